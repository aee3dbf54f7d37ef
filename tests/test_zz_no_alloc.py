"""The allocation-free dense entry point, dg_fp8_gemm_nt_noalloc, through the C ABI.

It exists for callers that cannot let libdg call cudaMalloc (a framework whose caching allocator
owns the device memory, a serving loop that must not block on cudaMalloc's synchronisation). Its
split-K scratch is a fixed array inside the library that every call reuses. The shapes here are
chosen so that the array is really used: split-K with the exchange through global memory (split-K
inside thread-block clusters, which needs no scratch, is switched off around them) and a tail
split; one shape needs none. Each is called twice in a row (the array keeps the previous call's
contents) and checked against the allocating entry point, dg_fp8_gemm_nt — bit for bit, since both
run one code path with the same schedule — and against the oracle on sampled elements within the
parity tests' tolerance. A shape whose partials exceed the array must be refused. The file name
sorts last so that a run stopping at the first failure has already run every other test; it passes
alone in a fresh process too.
"""
import os

import numpy as np
import pytest
import torch

import dg_inputs
import oracle
from _dg_testlib import COS_TOL, MAX_REL_TOL, assert_accurate, bf16_sentinel, bits16, boundary_samples, dev, metrics

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import moe_grouped_gemm_e4m3_gb300 as m
    m.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return m


@pytest.fixture
def global_split_k(dg):
    """Split-K through global memory (and so through the fixed array): no cluster exchange."""
    prev = dg.dg_set_cluster_split(False)
    try:
        yield
    finally:
        dg.dg_set_cluster_split(prev)


def _check_twice(dg, M, N, K, seed):
    a = dg_inputs.make_a(M, K, seed=seed)
    b = dg_inputs.make_b(1, N, K, seed=seed + 1)
    A, sA, B, sB = dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0])
    ref = bf16_sentinel((M, N))
    ref32 = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    dg.dg_fp8_gemm_nt(A, sA, B, sB, ref)
    dg.dg_fp8_gemm_nt_f32(A, sA, B, sB, ref32)
    outs = []
    for _ in range(2):                       # the scratch array keeps the previous call's contents
        D = bf16_sentinel((M, N))
        dg.dg_fp8_gemm_nt_noalloc(A, sA, B, sB, D)
        outs.append(D)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    r = ref.float().cpu().numpy()
    for D in outs:
        assert not torch.any(bits16(D) == -1), "output not fully written"
        m = metrics(D.float().cpu().numpy(), r)
        assert m["finite"] and m["max_rel"] <= MAX_REL_TOL and m["one_minus_cos"] <= COS_TOL, m
        assert torch.equal(bits16(D), bits16(ref))
    # the shared result against the oracle, on samples that cover every tile edge
    ms, ns = boundary_samples(M, N, 1024, seed=seed, block_cols=256)
    ref64 = oracle.gemm_nt_sampled(a.A, a.sA, b.B[0], b.sB[0], ms, ns)
    d32 = ref32.cpu().numpy()[ms, ns]
    assert_accurate(d32, bits16(outs[1]).cpu().numpy()[ms, ns], ref64, f"noalloc {M}x{N}x{K}")


# few output tiles: every tile's K is split and the partials go through the fixed array
@pytest.mark.parametrize("M,N,K", [(64, 2112, 7168), (128, 4096, 7168), (100, 1000, 2048)])
def test_noalloc_split_k_through_the_array(dg, global_split_k, M, N, K):
    cfg = dg.dg_query_config(0, M, N, K)
    assert cfg["splits"] > 1, cfg                 # the global split-K path, which uses the array
    _check_twice(dg, M, N, K, seed=M + K)


def test_noalloc_tail_split_through_the_array(dg):
    # 512 tiles on 152 SMs leave a last wave of 56 tiles (at most half the grid): the kernel cuts
    # them along K, and their partials go through the fixed array
    # (single CTAs: a launch by pairs of CTAs sharing B tiles has no tail split)
    M, N, K = 4096, 4096, 7168
    prev_pair = dg.dg_set_pair_b(False)
    prev = dg.dg_set_tail_splits(4)
    try:
        cfg = dg.dg_query_config(0, M, N, K)
        assert cfg["splits"] == 1 and 0 < cfg["tiles"] % cfg["grid"] <= cfg["grid"] // 2, cfg
        _check_twice(dg, M, N, K, seed=7)
    finally:
        dg.dg_set_tail_splits(prev)
        dg.dg_set_pair_b(prev_pair)


def test_noalloc_pairs_sharing_b(dg):
    # pairs of CTAs sharing B tiles (opt-in): no scratch
    prev = dg.dg_set_pair_b(True)
    try:
        assert dg.dg_query_config(0, 4096, 2112, 1024)["block_m"] == 256
        _check_twice(dg, 4096, 2112, 1024, seed=11)
    finally:
        dg.dg_set_pair_b(prev)


def test_noalloc_needs_no_scratch(dg):
    _check_twice(dg, 4096, 2112, 1024, seed=3)


def test_noalloc_refuses_a_shape_beyond_the_array(dg, global_split_k):
    # 28 tiles x 16 K ranges x 128 KiB of FP32 partials = 56 MiB > the 20 MiB the array holds
    M, N, K = 128, 7168, 16384
    a = dg_inputs.make_a(M, K, seed=5)
    b = dg_inputs.make_b(1, N, K, seed=5)
    A, sA, B, sB = dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0])
    D = bf16_sentinel((M, N))
    os.environ["DG_SPLITS"] = "16"
    try:
        with pytest.raises(dg.DGError) as e:
            dg.dg_fp8_gemm_nt_noalloc(A, sA, B, sB, D)
        assert e.value.status == dg.DG_ERR_UNSUPPORTED
        assert "fixed scratch" in str(e.value)
        # the allocating entry point has no such limit
        dg.dg_fp8_gemm_nt(A, sA, B, sB, D)
        torch.cuda.synchronize()
        assert not torch.any(bits16(D) == -1)
    finally:
        del os.environ["DG_SPLITS"]
    assert dg.dg_get_device_status() == 0


def test_noalloc_rejects_bad_arguments(dg):
    a = dg_inputs.make_a(16, 128, seed=1)
    b = dg_inputs.make_b(1, 64, 128, seed=1)
    D = bf16_sentinel((16, 60))
    with pytest.raises(dg.DGError) as e:
        dg.dg_fp8_gemm_nt_noalloc(dev(a.A), dev(a.sA), dev(b.B[0][:60].copy()), dev(b.sB[0]), D)
    assert e.value.status == dg.DG_ERR_ALIGNMENT
