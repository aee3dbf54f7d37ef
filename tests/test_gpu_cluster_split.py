"""GPU parity of split-K inside thread-block clusters (dense and contiguous, FP32 scales).

When a call splits K into at most 8 ranges and every tile's ranges fit on the GPU at once as one
cluster, the ranges reduce through distributed shared memory. Otherwise they use the global
workspace. Both sum the partials in range order, so each case checks that:
- the two paths give bitwise-equal results (dg_set_cluster_split on / off) when they split K the
  same way (a split count whose clusters do not all fit is lowered by one or two in cluster mode);
- the cluster path really ran (the DG_PRINT_CONFIGS line says "(cluster)");
- the result is accurate against the FP64 oracle;
- rows that must stay untouched are untouched.
"""
import os

import numpy as np
import pytest
import torch

import dg_inputs
import oracle
from _dg_testlib import assert_accurate, bf16_sentinel, bits16, boundary_samples, dev, f32_sentinel, rne_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import moe_grouped_gemm_e4m3_gb300 as m
    m.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield m
    assert m.dg_get_device_status() == 0


def _both(dg, run, capfd):
    """run() with clusters allowed (checking that they were used), then with the global workspace."""
    os.environ["DG_PRINT_CONFIGS"] = "1"
    try:
        capfd.readouterr()
        on = run()
        err = capfd.readouterr().err
    finally:
        del os.environ["DG_PRINT_CONFIGS"]
    assert "(cluster)" in err, f"the cluster split-K did not run:\n{err}"
    prev = dg.dg_set_cluster_split(False)
    try:
        off = run()
    finally:
        dg.dg_set_cluster_split(prev)
    return on, off


@pytest.mark.parametrize("M,N,K", [(64, 7168, 16384), (128, 7168, 16384), (64, 4096, 7168), (100, 7168, 2048), (64, 2112, 7168),
                                   (128, 512, 1024), (16, 264, 3072)])
def test_cluster_split_dense(dg, capfd, M, N, K):
    cfg = dg.dg_query_config(0, M, N, K)
    if not (2 <= cfg["splits"] <= 8):
        pytest.skip(f"configuration does not split K into 2..8 ranges: {cfg}")
    a = dg_inputs.make_a(M, K, seed=M + N)
    b = dg_inputs.make_b(1, N, K, seed=M + N)
    A, sA, B, sB = dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0])

    def run():
        D = bf16_sentinel((M, N))
        D32 = f32_sentinel((M, N))
        dg.dg_fp8_gemm_nt(A, sA, B, sB, D)
        dg.dg_fp8_gemm_nt_f32(A, sA, B, sB, D32)
        torch.cuda.synchronize()
        return bits16(D).cpu(), D32.cpu()

    (d_on, f_on), (d_off, f_off) = _both(dg, run, capfd)
    prev = dg.dg_set_cluster_split(False)
    try:
        cfg_off = dg.dg_query_config(0, M, N, K)
    finally:
        dg.dg_set_cluster_split(prev)
    if cfg_off["splits"] == cfg["splits"]:
        assert torch.equal(d_on, d_off) and torch.equal(f_on.view(torch.int32), f_off.view(torch.int32))
    assert torch.equal(d_on, rne_bf16_bits(f_on))
    ms, ns = boundary_samples(M, N, 1500, seed=3, block_cols=128)
    ref = oracle.gemm_nt_sampled(a.A, a.sA, b.B[0], b.sB[0], ms, ns)
    assert_accurate(f_on.numpy()[ms, ns], d_on.numpy()[ms, ns], ref, f"cluster split {M}x{N}x{K}")
    assert_accurate(f_off.numpy()[ms, ns], d_off.numpy()[ms, ns], ref, f"global split {M}x{N}x{K}")


def test_cluster_split_contiguous_with_padding(dg, capfd):
    # 3 groups with 70, 0 and 120 rows (two 128-row blocks); K long enough to split
    m_idx = dg_inputs.contiguous_m_indices([70, 0, 120])
    rows, N, K, G = len(m_idx), 1024, 4096, 3
    cfg = dg.dg_query_config(1, rows, N, K, G)
    if not (2 <= cfg["splits"] <= 8):
        pytest.skip(f"configuration does not split K into 2..8 ranges: {cfg}")
    a = dg_inputs.make_a(rows, K, seed=8)
    b = dg_inputs.make_b(G, N, K, seed=8)
    A, sA, B, sB, I = dev(a.A), dev(a.sA), dev(b.B), dev(b.sB), dev(m_idx)

    def run():
        D32 = f32_sentinel((rows, N))
        dg.dg_fp8_grouped_contiguous_f32(A, sA, B, sB, I, D32)
        torch.cuda.synchronize()
        return D32.cpu()

    f_on, f_off = _both(dg, run, capfd)
    assert torch.equal(f_on.view(torch.int32), f_off.view(torch.int32))
    pad = torch.from_numpy(m_idx < 0)
    assert bool(torch.isnan(f_on[pad]).all()), "padding rows were written"
    v = m_idx >= 0
    ref64, _, _ = oracle.grouped_contiguous(a.A, a.sA, b.B, b.sB, m_idx)
    d = f_on.numpy()[v]
    bits = torch.from_numpy(d.copy()).to(torch.bfloat16).view(torch.int16).numpy()
    assert_accurate(d, bits, ref64[v], "cluster split contiguous")


def test_cluster_split_accumulate_and_layout(dg, capfd):
    M, N, K = 64, 4096, 7168
    cfg = dg.dg_query_config(0, M, N, K)
    if not (2 <= cfg["splits"] <= 8):
        pytest.skip(f"configuration does not split K into 2..8 ranges: {cfg}")
    a = dg_inputs.make_a(M, K, seed=9)
    b = dg_inputs.make_b(1, N, K, seed=9)
    A, sA, B, sB = dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0])
    C = dg_inputs.draw(9, 6, M * N).reshape(M, N) * np.float32(30.0)

    def run():
        D32 = torch.full((M, N), float("nan"), device="cuda")
        dg.dg_fp8_gemm_nt_f32(A, sA, B, sB, D32)
        Ct = dev(C)
        dg.dg_fp8_gemm_nt_acc_f32(A, sA, B, sB, Ct, Ct)
        Dnn = f32_sentinel((M, N))
        dg.dg_fp8_gemm_nn_f32(A, sA, dev(np.ascontiguousarray(b.B[0].T)), sB, Dnn, M, N, K)
        torch.cuda.synchronize()
        return D32.cpu().numpy(), Ct.cpu().numpy(), Dnn.cpu().numpy()

    (d32, acc, dnn), (d32_off, acc_off, dnn_off) = _both(dg, run, capfd)
    want = (C.astype(np.float32) + d32).astype(np.float32)
    assert np.array_equal(acc.view(np.int32), want.view(np.int32)), "D != fl32(C + A·Bᵀ) bitwise"
    assert np.array_equal(dnn.view(np.int32), d32.view(np.int32)), "NN layout differs from NT"
    for x, y in ((d32, d32_off), (acc, acc_off), (dnn, dnn_off)):
        assert np.array_equal(x.view(np.int32), y.view(np.int32))


def _ue8m0(a, b):
    """Packed UE8M0 words (what the GPU gets) and the FP32 scales the oracle decodes from them."""
    nkb = -(-a.A.shape[-1] // 128)
    pa, pb = dg_inputs.pack_ue8m0_a(a.sA), dg_inputs.pack_ue8m0_b(b.sB)
    return pa, pb, oracle.unpack_ue8m0_a(pa, nkb), oracle.unpack_ue8m0_b(pb, nkb)


@pytest.mark.parametrize("M,N,K", [(64, 7168, 16384), (64, 4096, 7168), (64, 2112, 7168), (128, 512, 1024)])
def test_cluster_split_dense_ue8m0(dg, capfd, M, N, K):
    cfg = dg.dg_query_config_ue8m0(0, M, N, K)
    if not (2 <= cfg["splits"] <= 8):
        pytest.skip(f"configuration does not split K into 2..8 ranges: {cfg}")
    a = dg_inputs.make_a(M, K, seed=M + N + 1, ue8m0=True)
    b = dg_inputs.make_b(1, N, K, seed=M + N + 1, ue8m0=True)
    pa, pb, osA, osB = _ue8m0(a, b)
    A, sA, B, sB = dev(a.A), dev(pa), dev(b.B[0]), dev(pb[0])

    def run():
        D = bf16_sentinel((M, N))
        D32 = f32_sentinel((M, N))
        dg.dg_fp8_gemm_nt_ue8m0(A, sA, B, sB, D)
        dg.dg_fp8_gemm_nt_ue8m0_f32(A, sA, B, sB, D32)
        torch.cuda.synchronize()
        return bits16(D).cpu(), D32.cpu()

    (d_on, f_on), (d_off, f_off) = _both(dg, run, capfd)
    prev = dg.dg_set_cluster_split(False)
    try:
        cfg_off = dg.dg_query_config_ue8m0(0, M, N, K)
    finally:
        dg.dg_set_cluster_split(prev)
    if cfg_off["splits"] == cfg["splits"]:
        assert torch.equal(d_on, d_off) and torch.equal(f_on.view(torch.int32), f_off.view(torch.int32))
    assert torch.equal(d_on, rne_bf16_bits(f_on))
    ms, ns = boundary_samples(M, N, 1500, seed=4, block_cols=128)
    ref = oracle.gemm_nt_sampled(a.A, osA, b.B[0], osB[0], ms, ns)
    assert_accurate(f_on.numpy()[ms, ns], d_on.numpy()[ms, ns], ref, f"ue8m0 cluster split {M}x{N}x{K}")
    assert_accurate(f_off.numpy()[ms, ns], d_off.numpy()[ms, ns], ref, f"ue8m0 global split {M}x{N}x{K}")


def test_cluster_split_contiguous_ue8m0_with_padding(dg, capfd):
    m_idx = dg_inputs.contiguous_m_indices([70, 0, 120])
    rows, N, K, G = len(m_idx), 1024, 4096, 3
    cfg = dg.dg_query_config_ue8m0(1, rows, N, K, G)
    if not (2 <= cfg["splits"] <= 8):
        pytest.skip(f"configuration does not split K into 2..8 ranges: {cfg}")
    a = dg_inputs.make_a(rows, K, seed=10, ue8m0=True)
    b = dg_inputs.make_b(G, N, K, seed=10, ue8m0=True)
    pa, pb, osA, osB = _ue8m0(a, b)
    A, sA, B, sB, I = dev(a.A), dev(pa), dev(b.B), dev(pb), dev(m_idx)

    def run():
        D32 = f32_sentinel((rows, N))
        dg.dg_fp8_grouped_contiguous_ue8m0_f32(A, sA, B, sB, I, D32)
        torch.cuda.synchronize()
        return D32.cpu()

    f_on, f_off = _both(dg, run, capfd)
    pad = torch.from_numpy(m_idx < 0)
    assert bool(torch.isnan(f_on[pad]).all()), "padding rows were written"
    v = m_idx >= 0
    ref64, _, _ = oracle.grouped_contiguous(a.A, osA, b.B, osB, m_idx)
    for f, what in ((f_on, "on"), (f_off, "off")):
        d = f.numpy()[v]
        bits = torch.from_numpy(d.copy()).to(torch.bfloat16).view(torch.int16).numpy()
        assert_accurate(d, bits, ref64[v], f"ue8m0 cluster split contiguous {what}")
