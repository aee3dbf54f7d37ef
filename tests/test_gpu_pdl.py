"""Programmatic dependent launch (dg_set_pdl): back-to-back calls on one stream, each launched so that
it may start while the previous kernel still runs, must give the same bits as calls in plain stream
order.

The chains are built so that a kernel that read its inputs before the previous kernel finished would
be caught. The fused SwiGLU with FP8 H writes Hq and sH, and the masked GEMM right after it reads
them as A and sA; the first launch is small, so the second one's CTAs find idle SMs and start early.
The buffers are poisoned before every chain. Split-K launches reuse the workspace and arrival
counters of the call before them.
"""
import numpy as np
import pytest
import torch

import dg_inputs
from _dg_testlib import bf16_sentinel, bits16, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import moe_grouped_gemm_e4m3_gb300 as m
    m.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    prev = m.dg_set_pdl(False)
    yield m
    m.dg_set_pdl(prev)
    assert m.dg_get_device_status() == 0


def _with_pdl(dg, on, fn):
    prev = dg.dg_set_pdl(on)
    try:
        assert dg.dg_get_pdl() == on
        return fn()
    finally:
        dg.dg_set_pdl(prev)


def test_pdl_swiglu_fp8_then_down_projection(dg):
    G, M_max, I, K, N2 = 2, 64, 256, 1024, 2048
    masked_m = np.array([40, 64], np.int32)
    a = dg_inputs.make_masked_a(G, M_max, K, seed=21)
    b = dg_inputs.make_b(G, 2 * I, K, seed=21)
    w2 = dg_inputs.make_b(G, N2, I, seed=22)
    A, sA, B, sB, MM = dev(a.A), dev(a.sA), dev(b.B), dev(b.sB), dev(masked_m)
    W2, sW2 = dev(w2.B), dev(w2.sB)
    Hq = torch.empty((G, M_max, I), dtype=torch.uint8, device="cuda")
    sH = torch.empty((G, I // 128, M_max), dtype=torch.float32, device="cuda")

    def chain(reps):
        outs = []
        for _ in range(reps):
            Hq.fill_(0x7F)                       # NaN codes: a read before the cast finished shows up
            sH.fill_(float("nan"))
            D2 = bf16_sentinel((G, M_max, N2))
            dg.dg_fp8_grouped_masked_swiglu_fp8(A, sA, B, sB, MM, Hq, sH)
            dg.dg_fp8_grouped_masked(Hq, sH, W2, sW2, MM, D2)
            outs.append(D2)
        torch.cuda.synchronize()
        return [bits16(d).cpu() for d in outs]

    ref = _with_pdl(dg, False, lambda: chain(1))[0]
    got = _with_pdl(dg, True, lambda: chain(20))
    assert dg.dg_get_device_status() == 0
    for i, g in enumerate(got):
        assert torch.equal(g, ref), f"chain {i} with PDL differs from plain stream order"


@pytest.mark.parametrize("cluster", [True, False])
def test_pdl_back_to_back_split_k(dg, cluster):
    # small-M launches that split K: in clusters, or through the shared workspace and its counters
    shapes = [(64, 2112, 7168), (128, 4096, 7168), (64, 7168, 2048)]
    calls = []
    for i, (M, N, K) in enumerate(shapes):
        a = dg_inputs.make_a(M, K, seed=30 + i)
        b = dg_inputs.make_b(1, N, K, seed=30 + i)
        calls.append((dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0]), (M, N)))

    def run(reps):
        outs = []
        for _ in range(reps):
            for (A, sA, B, sB, (M, N)) in calls:
                D = bf16_sentinel((M, N))
                dg.dg_fp8_gemm_nt(A, sA, B, sB, D)
                outs.append(D)
        torch.cuda.synchronize()
        return [bits16(d).cpu() for d in outs]

    prev = dg.dg_set_cluster_split(cluster)
    try:
        ref = _with_pdl(dg, False, lambda: run(1))
        got = _with_pdl(dg, True, lambda: run(8))
    finally:
        dg.dg_set_cluster_split(prev)
    assert dg.dg_get_device_status() == 0
    for i, g in enumerate(got):
        assert torch.equal(g, ref[i % len(calls)]), f"call {i} with PDL differs from plain stream order"


def test_pdl_block_scaled_back_to_back(dg):
    M, N, K = 64, 7168, 16384
    a = dg_inputs.make_a(M, K, seed=40, ue8m0=True)
    b = dg_inputs.make_b(1, N, K, seed=40, ue8m0=True)
    A, B = dev(a.A), dev(b.B[0])
    sA, sB = dev(dg_inputs.pack_ue8m0_a(a.sA)), dev(dg_inputs.pack_ue8m0_b(b.sB)[0])

    def run(reps):
        outs = []
        for _ in range(reps):
            D = bf16_sentinel((M, N))
            dg.dg_fp8_gemm_nt_ue8m0(A, sA, B, sB, D)
            outs.append(D)
        torch.cuda.synchronize()
        return [bits16(d).cpu() for d in outs]

    ref = _with_pdl(dg, False, lambda: run(1))[0]
    for i, g in enumerate(_with_pdl(dg, True, lambda: run(10))):
        assert torch.equal(g, ref), f"call {i} with PDL differs"
