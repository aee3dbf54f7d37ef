"""The kernels' bounded waits, made to run out on purpose, on every kernel form.

Every pipeline wait inside the kernels has a time limit (dg_set_wait_limit_us; default 2 s). A
limit of 0 makes each wait that is not already satisfied give up at once: the kernel then records
DG_DEV_TIMEOUT, stops issuing, waits (with its own fixed bound) for the copies and MMAs already in
flight, frees its tensor memory and returns. No fault, trap or hang is involved: the test checks
that such a launch sets the status bit, and that with the default limit restored the very next call
on the same stream gives the same bits as before (which the other GPU tests tie to the oracle), so
the context, the split-K counters and the scratch all recovered.
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
    assert m.dg_get_device_status() == 0
    yield m
    m.dg_set_wait_limit_us(-1)
    assert m.dg_get_device_status() == 0


def _timeout_then_recover(dg, call, out):
    """call() writes `out`; returns after checking the timeout and the recovery."""
    call()
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    ref = out.clone()
    prev = dg.dg_set_wait_limit_us(0)
    try:
        assert prev == 2000000
        call()
        status = dg.dg_get_device_status()    # synchronises; reads and clears the status word
    finally:
        dg.dg_set_wait_limit_us(prev)
    assert status & dg.DG_DEV_TIMEOUT, f"no wait gave up (status 0x{status:x})"
    out.view(torch.int8).fill_(-1)
    call()
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    assert torch.equal(out.view(torch.int8), ref.view(torch.int8)), "the call after a timeout differs"


def _dense(dg, M, N, K, seed=0):
    a = dg_inputs.make_a(M, K, seed=seed)
    b = dg_inputs.make_b(1, N, K, seed=seed)
    A, sA, B, sB = dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0])
    D = bf16_sentinel((M, N))
    return (lambda: dg.dg_fp8_gemm_nt(A, sA, B, sB, D)), D


def test_timeout_dense_persistent(dg):
    call, D = _dense(dg, 4096, 2112, 1024)
    _timeout_then_recover(dg, call, D)


def test_timeout_dense_global_split_k(dg):
    prev = dg.dg_set_cluster_split(False)     # partials and arrival counters in global memory
    try:
        call, D = _dense(dg, 128, 4096, 7168, seed=1)
        assert dg.dg_query_config(0, 128, 4096, 7168)["splits"] > 1
        _timeout_then_recover(dg, call, D)
    finally:
        dg.dg_set_cluster_split(prev)


def test_timeout_dense_cluster_split_k(dg):
    # split-K inside thread-block clusters: a CTA that gives up holds no partial, and the cluster
    # leaves D alone instead of summing stale shared memory
    call, D = _dense(dg, 64, 2112, 7168, seed=2)
    _timeout_then_recover(dg, call, D)


def test_timeout_dense_tail_split(dg):
    call, D = _dense(dg, 4096, 4096, 7168, seed=3)
    _timeout_then_recover(dg, call, D)


def test_timeout_noalloc(dg):
    prev = dg.dg_set_cluster_split(False)
    try:
        M, N, K = 64, 2112, 7168
        a = dg_inputs.make_a(M, K, seed=4)
        b = dg_inputs.make_b(1, N, K, seed=4)
        A, sA, B, sB = dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0])
        D = bf16_sentinel((M, N))
        _timeout_then_recover(dg, lambda: dg.dg_fp8_gemm_nt_noalloc(A, sA, B, sB, D), D)
    finally:
        dg.dg_set_cluster_split(prev)


def test_timeout_contiguous(dg):
    m_idx = dg_inputs.contiguous_m_indices([300, 0, 520, 128])
    K, N, G = 2048, 1024, 4
    a = dg_inputs.make_a(len(m_idx), K, seed=5)
    b = dg_inputs.make_b(G, N, K, seed=5)
    A, sA, B, sB, I = dev(a.A), dev(a.sA), dev(b.B), dev(b.sB), dev(m_idx)
    D = bf16_sentinel((len(m_idx), N))
    _timeout_then_recover(dg, lambda: dg.dg_fp8_grouped_contiguous(A, sA, B, sB, I, D), D)


def test_timeout_masked(dg):
    G, M_max, N, K = 16, 256, 2048, 2048
    mm = dg_inputs.make_masked_m(G, M_max, seed=6)
    a = dg_inputs.make_masked_a(G, M_max, K, seed=6)
    b = dg_inputs.make_b(G, N, K, seed=6)
    A, sA, B, sB, MM = dev(a.A), dev(a.sA), dev(b.B), dev(b.sB), dev(mm)
    D = bf16_sentinel((G, M_max, N))
    _timeout_then_recover(dg, lambda: dg.dg_fp8_grouped_masked(A, sA, B, sB, MM, D), D)


def test_timeout_masked_swiglu(dg):
    G, M_max, N2, K = 8, 192, 1024, 1024
    mm = dg_inputs.make_masked_m(G, M_max, seed=7)
    a = dg_inputs.make_masked_a(G, M_max, K, seed=7)
    b = dg_inputs.make_b(G, N2, K, seed=7)
    A, sA, B, sB, MM = dev(a.A), dev(a.sA), dev(b.B), dev(b.sB), dev(mm)
    H = bf16_sentinel((G, M_max, N2 // 2))
    _timeout_then_recover(dg, lambda: dg.dg_fp8_grouped_masked_swiglu(A, sA, B, sB, MM, H), H)


def test_timeout_masked_swiglu_fp8(dg):
    # H cast to FP8: the codes (Hq) and the scales (sH) both come back unchanged after a timeout
    G, M_max, N2, K = 8, 192, 1024, 1024
    mm = dg_inputs.make_masked_m(G, M_max, seed=8)
    a = dg_inputs.make_masked_a(G, M_max, K, seed=8)
    b = dg_inputs.make_b(G, N2, K, seed=8)
    A, sA, B, sB, MM = dev(a.A), dev(a.sA), dev(b.B), dev(b.sB), dev(mm)
    Hq = torch.full((G, M_max, N2 // 2), 0xFF, dtype=torch.uint8, device="cuda")
    sH = torch.full((G, N2 // 2 // 128, M_max), float("nan"), dtype=torch.float32, device="cuda")
    call = lambda: dg.dg_fp8_grouped_masked_swiglu_fp8(A, sA, B, sB, MM, Hq, sH)
    call()
    torch.cuda.synchronize()
    ref_s = sH.clone()
    _timeout_then_recover(dg, call, Hq)
    assert torch.equal(sH.view(torch.int32), ref_s.view(torch.int32)), "the scales after a timeout differ"


def test_timeout_masked_swiglu_ue8m0(dg):
    G, M_max, N2, K = 8, 192, 1024, 1024
    mm = dg_inputs.make_masked_m(G, M_max, seed=9)
    a = dg_inputs.make_masked_a(G, M_max, K, seed=9, ue8m0=True)
    b = dg_inputs.make_b(G, N2, K, seed=9, ue8m0=True)
    A, B, MM = dev(a.A), dev(b.B), dev(mm)
    sA, sB = dev(dg_inputs.pack_ue8m0_a(a.sA)), dev(dg_inputs.pack_ue8m0_b(b.sB))
    H = bf16_sentinel((G, M_max, N2 // 2))
    _timeout_then_recover(dg, lambda: dg.dg_fp8_grouped_masked_swiglu_ue8m0(A, sA, B, sB, MM, H), H)


def test_timeout_k_grouped(dg):
    M, N, off = 512, 1024, np.array([0, 1024, 1024, 3072], np.int32)
    K = int(off[-1])
    a = dg_inputs.make_a(M, K, seed=8)
    b = dg_inputs.make_b(1, N, K, seed=8)
    A, B = dev(np.ascontiguousarray(a.A.T)), dev(np.ascontiguousarray(b.B[0].T))
    sA, sB, O = dev(a.sA), dev(b.sB[0]), dev(off)
    D = bf16_sentinel((len(off) - 1, M, N))
    _timeout_then_recover(dg, lambda: dg.dg_fp8_k_grouped_gemm_tn_contiguous(A, sA, B, sB, O, D), D)


@pytest.mark.parametrize("M,N,K", [(4096, 2112, 2048), (64, 2112, 7168)])
def test_timeout_block_scaled(dg, M, N, K):
    a = dg_inputs.make_a(M, K, seed=9, ue8m0=True)
    b = dg_inputs.make_b(1, N, K, seed=9, ue8m0=True)
    pa, pb = dg_inputs.pack_ue8m0_a(a.sA), dg_inputs.pack_ue8m0_b(b.sB)
    A, sA, B, sB = dev(a.A), dev(pa), dev(b.B[0]), dev(pb[0])
    D = bf16_sentinel((M, N))
    _timeout_then_recover(dg, lambda: dg.dg_fp8_gemm_nt_ue8m0(A, sA, B, sB, D), D)


def test_timeout_k_grouped_ue8m0(dg):
    M, N, off = 512, 1024, np.array([0, 1024, 1024, 3072], np.int32)
    K = int(off[-1])
    a = dg_inputs.make_a(M, K, seed=10, ue8m0=True)
    b = dg_inputs.make_b(1, N, K, seed=10, ue8m0=True)
    A, B = dev(np.ascontiguousarray(a.A.T)), dev(np.ascontiguousarray(b.B[0].T))
    sA, sB, O = dev(dg_inputs.pack_ue8m0_a(a.sA)), dev(dg_inputs.pack_ue8m0_b(b.sB)[0]), dev(off)
    D = bf16_sentinel((len(off) - 1, M, N))
    _timeout_then_recover(dg, lambda: dg.dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0(A, sA, B, sB, O, D), D)
