"""GPU parity of the accumulating form D = C + A·Bᵀ (FP32 C and D) against the CPU oracle.

Besides the accuracy bar against the FP64 oracle (tests/_dg_testlib.py), each case checks that the
accumulating call equals fl32(C + D32) bit for bit, where D32 is the plain FP32 call's output: the
product reaches every element of D exactly once, with the same tile configuration and order.
"""
import numpy as np
import pytest
import torch

import dg_inputs
import oracle
from _dg_testlib import boundary_samples, dev, metrics, MAX_REL_TOL, COS_TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import moe_grouped_gemm_e4m3_gb300 as m
    m.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield m
    assert m.dg_get_device_status() == 0


def _inputs(M, N, K, ue8m0, seed):
    a = dg_inputs.make_a(M, K, seed=seed, ue8m0=ue8m0)
    b = dg_inputs.make_b(1, N, K, seed=seed, ue8m0=ue8m0)
    C = dg_inputs.draw(seed, 6, M * N).reshape(M, N) * np.float32(30.0)
    if ue8m0:
        nkb = (K + 127) // 128
        pa, pb = dg_inputs.pack_ue8m0_a(a.sA), dg_inputs.pack_ue8m0_b(b.sB)
        return a, b, C, pa, pb[0], oracle.unpack_ue8m0_a(pa, nkb), oracle.unpack_ue8m0_b(pb, nkb)[0]
    return a, b, C, a.sA, b.sB[0], a.sA, b.sB[0]


def _run(dg, ue8m0, a, b, C, gsA, gsB, in_place):
    M, K = a.A.shape
    N = b.B.shape[1]
    A, SA, B, SB = dev(a.A), dev(gsA), dev(b.B[0]), dev(gsB)
    plain = dg.dg_fp8_gemm_nt_ue8m0_f32 if ue8m0 else dg.dg_fp8_gemm_nt_f32
    acc = dg.dg_fp8_gemm_nt_ue8m0_acc_f32 if ue8m0 else dg.dg_fp8_gemm_nt_acc_f32
    D32 = torch.full((M, N), float("nan"), device="cuda")
    plain(A, SA, B, SB, D32)
    Ct = dev(C)
    if in_place:
        acc(A, SA, B, SB, Ct, Ct)
        Dacc = Ct
    else:
        Dacc = torch.full((M, N), float("nan"), device="cuda")
        acc(A, SA, B, SB, Ct, Dacc)
    torch.cuda.synchronize()
    return D32.cpu().numpy(), Dacc.cpu().numpy()


def _check(d_acc, d32, C, ref, what):
    want = (C.astype(np.float32) + d32.astype(np.float32)).astype(np.float32)
    assert np.array_equal(d_acc.view(np.int32), want.view(np.int32)), f"{what}: D != fl32(C + A·Bᵀ) bitwise"
    m = metrics(d_acc, ref)
    assert m["finite"] and m["max_rel"] <= MAX_REL_TOL and m["one_minus_cos"] <= COS_TOL, f"{what}: {m}"


@pytest.mark.parametrize("ue8m0", [False, True])
@pytest.mark.parametrize("M,N,K,in_place", [(128, 512, 1024, False), (200, 136, 1024, True), (65, 112, 400, False),
                                            (64, 2112, 7168, True), (300, 264, 768, False)])
def test_acc_full_parity(dg, ue8m0, M, N, K, in_place):
    a, b, C, gsA, gsB, osA, osB = _inputs(M, N, K, ue8m0, seed=M + N)
    d32, d_acc = _run(dg, ue8m0, a, b, C, gsA, gsB, in_place)
    ref = oracle.gemm_nt_acc(a.A, osA, b.B[0], osB, C)
    _check(d_acc, d32, C, ref, f"acc {'ue8m0' if ue8m0 else 'fp32'} {M}x{N}x{K}")


@pytest.mark.parametrize("ue8m0", [False, True])
def test_acc_large_sampled(dg, ue8m0):
    M, N, K = 4096, 7168, 2048
    a, b, C, gsA, gsB, osA, osB = _inputs(M, N, K, ue8m0, seed=3)
    d32, d_acc = _run(dg, ue8m0, a, b, C, gsA, gsB, in_place=True)
    want = (C + d32).astype(np.float32)
    assert np.array_equal(d_acc.view(np.int32), want.view(np.int32))
    ms, ns = boundary_samples(M, N, 1500, seed=5, block_cols=256)
    ref = oracle.gemm_nt_acc_sampled(a.A, osA, b.B[0], osB, C, ms, ns)
    m = metrics(d_acc[ms, ns], ref)
    assert m["max_rel"] <= MAX_REL_TOL and m["one_minus_cos"] <= COS_TOL, m


def test_acc_host_validation(dg):
    a, b, C, gsA, gsB, _, _ = _inputs(16, 64, 128, False, seed=1)
    A, SA, B, SB = dev(a.A), dev(gsA), dev(b.B[0]), dev(gsB)
    big = torch.zeros(16 * 64 + 64, dtype=torch.float32, device="cuda")
    Cv, Dv = big[:16 * 64].view(16, 64), big[64:].view(16, 64)      # overlapping, not identical
    with pytest.raises(dg.DGError) as e:
        dg.dg_fp8_gemm_nt_acc_f32(A, SA, B, SB, Cv, Dv)
    assert e.value.status == dg.DG_ERR_INVALID_ARG
    D = torch.zeros(16, 64, dtype=torch.float32, device="cuda")
    dg.dg_fp8_gemm_nt_acc_f32(A, SA, B, SB, dev(C), D)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(D).all())
