"""GPU parity of the NN, TN and TT layouts (dense; FP32 scales and packed UE8M0 scales) against the
CPU oracle.

The product is always D = A·Bᵀ of the logical A[M,K] and B[N,K]; the layouts only store A as [K,M]
(t) and/or B as [K,N] (second letter n). The oracle computes the logical product; the tests also
check that each layout gives the NT call's result bit for bit (same tile configuration and
accumulation order; the tensor core reads the transposed tiles directly).
"""
import numpy as np
import pytest
import torch

import dg_inputs
import oracle
from _dg_testlib import assert_accurate, bf16_sentinel, bits16, boundary_samples, dev, f32_sentinel, rne_bf16_bits

pytestmark = pytest.mark.gpu

LAYOUTS = {"nn": (False, True), "tn": (True, True), "tt": (True, False)}


@pytest.fixture(scope="module")
def dg():
    import moe_grouped_gemm_e4m3_gb300 as m
    m.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield m
    assert m.dg_get_device_status() == 0


def _run(dg, layout, a, b):
    M, K = a.A.shape
    N = b.B.shape[1]
    a_t, b_t = LAYOUTS[layout]
    A = dev(np.ascontiguousarray(a.A.T) if a_t else a.A)
    B = dev(np.ascontiguousarray(b.B[0].T) if b_t else b.B[0])
    sA, sB = dev(a.sA), dev(b.sB[0])
    D = bf16_sentinel((M, N))
    D32 = f32_sentinel((M, N))
    getattr(dg, f"dg_fp8_gemm_{layout}")(A, sA, B, sB, D, M, N, K)
    getattr(dg, f"dg_fp8_gemm_{layout}_f32")(A, sA, B, sB, D32, M, N, K)
    # the same product in the NT layout
    Dnt = f32_sentinel((M, N))
    dg.dg_fp8_gemm_nt_f32(dev(a.A), sA, dev(b.B[0]), sB, Dnt)
    torch.cuda.synchronize()
    return D, D32, Dnt


@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("M,N,K", [(128, 512, 1024), (256, 256, 384), (64, 2112, 7168), (320, 528, 640),
                                   (16, 16, 128), (1024, 4096, 512)])
def test_layout_full_parity(dg, layout, M, N, K):
    a = dg_inputs.make_a(M, K, seed=M + 3 * N)
    b = dg_inputs.make_b(1, N, K, seed=M + 3 * N)
    D, D32, Dnt = _run(dg, layout, a, b)
    assert torch.equal(D32.view(torch.int32), Dnt.view(torch.int32)), f"{layout}: differs from the NT result"
    ref64, _ = oracle.gemm_nt(a.A, a.sA, b.B[0], b.sB[0], want_bf16=False)
    dbits = bits16(D).cpu()
    assert torch.equal(dbits, rne_bf16_bits(D32))
    assert_accurate(D32.cpu().numpy(), dbits.numpy(), ref64, f"{layout} {M}x{N}x{K}")


@pytest.mark.parametrize("layout", list(LAYOUTS))
def test_layout_large_sampled(dg, layout):
    M, N, K = 4096, 7168, 2048
    a = dg_inputs.make_a(M, K, seed=0)
    b = dg_inputs.make_b(1, N, K, seed=0)
    D, D32, Dnt = _run(dg, layout, a, b)
    assert torch.equal(D32.view(torch.int32), Dnt.view(torch.int32))
    ms, ns = boundary_samples(M, N, 1500, seed=11, block_cols=256)
    ref = oracle.gemm_nt_sampled(a.A, a.sA, b.B[0], b.sB[0], ms, ns)
    assert_accurate(D32.cpu().numpy()[ms, ns], bits16(D).cpu().numpy()[ms, ns], ref, f"{layout} large")


def test_layout_alignment_errors(dg):
    a = dg_inputs.make_a(72, 128, seed=2)      # M = 72: not a multiple of 16
    b = dg_inputs.make_b(1, 136, 128, seed=2)  # N = 136: not a multiple of 16
    D = bf16_sentinel((72, 136))
    with pytest.raises(dg.DGError) as e:
        dg.dg_fp8_gemm_tt(dev(np.ascontiguousarray(a.A.T)), dev(a.sA), dev(b.B[0]), dev(b.sB[0]), D, 72, 136, 128)
    assert e.value.status == dg.DG_ERR_ALIGNMENT
    with pytest.raises(dg.DGError) as e:
        dg.dg_fp8_gemm_nn(dev(a.A), dev(a.sA), dev(np.ascontiguousarray(b.B[0].T)), dev(b.sB[0]), D, 72, 136, 128)
    assert e.value.status == dg.DG_ERR_ALIGNMENT


# ----------------------------------------------------------------------------------------------
# The same layouts on the block-scaled kernel (power-of-two scales packed as UE8M0): each must give
# the packed-UE8M0 NT call's result bit for bit, and match the oracle with the unpacked scales.

def _run_ue8m0(dg, layout, a, b):
    M, K = a.A.shape
    N = b.B.shape[1]
    a_t, b_t = LAYOUTS[layout]
    A = dev(np.ascontiguousarray(a.A.T) if a_t else a.A)
    B = dev(np.ascontiguousarray(b.B[0].T) if b_t else b.B[0])
    sA, sB = dev(dg_inputs.pack_ue8m0_a(a.sA)), dev(dg_inputs.pack_ue8m0_b(b.sB)[0])
    D = bf16_sentinel((M, N))
    D32 = f32_sentinel((M, N))
    getattr(dg, f"dg_fp8_gemm_{layout}_ue8m0")(A, sA, B, sB, D, M, N, K)
    getattr(dg, f"dg_fp8_gemm_{layout}_ue8m0_f32")(A, sA, B, sB, D32, M, N, K)
    Dnt = f32_sentinel((M, N))
    dg.dg_fp8_gemm_nt_ue8m0_f32(dev(a.A), sA, dev(b.B[0]), sB, Dnt)
    torch.cuda.synchronize()
    return D, D32, Dnt


@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("M,N,K", [(128, 512, 1024), (256, 256, 384), (64, 2112, 7168), (320, 528, 640),
                                   (16, 16, 128), (1024, 4096, 512)])
def test_layout_ue8m0_full_parity(dg, layout, M, N, K):
    a = dg_inputs.make_a(M, K, seed=M + 5 * N, ue8m0=True)
    b = dg_inputs.make_b(1, N, K, seed=M + 5 * N, ue8m0=True)
    D, D32, Dnt = _run_ue8m0(dg, layout, a, b)
    assert torch.equal(D32.view(torch.int32), Dnt.view(torch.int32)), f"{layout}/ue8m0: differs from the NT result"
    ref64, _ = oracle.gemm_nt(a.A, a.sA, b.B[0], b.sB[0], want_bf16=False)
    dbits = bits16(D).cpu()
    assert torch.equal(dbits, rne_bf16_bits(D32))
    assert_accurate(D32.cpu().numpy(), dbits.numpy(), ref64, f"{layout}/ue8m0 {M}x{N}x{K}")


@pytest.mark.parametrize("layout", list(LAYOUTS))
def test_layout_ue8m0_large_sampled(dg, layout):
    M, N, K = 4096, 7168, 2048
    a = dg_inputs.make_a(M, K, seed=1, ue8m0=True)
    b = dg_inputs.make_b(1, N, K, seed=1, ue8m0=True)
    D, D32, Dnt = _run_ue8m0(dg, layout, a, b)
    assert torch.equal(D32.view(torch.int32), Dnt.view(torch.int32))
    ms, ns = boundary_samples(M, N, 1500, seed=12, block_cols=256)
    ref = oracle.gemm_nt_sampled(a.A, a.sA, b.B[0], b.sB[0], ms, ns)
    assert_accurate(D32.cpu().numpy()[ms, ns], bits16(D).cpu().numpy()[ms, ns], ref, f"{layout}/ue8m0 large")
