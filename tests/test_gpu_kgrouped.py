"""GPU parity of the K-grouped contiguous GEMM (groups along K; A stored [K,M], B stored [K,N]), with
FP32 scales and with packed UE8M0 scales (the block-scaled kernel).

D[g] sums the K-blocks of segment g (k_offsets on the device). Checked against the oracle on the
logical A[M,K] and B[N,K]: whole-output parity with an empty segment (zeros), BF16 == RNE(FP32), a
large weight-gradient-sized case sampled, and invalid offsets flagged with that group untouched.
"""
import numpy as np
import pytest
import torch

import dg_inputs
import oracle
from _dg_testlib import assert_accurate, bf16_sentinel, bits16, dev, f32_sentinel, rne_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import moe_grouped_gemm_e4m3_gb300 as m
    m.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield m
    assert m.dg_get_device_status() == 0


def _run(dg, a, b, off):
    M, K = a.A.shape
    N = b.B.shape[1]
    G = len(off) - 1
    A, B = dev(np.ascontiguousarray(a.A.T)), dev(np.ascontiguousarray(b.B[0].T))
    sA, sB, O = dev(a.sA), dev(b.sB[0]), dev(np.asarray(off, np.int32))
    D = bf16_sentinel((G, M, N))
    D32 = f32_sentinel((G, M, N))
    dg.dg_fp8_k_grouped_gemm_tn_contiguous(A, sA, B, sB, O, D)
    dg.dg_fp8_k_grouped_gemm_tn_contiguous_f32(A, sA, B, sB, O, D32)
    torch.cuda.synchronize()
    return D, D32


@pytest.mark.parametrize("M,N,off", [(192, 272, [0, 256, 256, 640, 1024]), (128, 128, [0, 128]),
                                     (64, 528, [0, 512, 1024, 1024]), (320, 256, [0, 0, 384, 1152])])
def test_k_grouped_full_parity(dg, M, N, off):
    K = off[-1]
    a = dg_inputs.make_a(M, K, seed=M + N)
    b = dg_inputs.make_b(1, N, K, seed=M + N)
    D, D32 = _run(dg, a, b, off)
    ref = oracle.k_grouped(a.A, a.sA, b.B[0], b.sB[0], np.array(off, np.int32))
    db = bits16(D).cpu()
    assert torch.equal(db, rne_bf16_bits(D32))
    for g in range(len(off) - 1):
        if off[g] == off[g + 1]:
            assert torch.all(D32[g] == 0) and torch.all(db[g] == 0), f"empty group {g} is not zero"
    nz = [g for g in range(len(off) - 1) if off[g] != off[g + 1]]
    assert_accurate(D32.cpu().numpy()[nz], db.numpy()[nz], ref[nz], f"k-grouped {M}x{N} {off}")


def test_k_grouped_large_sampled(dg):
    M, N = 2048, 7168
    off = [0, 1024, 1024, 3072, 3584]
    K = off[-1]
    a = dg_inputs.make_a(M, K, seed=0)
    b = dg_inputs.make_b(1, N, K, seed=0)
    D, D32 = _run(dg, a, b, off)
    assert torch.equal(bits16(D).cpu(), rne_bf16_bits(D32))
    assert torch.all(D32[1] == 0)
    rng = np.random.default_rng(3)
    for g in (0, 2, 3):
        k0, k1 = off[g], off[g + 1]
        ms, ns = rng.integers(0, M, 600), rng.integers(0, N, 600)
        kb = slice(k0 // 128, k1 // 128)
        ref = oracle.gemm_nt_sampled(np.ascontiguousarray(a.A[:, k0:k1]), np.ascontiguousarray(a.sA[kb]),
                                     np.ascontiguousarray(b.B[0][:, k0:k1]), np.ascontiguousarray(b.sB[0][:, kb]),
                                     ms, ns)
        assert_accurate(D32[g].cpu().numpy()[ms, ns], bits16(D[g]).cpu().numpy()[ms, ns], ref, f"k-grouped g={g}")


def test_k_grouped_bad_offsets_flagged_and_untouched(dg):
    M, N = 64, 128
    off = [0, 100, 256]                 # 100 is not a multiple of 128: both groups touching it are invalid
    a = dg_inputs.make_a(M, 256, seed=4)
    b = dg_inputs.make_b(1, N, 256, seed=4)
    assert dg.dg_get_device_status() == 0
    D, _ = _run(dg, a, b, off)
    assert dg.dg_get_device_status() & dg.DG_DEV_BAD_GROUP_INDEX
    assert torch.all(bits16(D).cpu() == -1)


# ----------------------------------------------------------------------------------------------
# The K-grouped form on the block-scaled kernel (power-of-two scales packed as UE8M0, four K-blocks
# per word along K_total). Offsets that are not multiples of 512 start a group inside a word; an
# empty group must store zeros although the tensor memory still holds the previous tile.

def _run_ue8m0(dg, a, b, off):
    M, K = a.A.shape
    N = b.B.shape[1]
    G = len(off) - 1
    A, B = dev(np.ascontiguousarray(a.A.T)), dev(np.ascontiguousarray(b.B[0].T))
    sA, sB = dev(dg_inputs.pack_ue8m0_a(a.sA)), dev(dg_inputs.pack_ue8m0_b(b.sB)[0])
    O = dev(np.asarray(off, np.int32))
    D = bf16_sentinel((G, M, N))
    D32 = f32_sentinel((G, M, N))
    dg.dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0(A, sA, B, sB, O, D)
    dg.dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0_f32(A, sA, B, sB, O, D32)
    torch.cuda.synchronize()
    return D, D32


@pytest.mark.parametrize("M,N,off", [(192, 272, [0, 256, 256, 640, 1024]), (128, 128, [0, 128]),
                                     (64, 528, [0, 512, 1024, 1024]), (320, 256, [0, 0, 384, 1152]),
                                     (256, 384, [0, 128, 128, 896, 1280, 1408])])
def test_k_grouped_ue8m0_full_parity(dg, M, N, off):
    K = off[-1]
    a = dg_inputs.make_a(M, K, seed=M + 2 * N, ue8m0=True)
    b = dg_inputs.make_b(1, N, K, seed=M + 2 * N, ue8m0=True)
    D, D32 = _run_ue8m0(dg, a, b, off)
    ref = oracle.k_grouped(a.A, a.sA, b.B[0], b.sB[0], np.array(off, np.int32))
    db = bits16(D).cpu()
    assert torch.equal(db, rne_bf16_bits(D32))
    for g in range(len(off) - 1):
        if off[g] == off[g + 1]:
            assert torch.all(D32[g] == 0) and torch.all(db[g] == 0), f"empty group {g} is not zero"
    nz = [g for g in range(len(off) - 1) if off[g] != off[g + 1]]
    assert_accurate(D32.cpu().numpy()[nz], db.numpy()[nz], ref[nz], f"k-grouped/ue8m0 {M}x{N} {off}")


def test_k_grouped_ue8m0_large_sampled(dg):
    M, N = 2048, 7168
    off = [0, 1024, 1024, 3072, 3584]
    K = off[-1]
    a = dg_inputs.make_a(M, K, seed=5, ue8m0=True)
    b = dg_inputs.make_b(1, N, K, seed=5, ue8m0=True)
    D, D32 = _run_ue8m0(dg, a, b, off)
    assert torch.equal(bits16(D).cpu(), rne_bf16_bits(D32))
    assert torch.all(D32[1] == 0)
    rng = np.random.default_rng(4)
    for g in (0, 2, 3):
        k0, k1 = off[g], off[g + 1]
        ms, ns = rng.integers(0, M, 600), rng.integers(0, N, 600)
        kb = slice(k0 // 128, k1 // 128)
        ref = oracle.gemm_nt_sampled(np.ascontiguousarray(a.A[:, k0:k1]), np.ascontiguousarray(a.sA[kb]),
                                     np.ascontiguousarray(b.B[0][:, k0:k1]), np.ascontiguousarray(b.sB[0][:, kb]),
                                     ms, ns)
        assert_accurate(D32[g].cpu().numpy()[ms, ns], bits16(D[g]).cpu().numpy()[ms, ns], ref,
                        f"k-grouped/ue8m0 g={g}")
