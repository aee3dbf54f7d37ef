"""GPU parity: libdg (through its C ABI) against the CPU oracle on the same seeded inputs.

Small and medium shapes are compared element by element over the whole output; the full-size
workloads (dense sweep, contiguous and masked MoE shapes, long-K outlier stress) on sampled
elements — random positions plus tile boundaries and tails — computed one by one by the oracle,
and on properties that hold at any size (BF16 == RNE(FP32) everywhere, finite outputs, rows
outside the valid region untouched). See tests/_dg_testlib.py for the accuracy bar.
"""
import numpy as np
import pytest
import torch

import dg_inputs
import oracle
from _dg_testlib import (assert_accurate, bf16_sentinel, bits16, boundary_samples, dev, f32_sentinel, metrics,
                         rne_bf16_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import moe_grouped_gemm_e4m3_gb300 as m
    m.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield m
    assert m.dg_get_device_status() == 0


def _dense_inputs(M, N, K, seed=0, dist=dg_inputs.NORMAL, outliers=0.0):
    a = dg_inputs.make_a(M, K, seed=seed, dist=dist, outlier_frac=outliers)
    b = dg_inputs.make_b(1, N, K, seed=seed, dist=dist)
    return a, b


def _run_dense(dg, a, b):
    M, K = a.A.shape
    N = b.B.shape[1]
    A, sA, B, sB = dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0])
    D = bf16_sentinel((M, N))
    D32 = f32_sentinel((M, N))
    dg.dg_fp8_gemm_nt(A, sA, B, sB, D)
    dg.dg_fp8_gemm_nt_f32(A, sA, B, sB, D32)
    torch.cuda.synchronize()
    return D, D32


# ----------------------------------------------------------------------------------------------
# Dense, whole-output parity


DENSE_SMALL = [
    (128, 512, 1024),     # the small dense case: M=128, N=512, K=1024
    (1, 16, 128), (63, 48, 256), (65, 112, 400), (200, 136, 1024), (129, 576, 512),
    (300, 264, 768), (64, 2112, 1024), (512, 2112, 1024), (1024, 4096, 512), (257, 520, 2048),
]


@pytest.mark.parametrize("M,N,K", DENSE_SMALL)
def test_dense_full_parity(dg, M, N, K):
    a, b = _dense_inputs(M, N, K, seed=M + N + K)
    D, D32 = _run_dense(dg, a, b)
    ref64, _ = oracle.gemm_nt(a.A, a.sA, b.B[0], b.sB[0], want_bf16=False)
    dbits = bits16(D).cpu()
    assert torch.equal(dbits, rne_bf16_bits(D32)), "BF16 output is not RNE of the FP32 accumulator"
    assert_accurate(D32.cpu().numpy(), dbits.numpy(), ref64, f"dense {M}x{N}x{K}")


def test_dense_student_t_outliers_full_parity(dg):
    a, b = _dense_inputs(256, 576, 4096, seed=5, dist=dg_inputs.STUDENT_T3, outliers=0.01)
    D, D32 = _run_dense(dg, a, b)
    ref64, _ = oracle.gemm_nt(a.A, a.sA, b.B[0], b.sB[0], want_bf16=False)
    dbits = bits16(D).cpu()
    assert torch.equal(dbits, rne_bf16_bits(D32))
    assert_accurate(D32.cpu().numpy(), dbits.numpy(), ref64, "student-t outliers")


def test_dense_is_deterministic(dg):
    a, b = _dense_inputs(64, 2112, 7168, seed=3)       # few tiles: split-K path
    D1, D32a = _run_dense(dg, a, b)
    D2, D32b = _run_dense(dg, a, b)
    assert torch.equal(bits16(D1), bits16(D2))
    assert torch.equal(D32a.view(torch.int32), D32b.view(torch.int32))


# ----------------------------------------------------------------------------------------------
# Dense, full-size sweep (sampled parity)

SWEEP = [(M, N, K) for M in (64, 128, 4096)
         for (N, K) in ((2112, 7168), (24576, 1536), (32768, 512), (7168, 16384), (4096, 7168), (7168, 2048))]


@pytest.mark.parametrize("M,N,K", SWEEP)
def test_dense_sweep_sampled(dg, M, N, K):
    a, b = _dense_inputs(M, N, K, seed=0)
    D, D32 = _run_dense(dg, a, b)
    assert torch.equal(bits16(D).cpu(), rne_bf16_bits(D32))
    assert bool(torch.isfinite(D32).all())
    ms, ns = boundary_samples(M, N, 1500, seed=M ^ N ^ K, block_cols=256)
    ref = oracle.gemm_nt_sampled(a.A, a.sA, b.B[0], b.sB[0], ms, ns)
    d32 = D32.cpu().numpy()[ms, ns]
    dbf = bits16(D).cpu().numpy()[ms, ns]
    assert_accurate(d32, dbf, ref, f"sweep {M}x{N}x{K}")


STRESS = [(4096, 2112, 7168), (4096, 576, 7168), (4096, 7168, 32768)]


@pytest.mark.parametrize("M,N,K", STRESS)
def test_dense_accuracy_stress_sampled(dg, M, N, K):
    a, b = _dense_inputs(M, N, K, seed=0, dist=dg_inputs.STUDENT_T3, outliers=0.01)
    D, D32 = _run_dense(dg, a, b)
    assert torch.equal(bits16(D).cpu(), rne_bf16_bits(D32))
    ms, ns = boundary_samples(M, N, 1500, seed=7, block_cols=256)
    ref = oracle.gemm_nt_sampled(a.A, a.sA, b.B[0], b.sB[0], ms, ns)
    assert_accurate(D32.cpu().numpy()[ms, ns], bits16(D).cpu().numpy()[ms, ns], ref, f"stress {M}x{N}x{K}")


# ----------------------------------------------------------------------------------------------
# Contiguous grouped


def _run_contig(dg, a, b, m_idx):
    M = a.A.shape[0]
    G, N, _ = b.B.shape
    A, sA, B, sB, I = dev(a.A), dev(a.sA), dev(b.B), dev(b.sB), dev(m_idx)
    D = bf16_sentinel((M, N))
    D32 = f32_sentinel((M, N))
    dg.dg_fp8_grouped_contiguous(A, sA, B, sB, I, D)
    dg.dg_fp8_grouped_contiguous_f32(A, sA, B, sB, I, D32)
    torch.cuda.synchronize()
    return D, D32


@pytest.mark.parametrize("rows,N,K", [([100, 0, 200, 128, 1], 136, 256), ([300, 129, 5], 264, 400),
                                      ([128, 128], 512, 1024), ([1, 2, 3, 4, 5, 6, 7, 8], 64, 128)])
def test_contiguous_full_parity(dg, rows, N, K):
    m_idx = dg_inputs.contiguous_m_indices(rows, pad_to=128)
    M, G = len(m_idx), len(rows)
    a = dg_inputs.make_a(M, K, seed=21)
    b = dg_inputs.make_b(G, N, K, seed=21)
    D, D32 = _run_contig(dg, a, b, m_idx)
    ref64, _, bad = oracle.grouped_contiguous(a.A, a.sA, b.B, b.sB, m_idx)
    assert bad == 0
    valid = m_idx >= 0
    dbits = bits16(D).cpu()
    assert torch.all(dbits[~torch.from_numpy(valid)] == -1), "padding rows were written"
    assert torch.all(torch.isnan(D32.cpu()[~torch.from_numpy(valid)])), "padding rows were written (FP32)"
    assert torch.equal(dbits[valid], rne_bf16_bits(D32)[valid])
    assert_accurate(D32.cpu().numpy()[valid], dbits.numpy()[valid], ref64[valid], f"contiguous {rows}")


def test_contiguous_equals_dense_per_group_bitwise(dg):
    # Same tile configuration (no split-K) => the same accumulation order => identical bits.
    rows, N, K = [256, 384, 128], 512, 1024
    m_idx = dg_inputs.contiguous_m_indices(rows)
    a = dg_inputs.make_a(len(m_idx), K, seed=4)
    b = dg_inputs.make_b(len(rows), N, K, seed=4)
    dg.dg_set_num_sms(2)
    try:
        _, D32 = _run_contig(dg, a, b, m_idx)
        r0 = 0
        for g, r in enumerate(rows):
            sl = slice(r0, r0 + r)
            sA = np.zeros((a.sA.shape[0], dg_inputs.align4(r)), np.float32)
            sA[:, :r] = a.sA[:, sl]
            ag = dg_inputs.OperandA(np.ascontiguousarray(a.A[sl]), sA)
            bg = dg_inputs.OperandB(b.B[g:g + 1], b.sB[g:g + 1])
            assert dg.dg_query_config(0, r, N, K)["splits"] == 1
            _, Dg32 = _run_dense(dg, ag, bg)
            assert torch.equal(D32[sl].view(torch.int32), Dg32.view(torch.int32)), f"group {g}"
            r0 += r
    finally:
        dg.dg_set_num_sms(0)


@pytest.mark.parametrize("G,N,K", [(4, 4096, 7168), (4, 7168, 2048), (8, 4096, 7168), (8, 7168, 2048)])
def test_contiguous_moe_sampled(dg, G, N, K):
    rows_per = 8192
    m_idx = np.repeat(np.arange(G, dtype=np.int32), rows_per)
    a = dg_inputs.make_a(G * rows_per, K, seed=0)
    b = dg_inputs.make_b(G, N, K, seed=0)
    D, D32 = _run_contig(dg, a, b, m_idx)
    assert torch.equal(bits16(D).cpu(), rne_bf16_bits(D32))
    # group boundaries and edges, plus every 128 x 256 output tile
    ms, ns = boundary_samples(G * rows_per, N, 2000, seed=G * N, block_rows=rows_per, block_cols=256, per_tile=0)
    mt, nt = boundary_samples(G * rows_per, N, 0, seed=G * N + 1, block_rows=128, block_cols=256)
    ms, ns = np.concatenate([ms, mt]), np.concatenate([ns, nt])
    ref = oracle.contiguous_sampled(a.A, a.sA, b.B, b.sB, m_idx, ms, ns)
    assert_accurate(D32.cpu().numpy()[ms, ns], bits16(D).cpu().numpy()[ms, ns], ref, f"contiguous G={G} {N}x{K}")


# ----------------------------------------------------------------------------------------------
# Masked grouped


def _run_masked(dg, a, b, masked_m):
    G, M_max, _ = a.A.shape
    N = b.B.shape[1]
    A, sA, B, sB, MM = dev(a.A), dev(a.sA), dev(b.B), dev(b.sB), dev(masked_m)
    D = bf16_sentinel((G, M_max, N))
    D32 = f32_sentinel((G, M_max, N))
    dg.dg_fp8_grouped_masked(A, sA, B, sB, MM, D)
    dg.dg_fp8_grouped_masked_f32(A, sA, B, sB, MM, D32)
    torch.cuda.synchronize()
    return D, D32


def _valid_mask(masked_m, M_max):
    return np.arange(M_max)[None, :] < np.clip(masked_m, 0, M_max)[:, None]


@pytest.mark.parametrize("N,K", [(112, 384), (264, 256), (512, 1024)])
def test_masked_full_parity(dg, N, K):
    masked_m = np.array([0, 1, 127, 128, 129, 256], np.int32)
    G, M_max = len(masked_m), 256
    a = dg_inputs.make_masked_a(G, M_max, K, seed=31)
    b = dg_inputs.make_b(G, N, K, seed=31)
    D, D32 = _run_masked(dg, a, b, masked_m)
    ref64, _, bad = oracle.grouped_masked(a.A, a.sA, b.B, b.sB, masked_m)
    assert bad == 0
    valid = torch.from_numpy(_valid_mask(masked_m, M_max))
    dbits = bits16(D).cpu()
    assert torch.all(dbits[~valid] == -1), "rows past masked_m were written"
    assert torch.all(torch.isnan(D32.cpu()[~valid]))
    assert torch.equal(dbits[valid], rne_bf16_bits(D32)[valid])
    v = valid.numpy()
    assert_accurate(D32.cpu().numpy()[v], dbits.numpy()[v], ref64[v], f"masked {N}x{K}")


@pytest.mark.parametrize("N,K", [(4096, 7168), (7168, 2048)])
def test_masked_decode_sampled(dg, N, K):
    G, M_max = 16, 256
    masked_m = dg_inputs.make_masked_m(G, M_max, seed=0)
    assert masked_m[0] == 0 and masked_m[-1] == M_max
    a = dg_inputs.make_masked_a(G, M_max, K, seed=0)
    b = dg_inputs.make_b(G, N, K, seed=0)
    D, D32 = _run_masked(dg, a, b, masked_m)
    valid = _valid_mask(masked_m, M_max)
    dbits = bits16(D).cpu()
    vt = torch.from_numpy(valid)
    assert torch.all(dbits[~vt] == -1), "rows past masked_m were written"
    assert torch.equal(dbits[vt], rne_bf16_bits(D32)[vt])
    rng = np.random.default_rng(N)
    gs, ms = np.nonzero(valid)
    pick = rng.choice(len(gs), size=3000, replace=len(gs) < 3000)
    gs, ms = gs[pick], ms[pick]
    ns = rng.integers(0, N, len(gs))
    ref = oracle.masked_sampled(a.A, a.sA, b.B, b.sB, gs, ms, ns)
    d32 = D32.cpu().numpy()[gs, ms, ns]
    assert_accurate(d32, dbits.numpy()[gs, ms, ns], ref, f"masked decode {N}x{K}")


# ----------------------------------------------------------------------------------------------
# Device-detected errors (no trap: status word, rows untouched)


def test_contiguous_bad_index_sets_status(dg):
    N, K, G = 64, 128, 2
    m_idx = np.full(256, -1, np.int32)
    m_idx[:10] = 0
    m_idx[128:140] = 1
    m_idx[140] = 7              # out of range
    a = dg_inputs.make_a(256, K, seed=2)
    b = dg_inputs.make_b(G, N, K, seed=2)
    assert dg.dg_get_device_status() == 0
    D, _ = _run_contig(dg, a, b, m_idx)
    code = dg.dg_get_device_status()
    assert code & dg.DG_DEV_BAD_GROUP_INDEX
    dbits = bits16(D).cpu()
    assert torch.all(dbits[140] == -1) and torch.all(dbits[10:128] == -1)
    assert not torch.any(dbits[:10] == -1) and not torch.any(dbits[128:140] == -1)


def test_masked_out_of_range_count_is_clamped(dg):
    N, K, G, M_max = 64, 128, 2, 128
    masked_m = np.array([300, -4], np.int32)
    a = dg_inputs.make_masked_a(G, M_max, K, seed=3)
    b = dg_inputs.make_b(G, N, K, seed=3)
    D, D32 = _run_masked(dg, a, b, masked_m)
    code = dg.dg_get_device_status()
    assert code & dg.DG_DEV_BAD_MASKED_M
    ref64, _, bad = oracle.grouped_masked(a.A, a.sA, b.B, b.sB, masked_m)
    assert bad == 2
    dbits = bits16(D).cpu()
    assert torch.all(dbits[1] == -1)
    assert_accurate(D32.cpu().numpy()[0], dbits.numpy()[0], ref64[0], "clamped masked")


def test_host_validation_errors(dg):
    a, b = _dense_inputs(16, 64, 128)
    A, sA, B, sB = dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0])
    D = bf16_sentinel((16, 64))
    with pytest.raises(dg.DGError) as e:
        dg.dg_fp8_gemm_nt(A[:, :120].contiguous(), sA, B[:, :120].contiguous(), sB, D)   # K = 120
    assert e.value.status == dg.DG_ERR_ALIGNMENT
    with pytest.raises(dg.DGError) as e:
        dg.dg_fp8_gemm_nt(A, sA, B[:60].contiguous(), sB, D[:, :60].contiguous())   # N = 60
    assert e.value.status == dg.DG_ERR_ALIGNMENT
    # the valid call still works afterwards
    dg.dg_fp8_gemm_nt(A, sA, B, sB, D)
    torch.cuda.synchronize()
    assert not torch.any(bits16(D) == -1)
