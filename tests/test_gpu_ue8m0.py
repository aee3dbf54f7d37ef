"""GPU parity of the packed-UE8M0 calls (block-scaled tensor-core kernel) against the CPU oracle.

The scales are powers of two (the smallest 2^p >= amax/448) packed four K-groups to an int32
word. The oracle decodes exactly the words the GPU receives (``oracle.unpack_ue8m0_*``) and runs
its FP64 two-level GEMM; the accuracy bar is that of the FP32-scale calls (tests/_dg_testlib.py).
Because the tensor core applies these scales inside the MMA, a scale read from the wrong row,
block or byte is a gross error: the "wide scales" cases give every row, B block and K-group its
own exponent so that any such mix-up fails the bar.
"""
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


def _nkb(K):
    return (K + 127) // 128


def _packed(a, b):
    """Packed words (what the GPU gets) and the oracle's FP32 scales decoded from those words."""
    K = a.A.shape[-1]
    pa, pb = dg_inputs.pack_ue8m0_a(a.sA), dg_inputs.pack_ue8m0_b(b.sB)
    return pa, pb, oracle.unpack_ue8m0_a(pa, _nkb(K)), oracle.unpack_ue8m0_b(pb, _nkb(K))


def _dense_inputs(M, N, K, seed=0, dist=dg_inputs.NORMAL, outliers=0.0):
    a = dg_inputs.make_a(M, K, seed=seed, dist=dist, outlier_frac=outliers, ue8m0=True)
    b = dg_inputs.make_b(1, N, K, seed=seed, dist=dist, ue8m0=True)
    return a, b


def _wide_scale_inputs(M, N, K, seed):
    """N(0,1) values times 2^(row term + K-group term) for A and 2^(block term + K-group term) for
    B, so that neighbouring rows, B blocks and K-groups all get different scale exponents."""
    nkb = _nkb(K)
    kb = np.arange(K) // 128
    xa = dg_inputs.draw(seed, 0, M * K).reshape(M, K)
    xa *= np.exp2(((np.arange(M) * 7) % 13 - 6)[:, None] + ((kb * 5) % 11 - 5)[None, :]).astype(np.float32)
    xb = dg_inputs.draw(seed, 1, N * K).reshape(N, K)
    nb = np.arange(N) // 128
    xb *= np.exp2(((nb * 3) % 5 - 2)[:, None] + ((kb * 3) % 7 - 3)[None, :]).astype(np.float32)
    a = dg_inputs.quantize_a(xa, ue8m0=True)
    b = dg_inputs.quantize_b(xb, ue8m0=True)
    assert len(np.unique(a.sA[:min(nkb, 4), :M])) > 3
    return a, b


def _run_dense(dg, pa, a, b, pb):
    M, K = a.A.shape
    N = b.B.shape[1]
    A, sA, B, sB = dev(a.A), dev(pa), dev(b.B[0]), dev(pb[0])
    D = bf16_sentinel((M, N))
    D32 = f32_sentinel((M, N))
    dg.dg_fp8_gemm_nt_ue8m0(A, sA, B, sB, D)
    dg.dg_fp8_gemm_nt_ue8m0_f32(A, sA, B, sB, D32)
    torch.cuda.synchronize()
    return D, D32


def _check_full(dg, a, b, what):
    pa, pb, sA, sB = _packed(a, b)
    D, D32 = _run_dense(dg, pa, a, b, pb)
    ref64, _ = oracle.gemm_nt(a.A, sA, b.B[0], sB[0], want_bf16=False)
    dbits = bits16(D).cpu()
    assert torch.equal(dbits, rne_bf16_bits(D32)), f"{what}: BF16 output is not RNE of the FP32 accumulator"
    assert_accurate(D32.cpu().numpy(), dbits.numpy(), ref64, what)


# ----------------------------------------------------------------------------------------------
# Dense, whole-output parity

DENSE_SMALL = [
    (128, 512, 1024),
    (1, 16, 128), (63, 48, 256), (65, 112, 400), (200, 136, 1024), (129, 576, 512),
    (300, 264, 768), (64, 2112, 1024), (512, 2112, 1024), (1024, 4096, 512), (257, 520, 2048),
    (130, 304, 1680),
]


@pytest.mark.parametrize("M,N,K", DENSE_SMALL)
def test_ue8m0_dense_full_parity(dg, M, N, K):
    a, b = _dense_inputs(M, N, K, seed=M + N + K)
    _check_full(dg, a, b, f"ue8m0 dense {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(160, 392, 1152), (33, 136, 400), (256, 512, 2560), (64, 2112, 7168)])
def test_ue8m0_wide_scales_full_parity(dg, M, N, K):
    a, b = _wide_scale_inputs(M, N, K, seed=M * 3 + K)
    _check_full(dg, a, b, f"ue8m0 wide scales {M}x{N}x{K}")


def test_ue8m0_student_t_outliers_full_parity(dg):
    a, b = _dense_inputs(256, 576, 4096, seed=5, dist=dg_inputs.STUDENT_T3, outliers=0.01)
    _check_full(dg, a, b, "ue8m0 student-t outliers")


def test_ue8m0_dense_is_deterministic(dg):
    a, b = _dense_inputs(64, 2112, 7168, seed=3)       # few tiles: split-K path
    pa, pb, _, _ = _packed(a, b)
    assert dg.dg_query_config_ue8m0(0, 64, 2112, 7168)["splits"] > 1
    D1, D32a = _run_dense(dg, pa, a, b, pb)
    D2, D32b = _run_dense(dg, pa, a, b, pb)
    assert torch.equal(bits16(D1), bits16(D2))
    assert torch.equal(D32a.view(torch.int32), D32b.view(torch.int32))


# ----------------------------------------------------------------------------------------------
# Dense, full-size sweep and long-K stress (sampled parity)

SWEEP = [(M, N, K) for M in (64, 128, 4096)
         for (N, K) in ((2112, 7168), (24576, 1536), (32768, 512), (7168, 16384), (4096, 7168), (7168, 2048))]


@pytest.mark.parametrize("M,N,K", SWEEP)
def test_ue8m0_dense_sweep_sampled(dg, M, N, K):
    a, b = _dense_inputs(M, N, K, seed=0)
    pa, pb, sA, sB = _packed(a, b)
    D, D32 = _run_dense(dg, pa, a, b, pb)
    assert torch.equal(bits16(D).cpu(), rne_bf16_bits(D32))
    assert bool(torch.isfinite(D32).all())
    ms, ns = boundary_samples(M, N, 1500, seed=M ^ N ^ K, block_cols=256)
    ref = oracle.gemm_nt_sampled(a.A, sA, b.B[0], sB[0], ms, ns)
    assert_accurate(D32.cpu().numpy()[ms, ns], bits16(D).cpu().numpy()[ms, ns], ref, f"ue8m0 sweep {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(4096, 2112, 7168), (4096, 576, 7168), (4096, 7168, 32768)])
def test_ue8m0_accuracy_stress_sampled(dg, M, N, K):
    a, b = _dense_inputs(M, N, K, seed=0, dist=dg_inputs.STUDENT_T3, outliers=0.01)
    pa, pb, sA, sB = _packed(a, b)
    D, D32 = _run_dense(dg, pa, a, b, pb)
    assert torch.equal(bits16(D).cpu(), rne_bf16_bits(D32))
    ms, ns = boundary_samples(M, N, 1500, seed=7, block_cols=256)
    ref = oracle.gemm_nt_sampled(a.A, sA, b.B[0], sB[0], ms, ns)
    assert_accurate(D32.cpu().numpy()[ms, ns], bits16(D).cpu().numpy()[ms, ns], ref, f"ue8m0 stress {M}x{N}x{K}")


# ----------------------------------------------------------------------------------------------
# Contiguous grouped


def _run_contig(dg, a, pa, b, pb, m_idx):
    M = a.A.shape[0]
    G, N, _ = b.B.shape
    A, sA, B, sB, I = dev(a.A), dev(pa), dev(b.B), dev(pb), dev(m_idx)
    D = bf16_sentinel((M, N))
    D32 = f32_sentinel((M, N))
    dg.dg_fp8_grouped_contiguous_ue8m0(A, sA, B, sB, I, D)
    dg.dg_fp8_grouped_contiguous_ue8m0_f32(A, sA, B, sB, I, D32)
    torch.cuda.synchronize()
    return D, D32


@pytest.mark.parametrize("rows,N,K", [([100, 0, 200, 128, 1], 136, 256), ([300, 129, 5], 264, 400),
                                      ([128, 128], 512, 1024), ([1, 2, 3, 4, 5, 6, 7, 8], 64, 128)])
def test_ue8m0_contiguous_full_parity(dg, rows, N, K):
    m_idx = dg_inputs.contiguous_m_indices(rows, pad_to=128)
    M, G = len(m_idx), len(rows)
    a = dg_inputs.make_a(M, K, seed=21, ue8m0=True)
    b = dg_inputs.make_b(G, N, K, seed=21, ue8m0=True)
    pa, pb, sA, sB = _packed(a, b)
    D, D32 = _run_contig(dg, a, pa, b, pb, m_idx)
    ref64, _, bad = oracle.grouped_contiguous(a.A, sA, b.B, sB, m_idx)
    assert bad == 0
    valid = m_idx >= 0
    dbits = bits16(D).cpu()
    assert torch.all(dbits[~torch.from_numpy(valid)] == -1), "padding rows were written"
    assert torch.all(torch.isnan(D32.cpu()[~torch.from_numpy(valid)])), "padding rows were written (FP32)"
    assert torch.equal(dbits[valid], rne_bf16_bits(D32)[valid])
    assert_accurate(D32.cpu().numpy()[valid], dbits.numpy()[valid], ref64[valid], f"ue8m0 contiguous {rows}")


@pytest.mark.parametrize("G,N,K", [(4, 4096, 7168), (4, 7168, 2048), (8, 4096, 7168), (8, 7168, 2048)])
def test_ue8m0_contiguous_moe_sampled(dg, G, N, K):
    rows_per = 8192
    m_idx = np.repeat(np.arange(G, dtype=np.int32), rows_per)
    a = dg_inputs.make_a(G * rows_per, K, seed=0, ue8m0=True)
    b = dg_inputs.make_b(G, N, K, seed=0, ue8m0=True)
    pa, pb, sA, sB = _packed(a, b)
    D, D32 = _run_contig(dg, a, pa, b, pb, m_idx)
    assert torch.equal(bits16(D).cpu(), rne_bf16_bits(D32))
    # group boundaries and edges, plus every 128 x 256 output tile
    ms, ns = boundary_samples(G * rows_per, N, 2000, seed=G * N, block_rows=rows_per, block_cols=256, per_tile=0)
    mt, nt = boundary_samples(G * rows_per, N, 0, seed=G * N + 1, block_rows=128, block_cols=256)
    ms, ns = np.concatenate([ms, mt]), np.concatenate([ns, nt])
    ref = oracle.contiguous_sampled(a.A, sA, b.B, sB, m_idx, ms, ns)
    assert_accurate(D32.cpu().numpy()[ms, ns], bits16(D).cpu().numpy()[ms, ns], ref,
                    f"ue8m0 contiguous G={G} {N}x{K}")


# ----------------------------------------------------------------------------------------------
# Masked grouped


def _run_masked(dg, a, pa, b, pb, masked_m):
    G, M_max, _ = a.A.shape
    N = b.B.shape[1]
    A, sA, B, sB, MM = dev(a.A), dev(pa), dev(b.B), dev(pb), dev(masked_m)
    D = bf16_sentinel((G, M_max, N))
    D32 = f32_sentinel((G, M_max, N))
    dg.dg_fp8_grouped_masked_ue8m0(A, sA, B, sB, MM, D)
    dg.dg_fp8_grouped_masked_ue8m0_f32(A, sA, B, sB, MM, D32)
    torch.cuda.synchronize()
    return D, D32


def _valid_mask(masked_m, M_max):
    return np.arange(M_max)[None, :] < np.clip(masked_m, 0, M_max)[:, None]


@pytest.mark.parametrize("N,K", [(112, 384), (264, 256), (512, 1024)])
def test_ue8m0_masked_full_parity(dg, N, K):
    masked_m = np.array([0, 1, 127, 128, 129, 256], np.int32)
    G, M_max = len(masked_m), 256
    a = dg_inputs.make_masked_a(G, M_max, K, seed=31, ue8m0=True)
    b = dg_inputs.make_b(G, N, K, seed=31, ue8m0=True)
    pa, pb, sA, sB = _packed(a, b)
    D, D32 = _run_masked(dg, a, pa, b, pb, masked_m)
    ref64, _, bad = oracle.grouped_masked(a.A, sA, b.B, sB, masked_m)
    assert bad == 0
    valid = torch.from_numpy(_valid_mask(masked_m, M_max))
    dbits = bits16(D).cpu()
    assert torch.all(dbits[~valid] == -1), "rows past masked_m were written"
    assert torch.all(torch.isnan(D32.cpu()[~valid]))
    assert torch.equal(dbits[valid], rne_bf16_bits(D32)[valid])
    v = valid.numpy()
    assert_accurate(D32.cpu().numpy()[v], dbits.numpy()[v], ref64[v], f"ue8m0 masked {N}x{K}")


@pytest.mark.parametrize("N,K", [(4096, 7168), (7168, 2048)])
def test_ue8m0_masked_decode_sampled(dg, N, K):
    G, M_max = 16, 256
    masked_m = dg_inputs.make_masked_m(G, M_max, seed=0)
    a = dg_inputs.make_masked_a(G, M_max, K, seed=0, ue8m0=True)
    b = dg_inputs.make_b(G, N, K, seed=0, ue8m0=True)
    pa, pb, sA, sB = _packed(a, b)
    D, D32 = _run_masked(dg, a, pa, b, pb, masked_m)
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
    ref = oracle.masked_sampled(a.A, sA, b.B, sB, gs, ms, ns)
    assert_accurate(D32.cpu().numpy()[gs, ms, ns], dbits.numpy()[gs, ms, ns], ref, f"ue8m0 masked decode {N}x{K}")


# ----------------------------------------------------------------------------------------------
# Device-detected errors and host validation


def test_ue8m0_contiguous_bad_index_sets_status(dg):
    N, K, G = 64, 128, 2
    m_idx = np.full(256, -1, np.int32)
    m_idx[:10] = 0
    m_idx[128:140] = 1
    m_idx[140] = 7              # out of range
    a = dg_inputs.make_a(256, K, seed=2, ue8m0=True)
    b = dg_inputs.make_b(G, N, K, seed=2, ue8m0=True)
    pa, pb, _, _ = _packed(a, b)
    assert dg.dg_get_device_status() == 0
    D, _ = _run_contig(dg, a, pa, b, pb, m_idx)
    assert dg.dg_get_device_status() & dg.DG_DEV_BAD_GROUP_INDEX
    dbits = bits16(D).cpu()
    assert torch.all(dbits[140] == -1) and torch.all(dbits[10:128] == -1)
    assert not torch.any(dbits[:10] == -1) and not torch.any(dbits[128:140] == -1)


def test_ue8m0_host_validation(dg):
    a, b = _dense_inputs(16, 64, 128)
    pa, pb, _, _ = _packed(a, b)
    A, sA, B, sB = dev(a.A), dev(pa), dev(b.B[0]), dev(pb[0])
    D = bf16_sentinel((16, 64))
    with pytest.raises(TypeError):
        dg.dg_fp8_gemm_nt_ue8m0(A, dev(a.sA), B, sB, D)           # FP32 scales to a UE8M0 call
    with pytest.raises(dg.DGError) as e:
        dg.dg_fp8_gemm_nt_ue8m0(A[:, :120].contiguous(), sA, B[:, :120].contiguous(), sB, D)   # K = 120
    assert e.value.status == dg.DG_ERR_ALIGNMENT
    dg.dg_fp8_gemm_nt_ue8m0(A, sA, B, sB, D)
    torch.cuda.synchronize()
    assert not torch.any(bits16(D) == -1)
