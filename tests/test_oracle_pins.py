"""Pins of the CPU oracle against things other than itself (CPU only).

* E4M3 decode: the OCP table (golden file), torch's float8_e4m3fn conversion for all 256 codes,
  and format invariants (signed zeros, sign symmetry, strict monotonicity, NaN codes).
* BF16 rounding: hand-derived IEEE cases (golden file, including a double-rounding trap) and
  torch's float32 -> bfloat16 conversion for float32-representable inputs.
* GEMM: exact brute force with integer-valued E4M3 inputs and power-of-two scales, computed with
  Python integers and fractions; the plain dequantise-then-matmul definition computed by numpy on
  random inputs (pins the scale indexing); identity B; scale linearity; a single K-block.
* Grouped forms: contiguous and masked equal the dense oracle per group, bit for bit, and rows
  outside the valid region stay untouched.
* Accumulating form D = C + A·Bᵀ: the hand-worked example with a C added, A = 0 gives C exactly,
  C = 0 gives the plain GEMM bit for bit.
* K-grouped GEMM: each group equals the dense oracle on its K slice, an empty group gives zeros, one
  group over all of K equals the dense GEMM bit for bit, and the groups sum to the dense GEMM.
* Masked GEMM fused with SwiGLU: silu against scipy's logistic function (x·expit(x)) and its limits;
  the fused output against silu(gate)·up formed from the plain masked oracle's two halves.
* Packed UE8M0 scales: the OCP MX E8M0 table (golden file) and torch's float8_e8m0fnu conversion
  for all 256 codes; a GEMM with packed scales worked by hand (golden file, pins the byte order
  and both packed layouts); the unpacker against the input generator's independent packer; the
  dequantise-then-matmul definition with power-of-two scales.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import dg_inputs
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_e4m3_table() -> np.ndarray:
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _e4m3_bytes_of_exact(values: np.ndarray) -> np.ndarray:
    """E4M3 bytes of values that E4M3 represents exactly, via torch's conversion."""
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32))
    b = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    back = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    assert np.array_equal(back, values.astype(np.float32)), "test values must be exact in E4M3"
    return b


# ----------------------------------------------------------------------------------------------
# E4M3 decode


def test_e4m3_golden_table():
    with open(os.path.join(GOLDEN, "e4m3_ocp_values.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 16
    for code_s, val_s in rows:
        code = int(code_s, 16)
        got = float(oracle.e4m3_decode(np.array([code], np.uint8))[0])
        if val_s == "nan":
            assert math.isnan(got), hex(code)
        else:
            want = float(val_s)
            assert got == want and math.copysign(1, got) == math.copysign(1, want), hex(code)


def test_e4m3_all_codes_vs_torch():
    ours = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = _torch_e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_e4m3_invariants():
    v = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert v[0x00] == 0 and not np.signbit(v[0x00])
    assert v[0x80] == 0 and np.signbit(v[0x80])
    assert v[0x7E] == 448.0 and v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    pos = v[0x00:0x7F]
    assert np.all(np.diff(pos) > 0)                       # strictly increasing over 0x00..0x7E
    assert np.array_equal(v[0x80:0xFF], -pos)             # sign symmetry
    # every finite value has at most 4 significant bits (1 implicit + 3 stored)
    for x in pos[1:]:
        m, e = math.frexp(x)
        assert (m * 16) == int(m * 16)


# ----------------------------------------------------------------------------------------------
# BF16 rounding


def test_bf16_golden_cases():
    with open(os.path.join(GOLDEN, "bf16_rne_cases.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    xs = np.array([float.fromhex(a) for a, _ in rows], np.float64)
    want = np.array([int(b, 16) for _, b in rows], np.uint16)
    got = oracle.bf16_from_f64(xs)
    assert np.array_equal(got, want), [(r, hex(g)) for r, g in zip(rows, got) if int(r[1], 16) != g]


def test_bf16_vs_torch_on_float32_inputs():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(5000) * 1e-39).astype(np.float32),          # FP32 subnormals
        (rng.standard_normal(5000) * 1e30).astype(np.float32),
        # exact ties: low 16 bits 0x8000, both parities of the kept part
        (rng.integers(0x3F000000, 0x47000000, 4000, dtype=np.uint32) & ~np.uint32(0xFFFF)
         | np.uint32(0x8000)).view(np.float32),
    ]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_from_f64(x.astype(np.float64))
    assert np.array_equal(got, want)


# ----------------------------------------------------------------------------------------------
# GEMM: exact brute force


def _rne_bf16_exact(fr: Fraction) -> int:
    """BF16 bits of an exact rational, by integer arithmetic (normal range only)."""
    if fr == 0:
        return 0
    sign = 0x8000 if fr < 0 else 0
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = a / Fraction(2) ** (e - 7)               # in [128, 256)
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    if fl == 256:
        fl, e = 128, e + 1
    assert -126 <= e <= 127
    return sign | ((e + 127) << 7) | (fl - 128)


def _pow2_problem(M, N, K, seed, G=1):
    rng = np.random.default_rng(seed)
    nkb, nnb = (K + 127) // 128, (N + 127) // 128
    a_int = rng.integers(-16, 17, size=(M, K))
    b_int = rng.integers(-16, 17, size=(G, N, K))
    ea = rng.integers(-6, 7, size=(nkb, M))
    eb = rng.integers(-6, 7, size=(G, nnb, nkb))
    ldsa = dg_inputs.align4(M)
    sA = np.zeros((nkb, ldsa), np.float32)
    sA[:, :M] = np.ldexp(1.0, ea)
    sB = np.ldexp(1.0, eb).astype(np.float32)
    A = _e4m3_bytes_of_exact(a_int.astype(np.float32))
    B = _e4m3_bytes_of_exact(b_int.astype(np.float32))
    return a_int, b_int, ea, eb, A, sA, B, sB


def _exact_dense(a_int, b_int, ea, eb, m, n, K):
    total = Fraction(0)
    for kb in range((K + 127) // 128):
        k0, k1 = kb * 128, min(K, kb * 128 + 128)
        dot = int(np.dot(a_int[m, k0:k1].astype(np.int64), b_int[n, k0:k1].astype(np.int64)))
        total += Fraction(dot) * Fraction(2) ** int(ea[kb, m] + eb[n // 128, kb])
    return total


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 128, 0), (3, 5, 256, 1), (8, 8, 384, 2),
                                        (7, 3, 200, 3), (5, 130, 256, 4), (2, 2, 16, 5)])
def test_gemm_bruteforce_integer_inputs(M, N, K, seed):
    a_int, b_int, ea, eb, A, sA, B, sB = _pow2_problem(M, N, K, seed)
    ref64, D = oracle.gemm_nt(A, sA, B[0], sB[0], threads=2)
    for m in range(M):
        for n in range(N):
            want = _exact_dense(a_int, b_int[0], ea, eb[0], m, n, K)
            assert Fraction(ref64[m, n]) == want, (m, n)
            assert int(D[m, n]) == _rne_bf16_exact(want), (m, n)


def test_gemm_worked_example_by_hand():
    # Two rows, two columns, K = 256 (two K-blocks). Row 0 of A is all 1.0, row 1 all 2.0;
    # row 0 of B is all 0.5, row 1 alternates +1/-1. sA = [[1, 0.5], [0.25, 8]] (kb-major, per row),
    # sB = [2, 4] (one N-block). By hand:
    #   D[0,0] = 1*2*(128*1*0.5) + 0.25*4*(128*1*0.5) = 128 + 64 = 192
    #   D[1,0] = 0.5*2*(128*2*0.5) + 8*4*(128*2*0.5) = 128 + 4096 = 4224
    #   D[:,1] = 0 (each K-block of B row 1 sums to zero against a constant row)
    A = np.array([[0x38] * 256, [0x40] * 256], np.uint8)
    B = np.array([[0x30] * 256, [0x38, 0xB8] * 128], np.uint8)
    sA = np.array([[1.0, 0.5, 0, 0], [0.25, 8.0, 0, 0]], np.float32)
    sB = np.array([[2.0, 4.0]], np.float32)
    ref64, D = oracle.gemm_nt(A, sA, B, sB, threads=1)
    assert ref64.tolist() == [[192.0, 0.0], [4224.0, 0.0]]
    assert D.tolist() == [[0x4340, 0x0000], [0x4584, 0x0000]]   # 192 = 1.5*2^7, 4224 = 1.03125*2^12


# ----------------------------------------------------------------------------------------------
# GEMM: the plain definition (dequantise, then FP64 matmul) computed independently by numpy


def _numpy_definition(A, sA, B, sB):
    table = _torch_e4m3_table()
    M, K = A.shape
    N = B.shape[0]
    sa = np.repeat(sA[:, :M].T.astype(np.float64), 128, axis=1)[:, :K]            # [M, K]
    sb = np.repeat(np.repeat(sB.astype(np.float64), 128, axis=0)[:N], 128, axis=1)[:, :K]  # [N, K]
    return (table[A] * sa) @ (table[B] * sb).T


@pytest.mark.parametrize("M,N,K,dist,outliers", [
    (33, 70, 300, dg_inputs.NORMAL, 0.0),
    (128, 200, 512, dg_inputs.NORMAL, 0.0),
    (17, 257, 1024, dg_inputs.STUDENT_T3, 0.01),
    (130, 48, 144, dg_inputs.STUDENT_T3, 0.05),
])
def test_gemm_matches_dequantised_definition(M, N, K, dist, outliers):
    a = dg_inputs.make_a(M, K, seed=11, dist=dist, outlier_frac=outliers)
    b = dg_inputs.make_b(1, N, K, seed=11, dist=dist)
    ref64, D = oracle.gemm_nt(a.A, a.sA, b.B[0], b.sB[0], threads=4)
    want = _numpy_definition(a.A, a.sA, b.B[0], b.sB[0])
    scale = np.abs(want).max()
    assert scale > 0
    assert np.abs(ref64 - want).max() <= 1e-13 * scale
    # a transposed or shifted scale index would move results by O(1) relative
    assert np.allclose(ref64, want, rtol=1e-12, atol=1e-13 * scale)


def test_identity_b():
    K = 256
    a = dg_inputs.make_a(20, K, seed=3)
    B = np.zeros((K, K), np.uint8)
    B[np.arange(K), np.arange(K)] = 0x38                    # 1.0
    sB = np.ones((2, 2), np.float32)
    ref64, D = oracle.gemm_nt(a.A, a.sA, B, sB, threads=2)
    table = _torch_e4m3_table()
    want = table[a.A] * np.repeat(a.sA[:, :20].T.astype(np.float64), 128, axis=1)
    assert np.array_equal(ref64, want)                    # dec(a)*sA is exact in FP64
    want_bits = np.array([_rne_bf16_exact(Fraction(float(v))) for v in want.ravel()], np.uint16)
    assert np.array_equal(D.ravel(), want_bits)


def test_single_k_block_is_exact_scaled_partial():
    a = dg_inputs.make_a(9, 128, seed=4)
    b = dg_inputs.make_b(1, 11, 128, seed=4)
    ref64, _ = oracle.gemm_nt(a.A, a.sA, b.B[0], b.sB[0], threads=1)
    table = _torch_e4m3_table()
    P = table[a.A] @ table[b.B[0]].T                         # exact: short products, 128 terms
    want = (a.sA[0, :9].astype(np.float64)[:, None] * float(b.sB[0, 0, 0])) * P
    assert np.array_equal(ref64, want)


def test_scale_linearity():
    M, N, K = 6, 9, 384
    a_int, b_int, ea, eb, A, sA, B, sB = _pow2_problem(M, N, K, seed=7)
    ref64, _ = oracle.gemm_nt(A, sA, B[0], sB[0], threads=1)
    kb = 1
    sA2 = sA.copy()
    sA2[kb, :] *= 2
    ref64_2, _ = oracle.gemm_nt(A, sA2, B[0], sB[0], threads=1)
    # contribution of K-block kb alone: the same problem restricted to those 128 columns
    sl = slice(kb * 128, kb * 128 + 128)
    contrib, _ = oracle.gemm_nt(np.ascontiguousarray(A[:, sl]), np.ascontiguousarray(sA[kb:kb + 1]),
                                np.ascontiguousarray(B[0][:, sl]), np.ascontiguousarray(sB[0][:, kb:kb + 1]),
                                threads=1)
    assert np.array_equal(ref64_2 - ref64, contrib)
    assert np.abs(contrib).max() > 0


# ----------------------------------------------------------------------------------------------
# Grouped forms


def test_contiguous_equals_per_group_dense_and_padding_untouched():
    G, N, K = 3, 136, 256
    rows = [100, 0, 200]
    m_idx = dg_inputs.contiguous_m_indices(rows, pad_to=128)
    M = len(m_idx)
    a = dg_inputs.make_a(M, K, seed=5)
    b = dg_inputs.make_b(G, N, K, seed=5)
    D0 = np.full((M, N), 0xFFFF, np.uint16)
    r0 = np.full((M, N), np.nan)
    ref64, D, bad = oracle.grouped_contiguous(a.A, a.sA, b.B, b.sB, m_idx, r0, D0, threads=4)
    assert bad == 0
    pad = m_idx < 0
    assert np.all(D[pad] == 0xFFFF) and np.all(np.isnan(ref64[pad]))
    for g in range(G):
        rr = np.nonzero(m_idx == g)[0]
        if len(rr) == 0:
            continue
        # the dense oracle on exactly those rows of A (with their scales)
        sA_g = np.zeros((a.sA.shape[0], dg_inputs.align4(len(rr))), np.float32)
        sA_g[:, :len(rr)] = a.sA[:, rr]
        rg, Dg = oracle.gemm_nt(a.A[rr], sA_g, b.B[g], b.sB[g], threads=2)
        assert np.array_equal(D[rr], Dg) and np.array_equal(ref64[rr], rg)


def test_contiguous_invalid_indices_untouched_and_counted():
    G, N, K = 2, 16, 128
    m_idx = np.array([0, 1, -1, 2, -2, 1], np.int32)
    a = dg_inputs.make_a(len(m_idx), K, seed=6)
    b = dg_inputs.make_b(G, N, K, seed=6)
    D0 = np.full((len(m_idx), N), 0xFFFF, np.uint16)
    _, D, bad = oracle.grouped_contiguous(a.A, a.sA, b.B, b.sB, m_idx, None, D0, threads=1)
    assert bad == 2
    assert np.all(D[[2, 3, 4]] == 0xFFFF)
    assert not np.any(D[[0, 1, 5]] == 0xFFFF)


def test_masked_equals_per_group_dense_and_tail_untouched():
    G, M_max, N, K = 4, 64, 40, 256
    masked_m = np.array([0, 64, 17, 33], np.int32)
    a = dg_inputs.make_masked_a(G, M_max, K, seed=8)
    b = dg_inputs.make_b(G, N, K, seed=8)
    D0 = np.full((G, M_max, N), 0xFFFF, np.uint16)
    ref64, D, bad = oracle.grouped_masked(a.A, a.sA, b.B, b.sB, masked_m, None, D0, threads=4)
    assert bad == 0
    for g in range(G):
        v = masked_m[g]
        assert np.all(D[g, v:] == 0xFFFF)
        rg, Dg = oracle.gemm_nt(a.A[g], a.sA[g], b.B[g], b.sB[g], threads=2)
        assert np.array_equal(D[g, :v], Dg[:v]) and np.array_equal(ref64[g, :v], rg[:v])


def test_masked_clamps_out_of_range_counts():
    G, M_max, N, K = 2, 8, 16, 128
    a = dg_inputs.make_masked_a(G, M_max, K, seed=9)
    b = dg_inputs.make_b(G, N, K, seed=9)
    D0 = np.full((G, M_max, N), 0xFFFF, np.uint16)
    _, D, bad = oracle.grouped_masked(a.A, a.sA, b.B, b.sB, np.array([-3, 99], np.int32), None, D0)
    assert bad == 2
    assert np.all(D[0] == 0xFFFF) and not np.any(D[1] == 0xFFFF)


def test_sampled_matches_full():
    M, N, K = 50, 300, 640
    a = dg_inputs.make_a(M, K, seed=10)
    b = dg_inputs.make_b(1, N, K, seed=10)
    ref64, _ = oracle.gemm_nt(a.A, a.sA, b.B[0], b.sB[0], threads=4)
    rng = np.random.default_rng(0)
    ms, ns = rng.integers(0, M, 200), rng.integers(0, N, 200)
    got = oracle.gemm_nt_sampled(a.A, a.sA, b.B[0], b.sB[0], ms, ns, threads=3)
    assert np.array_equal(got, ref64[ms, ns])


# ----------------------------------------------------------------------------------------------
# Packed UE8M0 scales


def test_ue8m0_golden_table():
    with open(os.path.join(GOLDEN, "ue8m0_values.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 10
    for code_s, val_s in rows:
        got = float(oracle.ue8m0_decode(np.array([int(code_s, 16)], np.uint8))[0])
        if val_s == "nan":
            assert math.isnan(got), code_s
        else:
            assert got == float(val_s), code_s


def test_ue8m0_all_codes_vs_torch():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this torch has no float8_e8m0fnu")
    ours = oracle.ue8m0_decode(np.arange(256, dtype=np.uint8))
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.isnan(ours[255]) and np.isnan(ref[255])
    assert np.array_equal(ours[:255], ref[:255])
    assert np.all(np.diff(ours[:255]) > 0) and np.all(ours[1:255] == 2 * ours[:254])


def _read_packed_example():
    vals = {}
    rows_a, rows_b = {}, {}
    with open(os.path.join(GOLDEN, "ue8m0_packed_example.txt")) as f:
        for ln in f:
            if not ln.strip() or ln.startswith("#"):
                continue
            key, *rest = ln.split()
            if key == "A_row_group_values":
                rows_a[int(rest[0])] = [float(v) for v in rest[1:]]
            elif key == "B_row_group_values":
                rows_b[int(rest[0])] = [float(v) for v in rest[1:]]
            else:
                vals[key] = rest
    return vals, rows_a, rows_b


def test_ue8m0_packed_worked_example_by_hand():
    vals, rows_a, rows_b = _read_packed_example()
    M, N, K = int(vals["M"][0]), int(vals["N"][0]), int(vals["K"][0])
    nkb = K // 128
    a_val = np.array([np.repeat(rows_a[m], 128) for m in range(M)], np.float32)
    b_val = np.array([np.repeat(rows_b[n], 128) for n in range(N)], np.float32)
    A, B = _e4m3_bytes_of_exact(a_val), _e4m3_bytes_of_exact(b_val)
    words = lambda key: np.array([int(w, 16) for w in vals[key]], np.uint32).view(np.int32)
    sA_packed = words("sA_packed").reshape((nkb + 3) // 4, dg_inputs.align4(M))
    sB_packed = words("sB_packed").reshape(1, (nkb + 3) // 4)
    sA = oracle.unpack_ue8m0_a(sA_packed, nkb)
    sB = oracle.unpack_ue8m0_b(sB_packed, nkb)
    ref64, D = oracle.gemm_nt(A, sA, B, sB, threads=1)
    assert ref64.ravel().tolist() == [float(v) for v in vals["D64"]]
    assert D.ravel().tolist() == [int(v, 16) for v in vals["D_bf16"]]


@pytest.mark.parametrize("G,M,N,K", [(1, 7, 130, 640), (2, 130, 40, 1024), (3, 1, 257, 200)])
def test_ue8m0_unpack_inverts_the_generators_packer(G, M, N, K):
    a = dg_inputs.make_a(M, K, seed=12, ue8m0=True)
    b = dg_inputs.make_b(G, N, K, seed=12, ue8m0=True)
    nkb = (K + 127) // 128
    sA = oracle.unpack_ue8m0_a(dg_inputs.pack_ue8m0_a(a.sA), nkb)
    sB = oracle.unpack_ue8m0_b(dg_inputs.pack_ue8m0_b(b.sB), nkb)
    assert np.array_equal(sA[:, :M], a.sA[:, :M])
    assert np.all(sA[:, M:] == 1.0)                     # padding columns pack as code 127
    assert np.array_equal(sB, b.sB)


@pytest.mark.parametrize("M,N,K,dist", [(40, 300, 896, dg_inputs.NORMAL), (129, 64, 272, dg_inputs.STUDENT_T3)])
def test_ue8m0_gemm_matches_dequantised_definition(M, N, K, dist):
    a = dg_inputs.make_a(M, K, seed=13, dist=dist, ue8m0=True)
    b = dg_inputs.make_b(1, N, K, seed=13, dist=dist, ue8m0=True)
    nkb = (K + 127) // 128
    sA = oracle.unpack_ue8m0_a(dg_inputs.pack_ue8m0_a(a.sA), nkb)
    sB = oracle.unpack_ue8m0_b(dg_inputs.pack_ue8m0_b(b.sB[0]), nkb)
    ref64, _ = oracle.gemm_nt(a.A, sA, b.B[0], sB, threads=4)
    want = _numpy_definition(a.A, a.sA, b.B[0], b.sB[0])
    scale = np.abs(want).max()
    assert np.abs(ref64 - want).max() <= 1e-13 * scale


# ----------------------------------------------------------------------------------------------
# Accumulating form D = C + A·Bᵀ


def test_gemm_acc_worked_example_by_hand():
    # The 2x2 example above (A·Bᵀ = [[192, 0], [4224, 0]]) plus C = [[1, 2], [3, 4]].
    A = np.array([[0x38] * 256, [0x40] * 256], np.uint8)
    B = np.array([[0x30] * 256, [0x38, 0xB8] * 128], np.uint8)
    sA = np.array([[1.0, 0.5, 0, 0], [0.25, 8.0, 0, 0]], np.float32)
    sB = np.array([[2.0, 4.0]], np.float32)
    C = np.array([[1.0, 2.0], [3.0, 4.0]], np.float32)
    assert oracle.gemm_nt_acc(A, sA, B, sB, C, threads=1).tolist() == [[193.0, 2.0], [4227.0, 4.0]]


def test_gemm_acc_reduces_to_its_parts():
    M, N, K = 37, 200, 640
    a = dg_inputs.make_a(M, K, seed=14)
    b = dg_inputs.make_b(1, N, K, seed=14)
    C = dg_inputs.draw(14, 5, M * N).reshape(M, N) * 100
    ref, _ = oracle.gemm_nt(a.A, a.sA, b.B[0], b.sB[0], threads=2)
    assert np.array_equal(oracle.gemm_nt_acc(a.A, a.sA, b.B[0], b.sB[0], np.zeros_like(C), threads=2), ref)
    zero_a = np.zeros_like(a.A)
    assert np.array_equal(oracle.gemm_nt_acc(zero_a, a.sA, b.B[0], b.sB[0], C, threads=2), C.astype(np.float64))
    rng = np.random.default_rng(1)
    ms, ns = rng.integers(0, M, 100), rng.integers(0, N, 100)
    full = oracle.gemm_nt_acc(a.A, a.sA, b.B[0], b.sB[0], C, threads=2)
    assert np.array_equal(oracle.gemm_nt_acc_sampled(a.A, a.sA, b.B[0], b.sB[0], C, ms, ns), full[ms, ns])


# ----------------------------------------------------------------------------------------------
# Masked GEMM fused with SwiGLU


def test_silu_against_scipy_and_limits():
    from scipy.special import expit
    x = np.concatenate([np.linspace(-30, 30, 601), [0.0, 1e-8, -1e-8, 700.0, -700.0]])
    got = oracle.silu(x)
    want = x * expit(x)
    assert np.allclose(got, want, rtol=1e-14, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert oracle.silu(np.array([50.0]))[0] == 50.0
    assert abs(oracle.silu(np.array([-50.0]))[0]) < 1e-19


def test_masked_swiglu_equals_silu_gate_times_up():
    G, M_max, I, K = 3, 160, 256, 384
    masked_m = np.array([0, 1, 160], np.int32)
    a = dg_inputs.make_masked_a(G, M_max, K, seed=15)
    b = dg_inputs.make_b(G, 2 * I, K, seed=15)
    H0 = np.full((G, M_max, I), 0xFFFF, np.uint16)
    ref, H, bad = oracle.grouped_masked_swiglu(a.A, a.sA, b.B, b.sB, masked_m, None, H0, threads=4)
    assert bad == 0
    full, _, _ = oracle.grouped_masked(a.A, a.sA, b.B, b.sB, masked_m, threads=4)
    from scipy.special import expit
    for g in range(G):
        v = masked_m[g]
        gate, up = full[g, :v, :I], full[g, :v, I:]
        assert np.allclose(ref[g, :v], gate * expit(gate) * up, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
        assert np.all(H[g, v:] == 0xFFFF)
    assert np.array_equal(H[2], oracle.bf16_from_f64(ref[2]))
    gs, ms, js = np.array([1, 2, 2]), np.array([0, 5, 159]), np.array([0, 255, 128])
    assert np.allclose(oracle.masked_swiglu_sampled(a.A, a.sA, b.B, b.sB, gs, ms, js), ref[gs, ms, js], rtol=1e-12)


# ----------------------------------------------------------------------------------------------
# K-grouped GEMM (groups along K)


def test_k_grouped_equals_dense_on_slices():
    M, N = 40, 136
    off = np.array([0, 256, 256, 640, 1024], np.int32)        # group 1 is empty
    K = int(off[-1])
    a = dg_inputs.make_a(M, K, seed=16)
    b = dg_inputs.make_b(1, N, K, seed=16)
    ref = oracle.k_grouped(a.A, a.sA, b.B[0], b.sB[0], off, threads=4)
    for g in range(len(off) - 1):
        k0, k1 = int(off[g]), int(off[g + 1])
        if k0 == k1:
            assert np.all(ref[g] == 0)
            continue
        kb = slice(k0 // 128, k1 // 128)
        sl, _ = oracle.gemm_nt(np.ascontiguousarray(a.A[:, k0:k1]), np.ascontiguousarray(a.sA[kb]),
                               np.ascontiguousarray(b.B[0][:, k0:k1]), np.ascontiguousarray(b.sB[0][:, kb]), threads=2)
        assert np.array_equal(ref[g], sl)
    full, _ = oracle.gemm_nt(a.A, a.sA, b.B[0], b.sB[0], threads=2)
    one = oracle.k_grouped(a.A, a.sA, b.B[0], b.sB[0], np.array([0, K], np.int32), threads=2)
    assert np.array_equal(one[0], full)
    assert np.allclose(ref.sum(axis=0), full, rtol=1e-12, atol=1e-12 * np.abs(full).max())
    with pytest.raises(ValueError):
        oracle.k_grouped(a.A, a.sA, b.B[0], b.sB[0], np.array([0, 100, K], np.int32))


# ----------------------------------------------------------------------------------------------
# The FP8 cast of H (e4m3_encode_rne, quantize_rows_e4m3), the reference of the fused SwiGLU with
# FP8 output: pinned against the OCP table round trip, torch's own float32 -> float8_e4m3fn
# conversion (round to nearest even), hand-worked ties and closed forms of the 1x128 scale rule.

def test_e4m3_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)   # all but the NaNs
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    back = oracle.e4m3_encode_rne(vals)
    # +0 and -0 keep their sign; every other code comes back as itself
    assert np.array_equal(back, codes)


def test_e4m3_encode_matches_torch_and_ties_go_to_even():
    rng = np.random.default_rng(0)
    y = np.concatenate([rng.uniform(-448, 448, 50000), rng.normal(0, 1e-2, 50000)]).astype(np.float32)
    ours = oracle.e4m3_encode_rne(y)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    # every midpoint between adjacent representable magnitudes goes to the even code
    vals = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (vals[:-1] + vals[1:]) / 2)   # exact in FP32
    want = np.where(np.arange(126) % 2 == 0, np.arange(126), np.arange(1, 127)).astype(np.uint8)
    assert np.array_equal(oracle.e4m3_encode_rne(mids), want)
    assert np.array_equal(oracle.e4m3_encode_rne(-mids), want | 0x80)
    # worked by hand: 1.0625 lies between 1.0 (0x38) and 1.125 (0x39) -> 0x38; 1.1875 between
    # 1.125 (0x39) and 1.25 (0x3A) -> 0x3A; 2^-10, half the smallest subnormal -> +0
    assert list(oracle.e4m3_encode_rne(np.array([1.0625, 1.1875, 2.0 ** -10], np.float32))) == [0x38, 0x3A, 0x00]


def test_quantize_rows_scale_rule_closed_forms():
    rng = np.random.default_rng(1)
    # a row whose group maximum is 448 has scale exactly 1: the codes are the values' own codes
    vals = oracle.e4m3_decode(rng.integers(0, 126, 256).astype(np.uint8)).astype(np.float32)
    vals[0], vals[128] = 448.0, -448.0
    codes, s = oracle.quantize_rows_e4m3(vals[None, :])
    assert s.shape == (2, 1) and np.all(s == 1.0)
    assert np.array_equal(codes[0], oracle.e4m3_encode_rne(vals))
    # an all-zero group has scale 1 and codes 0; the other group is unaffected by it
    h = rng.normal(0, 3, (3, 256)).astype(np.float32)
    h[1, :128] = 0.0
    codes, s = oracle.quantize_rows_e4m3(h)
    assert s[0, 1] == 1.0 and np.all(codes[1, :128] == 0)
    assert s[1, 1] == np.float32(np.max(np.abs(h[1, 128:]))) / np.float32(448.0)
    # scaling a group by a power of two scales its scale (the all-zero group keeps 1) and leaves its
    # codes as they are
    codes2, s2 = oracle.quantize_rows_e4m3(h * np.float32(2.0 ** -7))
    want = np.where(np.swapaxes(np.max(np.abs(h.reshape(3, 2, 128)), axis=-1), 0, 1) > 0, s * np.float32(2.0 ** -7), 1.0)
    assert np.array_equal(codes2, codes) and np.array_equal(s2, want.astype(np.float32))
    # dequantised values are within half an E4M3 step of the top binade of each group
    deq = oracle.e4m3_decode(codes).reshape(3, 2, 128) * np.swapaxes(s, 0, 1)[..., None]
    err = np.abs(deq - h.reshape(3, 2, 128).astype(np.float64))
    assert np.all(err <= (16.0 / 448.0) * np.max(np.abs(h.reshape(3, 2, 128)), axis=-1, keepdims=True) * 1.0001)
