"""CPU oracle of the FP8 (E4M3) fine-grained-scaled GEMM — TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and its
``--impl reference`` arm) may import this package. The CUDA path never does; the two share no
code. ``dg_oracle.cpp`` holds the arithmetic and documents, function by function, which passage
of the DeepGEMM pages (or which outside definition: OCP E4M3, IEEE rounding, the DeepSeek-V3
scale granularity) it follows.

Every function here is pinned by ``tests/test_oracle_pins.py`` against things other than itself:
the OCP E4M3 and E8M0 tables and torch's float8 conversions, torch's float32->bfloat16 rounding,
exact integer brute force, closed forms, a hand-worked packed-UE8M0 example, and the plain
dequantise-then-matmul definition computed by numpy.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dg_oracle.cpp")
_LIB = os.path.join(_HERE, "libdg_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``dg_oracle.cpp`` into ``libdg_oracle.so`` (g++, -ffp-contract=off, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_int64
        lib.dgo_e4m3_decode.restype = ctypes.c_double
        lib.dgo_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.dgo_bf16_from_f64.restype = ctypes.c_uint16
        lib.dgo_bf16_from_f64.argtypes = [ctypes.c_double]
        lib.dgo_bf16_from_f64_array.argtypes = [P, P, i64]
        lib.dgo_gemm_nt.argtypes = [P, P, i64, P, P, i32, i32, i32, P, P, i32]
        lib.dgo_grouped_contiguous.restype = i32
        lib.dgo_grouped_contiguous.argtypes = [P, P, i64, P, P, P, i32, i32, i32, i32, P, P, i32]
        lib.dgo_grouped_masked.restype = i32
        lib.dgo_grouped_masked.argtypes = [P, P, i64, P, P, P, i32, i32, i32, i32, P, P, i32]
        lib.dgo_gemm_nt_sampled.argtypes = [P, P, i64, P, P, i32, i32, i32, i64, P, P, P, i32]
        lib.dgo_gemm_nt_acc.argtypes = [P, P, i64, P, P, P, i32, i32, i32, P, i32]
        lib.dgo_grouped_masked_swiglu.restype = i32
        lib.dgo_grouped_masked_swiglu.argtypes = [P, P, i64, P, P, P, i32, i32, i32, i32, P, P, i32]
        lib.dgo_k_grouped.restype = i32
        lib.dgo_k_grouped.argtypes = [P, P, i64, P, P, P, i32, i32, i32, i32, P, i32]
        lib.dgo_silu.restype = ctypes.c_double
        lib.dgo_silu.argtypes = [ctypes.c_double]
        lib.dgo_hardware_threads.restype = i32
        lib.dgo_ue8m0_decode.restype = ctypes.c_double
        lib.dgo_ue8m0_decode.argtypes = [ctypes.c_uint8]
        lib.dgo_ue8m0_unpack.argtypes = [P, i64, i32, i64, i64, P, i64, i64]
        _lib = lib
    return _lib


def hardware_threads() -> int:
    return int(_load().dgo_hardware_threads())


def _threads(threads):
    return int(threads) if threads else hardware_threads()


def _p(a: np.ndarray):
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle inputs must be C-contiguous")
    return a.ctypes.data_as(ctypes.c_void_p)


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def e4m3_decode(codes) -> np.ndarray:
    """FP64 value of each E4M3 byte (OCP definition)."""
    codes = np.asarray(codes, dtype=np.uint8)
    lib = _load()
    return np.array([lib.dgo_e4m3_decode(int(c)) for c in codes.ravel()], dtype=np.float64).reshape(codes.shape)


def bf16_from_f64(x) -> np.ndarray:
    """BF16 bit patterns (uint16) of FP64 values, rounded to nearest-even directly from FP64."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, dtype=np.uint16)
    _load().dgo_bf16_from_f64_array(_p(x), _p(out), x.size)
    return out


def gemm_nt(A, sA, B, sB, threads=None, want_ref64=True, want_bf16=True):
    """Dense D = A·Bᵀ. A[M,K] u8, sA[ceil(K/128)][ldsa] f32, B[N,K] u8, sB[ceil(N/128)][ceil(K/128)].

    Returns (ref64 [M,N] float64 or None, D [M,N] uint16 BF16 bits or None)."""
    A, B, sA, sB = _u8(A), _u8(B), _f32(sA), _f32(sB)
    if B.ndim == 3:
        B, sB = B[0], sB[0]
    M, K = A.shape
    N = B.shape[0]
    ref = np.zeros((M, N), np.float64) if want_ref64 else None
    D = np.zeros((M, N), np.uint16) if want_bf16 else None
    _load().dgo_gemm_nt(_p(A), _p(sA), sA.shape[-1], _p(B), _p(sB), M, N, K,
                        _p(ref) if ref is not None else None, _p(D) if D is not None else None,
                        _threads(threads))
    return ref, D


def gemm_nt_acc(A, sA, B, sB, C, threads=None) -> np.ndarray:
    """Accumulating dense D = C + A·Bᵀ in FP64 (C float32 [M,N]). Returns ref64 [M,N]."""
    A, B, sA, sB = _u8(A), _u8(B), _f32(sA), _f32(sB)
    if B.ndim == 3:
        B, sB = B[0], sB[0]
    C = _f32(C)
    M, K = A.shape
    N = B.shape[0]
    assert C.shape == (M, N)
    ref = np.empty((M, N), np.float64)
    _load().dgo_gemm_nt_acc(_p(A), _p(sA), sA.shape[-1], _p(B), _p(sB), _p(C), M, N, K, _p(ref), _threads(threads))
    return ref


def gemm_nt_acc_sampled(A, sA, B, sB, C, ms, ns, threads=None) -> np.ndarray:
    """FP64 values of sampled elements of D = C + A·Bᵀ."""
    ms = np.asarray(ms, np.int64)
    ns = np.asarray(ns, np.int64)
    return np.asarray(C, np.float32)[ms, ns].astype(np.float64) + gemm_nt_sampled(A, sA, B, sB, ms, ns, threads)


def grouped_contiguous(A, sA, B, sB, m_indices, ref64_init=None, D_init=None, threads=None):
    """Contiguous grouped D. Rows whose m_indices is -1 (or invalid) keep the initial contents.

    Returns (ref64, D, n_invalid_rows)."""
    A, B, sA, sB = _u8(A), _u8(B), _f32(sA), _f32(sB)
    m_indices = np.ascontiguousarray(m_indices, dtype=np.int32)
    M, K = A.shape
    G, N, _ = B.shape
    ref = np.array(ref64_init, dtype=np.float64, copy=True) if ref64_init is not None else np.zeros((M, N), np.float64)
    D = np.array(D_init, dtype=np.uint16, copy=True) if D_init is not None else np.zeros((M, N), np.uint16)
    bad = _load().dgo_grouped_contiguous(_p(A), _p(sA), sA.shape[-1], _p(B), _p(sB), _p(m_indices),
                                         M, N, K, G, _p(ref), _p(D), _threads(threads))
    return ref, D, int(bad)


def grouped_masked(A, sA, B, sB, masked_m, ref64_init=None, D_init=None, threads=None):
    """Masked grouped D[G,M_max,N]: rows m >= masked_m[g] keep the initial contents.

    Returns (ref64, D, n_clamped_groups)."""
    A, B, sA, sB = _u8(A), _u8(B), _f32(sA), _f32(sB)
    masked_m = np.ascontiguousarray(masked_m, dtype=np.int32)
    G, M_max, K = A.shape
    N = B.shape[1]
    ref = np.array(ref64_init, dtype=np.float64, copy=True) if ref64_init is not None else np.zeros((G, M_max, N), np.float64)
    D = np.array(D_init, dtype=np.uint16, copy=True) if D_init is not None else np.zeros((G, M_max, N), np.uint16)
    bad = _load().dgo_grouped_masked(_p(A), _p(sA), sA.shape[-1], _p(B), _p(sB), _p(masked_m),
                                     G, M_max, N, K, _p(ref), _p(D), _threads(threads))
    return ref, D, int(bad)


def silu(x) -> np.ndarray:
    """x / (1 + e^-x) in FP64."""
    x = np.asarray(x, np.float64)
    lib = _load()
    return np.array([lib.dgo_silu(float(v)) for v in x.ravel()], np.float64).reshape(x.shape)


def e4m3_encode_rne(y) -> np.ndarray:
    """E4M3 code of each FP32 value y with |y| <= 448: the representable value nearest to y (the
    finite values of the OCP table, from ``e4m3_decode``), a tie going to the even code (even
    mantissa), the sign of y kept (a negative value that rounds to zero gives -0, code 0x80).
    Values beyond ±448 must have been clamped by the caller."""
    y = np.asarray(y, np.float32)
    if np.any(np.abs(y) > 448.0) or np.any(np.isnan(y)):
        raise ValueError("e4m3_encode_rne takes finite values with |y| <= 448")
    codes = np.arange(0, 127, dtype=np.uint8)                 # 0x00..0x7E: +0 .. 448
    vals = e4m3_decode(codes)                                  # increasing
    a = np.abs(y.astype(np.float64)).ravel()
    hi = np.searchsorted(vals, a, side="left")                 # vals[hi-1] < a <= vals[hi]
    hi = np.clip(hi, 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick = np.where(d_hi < d_lo, hi, np.where(d_lo < d_hi, lo, np.where(codes[hi] % 2 == 0, hi, lo)))
    out = codes[pick].astype(np.uint8)
    out = np.where(np.signbit(y.ravel()), out | np.uint8(0x80), out).astype(np.uint8)
    return out.reshape(y.shape)


def quantize_rows_e4m3(H, group: int = 128):
    """FP8 cast of H [..., R, C] per 1 x ``group`` group of each row: the group is mapped onto the
    E4M3 range by the factor 448/amax (an FP32 division, once per group) and its dequantisation scale
    is s = amax/448 (FP32); codes = e4m3_rne(clamp(H · (448/amax), ±448)) with the FP32 product. An
    all-zero group has factor 1 and scale 1. Returns (codes [..., R, C] uint8, scales [..., C/group, R]
    float32: the MN-major LHS scale layout, unpadded)."""
    H = np.asarray(H, np.float32)
    *lead, R, C = H.shape
    if C % group:
        raise ValueError("the row length must be a multiple of the group")
    Hg = H.reshape(*lead, R, C // group, group)
    amax = np.max(np.abs(Hg), axis=-1)                                     # [..., R, C/group] FP32
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1.0)).astype(np.float32)
    s = np.where(nz, (safe / np.float32(448.0)).astype(np.float32), np.float32(1.0)).astype(np.float32)
    inv = np.where(nz, (np.float32(448.0) / safe).astype(np.float32), np.float32(1.0)).astype(np.float32)
    y = (Hg * inv[..., None]).astype(np.float32)                          # FP32 product, rounded once
    y = np.clip(y, np.float32(-448.0), np.float32(448.0))
    codes = e4m3_encode_rne(y).reshape(*lead, R, C)
    return codes, np.swapaxes(s, -1, -2).copy()


def grouped_masked_swiglu(A, sA, B, sB, masked_m, ref64_init=None, H_init=None, threads=None):
    """Masked grouped GEMM fused with SwiGLU: B [G, 2I, K] (gate rows then up rows),
    H[g,m,j] = silu(D[g,m,j])·D[g,m,I+j] for m < masked_m[g]. Returns (ref64, H bf16 bits, n_clamped)."""
    A, B, sA, sB = _u8(A), _u8(B), _f32(sA), _f32(sB)
    masked_m = np.ascontiguousarray(masked_m, dtype=np.int32)
    G, M_max, K = A.shape
    I = B.shape[1] // 2
    ref = np.array(ref64_init, np.float64, copy=True) if ref64_init is not None else np.zeros((G, M_max, I), np.float64)
    H = np.array(H_init, np.uint16, copy=True) if H_init is not None else np.zeros((G, M_max, I), np.uint16)
    bad = _load().dgo_grouped_masked_swiglu(_p(A), _p(sA), sA.shape[-1], _p(B), _p(sB), _p(masked_m), G, M_max, I,
                                            K, _p(ref), _p(H), _threads(threads))
    return ref, H, int(bad)


def masked_swiglu_sampled(A, sA, B, sB, gs, ms, js, threads=None) -> np.ndarray:
    """FP64 values H[g,m,j] of the fused SwiGLU output at sampled positions (rows must be valid)."""
    I = B.shape[1] // 2
    js = np.asarray(js, np.int64)
    gate = masked_sampled(A, sA, B, sB, gs, ms, js, threads)
    up = masked_sampled(A, sA, B, sB, gs, ms, js + I, threads)
    return silu(gate) * up


def k_grouped(A, sA, B, sB, offsets, threads=None) -> np.ndarray:
    """K-grouped D[g] = Σ_{k in [off[g], off[g+1])} of the logical A[M,K_total]·B[N,K_total]ᵀ terms,
    with the scales of those K-blocks. Returns ref64 [G,M,N]."""
    A, B, sA, sB = _u8(A), _u8(B), _f32(sA), _f32(sB)
    if B.ndim == 3:
        B, sB = B[0], sB[0]
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    M, K = A.shape
    N = B.shape[0]
    G = len(off) - 1
    ref = np.zeros((G, M, N), np.float64)
    bad = _load().dgo_k_grouped(_p(A), _p(sA), sA.shape[-1], _p(B), _p(sB), _p(off), G, M, N, K, _p(ref),
                                _threads(threads))
    if bad:
        raise ValueError(f"{bad} invalid K offsets")
    return ref


def gemm_nt_sampled(A, sA, B, sB, ms, ns, threads=None) -> np.ndarray:
    """FP64 values of the elements (ms[i], ns[i]) of a dense D = A·Bᵀ."""
    A, B, sA, sB = _u8(A), _u8(B), _f32(sA), _f32(sB)
    if B.ndim == 3:
        B, sB = B[0], sB[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(len(ms), np.float64)
    M, K = A.shape
    _load().dgo_gemm_nt_sampled(_p(A), _p(sA), sA.shape[-1], _p(B), _p(sB), M, B.shape[0], K,
                                len(ms), _p(ms), _p(ns), _p(out), _threads(threads))
    return out


def contiguous_sampled(A, sA, B, sB, m_indices, ms, ns, threads=None) -> np.ndarray:
    """FP64 values of sampled elements of a contiguous grouped problem (rows must be valid)."""
    m_indices = np.asarray(m_indices)
    ms = np.asarray(ms, np.int64)
    ns = np.asarray(ns, np.int64)
    out = np.empty(len(ms), np.float64)
    groups = m_indices[ms]
    for g in np.unique(groups):
        sel = np.nonzero(groups == g)[0]
        out[sel] = gemm_nt_sampled(A, sA, B[g], sB[g], ms[sel], ns[sel], threads)
    return out


def masked_sampled(A, sA, B, sB, gs, ms, ns, threads=None) -> np.ndarray:
    """FP64 values of sampled elements (g, m, n) of a masked grouped problem."""
    gs = np.asarray(gs, np.int64)
    ms = np.asarray(ms, np.int64)
    ns = np.asarray(ns, np.int64)
    out = np.empty(len(ms), np.float64)
    for g in np.unique(gs):
        sel = np.nonzero(gs == g)[0]
        out[sel] = gemm_nt_sampled(A[g], sA[g], B[g], sB[g], ms[sel], ns[sel], threads)
    return out


# ---------------------------------------------------------------------------------------------
# Packed UE8M0 scales (four OCP E8M0 codes per int32; byte j of word q is K-group 4q+j). The GEMM
# with such scales is the GEMM above with the unpacked (exact, power-of-two) FP32 scales.


def ue8m0_decode(codes) -> np.ndarray:
    """FP64 value of each E8M0 byte: 2^(e-127), NaN for 0xFF."""
    codes = np.asarray(codes, dtype=np.uint8)
    lib = _load()
    return np.array([lib.dgo_ue8m0_decode(int(c)) for c in codes.ravel()], dtype=np.float64).reshape(codes.shape)


def unpack_ue8m0_a(sA_packed, nkb: int) -> np.ndarray:
    """A's MN-major packed scales [..., ceil(nkb/4), ldsa] int32 -> FP32 [..., nkb, ldsa]."""
    p = np.ascontiguousarray(sA_packed, dtype=np.int32)
    lead, (nkq, ldsa) = p.shape[:-2], p.shape[-2:]
    assert nkq == (nkb + 3) // 4
    p2 = p.reshape(-1, nkq, ldsa)
    out = np.empty((p2.shape[0], nkb, ldsa), np.float32)
    lib = _load()
    for g in range(p2.shape[0]):
        pg = np.ascontiguousarray(p2[g])
        og = np.empty((nkb, ldsa), np.float32)
        lib.dgo_ue8m0_unpack(_p(pg), ldsa, nkb, 1, ldsa, _p(og), 1, ldsa)
        out[g] = og
    return out.reshape(*lead, nkb, ldsa)


def unpack_ue8m0_b(sB_packed, nkb: int) -> np.ndarray:
    """B's packed scales [..., nnb, ceil(nkb/4)] int32 -> FP32 [..., nnb, nkb]."""
    p = np.ascontiguousarray(sB_packed, dtype=np.int32)
    lead, (nnb, nkq) = p.shape[:-2], p.shape[-2:]
    assert nkq == (nkb + 3) // 4
    flat = np.ascontiguousarray(p.reshape(-1, nkq))
    out = np.empty((flat.shape[0], nkb), np.float32)
    _load().dgo_ue8m0_unpack(_p(flat), flat.shape[0], nkb, nkq, 1, _p(out), nkb, 1)
    return out.reshape(*lead, nnb, nkb)
