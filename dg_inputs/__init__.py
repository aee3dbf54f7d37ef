"""Seeded synthetic operands for the FP8 (E4M3) fine-grained-scaled GEMM.

Input preparation shared by the CUDA path, the CPU oracle, the tests and the benchmark. It holds
no GEMM arithmetic: it draws values from a counter-based SplitMix64 generator (Box-Muller
normals, Student-t with three degrees of freedom), applies optional activation-channel
outliers, and quantises to E4M3 bytes with the DeepSeek-V3 fine-grained scheme (one FP32 scale
per 1x128 K-group of each A row, one per 128x128 block of B, s = amax/448). The C source,
``dg_inputs.c``, documents every step.

Streams: A is stream 0, B stream 1, outlier channels stream 2, ``masked_m`` stream 3.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dg_inputs.c")
_LIB = os.path.join(_HERE, "libdg_inputs.so")
_lib = None

NORMAL = 0
STUDENT_T3 = 1


def build(force: bool = False) -> str:
    """Compile ``dg_inputs.c`` into ``libdg_inputs.so`` next to it (gcc, no -march flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, u64, f32, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_double
        lib.dgi_e4m3_encode.restype = ctypes.c_uint8
        lib.dgi_e4m3_encode.argtypes = [f32]
        lib.dgi_e4m3_encode_array.argtypes = [P, P, i64]
        lib.dgi_fill.argtypes = [u64, u64, i32, i64, i64, P, i32]
        lib.dgi_outlier_channels.restype = i32
        lib.dgi_outlier_channels.argtypes = [u64, i32, dbl, P]
        lib.dgi_make_a.argtypes = [u64, u64, i32, i64, i32, i32, P, i32, f32, P, P, i64, i32, i32]
        lib.dgi_quantize_a.argtypes = [P, i32, i32, P, P, i64, i32, i32]
        lib.dgi_make_b.argtypes = [u64, u64, i32, i32, i32, i32, P, P, i32, i32]
        lib.dgi_quantize_b.argtypes = [P, i32, i32, i32, P, P, i32, i32]
        lib.dgi_make_masked_m.argtypes = [u64, i32, i32, i32, P]
        _lib = lib
    return _lib


def _threads(threads):
    return int(threads) if threads else (os.cpu_count() or 1)


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def ceil_div(a: int, b: int) -> int:
    return (a + b - 1) // b


def align4(x: int) -> int:
    """Row stride of the MN-major A scales: x rounded up to 4 floats (16 bytes)."""
    return (x + 3) // 4 * 4


def e4m3_encode(x) -> np.ndarray:
    """Nearest-even E4M3 bytes of float32 values, saturating at +-448 (input preparation)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint8)
    _load().dgi_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def draw(seed: int, stream: int, n: int, dist: int = NORMAL, base: int = 0, threads=None) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().dgi_fill(seed, stream, dist, base, n, _ptr(out), _threads(threads))
    return out


def outlier_channels(seed: int, K: int, frac: float) -> np.ndarray:
    n = int(np.floor(frac * K + 0.5))
    out = np.empty(max(n, 1), dtype=np.int32)
    got = _load().dgi_outlier_channels(seed, K, frac, _ptr(out))
    if got < 0:
        raise MemoryError("dgi_outlier_channels")
    return out[:got].copy()


@dataclass
class OperandA:
    """A[M,K] E4M3 bytes (K contiguous) and its MN-major scales sA[ceil(K/128)][align4(M)]."""
    A: np.ndarray
    sA: np.ndarray

    @property
    def ldsa(self) -> int:
        return self.sA.shape[-1]


@dataclass
class OperandB:
    """B[G,N,K] E4M3 bytes (K contiguous) and scales sB[G][ceil(N/128)][ceil(K/128)]."""
    B: np.ndarray
    sB: np.ndarray


def make_a(M: int, K: int, seed: int = 0, dist: int = NORMAL, base_row: int = 0,
           outlier_frac: float = 0.0, outlier_scale: float = 64.0, stream: int = 0,
           threads=None, ue8m0: bool = False) -> OperandA:
    """ue8m0=True quantises with power-of-two scales (smallest 2^p >= amax/448), the scales that
    the packed-UE8M0 entry points take (pack them with ``pack_ue8m0_a``)."""
    A = np.empty((M, K), dtype=np.uint8)
    sA = np.empty((ceil_div(K, 128), align4(M)), dtype=np.float32)
    ch = outlier_channels(seed, K, outlier_frac) if outlier_frac > 0 else np.zeros(1, np.int32)
    n_out = len(ch) if outlier_frac > 0 else 0
    _load().dgi_make_a(seed, stream, dist, base_row, M, K, _ptr(ch), n_out, outlier_scale,
                       _ptr(A), _ptr(sA), sA.shape[1], 1 if ue8m0 else 0, _threads(threads))
    return OperandA(A, sA)


def quantize_a(x: np.ndarray, threads=None, ue8m0: bool = False) -> OperandA:
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    A = np.empty((M, K), dtype=np.uint8)
    sA = np.empty((ceil_div(K, 128), align4(M)), dtype=np.float32)
    _load().dgi_quantize_a(_ptr(x), M, K, _ptr(A), _ptr(sA), sA.shape[1], 1 if ue8m0 else 0,
                           _threads(threads))
    return OperandA(A, sA)


def make_b(G: int, N: int, K: int, seed: int = 0, dist: int = NORMAL, stream: int = 1,
           threads=None, ue8m0: bool = False) -> OperandB:
    B = np.empty((G, N, K), dtype=np.uint8)
    sB = np.empty((G, ceil_div(N, 128), ceil_div(K, 128)), dtype=np.float32)
    _load().dgi_make_b(seed, stream, dist, G, N, K, _ptr(B), _ptr(sB), 1 if ue8m0 else 0,
                       _threads(threads))
    return OperandB(B, sB)


def quantize_b(x: np.ndarray, threads=None, ue8m0: bool = False) -> OperandB:
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 2:
        x = x[None]
    G, N, K = x.shape
    B = np.empty((G, N, K), dtype=np.uint8)
    sB = np.empty((G, ceil_div(N, 128), ceil_div(K, 128)), dtype=np.float32)
    _load().dgi_quantize_b(_ptr(x), G, N, K, _ptr(B), _ptr(sB), 1 if ue8m0 else 0, _threads(threads))
    return OperandB(B, sB)


def _e8m0_codes(s: np.ndarray) -> np.ndarray:
    """E8M0 code of each power-of-two FP32 scale in [2^-127, 2^127] (the exponent field; 2^-127,
    an FP32 subnormal, has exponent field 0 = code 0)."""
    s = np.ascontiguousarray(s, dtype=np.float32)
    bits = s.view(np.uint32)
    frac = bits & 0x7FFFFF
    expo = (bits >> 23) & 0xFF
    ok = (s > 0) & (((expo > 0) & (frac == 0)) | ((expo == 0) & (frac == 0x400000)))
    if not np.all(ok):
        raise ValueError("scales must be powers of two in [2^-127, 2^127] to pack as UE8M0")
    return expo.astype(np.uint32)


def _pack4(codes: np.ndarray, axis: int) -> np.ndarray:
    """Packs codes four at a time along `axis` into int32: byte j of word q = entry 4q+j; the
    bytes past the end are 127 (the scale 1.0)."""
    codes = np.moveaxis(codes, axis, -1)
    n = codes.shape[-1]
    nq = ceil_div(n, 4)
    padded = np.full(codes.shape[:-1] + (nq * 4,), 127, np.uint32)
    padded[..., :n] = codes
    q = padded.reshape(codes.shape[:-1] + (nq, 4))
    words = q[..., 0] | (q[..., 1] << 8) | (q[..., 2] << 16) | (q[..., 3] << 24)
    return np.ascontiguousarray(np.moveaxis(words.astype(np.uint32).view(np.int32), -1, axis))


def pack_ue8m0_a(sA: np.ndarray) -> np.ndarray:
    """A's MN-major FP32 scales [..., nkb, ldsa] (powers of two) -> packed UE8M0
    [..., ceil(nkb/4), ldsa] int32. Padding columns (m >= M, scale 0) pack as 127."""
    sA = np.array(sA, dtype=np.float32, copy=True)
    sA[sA == 0] = 1.0
    return _pack4(_e8m0_codes(sA), axis=-2)


def pack_ue8m0_b(sB: np.ndarray) -> np.ndarray:
    """B's FP32 scales [..., nnb, nkb] (powers of two) -> packed UE8M0 [..., nnb, ceil(nkb/4)]."""
    return _pack4(_e8m0_codes(sB), axis=-1)


def make_masked_m(G: int, M_max: int, seed: int = 0, force_ends: bool = True) -> np.ndarray:
    out = np.empty(G, dtype=np.int32)
    _load().dgi_make_masked_m(seed, G, M_max, 1 if force_ends else 0, _ptr(out))
    return out


def make_masked_a(G: int, M_max: int, K: int, seed: int = 0, dist: int = NORMAL, threads=None,
                  ue8m0: bool = False) -> OperandA:
    """A[G,M_max,K] and sA[G][ceil(K/128)][align4(M_max)]: group g is rows [g*M_max, (g+1)*M_max)
    of stream 0, each group quantised with its own MN-major scale block."""
    ldsa = align4(M_max)
    A = np.empty((G, M_max, K), dtype=np.uint8)
    sA = np.empty((G, ceil_div(K, 128), ldsa), dtype=np.float32)
    ch = np.zeros(1, np.int32)
    lib = _load()
    for g in range(G):
        Ag = np.empty((M_max, K), dtype=np.uint8)
        sAg = np.empty((ceil_div(K, 128), ldsa), dtype=np.float32)
        lib.dgi_make_a(seed, 0, dist, g * M_max, M_max, K, _ptr(ch), 0, 64.0,
                       _ptr(Ag), _ptr(sAg), ldsa, 1 if ue8m0 else 0, _threads(threads))
        A[g] = Ag
        sA[g] = sAg
    return OperandA(A, sA)


def contiguous_m_indices(rows_per_group, pad_to: int = 128) -> np.ndarray:
    """Per-row group index of the contiguous layout: group g's rows follow group g-1's, each
    segment padded with -1 rows up to a multiple of ``pad_to``."""
    out = []
    for g, r in enumerate(rows_per_group):
        seg = ceil_div(r, pad_to) * pad_to if pad_to else r
        out.append(np.full(r, g, dtype=np.int32))
        out.append(np.full(seg - r, -1, dtype=np.int32))
    return np.concatenate(out) if out else np.zeros(0, np.int32)
