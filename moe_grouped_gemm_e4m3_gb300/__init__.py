"""FP8 (E4M3) fine-grained-scaled GEMM for GB300 — thin Python binding of libdg (include/dg.h).

Argument marshalling only: every step of the GEMM runs in the sm_103a kernels of ``libdg.so``.
PyTorch supplies device memory and the current CUDA stream. There is no fallback: if the library
is missing or cannot load, every call raises.

The names mirror the C ABI:

* ``dg_fp8_gemm_nt(A, sA, B, sB, D)``                       dense D = A·Bᵀ
* ``dg_fp8_grouped_contiguous(A, sA, B, sB, m_indices, D)``  M-grouped, contiguous layout
* ``dg_fp8_grouped_masked(A, sA, B, sB, masked_m, D)``       M-grouped, masked layout
* ``*_f32`` variants store the FP32 accumulator instead of BF16 (same kernel and order).
* ``dg_fp8_gemm_{nn,tn,tt}(A, sA, B, sB, D, M=, N=, K=)``     dense D = A·Bᵀ with A stored [K,M] (t) and/or
  B stored [K,N] (second letter n); the scales keep dg_fp8_gemm_nt's layouts
* ``dg_fp8_k_grouped_gemm_tn_contiguous(A, sA, B, sB, k_offsets, D)``  groups along K: A [K,M], B [K,N],
  D [G,M,N]
* ``dg_fp8_grouped_masked_swiglu(A, sA, B, sB, masked_m, H)``  masked GEMM + SwiGLU: B [G, 2I, K], H [G, M_max, I]
* ``dg_fp8_gemm_nt_acc_f32(A, sA, B, sB, C, D)``             D = C + A·Bᵀ (FP32 C and D; C may be D)
* ``*_ue8m0`` variants take power-of-two scales as packed UE8M0 int32 words (four K-groups per
  word, byte j = K-group 4q+j): sA int32 [ceil(ceil(K/128)/4), align4(rows)] (masked: leading G),
  sB int32 [G, ceil(N/128), ceil(ceil(K/128)/4)]. They run the block-scaled tensor-core kernel.

Tensor contract (all CUDA, contiguous): A uint8/float8_e4m3fn [rows, K] (masked: [G, M_max, K]);
B uint8/float8_e4m3fn [N, K] or [G, N, K]; sA float32 MN-major [ceil(K/128), align4(rows)]
(masked: [G, ceil(K/128), align4(M_max)]); sB float32 [G, ceil(N/128), ceil(K/128)]; D bfloat16
(or float32) [rows, N] (masked: [G, M_max, N]); m_indices / masked_m int32.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build_mod

__all__ = [
    "DGError", "load", "dg_fp8_gemm_nt", "dg_fp8_gemm_nt_f32", "dg_fp8_grouped_contiguous",
    "dg_fp8_grouped_contiguous_f32", "dg_fp8_grouped_masked", "dg_fp8_grouped_masked_f32", "dg_fp8_gemm_nt_noalloc",
    "dg_get_tma_aligned_size", "dg_get_mk_alignment_for_contiguous_layout", "dg_set_num_sms",
    "dg_get_num_sms", "dg_get_device_status", "dg_last_error_string", "dg_query_config",
    "dg_set_tail_splits", "dg_set_cluster_split", "dg_set_wait_limit_us", "dg_set_pair_b", "dg_set_pdl", "dg_get_pdl",
    "dg_transform_sf_into_ue8m0_a", "dg_transform_sf_into_ue8m0_b", "dg_transform_sf_a_into_mn_major",
    "dg_fp8_gemm_nt_ue8m0", "dg_fp8_gemm_nt_ue8m0_f32", "dg_fp8_grouped_contiguous_ue8m0",
    "dg_fp8_grouped_contiguous_ue8m0_f32", "dg_fp8_grouped_masked_ue8m0", "dg_fp8_grouped_masked_ue8m0_f32",
    "dg_query_config_ue8m0", "dg_fp8_gemm_nt_acc_f32", "dg_fp8_gemm_nt_ue8m0_acc_f32",
    "dg_fp8_grouped_masked_swiglu", "dg_fp8_grouped_masked_swiglu_f32", "dg_fp8_grouped_masked_swiglu_fp8",
    "dg_fp8_grouped_masked_swiglu_ue8m0",
    "dg_fp8_grouped_masked_swiglu_ue8m0_f32", "dg_fp8_gemm_nn", "dg_fp8_gemm_nn_f32",
    "dg_fp8_gemm_tn", "dg_fp8_gemm_tn_f32", "dg_fp8_gemm_tt", "dg_fp8_gemm_tt_f32",
    "dg_fp8_gemm_nn_ue8m0", "dg_fp8_gemm_nn_ue8m0_f32", "dg_fp8_gemm_tn_ue8m0", "dg_fp8_gemm_tn_ue8m0_f32", "dg_fp8_gemm_tt_ue8m0", "dg_fp8_gemm_tt_ue8m0_f32",
    "dg_fp8_k_grouped_gemm_tn_contiguous", "dg_fp8_k_grouped_gemm_tn_contiguous_f32",
    "dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0", "dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0_f32", "EXPORTED_SYMBOLS", "DG_OK", "DG_ERR_INVALID_ARG", "DG_ERR_ALIGNMENT", "DG_ERR_UNSUPPORTED",
    "DG_ERR_CUDA", "DG_ERR_DEVICE_STATUS", "DG_DEV_BAD_GROUP_INDEX", "DG_DEV_BAD_MASKED_M",
    "DG_DEV_TIMEOUT", "DG_DEV_BAD_SCALE",
]

DG_OK, DG_ERR_INVALID_ARG, DG_ERR_ALIGNMENT, DG_ERR_UNSUPPORTED, DG_ERR_CUDA, DG_ERR_DEVICE_STATUS = range(6)
DG_DEV_BAD_GROUP_INDEX, DG_DEV_BAD_MASKED_M, DG_DEV_TIMEOUT, DG_DEV_BAD_SCALE = 0x1, 0x2, 0x4, 0x8

# Every symbol include/dg.h declares (checked against the built library by the CPU tests).
EXPORTED_SYMBOLS = (
    "dg_fp8_gemm_nt", "dg_fp8_gemm_nt_f32", "dg_fp8_grouped_contiguous", "dg_fp8_grouped_contiguous_f32",
    "dg_fp8_grouped_masked", "dg_fp8_grouped_masked_f32", "dg_get_tma_aligned_size",
    "dg_get_mk_alignment_for_contiguous_layout", "dg_set_num_sms", "dg_get_num_sms", "dg_get_device_status",
    "dg_last_error_string", "dg_query_config", "dg_fp8_gemm_nt_noalloc", "dg_set_tail_splits",
    "dg_set_cluster_split", "dg_set_wait_limit_us", "dg_set_pair_b", "dg_set_pdl", "dg_get_pdl",
    "dg_transform_sf_into_ue8m0_a", "dg_transform_sf_into_ue8m0_b", "dg_transform_sf_a_into_mn_major",
    "dg_fp8_gemm_nt_ue8m0", "dg_fp8_gemm_nt_ue8m0_f32", "dg_fp8_grouped_contiguous_ue8m0",
    "dg_fp8_grouped_contiguous_ue8m0_f32", "dg_fp8_grouped_masked_ue8m0", "dg_fp8_grouped_masked_ue8m0_f32",
    "dg_query_config_ue8m0", "dg_fp8_gemm_nt_acc_f32", "dg_fp8_gemm_nt_ue8m0_acc_f32",
    "dg_fp8_grouped_masked_swiglu", "dg_fp8_grouped_masked_swiglu_f32", "dg_fp8_grouped_masked_swiglu_fp8",
    "dg_fp8_grouped_masked_swiglu_ue8m0",
    "dg_fp8_grouped_masked_swiglu_ue8m0_f32", "dg_fp8_gemm_nn", "dg_fp8_gemm_nn_f32",
    "dg_fp8_gemm_tn", "dg_fp8_gemm_tn_f32", "dg_fp8_gemm_tt", "dg_fp8_gemm_tt_f32",
    "dg_fp8_gemm_nn_ue8m0", "dg_fp8_gemm_nn_ue8m0_f32", "dg_fp8_gemm_tn_ue8m0", "dg_fp8_gemm_tn_ue8m0_f32", "dg_fp8_gemm_tt_ue8m0", "dg_fp8_gemm_tt_ue8m0_f32",
    "dg_fp8_k_grouped_gemm_tn_contiguous", "dg_fp8_k_grouped_gemm_tn_contiguous_f32",
    "dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0", "dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0_f32",
)


class DGError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libdg status {status}: {msg}")
        self.status = status


_lib = None


def load(build_if_missing: bool = True):
    """Loads libdg.so (building it first if it is missing or stale and nvcc is available)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build_mod.LIB
    if build_if_missing and not _build_mod.up_to_date():
        _build_mod.build()
    if not os.path.exists(path):
        raise DGError(DG_ERR_UNSUPPORTED, f"libdg.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, i32 = ctypes.c_void_p, ctypes.c_int
    for name in ("dg_fp8_gemm_nt", "dg_fp8_gemm_nt_f32", "dg_fp8_gemm_nt_noalloc", "dg_fp8_gemm_nt_ue8m0",
                 "dg_fp8_gemm_nt_ue8m0_f32", "dg_fp8_gemm_nn", "dg_fp8_gemm_nn_f32", "dg_fp8_gemm_tn",
                 "dg_fp8_gemm_tn_f32", "dg_fp8_gemm_tt", "dg_fp8_gemm_tt_f32", "dg_fp8_gemm_nn_ue8m0", "dg_fp8_gemm_nn_ue8m0_f32", "dg_fp8_gemm_tn_ue8m0", "dg_fp8_gemm_tn_ue8m0_f32", "dg_fp8_gemm_tt_ue8m0", "dg_fp8_gemm_tt_ue8m0_f32"):
        f = getattr(lib, name)
        f.restype, f.argtypes = i32, [P, P, P, P, P, i32, i32, i32, P]
    for name in ("dg_fp8_grouped_contiguous", "dg_fp8_grouped_contiguous_f32", "dg_fp8_grouped_contiguous_ue8m0",
                 "dg_fp8_grouped_contiguous_ue8m0_f32"):
        f = getattr(lib, name)
        f.restype, f.argtypes = i32, [P, P, P, P, P, P, i32, i32, i32, i32, P]
    for name in ("dg_fp8_grouped_masked", "dg_fp8_grouped_masked_f32", "dg_fp8_grouped_masked_ue8m0",
                 "dg_fp8_grouped_masked_ue8m0_f32", "dg_fp8_grouped_masked_swiglu",
                 "dg_fp8_grouped_masked_swiglu_f32", "dg_fp8_grouped_masked_swiglu_ue8m0",
                 "dg_fp8_grouped_masked_swiglu_ue8m0_f32"):
        f = getattr(lib, name)
        f.restype, f.argtypes = i32, [P, P, P, P, P, P, i32, i32, i32, i32, P]
    lib.dg_fp8_grouped_masked_swiglu_fp8.restype = i32
    lib.dg_fp8_grouped_masked_swiglu_fp8.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, P]
    lib.dg_get_tma_aligned_size.restype, lib.dg_get_tma_aligned_size.argtypes = i32, [i32, i32]
    lib.dg_get_mk_alignment_for_contiguous_layout.restype = i32
    lib.dg_get_mk_alignment_for_contiguous_layout.argtypes = []
    lib.dg_set_num_sms.restype, lib.dg_set_num_sms.argtypes = None, [i32]
    lib.dg_get_num_sms.restype, lib.dg_get_num_sms.argtypes = i32, []
    lib.dg_set_tail_splits.restype, lib.dg_set_tail_splits.argtypes = i32, [i32]
    lib.dg_set_cluster_split.restype, lib.dg_set_cluster_split.argtypes = i32, [i32]
    lib.dg_set_pair_b.restype, lib.dg_set_pair_b.argtypes = i32, [i32]
    lib.dg_set_pdl.restype, lib.dg_set_pdl.argtypes = i32, [i32]
    lib.dg_get_pdl.restype, lib.dg_get_pdl.argtypes = i32, []
    for name in ("dg_transform_sf_into_ue8m0_a", "dg_transform_sf_into_ue8m0_b", "dg_transform_sf_a_into_mn_major"):
        f = getattr(lib, name)
        f.restype, f.argtypes = i32, [P, P, i32, i32, i32, P]
    lib.dg_set_wait_limit_us.restype, lib.dg_set_wait_limit_us.argtypes = ctypes.c_longlong, [ctypes.c_longlong]
    lib.dg_get_device_status.restype, lib.dg_get_device_status.argtypes = i32, [ctypes.POINTER(i32), P]
    lib.dg_last_error_string.restype, lib.dg_last_error_string.argtypes = ctypes.c_char_p, []
    for name in ("dg_fp8_gemm_nt_acc_f32", "dg_fp8_gemm_nt_ue8m0_acc_f32"):
        f = getattr(lib, name)
        f.restype, f.argtypes = i32, [P, P, P, P, P, P, i32, i32, i32, P]
    for name in ("dg_fp8_k_grouped_gemm_tn_contiguous", "dg_fp8_k_grouped_gemm_tn_contiguous_f32",
                 "dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0", "dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0_f32"):
        f = getattr(lib, name)
        f.restype, f.argtypes = i32, [P, P, P, P, P, P, i32, i32, i32, i32, P]
    for name in ("dg_query_config", "dg_query_config_ue8m0"):
        f = getattr(lib, name)
        f.restype, f.argtypes = i32, [i32, i32, i32, i32, i32, i32, ctypes.POINTER(i32)]
    _lib = lib
    return lib


def _check(status: int):
    if status != DG_OK:
        raise DGError(status, load().dg_last_error_string().decode(errors="replace"))


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t, name, dtypes):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _shape(t, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    return tuple(int(x) for x in t.shape)


def _expect(t, name, shape):
    """Raises ValueError unless tensor `t` has exactly `shape` (checked before any pointer is taken,
    so that a mis-shaped call never reaches a kernel, whose TMA boxes would read out of bounds)."""
    got = _shape(t, name)
    if got != tuple(shape):
        raise ValueError(f"{name} has shape {list(got)}, expected {list(shape)}")


def _cdiv(a, b):
    return -(-a // b)


def _align4(x):
    return -(-x // 4) * 4


def _scale_k(name, K):
    """Scale entries along K: one per 128-deep K-block (FP32 scales), or one int32 word per four
    K-blocks (packed UE8M0)."""
    nkb = _cdiv(K, 128)
    return _cdiv(nkb, 4) if "_ue8m0" in name else nkb


def _fp8_types():
    import torch
    return (torch.uint8, torch.float8_e4m3fn)


def _f32():
    import torch
    return (torch.float32,)


def _scale_types(name):
    import torch
    return (torch.int32,) if "_ue8m0" in name else (torch.float32,)


def _d_types(f32: bool):
    import torch
    return (torch.float32,) if f32 else (torch.bfloat16, torch.int16, torch.uint16)


def _dense_shapes(name, A, B):
    """(M, N, K) of a dense call: A [M, K], B [N, K] (or [1, N, K])."""
    a, b = _shape(A, "A"), _shape(B, "B")
    if len(a) != 2:
        raise ValueError(f"A must be [M, K], got {list(a)}")
    if not (len(b) == 2 or (len(b) == 3 and b[0] == 1)):
        raise ValueError(f"B must be [N, K] (or [1, N, K]), got {list(b)}")
    M, K = a
    N = b[-2]
    if b[-1] != K:
        raise ValueError(f"B has K = {b[-1]}, A has K = {K}")
    return M, N, K


def _check_scales_2d(name, sA, sB, M, N, K):
    nks = _scale_k(name, K)
    _expect(sA, "sA", (nks, _align4(M)))
    sb = _shape(sB, "sB")
    want = (_cdiv(N, 128), nks)
    if sb != want and sb != (1,) + want:
        raise ValueError(f"sB has shape {list(sb)}, expected {list(want)}")


def _dense(name, f32, A, sA, B, sB, D, stream):
    M, N, K = _dense_shapes(name, A, B)
    _check_scales_2d(name, sA, sB, M, N, K)
    _expect(D, "D", (M, N))
    lib = load()
    _check(getattr(lib, name)(_ptr(A, "A", _fp8_types()), _ptr(sA, "sA", _scale_types(name)), _ptr(B, "B", _fp8_types()),
                              _ptr(sB, "sB", _scale_types(name)), _ptr(D, "D", _d_types(f32)), M, N, K, _stream(stream)))
    return D


def dg_fp8_gemm_nt(A, sA, B, sB, D, stream=None):
    """D[M,N] (bfloat16) = A[M,K]·B[N,K]ᵀ with fine-grained scales."""
    return _dense("dg_fp8_gemm_nt", False, A, sA, B, sB, D, stream)


def dg_fp8_gemm_nt_f32(A, sA, B, sB, D, stream=None):
    """As dg_fp8_gemm_nt, storing the FP32 accumulator."""
    return _dense("dg_fp8_gemm_nt_f32", True, A, sA, B, sB, D, stream)


def dg_fp8_gemm_nt_noalloc(A, sA, B, sB, D, stream=None):
    """As dg_fp8_gemm_nt, without any allocation: for callers that cannot let the library call
    cudaMalloc (a framework whose caching allocator owns device memory, a serving loop that must not
    block on cudaMalloc's synchronisation). Split-K scratch comes from a fixed 20 MiB array inside
    libdg shared by all calls on a device, so calls that overlap on the GPU race; a shape that needs
    more scratch raises DGError(DG_ERR_UNSUPPORTED). The first call on a device looks up the array's
    address; make it before any stream capture."""
    return _dense("dg_fp8_gemm_nt_noalloc", False, A, sA, B, sB, D, stream)


def _contig(name, f32, A, sA, B, sB, m_indices, D, stream):
    import torch
    a, b = _shape(A, "A"), _shape(B, "B")
    if len(a) != 2 or len(b) != 3:
        raise ValueError(f"contiguous layout: A must be [M_total, K] and B [G, N, K], got {list(a)} and {list(b)}")
    M, K = a
    G, N = b[0], b[1]
    if b[2] != K:
        raise ValueError(f"B has K = {b[2]}, A has K = {K}")
    nks = _scale_k(name, K)
    _expect(sA, "sA", (nks, _align4(M)))
    _expect(sB, "sB", (G, _cdiv(N, 128), nks))
    _expect(m_indices, "m_indices", (M,))
    _expect(D, "D", (M, N))
    lib = load()
    _check(getattr(lib, name)(_ptr(A, "A", _fp8_types()), _ptr(sA, "sA", _scale_types(name)), _ptr(B, "B", _fp8_types()),
                              _ptr(sB, "sB", _scale_types(name)), _ptr(m_indices, "m_indices", (torch.int32,)),
                              _ptr(D, "D", _d_types(f32)), M, N, K, G, _stream(stream)))
    return D


def dg_fp8_grouped_contiguous(A, sA, B, sB, m_indices, D, stream=None):
    """Contiguous-layout grouped GEMM: row m of D uses expert m_indices[m] (-1: padding, untouched)."""
    return _contig("dg_fp8_grouped_contiguous", False, A, sA, B, sB, m_indices, D, stream)


def dg_fp8_grouped_contiguous_f32(A, sA, B, sB, m_indices, D, stream=None):
    return _contig("dg_fp8_grouped_contiguous_f32", True, A, sA, B, sB, m_indices, D, stream)


def _masked(name, f32, A, sA, B, sB, masked_m, D, stream):
    import torch
    a, b = _shape(A, "A"), _shape(B, "B")
    if len(a) != 3 or len(b) != 3:
        raise ValueError(f"masked layout: A must be [G, M_max, K] and B [G, N, K], got {list(a)} and {list(b)}")
    G, M_max, K = a
    N = b[1]
    if b[0] != G or b[2] != K:
        raise ValueError(f"B has shape {list(b)}, expected [{G}, N, {K}]")
    nks = _scale_k(name, K)
    _expect(sA, "sA", (G, nks, _align4(M_max)))
    _expect(sB, "sB", (G, _cdiv(N, 128), nks))
    _expect(masked_m, "masked_m", (G,))
    # the fused SwiGLU writes H = silu(gate)·up, half as wide as B's 2I rows
    _expect(D, "H" if "swiglu" in name else "D", (G, M_max, N // 2 if "swiglu" in name else N))
    lib = load()
    _check(getattr(lib, name)(_ptr(A, "A", _fp8_types()), _ptr(sA, "sA", _scale_types(name)), _ptr(B, "B", _fp8_types()),
                              _ptr(sB, "sB", _scale_types(name)), _ptr(masked_m, "masked_m", (torch.int32,)),
                              _ptr(D, "D", _d_types(f32)), G, M_max, N, K, _stream(stream)))
    return D


def dg_fp8_grouped_masked(A, sA, B, sB, masked_m, D, stream=None):
    """Masked-layout grouped GEMM: rows m < masked_m[g] of group g are computed, the rest untouched."""
    return _masked("dg_fp8_grouped_masked", False, A, sA, B, sB, masked_m, D, stream)


def dg_fp8_grouped_masked_f32(A, sA, B, sB, masked_m, D, stream=None):
    return _masked("dg_fp8_grouped_masked_f32", True, A, sA, B, sB, masked_m, D, stream)


def _dense_acc(name, A, sA, B, sB, C, D, stream):
    M, N, K = _dense_shapes(name, A, B)
    _check_scales_2d(name, sA, sB, M, N, K)
    _expect(C, "C", (M, N))
    _expect(D, "D", (M, N))
    lib = load()
    _check(getattr(lib, name)(_ptr(A, "A", _fp8_types()), _ptr(sA, "sA", _scale_types(name)),
                              _ptr(B, "B", _fp8_types()), _ptr(sB, "sB", _scale_types(name)), _ptr(C, "C", _f32()),
                              _ptr(D, "D", _f32()), M, N, K, _stream(stream)))
    return D


def dg_fp8_gemm_nt_acc_f32(A, sA, B, sB, C, D, stream=None):
    """D (float32) = C + A·Bᵀ; C (float32 [M,N]) may be D itself."""
    return _dense_acc("dg_fp8_gemm_nt_acc_f32", A, sA, B, sB, C, D, stream)


def dg_fp8_gemm_nt_ue8m0_acc_f32(A, sA, B, sB, C, D, stream=None):
    """As dg_fp8_gemm_nt_acc_f32 with packed UE8M0 scales."""
    return _dense_acc("dg_fp8_gemm_nt_ue8m0_acc_f32", A, sA, B, sB, C, D, stream)


# The layouts' names: the first letter says how A is stored (n: [M, K], t: [K, M]), the second how
# B is stored (t: [N, K], n: [K, N]).
_LAYOUTS = {"nn": (False, True), "tn": (True, True), "tt": (True, False)}


def _dense_layout(name, f32, A, sA, B, sB, D, M, N, K, stream):
    a_t, b_n = _LAYOUTS[name[len("dg_fp8_gemm_"):len("dg_fp8_gemm_") + 2]]
    M, N, K = int(M), int(N), int(K)
    nks = _scale_k(name, K)
    _expect(A, "A", (K, M) if a_t else (M, K))
    _expect(B, "B", (K, N) if b_n else (N, K))
    _expect(sA, "sA", (nks, _align4(M)))
    _expect(sB, "sB", (_cdiv(N, 128), nks))
    _expect(D, "D", (M, N))
    lib = load()
    st = _scale_types(name)
    _check(getattr(lib, name)(_ptr(A, "A", _fp8_types()), _ptr(sA, "sA", st), _ptr(B, "B", _fp8_types()),
                              _ptr(sB, "sB", st), _ptr(D, "D", _d_types(f32)), M, N, K, _stream(stream)))
    return D


def dg_fp8_gemm_nn(A, sA, B, sB, D, M, N, K, stream=None):
    """D[M,N] = A·Bᵀ with A stored [M,K] and B stored [K,N] (N contiguous)."""
    return _dense_layout("dg_fp8_gemm_nn", False, A, sA, B, sB, D, M, N, K, stream)


def dg_fp8_gemm_nn_f32(A, sA, B, sB, D, M, N, K, stream=None):
    return _dense_layout("dg_fp8_gemm_nn_f32", True, A, sA, B, sB, D, M, N, K, stream)


def dg_fp8_gemm_tn(A, sA, B, sB, D, M, N, K, stream=None):
    """D[M,N] = A·Bᵀ with A stored [K,M] and B stored [K,N] (both M/N contiguous)."""
    return _dense_layout("dg_fp8_gemm_tn", False, A, sA, B, sB, D, M, N, K, stream)


def dg_fp8_gemm_tn_f32(A, sA, B, sB, D, M, N, K, stream=None):
    return _dense_layout("dg_fp8_gemm_tn_f32", True, A, sA, B, sB, D, M, N, K, stream)


def dg_fp8_gemm_tt(A, sA, B, sB, D, M, N, K, stream=None):
    """D[M,N] = A·Bᵀ with A stored [K,M] and B stored [N,K]."""
    return _dense_layout("dg_fp8_gemm_tt", False, A, sA, B, sB, D, M, N, K, stream)


def dg_fp8_gemm_tt_f32(A, sA, B, sB, D, M, N, K, stream=None):
    return _dense_layout("dg_fp8_gemm_tt_f32", True, A, sA, B, sB, D, M, N, K, stream)


def dg_fp8_gemm_nn_ue8m0(A, sA, B, sB, D, M, N, K, stream=None):
    """dg_fp8_gemm_nn with packed UE8M0 scales (sA [ceil(nkb/4), align4(M)], sB [ceil(N/128), ceil(nkb/4)] int32)."""
    return _dense_layout("dg_fp8_gemm_nn_ue8m0", False, A, sA, B, sB, D, M, N, K, stream)


def dg_fp8_gemm_nn_ue8m0_f32(A, sA, B, sB, D, M, N, K, stream=None):
    return _dense_layout("dg_fp8_gemm_nn_ue8m0_f32", True, A, sA, B, sB, D, M, N, K, stream)


def dg_fp8_gemm_tn_ue8m0(A, sA, B, sB, D, M, N, K, stream=None):
    """dg_fp8_gemm_tn with packed UE8M0 scales."""
    return _dense_layout("dg_fp8_gemm_tn_ue8m0", False, A, sA, B, sB, D, M, N, K, stream)


def dg_fp8_gemm_tn_ue8m0_f32(A, sA, B, sB, D, M, N, K, stream=None):
    return _dense_layout("dg_fp8_gemm_tn_ue8m0_f32", True, A, sA, B, sB, D, M, N, K, stream)


def dg_fp8_gemm_tt_ue8m0(A, sA, B, sB, D, M, N, K, stream=None):
    """dg_fp8_gemm_tt with packed UE8M0 scales."""
    return _dense_layout("dg_fp8_gemm_tt_ue8m0", False, A, sA, B, sB, D, M, N, K, stream)


def dg_fp8_gemm_tt_ue8m0_f32(A, sA, B, sB, D, M, N, K, stream=None):
    return _dense_layout("dg_fp8_gemm_tt_ue8m0_f32", True, A, sA, B, sB, D, M, N, K, stream)


def _k_grouped(name, f32, A, sA, B, sB, k_offsets, D, stream):
    import torch
    a, b, o = _shape(A, "A"), _shape(B, "B"), _shape(k_offsets, "k_offsets")
    if len(a) != 2 or len(b) != 2 or len(o) != 1 or o[0] < 1:
        raise ValueError(f"K-grouped: A must be [K_total, M], B [K_total, N], k_offsets [G + 1]; got "
                         f"{list(a)}, {list(b)}, {list(o)}")
    K_total, M = a
    N = b[1]
    G = o[0] - 1
    if b[0] != K_total:
        raise ValueError(f"B has K_total = {b[0]}, A has K_total = {K_total}")
    nks = _scale_k(name, K_total)
    _expect(sA, "sA", (nks, _align4(M)))
    _expect(sB, "sB", (_cdiv(N, 128), nks))
    _expect(D, "D", (G, M, N))
    lib = load()
    st = _scale_types(name)
    _check(getattr(lib, name)(_ptr(A, "A", _fp8_types()), _ptr(sA, "sA", st), _ptr(B, "B", _fp8_types()),
                              _ptr(sB, "sB", st), _ptr(k_offsets, "k_offsets", (torch.int32,)),
                              _ptr(D, "D", _d_types(f32)), G, M, N, K_total, _stream(stream)))
    return D


def dg_fp8_k_grouped_gemm_tn_contiguous(A, sA, B, sB, k_offsets, D, stream=None):
    """Groups along K: A [K_total, M], B [K_total, N], k_offsets [G+1] int32 (multiples of 128),
    D [G, M, N] (bfloat16) = Σ over each group's K range."""
    return _k_grouped("dg_fp8_k_grouped_gemm_tn_contiguous", False, A, sA, B, sB, k_offsets, D, stream)


def dg_fp8_k_grouped_gemm_tn_contiguous_f32(A, sA, B, sB, k_offsets, D, stream=None):
    return _k_grouped("dg_fp8_k_grouped_gemm_tn_contiguous_f32", True, A, sA, B, sB, k_offsets, D, stream)


def dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0(A, sA, B, sB, k_offsets, D, stream=None):
    """The K-grouped GEMM with packed UE8M0 scales: sA [ceil(K_total/512), align4(M)], sB
    [ceil(N/128), ceil(K_total/512)] int32 (four K-blocks per word along K_total)."""
    return _k_grouped("dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0", False, A, sA, B, sB, k_offsets, D, stream)


def dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0_f32(A, sA, B, sB, k_offsets, D, stream=None):
    return _k_grouped("dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0_f32", True, A, sA, B, sB, k_offsets, D, stream)


def dg_fp8_grouped_masked_swiglu(A, sA, B, sB, masked_m, H, stream=None):
    """Masked grouped GEMM fused with SwiGLU: B [G, 2I, K] (gate rows, then up rows),
    H [G, M_max, I] = silu(gate)·up over the rows m < masked_m[g]; other rows untouched."""
    return _masked("dg_fp8_grouped_masked_swiglu", False, A, sA, B, sB, masked_m, H, stream)


def dg_fp8_grouped_masked_swiglu_f32(A, sA, B, sB, masked_m, H, stream=None):
    return _masked("dg_fp8_grouped_masked_swiglu_f32", True, A, sA, B, sB, masked_m, H, stream)


def dg_fp8_grouped_masked_swiglu_fp8(A, sA, B, sB, masked_m, Hq, sH, stream=None):
    """The fused SwiGLU with H cast to FP8 for the down projection: Hq [G, M_max, I] E4M3 codes
    (uint8 or float8_e4m3fn), e4m3_rne(H · (448/amax)), and sH [G, I/128, align4(M_max)] float32, the
    dequantisation scale amax/448 of each 1x128 group of each valid row; the A and sA layouts of
    dg_fp8_grouped_masked. Rows past masked_m are
    untouched in both."""
    import torch
    a, b = _shape(A, "A"), _shape(B, "B")
    if len(a) != 3 or len(b) != 3:
        raise ValueError(f"masked layout: A must be [G, M_max, K] and B [G, 2I, K], got {list(a)} and {list(b)}")
    G, M_max, K = a
    N = b[1]
    if b[0] != G or b[2] != K:
        raise ValueError(f"B has shape {list(b)}, expected [{G}, 2I, {K}]")
    nkb = _cdiv(K, 128)
    _expect(sA, "sA", (G, nkb, _align4(M_max)))
    _expect(sB, "sB", (G, _cdiv(N, 128), nkb))
    _expect(masked_m, "masked_m", (G,))
    _expect(Hq, "Hq", (G, M_max, N // 2))
    _expect(sH, "sH", (G, (N // 2) // 128, _align4(M_max)))
    lib = load()
    _check(lib.dg_fp8_grouped_masked_swiglu_fp8(
        _ptr(A, "A", _fp8_types()), _ptr(sA, "sA", _f32()), _ptr(B, "B", _fp8_types()), _ptr(sB, "sB", _f32()),
        _ptr(masked_m, "masked_m", (torch.int32,)), _ptr(Hq, "Hq", _fp8_types()), _ptr(sH, "sH", _f32()),
        G, M_max, N, K, _stream(stream)))
    return Hq, sH


def dg_fp8_grouped_masked_swiglu_ue8m0(A, sA, B, sB, masked_m, H, stream=None):
    """The fused SwiGLU with packed UE8M0 scales (int32 words, four K-groups each)."""
    return _masked("dg_fp8_grouped_masked_swiglu_ue8m0", False, A, sA, B, sB, masked_m, H, stream)


def dg_fp8_grouped_masked_swiglu_ue8m0_f32(A, sA, B, sB, masked_m, H, stream=None):
    return _masked("dg_fp8_grouped_masked_swiglu_ue8m0_f32", True, A, sA, B, sB, masked_m, H, stream)


def dg_transform_sf_into_ue8m0_a(sA, sA_packed, M, K, stream=None):
    """A's FP32 scales sA [ceil(K/128), align4(M)] (or [G, ...]; powers of two, zero for padding rows)
    -> packed UE8M0 words sA_packed [ceil(ceil(K/128)/4), align4(M)] (or [G, ...]) int32, on the GPU.
    A value that is not a power of two sets DG_DEV_BAD_SCALE (dg_get_device_status)."""
    import torch
    s = _shape(sA, "sA")
    if len(s) not in (2, 3):
        raise ValueError(f"sA must be [ceil(K/128), align4(M)] or [G, ceil(K/128), align4(M)], got {list(s)}")
    G = s[0] if len(s) == 3 else 1
    nkb, ldsa = -(-K // 128), dg_get_tma_aligned_size(M, 4)
    _expect(sA, "sA", s[:-2] + (nkb, ldsa))
    _expect(sA_packed, "sA_packed", s[:-2] + (-(-nkb // 4), ldsa))
    _check(load().dg_transform_sf_into_ue8m0_a(_ptr(sA, "sA", (torch.float32,)),
                                               _ptr(sA_packed, "sA_packed", (torch.int32,)), G, M, K, _stream(stream)))


def dg_transform_sf_a_into_mn_major(sA_rows, sA, M, K, stream=None):
    """A's FP32 scales row-major sA_rows [M, ceil(K/128)] (or [G, M, ceil(K/128)]) -> the MN-major
    layout of every call, sA [ceil(K/128), align4(M)] (or [G, ...]), padding rows zero, on the GPU."""
    import torch
    s = _shape(sA_rows, "sA_rows")
    if len(s) not in (2, 3):
        raise ValueError(f"sA_rows must be [M, ceil(K/128)] or [G, M, ceil(K/128)], got {list(s)}")
    G = s[0] if len(s) == 3 else 1
    nkb = -(-K // 128)
    _expect(sA_rows, "sA_rows", s[:-2] + (M, nkb))
    _expect(sA, "sA", s[:-2] + (nkb, dg_get_tma_aligned_size(M, 4)))
    _check(load().dg_transform_sf_a_into_mn_major(_ptr(sA_rows, "sA_rows", (torch.float32,)),
                                                  _ptr(sA, "sA", (torch.float32,)), G, M, K, _stream(stream)))


def dg_transform_sf_into_ue8m0_b(sB, sB_packed, N, K, stream=None):
    """B's FP32 scales sB [ceil(N/128), ceil(K/128)] (or [G, ...]; powers of two) -> packed UE8M0 words
    sB_packed [ceil(N/128), ceil(ceil(K/128)/4)] (or [G, ...]) int32, on the GPU. A value that is not a
    power of two sets DG_DEV_BAD_SCALE (dg_get_device_status)."""
    import torch
    s = _shape(sB, "sB")
    if len(s) not in (2, 3):
        raise ValueError(f"sB must be [ceil(N/128), ceil(K/128)] or [G, ceil(N/128), ceil(K/128)], got {list(s)}")
    G = s[0] if len(s) == 3 else 1
    nnb, nkb = -(-N // 128), -(-K // 128)
    _expect(sB, "sB", s[:-2] + (nnb, nkb))
    _expect(sB_packed, "sB_packed", s[:-2] + (nnb, -(-nkb // 4)))
    _check(load().dg_transform_sf_into_ue8m0_b(_ptr(sB, "sB", (torch.float32,)),
                                               _ptr(sB_packed, "sB_packed", (torch.int32,)), G, N, K, _stream(stream)))


def dg_fp8_gemm_nt_ue8m0(A, sA, B, sB, D, stream=None):
    """Dense D (bfloat16) with power-of-two scales given as packed UE8M0 int32 words."""
    return _dense("dg_fp8_gemm_nt_ue8m0", False, A, sA, B, sB, D, stream)


def dg_fp8_gemm_nt_ue8m0_f32(A, sA, B, sB, D, stream=None):
    return _dense("dg_fp8_gemm_nt_ue8m0_f32", True, A, sA, B, sB, D, stream)


def dg_fp8_grouped_contiguous_ue8m0(A, sA, B, sB, m_indices, D, stream=None):
    return _contig("dg_fp8_grouped_contiguous_ue8m0", False, A, sA, B, sB, m_indices, D, stream)


def dg_fp8_grouped_contiguous_ue8m0_f32(A, sA, B, sB, m_indices, D, stream=None):
    return _contig("dg_fp8_grouped_contiguous_ue8m0_f32", True, A, sA, B, sB, m_indices, D, stream)


def dg_fp8_grouped_masked_ue8m0(A, sA, B, sB, masked_m, D, stream=None):
    return _masked("dg_fp8_grouped_masked_ue8m0", False, A, sA, B, sB, masked_m, D, stream)


def dg_fp8_grouped_masked_ue8m0_f32(A, sA, B, sB, masked_m, D, stream=None):
    return _masked("dg_fp8_grouped_masked_ue8m0_f32", True, A, sA, B, sB, masked_m, D, stream)


def dg_get_tma_aligned_size(x: int, elem_bytes: int) -> int:
    return int(load().dg_get_tma_aligned_size(x, elem_bytes))


def dg_get_mk_alignment_for_contiguous_layout() -> int:
    return int(load().dg_get_mk_alignment_for_contiguous_layout())


def dg_set_num_sms(n: int) -> None:
    load().dg_set_num_sms(int(n))


def dg_get_num_sms() -> int:
    return int(load().dg_get_num_sms())


def dg_set_cluster_split(on: bool) -> bool:
    """Allow (default) or forbid split-K inside thread-block clusters. Returns the previous value."""
    return bool(load().dg_set_cluster_split(1 if on else 0))


def dg_set_wait_limit_us(us: int) -> int:
    """Time limit of the kernels' pipeline waits in microseconds (default 2 s; < 0 restores it; 0 makes
    every wait that is not already satisfied give up, which exercises the timeout path). A launch that
    gives up sets DG_DEV_TIMEOUT; its output is undefined. Returns the previous value."""
    return int(load().dg_set_wait_limit_us(int(us)))


def dg_set_pair_b(on: bool) -> bool:
    """Allow or forbid (default) pairs of CTAs that share B tiles through TMA multicast. Returns the
    previous value; results are bit-identical either way."""
    return bool(load().dg_set_pair_b(1 if on else 0))


def dg_set_pdl(on: bool) -> bool:
    """Launch every GEMM with programmatic dependent launch (it may start before the previous kernel
    in the stream ends, and waits for that kernel's results before reading its inputs), or not (the
    default). Returns the previous value; results are bit-identical either way."""
    return bool(load().dg_set_pdl(1 if on else 0))


def dg_get_pdl() -> bool:
    return bool(load().dg_get_pdl())


def dg_set_tail_splits(n: int) -> int:
    """Most K ranges a tile of a last, partial wave may be cut into (1: off; <= 0: default 4).
    Returns the previous value."""
    return int(load().dg_set_tail_splits(int(n)))


def dg_get_device_status(stream=None) -> int:
    """Synchronises `stream`, reads and clears the device status word; returns its DG_DEV_* bits."""
    code = ctypes.c_int(0)
    st = load().dg_get_device_status(ctypes.byref(code), _stream(stream))
    if st not in (DG_OK, DG_ERR_DEVICE_STATUS):
        _check(st)
    return int(code.value)


def dg_last_error_string() -> str:
    return load().dg_last_error_string().decode(errors="replace")


def dg_query_config(mode: int, M: int, N: int, K: int, G: int = 1, out_f32: bool = False) -> dict:
    """Tile configuration a call would launch: mode 0 dense, 1 contiguous, 2 masked."""
    cfg = (ctypes.c_int * 6)()
    _check(load().dg_query_config(mode, M, N, K, G, 1 if out_f32 else 0, cfg))
    keys = ("block_m", "block_n", "stages", "splits", "grid", "tiles")
    return dict(zip(keys, [int(v) for v in cfg]))


def dg_query_config_ue8m0(mode: int, M: int, N: int, K: int, G: int = 1, out_f32: bool = False) -> dict:
    """Tile configuration of the packed-UE8M0 (block-scaled) calls."""
    cfg = (ctypes.c_int * 6)()
    _check(load().dg_query_config_ue8m0(mode, M, N, K, G, 1 if out_f32 else 0, cfg))
    keys = ("block_m", "block_n", "stages", "splits", "grid", "tiles")
    return dict(zip(keys, [int(v) for v in cfg]))
