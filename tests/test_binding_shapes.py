"""The Python binding checks every tensor's shape against the documented layouts before it takes a
pointer, so that a mis-shaped call is refused on the host instead of sending a kernel's TMA boxes
out of bounds. CPU tensors suffice: a well-shaped call gets past every shape check and stops only at
the "must be a CUDA tensor" check, and a mis-shaped one fails earlier with a shape message."""
import pytest
import torch

import moe_grouped_gemm_e4m3_gb300 as dg

SHAPE_ERR = r"shape|expected|must be \[|has K"
CUDA_ERR = r"CUDA tensor"


def cdiv(a, b):
    return -(-a // b)


def a4(x):
    return -(-x // 4) * 4


def u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8)


def f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def _refused(fn, args, i, bad):
    """Calls fn with argument i replaced by `bad`; the binding must refuse the shape."""
    a = list(args)
    a[i] = bad
    with pytest.raises(ValueError, match=SHAPE_ERR):
        fn(*a)


def _accepted(fn, args):
    with pytest.raises(ValueError, match=CUDA_ERR):
        fn(*args)


M, N, K, G = 198, 392, 1152, 3          # ragged M/N tails (M not a multiple of 4); K = 9 K-blocks
NKB, NNB = cdiv(K, 128), cdiv(N, 128)


def test_dense_shapes():
    args = [u8(M, K), f32(NKB, a4(M)), u8(N, K), f32(NNB, NKB), bf16(M, N)]
    for fn in (dg.dg_fp8_gemm_nt, dg.dg_fp8_gemm_nt_noalloc):
        _accepted(fn, args)
        _refused(fn, args, 0, u8(M, K + 16))            # A's K differs from B's
        _refused(fn, args, 0, u8(M * K))                # A not 2-D
        _refused(fn, args, 1, f32(NKB, M))              # sA rows not padded to 4
        _refused(fn, args, 1, f32(NKB + 1, a4(M)))      # sA K-blocks
        _refused(fn, args, 2, u8(N, K - 16))            # B's K
        _refused(fn, args, 2, u8(2, N, K))              # B with G != 1
        _refused(fn, args, 3, f32(NNB + 1, NKB))        # sB N-blocks
        _refused(fn, args, 3, f32(NNB, NKB - 1))        # sB K-blocks
        _refused(fn, args, 4, bf16(M, N + 8))           # D columns
        _refused(fn, args, 4, bf16(M + 1, N))           # D rows
    f32_args = args[:4] + [f32(M, N)]
    _accepted(dg.dg_fp8_gemm_nt_f32, f32_args)
    _refused(dg.dg_fp8_gemm_nt_f32, f32_args, 4, f32(N, M))


def test_dense_ue8m0_shapes():
    nkq = cdiv(NKB, 4)
    args = [u8(M, K), i32(nkq, a4(M)), u8(N, K), i32(NNB, nkq), bf16(M, N)]
    _accepted(dg.dg_fp8_gemm_nt_ue8m0, args)
    _refused(dg.dg_fp8_gemm_nt_ue8m0, args, 1, i32(NKB, a4(M)))     # FP32-scale layout to the packed call
    _refused(dg.dg_fp8_gemm_nt_ue8m0, args, 3, i32(NNB, NKB))


def test_accumulating_shapes():
    args = [u8(M, K), f32(NKB, a4(M)), u8(N, K), f32(NNB, NKB), f32(M, N), f32(M, N)]
    _accepted(dg.dg_fp8_gemm_nt_acc_f32, args)
    _refused(dg.dg_fp8_gemm_nt_acc_f32, args, 4, f32(M, N - 4))     # C
    _refused(dg.dg_fp8_gemm_nt_acc_f32, args, 5, f32(M - 1, N))     # D
    _refused(dg.dg_fp8_gemm_nt_acc_f32, args, 2, u8(N, K + 128))


def test_contiguous_shapes():
    MT = 384
    args = [u8(MT, K), f32(NKB, a4(MT)), u8(G, N, K), f32(G, NNB, NKB), i32(MT), bf16(MT, N)]
    fn = dg.dg_fp8_grouped_contiguous
    _accepted(fn, args)
    _refused(fn, args, 0, u8(MT, K - 16))
    _refused(fn, args, 1, f32(NKB, MT + 4))
    _refused(fn, args, 2, u8(N, K))                     # B without the group axis
    _refused(fn, args, 2, u8(G, N, K + 16))
    _refused(fn, args, 3, f32(G + 1, NNB, NKB))
    _refused(fn, args, 4, i32(MT - 1))                  # m_indices length
    _refused(fn, args, 5, bf16(MT, N - 8))
    _accepted(dg.dg_fp8_grouped_contiguous_f32, args[:5] + [f32(MT, N)])


def test_masked_shapes():
    MM = 256
    args = [u8(G, MM, K), f32(G, NKB, a4(MM)), u8(G, N, K), f32(G, NNB, NKB), i32(G), bf16(G, MM, N)]
    fn = dg.dg_fp8_grouped_masked
    _accepted(fn, args)
    _refused(fn, args, 0, u8(MM, K))                    # A without the group axis
    _refused(fn, args, 1, f32(NKB, a4(MM)))             # sA without the group axis
    _refused(fn, args, 2, u8(G + 1, N, K))              # B's group count
    _refused(fn, args, 3, f32(G, NNB, NKB + 1))
    _refused(fn, args, 4, i32(G + 1))                   # masked_m length
    _refused(fn, args, 5, bf16(G, MM, N // 2))
    nkq = cdiv(NKB, 4)
    pargs = [u8(G, MM, K), i32(G, nkq, a4(MM)), u8(G, N, K), i32(G, NNB, nkq), i32(G), bf16(G, MM, N)]
    _accepted(dg.dg_fp8_grouped_masked_ue8m0, pargs)
    _refused(dg.dg_fp8_grouped_masked_ue8m0, pargs, 1, i32(G, NKB, a4(MM)))


def test_swiglu_shapes():
    MM, N2 = 64, 512
    args = [u8(G, MM, K), f32(G, NKB, a4(MM)), u8(G, N2, K), f32(G, N2 // 128, NKB), i32(G), bf16(G, MM, N2 // 2)]
    fn = dg.dg_fp8_grouped_masked_swiglu
    _accepted(fn, args)
    _refused(fn, args, 5, bf16(G, MM, N2))              # H is I = N2/2 wide
    _refused(fn, args, 3, f32(G, N2 // 256, NKB))
    nkq = cdiv(NKB, 4)
    pargs = [u8(G, MM, K), i32(G, nkq, a4(MM)), u8(G, N2, K), i32(G, N2 // 128, nkq), i32(G), bf16(G, MM, N2 // 2)]
    _accepted(dg.dg_fp8_grouped_masked_swiglu_ue8m0, pargs)
    _accepted(dg.dg_fp8_grouped_masked_swiglu_ue8m0_f32, pargs[:5] + [f32(G, MM, N2 // 2)])
    _refused(dg.dg_fp8_grouped_masked_swiglu_ue8m0, pargs, 1, i32(G, NKB, a4(MM)))
    _refused(dg.dg_fp8_grouped_masked_swiglu_ue8m0, pargs, 5, bf16(G, MM, N2))
    qargs = args[:5] + [u8(G, MM, N2 // 2), f32(G, N2 // 256, a4(MM))]
    _accepted(dg.dg_fp8_grouped_masked_swiglu_fp8, qargs)
    _refused(dg.dg_fp8_grouped_masked_swiglu_fp8, qargs, 5, u8(G, MM, N2))       # Hq is I wide
    _refused(dg.dg_fp8_grouped_masked_swiglu_fp8, qargs, 6, f32(G, N2 // 128, a4(MM)))   # sH has I/128 groups
    _refused(dg.dg_fp8_grouped_masked_swiglu_fp8, qargs, 6, f32(G, N2 // 256, MM + 1))


@pytest.mark.parametrize("layout", ["nn", "tn", "tt"])
def test_layout_shapes(layout):
    a_t, b_n = {"nn": (False, True), "tn": (True, True), "tt": (True, False)}[layout]
    fn = getattr(dg, f"dg_fp8_gemm_{layout}")
    A = u8(K, M) if a_t else u8(M, K)
    B = u8(K, N) if b_n else u8(N, K)
    args = [A, f32(NKB, a4(M)), B, f32(NNB, NKB), bf16(M, N), M, N, K]
    _accepted(fn, args)
    _refused(fn, args, 0, u8(M, K) if a_t else u8(K, M))   # A stored the other way
    _refused(fn, args, 2, u8(N, K) if b_n else u8(K, N))   # B stored the other way
    _refused(fn, args, 1, f32(NKB, a4(M) + 4))
    _refused(fn, args, 3, f32(NNB, NKB + 1))
    _refused(fn, args, 4, bf16(M, N + 8))
    _refused(fn, args, 5, M + 16)                          # sizes that disagree with the tensors


@pytest.mark.parametrize("layout", ["nn", "tn", "tt"])
def test_layout_ue8m0_shapes(layout):
    a_t, b_n = {"nn": (False, True), "tn": (True, True), "tt": (True, False)}[layout]
    fn = getattr(dg, f"dg_fp8_gemm_{layout}_ue8m0")
    nkq = cdiv(NKB, 4)
    A = u8(K, M) if a_t else u8(M, K)
    B = u8(K, N) if b_n else u8(N, K)
    args = [A, i32(nkq, a4(M)), B, i32(NNB, nkq), bf16(M, N), M, N, K]
    _accepted(fn, args)
    _refused(fn, args, 1, i32(NKB, a4(M)))                 # FP32-scale layout to the packed call
    _refused(fn, args, 3, i32(NNB, NKB))
    _refused(fn, args, 0, u8(M, K) if a_t else u8(K, M))
    _accepted(getattr(dg, f"dg_fp8_gemm_{layout}_ue8m0_f32"), args[:4] + [f32(M, N), M, N, K])


def test_k_grouped_shapes():
    KT, MG, NG = 1024, 256, 384
    args = [u8(KT, MG), f32(KT // 128, a4(MG)), u8(KT, NG), f32(cdiv(NG, 128), KT // 128), i32(G + 1), bf16(G, MG, NG)]
    fn = dg.dg_fp8_k_grouped_gemm_tn_contiguous
    _accepted(fn, args)
    _refused(fn, args, 0, u8(MG, KT))                      # A must be [K_total, M]
    _refused(fn, args, 2, u8(KT + 128, NG))                # B's K_total
    _refused(fn, args, 1, f32(KT // 128 + 1, a4(MG)))
    _refused(fn, args, 3, f32(cdiv(NG, 128), KT // 128 - 1))
    _refused(fn, args, 5, bf16(G + 1, MG, NG))             # D's group count follows k_offsets
    _refused(fn, args, 4, i32(G + 1, 1))                   # k_offsets not 1-D
    nkq = cdiv(KT // 128, 4)
    pargs = [u8(KT, MG), i32(nkq, a4(MG)), u8(KT, NG), i32(cdiv(NG, 128), nkq), i32(G + 1), bf16(G, MG, NG)]
    _accepted(dg.dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0, pargs)
    _refused(dg.dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0, pargs, 1, i32(KT // 128, a4(MG)))
    _refused(dg.dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0, pargs, 3, i32(cdiv(NG, 128), KT // 128))


def test_transform_sf_shapes():
    nkq = cdiv(NKB, 4)
    fa = lambda s, p: dg.dg_transform_sf_into_ue8m0_a(s, p, M, K)
    fb = lambda s, p: dg.dg_transform_sf_into_ue8m0_b(s, p, N, K)
    for args in ([f32(NKB, a4(M)), i32(nkq, a4(M))], [f32(G, NKB, a4(M)), i32(G, nkq, a4(M))]):
        _accepted(fa, args)
        _refused(fa, args, 1, i32(*args[1].shape[:-2], NKB, a4(M)))      # unpacked K extent
        _refused(fa, args, 0, f32(*args[0].shape[:-2], NKB, M))          # rows not padded to 4
    for args in ([f32(NNB, NKB), i32(NNB, nkq)], [f32(G, NNB, NKB), i32(G, NNB, nkq)]):
        _accepted(fb, args)
        _refused(fb, args, 1, i32(*args[1].shape[:-1], NKB))
        _refused(fb, args, 0, f32(*args[0].shape[:-2], NNB + 1, NKB))
    _refused(fa, [f32(NKB), i32(nkq)], 0, f32(NKB))                       # 1-D is not a layout


def test_transform_sf_rows_shapes():
    f = lambda r, s: dg.dg_transform_sf_a_into_mn_major(r, s, M, K)
    for args in ([f32(M, NKB), f32(NKB, a4(M))], [f32(G, M, NKB), f32(G, NKB, a4(M))]):
        _accepted(f, args)
        _refused(f, args, 0, f32(*args[0].shape[:-2], NKB, M))           # already MN-major
        _refused(f, args, 1, f32(*args[1].shape[:-2], NKB, M))           # output rows not padded
