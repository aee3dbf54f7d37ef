"""GPU parity of the masked grouped GEMM fused with SwiGLU against the CPU oracle, with FP32 scales
(the FP32-scale kernel) and with power-of-two scales packed as UE8M0 (the block-scaled kernel).

H[g,m,j] = silu(D[g,m,j]) · D[g,m,I+j] over the valid rows m < masked_m[g] (B holds the I gate rows,
then the I up rows, of each group). Checked: rows past masked_m untouched (sentinel bits), the BF16
output equal to RNE of the FP32 output of the same kernel, and the accuracy bar of
tests/_dg_testlib.py against the FP64 oracle.
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


SCALES = ["fp32", "ue8m0"]


def _run(dg, a, b, masked_m, scales="fp32"):
    G, M_max, _ = a.A.shape
    I = b.B.shape[1] // 2
    A, B, MM = dev(a.A), dev(b.B), dev(masked_m)
    H = bf16_sentinel((G, M_max, I))
    H32 = f32_sentinel((G, M_max, I))
    if scales == "ue8m0":
        sA, sB = dev(dg_inputs.pack_ue8m0_a(a.sA)), dev(dg_inputs.pack_ue8m0_b(b.sB))
        dg.dg_fp8_grouped_masked_swiglu_ue8m0(A, sA, B, sB, MM, H)
        dg.dg_fp8_grouped_masked_swiglu_ue8m0_f32(A, sA, B, sB, MM, H32)
    else:
        sA, sB = dev(a.sA), dev(b.sB)
        dg.dg_fp8_grouped_masked_swiglu(A, sA, B, sB, MM, H)
        dg.dg_fp8_grouped_masked_swiglu_f32(A, sA, B, sB, MM, H32)
    torch.cuda.synchronize()
    return H, H32


def _valid(masked_m, M_max):
    return np.arange(M_max)[None, :] < np.clip(masked_m, 0, M_max)[:, None]


@pytest.mark.parametrize("scales", SCALES)
@pytest.mark.parametrize("I,K", [(128, 384), (256, 1024), (384, 256), (256, 640)])
def test_swiglu_full_parity(dg, I, K, scales):
    masked_m = np.array([0, 1, 127, 128, 129, 256], np.int32)
    G, M_max = len(masked_m), 256
    ue = scales == "ue8m0"
    a = dg_inputs.make_masked_a(G, M_max, K, seed=41, ue8m0=ue)
    b = dg_inputs.make_b(G, 2 * I, K, seed=41, ue8m0=ue)
    H, H32 = _run(dg, a, b, masked_m, scales)
    ref, _, bad = oracle.grouped_masked_swiglu(a.A, a.sA, b.B, b.sB, masked_m)
    assert bad == 0
    valid = torch.from_numpy(_valid(masked_m, M_max))
    hb = bits16(H).cpu()
    assert torch.all(hb[~valid] == -1), "rows past masked_m were written"
    assert torch.all(torch.isnan(H32.cpu()[~valid]))
    assert torch.equal(hb[valid], rne_bf16_bits(H32)[valid])
    v = valid.numpy()
    assert_accurate(H32.cpu().numpy()[v], hb.numpy()[v], ref[v], f"swiglu/{scales} I={I} K={K}")


@pytest.mark.parametrize("scales", SCALES)
def test_swiglu_decode_sampled(dg, scales):
    G, M_max, I, K = 16, 256, 2048, 7168
    ue = scales == "ue8m0"
    masked_m = dg_inputs.make_masked_m(G, M_max, seed=0)
    a = dg_inputs.make_masked_a(G, M_max, K, seed=0, ue8m0=ue)
    b = dg_inputs.make_b(G, 2 * I, K, seed=0, ue8m0=ue)
    H, H32 = _run(dg, a, b, masked_m, scales)
    valid = _valid(masked_m, M_max)
    vt = torch.from_numpy(valid)
    hb = bits16(H).cpu()
    assert torch.all(hb[~vt] == -1)
    assert torch.equal(hb[vt], rne_bf16_bits(H32)[vt])
    rng = np.random.default_rng(9)
    gs, ms = np.nonzero(valid)
    pick = rng.choice(len(gs), size=2000, replace=len(gs) < 2000)
    gs, ms = gs[pick], ms[pick]
    js = rng.integers(0, I, len(gs))
    ref = oracle.masked_swiglu_sampled(a.A, a.sA, b.B, b.sB, gs, ms, js)
    assert_accurate(H32.cpu().numpy()[gs, ms, js], hb.numpy()[gs, ms, js], ref, f"swiglu/{scales} decode")


def test_swiglu_rejects_bad_width(dg):
    a = dg_inputs.make_masked_a(2, 64, 128, seed=1)
    b = dg_inputs.make_b(2, 192, 128, seed=1)          # 2I = 192: I is not a multiple of 128
    H = bf16_sentinel((2, 64, 96))
    with pytest.raises(dg.DGError) as e:
        dg.dg_fp8_grouped_masked_swiglu(dev(a.A), dev(a.sA), dev(b.B), dev(b.sB), dev(np.array([5, 6], np.int32)), H)
    assert e.value.status == dg.DG_ERR_ALIGNMENT


# ----------------------------------------------------------------------------------------------
# The fused SwiGLU with H cast to FP8 (dg_fp8_grouped_masked_swiglu_fp8). The cast is a decision
# per element, so it is checked in the kernel's own precision: the codes and scales must equal,
# bit for bit, the oracle's plain 1x128 quantiser applied to the FP32 H of the same kernel
# (dg_fp8_grouped_masked_swiglu_f32). The dequantised H is checked against the FP64 oracle within
# half an E4M3 step of each group's top binade, and the down projection consumes Hq/sH as its A/sA.

def _align4(x):
    return -(-x // 4) * 4


def _fp8_h(dg, a, b, masked_m):
    G, M_max, _ = a.A.shape
    I = b.B.shape[1] // 2
    Hq = torch.full((G, M_max, I), 0x7F, dtype=torch.uint8, device="cuda")          # NaN codes
    sH = torch.full((G, I // 128, _align4(M_max)), float("nan"), dtype=torch.float32, device="cuda")
    dg.dg_fp8_grouped_masked_swiglu_fp8(dev(a.A), dev(a.sA), dev(b.B), dev(b.sB), dev(masked_m), Hq, sH)
    torch.cuda.synchronize()
    return Hq.cpu().numpy(), sH.cpu().numpy()


def _check_fp8_h(dg, a, b, masked_m, label, ref64=None):
    G, M_max, _ = a.A.shape
    I = b.B.shape[1] // 2
    _, H32 = _run(dg, a, b, masked_m)
    Hq, sH = _fp8_h(dg, a, b, masked_m)
    valid = _valid(masked_m, M_max)
    h32 = H32.cpu().numpy()
    h32 = np.where(valid[..., None], h32, 0.0).astype(np.float32)
    codes, scales = oracle.quantize_rows_e4m3(h32)          # scales [G, I/128, M_max]
    assert np.all(Hq[~valid] == 0x7F), f"{label}: rows past masked_m were written"
    assert np.array_equal(Hq[valid], codes[valid]), f"{label}: codes differ from the 1x128 cast of H"
    sv = np.swapaxes(sH[:, :, :M_max], 1, 2)                # [G, M_max, I/128]
    assert np.all(np.isnan(sv[~valid])) and np.all(np.isnan(sH[:, :, M_max:]))
    assert np.array_equal(sv[valid].view(np.int32), np.swapaxes(scales, 1, 2)[valid].view(np.int32)), \
        f"{label}: scales differ"
    if ref64 is not None:
        deq = oracle.e4m3_decode(Hq).reshape(G, M_max, I // 128, 128) * sv[..., None]
        h64 = ref64.reshape(G, M_max, I // 128, 128)
        amax = np.max(np.abs(h32.reshape(G, M_max, I // 128, 128)), axis=-1, keepdims=True)
        bound = (16.0 / 448.0) * amax * 1.0001 + 2e-3 * np.max(np.abs(ref64))
        assert np.all(np.abs(deq - h64)[valid] <= bound[valid]), f"{label}: dequantised H off the oracle"
    return Hq, sH


@pytest.mark.parametrize("I,K", [(128, 384), (256, 1024), (384, 256)])
def test_swiglu_fp8_h_full(dg, I, K):
    masked_m = np.array([0, 1, 127, 128, 129, 256], np.int32)
    G, M_max = len(masked_m), 256
    a = dg_inputs.make_masked_a(G, M_max, K, seed=43)
    b = dg_inputs.make_b(G, 2 * I, K, seed=43)
    ref, _, bad = oracle.grouped_masked_swiglu(a.A, a.sA, b.B, b.sB, masked_m)
    assert bad == 0
    _check_fp8_h(dg, a, b, masked_m, f"fp8 H I={I} K={K}", ref64=ref)


def test_swiglu_fp8_h_decode_and_down_projection(dg):
    G, M_max, I, K, N2 = 16, 256, 2048, 7168, 1024
    masked_m = dg_inputs.make_masked_m(G, M_max, seed=0)
    a = dg_inputs.make_masked_a(G, M_max, K, seed=0)
    b = dg_inputs.make_b(G, 2 * I, K, seed=0)
    Hq, sH = _check_fp8_h(dg, a, b, masked_m, "fp8 H decode")
    # the down projection reads Hq and sH as its A and sA, exactly as they are
    w2 = dg_inputs.make_b(G, N2, I, seed=2)
    D2 = bf16_sentinel((G, M_max, N2))
    D2_32 = f32_sentinel((G, M_max, N2))
    args = (dev(Hq), dev(np.ascontiguousarray(sH)), dev(w2.B), dev(w2.sB), dev(masked_m))
    dg.dg_fp8_grouped_masked(*args, D2)
    dg.dg_fp8_grouped_masked_f32(*args, D2_32)
    torch.cuda.synchronize()
    valid = _valid(masked_m, M_max)
    ref2, _, bad = oracle.grouped_masked(Hq, sH, w2.B, w2.sB, masked_m)
    assert bad == 0
    db = bits16(D2).cpu()
    assert torch.all(db[~torch.from_numpy(valid)] == -1)
    assert_accurate(D2_32.cpu().numpy()[valid], db.numpy()[valid], ref2[valid], "down projection of FP8 H")
