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
