"""dg_transform_sf_into_ue8m0_a/_b: FP32 power-of-two scales packed on the GPU into the UE8M0 words of
the block-scaled calls.

Checked against the oracle's independent unpacker (every valid scale comes back exactly, padding
bytes and padding rows hold 127), against a GEMM (the block-scaled call on the packed words matches
the FP64 oracle run on the FP32 scales), and on values that are not powers of two (the status bit is
set and the code is that of the next power of two up).
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
    assert m.dg_get_device_status() == 0
    yield m
    assert m.dg_get_device_status() == 0


def _pack_a(dg, sA, M, K):
    nkb = -(-K // 128)
    out = torch.full(sA.shape[:-2] + (-(-nkb // 4), sA.shape[-1]), -1, dtype=torch.int32, device="cuda")
    dg.dg_transform_sf_into_ue8m0_a(dev(sA), out, M, K)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _pack_b(dg, sB, N, K):
    nkb = -(-K // 128)
    out = torch.full(sB.shape[:-1] + (-(-nkb // 4),), -1, dtype=torch.int32, device="cuda")
    dg.dg_transform_sf_into_ue8m0_b(dev(sB), out, N, K)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _bytes(words):
    return words.view(np.uint8).reshape(words.shape + (4,))   # little-endian: byte j = K-block 4q + j


@pytest.mark.parametrize("M,K", [(198, 1152), (64, 128), (4096, 7168), (130, 640)])
def test_pack_a_round_trip(dg, M, K):
    a = dg_inputs.make_a(M, K, seed=M + K, ue8m0=True)          # sA [nkb, align4(M)], powers of two
    nkb = -(-K // 128)
    words = _pack_a(dg, a.sA, M, K)
    assert dg.dg_get_device_status() == 0
    back = oracle.unpack_ue8m0_a(words, nkb)
    assert np.array_equal(back[:, :M], a.sA[:, :M]), "a scale did not come back exactly"
    assert np.all(back[:, M:] == 1.0), "padding rows must pack as 127 (the scale 1)"
    b = _bytes(words).reshape(words.shape[0], words.shape[1], 4)
    for q in range(words.shape[0]):
        for j in range(4):
            if 4 * q + j >= nkb:
                assert np.all(b[q, :, j] == 127), "bytes past the last K-block must be 127"


@pytest.mark.parametrize("G,N,K", [(1, 392, 1152), (4, 4096, 7168), (3, 256, 384)])
def test_pack_b_round_trip(dg, G, N, K):
    b = dg_inputs.make_b(G, N, K, seed=N + K, ue8m0=True)        # sB [G, nnb, nkb]
    nkb = -(-K // 128)
    words = _pack_b(dg, b.sB, N, K)
    assert dg.dg_get_device_status() == 0
    assert np.array_equal(oracle.unpack_ue8m0_b(words, nkb), b.sB)
    pad = _bytes(words)[..., :]
    for q in range(words.shape[-1]):
        for j in range(4):
            if 4 * q + j >= nkb:
                assert np.all(pad[..., q, j] == 127)


def test_packed_scales_drive_the_block_scaled_gemm(dg):
    M, N, K = 320, 640, 1664
    a = dg_inputs.make_a(M, K, seed=7, ue8m0=True)
    b = dg_inputs.make_b(1, N, K, seed=7, ue8m0=True)
    sA = torch.from_numpy(_pack_a(dg, a.sA, M, K)).cuda()
    sB = torch.from_numpy(_pack_b(dg, b.sB[0], N, K)).cuda()
    D, D32 = bf16_sentinel((M, N)), f32_sentinel((M, N))
    dg.dg_fp8_gemm_nt_ue8m0(dev(a.A), sA, dev(b.B[0]), sB, D)
    dg.dg_fp8_gemm_nt_ue8m0_f32(dev(a.A), sA, dev(b.B[0]), sB, D32)
    torch.cuda.synchronize()
    ref64, _ = oracle.gemm_nt(a.A, a.sA, b.B[0], b.sB[0], want_bf16=False)
    assert torch.equal(bits16(D).cpu(), rne_bf16_bits(D32))
    assert_accurate(D32.cpu().numpy(), bits16(D).cpu().numpy(), ref64, "block-scaled GEMM on transformed scales")


def test_values_that_are_not_powers_of_two(dg):
    # one K-block per row of B's layout: [rows, 1]; the codes are the exponent fields
    vals = np.array([3.0, 0.75, -2.0, np.inf, np.nan, 1e-45, 2.0 ** 127 * 1.5, 2.0 ** -127 * 1.5, 8.0],
                    dtype=np.float32)
    want = np.array([129, 127, 128, 254, 127, 0, 254, 1, 130], dtype=np.uint8)
    sB = vals.reshape(-1, 1)
    out = torch.full((len(vals), 1), -1, dtype=torch.int32, device="cuda")
    dg.dg_transform_sf_into_ue8m0_b(dev(sB), out, 128 * len(vals), 128)
    assert dg.dg_get_device_status() & dg.DG_DEV_BAD_SCALE
    got = _bytes(out.cpu().numpy())[:, 0, :]
    assert np.array_equal(got[:, 0], want), got[:, 0]
    assert np.all(got[:, 1:] == 127)
    # exact powers of two alone leave the status word clear
    ok = np.array([[1.0], [0.5], [2.0 ** -127], [2.0 ** 127]], dtype=np.float32)
    out2 = torch.empty((4, 1), dtype=torch.int32, device="cuda")
    dg.dg_transform_sf_into_ue8m0_b(dev(ok), out2, 512, 128)
    assert dg.dg_get_device_status() == 0
    assert np.array_equal(_bytes(out2.cpu().numpy())[:, 0, 0], np.array([127, 126, 0, 254], np.uint8))


def test_masked_layouts_pack_and_drive_the_masked_gemm(dg):
    # 3-D layouts of the masked form: sA [G, nkb, align4(M_max)], sB [G, nnb, nkb]
    G, M_max, N, K = 4, 96, 384, 896
    masked_m = np.array([0, 96, 37, 1], np.int32)
    a = dg_inputs.make_masked_a(G, M_max, K, seed=13, ue8m0=True)
    b = dg_inputs.make_b(G, N, K, seed=13, ue8m0=True)
    nkb = -(-K // 128)
    pa, pb = _pack_a(dg, a.sA, M_max, K), _pack_b(dg, b.sB, N, K)
    assert dg.dg_get_device_status() == 0
    assert np.array_equal(oracle.unpack_ue8m0_a(pa, nkb)[..., :M_max], a.sA[..., :M_max])
    assert np.array_equal(oracle.unpack_ue8m0_b(pb, nkb), b.sB)
    D32 = f32_sentinel((G, M_max, N))
    dg.dg_fp8_grouped_masked_ue8m0_f32(dev(a.A), torch.from_numpy(pa).cuda(), dev(b.B), torch.from_numpy(pb).cuda(),
                                       dev(masked_m), D32)
    torch.cuda.synchronize()
    ref, _, bad = oracle.grouped_masked(a.A, a.sA, b.B, b.sB, masked_m)
    assert bad == 0
    valid = np.arange(M_max)[None, :] < masked_m[:, None]
    d = D32.cpu().numpy()
    assert np.all(np.isnan(d[~valid])), "rows past masked_m were written"
    err = np.abs(d[valid].astype(np.float64) - ref[valid]).max() / np.abs(ref[valid]).max()
    assert err <= 2e-3, err


@pytest.mark.parametrize("G,M,K", [(1, 198, 1152), (1, 4096, 7168), (3, 70, 640), (2, 1, 128)])
def test_row_major_scales_to_mn_major(dg, G, M, K):
    # the MN-major layout of the input generator, handed over row-major and converted back on the GPU
    a = dg_inputs.make_masked_a(G, M, K, seed=G + M, ue8m0=False)   # sA [G, nkb, align4(M)]
    rows = np.ascontiguousarray(np.swapaxes(a.sA[..., :M], -1, -2))  # [G, M, nkb]
    out = torch.full(a.sA.shape, float("nan"), dtype=torch.float32, device="cuda")
    dg.dg_transform_sf_a_into_mn_major(dev(rows), out, M, K)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.array_equal(got[..., :M], a.sA[..., :M])
    assert np.all(got[..., M:] == 0.0), "padding rows must be zero"


def test_row_major_scales_drive_the_gemm(dg):
    M, N, K = 200, 264, 768
    a = dg_inputs.make_a(M, K, seed=17)
    b = dg_inputs.make_b(1, N, K, seed=17)
    rows = np.ascontiguousarray(a.sA[:, :M].T)                      # [M, nkb]
    sA = torch.empty(a.sA.shape, dtype=torch.float32, device="cuda")
    dg.dg_transform_sf_a_into_mn_major(dev(rows), sA, M, K)
    D32 = f32_sentinel((M, N))
    dg.dg_fp8_gemm_nt_f32(dev(a.A), sA, dev(b.B[0]), dev(b.sB[0]), D32)
    torch.cuda.synchronize()
    ref64, _ = oracle.gemm_nt(a.A, a.sA, b.B[0], b.sB[0], want_bf16=False)
    err = np.abs(D32.cpu().numpy().astype(np.float64) - ref64).max() / np.abs(ref64).max()
    assert err <= 2e-3, err
