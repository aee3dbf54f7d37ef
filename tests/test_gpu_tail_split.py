"""GPU parity of the tail split: the tiles of a last, partial wave cut along K (both kernels).

Each case runs the same call with the tail split on (default) and off (dg_set_tail_splits(1)) and
checks:
- the tiles computed whole are bitwise identical in the two runs;
- the tail tiles differ somewhere (their partial sums are added in another order, so the split
  path really ran) and are accurate against the FP64 oracle either way;
- BF16 == RNE(FP32), and rows that must stay untouched are untouched.

Which tiles form the tail follows the kernel's rule: tiles % grid of them at the end of the linear
tile order when that is at most half the grid, cut into the number of K ranges that the kernel's
cost model prefers (up to 4).
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
    # a launch by pairs of CTAs sharing B tiles has no tail split: these tests use single CTAs
    prev = m.dg_set_pair_b(False)
    yield m
    m.dg_set_pair_b(prev)
    assert m.dg_get_device_status() == 0


KB_NS = {"fp32": 534, "ue8m0": 300}   # the kernels' cost of one K-block in their tail-split model


def _tail(tiles, grid, nkb, bn, kb_ns=534, max_splits=4):
    """(first tail tile, K ranges per tail tile) under the kernel's rule; (tiles, 1) if none."""
    rem = tiles % grid
    if not (max_splits > 1 and rem > 0 and 2 * rem <= grid):
        return tiles, 1
    pub, red, kb = (2500, 1000, kb_ns) if bn == 256 else (1600, 600, kb_ns)
    best, out = 0, (tiles, 1)
    s = 2
    while s <= max_splits and s * rem <= grid:
        kps = -(-nkb // s)
        eff = -(-nkb // kps)
        gain = (nkb - kps) * kb - (pub + eff * red)
        if eff > 1 and gain > best:
            best, out = gain, (tiles - rem, eff)
        s += 1
    return out


def _dense_tile(u, mb, nb):
    """(m_blk, n_blk) of linear tile u: rasterised in groups of min(mb, 16) m-blocks."""
    rm = min(mb, 16)
    per_group = rm * nb
    grp, local = divmod(u, per_group)
    first_m = grp * rm
    gsz = min(mb - first_m, rm)
    return first_m + local % gsz, local // gsz


def _both(dg, run):
    """run() with the tail split on, then off; the setting is restored afterwards."""
    on = run()
    prev = dg.dg_set_tail_splits(1)
    try:
        off = run()
    finally:
        dg.dg_set_tail_splits(prev)
    return on, off


def _dense_shape(dg):
    """M, N, K whose BN=256 tiles leave a tail of 8 to 15 tiles on this GPU's grid."""
    sms = dg.dg_get_num_sms()
    nb = 8
    mb = -(-(sms + 8) // nb)
    return 128 * mb, 256 * nb, 4096


def _scales(a, b, scales):
    """(device sA, device sB, oracle sA, oracle sB): FP32 scales, or packed UE8M0 words and the
    FP32 scales the oracle decodes from those words."""
    if scales == "fp32":
        return a.sA, b.sB, a.sA, b.sB
    nkb = -(-a.A.shape[-1] // 128)
    pa, pb = dg_inputs.pack_ue8m0_a(a.sA), dg_inputs.pack_ue8m0_b(b.sB)
    return pa, pb, oracle.unpack_ue8m0_a(pa, nkb), oracle.unpack_ue8m0_b(pb, nkb)


@pytest.mark.parametrize("scales", ["fp32", "ue8m0"])
def test_tail_split_dense(dg, scales):
    ue = scales == "ue8m0"
    M, N, K = _dense_shape(dg)
    cfg = (dg.dg_query_config_ue8m0 if ue else dg.dg_query_config)(0, M, N, K)
    assert cfg["splits"] == 1 and cfg["block_n"] == 256
    mb, nb = M // 128, N // 256
    tiles = mb * nb
    first, splits = _tail(tiles, cfg["grid"], K // 128, 256, KB_NS[scales])
    assert splits > 1, f"expected a tail split: tiles={tiles} grid={cfg['grid']}"
    a = dg_inputs.make_a(M, K, seed=41, ue8m0=ue)
    b = dg_inputs.make_b(1, N, K, seed=41, ue8m0=ue)
    gsA, gsB, osA, osB = _scales(a, b, scales)
    A, sA, B, sB = dev(a.A), dev(gsA), dev(b.B[0]), dev(gsB[0])
    f_bf16 = dg.dg_fp8_gemm_nt_ue8m0 if ue else dg.dg_fp8_gemm_nt
    f_f32 = dg.dg_fp8_gemm_nt_ue8m0_f32 if ue else dg.dg_fp8_gemm_nt_f32

    def run():
        D = bf16_sentinel((M, N))
        D32 = f32_sentinel((M, N))
        f_bf16(A, sA, B, sB, D)
        f_f32(A, sA, B, sB, D32)
        torch.cuda.synchronize()
        return bits16(D).cpu(), D32.cpu().numpy()

    (d_on, f_on), (d_off, f_off) = _both(dg, run)
    assert torch.equal(d_on, rne_bf16_bits(torch.from_numpy(f_on)))
    in_tail = np.zeros((M, N), bool)
    for u in range(first, tiles):
        m_blk, n_blk = _dense_tile(u, mb, nb)
        in_tail[m_blk * 128:(m_blk + 1) * 128, n_blk * 256:(n_blk + 1) * 256] = True
    assert in_tail.sum() == (tiles - first) * 128 * 256
    assert np.array_equal(f_on.view(np.int32)[~in_tail], f_off.view(np.int32)[~in_tail]), \
        "tiles computed whole differ between tail split on and off"
    assert not np.array_equal(f_on.view(np.int32)[in_tail], f_off.view(np.int32)[in_tail]), \
        "the tail tiles are bitwise identical: the split path did not run"
    rng = np.random.default_rng(5)
    tm, tn = np.nonzero(in_tail)
    pick = rng.choice(len(tm), 1500, replace=False)
    ms = np.concatenate([tm[pick], rng.integers(0, M, 500)])
    ns = np.concatenate([tn[pick], rng.integers(0, N, 500)])
    ref = oracle.gemm_nt_sampled(a.A, osA, b.B[0], osB[0], ms, ns)
    assert_accurate(f_on[ms, ns], d_on.numpy()[ms, ns], ref, f"{scales} tail split on")
    assert_accurate(f_off[ms, ns], d_off.numpy()[ms, ns], ref, f"{scales} tail split off")


def test_tail_split_contiguous_with_padding(dg):
    # 2560 rows in 20 m-blocks; the tail tiles hold group 3's last rows and its padding rows
    M, N, K = _dense_shape(dg)
    if M != 2560:
        pytest.skip("shape laid out for a 152-SM grid")
    m_idx = dg_inputs.contiguous_m_indices([600, 0, 700, 1100])
    assert len(m_idx) == M
    G = 4
    a = dg_inputs.make_a(M, K, seed=43)
    b = dg_inputs.make_b(G, N, K, seed=43)
    A, sA, B, sB, I = dev(a.A), dev(a.sA), dev(b.B), dev(b.sB), dev(m_idx)

    def run():
        D32 = f32_sentinel((M, N))
        dg.dg_fp8_grouped_contiguous_f32(A, sA, B, sB, I, D32)
        torch.cuda.synchronize()
        return D32.cpu().numpy()

    f_on, f_off = _both(dg, run)
    pad = m_idx < 0
    assert np.all(np.isnan(f_on[pad])) and np.all(np.isnan(f_off[pad])), "padding rows were written"
    mb, nb = M // 128, N // 256
    first, splits = _tail(mb * nb, dg.dg_query_config(1, M, N, K, G)["grid"], K // 128, 256)
    assert splits > 1
    in_tail = np.zeros((M, N), bool)
    for u in range(first, mb * nb):
        m_blk, n_blk = _dense_tile(u, mb, nb)
        in_tail[m_blk * 128:(m_blk + 1) * 128, n_blk * 256:(n_blk + 1) * 256] = True
    valid = ~pad[:, None] & np.ones((1, N), bool)
    assert np.array_equal(f_on.view(np.int32)[valid & ~in_tail], f_off.view(np.int32)[valid & ~in_tail])
    assert not np.array_equal(f_on.view(np.int32)[valid & in_tail], f_off.view(np.int32)[valid & in_tail])
    rng = np.random.default_rng(6)
    tm, tn = np.nonzero(valid & in_tail)
    pick = rng.choice(len(tm), 1200, replace=False)
    ms, ns = tm[pick], tn[pick]
    ref = oracle.contiguous_sampled(a.A, a.sA, b.B, b.sB, m_idx, ms, ns)
    for f, what in ((f_on, "on"), (f_off, "off")):
        d = f[ms, ns]
        bits = torch.from_numpy(d.copy()).to(torch.bfloat16).view(torch.int16).numpy()
        assert_accurate(d, bits, ref, f"contiguous tail split {what}")


@pytest.mark.parametrize("scales", ["fp32", "ue8m0"])
def test_tail_split_masked_decode(dg, scales):
    # the decode shape: 16 groups, masked_m from seed 0, N=4096, K=7168 (320 tiles: a tail of 16)
    ue = scales == "ue8m0"
    G, M_max, N, K = 16, 256, 4096, 7168
    masked_m = dg_inputs.make_masked_m(G, M_max, seed=0)
    mbs = [-(-int(m) // 128) for m in masked_m]
    nb = N // 256
    tiles = sum(mbs) * nb
    grid = (dg.dg_query_config_ue8m0 if ue else dg.dg_query_config)(2, M_max, N, K, G)["grid"]
    first, splits = _tail(tiles, grid, K // 128, 256, KB_NS[scales])
    if splits == 1:
        pytest.skip(f"no tail split for tiles={tiles} on grid={grid}")
    a = dg_inputs.make_masked_a(G, M_max, K, seed=0, ue8m0=ue)
    b = dg_inputs.make_b(G, N, K, seed=0, ue8m0=ue)
    gsA, gsB, osA, osB = _scales(a, b, scales)
    A, sA, B, sB, MM = dev(a.A), dev(gsA), dev(b.B), dev(gsB), dev(masked_m)
    f_bf16 = dg.dg_fp8_grouped_masked_ue8m0 if ue else dg.dg_fp8_grouped_masked
    f_f32 = dg.dg_fp8_grouped_masked_ue8m0_f32 if ue else dg.dg_fp8_grouped_masked_f32

    def run():
        D = bf16_sentinel((G, M_max, N))
        D32 = f32_sentinel((G, M_max, N))
        f_bf16(A, sA, B, sB, MM, D)
        f_f32(A, sA, B, sB, MM, D32)
        torch.cuda.synchronize()
        return bits16(D).cpu(), D32.cpu().numpy()

    (d_on, f_on), (d_off, f_off) = _both(dg, run)
    valid = np.arange(M_max)[None, :, None] < masked_m[:, None, None]
    valid = np.broadcast_to(valid, (G, M_max, N))
    assert torch.all(d_on[torch.from_numpy(~valid)] == -1), "rows past masked_m were written"
    assert np.all(np.isnan(f_on[~valid]))
    vt = torch.from_numpy(np.ascontiguousarray(valid))
    assert torch.equal(d_on[vt], rne_bf16_bits(torch.from_numpy(f_on))[vt])
    # tiles in order: groups in turn, within a group m-blocks fastest, then n-blocks
    in_tail = np.zeros((G, M_max, N), bool)
    u = 0
    for g in range(G):
        for local in range(mbs[g] * nb):
            if u >= first:
                m_blk, n_blk = local % mbs[g], local // mbs[g]
                in_tail[g, m_blk * 128:(m_blk + 1) * 128, n_blk * 256:(n_blk + 1) * 256] = True
            u += 1
    assert u == tiles
    sel_whole, sel_tail = valid & ~in_tail, valid & in_tail
    assert np.array_equal(f_on.view(np.int32)[sel_whole], f_off.view(np.int32)[sel_whole])
    assert not np.array_equal(f_on.view(np.int32)[sel_tail], f_off.view(np.int32)[sel_tail])
    rng = np.random.default_rng(7)
    gs, ms, ns = np.nonzero(sel_tail)
    pick = rng.choice(len(gs), 1500, replace=False)
    gs, ms, ns = gs[pick], ms[pick], ns[pick]
    ref = oracle.masked_sampled(a.A, osA, b.B, osB, gs, ms, ns)
    assert_accurate(f_on[gs, ms, ns], d_on.numpy()[gs, ms, ns], ref, f"{scales} masked tail split on")
    assert_accurate(f_off[gs, ms, ns], d_off.numpy()[gs, ms, ns], ref, f"{scales} masked tail split off")


def test_tail_split_setting_round_trip(dg):
    prev = dg.dg_set_tail_splits(2)
    try:
        assert dg.dg_set_tail_splits(99) == 2
        assert dg.dg_set_tail_splits(0) == 16          # clamped to 16
        assert dg.dg_set_tail_splits(prev) == 4        # 0 restored the default
    finally:
        dg.dg_set_tail_splits(prev)


@pytest.mark.parametrize("layout", ["nn", "tt"])
def test_tail_split_layouts_match_nt(dg, layout):
    # the transposed layouts take the same schedule: bitwise equal to the NT call, tail included
    M, N, K = _dense_shape(dg)
    a = dg_inputs.make_a(M, K, seed=44)
    b = dg_inputs.make_b(1, N, K, seed=44)
    sA, sB = dev(a.sA), dev(b.sB[0])
    a_t, b_t = {"nn": (False, True), "tt": (True, False)}[layout]   # A stored [K,M] / B stored [K,N]
    A = dev(np.ascontiguousarray(a.A.T)) if a_t else dev(a.A)
    B = dev(np.ascontiguousarray(b.B[0].T)) if b_t else dev(b.B[0])
    D32 = f32_sentinel((M, N))
    getattr(dg, f"dg_fp8_gemm_{layout}_f32")(A, sA, B, sB, D32, M, N, K)
    Dnt = f32_sentinel((M, N))
    dg.dg_fp8_gemm_nt_f32(dev(a.A), sA, dev(b.B[0]), sB, Dnt)
    torch.cuda.synchronize()
    assert torch.equal(D32.view(torch.int32), Dnt.view(torch.int32))


def test_tail_split_accumulate(dg):
    # D = C + A·Bᵀ: the split tiles are reduced once, then added onto C once
    M, N, K = _dense_shape(dg)
    a = dg_inputs.make_a(M, K, seed=45)
    b = dg_inputs.make_b(1, N, K, seed=45)
    A, sA, B, sB = dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0])
    C = dg_inputs.draw(45, 6, M * N).reshape(M, N) * np.float32(30.0)
    D32 = torch.full((M, N), float("nan"), device="cuda")
    dg.dg_fp8_gemm_nt_f32(A, sA, B, sB, D32)
    Ct = dev(C)
    dg.dg_fp8_gemm_nt_acc_f32(A, sA, B, sB, Ct, Ct)
    torch.cuda.synchronize()
    want = (C.astype(np.float32) + D32.cpu().numpy()).astype(np.float32)
    assert np.array_equal(Ct.cpu().numpy().view(np.int32), want.view(np.int32))
