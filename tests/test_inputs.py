"""The seeded input generator and quantiser (input preparation shared by both sides; CPU only)."""
import numpy as np
import torch

import dg_inputs


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(50000) * 100, rng.standard_normal(5000) * 0.01,
                        rng.uniform(-463.9, 463.9, 5000)]).astype(np.float32)
    x = x[np.abs(x) < 464]            # beyond the 448/480 midpoint torch gives NaN; we saturate
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = dg_inputs.e4m3_encode(x)
    assert np.array_equal(got, want)


def test_e4m3_encode_round_trip_and_saturation():
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(dg_inputs.e4m3_encode(table[codes]), codes)
    sat = dg_inputs.e4m3_encode(np.array([448.0, 470.0, 1e6, -1e6, -449.0], np.float32))
    assert sat.tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_draw_is_thread_independent_and_normal():
    a = dg_inputs.draw(0, 0, 200001, threads=1)
    b = dg_inputs.draw(0, 0, 200001, threads=7)
    assert np.array_equal(a, b)
    assert abs(a.mean()) < 0.01 and abs(a.std() - 1) < 0.01
    c = dg_inputs.draw(0, 0, 1000, base=500)
    assert np.array_equal(c, a[500:1500])
    assert not np.array_equal(dg_inputs.draw(0, 1, 1000), a[:1000])
    t = dg_inputs.draw(0, 0, 200000, dist=dg_inputs.STUDENT_T3)
    # Student-t(3): variance 3, heavy tails
    assert abs(t.var() - 3) < 0.6 and np.abs(t).max() > 20


def test_quantize_a_scales_and_error_bound():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((37, 300)).astype(np.float32)
    x[3, :128] = 0                                    # an all-zero group gets s = 1
    qa = dg_inputs.quantize_a(x)
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert qa.sA.shape == (3, 40)
    assert np.all(qa.sA[:, 37:] == 0)
    for kb in range(3):
        sl = slice(kb * 128, min(300, kb * 128 + 128))
        amax = np.abs(x[:, sl]).max(axis=1)
        want = np.where(amax > 0, amax / np.float32(448), np.float32(1)).astype(np.float32)
        assert np.array_equal(qa.sA[kb, :37], want)
        deq = table[qa.A[:, sl]] * qa.sA[kb, :37, None]
        # E4M3 keeps 4 significant bits: relative error <= 2^-4 for normals, plus subnormal quantum
        err = np.abs(deq - x[:, sl])
        bound = np.abs(x[:, sl]) * 2.0 ** -4 + qa.sA[kb, :37, None] * 2.0 ** -10
        assert np.all(err <= bound)
    assert np.all(qa.A[3, :128] == 0) and qa.sA[0, 3] == 1.0


def test_quantize_b_block_scales():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 200, 256)).astype(np.float32)
    qb = dg_inputs.quantize_b(x)
    assert qb.sB.shape == (2, 2, 2)
    for g in range(2):
        for nb in range(2):
            for kb in range(2):
                blk = x[g, nb * 128:min(200, nb * 128 + 128), kb * 128:kb * 128 + 128]
                assert qb.sB[g, nb, kb] == np.float32(np.abs(blk).max()) / np.float32(448)


def test_make_a_matches_quantize_of_drawn_values():
    M, K = 5, 260
    a = dg_inputs.make_a(M, K, seed=3, base_row=7)
    x = dg_inputs.draw(3, 0, M * K, base=7 * K).reshape(M, K)
    q = dg_inputs.quantize_a(x)
    assert np.array_equal(a.A, q.A) and np.array_equal(a.sA, q.sA)


def test_outliers_and_masked_m():
    ch = dg_inputs.outlier_channels(0, 7168, 0.01)
    assert len(ch) == 72 and len(set(ch.tolist())) == 72 and ch.min() >= 0 and ch.max() < 7168
    mm = dg_inputs.make_masked_m(16, 256, seed=0)
    assert mm[0] == 0 and mm[-1] == 256 and np.all((mm >= 0) & (mm <= 256))
    idx = dg_inputs.contiguous_m_indices([3, 0, 130], pad_to=128)
    assert len(idx) == 128 + 256 and (idx == -1).sum() == 125 + 126


def test_ue8m0_scales_are_the_smallest_sufficient_powers_of_two():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((21, 400)) * np.exp(rng.uniform(-20, 20, (21, 1)))).astype(np.float32)
    x[5, 128:256] = 0
    qa = dg_inputs.quantize_a(x, ue8m0=True)
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for kb in range(4):
        sl = slice(kb * 128, min(400, kb * 128 + 128))
        t = np.abs(x[:, sl]).max(axis=1) / np.float32(448)
        s = qa.sA[kb, :21].astype(np.float64)
        m, _ = np.frexp(s)
        assert np.all(m == 0.5)                                   # powers of two
        nz = t > 0
        assert np.all(s[nz] >= t[nz]) and np.all(s[nz] / 2 < t[nz])
        assert np.all(s[~nz] == 1.0)
        assert np.all(np.abs(table[qa.A[:, sl]]) <= 448)
    qb = dg_inputs.quantize_b(x[None, :, :256], ue8m0=True)
    m, _ = np.frexp(qb.sB.astype(np.float64))
    assert np.all(m == 0.5)


def test_pack_ue8m0_layout_and_padding():
    sA = np.array([[1.0, 2.0, 0.0, 0.0], [0.5, 4.0, 0.0, 0.0], [2.0 ** -127, 2.0 ** 127, 0.0, 0.0],
                   [1.0, 1.0, 0.0, 0.0], [8.0, 0.25, 0.0, 0.0]], np.float32)      # [nkb=5][ldsa=4]
    p = dg_inputs.pack_ue8m0_a(sA).view(np.uint32)
    assert p.shape == (2, 4)
    assert hex(p[0, 0]) == hex(0x7F007E7F) and hex(p[0, 1]) == hex(0x7FFE8180)
    assert hex(p[1, 0]) == hex(0x7F7F7F82) and hex(p[1, 1]) == hex(0x7F7F7F7D)
    assert np.all(p[:, 2:] == 0x7F7F7F7F)
    sB = np.array([[[1.0, 2.0, 4.0, 8.0, 16.0]]], np.float32)                    # [G=1][nnb=1][nkb=5]
    q = dg_inputs.pack_ue8m0_b(sB).view(np.uint32)
    assert q.shape == (1, 1, 2) and q[0, 0, 0] == 0x8281807F and q[0, 0, 1] == 0x7F7F7F83
    with np.testing.assert_raises(ValueError):
        dg_inputs.pack_ue8m0_b(np.array([[[3.0]]], np.float32))
