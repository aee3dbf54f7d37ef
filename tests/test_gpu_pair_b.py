"""GPU parity of pairs of CTAs that share B tiles (TMA multicast; dg_set_pair_b).

A paired launch runs clusters of two CTAs over pairs of 128-row blocks: each loads its own A tile
and half of the B tile, multicast into both. The sum over K is taken in the same order, so every
case must be bit-identical to the single-CTA schedule (pairing off) — and accurate against the
FP64 oracle on samples that hit every output tile. Covered: ragged and odd M (the second block of
the last pair lies past M), BF16 and FP32 output, the accumulating form, and contiguous layouts whose
pairs straddle two groups (each CTA then loads its own group's B tile), hold a padding block, or are
all padding.
"""
import numpy as np
import pytest
import torch

import dg_inputs
import oracle
from _dg_testlib import assert_accurate, bf16_sentinel, bits16, boundary_samples, dev, f32_sentinel, rne_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import moe_grouped_gemm_e4m3_gb300 as m
    m.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield m
    m.dg_set_pair_b(False)
    assert m.dg_get_device_status() == 0


def _paired_and_single(dg, run):
    prev = dg.dg_set_pair_b(True)
    try:
        on = run()
        dg.dg_set_pair_b(False)
        off = run()
    finally:
        dg.dg_set_pair_b(prev)
    return on, off


@pytest.mark.parametrize("M,N,K", [(896, 3072, 1536), (1664, 2600, 768), (2304, 4096, 512), (4096, 7168, 2048)])
def test_pair_dense(dg, M, N, K):
    a = dg_inputs.make_a(M, K, seed=M + N)
    b = dg_inputs.make_b(1, N, K, seed=M + K)
    A, sA, B, sB = dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0])
    prev = dg.dg_set_pair_b(True)
    try:
        cfg = dg.dg_query_config(0, M, N, K)
    finally:
        dg.dg_set_pair_b(prev)
    assert cfg["block_m"] == 256 and cfg["grid"] % 2 == 0, cfg

    def run():
        D = bf16_sentinel((M, N))
        D32 = f32_sentinel((M, N))
        dg.dg_fp8_gemm_nt(A, sA, B, sB, D)
        dg.dg_fp8_gemm_nt_f32(A, sA, B, sB, D32)
        torch.cuda.synchronize()
        return bits16(D).cpu(), D32.cpu()

    (d_on, f_on), (d_off, f_off) = _paired_and_single(dg, run)
    assert torch.equal(f_on.view(torch.int32), f_off.view(torch.int32)), "FP32 differs with pairs"
    assert torch.equal(d_on, d_off), "BF16 differs with pairs"
    assert torch.equal(d_on, rne_bf16_bits(f_on))
    ms, ns = boundary_samples(M, N, 800, seed=M ^ N, block_cols=256)
    ref = oracle.gemm_nt_sampled(a.A, a.sA, b.B[0], b.sB[0], ms, ns)
    assert_accurate(f_on.numpy()[ms, ns], d_on.numpy()[ms, ns], ref, f"pairs {M}x{N}x{K}")


def test_pair_accumulate(dg):
    M, N, K = 2048, 3072, 1024
    a = dg_inputs.make_a(M, K, seed=3)
    b = dg_inputs.make_b(1, N, K, seed=4)
    C = torch.from_numpy(dg_inputs.draw(5, 0, M * N).reshape(M, N).astype(np.float32)).cuda()
    A, sA, B, sB = dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0])

    def run():
        D = C.clone()
        dg.dg_fp8_gemm_nt_acc_f32(A, sA, B, sB, D, D)
        torch.cuda.synchronize()
        return D.cpu()

    on, off = _paired_and_single(dg, run)
    assert torch.equal(on.view(torch.int32), off.view(torch.int32))


def _contiguous_indices():
    """13 row blocks of 128: g0 | g1 g1 | g2 (100 rows + padding) | padding | g4 g4 g4 | padding
    padding | g5 (30 rows) | g6 g6. Pairs (0,1), (2,3) and (10,11) straddle two groups; (4,5) is
    padding and g4; (6,7) is g4 alone; (8,9) is all padding; block 12 is the odd last one (its pair's
    second block lies past M)."""
    idx = []
    def block(g, valid=128):
        idx.extend([g] * valid + [-1] * (128 - valid))
    block(0); block(1); block(1); block(2, 100); block(-1, 0); block(4); block(4); block(4)
    block(-1, 0); block(-1, 0); block(5, 30); block(6); block(6)
    return np.array(idx, np.int32)


def test_pair_contiguous(dg):
    m_idx = _contiguous_indices()
    M, N, K, G = len(m_idx), 2048, 1024, 7
    a = dg_inputs.make_a(M, K, seed=21)
    b = dg_inputs.make_b(G, N, K, seed=22)
    A, sA, B, sB, I = dev(a.A), dev(a.sA), dev(b.B), dev(b.sB), dev(m_idx)

    def run():
        D = bf16_sentinel((M, N))
        D32 = f32_sentinel((M, N))
        dg.dg_fp8_grouped_contiguous(A, sA, B, sB, I, D)
        dg.dg_fp8_grouped_contiguous_f32(A, sA, B, sB, I, D32)
        torch.cuda.synchronize()
        return bits16(D).cpu(), D32.cpu()

    prev = dg.dg_set_pair_b(True)
    try:
        assert dg.dg_query_config(1, M, N, K, G)["block_m"] == 256
    finally:
        dg.dg_set_pair_b(prev)
    (d_on, f_on), (d_off, f_off) = _paired_and_single(dg, run)
    assert dg.dg_get_device_status() == 0
    assert torch.equal(f_on.view(torch.int32), f_off.view(torch.int32)), "FP32 differs with pairs"
    assert torch.equal(d_on, d_off)
    pad = m_idx < 0
    assert torch.all(d_on[torch.from_numpy(pad)] == -1), "padding rows were written"
    ref, _, _ = oracle.grouped_contiguous(a.A, a.sA, b.B, b.sB, m_idx)
    v = ~pad
    assert_accurate(f_on.numpy()[v], d_on.numpy()[v], ref[v], "pairs contiguous")
