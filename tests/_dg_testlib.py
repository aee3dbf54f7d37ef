"""Helpers shared by the GPU parity tests: device transfer, accuracy metrics, sampling.

The accuracy bar. A BF16 output cannot meet max|D - ref| / max|ref| <= 2e-3 literally: rounding an
element in the top binade to BF16's 8 significant bits already moves it by up to 2^(e-8), 1.95e-3 to
3.9e-3 of max|ref|. So the bound is applied to the FP32 accumulator, and the BF16 output is tied to it:
* the FP32 accumulator (``*_f32`` entry points) must satisfy
  max|D32 - ref64| / max|ref64| <= 2e-3 and 1 - cos(D32, ref64) <= 1e-5 against the FP64 oracle;
* the BF16 output must equal RNE(D32) bit for bit (same kernel, same accumulation order), and
  1 - cos(D_bf16, ref64) <= 1e-5;
* group/mask indexing is bit-exact: rows outside the valid region keep their sentinel bits.
"""
from __future__ import annotations

import numpy as np
import torch

MAX_REL_TOL = 2e-3
COS_TOL = 1e-5
SENTINEL_BF16_BITS = -1          # 0xFFFF as int16: a NaN pattern no kernel output produces


def dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def bf16_sentinel(shape) -> torch.Tensor:
    return torch.full(shape, SENTINEL_BF16_BITS, dtype=torch.int16, device="cuda").view(torch.bfloat16)


def f32_sentinel(shape) -> torch.Tensor:
    return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")


def bits16(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16)


def rne_bf16_bits(d32: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even of FP32 values to BF16, on the CPU for moderate sizes."""
    if d32.numel() <= (1 << 24):
        return d32.detach().cpu().to(torch.bfloat16).view(torch.int16)
    return d32.to(torch.bfloat16).view(torch.int16).cpu()


def metrics(d: np.ndarray, ref: np.ndarray) -> dict:
    d = np.asarray(d, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    scale = np.abs(ref).max()
    max_rel = float(np.abs(d - ref).max() / scale) if scale > 0 else float(np.abs(d).max())
    nd, nr = np.linalg.norm(d), np.linalg.norm(ref)
    cos = float(np.dot(d, ref) / (nd * nr)) if nd > 0 and nr > 0 else (1.0 if nd == nr else 0.0)
    return {"max_rel": max_rel, "one_minus_cos": 1.0 - cos, "finite": bool(np.all(np.isfinite(d)))}


def assert_accurate(d32: np.ndarray, d_bf16_bits: np.ndarray, ref64: np.ndarray, what: str = ""):
    m32 = metrics(d32, ref64)
    assert m32["finite"], f"{what}: non-finite FP32 output"
    assert m32["max_rel"] <= MAX_REL_TOL, f"{what}: FP32 max_rel {m32['max_rel']:.3e}"
    assert m32["one_minus_cos"] <= COS_TOL, f"{what}: FP32 1-cos {m32['one_minus_cos']:.3e}"
    dbf = torch.from_numpy(np.ascontiguousarray(d_bf16_bits).astype(np.int16)).view(torch.bfloat16)
    mbf = metrics(dbf.to(torch.float64).numpy(), ref64)
    assert mbf["one_minus_cos"] <= COS_TOL, f"{what}: BF16 1-cos {mbf['one_minus_cos']:.3e}"
    return m32, mbf


def boundary_samples(rows: int, cols: int, n_random: int, seed: int = 0, block_rows=128, block_cols=128,
                     per_tile: int = 8):
    """Random (m, n) pairs, the first/last rows and columns and tile boundaries, and `per_tile`
    elements inside every block_rows x block_cols output tile whose rows take every residue mod 8
    (so that a wrong tile, a wrong K range of a split tile, or a wrong rank's rows of a split-K
    cluster — which reduces rows r with r % S = rank, S <= 8 — is hit by some sample)."""
    rng = np.random.default_rng(seed)
    ms = list(rng.integers(0, rows, n_random))
    ns = list(rng.integers(0, cols, n_random))
    if per_tile > 0:
        tm = np.arange(0, rows, block_rows)
        tn = np.arange(0, cols, block_cols)
        th = np.minimum(block_rows, rows - tm)                 # rows of each tile row (ragged tail)
        tw = np.minimum(block_cols, cols - tn)
        tmi, tni = np.meshgrid(np.arange(len(tm)), np.arange(len(tn)), indexing="ij")
        tmi = np.repeat(tmi.ravel(), per_tile)
        tni = np.repeat(tni.ravel(), per_tile)
        res = np.tile(np.arange(per_tile) % 8, len(tm) * len(tn))   # every residue mod 8 in each tile
        r = res + 8 * rng.integers(0, np.maximum(1, th[tmi] // 8))
        ms += list(tm[tmi] + np.minimum(r, th[tmi] - 1))
        ns += list(tn[tni] + rng.integers(0, tw[tni]))
    edge_m = sorted({0, rows - 1} | {x for b in range(block_rows, rows, block_rows) for x in (b - 1, b)})
    edge_n = sorted({0, cols - 1} | {x for b in range(block_cols, cols, block_cols) for x in (b - 1, b)})
    for m in edge_m[:64]:
        for n in rng.choice(edge_n, size=min(8, len(edge_n)), replace=False):
            ms.append(m)
            ns.append(int(n))
    for n in edge_n[:64]:
        ms.append(int(rng.integers(0, rows)))
        ns.append(n)
    return np.array(ms, np.int64), np.array(ns, np.int64)
