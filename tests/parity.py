"""Parity rules between the CUDA path and the fp64 oracle.

* scores: |gpu - oracle| <= 2e-3 * max(|oracle|, 1e-3 * max_row |oracle|) on
  visible positions (scores are >= 0 when w >= 0, so the floor guards values
  near 0); exactly -inf after the query's position.
* top-k: same count; every position in the symmetric difference has an oracle
  score within 1e-4 relative of the oracle's k-th score tau (a boundary tie,
  counted and reported); indices ascending, -1 only as trailing padding.
* attention: on the bf16 output against fp64, max-abs <= 2e-2 and
  mean-abs <= 2e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

SCORE_RTOL = 2e-3
SCORE_FLOOR = 1e-3
TIE_RTOL = 1e-4
ATTN_MAX_ABS = 2e-2
ATTN_MEAN_ABS = 2e-3


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact fp64 copy of a CPU/GPU tensor (bf16 through its bit pattern)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))
    return t.double().numpy()


def check_scores_row(gpu: np.ndarray, ora: np.ndarray, pos: int) -> float:
    T = ora.shape[0]
    L = min(pos + 1, T)
    g, o = gpu[:L], ora[:L]
    assert np.all(np.isfinite(g)), "non-finite score at a visible position"
    floor = SCORE_FLOOR * (np.abs(o).max() if L else 0.0)
    tol = SCORE_RTOL * np.maximum(np.abs(o), floor)
    err = np.abs(g - o)
    bad = np.nonzero(err > tol)[0]
    assert bad.size == 0, f"{bad.size} scores out of tolerance, first at s={bad[:5]}: gpu={g[bad[:5]]} ora={o[bad[:5]]}"
    assert np.all(np.isneginf(gpu[L:])), "masked positions must be -inf"
    return float((err / np.maximum(np.abs(o), floor if floor > 0 else 1.0)).max()) if L else 0.0


def check_topk_row(gpu_idx: np.ndarray, ora_idx: np.ndarray, ora_scores: np.ndarray, pos: int, k: int) -> int:
    """Returns the number of boundary ties (positions in the symmetric difference)."""
    L = min(pos + 1, ora_scores.shape[0])
    n = min(k, L)
    g = gpu_idx[:n]
    assert np.all(gpu_idx[n:] == -1), "padding must be -1"
    assert np.all(g >= 0) and np.all(g < L), "index outside the visible range"
    assert np.all(np.diff(g) > 0), "indices must be strictly ascending"
    o = ora_idx[:n]
    diff = np.setxor1d(g, o)
    if diff.size == 0:
        return 0
    tau = ora_scores[o].min()
    dev = np.abs(ora_scores[diff] - tau)
    assert np.all(dev < TIE_RTOL * abs(tau)), (
        f"{diff.size} index mismatches, not all boundary ties: tau={tau}, worst rel dev={dev.max() / abs(tau):.3g}")
    return int(diff.size)


def check_attention(gpu: np.ndarray, ora: np.ndarray) -> tuple:
    err = np.abs(gpu - ora)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= ATTN_MAX_ABS, f"max-abs error {mx:.3g} > {ATTN_MAX_ABS}"
    assert mean <= ATTN_MEAN_ABS, f"mean-abs error {mean:.3g} > {ATTN_MEAN_ABS}"
    return mx, mean
