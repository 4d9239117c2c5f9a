"""Comparison rules between the CUDA path's outputs and the oracle's --
TEST INFRASTRUCTURE ONLY (tests, smoke, benchmark baseline).

Plain numpy on arrays the caller passes in; nothing here computes a step of
the method.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

SCORE_RTOL = 2e-3   # group scores (probabilities), relative
ATTN_ATOL = 1e-2    # attention output, absolute (the stated bar)


def forced_mask(length: int, n_sink: int, n_recent: int) -> np.ndarray:
    m = np.zeros(length, bool)
    m[:min(n_sink, length)] = True
    m[max(0, length - n_recent):] = True
    return m


def selection_within_tie_band(gpu_sel: np.ndarray, ora_sel: np.ndarray, ora_scores: np.ndarray,
                              budget: int, n_sink: int, n_recent: int,
                              rtol: float = SCORE_RTOL) -> Tuple[bool, int, str]:
    """GPU and oracle selections of one KV head agree up to tie-band swaps.

    gpu_sel: int [budget] (ascending, -1 padded); ora_sel: the oracle's
    ascending selection; ora_scores: oracle group scores [len]. Every position
    in the symmetric difference must score within rtol of the oracle's K-th
    (smallest non-forced kept) score. Returns (ok, swaps, message).
    """
    length = ora_scores.shape[0]
    g = np.asarray(gpu_sel)
    n = min(budget, length)
    if np.any(g[n:] != -1):
        return False, 0, "padding is not -1"
    g = g[:n]
    if np.any(np.diff(g) <= 0):
        return False, 0, "not strictly ascending"
    if np.any(g < 0) or np.any(g >= max(length, 1)):
        return False, 0, "position out of range"
    o = np.asarray(ora_sel)
    if len(o) != n:
        return False, 0, "oracle size mismatch"
    if np.array_equal(g, o):
        return True, 0, ""
    fm = forced_mask(length, n_sink, n_recent)
    if not np.all(np.isin(np.nonzero(fm)[0], g)) and length > budget:
        return False, 0, "forced position missing"
    kept_nf = o[~fm[o]]
    tau = ora_scores[kept_nf].min() if kept_nf.size else 0.0
    diff = np.setxor1d(g, o)
    dev = np.abs(ora_scores[diff] - tau)
    ok = bool(np.all(dev <= rtol * abs(tau)))
    swaps = int(np.setdiff1d(g, o).size)
    msg = "" if ok else f"{swaps} swaps outside the tie band (max rel dev {np.max(dev) / max(abs(tau), 1e-300):.3g})"
    return ok, swaps, msg


def max_rel_err(a: np.ndarray, b: np.ndarray, floor: float = 0.0) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.maximum(np.abs(b), floor)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(den > 0, np.abs(a - b) / den, np.abs(a - b))
    return float(r.max()) if r.size else 0.0


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in units in the last place between bf16 bit patterns of equal sign."""
    a = np.asarray(a_bits, np.uint16).astype(np.int32)
    b = np.asarray(b_bits, np.uint16).astype(np.int32)
    def ordered(x):
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)
    return np.abs(ordered(a) - ordered(b))
