"""Tie-band swap counts of the GPU parity tests, printed in pytest's terminal
summary (kept with -q, unlike print()).

A swap is a position that the GPU selection holds and the oracle's does not,
allowed when every position of the symmetric difference scores within 2e-3
(relative) of the oracle's K-th score.
"""
from __future__ import annotations

from typing import Dict, List

import numpy as np

from oracle.checks import selection_within_tie_band

# test id -> [swapped positions, selections checked, selections with a swap]
COUNTS: Dict[str, List[int]] = {}


def record(test_id: str, swaps: int, checked: int, heads_swapped: int) -> None:
    c = COUNTS.setdefault(test_id, [0, 0, 0])
    c[0] += swaps
    c[1] += checked
    c[2] += heads_swapped


def check_selection(test_id: str, gsel: np.ndarray, osel, oss, budget: int, n_sink: int, n_recent: int,
                    where: str = ""):
    """Check the GPU's selections [B][n_kv][budget] against the oracle's within
    the tie band; record the swaps; return the GPU's selections as the lists
    of positions a chain continues from (the oracle's own when they agree)."""
    B, n_kv = gsel.shape[:2]
    swaps = heads = 0
    adopted = []
    for b in range(B):
        row = []
        for g in range(n_kv):
            ok, sw, msg = selection_within_tie_band(gsel[b, g], osel[b][g], oss[b][g], budget, n_sink, n_recent)
            assert ok, f"{where} b={b} g={g}: {msg}"
            swaps += sw
            heads += 1 if sw else 0
            row.append(np.asarray(osel[b][g]) if sw == 0 else gsel[b, g][gsel[b, g] >= 0].astype(np.int64))
        adopted.append(row)
    record(test_id, swaps, B * n_kv, heads)
    return adopted, swaps
