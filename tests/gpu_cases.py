"""Helpers shared by the GPU parity tests: run one C-ABI call on seeded inputs
and the matching oracle computation. Every input comes from the seeded
generator (or a numpy RNG seeded here); the oracle never sees a value the
CUDA path produced.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

import oracle.spc_oracle as O
from oracle.checks import SCORE_RTOL, max_rel_err, selection_within_tie_band
from sparse_kv_cache_retrieval_gb300 import binding as spc
from sparse_kv_cache_retrieval_gb300.configs import Workload
from sparse_kv_cache_retrieval_gb300.synth import make_inputs

DEV = "cuda"


def workload(name="t", B=1, lens=(300,), H=256, n_q=8, n_kv=2, budget=96, n_layers=1, steps=1,
             cap=None, append=False, hot_frac=0.01, seed=0, n_sink=4, n_recent=64, rho=0.9,
             gpu_layers=None):
    lens = tuple(lens)
    cap = cap if cap is not None else max(max(lens), 1, budget) + (steps if append else 0)
    return Workload(name=name, B=B, lens=lens, H=H, n_q=n_q, n_kv=n_kv, d=128, budget=budget,
                    n_layers=n_layers, gpu_layers=tuple(gpu_layers or (0,) * B), steps=steps,
                    rho=(rho,) * B, hot=tuple(max(1, int(hot_frac * L)) for L in lens), seed=seed,
                    append=append, cap=cap, n_sink=n_sink, n_recent=n_recent)


def u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)


class ScoreRun:
    """GPU spc_score_select on a workload's inputs, one call per head input."""

    def __init__(self, cfg: Workload, inputs=None):
        self.cfg = cfg
        self.inp = inputs if inputs is not None else make_inputs(cfg, steps=cfg.steps, n_layers=1)
        c = cfg
        self.Wq, self.Wk, self.K = u16(self.inp.Wq), u16(self.inp.Wk), u16(self.inp.K_dlm)
        self.len = torch.from_numpy(self.inp.lens.astype(np.int32)).to(DEV)
        self.ws = torch.zeros(spc.spc_score_select_workspace_size(c.B, c.H, c.n_q, c.n_kv, 128, c.cap,
                                                                  c.budget), dtype=torch.uint8, device=DEV)
        self.q = torch.zeros(c.B, c.n_q, 128, dtype=torch.float32, device=DEV)
        self.scores = torch.zeros(c.B, c.n_kv, c.cap, dtype=torch.float32, device=DEV)
        self.sel = torch.full((c.B, c.n_kv, c.budget), -7, dtype=torch.int32, device=DEV)

    def call(self, t: int, append: int):
        c = self.cfg
        x = u16(self.inp.x[t])
        spc.spc_score_select(x, self.Wq, self.Wk if append else None, self.K, self.len, append, c.B,
                             c.H, c.n_q, c.n_kv, 128, c.cap, c.budget, c.n_sink, c.n_recent, self.q,
                             self.scores, self.sel, self.ws)
        torch.cuda.synchronize()
        return (self.q.cpu().numpy().astype(np.float64), self.scores.cpu().numpy(),
                self.sel.cpu().numpy(), self.len.cpu().numpy(), self.K.cpu().numpy().view(np.uint16))

    def status(self) -> int:
        return int(self.ws[:4].view(torch.int32).item())


def oracle_score(cfg: Workload, K_bits: np.ndarray, lens, x_bits, Wq, Wk, append: bool):
    """Oracle q, k_new, per-request group scores and selections on its own cache."""
    q, k_new = O.project(x_bits, Wq, Wk if append else None, cfg.n_q, cfg.n_kv, 128)
    lens = [int(v) for v in lens]
    K = K_bits
    if append:
        K = K_bits.copy()
        for b in range(cfg.B):
            if lens[b] < cfg.cap:
                K[b, :, lens[b]] = k_new[b]
                lens[b] += 1
    s_all, sel_all = [], []
    for b in range(cfg.B):
        P = O.head_probabilities(q[b], K[b], lens[b])
        s = O.group_scores(P, cfg.n_kv)
        s_all.append(s)
        sel_all.append([O.select(s[g], cfg.budget, cfg.n_sink, cfg.n_recent) for g in range(cfg.n_kv)])
    return q, k_new, K, lens, s_all, sel_all


def check_score_call(cfg, gq, gscores, gsel, glen, oq, olens, os_all, osel_all, q_atol=None):
    """Assert q, scores and selections of one call; returns the tie-band swap count."""
    # q: fp32 accumulation of H bf16 products vs exact: |err| <= H * 2^-23 * sum|x w|
    scale = np.abs(oq).max() + 1e-30
    assert np.abs(gq - oq).max() <= (q_atol if q_atol is not None else 1e-5 * scale), "projection"
    assert list(glen) == list(olens), "len update"
    swaps = 0
    for b in range(cfg.B):
        L = olens[b]
        err = max_rel_err(gscores[b, :, :L], os_all[b], floor=1e-30)
        assert err <= SCORE_RTOL, f"scores b={b}: max rel err {err:.3g}"
        for g in range(cfg.n_kv):
            ok, sw, msg = selection_within_tie_band(gsel[b, g], osel_all[b][g], os_all[b][g], cfg.budget,
                                                    cfg.n_sink, cfg.n_recent)
            assert ok, f"selection b={b} g={g}: {msg}"
            swaps += sw
    return swaps
