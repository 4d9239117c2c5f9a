"""Parity at the benchmark's full sizes and in its launch configuration: every
layer of the workload, the layer chunk and schedule bench.py times, two
decode steps; the oracle recomputes the selections and the attention of a
sample of the layers (the attention of a layer depends only on that layer's
rows and the selection, so the oracle holds the sampled layers only)."""
import math

import numpy as np
import pytest
import torch

import oracle.mla_oracle as M
import oracle.spc_oracle as O
from oracle.checks import ATTN_ATOL, selection_within_tie_band
from sparse_kv_cache_retrieval_gb300.configs import CONFIGS
from sparse_kv_cache_retrieval_gb300.pipeline import DecodePipeline
from sparse_kv_cache_retrieval_gb300.synth import fill_llm_kv, fill_mla_layer, make_inputs, make_mla_inputs

pytestmark = pytest.mark.gpu


def test_cfg2_all_layers_bench_launch_configuration():
    cfg = CONFIGS["cfg2"]
    steps, sample = 2, [0, 15, 16, 31]
    inp = make_inputs(cfg, steps=steps)
    pipe = DecodePipeline(cfg, inp, layers_per_launch=cfg.layers_per_launch)
    assert pipe.L == 32 and pipe.front_after == cfg.front_after
    stores = []
    for b in range(cfg.B):
        st = np.empty((len(sample), 2, cfg.n_kv, cfg.cap, cfg.d), np.uint16)
        for i, l in enumerate(sample):
            fill_llm_kv(cfg, b, l, st[i:i + 1])
        stores.append(st)
    ost = O.DecodeState(inp.K_dlm, inp.lens, stores, [0] * cfg.B, cfg.budget, cfg.n_sink, cfg.n_recent)
    _, _, _, oss, osel = ost.score_select(inp.x[0], inp.Wq, inp.Wk, cfg.n_q, False)
    ost.diff_and_gather(osel)
    pipe.prologue()
    swapped = np.zeros((cfg.B, cfg.n_kv), bool)
    g0 = pipe.selected[0].cpu().numpy()
    for g in range(cfg.n_kv):
        ok, sw, msg = selection_within_tie_band(g0[0, g], osel[0][g], oss[0][g], cfg.budget, cfg.n_sink, cfg.n_recent)
        assert ok, msg
        swapped[0, g] |= sw > 0
    for t in range(steps):
        pn = (t + 1) % 2
        pipe.run(t, 1)
        torch.cuda.synchronize()
        _, _, _, oss, osel = ost.score_select(inp.x[t + 1], inp.Wq, inp.Wk, cfg.n_q, False)
        oout = ost.attention(inp.q_llm[t][sample], 1 / math.sqrt(cfg.d))
        ost.diff_and_gather(osel)
        gout = pipe.out.cpu().numpy()[sample]
        gsel = pipe.selected[pn].cpu().numpy()
        for g in range(cfg.n_kv):
            hs = slice(g * cfg.G, (g + 1) * cfg.G)
            if not swapped[0, g]:
                assert float(np.abs(gout[:, 0, hs] - oout[:, 0, hs]).max()) <= ATTN_ATOL, f"t={t} g={g}"
            ok, sw, msg = selection_within_tie_band(gsel[0, g], osel[0][g], oss[0][g], cfg.budget, cfg.n_sink,
                                                    cfg.n_recent)
            assert ok, f"t={t} g={g}: {msg}"
            swapped[0, g] |= sw > 0
            if not swapped[0, g]:
                assert np.array_equal(pipe.slot_pos[pn].cpu().numpy()[0, g], ost.slot_pos[0, g])


def test_mla_all_layers_bench_launch_configuration():
    cfg = CONFIGS["mla"]
    steps, sample = 2, [0, 13, 26]
    inp = make_mla_inputs(cfg, steps=steps)
    pipe = DecodePipeline(cfg, inp, layers_per_launch=cfg.layers_per_launch)
    assert pipe.L == 27 and len(pipe.chunks) == 1
    stores = []
    for b in range(cfg.B):
        st = np.empty((len(sample), cfg.cap, M.D_LAT), np.uint16)
        for i, l in enumerate(sample):
            fill_mla_layer(cfg, b, l, st[i])
        stores.append(st)
    ost = M.MlaDecodeState(inp.C_dlm, inp.lens, stores, [0] * cfg.B, cfg.budget, cfg.n_sink, cfg.n_recent)
    _, _, _, oss, osel = ost.score_select(inp.x[0], inp.Wq, inp.Wuk, inp.Wdkv, cfg.n_q, False)
    ost.diff_and_gather(osel)
    pipe.prologue()
    g0 = pipe.selected[0].cpu().numpy()
    ok, sw, msg = selection_within_tie_band(g0[0, 0], osel[0][0], oss[0][0], cfg.budget, cfg.n_sink, cfg.n_recent)
    assert ok, msg
    swapped = sw > 0
    for t in range(steps):
        pn = (t + 1) % 2
        pipe.run(t, 1)
        torch.cuda.synchronize()
        _, _, _, oss, osel = ost.score_select(inp.x[t + 1], inp.Wq, inp.Wuk, inp.Wdkv, cfg.n_q, False)
        oout = ost.attention(inp.q_llm[t][sample], inp.Wuk_llm[sample], inp.Wuv_llm[sample], 1 / math.sqrt(M.D_QK))
        ost.diff_and_gather(osel)
        if not swapped:
            assert float(np.abs(pipe.out.cpu().numpy()[sample] - oout).max()) <= ATTN_ATOL, f"t={t}"
        gsel = pipe.selected[pn].cpu().numpy()
        ok, sw, msg = selection_within_tie_band(gsel[0, 0], osel[0][0], oss[0][0], cfg.budget, cfg.n_sink,
                                                cfg.n_recent)
        assert ok, f"t={t}: {msg}"
        swapped |= sw > 0
        if not swapped:
            assert np.array_equal(pipe.slot_pos[pn].cpu().numpy()[0, 0], ost.slot_pos[0, 0])
