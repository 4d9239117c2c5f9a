"""Parity at the benchmark's full sizes and in its launch configuration: every
layer of the workload, the layer chunks and schedule bench.py times, two
decode steps; the oracle recomputes the selections and the attention of a
sample of the layers (the attention of a layer depends only on that layer's
rows and the selection, so the oracle holds the sampled layers only).

Selections must equal the oracle's up to tie-band swaps (counted in the
terminal summary); the chain then continues from the GPU's valid choice, so
slot maps and the attention of every head stay checked at every step.
"""
import math

import numpy as np
import pytest
import torch

import oracle.mla_oracle as M
import oracle.spc_oracle as O
from oracle.checks import ATTN_ATOL
from sparse_kv_cache_retrieval_gb300.configs import CONFIGS
from sparse_kv_cache_retrieval_gb300.pipeline import DecodePipeline
from sparse_kv_cache_retrieval_gb300.synth import fill_llm_kv, fill_mla_layer, make_inputs, make_mla_inputs
from tests import swap_log

pytestmark = pytest.mark.gpu


def _release_pinned():
    # the pinned stores of a large workload go back to the OS, not to torch's
    # host-allocator cache, before the next test allocates its own
    torch.cuda.synchronize()
    fn = getattr(torch._C, "_host_emptyCache", None)
    if fn is not None:
        fn()


def _gqa_full_launch(key, steps, sample):
    cfg = CONFIGS[key]
    tid = f"full launch {key} ({cfg.n_layers} layers)"
    inp = make_inputs(cfg, steps=steps)
    pipe = DecodePipeline(cfg, inp, layers_per_launch=cfg.layers_per_launch)
    assert pipe.L == cfg.n_layers and pipe.front_after == cfg.front_after
    n_chunks = -(-cfg.n_layers // cfg.layers_per_launch)
    assert len(pipe.chunks) == n_chunks
    # the oracle's stores hold the sampled layers only; requests sharing
    # K/V contents share one array, as the pipeline shares one pinned store
    by_src, stores = {}, []
    for b in range(cfg.B):
        src = cfg.kv_source(b)
        if src not in by_src:
            st = np.empty((len(sample), 2, cfg.n_kv, cfg.cap, cfg.d), np.uint16)
            for i, l in enumerate(sample):
                fill_llm_kv(cfg, b, l, st[i:i + 1])
            by_src[src] = st
        stores.append(by_src[src])
    ost = O.DecodeState(inp.K_dlm, inp.lens, stores, [0] * cfg.B, cfg.budget, cfg.n_sink, cfg.n_recent)
    _, _, _, oss, osel = ost.score_select(inp.x[0], inp.Wq, inp.Wk, cfg.n_q, False)
    pipe.prologue()
    sel, _ = swap_log.check_selection(tid, pipe.selected[0].cpu().numpy(), osel, oss, cfg.budget, cfg.n_sink,
                                      cfg.n_recent, "prologue")
    ost.diff_and_gather(sel)
    for t in range(steps):
        pn = (t + 1) % 2
        pipe.run(t, 1)
        torch.cuda.synchronize()
        _, _, _, oss, osel = ost.score_select(inp.x[t + 1], inp.Wq, inp.Wk, cfg.n_q, False)
        oout = ost.attention(inp.q_llm[t][sample], 1 / math.sqrt(cfg.d))
        gout = pipe.out.cpu().numpy()[sample]
        err = np.abs(gout - oout)
        assert err.max() <= ATTN_ATOL, f"t={t}: attention max err {err.max():.3g}"
        assert np.all(err <= 2e-5 + 1e-4 * np.abs(oout)), f"t={t}: attention"
        sel, _ = swap_log.check_selection(tid, pipe.selected[pn].cpu().numpy(), osel, oss, cfg.budget, cfg.n_sink,
                                          cfg.n_recent, f"t={t}")
        ost.diff_and_gather(sel)
        assert np.array_equal(pipe.slot_pos[pn].cpu().numpy(), ost.slot_pos), f"t={t}: slot maps"
        # the slots of the sampled host layers hold the rows the slot map names
        gslot = pipe.slot_pos[pn].cpu().numpy()
        for b in (0, cfg.B - 1):
            hs = pipe.host_slots(b)
            h0 = pipe.gpu_layers[b]
            for i, l in enumerate(sample):
                if l < h0:
                    continue
                sl = hs[l - h0].cpu().numpy().view(np.uint16)
                for g in (0, cfg.n_kv - 1):
                    idx = np.nonzero(gslot[b, g] >= 0)[0]
                    assert np.array_equal(sl[:, g, idx], stores[b][i][:, g, gslot[b, g][idx]]), \
                        f"t={t} b={b} layer {l} g={g}: slot contents"
    del pipe
    _release_pinned()


def test_cfg2_all_layers_bench_launch_configuration():
    _gqa_full_launch("cfg2", 2, [0, 15, 16, 31])


def test_cfg5_all_80_layers_bench_launch_configuration():
    # the benchmark's default workload: 8 requests x 65536 positions, 64/8
    # heads, budget 4096, layer 0 in HBM and 79 host layers gathered in five
    # 16-layer chunks (each chunk's gather beside the next chunk's attention)
    _gqa_full_launch("cfg5", 2, [0, 1, 15, 16, 40, 79])


def test_cfg5_mqa_all_80_layers_bench_launch_configuration():
    # the MQA variant: all 64 query heads on one KV head (the tensor-core
    # attention, 16 layers x 8 requests x 32 tiles per launch over 152 CTAs,
    # so runs of tiles cross segment boundaries and segments merge partials)
    _gqa_full_launch("cfg5mqa", 2, [0, 1, 15, 16, 79])


def test_mla_all_layers_bench_launch_configuration():
    cfg = CONFIGS["mla"]
    tid = "full launch mla (27 layers)"
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
    pipe.prologue()
    sel, _ = swap_log.check_selection(tid, pipe.selected[0].cpu().numpy(), osel, oss, cfg.budget, cfg.n_sink,
                                      cfg.n_recent, "prologue")
    ost.diff_and_gather(sel)
    for t in range(steps):
        pn = (t + 1) % 2
        pipe.run(t, 1)
        torch.cuda.synchronize()
        _, _, _, oss, osel = ost.score_select(inp.x[t + 1], inp.Wq, inp.Wuk, inp.Wdkv, cfg.n_q, False)
        oout = ost.attention(inp.q_llm[t][sample], inp.Wuk_llm[sample], inp.Wuv_llm[sample], 1 / math.sqrt(M.D_QK))
        assert float(np.abs(pipe.out.cpu().numpy()[sample] - oout).max()) <= ATTN_ATOL, f"t={t}"
        sel, _ = swap_log.check_selection(tid, pipe.selected[pn].cpu().numpy(), osel, oss, cfg.budget, cfg.n_sink,
                                          cfg.n_recent, f"t={t}")
        ost.diff_and_gather(sel)
        assert np.array_equal(pipe.slot_pos[pn].cpu().numpy(), ost.slot_pos), f"t={t}: slot map"
