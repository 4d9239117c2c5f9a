"""GPU parity of the batch-level selection (spc_batch_select) against the
oracle's `batch_level_select`, on seeded group scores given to both sides.

Bar: the selection equals the oracle's except swaps inside the 2e-3 tie band
of the K-th merged score (the kernel ranks the merged score after a
log2 / exp2 round trip in fp32), identical for every KV head of a request.
"""
import numpy as np
import pytest
import torch

import oracle.spc_oracle as O
from oracle.checks import selection_within_tie_band
from sparse_kv_cache_retrieval_gb300 import binding as spc

from tests import swap_log  # noqa: E402

pytestmark = pytest.mark.gpu


def _case(lens, n_kv, budget, cap=None, seed=0, n_sink=4, n_recent=64, equal=False):
    rng = np.random.default_rng(seed)
    B = len(lens)
    cap = cap or max(max(lens), budget)
    s = (rng.random((B, n_kv, cap)) ** 6).astype(np.float32)
    if equal:
        s[:] = np.float32(0.25)
    scores = torch.from_numpy(s).cuda()
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    sel = torch.full((B, n_kv, budget), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(spc.spc_batch_select_workspace_size(B, cap, budget), dtype=torch.uint8, device="cuda")
    spc.spc_batch_select(scores, ln, B, n_kv, cap, budget, n_sink, n_recent, sel, ws)
    torch.cuda.synchronize()
    g = sel.cpu().numpy()
    for b, L in enumerate(lens):
        sg = s[b, :, :L].astype(np.float64)
        want = O.batch_level_select(sg, budget, n_sink, n_recent)
        merged = sg.max(axis=0)
        for kv in range(n_kv):
            assert np.array_equal(g[b, kv], g[b, 0]), "the same set for every KV head"
        ok, _, msg = selection_within_tie_band(g[b, 0], want, merged, budget, n_sink, n_recent)
        assert ok, f"request {b}: {msg}"
    return g


def test_batch_select_ragged_batch():
    _case([1000, 300, 50], n_kv=8, budget=128)


def test_batch_select_long_context_many_ctas():
    _case([20000], n_kv=4, budget=300, seed=3)


def test_batch_select_all_equal_scores_take_the_lowest_positions():
    g = _case([5000], n_kv=2, budget=200, seed=5, equal=True)
    assert g[0, 0].tolist() == list(range(4 + 132)) + list(range(5000 - 64, 5000))


def test_batch_select_one_group_equals_the_head_level_rule():
    _case([3000, 2000], n_kv=1, budget=256, seed=7)


def test_batch_level_pipeline_chain():
    """The decode step with batch-level retrieval against the oracle's own
    chain using the batch-level rule: the same set for every KV head, within
    the tie band of the oracle's merged scores; the chain continues from the
    GPU's set, so slot maps match and attention is within the bar at every
    step; the head-level selection of the same step is kept beside it and
    matches the head-level rule."""
    import math
    from oracle.checks import ATTN_ATOL
    from sparse_kv_cache_retrieval_gb300.configs import CONFIGS, scaled
    from sparse_kv_cache_retrieval_gb300.pipeline import DecodePipeline
    from sparse_kv_cache_retrieval_gb300.synth import fill_llm_kv, make_inputs
    cfg = scaled(CONFIGS["cfg2"], lens=(6000,), n_layers=2, steps=3, budget=512)
    L = 2
    inp = make_inputs(cfg, steps=3, n_layers=L)
    pipe = DecodePipeline(cfg, inp, n_layers=L, layers_per_launch=2, retrieval="batch")
    stores = []
    for b in range(cfg.B):
        st = np.empty((L, 2, cfg.n_kv, cfg.cap, cfg.d), np.uint16)
        fill_llm_kv(cfg, b, 0, st)
        stores.append(st)
    ost = O.DecodeState(inp.K_dlm, inp.lens, stores, pipe.gpu_layers, cfg.budget, cfg.n_sink, cfg.n_recent)

    def batch_sel(ss):
        return [[O.batch_level_select(ss[b], cfg.budget, cfg.n_sink, cfg.n_recent)] * cfg.n_kv
                for b in range(cfg.B)]

    tid = "batch-level chain"

    def adopt(g, osel, oss, where):
        # the GPU's batch-level set, within the tie band of the oracle's merged
        # scores, is the one the chain continues from
        out = []
        for b in range(cfg.B):
            merged = np.max(np.stack(oss[b]), axis=0)
            ok, sw, msg = selection_within_tie_band(g[b, 0], osel[b][0], merged, cfg.budget, cfg.n_sink,
                                                    cfg.n_recent)
            assert ok, f"{where}: {msg}"
            swap_log.record(tid, sw, 1, 1 if sw else 0)
            for kv in range(cfg.n_kv):
                assert np.array_equal(g[b, kv], g[b, 0])
            out.append([g[b, 0][g[b, 0] >= 0].astype(np.int64)] * cfg.n_kv)
        return out

    _, _, _, oss, ohead = ost.score_select(inp.x[0], inp.Wq, inp.Wk, cfg.n_q, False)
    pipe.prologue()
    ost.diff_and_gather(adopt(pipe.selected[0].cpu().numpy(), batch_sel(oss), oss, "prologue"))
    for t in range(3):
        pn = (t + 1) % 2
        pipe.step(t)
        pipe.join()
        torch.cuda.synchronize()
        _, _, _, oss, ohead = ost.score_select(inp.x[t + 1], inp.Wq, inp.Wk, cfg.n_q, False)
        oout = ost.attention(inp.q_llm[t, :L], 1 / math.sqrt(cfg.d))
        g = pipe.selected[pn].cpu().numpy()
        gh = pipe.selected_head[pn].cpu().numpy()
        ost.diff_and_gather(adopt(g, batch_sel(oss), oss, f"t={t}"))
        for b in range(cfg.B):
            for kv in range(cfg.n_kv):
                okh, _, msgh = selection_within_tie_band(gh[b, kv], ohead[b][kv], oss[b][kv], cfg.budget,
                                                         cfg.n_sink, cfg.n_recent)
                assert okh, f"t={t} head-level kv={kv}: {msgh}"
            assert float(np.abs(pipe.out.cpu().numpy()[:, b] - oout[:, b]).max()) <= ATTN_ATOL
            assert np.array_equal(pipe.slot_pos[pn].cpu().numpy()[b], ost.slot_pos[b])
