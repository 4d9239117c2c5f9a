"""GPU parity of the whole decode step (two streams, all four calls) against
the oracle, plus graph-vs-eager and host-I/O equivalence.

Every step the oracle computes its own selection, and the GPU's must equal
it up to tie-band swaps (positions whose oracle scores lie within 2e-3 of the
oracle's K-th score; counted and reported in the terminal summary). Several
selections are then correct, so the chain continues from the one the GPU
made: the oracle's diff, gather and attention take it as their input, and the
GPU's load lists, slot maps and slot contents must match the oracle's bit for
bit and its attention within tolerance, for every KV head at every step (a
swap never switches a check off).
"""
import math

import numpy as np
import pytest
import torch

import oracle.spc_oracle as O
from oracle.checks import ATTN_ATOL
from sparse_kv_cache_retrieval_gb300.configs import CONFIGS, scaled
from sparse_kv_cache_retrieval_gb300.pipeline import DecodePipeline
from sparse_kv_cache_retrieval_gb300.synth import fill_llm_kv, make_inputs
from tests import swap_log

pytestmark = pytest.mark.gpu


def oracle_stores(cfg, L):
    stores = []
    for b in range(cfg.B):
        st = np.empty((L, 2, cfg.n_kv, cfg.cap, cfg.d), np.uint16)
        fill_llm_kv(cfg, b, 0, st)
        stores.append(st)
    return stores


def run_chain(cfg, steps, L, layers_per_launch=1, on_step=None, test_id=None, **pipe_kw):
    tid = test_id or cfg.name
    inp = make_inputs(cfg, steps=steps, n_layers=L)
    pipe = DecodePipeline(cfg, inp, n_layers=L, layers_per_launch=layers_per_launch, **pipe_kw)
    stores = oracle_stores(cfg, L)
    ost = O.DecodeState(inp.K_dlm, inp.lens, stores, pipe.gpu_layers, cfg.budget, cfg.n_sink,
                        cfg.n_recent)
    _, _, _, oss, osel = ost.score_select(inp.x[0], inp.Wq, inp.Wk, cfg.n_q, append=False)
    pipe.prologue()
    swaps_total = 0
    # the prologue's selection S_0 is held to the same tie band; the chain
    # continues from the GPU's (valid) choice
    sel, sw = swap_log.check_selection(tid, pipe.selected[0].cpu().numpy(), osel, oss, cfg.budget, cfg.n_sink,
                                       cfg.n_recent, "prologue")
    swaps_total += sw
    ost.diff_and_gather(sel)
    scale = 1 / math.sqrt(cfg.d)
    for t in range(steps):
        p, pn = t % 2, (t + 1) % 2
        pipe.step(t)
        pipe.join()
        torch.cuda.synchronize()
        if on_step is not None:
            on_step(t, pipe)
        _, _, _, oss, osel = ost.score_select(inp.x[t + 1], inp.Wq, inp.Wk, cfg.n_q, append=cfg.append)
        # attention of step t runs over S_t, the selection the previous step adopted
        oout = ost.attention(inp.q_llm[t, :L], scale)
        gsel = pipe.selected[pn].cpu().numpy()
        sel, sw = swap_log.check_selection(tid, gsel, osel, oss, cfg.budget, cfg.n_sink, cfg.n_recent, f"t={t}")
        swaps_total += sw
        loads = ost.diff_and_gather(sel)
        gslot = pipe.slot_pos[pn].cpu().numpy()
        gnl = pipe.n_load[pn].cpu().numpy()
        gls = pipe.load_slot[pn].cpu().numpy()
        glp = pipe.load_pos[pn].cpu().numpy()
        gout = pipe.out.cpu().numpy()
        assert pipe.len.cpu().numpy().tolist() == ost.lens
        e = np.abs(gout - oout)
        assert e.max() <= ATTN_ATOL, f"t={t}: attention max err {e.max():.3g}"
        assert np.all(e <= 2e-5 + 1e-4 * np.abs(oout)), f"t={t}: attention"
        for b in range(cfg.B):
            for g in range(cfg.n_kv):
                ls, lp = loads[b][g]
                assert gnl[b, g] == lp.size, f"t={t} b={b} g={g} n_load"
                assert np.array_equal(glp[b, g, :lp.size], lp) and np.array_equal(gls[b, g, :ls.size], ls)
                assert np.array_equal(gslot[b, g], ost.slot_pos[b, g]), f"t={t} b={b} g={g} slot map"
        # slots hold the rows their slot map names, byte for byte (host layers)
        for b in range(cfg.B):
            if pipe.host_slots(b) is None:
                continue
            sl = pipe.host_slots(b).cpu().numpy().view(np.uint16)
            h0 = pipe.gpu_layers[b]
            for g in range(cfg.n_kv):
                held = gslot[b, g]
                idx = np.nonzero(held >= 0)[0]
                assert np.array_equal(sl[:, :, g, idx], stores[b][h0:, :, g, held[idx]]), \
                    f"t={t} b={b} g={g} slot contents"
    return swaps_total, pipe


def test_chain_cfg1_full_size():
    cfg = CONFIGS["cfg1"]
    run_chain(cfg, cfg.steps, cfg.n_layers)


def test_chain_cfg4a_append_select_all_then_topk():
    cfg = scaled(CONFIGS["cfg4a"], B=2, n_layers=2, steps=4, lens=(2046, 2047))
    swaps, pipe = run_chain(cfg, 4, 2, layers_per_launch=2)
    assert pipe.len.cpu().tolist() == [2050, 2051]


def test_chain_cfg3_ragged_hbm_host_split():
    cfg = scaled(CONFIGS["cfg3"], n_layers=2, steps=2)
    assert any(g == 2 for g in cfg.gpu_layers) and any(g == 0 for g in cfg.gpu_layers)
    run_chain(cfg, 2, 2, layers_per_launch=2)


def test_chain_cfg2_shape_two_layers():
    cfg = scaled(CONFIGS["cfg2"], n_layers=3, steps=3)
    run_chain(cfg, 3, 3, layers_per_launch=2)


def test_chain_cfg4b_128k_context_append_full_shape():
    # full cfg4b shapes (4 requests at 131072 positions, capacity 131328,
    # budget 2048, appending) on two host layers and two steps
    cfg = scaled(CONFIGS["cfg4b"], n_layers=2, steps=2)
    assert cfg.cap == 131072 + 256
    swaps, pipe = run_chain(cfg, 2, 2, layers_per_launch=2)
    assert pipe.len.cpu().tolist() == [131074] * 4


def test_chain_cfg5_70b_shape_hbm_and_host_layers():
    # full cfg5 shapes (8 requests x 65536 positions, 64/8 heads, H 8192,
    # budget 4096): layer 0 resident in HBM (attention by position), layer 1
    # through the host slots
    cfg = scaled(CONFIGS["cfg5"], n_layers=2, steps=1)
    assert cfg.gpu_layers == (1,) * 8
    run_chain(cfg, 1, 2, layers_per_launch=2)


def test_chain_shared_host_stores():
    # cfg5's layout on a small context: requests b and b + 2 hold the same
    # K/V contents and share one pinned store, yet each selects, diffs and
    # gathers its own positions into its own slots
    cfg = scaled(CONFIGS["cfg5"], B=4, lens=(3000, 2900, 3000, 2800), n_layers=3, steps=2, budget=512, H=1024)
    assert cfg.host_store_copies == 2 and cfg.kv_source(2) == 0 and cfg.kv_source(3) == 1
    swaps, pipe = run_chain(cfg, 2, 3, layers_per_launch=2)
    assert pipe.host_stores[2] is pipe.host_stores[0] and pipe.host_stores[3] is pipe.host_stores[1]
    assert pipe.host_stores[1] is not pipe.host_stores[0]
    assert pipe.slots[2] is not pipe.slots[0]


def test_chain_cfg5_mqa_full_shape():
    cfg = scaled(CONFIGS["cfg5mqa"], n_layers=2, steps=1)
    run_chain(cfg, 1, 2, layers_per_launch=2)


def test_chain_mqa_short_last_chunk():
    # 64 heads on one KV head, a 16-layer chunk and a last chunk of 1: the
    # 1-layer launch splits its segments over several CTAs (and needs merge
    # workspace), the 16-layer launch keeps whole segments (and needs none)
    cfg = scaled(CONFIGS["cfg5mqa"], B=8, lens=(1000,) * 8, n_layers=17, steps=2, budget=256, H=1024)
    run_chain(cfg, 2, 17, layers_per_launch=16)


def _growing_small(steps=8):
    from tests.gpu_cases import workload
    return workload(name="c3_small", B=2, lens=(100, 98), H=256, n_q=8, n_kv=2, budget=96, n_layers=4,
                    steps=steps, append=True)


@pytest.mark.parametrize("policy", ["progressive", "static"])
def test_chain_adaptive_offload_crosses_thresholds(policy):
    # adaptive memory management: a growing context crosses the memory model's
    # thresholds during the run; every step still matches the oracle (selections,
    # load lists, slot maps and contents, attention), the number of offloaded
    # layers follows the rule at every step, and the last layers go first
    cfg = _growing_small()
    L, B = 4, cfg.B
    row = 2 * cfg.n_kv * 128 * 2
    kv_bytes = B * 408 * row
    thr = O.offload_thresholds(L, cfg.n_kv, 128, B, cfg.budget, kv_bytes)
    assert thr[:3] == [103, 105, 109]
    seen = []

    def on_step(t, pipe):
        for b in range(B):
            length = int(cfg.lens[b]) + t + 1
            n_off = L - pipe.gpu_layers[b]
            if policy == "progressive":
                assert n_off == O.layers_to_offload(length, thr, 0)
                assert O.gpu_kv_bytes(length, n_off, L, cfg.n_kv, 128, B, cfg.budget) <= kv_bytes
            else:
                assert n_off == (L if length >= thr[0] else 0)
        seen.append([L - g for g in pipe.gpu_layers])

    swaps, pipe = run_chain(cfg, 8, L, layers_per_launch=2, on_step=on_step, kv_bytes=kv_bytes,
                            offload_policy=policy)
    moved = [(b, l) for (_, b, l) in pipe.offload_log]
    for b in range(B):
        layers = [l for (bb, l) in moved if bb == b]
        assert layers == sorted(layers, reverse=True)          # last layers first
        assert layers == list(range(L - 1, L - 1 - len(layers), -1))
    assert seen[-1] != seen[0]                                  # something moved during the run


def test_full_reload_mode_loads_every_selected_row_and_matches_elastic():
    # the baseline elastic loading is measured against: each step reloads its
    # whole selection; selections and attention outputs are those of the
    # elastic path, only the traffic differs
    cfg = scaled(CONFIGS["cfg1"], steps=4)
    inp = make_inputs(cfg, steps=4)
    a = DecodePipeline(cfg, inp, layers_per_launch=1)
    b = DecodePipeline(cfg, inp, layers_per_launch=1, elastic=False)
    a.prologue()
    b.prologue()
    for t in range(4):
        for p_ in (a, b):
            p_.step(t)
            p_.join()
        torch.cuda.synchronize()
        pn = (t + 1) % 2
        assert torch.equal(a.selected[pn], b.selected[pn])
        n_sel = (b.selected[pn] >= 0).sum(dim=2)
        assert torch.equal(b.n_load[pn], n_sel.to(torch.int32))
        assert int(a.n_load[pn].sum()) < int(b.n_load[pn].sum())
        assert (a.out - b.out).abs().max().item() <= 2e-5


def _state(pipe):
    return [pipe.out.cpu(), pipe.selected.cpu(), pipe.slot_pos.cpu(), pipe.len.cpu()] + \
        [s.cpu() for s in pipe.slots if s is not None]


def test_graph_replay_equals_eager():
    cfg = scaled(CONFIGS["cfg1"], steps=4)
    inp = make_inputs(cfg, steps=4)
    a = DecodePipeline(cfg, inp, layers_per_launch=1)
    a.prologue()
    a.run(0, 4)
    torch.cuda.synchronize()
    b = DecodePipeline(cfg, inp, layers_per_launch=1)
    b.prologue()
    g = b.capture(0, 4)
    g.replay()
    torch.cuda.synchronize()
    for u, v in zip(_state(a), _state(b)):
        assert torch.equal(u, v)


def test_host_io_matches_device_resident():
    cfg = scaled(CONFIGS["cfg1"], steps=3)
    inp = make_inputs(cfg, steps=3)
    a = DecodePipeline(cfg, inp)
    a.prologue()
    outs = []
    for t in range(3):
        a.step(t)
        a.join()
        torch.cuda.synchronize()
        outs.append(a.out.cpu().clone())
    b = DecodePipeline(cfg, inp, host_io=True)
    b.prologue()
    b.run(0, 3)
    torch.cuda.synchronize()
    for t in range(3):
        assert torch.equal(b.out_host[t], outs[t])


def test_front_after_attention_gives_the_same_steps():
    """Issuing the next step's projection and key scan after the last
    attention instead of after the select changes only the schedule."""
    cfg = scaled(CONFIGS["cfg2"], n_layers=4, steps=4)
    inp = make_inputs(cfg, steps=4, n_layers=4)
    a = DecodePipeline(cfg, inp, n_layers=4, layers_per_launch=2)
    a.prologue()
    a.run(0, 4)
    torch.cuda.synchronize()
    b = DecodePipeline(cfg, inp, n_layers=4, layers_per_launch=2, front_after="attention")
    b.prologue()
    g = b.capture(0, 4)
    g.replay()
    torch.cuda.synchronize()
    for u, v in zip(_state(a), _state(b)):
        assert torch.equal(u, v)
