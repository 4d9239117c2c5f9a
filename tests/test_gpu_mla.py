"""GPU parity of the MLA variant against the MLA oracle, through the C ABI.

The oracle expands every selected latent row into per-head keys and values
and attends over them (the pages' wording); the CUDA path absorbs the query
into the latent space and up-projects the softmax-weighted latent sum once.
Bars: scores within 2e-3 relative; selections identical except swaps inside
the 2e-3 tie band of the K-th score; the appended latent row within 1 bf16
ulp; gathered rows bit-exact; attention within 1e-2 absolute (the bar of the
GQA path).
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle.mla_oracle as M
import oracle.spc_oracle as O
from oracle.checks import ATTN_ATOL, SCORE_RTOL, bf16_ulp_distance, max_rel_err, selection_within_tie_band
from sparse_kv_cache_retrieval_gb300 import binding as spc
from sparse_kv_cache_retrieval_gb300.configs import Workload
from sparse_kv_cache_retrieval_gb300.synth import make_mla_inputs

from tests import swap_log  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


def mla_workload(name="m", B=1, lens=(300,), H=256, budget=96, steps=1, cap=None, append=False, hot_frac=0.01,
                 seed=0, n_sink=4, n_recent=64):
    lens = tuple(lens)
    cap = cap if cap is not None else max(max(lens), 1, budget) + (steps if append else 0)
    return Workload(name=name, B=B, lens=lens, H=H, n_q=16, n_kv=1, d=128, budget=budget, n_layers=1,
                    gpu_layers=(0,) * B, steps=steps, rho=(0.9,) * B,
                    hot=tuple(max(1, int(hot_frac * L)) for L in lens), seed=seed, append=append, cap=cap,
                    n_sink=n_sink, n_recent=n_recent, mla=True)


def u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)


def _score_case(cfg, t=0, append=False):
    inp = make_mla_inputs(cfg, steps=max(1, cfg.steps), n_layers=1)
    C = u16(inp.C_dlm)
    ln = torch.from_numpy(inp.lens.astype(np.int32)).to(DEV)
    ws = torch.zeros(spc.spc_mla_score_select_workspace_size(cfg.B, cfg.H, cfg.cap, cfg.budget), dtype=torch.uint8,
                     device=DEV)
    scores = torch.zeros(cfg.B, cfg.cap, dtype=torch.float32, device=DEV)
    sel = torch.full((cfg.B, cfg.budget), -7, dtype=torch.int32, device=DEV)
    spc.spc_mla_score_select(u16(inp.x[t]), u16(inp.Wq), u16(inp.Wuk), u16(inp.Wdkv) if append else None, C, ln,
                             int(append), cfg.B, cfg.H, cfg.cap, cfg.budget, cfg.n_sink, cfg.n_recent, scores, sel,
                             ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    gsel, gs, glen = sel.cpu().numpy(), scores.cpu().numpy(), ln.cpu().numpy()
    gC = C.cpu().numpy().view(np.uint16)

    st = M.MlaDecodeState(inp.C_dlm, inp.lens, [np.zeros((1, cfg.cap, M.D_LAT), np.uint16)] * cfg.B, [0] * cfg.B,
                          cfg.budget, cfg.n_sink, cfg.n_recent)
    L0 = [int(v) for v in inp.lens]
    _, c_new, _, ss, osel = st.score_select(inp.x[t], inp.Wq, inp.Wuk, inp.Wdkv, cfg.n_q, append)
    assert list(glen) == st.lens
    swaps = 0
    for b in range(cfg.B):
        L = st.lens[b]
        err = max_rel_err(gs[b, :L], ss[b][0], floor=1e-30)
        assert err <= SCORE_RTOL, f"scores b={b}: max rel err {err:.3g}"
        ok, sw, msg = selection_within_tie_band(gsel[b], osel[b][0], ss[b][0], cfg.budget, cfg.n_sink,
                                                cfg.n_recent)
        assert ok, f"selection b={b}: {msg}"
        swaps += sw
        if append and L0[b] < cfg.cap:
            assert bf16_ulp_distance(gC[b, L0[b]], c_new[b]).max() <= 1
    return swaps


SCORE_CASES = [
    ("tiles_and_tail", dict(lens=(3001,), H=512, budget=512)),
    ("one_tile_partial", dict(lens=(33,), budget=16, n_sink=2, n_recent=8)),
    ("ragged_batch", dict(B=3, lens=(1500, 129, 700), H=256, budget=96)),
    ("batch17", dict(B=17, lens=tuple(200 + 37 * i for i in range(17)), H=256, budget=80)),
    ("len_le_budget", dict(lens=(50,), budget=96)),
    ("len_zero", dict(lens=(0,), budget=96)),
    ("hidden8", dict(lens=(400,), H=8, budget=96)),
    ("long_many_ctas", dict(lens=(20000,), H=512, budget=300, cap=20011)),
]


@pytest.mark.parametrize("name,kw", SCORE_CASES, ids=[c[0] for c in SCORE_CASES])
def test_mla_score_select(name, kw):
    _score_case(mla_workload(name=name, **kw))


def test_mla_score_select_appends_the_latent_row():
    cfg = mla_workload(name="append", B=2, lens=(700, 97), H=256, budget=96, steps=2, append=True)
    _score_case(cfg, t=1, append=True)


def test_mla_score_select_full_context_shape():
    """The 32K-context, 16-head shape of the benchmark workload (one step)."""
    cfg = mla_workload(name="full", lens=(32768,), H=2048, budget=2048, hot_frac=0.01, seed=6)
    assert _score_case(cfg) <= 8


# ------------------------------------------------------------------ gather
def test_mla_gather_is_a_byte_copy():
    rng = np.random.default_rng(71)
    B, cap, K = 3, 900, 200
    # request 0: store holds layers 1..4, host layers 2..4; request 1: store 0..4,
    # host 0..4; request 2: nothing to load
    specs = [(1, 4, 2, 3), (0, 5, 0, 5), (0, 5, 0, 5)]
    stores, slots, dptr, loads = [], [], [], []
    for b, (s0, sn, l0, nl) in enumerate(specs):
        hs = torch.from_numpy(rng.integers(0, 1 << 16, (cap, sn, M.D_LAT), dtype=np.uint16).view(np.int16)).pin_memory()
        stores.append(hs)
        sl = torch.from_numpy(rng.integers(0, 1 << 16, (nl, K, M.D_LAT), dtype=np.uint16).view(np.int16)).to(DEV)
        slots.append(sl)
        dptr.append(spc.spc_host_device_pointer(hs))
        n = 0 if b == 2 else int(rng.integers(1, K))
        lp = np.sort(rng.choice(cap, n, replace=False))
        ls = rng.choice(K, n, replace=False)
        loads.append((ls, lp))
    views = spc.gather_views(dptr, [s.data_ptr() for s in slots], [s[2] for s in specs], [s[3] for s in specs],
                             [s[0] for s in specs], [s[1] for s in specs])
    load_slot = np.zeros((B, K), np.int32)
    load_pos = np.zeros((B, K), np.int32)
    n_load = np.zeros(B, np.int32)
    for b, (ls, lp) in enumerate(loads):
        load_slot[b, :len(ls)], load_pos[b, :len(lp)], n_load[b] = ls, lp, len(ls)
    before = [s.cpu().numpy().view(np.uint16).copy() for s in slots]
    spc.spc_mla_gather(spc.to_device_bytes(views, DEV), 0, 5, torch.from_numpy(load_slot).to(DEV),
                       torch.from_numpy(load_pos).to(DEV), torch.from_numpy(n_load).to(DEV), B, cap, K)
    torch.cuda.synchronize()
    for b, (s0, sn, l0, nl) in enumerate(specs):
        want = before[b].copy()
        store = stores[b].numpy().view(np.uint16)
        # oracle layout [layers][cap][576] of the request's host layers
        M.mla_gather(np.ascontiguousarray(store[:, l0 - s0:l0 - s0 + nl].transpose(1, 0, 2)), want, *loads[b])
        assert np.array_equal(slots[b].cpu().numpy().view(np.uint16), want), f"request {b}"


# ------------------------------------------------------------------ attention
def _attn_case(B, n_layers, budget, hbm_layers, seed=73, empty_request=None, short=None, cap=700):
    rng = np.random.default_rng(seed)
    scale = 1 / math.sqrt(M.D_QK)
    full = [O.round_to_bf16(rng.standard_normal((n_layers, cap, M.D_LAT))) for _ in range(B)]
    q = O.round_to_bf16(rng.standard_normal((n_layers, B, 16, M.D_QK)))
    Wuk = O.round_to_bf16(rng.standard_normal((n_layers, 16, M.D_NOPE, M.D_C)) / math.sqrt(M.D_C))
    Wuv = O.round_to_bf16(rng.standard_normal((n_layers, 16, M.D_V, M.D_C)) / math.sqrt(M.D_C))
    selected = np.full((B, budget), -1, np.int32)
    slot_pos = np.full((B, budget), -1, np.int32)
    for b in range(B):
        if b == empty_request:
            continue
        n = budget if b != short else budget // 3
        pos = np.sort(rng.choice(cap, n, replace=False))
        selected[b, :n] = pos
        perm = rng.permutation(budget)[:n]          # slots in any order, some left empty
        slot_pos[b, perm] = pos
    # device tensors: HBM layers read full caches by position, host layers slots
    dev_full = [[u16(full[b][l]) for l in range(n_layers)] for b in range(B)]
    dev_slots = []
    for b in range(B):
        sl = np.zeros((n_layers, budget, M.D_LAT), np.uint16)
        for s, p in enumerate(slot_pos[b]):
            if p >= 0:
                sl[:, s] = full[b][:, p]
        dev_slots.append(u16(sl))
    ptrs, rows, use = [], [], []
    for l in range(n_layers):
        for b in range(B):
            if l < hbm_layers:
                ptrs.append(dev_full[b][l].data_ptr()); rows.append(cap); use.append(0)
            else:
                ptrs.append(dev_slots[b][l].data_ptr()); rows.append(budget); use.append(1)
    views = spc.to_device_bytes(spc.kv_views(ptrs, [0] * len(ptrs), rows, use), DEV)
    out = torch.full((n_layers, B, 16, M.D_V), 7.0, dtype=torch.float32, device=DEV)
    ws = torch.zeros(spc.spc_mla_decode_attn_workspace_size(n_layers, B, budget), dtype=torch.uint8, device=DEV)
    spc.spc_mla_decode_attn(u16(q), u16(Wuk), u16(Wuv), views, torch.from_numpy(selected).to(DEV),
                            torch.from_numpy(slot_pos).to(DEV), n_layers, B, budget, scale, out, ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    g = out.cpu().numpy()
    worst = 0.0
    for l in range(n_layers):
        for b in range(B):
            rows_b = selected[b][selected[b] >= 0]
            want = M.mla_sparse_attention(q[l, b], full[b][l], Wuk[l], Wuv[l], rows_b, scale)
            err = float(np.abs(g[l, b] - want).max())
            worst = max(worst, err)
            assert err <= ATTN_ATOL, f"layer {l} request {b}: {err:.3g}"
    return worst


def test_mla_attention_hbm_and_slot_layers_ragged_budget():
    worst = _attn_case(B=2, n_layers=3, budget=300, hbm_layers=1, short=1)
    assert worst <= 3e-3


def test_mla_attention_empty_selection_gives_zeros():
    _attn_case(B=3, n_layers=2, budget=64, hbm_layers=1, empty_request=1)


def test_mla_attention_many_splits():
    # one (layer, request) and the largest budget: 128 tiles of 32 rows over
    # 64 CTAs of two tiles each
    _attn_case(B=1, n_layers=1, budget=4096, hbm_layers=0, seed=79, cap=5000)


# ------------------------------------------------------------------ the decode step
def run_mla_chain(cfg, steps, L, layers_per_launch=1):
    """The pipelined MLA decode step against the oracle's own chain: while the
    GPU and oracle selections agree, load lists and slot maps match bit for
    bit and attention is within the bar; a tie-band swap makes that request's
    later steps comparable on sets only (band, slot contents)."""
    from sparse_kv_cache_retrieval_gb300.pipeline import DecodePipeline
    from sparse_kv_cache_retrieval_gb300.synth import fill_mla_layer
    inp = make_mla_inputs(cfg, steps=steps, n_layers=L)
    pipe = DecodePipeline(cfg, inp, n_layers=L, layers_per_launch=layers_per_launch)
    stores = []
    for b in range(cfg.B):
        st = np.empty((L, cfg.cap, M.D_LAT), np.uint16)
        for l in range(L):
            fill_mla_layer(cfg, b, l, st[l])
        stores.append(st)
    ost = M.MlaDecodeState(inp.C_dlm, inp.lens, stores, pipe.gpu_layers, cfg.budget, cfg.n_sink, cfg.n_recent)
    _, _, _, oss, osel = ost.score_select(inp.x[0], inp.Wq, inp.Wuk, inp.Wdkv, cfg.n_q, append=False)
    pipe.prologue()
    tid = f"mla chain {cfg.name}"
    # selections within the tie band of the oracle's; the chain continues from
    # the GPU's (valid) choice, so every later check covers every request
    sel, swaps = swap_log.check_selection(tid, pipe.selected[0].cpu().numpy(), osel, oss, cfg.budget, cfg.n_sink,
                                          cfg.n_recent, "prologue")
    ost.diff_and_gather(sel)
    scale = 1 / math.sqrt(M.D_QK)
    worst = 0.0
    for t in range(steps):
        pn = (t + 1) % 2
        pipe.step(t)
        pipe.join()
        torch.cuda.synchronize()
        _, _, _, oss, osel = ost.score_select(inp.x[t + 1], inp.Wq, inp.Wuk, inp.Wdkv, cfg.n_q, append=cfg.append)
        oout = ost.attention(inp.q_llm[t, :L], inp.Wuk_llm[:L], inp.Wuv_llm[:L], scale)
        gsel, gslot = pipe.selected[pn].cpu().numpy(), pipe.slot_pos[pn].cpu().numpy()
        sel, sw = swap_log.check_selection(tid, gsel, osel, oss, cfg.budget, cfg.n_sink, cfg.n_recent, f"t={t}")
        swaps += sw
        loads = ost.diff_and_gather(sel)
        gnl, gls, glp = pipe.n_load[pn].cpu().numpy(), pipe.load_slot[pn].cpu().numpy(), pipe.load_pos[pn].cpu().numpy()
        gout = pipe.out.cpu().numpy()
        assert pipe.len.cpu().numpy().tolist() == ost.lens
        for b in range(cfg.B):
            e = float(np.abs(gout[:, b] - oout[:, b]).max())
            worst = max(worst, e)
            assert e <= ATTN_ATOL, f"t={t} b={b}: attention error {e:.3g}"
            ls, lp = loads[b][0]
            assert gnl[b, 0] == lp.size
            assert np.array_equal(glp[b, 0, :lp.size], lp) and np.array_equal(gls[b, 0, :ls.size], ls)
            assert np.array_equal(gslot[b, 0], ost.slot_pos[b, 0])
            if pipe.host_slots(b) is not None:
                sl = pipe.host_slots(b).cpu().numpy().view(np.uint16)
                h0 = pipe.gpu_layers[b]
                idx = np.nonzero(gslot[b, 0] >= 0)[0]
                assert np.array_equal(sl[:, idx], stores[b][h0:, gslot[b, 0][idx]])
    return swaps, worst, pipe


def test_mla_chain_small_host_layers():
    from sparse_kv_cache_retrieval_gb300.configs import CONFIGS, scaled
    cfg = scaled(CONFIGS["mla"], lens=(3000,), n_layers=3, steps=3, budget=512)
    _, worst, _ = run_mla_chain(cfg, 3, 3, layers_per_launch=2)
    assert worst <= 3e-3


def test_mla_chain_ragged_batch_hbm_host_split_append():
    cfg = dataclasses.replace(mla_workload(name="chain", B=2, lens=(510, 900), H=256, budget=512, steps=3,
                                           append=True), n_layers=2, gpu_layers=(1, 0))
    _, _, pipe = run_mla_chain(cfg, 3, 2, layers_per_launch=2)
    assert pipe.len.cpu().tolist() == [513, 903]


def test_mla_chain_full_shape():
    """The benchmark workload's shapes (32K context, budget 2048, 16 heads) on
    two of its 27 host layers, two steps."""
    from sparse_kv_cache_retrieval_gb300.configs import CONFIGS, scaled
    cfg = scaled(CONFIGS["mla"], n_layers=2, steps=2)
    assert cfg.cap == 32768 and cfg.budget == 2048
    run_mla_chain(cfg, 2, 2, layers_per_launch=2)


def test_mla_graph_replay_equals_eager():
    from sparse_kv_cache_retrieval_gb300.configs import CONFIGS, scaled
    from sparse_kv_cache_retrieval_gb300.pipeline import DecodePipeline
    cfg = scaled(CONFIGS["mla"], lens=(2000,), n_layers=2, steps=3, budget=256)
    inp = make_mla_inputs(cfg, steps=3, n_layers=2)
    a = DecodePipeline(cfg, inp, n_layers=2, layers_per_launch=1)
    a.prologue()
    a.run(0, 3)
    torch.cuda.synchronize()
    b = DecodePipeline(cfg, inp, n_layers=2, layers_per_launch=1)
    b.prologue()
    g = b.capture(0, 3)
    g.replay()
    torch.cuda.synchronize()
    for u, v in ((a.out, b.out), (a.selected, b.selected), (a.slot_pos, b.slot_pos), (a.slots[0], b.slots[0])):
        assert torch.equal(u.cpu(), v.cpu())
