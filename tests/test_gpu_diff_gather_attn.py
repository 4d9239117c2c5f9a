"""GPU parity of spc_elastic_diff, spc_gather_kv and spc_sparse_decode_attn
against the CPU oracle, through the C ABI, on seeded synthetic inputs.

Bars: load lists, slot maps and gathered bytes bit-exact; attention within
1e-2 absolute (the stated bar) and, tighter, within 2e-5 + 1e-4 |o| (fp32
accumulation over at most 4096 rows of unit-scale products).
"""
import math

import numpy as np
import pytest
import torch

import oracle.spc_oracle as O
from oracle.checks import ATTN_ATOL
from sparse_kv_cache_retrieval_gb300 import binding as spc

pytestmark = pytest.mark.gpu
DEV = "cuda"


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)


def random_state(rng, B, n_kv, K, cap, churn=0.3, empty=0.05, n_sel=None):
    """Seeded selection/slot-map pairs with the structure a decode produces."""
    sel = np.full((B, n_kv, K), -1, np.int64)
    prev = np.full((B, n_kv, K), -1, np.int64)
    for b in range(B):
        for g in range(n_kv):
            m = K if n_sel is None else n_sel
            old = rng.choice(cap, size=K, replace=False)
            keep = old[rng.random(K) > churn]
            fresh = np.setdiff1d(rng.choice(cap, size=min(cap, 2 * K), replace=False), old)
            new = np.concatenate([keep, fresh])[:m]
            new = np.sort(rng.permutation(new)[:m])
            sel[b, g, :new.size] = new
            p = old.copy()
            p[rng.random(K) < empty] = -1
            prev[b, g] = p
    return sel, prev


def run_diff(sel, prev, cap, inplace=False):
    B, n_kv, K = sel.shape
    s, p = i32(sel), i32(prev)
    nxt = p if inplace else torch.full_like(p, -9)
    ls = torch.full_like(p, -9)
    lp = torch.full_like(p, -9)
    nl = torch.full((B, n_kv), -9, dtype=torch.int32, device=DEV)
    spc.spc_elastic_diff(s, p, nxt, ls, lp, nl, B, n_kv, K, cap)
    torch.cuda.synchronize()
    return ls.cpu().numpy(), lp.cpu().numpy(), nxt.cpu().numpy(), nl.cpu().numpy()


@pytest.mark.parametrize("B,n_kv,K,cap,churn,inplace", [
    (1, 8, 2048, 32768, 0.2, False),
    (2, 3, 100, 400, 0.5, True),
    (16, 8, 1024, 16384, 0.3, False),
    (1, 1, 4096, 262144, 0.9, False),      # maximum budget and capacity
    (3, 2, 64, 64, 1.0, False),           # every slot empty or replaced
    (2, 2, 1, 5, 0.5, True),
])
def test_elastic_diff_bit_exact(B, n_kv, K, cap, churn, inplace):
    rng = np.random.default_rng(1000 + K + cap)
    sel, prev = random_state(rng, B, n_kv, K, cap, churn)
    ls, lp, nxt, nl = run_diff(sel, prev, cap, inplace)
    for b in range(B):
        for g in range(n_kv):
            ols, olp, onxt = O.elastic_diff(sel[b, g], prev[b, g])
            n = nl[b, g]
            assert n == olp.size
            assert np.array_equal(ls[b, g, :n], ols) and np.array_equal(lp[b, g, :n], olp)
            assert np.array_equal(nxt[b, g], onxt)


def test_elastic_diff_worked_example_and_idempotence():
    sel = np.array([[[1, 8, 21, 50]]])
    prev = np.array([[[1, 8, 21, 35]]])
    ls, lp, nxt, nl = run_diff(sel, prev, 64)
    assert nl[0, 0] == 1 and lp[0, 0, 0] == 50 and ls[0, 0, 0] == 3
    assert nxt[0, 0].tolist() == [1, 8, 21, 50]
    ls, lp, nxt2, nl = run_diff(sel, nxt, 64)
    assert nl[0, 0] == 0 and np.array_equal(nxt2, nxt)


def test_elastic_diff_partial_selection():
    rng = np.random.default_rng(7)
    sel, prev = random_state(rng, 2, 4, 256, 3000, 0.4, n_sel=170)
    ls, lp, nxt, nl = run_diff(sel, prev, 3000)
    for b in range(2):
        for g in range(4):
            ols, olp, onxt = O.elastic_diff(sel[b, g], prev[b, g])
            assert np.array_equal(lp[b, g, :nl[b, g]], olp) and np.array_equal(nxt[b, g], onxt)


@pytest.mark.parametrize("whole_store", [False, True])
def test_gather_bit_exact_over_layers_and_requests(whole_store):
    # host stores are position-major [cap][n_kv][store_layers][2][d]; with
    # whole_store every request's store holds all L layers (the adaptive
    # layout) while only layers >= layer0 are host-resident
    rng = np.random.default_rng(11)
    B, n_kv, K, cap, L = 3, 4, 96, 700, 5
    layer0 = [0, 2, 5]                      # request 2 keeps every layer in HBM
    stores, slots, hptr, sptr, s0s, sns = [], [], [], [], [], []
    for b in range(B):
        nh = L - layer0[b]
        s0 = 0 if whole_store else layer0[b]
        if nh == 0:
            stores.append(None); slots.append(None); hptr.append(0); sptr.append(0)
            s0s.append(s0); sns.append(L - s0)
            continue
        bits = rng.integers(-32768, 32767, (L - s0, 2, n_kv, cap, 128), dtype=np.int16)   # layer-major
        hs = torch.from_numpy(np.ascontiguousarray(bits.transpose(3, 2, 0, 1, 4))).pin_memory()
        sl = torch.zeros((nh, 2, n_kv, K, 128), dtype=torch.int16, device=DEV)
        stores.append((bits, hs)); slots.append(sl)
        hptr.append(spc.spc_host_device_pointer(hs)); sptr.append(sl.data_ptr())
        s0s.append(s0); sns.append(L - s0)
    views = spc.to_device_bytes(spc.gather_views(hptr, sptr, layer0, [L - v for v in layer0], s0s, sns), DEV)
    sel, prev = random_state(rng, B, n_kv, K, cap, 0.5)
    loads = [[O.elastic_diff(sel[b, g], prev[b, g]) for g in range(n_kv)] for b in range(B)]
    ls = np.zeros((B, n_kv, K), np.int32)
    lp = np.zeros((B, n_kv, K), np.int32)
    nl = np.zeros((B, n_kv), np.int32)
    for b in range(B):
        for g in range(n_kv):
            a, p, _ = loads[b][g]
            ls[b, g, :a.size], lp[b, g, :p.size], nl[b, g] = a, p, a.size
    ls_d, lp_d, nl_d = i32(ls), i32(lp), i32(nl)
    # two launches over layer ranges [0, 3) and [3, 5)
    spc.spc_gather_kv(views, 0, 3, ls_d, lp_d, nl_d, B, n_kv, 128, cap, K)
    spc.spc_gather_kv(views, 3, 5, ls_d, lp_d, nl_d, B, n_kv, 128, cap, K)
    torch.cuda.synchronize()
    for b in range(B):
        if slots[b] is None:
            continue
        got = slots[b].cpu().numpy().view(np.uint16)
        want = np.zeros_like(got)
        bits = stores[b][0].view(np.uint16)[layer0[b] - s0s[b]:]
        O.gather(bits, want, [x[0] for x in loads[b]], [x[1] for x in loads[b]])
        assert np.array_equal(got, want)


def test_store_layer_writes_one_layer_position_major():
    # the copy half of an offload: a layer-major HBM cache into its layer of a
    # position-major pinned store, bit-exact, other layers untouched
    rng = np.random.default_rng(23)
    n_kv, cap, SL, layer, rows = 4, 300, 5, 3, 260
    src_bits = rng.integers(-32768, 32767, (2, n_kv, cap, 128), dtype=np.int16)
    src = torch.from_numpy(src_bits).to(DEV)
    store = torch.full((cap, n_kv, SL, 2, 128), 5, dtype=torch.int16).pin_memory()
    spc.spc_store_layer(spc.spc_host_device_pointer(store), src, n_kv, 128, cap, rows, SL, layer)
    torch.cuda.synchronize()
    got = store.numpy()
    want = np.full_like(got, 5)
    want[:rows, :, layer] = src_bits[:, :, :rows].transpose(2, 1, 0, 3)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("source", ["device", "host"])
def test_fill_slots_bit_exact(source):
    # the workspace of a layer entering CPU memory starts with the resident
    # rows: slots[s] = cache[slot_pos[s]] for every slot holding a position
    # (empty slots and out-of-range positions untouched), per request, K and V,
    # KV head; layers outside a request's view are skipped
    rng = np.random.default_rng(17)
    B, n_kv, K, cap, L = 3, 2, 100, 400, 4
    layer0 = [1, 3, 4]                  # request 2 has no layer in the view
    caches, slots, hptr, sptr = [], [], [], []
    for b in range(B):
        n = max(1, L - layer0[b])
        bits = rng.integers(-32768, 32767, (n, 2, n_kv, cap, 128), dtype=np.int16)
        if source == "device":
            c = torch.from_numpy(bits).to(DEV)
            hptr.append(c.data_ptr())
        else:
            c = torch.from_numpy(bits).pin_memory()
            hptr.append(spc.spc_host_device_pointer(c))
        sl = torch.full((n, 2, n_kv, K, 128), 7, dtype=torch.int16, device=DEV)
        caches.append((bits, c)); slots.append(sl); sptr.append(sl.data_ptr())
    views = spc.to_device_bytes(spc.gather_views(hptr, sptr, layer0, [L - v for v in layer0]), DEV)
    slot_pos = np.full((B, n_kv, K), -1, np.int64)
    for b in range(B):
        for g in range(n_kv):
            m = int(rng.integers(K // 2, K + 1))
            slot_pos[b, g, rng.choice(K, size=m, replace=False)] = rng.choice(cap, size=m, replace=False)
    slot_pos[0, 0, 0] = cap + 5                     # out of range: left untouched
    spc.spc_fill_slots(views, 2, 4, i32(slot_pos), B, n_kv, 128, cap, K)   # layers 2 and 3 only
    torch.cuda.synchronize()
    for b in range(B):
        got = slots[b].cpu().numpy()
        want = np.full_like(got, 7)
        bits = caches[b][0]
        for l in range(max(2, layer0[b]), 4):
            lr = l - layer0[b]
            for g in range(n_kv):
                for s_ in range(K):
                    p_ = slot_pos[b, g, s_]
                    if 0 <= p_ < cap:
                        want[lr, :, g, s_] = bits[lr, :, g, p_]
        assert np.array_equal(got, want), f"request {b}"


def _attn_case(rng, L, B, n_q, n_kv, K, cap, use_slots, n_valid=None, empty_group=False, q_gain=1.5,
               ramp=False, poison=False, pos_layers=0):
    """Returns GPU output and oracle output for one attention launch.

    ramp: K rows grow in norm with their row index (later tiles hold larger
    logits, so a running maximum keeps rising); poison: rows of the K/V
    buffers that no kept index names hold NaN (they must not reach the output);
    pos_layers: the first layers read positions from a full cache whatever
    use_slots says (a launch that mixes both kinds of view).
    """
    d = 128
    sel = np.full((B, n_kv, K), -1, np.int64)
    slot = np.full((B, n_kv, K), -1, np.int64)
    kept = []
    for b in range(B):
        kb = []
        for g in range(n_kv):
            m = K if n_valid is None else n_valid
            if empty_group and g == 0:
                m = 0
            pos = np.sort(rng.choice(cap, size=m, replace=False))
            sel[b, g, :m] = pos
            sl = rng.choice(K, size=m, replace=False)
            slot[b, g, sl] = pos
            kb.append(np.sort(sl) if use_slots else pos)
        kept.append(kb)
    caches, kp, vp, rows, use = [], [], [], [], []
    for l in range(L):
        for b in range(B):
            slots_here = use_slots and l >= pos_layers
            nrows = K if slots_here else cap
            kv = rng.standard_normal((2, n_kv, nrows, d)).astype(np.float32)
            if ramp:
                kv[0] *= (1.0 + 3.0 * np.arange(nrows) / nrows)[None, :, None].astype(np.float32)
            bits = O.round_to_bf16(kv.astype(np.float64))
            t = torch.from_numpy(bits.view(np.int16)).to(DEV)
            if poison:
                raw = bits.view(np.int16).copy()
                for g in range(n_kv):
                    unused = np.ones(nrows, bool)
                    unused[kept[b][g]] = False
                    raw[:, g, unused] = np.int16(0x7FC0)       # bf16 quiet NaN
                t = torch.from_numpy(raw).to(DEV)
            caches.append((bits, t))
            kp.append(t[0].data_ptr()); vp.append(t[1].data_ptr()); rows.append(nrows); use.append(int(slots_here))
    views = spc.to_device_bytes(spc.kv_views(kp, vp, rows, use), DEV)
    q = O.round_to_bf16(rng.standard_normal((L, B, n_q, d)) * q_gain)
    out = torch.full((L, B, n_q, d), 7.0, dtype=torch.float32, device=DEV)
    ws = torch.zeros(spc.spc_sparse_decode_attn_workspace_size(L, B, n_q, n_kv, d, K), dtype=torch.uint8,
                     device=DEV)
    qd = torch.from_numpy(q.view(np.int16)).to(DEV)
    scale = 1 / math.sqrt(d)
    spc.spc_sparse_decode_attn(qd, views, i32(sel), i32(slot), L, B, n_q, n_kv, d, K, scale, out, ws)
    spc.spc_sparse_decode_attn(qd, views, i32(sel), i32(slot), L, B, n_q, n_kv, d, K, scale, out, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    want = np.zeros_like(got, dtype=np.float64)
    for l in range(L):
        for b in range(B):
            bits = caches[l * B + b][0]
            rows_lb = kept[b] if (use_slots and l >= pos_layers) else \
                [sel[b, g][sel[b, g] >= 0] for g in range(n_kv)]
            want[l, b] = O.sparse_attention(q[l, b], bits[0], bits[1], rows_lb, scale)
    return got, want


ATTN_CASES = [
    # L, B, n_q, n_kv, K, cap, use_slots, n_valid
    (1, 1, 32, 8, 2048, 4096, 1, None),      # bench shape, one layer (split over the budget)
    (4, 1, 32, 8, 2048, 4096, 1, 1500),      # 4 layers per launch, partly empty slots
    (2, 2, 32, 8, 1000, 3000, 0, None),      # positions into a full cache, budget not /64
    (1, 3, 4, 4, 130, 500, 1, None),         # MHA
    (1, 2, 8, 4, 200, 700, 0, 150),          # G = 2
    (1, 1, 64, 8, 4096, 8192, 1, None),      # 70B shape, max budget
    (1, 1, 64, 1, 512, 2000, 0, None),       # MQA
    (1, 1, 16, 1, 64, 100, 1, 1),            # one kept row per group
    # 64 heads per KV head (the tensor-core kernel): CTA runs split segments,
    # partials merged by the last CTA of each segment
    (2, 3, 64, 1, 4096, 8192, 1, 3000),      # max budget, 16 CTAs per segment
    (3, 4, 64, 1, 4096, 4096, 1, 3900),      # 12 segments, 3 tiles per CTA: runs cross segment ends
    (1, 1, 64, 1, 1000, 3000, 1, None),      # budget not a multiple of the 128-row tile
    (2, 1, 128, 2, 700, 2000, 0, None),      # two KV heads, positions into a full cache
    (1, 1, 64, 1, 128, 128, 1, None),        # one tile, one CTA: no partials
    (3, 1, 64, 1, 256, 300, 1, 2),           # two kept rows in a 256-row budget
    (32, 8, 64, 1, 256, 300, 1, 200),        # 256 segments: two whole segments per CTA
    (16, 8, 64, 1, 512, 600, 1, None),       # 128 segments: one whole segment per CTA
]


@pytest.mark.parametrize("L,B,n_q,n_kv,K,cap,use_slots,n_valid", ATTN_CASES)
def test_attention_parity(L, B, n_q, n_kv, K, cap, use_slots, n_valid):
    rng = np.random.default_rng(L * 1000 + n_q * 10 + K)
    got, want = _attn_case(rng, L, B, n_q, n_kv, K, cap, use_slots, n_valid)
    err = np.abs(got - want)
    assert err.max() <= ATTN_ATOL
    assert np.all(err <= 2e-5 + 1e-4 * np.abs(want)), f"max err {err.max():.3g}"


@pytest.mark.parametrize("L,B,K,cap,n_valid", [(16, 8, 512, 2000, None), (4, 8, 1024, 3000, 900)])
def test_attention_mixed_views_64_heads(L, B, K, cap, n_valid):
    """Layer 0 read by position from a full cache, the others through slots, in
    one launch: with one segment per CTA the position-read segments are split
    over two CTAs each (their halves merged) while the others stay whole."""
    rng = np.random.default_rng(31 + L)
    got, want = _attn_case(rng, L, B, 64, 1, K, cap, 1, n_valid, pos_layers=1)
    err = np.abs(got - want)
    assert np.all(err <= 2e-5 + 1e-4 * np.abs(want)), f"max err {err.max():.3g}"


@pytest.mark.parametrize("n_q,n_kv", [(64, 1), (32, 8)])
def test_attention_rising_maximum(n_q, n_kv):
    """Large logits that grow tile by tile: the running maximum is raised and
    the partial sums and outputs rescaled many times."""
    rng = np.random.default_rng(11 + n_q)
    got, want = _attn_case(rng, 2, 2, n_q, n_kv, 2048, 2048, 1, None, q_gain=12.0, ramp=True)
    err = np.abs(got - want)
    assert np.all(err <= 2e-5 + 1e-4 * np.abs(want)), f"max err {err.max():.3g}"


@pytest.mark.parametrize("n_q,n_kv,use_slots", [(64, 1, 1), (64, 1, 0), (32, 8, 1)])
def test_attention_ignores_rows_not_kept(n_q, n_kv, use_slots):
    """NaN in every K/V row that no kept index names leaves the output finite
    and equal to the oracle's."""
    rng = np.random.default_rng(21 + n_q + use_slots)
    got, want = _attn_case(rng, 1, 2, n_q, n_kv, 1024, 2048, use_slots, 700, poison=True)
    assert np.all(np.isfinite(got))
    err = np.abs(got - want)
    assert np.all(err <= 2e-5 + 1e-4 * np.abs(want)), f"max err {err.max():.3g}"


@pytest.mark.parametrize("n_q,n_kv", [(64, 1), (8, 2)])
def test_attention_empty_group_is_zero_any_shape(n_q, n_kv):
    rng = np.random.default_rng(6 + n_q)
    got, want = _attn_case(rng, 2, 2, n_q, n_kv, 384, 500, 1, None, empty_group=True)
    G = n_q // n_kv
    assert np.all(got[:, :, :G] == 0.0)
    assert np.abs(got - want).max() <= 2e-5 + 1e-4 * np.abs(want).max()


def test_attention_empty_group_is_zero():
    rng = np.random.default_rng(5)
    got, want = _attn_case(rng, 1, 1, 8, 2, 128, 300, 1, None, empty_group=True)
    assert np.all(got[0, 0, :4] == 0.0)
    assert np.abs(got - want).max() <= 2e-5 + 1e-4 * np.abs(want).max()


def test_attention_all_rows_equals_dense():
    """Every position kept: sparse attention is dense attention (torch SDPA, fp64)."""
    rng = np.random.default_rng(3)
    d, n_q, n_kv, n = 128, 8, 2, 192
    got, want = _attn_case(rng, 1, 1, n_q, n_kv, n, n, 0, None)
    assert np.abs(got - want).max() <= 1e-4
