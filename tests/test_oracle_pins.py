"""Pins of the CPU oracle to facts outside itself.

Every oracle function is checked against something it cannot agree with by
construction: the pages' worked example and printed figures (tests/golden/),
closed forms, brute force over tiny inputs, invariants the pages state, and a
library routine on the special case that reduces to it. The mutation tests at
the end plant plausible mistakes in copies of oracle functions and check that
at least one pin fails for each.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle.spc_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


def _bits(values):
    """Exact fp64 -> bf16 bits for values that are exactly representable."""
    a = np.asarray(values, np.float64).astype(np.float32)
    assert np.array_equal(a.astype(np.float64), np.asarray(values, np.float64))
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


# ----------------------------------------------------------------- pin checks
# Each check takes the function under test so the mutation tests can reuse it.

def check_bf16_golden(round_fn):
    for row in _golden_rows("bf16_rounding.txt"):
        expr, hexbits = row.rsplit(None, 1)
        v = eval(expr, {"__builtins__": {}})
        if int(round_fn(np.array([v]))[0]) != int(hexbits, 16):
            return False
    return True


def check_bf16_bruteforce(round_fn, n=400, seed=11):
    """Nearest bf16 over ALL finite bf16 values, ties to the even bit pattern."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))
    # include exact halfway points
    base = rng.integers(0x3000, 0x4F00, 40).astype(np.uint32)
    lo = (base << 16).view(np.float32).astype(np.float64)
    hi = ((base + 1) << 16).view(np.float32).astype(np.float64)
    v = np.concatenate([v, (lo + hi) / 2, -(lo + hi) / 2])
    allbits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        allv = (allbits << 16).view(np.float32).astype(np.float64)
    finite = np.isfinite(allv)
    allbits, allv = allbits[finite], allv[finite]
    got = round_fn(v)
    for x, g in zip(v, got):
        dist = np.abs(allv - x)
        best = np.nonzero(dist == dist.min())[0]
        cands = allbits[best]
        if len(cands) > 1:
            cands = cands[(cands & 1) == 0]
        if int(g) not in set(int(c) for c in cands):
            return False
    return True


def check_projection_exact(project_fn):
    """Small-integer inputs: products and sums are exact in fp64, so the result
    must equal integer arithmetic done with Python ints, element by element."""
    B, H, n_q, n_kv, d = 2, 6, 4, 2, 3
    x = [[(3 * b + 2 * i) % 7 - 3 for i in range(H)] for b in range(B)]
    Wq = [[(5 * i + 3 * j) % 9 - 4 for j in range(n_q * d)] for i in range(H)]
    Wk = [[(2 * i + 7 * j) % 5 - 2 for j in range(n_kv * d)] for i in range(H)]
    q, k = project_fn(_bits(x), _bits(Wq), _bits(Wk), n_q, n_kv, d)
    for b in range(B):
        for h in range(n_q):
            for c in range(d):
                ref = sum(x[b][i] * Wq[i][h * d + c] for i in range(H))
                if q[b, h, c] != ref:
                    return False
        for g in range(n_kv):
            for c in range(d):
                ref = sum(x[b][i] * Wk[i][g * d + c] for i in range(H))
                if abs(ref) > 256:
                    continue
                if int(k[b, g, c]) != int(_bits([ref])[0]):
                    return False
    return True


def check_softmax_closed_form(prob_fn):
    """Two positions, K_0 = 0, K_1 = c e_0, q = a e_0: p_1 = 1/(1+exp(-a c/sqrt(d)))."""
    d = 128
    for a, c in [(1.0, 2.0), (3.0, -1.5), (0.5, 8.0), (-2.0, 4.0)]:
        K = np.zeros((1, 2, d))
        K[0, 1, 0] = c
        q = np.zeros((1, d))
        q[0, 0] = a
        P = prob_fn(q, _bits(K), 2)
        want = 1.0 / (1.0 + math.exp(-a * c / math.sqrt(d)))
        if abs(P[0, 1] - want) > 1e-13 or abs(P[0, 0] - (1 - want)) > 1e-13:
            return False
    return True


def check_softmax_uniform(prob_fn):
    """Identical keys: every weight is exactly 1/len."""
    rng = np.random.default_rng(3)
    for n in (1, 5, 64):
        row = _bits(np.round(rng.standard_normal(128) * 8) / 8)
        K = np.tile(row, (2, n, 1))
        q = rng.standard_normal((4, 128))
        P = prob_fn(q, K, n)
        if not np.allclose(P, 1.0 / n, rtol=0, atol=1e-15):
            return False
    return True


def check_softmax_vs_sdpa(prob_fn):
    """Library routine: scaled_dot_product_attention with V = identity returns
    the attention weights themselves (float64, CPU)."""
    rng = np.random.default_rng(5)
    n_q, n_kv, n, d = 8, 2, 37, 128
    Kb = O.round_to_bf16(rng.standard_normal((n_kv, n, d)))
    q = rng.standard_normal((n_q, d))
    P = prob_fn(q, Kb, n)
    Kf = torch.from_numpy(O.bf16_to_f64(Kb))
    G = n_q // n_kv
    for h in range(n_q):
        w = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[h]).view(1, 1, 1, d), Kf[h // G].view(1, 1, n, d),
            torch.eye(n, dtype=torch.float64).view(1, 1, n, n))
        if not np.allclose(P[h], w.view(-1).numpy(), rtol=1e-12, atol=1e-15):
            return False
    return True


def check_group_max(group_fn):
    rng = np.random.default_rng(7)
    for n_q, n_kv in [(8, 2), (32, 8), (6, 6), (64, 1)]:
        P = rng.random((n_q, 50))
        s = group_fn(P, n_kv)
        G = n_q // n_kv
        for g in range(n_kv):
            members = P[g * G:(g + 1) * G]
            if np.any(s[g] < members - 0):           # >= every member
                return False
            if not np.all(np.any(s[g] == members, axis=0)):  # attained by one member
                return False
        if n_q == n_kv and not np.array_equal(s, P):  # MHA: identity
            return False
    return True


def _is_valid_topk(sel, s, budget, n_sink, n_recent):
    """Definition check: forced set inside, size min(budget, len), ascending, and
    no kept candidate ranks below an excluded one by (score desc, index asc)."""
    n = len(s)
    sel = list(sel)
    if sel != sorted(set(sel)) or len(sel) != min(budget, n):
        return False
    if n <= budget:
        return sel == list(range(n))
    F = set(range(min(n_sink, n))) | set(range(max(0, n - n_recent), n))
    if not F <= set(sel):
        return False
    kept = [p for p in sel if p not in F]
    out = [p for p in range(n) if p not in F and p not in set(sel)]
    for p in kept:
        for q in out:
            if (s[p], -p) < (s[q], -q):
                return False
    return True


def check_select_bruteforce(select_fn):
    """Every subset of the candidates for tiny n, with scores drawn from a
    three-value set so that every tie pattern occurs; exactly one subset meets
    the definition and the oracle must return it."""
    rng = np.random.default_rng(9)
    for trial in range(120):
        n = int(rng.integers(1, 11))
        budget = int(rng.integers(2, 8))
        n_sink, n_recent = int(rng.integers(0, 2)), int(rng.integers(0, 2))
        if n_sink + n_recent > budget:
            continue
        s = rng.choice([0.0, 0.25, 0.5], size=n)
        got = list(select_fn(s, budget, n_sink, n_recent))
        if n <= budget:
            if got != list(range(n)):
                return False
            continue
        F = set(range(n_sink)) | set(range(n - n_recent, n))
        cand = [p for p in range(n) if p not in F]
        k = budget - len(F)
        valid = []
        for T in itertools.combinations(cand, k):
            S = sorted(F | set(T))
            if _is_valid_topk(S, s, budget, n_sink, n_recent):
                valid.append(S)
        if len(valid) != 1 or got != valid[0]:
            return False
    return True


def check_diff_worked_example(diff_fn):
    rows = dict(r.split(None, 1) for r in _golden_rows("elastic_loading_worked_example.txt"))
    S_last = [int(v) for v in rows["S_last"].split()]
    S_now = [int(v) for v in rows["S_now"].split()]
    to_load = [int(v) for v in rows["to_load"].split()]
    replaced = int(rows["replaced"])
    ls, lp, nxt = diff_fn(np.array(S_now), np.array(S_last))
    if list(lp) != to_load:
        return False
    if [S_last[i] for i in ls] != [replaced]:
        return False
    return sorted(nxt.tolist()) == sorted(S_now)


def check_diff_invariants(diff_fn):
    """resident ∪ loaded = selected; loaded ∩ previously resident = ∅; each
    load goes to a slot whose old position left the selection; idempotence."""
    rng = np.random.default_rng(13)
    for trial in range(200):
        K = int(rng.integers(1, 24))
        n = int(rng.integers(K, 4 * K + 2))
        prev = rng.choice(n, size=K, replace=False)
        prev = np.where(rng.random(K) < 0.15, -1, prev)
        m = int(rng.integers(0, K + 1))
        sel = np.full(K, -1)
        sel[:m] = np.sort(rng.choice(n, size=m, replace=False))
        ls, lp, nxt = diff_fn(sel, prev)
        S_new = set(int(p) for p in sel if p >= 0)
        resident = set(int(p) for p in prev if p >= 0)
        if set(int(p) for p in nxt if p >= 0) != S_new:
            return False
        if set(int(p) for p in lp) & resident:
            return False
        if set(int(p) for p in lp) != S_new - resident:
            return False
        for s_, p_ in zip(ls, lp):
            if prev[s_] >= 0 and int(prev[s_]) in S_new:
                return False
            if nxt[s_] != p_:
                return False
        kept_slots = [i for i in range(K) if prev[i] >= 0 and int(prev[i]) in S_new]
        if any(nxt[i] != prev[i] for i in kept_slots):
            return False
        ls2, lp2, nxt2 = diff_fn(sel, nxt)
        if len(lp2) or not np.array_equal(nxt2, nxt):
            return False
    return True


def check_diff_pairing_order(diff_fn):
    """Reading of the in-place rule: free slots (ascending) receive the missing
    positions (ascending). Hand example: slots hold [7, 3, 9, -1, 5]; the new
    selection is {2, 3, 5, 11}: slots 0, 2, 3 are free, positions 2 and 11
    are missing -> slot 0 <- 2, slot 2 <- 11, slot 3 stays empty."""
    ls, lp, nxt = diff_fn(np.array([2, 3, 5, 11, -1]), np.array([7, 3, 9, -1, 5]))
    return list(ls) == [0, 2] and list(lp) == [2, 11] and list(nxt) == [2, 3, 11, -1, 5]


def check_attention_vs_sdpa(attn_fn):
    """All rows kept: sparse attention equals dense attention (library SDPA, float64)."""
    rng = np.random.default_rng(17)
    n_q, n_kv, n, d = 8, 2, 29, 128
    q = O.round_to_bf16(rng.standard_normal((n_q, d)))
    K = O.round_to_bf16(rng.standard_normal((n_kv, n, d)))
    V = O.round_to_bf16(rng.standard_normal((n_kv, n, d)))
    out = attn_fn(q, K, V, [np.arange(n)] * n_kv, 1 / math.sqrt(d))
    qf, Kf, Vf = (torch.from_numpy(O.bf16_to_f64(a)) for a in (q, K, V))
    G = n_q // n_kv
    ref = torch.nn.functional.scaled_dot_product_attention(
        qf.view(1, n_q, 1, d), Kf.repeat_interleave(G, 0).view(1, n_q, n, d),
        Vf.repeat_interleave(G, 0).view(1, n_q, n, d)).view(n_q, d).numpy()
    return np.allclose(out, ref, rtol=1e-12, atol=1e-13)


def check_attention_subset_vs_sdpa(attn_fn):
    """A proper subset of rows equals dense attention over those rows only."""
    rng = np.random.default_rng(19)
    n_q, n_kv, n, d = 4, 2, 40, 128
    q = O.round_to_bf16(rng.standard_normal((n_q, d)))
    K = O.round_to_bf16(rng.standard_normal((n_kv, n, d)))
    V = O.round_to_bf16(rng.standard_normal((n_kv, n, d)))
    rows = [np.array([3, 17, 18, 39]), np.array([0, 5])]
    out = attn_fn(q, K, V, rows, 1 / math.sqrt(d))
    G = n_q // n_kv
    for h in range(n_q):
        r = rows[h // G]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(O.bf16_to_f64(q[h])).view(1, 1, 1, d),
            torch.from_numpy(O.bf16_to_f64(K[h // G, r])).view(1, 1, len(r), d),
            torch.from_numpy(O.bf16_to_f64(V[h // G, r])).view(1, 1, len(r), d)).view(d).numpy()
        if not np.allclose(out[h], ref, rtol=1e-12, atol=1e-13):
            return False
    return True


def check_attention_special(attn_fn):
    """One row: o = V_r exactly. Equal keys: o = mean of the V rows. No row: 0."""
    rng = np.random.default_rng(23)
    d = 128
    q = O.round_to_bf16(rng.standard_normal((2, d)))
    K = O.round_to_bf16(rng.standard_normal((1, 6, d)))
    V = O.round_to_bf16(rng.standard_normal((1, 6, d)))
    o = attn_fn(q, K, V, [np.array([4])], 0.1)
    if not np.array_equal(o, np.tile(O.bf16_to_f64(V[0, 4]), (2, 1))):
        return False
    Ke = np.tile(K[:, :1], (1, 6, 1))
    o = attn_fn(q, Ke, V, [np.array([0, 2, 5])], 0.1)
    if not np.allclose(o, np.tile(O.bf16_to_f64(V[0, [0, 2, 5]]).mean(0), (2, 1)), atol=1e-15):
        return False
    o = attn_fn(q, K, V, [np.array([], np.int64)], 0.1)
    return np.array_equal(o, np.zeros((2, d)))


# ----------------------------------------------------------------- the pins
# ---------------------------------------------------------------- C3 memory model
def _offload_cases():
    rng = np.random.default_rng(21)
    for _ in range(40):
        L = int(rng.integers(1, 9))
        n_kv = int(rng.integers(1, 4))
        d = int(rng.choice([2, 4, 8]))
        B = int(rng.integers(1, 4))
        K = int(rng.integers(1, 12))
        row = 2 * n_kv * d * 2
        # between "all workspaces just fit" and "the whole context fits 3x over"
        kv = int(B * row * rng.integers(L * K, L * K * 6 + 2))
        yield L, n_kv, d, B, K, kv


def check_offload_bruteforce(thr_fn):
    """For every length, the rule applied from the thresholds gives the fewest
    offloaded (last) layers whose GPU footprint fits the memory, found by trying
    every count."""
    for L, n_kv, d, B, K, kv in _offload_cases():
        thr = thr_fn(L, n_kv, d, B, K, kv)
        n = 0
        for length in range(1, 40 * K + 40):
            n = O.layers_to_offload(length, thr, n)
            best = next(k for k in range(L + 1) if O.gpu_kv_bytes(length, k, L, n_kv, d, B, K) <= kv)
            if n != best:
                return False
    return True


def check_offload_boundaries(thr_fn):
    """At threshold[k] - 1 the footprint with k offloaded layers fits; at
    threshold[k] it does not; thresholds never decrease."""
    for L, n_kv, d, B, K, kv in _offload_cases():
        thr = thr_fn(L, n_kv, d, B, K, kv)
        if thr[L] is not None or any(thr[k] > thr[k + 1] for k in range(L - 1)):
            return False
        for k in range(L):
            if O.gpu_kv_bytes(thr[k] - 1, k, L, n_kv, d, B, K) > kv:
                return False
            if thr[k] > K and O.gpu_kv_bytes(thr[k], k, L, n_kv, d, B, K) <= kv:
                return False
    return True


def check_offload_pages_example(thr_fn):
    """[Blog] §7 / [Summary] §6.2.1 narrative on a Llama3-8B-shaped model (32
    layers, 8 KV heads, d 128): below the first threshold every layer keeps its
    full KV on the GPU; past it the last layer (index 31) goes to the CPU;
    between the second and the third thresholds the last two are on the CPU."""
    L = 32
    thr = thr_fn(L, 8, 128, 1, 2048, 8 << 30)
    offl = lambda length: O.layers_to_offload(length, thr, 0)
    if offl(thr[0] - 1) != 0 or offl(thr[0]) != 1:
        return False
    if list(range(L - offl(thr[0]), L)) != [31]:
        return False
    mid = (thr[1] + thr[2]) // 2
    return offl(mid) == 2 and list(range(L - offl(mid), L)) == [30, 31]


def test_offload_thresholds_bruteforce():
    assert check_offload_bruteforce(O.offload_thresholds)


def test_offload_thresholds_boundaries():
    assert check_offload_boundaries(O.offload_thresholds)


def test_offload_follows_the_pages_example():
    assert check_offload_pages_example(O.offload_thresholds)


def test_offload_infeasible_memory_is_rejected():
    with pytest.raises(ValueError):
        O.offload_thresholds(32, 8, 128, 2, 2048, 2 * 32 * 2048 * 4096 - 1)
    O.offload_thresholds(32, 8, 128, 2, 2048, 2 * 32 * 2048 * 4096)


def test_offload_rule_is_monotone_along_a_growing_context():
    thr = O.offload_thresholds(8, 2, 16, 3, 50, 3 * 2 * 2 * 16 * 2 * 900)
    n, prev = 0, 0
    for length in range(1, 2000):
        n = O.layers_to_offload(length, thr, n)
        assert n >= prev
        assert O.gpu_kv_bytes(length, n, 8, 2, 16, 3, 50) <= 3 * 2 * 2 * 16 * 2 * 900
        prev = n


def test_bf16_decode_known_values():
    assert O.bf16_to_f64(np.array([0x3F80, 0xC000, 0x4049, 0x0000, 0x8000], np.uint16)).tolist() == \
        [1.0, -2.0, 3.140625, 0.0, -0.0]


def test_bf16_rounding_golden():
    assert check_bf16_golden(O.round_to_bf16)


def test_bf16_rounding_bruteforce():
    assert check_bf16_bruteforce(O.round_to_bf16)


def test_projection_exact_integers():
    assert check_projection_exact(O.project)


def test_softmax_closed_form():
    assert check_softmax_closed_form(O.head_probabilities)


def test_softmax_uniform_and_rows_sum_to_one():
    assert check_softmax_uniform(O.head_probabilities)
    rng = np.random.default_rng(1)
    P = O.head_probabilities(rng.standard_normal((8, 128)) * 3,
                             O.round_to_bf16(rng.standard_normal((2, 300, 128))), 300)
    assert np.allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(P > 0)


def test_softmax_vs_library_sdpa():
    assert check_softmax_vs_sdpa(O.head_probabilities)


def test_group_max():
    assert check_group_max(O.group_scores)


def test_select_bruteforce():
    assert check_select_bruteforce(O.select)


def test_select_special_cases():
    s = np.linspace(0, 1, 100)
    # len <= budget: everything
    assert O.select(s[:10], 16, 4, 64).tolist() == list(range(10))
    assert O.select(s[:16], 16, 4, 4).tolist() == list(range(16))
    # budget = |F|: only the forced set
    assert O.select(s, 8, 4, 4).tolist() == [0, 1, 2, 3, 96, 97, 98, 99]
    # all scores equal: the lowest non-forced positions
    assert O.select(np.zeros(50), 10, 2, 3).tolist() == [0, 1, 2, 3, 4, 5, 6, 47, 48, 49]
    # increasing scores: the highest non-forced positions
    assert O.select(s, 10, 2, 3).tolist() == [0, 1, 92, 93, 94, 95, 96, 97, 98, 99]


def test_select_planted_hot_set():
    """Positions sharing the query direction are the top-K when they fit."""
    rng = np.random.default_rng(29)
    n, d, n_hot = 2000, 128, 40
    q = rng.standard_normal((4, d))
    u = q.sum(0) / np.linalg.norm(q.sum(0))
    K = rng.standard_normal((1, n, d))
    hot = np.sort(rng.choice(np.arange(4, n - 64), n_hot, replace=False))
    K[0, hot] += 8.0 * 2.0 * u   # gamma * sqrt(G), G = 4: about +8 sigma
    P = O.head_probabilities(q, O.round_to_bf16(K), n)
    s = O.group_scores(P, 1)[0]
    sel = O.select(s, n_hot + 68, 4, 64)
    assert set(hot.tolist()) <= set(sel.tolist())


def test_diff_worked_example_from_the_page():
    assert check_diff_worked_example(O.elastic_diff)


def test_diff_invariants_and_idempotence():
    assert check_diff_invariants(O.elastic_diff)


def test_diff_pairing_order():
    assert check_diff_pairing_order(O.elastic_diff)


def test_gather_is_a_byte_copy():
    rng = np.random.default_rng(31)
    store = rng.integers(0, 1 << 16, (3, 2, 2, 50, 128), dtype=np.uint16)
    slots = np.zeros((3, 2, 2, 8, 128), np.uint16)
    ls = [np.array([1, 6]), np.array([0])]
    lp = [np.array([44, 2]), np.array([49])]
    O.gather(store, slots, ls, lp)
    for g in range(2):
        for s_, p_ in zip(ls[g], lp[g]):
            assert np.array_equal(slots[:, :, g, s_], store[:, :, g, p_])
    untouched = np.ones(8, bool)
    untouched[[1, 6]] = False
    assert not slots[:, :, 0, untouched].any()


def test_attention_vs_library_sdpa():
    assert check_attention_vs_sdpa(O.sparse_attention)
    assert check_attention_subset_vs_sdpa(O.sparse_attention)


def test_attention_special_cases():
    assert check_attention_special(O.sparse_attention)


def test_kv_footprint_matches_the_pages():
    from sparse_kv_cache_retrieval_gb300.configs import CONFIGS
    c = CONFIGS["cfg2"]
    for row in _golden_rows("kv_footprint.txt"):
        ctx, gib = (int(v) for v in row.split())
        assert 32 * c.kv_layer_bytes(ctx) == gib * (1 << 30)
    assert c.host_store_bytes() == 4 * (1 << 30)


def test_decode_state_chain_small():
    """A two-step chain on a tiny problem: the selection is consistent with the
    definitions, the slots always hold the selected rows, attention reads them."""
    rng = np.random.default_rng(37)
    B, n_q, n_kv, d, cap, L, budget = 2, 4, 2, 128, 40, 3, 12
    K_dlm = O.round_to_bf16(rng.standard_normal((B, n_kv, cap, d)))
    stores = [rng.integers(0, 1 << 16, (L, 2, n_kv, cap, d), dtype=np.uint16) & 0x3FFF
              for _ in range(B)]
    st = O.DecodeState(K_dlm, [30, 9], stores, [1, 0], budget, 2, 3)
    H = 16
    Wq = O.round_to_bf16(rng.standard_normal((H, n_q * d)) / 4)
    Wk = O.round_to_bf16(rng.standard_normal((H, n_kv * d)) / 4)
    for t in range(3):
        x = O.round_to_bf16(rng.standard_normal((B, H)))
        q, k_new, Ps, ss, sel = st.score_select(x, Wq, Wk, n_q, append=(t > 0))
        for b in range(B):
            for g in range(n_kv):
                assert _is_valid_topk(sel[b][g], ss[b][g], budget, 2, 3)
        st.diff_and_gather(sel)
        for b in range(B):
            h0 = st.host_layer0[b]
            for g in range(n_kv):
                held = st.slot_pos[b, g]
                assert set(int(p) for p in held if p >= 0) == set(sel[b][g].tolist())
                for s_, p_ in enumerate(held):
                    if p_ >= 0:
                        assert np.array_equal(st.slots[b][:, :, g, s_], stores[b][h0:, :, g, p_])
    assert st.lens == [32, 11]


# ----------------------------------------------------------------- mutations
def _mut_round_truncate(v):
    return (np.asarray(v, np.float64).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _mut_round_half_up(v):
    f, e = np.frexp(np.asarray(v, np.float64))
    r = np.ldexp(np.floor(f * 256.0 + 0.5) / 256.0, e)
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _mut_project_transposed(x_bits, Wq_bits, Wk_bits, n_q, n_kv, d):
    q, k = O.project(x_bits, Wq_bits, Wk_bits, n_q, n_kv, d)
    return q.reshape(q.shape[0], d, n_q).transpose(0, 2, 1), k


def _mut_prob_no_scale(q, K_bits, length):
    return O.head_probabilities(q * math.sqrt(q.shape[1]), K_bits, length)


def _mut_prob_wrong_group(q, K_bits, length):
    n_q = q.shape[0]
    n_kv = K_bits.shape[0]
    P = np.zeros((n_q, length))
    for h in range(n_q):
        P[h] = O.head_probabilities(q[h:h + 1], K_bits[h % n_kv:h % n_kv + 1], length)[0]
    return P


def _mut_group_mean(P, n_kv):
    G = P.shape[0] // n_kv
    return P.reshape(n_kv, G, -1).mean(axis=1)


def _mut_group_max_logits(P, n_kv):
    """Max taken before normalising: the group member with the largest raw weight
    times the group size (a dropped-normaliser mistake)."""
    G = P.shape[0] // n_kv
    return P.reshape(n_kv, G, -1).max(axis=1) * G


def _mut_select_high_index_ties(s, budget, n_sink, n_recent):
    n = len(s)
    if n <= budget:
        return np.arange(n)
    F = O.forced_positions(n, n_sink, n_recent)
    cand = np.setdiff1d(np.arange(n), F)
    order = np.lexsort((-cand, -s[cand]))
    return np.sort(np.concatenate([F, cand[order[:budget - F.size]]]))


def _mut_select_no_forced(s, budget, n_sink, n_recent):
    return O.select(s, budget, 0, 0)


def _mut_diff_descending_slots(selected, slot_pos):
    ls, lp, nxt = O.elastic_diff(selected, slot_pos)
    keep = np.array([p >= 0 and p in set(selected[selected >= 0].tolist()) for p in slot_pos])
    free = np.nonzero(~keep)[0][::-1]
    ls = free[:lp.size]
    nxt = np.where(keep, slot_pos, -1)
    nxt[ls] = lp
    return ls, lp, nxt


def _mut_diff_reload_all(selected, slot_pos):
    empty = np.full_like(np.asarray(slot_pos), -1)
    return O.elastic_diff(selected, empty)


def _mut_attn_no_softmax_norm(q_bits, K_bits, V_bits, rows, scale):
    out = O.sparse_attention(q_bits, K_bits, V_bits, rows, scale)
    return out * np.array([max(1, len(rows[h * len(rows) // q_bits.shape[0]])) for h in
                           range(q_bits.shape[0])])[:, None]


def _mut_attn_k_for_v(q_bits, K_bits, V_bits, rows, scale):
    return O.sparse_attention(q_bits, K_bits, K_bits, rows, scale)


def _mut_offload_last_fit(L, n_kv, d, B, K, kv):
    """Threshold at the longest length that still fits (off by one)."""
    thr = O.offload_thresholds(L, n_kv, d, B, K, kv)
    return [t - 1 if t is not None else None for t in thr]


def _mut_offload_no_workspace(L, n_kv, d, B, K, kv):
    """Offloaded layers counted as free (the budget workspace dropped)."""
    per_req = kv // (B * O.kv_row_bytes(n_kv, d))
    return [per_req // (L - k) + 1 for k in range(L)] + [None]


MUTANTS = [
    ("round truncates", [check_bf16_golden, check_bf16_bruteforce], _mut_round_truncate),
    ("round half up", [check_bf16_golden, check_bf16_bruteforce], _mut_round_half_up),
    ("projection transposed", [check_projection_exact], _mut_project_transposed),
    ("softmax without 1/sqrt(d)", [check_softmax_closed_form, check_softmax_vs_sdpa], _mut_prob_no_scale),
    ("query head mapped to wrong KV head", [check_softmax_vs_sdpa], _mut_prob_wrong_group),
    ("group mean instead of max", [check_group_max], _mut_group_mean),
    ("group max of unnormalised weights", [check_group_max], _mut_group_max_logits),
    ("ties to the higher index", [check_select_bruteforce], _mut_select_high_index_ties),
    ("forced set dropped", [check_select_bruteforce], _mut_select_no_forced),
    ("free slots paired descending", [check_diff_pairing_order], _mut_diff_descending_slots),
    ("reload everything", [check_diff_invariants, check_diff_worked_example], _mut_diff_reload_all),
    ("attention without normaliser", [check_attention_vs_sdpa, check_attention_special], _mut_attn_no_softmax_norm),
    ("K used as V", [check_attention_vs_sdpa, check_attention_subset_vs_sdpa], _mut_attn_k_for_v),
    ("offload threshold off by one", [check_offload_bruteforce, check_offload_boundaries], _mut_offload_last_fit),
    ("offloaded layer keeps no workspace", [check_offload_bruteforce, check_offload_boundaries],
     _mut_offload_no_workspace),
]


@pytest.mark.parametrize("name,checks,mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistakes(name, checks, mutant):
    assert not all(chk(mutant) for chk in checks), f"no pin caught: {name}"
