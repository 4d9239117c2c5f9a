"""CPU oracle for the SpeContext decode-step hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this module. The product path never calls it and never falls back to
it. It shares no code with the CUDA library and imports nothing from the
package: bf16 tensors come in as ``uint16`` bit patterns and every step is
written out here from its definition, in float64.

Pages cited (title, then section):
  [Blog]    "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog)
  [Summary] "SpeContext: Enabling Efficient Long-context Reasoning with
            Speculative Context Sparsity in LLMs" (paperlayer.ai summary of
            arXiv 2512.00722v1)
  [SparseSpec-L] news post on SparseSpec-L (a different paper; only its
            "sinks + recent window + top-K" retained set is used)

Readings where the pages are silent (each also listed in the design notes):
  * the head input is a hidden vector x (the embedding output); no RoPE;
  * softmax per query head comes before the group max ([Blog] §5 says the
    group max is taken over attention scores, [Summary] §4.3 over attention
    weights);
  * sinks 0..n_sink-1 and the last n_recent positions are always kept, counted
    inside the budget; when len <= budget every position is kept;
  * Top-K ties go to the lower position;
  * free slots and missing positions are paired in ascending order
    (slot index, position); slots left over become empty (-1);
  * attention over an empty row set returns zeros.

Every function here has a pin in ``tests/test_oracle_pins.py`` (closed forms,
invariants, brute force on tiny inputs, the page's worked example, a library
routine on the special case that reduces to it).
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np


# --------------------------------------------------------------------------
# bf16 encoding (plain definition: 1 sign, 8 exponent, 7 stored mantissa bits)
# --------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns: the 16 bits are the top half of an IEEE fp32."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16, ties to even; return bit patterns.

    bf16 keeps 8 significant bits. Writing v = f * 2**e with 0.5 <= |f| < 1,
    the bf16 value is rint(f * 256) / 256 * 2**e, and ``np.rint`` rounds halves
    to even. Normal range only (|v| in [2**-126, 2**128)), which the data here
    never leaves.
    """
    v = np.asarray(v, dtype=np.float64)
    f, e = np.frexp(v)
    r = np.ldexp(np.rint(f * 256.0) / 256.0, e)
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# --------------------------------------------------------------------------
# a1: retrieval-head projection ([Blog] §5 C1: the head keeps the embedding and
#     the Query/Key projections; [Summary] §4.3)
# --------------------------------------------------------------------------
def project(x_bits: np.ndarray, Wq_bits: np.ndarray, Wk_bits: Optional[np.ndarray],
            n_q: int, n_kv: int, d: int) -> Tuple[np.ndarray, Optional[np.ndarray]]:
    """q[b, h, :] = x_b . W_q[:, h*d:(h+1)*d] (float64, unrounded);
    k_new[b, g, :] = bf16(x_b . W_k[:, g*d:(g+1)*d]) when W_k is given."""
    x = bf16_to_f64(x_bits)
    q = (x @ bf16_to_f64(Wq_bits)).reshape(x.shape[0], n_q, d)
    k_new = None
    if Wk_bits is not None:
        k_new = round_to_bf16((x @ bf16_to_f64(Wk_bits)).reshape(x.shape[0], n_kv, d))
    return q, k_new


# --------------------------------------------------------------------------
# a2: per-head attention weights softmax(q K^T / sqrt(d)) ([Blog] §2 formula)
# --------------------------------------------------------------------------
def head_probabilities(q: np.ndarray, K_bits: np.ndarray, length: int) -> np.ndarray:
    """Attention weights of every query head of one request over its context.

    q: float64 [n_q][d]; K_bits: bf16 [n_kv][cap][d]; query head h reads KV head
    h // (n_q / n_kv). Returns float64 [n_q][length], each row summing to 1.
    """
    n_q, d = q.shape
    n_kv = K_bits.shape[0]
    G = n_q // n_kv
    P = np.zeros((n_q, length), np.float64)
    if length == 0:
        return P
    for g in range(n_kv):
        K = bf16_to_f64(K_bits[g, :length])
        for h in range(g * G, (g + 1) * G):
            logits = (K @ q[h]) / math.sqrt(d)
            w = np.exp(logits - logits.max())
            P[h] = w / w.sum()
    return P


# --------------------------------------------------------------------------
# a3: GQA group score ([Blog] §5: element-wise max over the query heads of a
#     group, then Top-K per group; MQA = one group; MHA = group of one)
# --------------------------------------------------------------------------
def group_scores(P: np.ndarray, n_kv: int) -> np.ndarray:
    """s[g, p] = max over query heads h of group g of P[h, p]; float64 [n_kv][len]."""
    n_q, length = P.shape
    G = n_q // n_kv
    s = np.empty((n_kv, length), np.float64)
    for g in range(n_kv):
        s[g] = P[g * G:(g + 1) * G].max(axis=0)
    return s


# --------------------------------------------------------------------------
# a4: forced set + Top-K under the KV budget ([Blog] §2: top-K per head, K is
#     the KV budget; [SparseSpec-L] and [Summary] §2.2: sinks + recent window)
# --------------------------------------------------------------------------
def forced_positions(length: int, n_sink: int, n_recent: int) -> np.ndarray:
    f = set(range(min(n_sink, length))) | set(range(max(0, length - n_recent), length))
    return np.array(sorted(f), dtype=np.int64)


def select(s: np.ndarray, budget: int, n_sink: int, n_recent: int) -> np.ndarray:
    """Positions kept for one KV head, ascending, size min(budget, len).

    All positions when len <= budget. Otherwise the forced sinks and recent
    window, plus the budget-|F| best other positions ranked by score
    (descending), ties to the lower position.
    """
    length = s.shape[0]
    if length <= budget:
        return np.arange(length, dtype=np.int64)
    F = forced_positions(length, n_sink, n_recent)
    is_forced = np.zeros(length, bool)
    is_forced[F] = True
    cand = np.nonzero(~is_forced)[0]
    k = budget - F.size
    # lexsort sorts by the last key first: primary -score, secondary position
    order = np.lexsort((cand, -s[cand]))
    taken = cand[order[:k]]
    return np.sort(np.concatenate([F, taken]))


def batch_level_select(s_groups: np.ndarray, budget: int, n_sink: int, n_recent: int) -> np.ndarray:
    """The batch-level alternative the pages compare head-level retrieval
    with ([Blog] §5: every head's weights merged into one Top-K): one selection
    for the whole request from the element-wise max over ALL groups' scores,
    shared by every KV head. s_groups: float64 [n_kv][len]."""
    return select(np.asarray(s_groups, np.float64).max(axis=0), budget, n_sink, n_recent)


# --------------------------------------------------------------------------
# a5: elastic loading ([Blog] §6: to_load = S_now - S_last, worked example
#     S_last={1,8,21,35}, S_now={1,8,21,50} -> {50}; [Summary] §5.4: reuse the
#     resident entries and overwrite in place under a fixed budget)
# --------------------------------------------------------------------------
def elastic_diff(selected: np.ndarray, slot_pos: np.ndarray):
    """Set difference between the new selection and the resident slots.

    selected: int [K] new positions (-1 = none); slot_pos: int [K] position
    held by each slot (-1 = empty). Returns (load_slot, load_pos, slot_pos_next)
    with load_pos = sorted(S_new - S_resident), load_slot = the free slots
    (slot position not in S_new, or empty) in ascending slot order, paired
    one-to-one with load_pos; unpaired free slots become empty.
    """
    S_new = set(int(p) for p in selected if p >= 0)
    keep = np.array([int(p) >= 0 and int(p) in S_new for p in slot_pos], bool)
    resident = set(int(p) for p, k in zip(slot_pos, keep) if k)
    load_pos = np.array(sorted(S_new - resident), dtype=np.int64)
    free = np.nonzero(~keep)[0]
    assert free.size >= load_pos.size
    load_slot = free[:load_pos.size].astype(np.int64)
    nxt = np.where(keep, np.asarray(slot_pos, np.int64), -1)
    nxt[load_slot] = load_pos
    return load_slot, load_pos, nxt


# --------------------------------------------------------------------------
# a6: gather of the missing rows into the slots ([Blog] §4 prefetcher, §7
#     budget-sized workspace of an offloaded layer; [Summary] §5.4 in place)
# --------------------------------------------------------------------------
def gather(store: np.ndarray, slots: np.ndarray, load_slot: Sequence[np.ndarray],
           load_pos: Sequence[np.ndarray]) -> None:
    """Byte copy: slots[l, kv, g, load_slot[g][i]] = store[l, kv, g, load_pos[g][i]].

    store: u16 [n_layers][2][n_kv][cap][d]; slots: u16 [n_layers][2][n_kv][K][d].
    """
    for g in range(store.shape[2]):
        if len(load_pos[g]):
            slots[:, :, g, load_slot[g]] = store[:, :, g, load_pos[g]]


# --------------------------------------------------------------------------
# a7: sparse decode attention over the kept rows ([Blog] §2 formula applied to
#     the selected rows; §4: the LLM runs on the sparse KV prepared earlier)
# --------------------------------------------------------------------------
def sparse_attention(q_bits: np.ndarray, K_bits: np.ndarray, V_bits: np.ndarray,
                     rows: Sequence[np.ndarray], scale: float) -> np.ndarray:
    """o[h] = sum_r softmax_r(q_h . K[g, r] * scale) V[g, r] over r in rows[g].

    q_bits: bf16 [n_q][d]; K_bits/V_bits: bf16 [n_kv][n_rows][d]; rows[g]:
    row indices kept for KV head g. Returns float64 [n_q][d]; zeros when a
    group keeps no row.
    """
    n_q, d = q_bits.shape
    n_kv = K_bits.shape[0]
    G = n_q // n_kv
    q = bf16_to_f64(q_bits)
    out = np.zeros((n_q, d), np.float64)
    for h in range(n_q):
        r = np.asarray(rows[h // G], dtype=np.int64)
        if r.size == 0:
            continue
        K = bf16_to_f64(K_bits[h // G, r])
        V = bf16_to_f64(V_bits[h // G, r])
        logits = (K @ q[h]) * scale
        w = np.exp(logits - logits.max())
        out[h] = (w / w.sum()) @ V
    return out


# --------------------------------------------------------------------------
# C3: adaptive memory management ([Blog] §7: sequence-length thresholds from
#     the model's layers, KV heads and head dimension, the free GPU memory,
#     the concurrent requests and the KV budget; past each threshold the last
#     layer still on the GPU moves to CPU memory and keeps a budget-sized
#     workspace; [Summary] §6.2 and §6.2.1)
# --------------------------------------------------------------------------
def kv_row_bytes(n_kv: int, d: int, elem_bytes: int = 2) -> int:
    """GPU bytes one position costs in one layer: K and V, every KV head."""
    return 2 * n_kv * d * elem_bytes


def gpu_kv_bytes(length: int, n_offloaded: int, n_layers: int, n_kv: int, d: int, B: int,
                 budget: int) -> int:
    """GPU KV bytes of B requests of `length` positions when the last
    `n_offloaded` layers live in CPU memory: every layer still on the GPU holds
    all `length` rows, every offloaded layer a `budget`-row workspace."""
    rows = (n_layers - n_offloaded) * length + n_offloaded * budget
    return B * rows * kv_row_bytes(n_kv, d)


def offload_thresholds(n_layers: int, n_kv: int, d: int, B: int, budget: int,
                       kv_bytes: int) -> List[int]:
    """threshold[k] (k = 0..n_layers-1): the shortest context at which k
    offloaded layers no longer fit in `kv_bytes`, so the (k+1)-th must go.
    threshold[n_layers] is None (nothing left to offload). Written from the
    definition: the largest length that fits with k offloaded layers, plus one.
    Raises ValueError when even every layer offloaded does not fit."""
    per_req_rows = kv_bytes // (B * kv_row_bytes(n_kv, d))   # rows one request may hold
    if per_req_rows < n_layers * budget:
        raise ValueError("the budget workspaces of all layers exceed the KV memory")
    out: List[int] = []
    for k in range(n_layers):
        fit = (per_req_rows - k * budget) // (n_layers - k)   # longest length that fits
        out.append(int(fit) + 1)
    out.append(None)
    return out


def layers_to_offload(length: int, thresholds: Sequence[Optional[int]], n_offloaded: int) -> int:
    """The runtime rule of [Blog] §7: while the length has reached the
    threshold for the current number of offloaded layers, offload one more.
    Returns the new number of offloaded layers (never fewer than before)."""
    n = n_offloaded
    while thresholds[n] is not None and length >= thresholds[n]:
        n += 1
    return n


# --------------------------------------------------------------------------
# the decode step ([Blog] §4 loop: select for the next step, load only the
# difference, run the LLM on the previously prepared sparse KV)
# --------------------------------------------------------------------------
class DecodeState:
    """Oracle state of a batch: key cache, lengths, current selection, slots.

    ``stores[b]`` is u16 [n_layers][2][n_kv][cap][d] holding every layer of
    request b (the oracle needs no HBM/host split: it reads rows by position);
    ``host_layer0[b]`` is the first layer whose KV lives in slots.
    """

    def __init__(self, K_dlm: np.ndarray, lens: Sequence[int], stores: List[np.ndarray],
                 host_layer0: Sequence[int], budget: int, n_sink: int, n_recent: int):
        self.K = np.array(K_dlm, copy=True)
        self.lens = [int(v) for v in lens]
        self.stores = stores
        self.host_layer0 = [int(v) for v in host_layer0]
        self.budget, self.n_sink, self.n_recent = budget, n_sink, n_recent
        B, n_kv = self.K.shape[0], self.K.shape[1]
        L = stores[0].shape[0]
        d = self.K.shape[3]
        self.slot_pos = np.full((B, n_kv, budget), -1, np.int64)
        self.slots = [np.zeros((L - self.host_layer0[b], 2, n_kv, budget, d), np.uint16)
                      for b in range(B)]
        self.S = [[np.zeros(0, np.int64) for _ in range(n_kv)] for _ in range(B)]

    def score_select(self, x_bits, Wq_bits, Wk_bits, n_q, append: bool):
        """a1-a4 for every request; returns (q, P list, s list, selections)."""
        B, n_kv, cap, d = self.K.shape
        q, k_new = project(x_bits, Wq_bits, Wk_bits if append else None, n_q, n_kv, d)
        if append:
            for b in range(B):
                if self.lens[b] < cap:
                    self.K[b, :, self.lens[b]] = k_new[b]
                    self.lens[b] += 1
        Ps, ss, sel = [], [], []
        for b in range(B):
            P = head_probabilities(q[b], self.K[b], self.lens[b])
            s = group_scores(P, n_kv)
            Ps.append(P)
            ss.append(s)
            sel.append([select(s[g], self.budget, self.n_sink, self.n_recent) for g in range(n_kv)])
        return q, k_new, Ps, ss, sel

    def attention(self, q_llm_bits: np.ndarray, scale: float) -> np.ndarray:
        """a7 for all layers with the current selection: float64 [L][B][n_q][d]."""
        L, B, n_q, d = q_llm_bits.shape
        out = np.zeros((L, B, n_q, d), np.float64)
        for l in range(L):
            for b in range(B):
                st = self.stores[b]
                out[l, b] = sparse_attention(q_llm_bits[l, b], st[l, 0], st[l, 1], self.S[b], scale)
        return out

    def diff_and_gather(self, new_sel):
        """a5 + a6: returns per (b, g) (load_slot, load_pos)."""
        loads = []
        B, n_kv = self.slot_pos.shape[:2]
        for b in range(B):
            lb = []
            for g in range(n_kv):
                sel_pad = np.full(self.budget, -1, np.int64)
                sel_pad[:new_sel[b][g].size] = new_sel[b][g]
                ls, lp, nxt = elastic_diff(sel_pad, self.slot_pos[b, g])
                self.slot_pos[b, g] = nxt
                lb.append((ls, lp))
            h0 = self.host_layer0[b]
            if self.slots[b].shape[0]:
                gather(self.stores[b][h0:], self.slots[b], [x[0] for x in lb], [x[1] for x in lb])
            loads.append(lb)
        self.S = [[np.asarray(new_sel[b][g]) for g in range(n_kv)] for b in range(B)]
        return loads


__all__ = ["bf16_to_f64", "round_to_bf16", "project", "head_probabilities", "group_scores",
           "forced_positions", "select", "batch_level_select", "elastic_diff", "gather", "sparse_attention", "kv_row_bytes",
           "gpu_kv_bytes", "offload_thresholds", "layers_to_offload", "DecodeState"]
