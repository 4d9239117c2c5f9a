"""CPU oracle for the MLA variant of the decode hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this module; the product path never calls it. Like the GQA oracle
it shares no code with the CUDA library, takes bf16 tensors as ``uint16`` bit
patterns and works in float64.

Pages cited (title, then section):
  [Blog]    "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog)
            §5: for DeepSeek's MLA the retrieval picks entries of the
            low-dimensional latent cache and only the hits are up-projected.
  [Summary] "SpeContext: Enabling Efficient Long-context Reasoning with
            Speculative Context Sparsity in LLMs" (paperlayer.ai summary)
            §4.3: with MLA the retrieval stays head-level and only the
            selected latent entries are expanded for attention.

Readings where the pages are silent (each also listed in the design notes):
  * MLA as in the DeepSeek-V2 architecture: every position caches one latent
    row of d_c = 512 values plus a d_rope = 64 decoupled key part shared by
    all heads; head h expands a latent c into its key [W_uk[h] c ; c_rope]
    (128 + 64 values) and its value W_uv[h] c (128 values); a query has 128
    "nope" and 64 rope values per head; the logit scale is 1/sqrt(192);
  * the latent row is shared by all query heads, so (as for MQA) all heads
    form one group: one selection per request, from the element-wise max of
    the heads' softmax weights;
  * the retrieval head keeps the query projection, the key up-projection
    W_uk and (when the context grows) the latent down-projection W_dkv; no
    RoPE is applied (the rope part is a plain projection), as for GQA;
  * a new latent row is rounded to bf16 once.

The attention here is written literally as the pages put it: the selected
latent rows are expanded into per-head keys and values, then ordinary softmax
attention runs over them. (The CUDA path computes the same quantity without
materialising the expanded rows.)
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence

import numpy as np

from .spc_oracle import bf16_to_f64, elastic_diff, group_scores, round_to_bf16, select

D_C = 512                   # latent width
D_ROPE = 64                 # decoupled rope key width
D_NOPE = 128                # per-head key part expanded from the latent
D_V = 128                   # per-head value width
D_LAT = D_C + D_ROPE        # one cached latent row: 576 values
D_QK = D_NOPE + D_ROPE      # per-head query / key width: 192


def mla_project(x_bits: np.ndarray, Wq_bits: np.ndarray, Wdkv_bits: Optional[np.ndarray], n_q: int):
    """q[b, h] = x_b . W_q[:, h*192:(h+1)*192] (128 nope values, then 64 rope
    values; float64, unrounded); c_new[b] = bf16(x_b . W_dkv) when W_dkv is given."""
    x = bf16_to_f64(x_bits)
    q = (x @ bf16_to_f64(Wq_bits)).reshape(x.shape[0], n_q, D_QK)
    c_new = None
    if Wdkv_bits is not None:
        c_new = round_to_bf16(x @ bf16_to_f64(Wdkv_bits))
    return q, c_new


def expand_keys(C_bits: np.ndarray, Wuk_h_bits: np.ndarray) -> np.ndarray:
    """Keys of one head for latent rows C: [W_uk[h] c[:512] ; c[512:]] per row.

    C_bits: bf16 [rows][576]; Wuk_h_bits: bf16 [128][512]. Returns float64 [rows][192].
    """
    C = bf16_to_f64(C_bits)
    k_nope = C[:, :D_C] @ bf16_to_f64(Wuk_h_bits).T
    return np.concatenate([k_nope, C[:, D_C:]], axis=1)


def expand_values(C_bits: np.ndarray, Wuv_h_bits: np.ndarray) -> np.ndarray:
    """Values of one head for latent rows C: W_uv[h] c[:512]; float64 [rows][128]."""
    return bf16_to_f64(C_bits)[:, :D_C] @ bf16_to_f64(Wuv_h_bits).T


def mla_head_probabilities(q: np.ndarray, C_bits: np.ndarray, Wuk_bits: np.ndarray, length: int) -> np.ndarray:
    """Attention weights of every head over the first `length` latent rows.

    q: float64 [n_q][192]; C_bits: bf16 [cap][576]; Wuk_bits: bf16 [n_q][128][512].
    Returns float64 [n_q][length], rows summing to 1.
    """
    n_q = q.shape[0]
    P = np.zeros((n_q, length), np.float64)
    if length == 0:
        return P
    for h in range(n_q):
        Kh = expand_keys(C_bits[:length], Wuk_bits[h])
        logits = (Kh @ q[h]) / math.sqrt(D_QK)
        w = np.exp(logits - logits.max())
        P[h] = w / w.sum()
    return P


def mla_sparse_attention(q_bits: np.ndarray, C_bits: np.ndarray, Wuk_bits: np.ndarray, Wuv_bits: np.ndarray,
                         rows: np.ndarray, scale: float) -> np.ndarray:
    """o[h] = sum_r softmax_r(q_h . key_h(C[r]) * scale) value_h(C[r]) over the
    selected latent rows r, each expanded on its own (the pages' "up-project
    only the hits").

    q_bits: bf16 [n_q][192]; C_bits: bf16 [n_rows][576]; Wuk_bits, Wuv_bits:
    bf16 [n_q][128][512]; rows: indices into C. Returns float64 [n_q][128];
    zeros when no row is kept.
    """
    n_q = q_bits.shape[0]
    q = bf16_to_f64(q_bits)
    out = np.zeros((n_q, D_V), np.float64)
    r = np.asarray(rows, dtype=np.int64)
    if r.size == 0:
        return out
    Csel = C_bits[r]
    for h in range(n_q):
        Kh = expand_keys(Csel, Wuk_bits[h])
        Vh = expand_values(Csel, Wuv_bits[h])
        logits = (Kh @ q[h]) * scale
        w = np.exp(logits - logits.max())
        out[h] = (w / w.sum()) @ Vh
    return out


def mla_gather(store: np.ndarray, slots: np.ndarray, load_slot: np.ndarray, load_pos: np.ndarray) -> None:
    """Byte copy of latent rows: slots[l, load_slot[i]] = store[l, load_pos[i]].

    store: u16 [n_layers][cap][576]; slots: u16 [n_layers][K][576].
    """
    if len(load_pos):
        slots[:, load_slot] = store[:, load_pos]


class MlaDecodeState:
    """Oracle state of an MLA batch: the retrieval head's latent cache, lengths,
    the current selection (one per request) and the slots of the host layers.

    ``stores[b]`` is u16 [n_layers][cap][576] holding the LLM's latent rows of
    every layer of request b; layers [host_layer0[b], n_layers) live in slots.
    """

    def __init__(self, C_dlm: np.ndarray, lens: Sequence[int], stores: List[np.ndarray],
                 host_layer0: Sequence[int], budget: int, n_sink: int, n_recent: int):
        self.C = np.array(C_dlm, copy=True)            # [B][cap][576]
        self.lens = [int(v) for v in lens]
        self.stores = stores
        self.host_layer0 = [int(v) for v in host_layer0]
        self.budget, self.n_sink, self.n_recent = budget, n_sink, n_recent
        B = self.C.shape[0]
        L = stores[0].shape[0]
        self.slot_pos = np.full((B, 1, budget), -1, np.int64)
        self.slots = [np.zeros((L - self.host_layer0[b], budget, D_LAT), np.uint16) for b in range(B)]
        self.S = [[np.zeros(0, np.int64)] for _ in range(B)]

    def score_select(self, x_bits, Wq_bits, Wuk_bits, Wdkv_bits, n_q, append: bool):
        """Retrieval head for every request: returns (q, c_new, P list, s list, selections)."""
        B, cap = self.C.shape[:2]
        q, c_new = mla_project(x_bits, Wq_bits, Wdkv_bits if append else None, n_q)
        if append:
            for b in range(B):
                if self.lens[b] < cap:
                    self.C[b, self.lens[b]] = c_new[b]
                    self.lens[b] += 1
        Ps, ss, sel = [], [], []
        for b in range(B):
            P = mla_head_probabilities(q[b], self.C[b], Wuk_bits, self.lens[b])
            s = group_scores(P, 1)
            Ps.append(P)
            ss.append(s)
            sel.append([select(s[0], self.budget, self.n_sink, self.n_recent)])
        return q, c_new, Ps, ss, sel

    def attention(self, q_llm_bits: np.ndarray, Wuk_llm: np.ndarray, Wuv_llm: np.ndarray,
                  scale: float) -> np.ndarray:
        """Sparse MLA attention of every layer with the current selection:
        float64 [L][B][n_q][128]. Wuk_llm, Wuv_llm: bf16 [L][n_q][128][512]."""
        L, B, n_q = q_llm_bits.shape[:3]
        out = np.zeros((L, B, n_q, D_V), np.float64)
        for l in range(L):
            for b in range(B):
                out[l, b] = mla_sparse_attention(q_llm_bits[l, b], self.stores[b][l], Wuk_llm[l], Wuv_llm[l],
                                                 self.S[b][0], scale)
        return out

    def diff_and_gather(self, new_sel):
        """Elastic diff of every request's selection and the gather of the
        missing latent rows into the host layers' slots."""
        loads = []
        for b in range(self.C.shape[0]):
            sel_pad = np.full(self.budget, -1, np.int64)
            sel_pad[:new_sel[b][0].size] = new_sel[b][0]
            ls, lp, nxt = elastic_diff(sel_pad, self.slot_pos[b, 0])
            self.slot_pos[b, 0] = nxt
            h0 = self.host_layer0[b]
            if self.slots[b].shape[0]:
                mla_gather(self.stores[b][h0:], self.slots[b], ls, lp)
            loads.append([(ls, lp)])
        self.S = [[np.asarray(new_sel[b][0])] for b in range(self.C.shape[0])]
        return loads


__all__ = ["D_C", "D_ROPE", "D_NOPE", "D_V", "D_LAT", "D_QK", "mla_project", "expand_keys", "expand_values",
           "mla_head_probabilities", "mla_sparse_attention", "mla_gather", "MlaDecodeState"]
