"""Seeded synthetic inputs for the decode hot path.

This module only draws input data: weights, caches, per-step head inputs and
LLM queries. It is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests, and it holds none of the method's arithmetic (no scoring, no
selection, no set difference, no attention).

bf16 tensors are held as ``uint16`` bit patterns (numpy has no bf16); fp32
values are encoded round-to-nearest-even.

Recipe (the stand-in for the models and datasets the pages evaluate on, which
are not available here):
  * retrieval-head weights W_q [H][n_q*d], W_k [H][n_kv*d] ~ N(0, 1/H);
  * head input x_0 ~ N(0, I_H); x_t = sqrt(H) * normalize(rho*x_{t-1} + (1-rho)*eps_t);
    x_0 is the prologue input (the last prompt token, which fills the slots
    before the first decode step), x_{t+1} the input of decode step t;
  * distilled-model key cache K_dlm[b][g][p] ~ N(0, I_d) for p < len_b, zero above;
    per (b, g) a set of planted hot positions (uniform, outside the forced sink
    and recent windows) gets K += gamma * sqrt(G) * u_g, u_g the unit direction
    of the group's summed initial query (data shaping only). A query head has
    cosine ~1/sqrt(G) with that sum, so the planted logits start about gamma
    (= 8) standard deviations above the rest for every group size;
  * LLM K/V rows ~ N(0, I_d) for every layer and position up to the capacity;
    a workload with ``host_store_copies`` = c > 0 draws c distinct contents
    and request b holds those of request b % c (``Workload.kv_source``);
  * LLM query per layer q'_{l,0} ~ N(0, I_d) rescaled to norm sqrt(d), then the
    same drift as the head input.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import os
from typing import List, Optional

import numpy as np

from .configs import Workload

# Stream tags: each tensor draws from its own SeedSequence child, so changing
# the number of steps or layers never changes any other tensor.
_TAG_WQ, _TAG_WK, _TAG_KDLM, _TAG_HOT, _TAG_X, _TAG_QLLM, _TAG_KV = 1, 2, 3, 4, 5, 6, 7
_TAG_WUK, _TAG_WDKV, _TAG_WUK_L, _TAG_WUV_L = 8, 9, 10, 11


def rng_for(seed: int, *tags: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=tuple(tags))))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    w = u >> np.uint32(16)
    w &= np.uint32(1)
    w += np.uint32(0x7FFF)
    w += u
    w >>= np.uint32(16)
    return w.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16_into(out: np.ndarray, rng: np.random.Generator, scale: float = 1.0,
                      chunk: int = 1 << 22) -> None:
    """Fill a uint16 array with bf16(N(0, scale^2)) draws."""
    flat = out.reshape(-1)
    buf = np.empty(min(chunk, flat.size), dtype=np.float32)
    for s in range(0, flat.size, chunk):
        n = min(chunk, flat.size - s)
        v = buf[:n]
        rng.standard_normal(out=v, dtype=np.float32)
        if scale != 1.0:
            v *= np.float32(scale)
        flat[s:s + n] = to_bf16_bits(v)


def _parallel(jobs, work, threads: Optional[int] = None) -> None:
    """Run work(job) for every job on a thread pool (numpy's generators and
    array operations release the GIL); jobs write disjoint outputs."""
    threads = threads or min(16, os.cpu_count() or 1)
    if threads <= 1 or len(jobs) <= 1:
        for j in jobs:
            work(j)
        return
    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, jobs))


def _drift(prev: np.ndarray, eps: np.ndarray, rho: float, norm: float) -> np.ndarray:
    v = rho * prev + (1.0 - rho) * eps
    return v * (norm / np.linalg.norm(v, axis=-1, keepdims=True))


@dataclasses.dataclass
class Inputs:
    cfg: Workload
    Wq: np.ndarray                  # u16 [H][n_q*d]
    Wk: np.ndarray                  # u16 [H][n_kv*d]
    K_dlm: np.ndarray               # u16 [B][n_kv][cap][d]
    hot: List[np.ndarray]           # per request: int64 [n_kv][hot_b] planted positions
    x: np.ndarray                   # u16 [steps+1][B][H]: x[0] prologue, x[t+1] step t
    q_llm: np.ndarray               # u16 [steps][n_layers][B][n_q][d]
    lens: np.ndarray                # int32 [B] context length at step 0


def make_inputs(cfg: Workload, steps: Optional[int] = None, n_layers: Optional[int] = None) -> Inputs:
    """Everything except the LLM K/V stores (see ``fill_llm_kv``)."""
    steps = cfg.steps if steps is None else steps
    L = cfg.n_layers if n_layers is None else n_layers
    B, H, n_q, n_kv, d, G, cap = cfg.B, cfg.H, cfg.n_q, cfg.n_kv, cfg.d, cfg.G, cfg.cap

    Wq = np.empty((H, n_q * d), np.uint16)
    _normal_bf16_into(Wq, rng_for(cfg.seed, _TAG_WQ), 1.0 / np.sqrt(H))
    Wk = np.empty((H, n_kv * d), np.uint16)
    _normal_bf16_into(Wk, rng_for(cfg.seed, _TAG_WK), 1.0 / np.sqrt(H))

    # head input sequence
    xs = np.empty((steps + 1, B, H), np.uint16)
    x0 = np.empty((B, H), np.float64)
    for b in range(B):
        r = rng_for(cfg.seed, _TAG_X, b)
        x = r.standard_normal(H)
        x0[b] = x
        for t in range(steps + 1):
            if t > 0:
                x = _drift(x, r.standard_normal(H), cfg.rho[b], np.sqrt(H))
            xs[t, b] = to_bf16_bits(x.astype(np.float32))

    # LLM queries, one drifting sequence per (layer, request, head)
    q_llm = np.empty((steps, L, B, n_q, d), np.uint16)
    for b in range(B):
        r = rng_for(cfg.seed, _TAG_QLLM, b)
        q = r.standard_normal((L, n_q, d))
        q *= np.sqrt(d) / np.linalg.norm(q, axis=-1, keepdims=True)
        for t in range(steps):
            if t > 0:
                q = _drift(q, r.standard_normal((L, n_q, d)), cfg.rho[b], np.sqrt(d))
            q_llm[t, :, b] = to_bf16_bits(q.astype(np.float32))

    # distilled-model key cache with planted hot positions (every (b, g) has
    # its own stream, so drawing them on several threads gives the same bits)
    K = np.zeros((B, n_kv, cap, d), np.uint16)
    _parallel([(b, g) for b in range(B) for g in range(n_kv)],
              lambda j: _normal_bf16_into(K[j[0], j[1], :int(cfg.lens[j[0]])],
                                          rng_for(cfg.seed, _TAG_KDLM, j[0], j[1])))
    Wq_f = bf16_bits_to_f32(Wq)
    hot = []
    for b in range(B):
        Lb = int(cfg.lens[b])
        # initial query direction of every group, only to aim the planted keys
        xq = bf16_bits_to_f32(xs[0, b]) @ Wq_f                       # [n_q*d]
        u = xq.reshape(n_kv, G, d).sum(axis=1)
        u /= np.linalg.norm(u, axis=-1, keepdims=True)
        r = rng_for(cfg.seed, _TAG_HOT, b)
        lo, hi = cfg.n_sink, max(cfg.n_sink, Lb - cfg.n_recent)
        n_hot = min(int(cfg.hot[b]), hi - lo)
        pos_b = np.empty((n_kv, n_hot), np.int64)
        for g in range(n_kv):
            pos = np.sort(r.choice(np.arange(lo, hi), size=n_hot, replace=False))
            pos_b[g] = pos
            boost = np.float32(cfg.gamma * np.sqrt(G))
            rows = bf16_bits_to_f32(K[b, g, pos]) + boost * u[g].astype(np.float32)
            K[b, g, pos] = to_bf16_bits(rows)
        hot.append(pos_b)
    return Inputs(cfg=cfg, Wq=Wq, Wk=Wk, K_dlm=K, hot=hot, x=xs, q_llm=q_llm,
                  lens=np.asarray(cfg.lens, np.int32))


def fill_llm_kv(cfg: Workload, b: int, layer0: int, out: np.ndarray, threads: Optional[int] = None) -> None:
    """Fill one request's LLM K/V rows for layers [layer0, layer0 + out.shape[0]).

    ``out`` is u16 [n_layers][2][n_kv][rows][d] (rows <= cap; the first rows of
    every (layer, K/V, head) are drawn, so a store sized to the capacity and a
    smaller prefix agree). Layer l of request b always gets the same values,
    whichever store (HBM or pinned host) it lands in.
    """
    nl = out.shape[0]
    src = cfg.kv_source(b)
    jobs = [(l, kv, g) for l in range(nl) for kv in range(2) for g in range(cfg.n_kv)]

    def work(job):
        l, kv, g = job
        _normal_bf16_into(out[l, kv, g], rng_for(cfg.seed, _TAG_KV, src, layer0 + l, kv, g))

    _parallel(jobs, work, threads)


def fill_llm_kv_store(cfg: Workload, b: int, layer_lo: int, layer_hi: int, store: np.ndarray,
                      store_layer0: int, threads: Optional[int] = None) -> None:
    """The rows of ``fill_llm_kv`` for layers [layer_lo, layer_hi) written into a
    position-major store, u16 [rows][n_kv][store_layers][2][d] (row p, head g,
    layer l, K or V at store[p, g, l - store_layer0, kv]); same values as
    ``fill_llm_kv`` gives the layer-major layout."""
    rows = store.shape[0]
    src = cfg.kv_source(b)
    jobs = [(l, kv, g) for l in range(layer_lo, layer_hi) for kv in range(2) for g in range(cfg.n_kv)]

    def work(job):
        l, kv, g = job
        tmp = np.empty((rows, cfg.d), np.uint16)
        _normal_bf16_into(tmp, rng_for(cfg.seed, _TAG_KV, src, l, kv, g))
        store[:, g, l - store_layer0, kv, :] = tmp

    _parallel(jobs, work, threads)


# ------------------------------------------------------------------ MLA
# Recipe of the MLA workloads (DeepSeek-V2-style latent attention, 16 heads):
#   * retrieval head: W_q [H][16*192] ~ N(0, 1/H) (per head 128 nope then 64
#     rope columns), W_uk [16][128][512] ~ N(0, 1/512), W_dkv [H][576] ~ N(0, 1/H);
#   * the head's latent cache C_dlm[b][p] ~ N(0, I_576) for p < len_b, zero
#     above; planted hot positions get C += gamma * sqrt(16) * u, u the unit
#     direction of the sum over heads of the heads' initial queries expressed
#     in latent coordinates, [W_uk[h]^T q_nope ; q_rope] (data shaping only),
#     so planted logits start about gamma standard deviations up;
#   * LLM: latent rows ~ N(0, I_576) per layer and position; W_uk, W_uv per
#     layer [16][128][512] ~ N(0, 1/512); queries [16][192] per layer drift as
#     for GQA with norm sqrt(192).
MLA_LAT, MLA_DC, MLA_NOPE, MLA_QK = 576, 512, 128, 192


@dataclasses.dataclass
class MlaInputs:
    cfg: Workload
    Wq: np.ndarray                  # u16 [H][16*192]
    Wuk: np.ndarray                 # u16 [16][128][512] (retrieval head)
    Wdkv: np.ndarray                # u16 [H][576]
    C_dlm: np.ndarray               # u16 [B][cap][576]
    hot: List[np.ndarray]           # per request: int64 [1][hot_b]
    x: np.ndarray                   # u16 [steps+1][B][H]
    q_llm: np.ndarray               # u16 [steps][n_layers][B][16][192]
    Wuk_llm: np.ndarray             # u16 [n_layers][16][128][512]
    Wuv_llm: np.ndarray             # u16 [n_layers][16][128][512]
    lens: np.ndarray


def make_mla_inputs(cfg: Workload, steps: Optional[int] = None, n_layers: Optional[int] = None) -> MlaInputs:
    """Everything of an MLA workload except the LLM latent stores."""
    steps = cfg.steps if steps is None else steps
    L = cfg.n_layers if n_layers is None else n_layers
    B, H, n_q, cap = cfg.B, cfg.H, cfg.n_q, cfg.cap
    Wq = np.empty((H, n_q * MLA_QK), np.uint16)
    _normal_bf16_into(Wq, rng_for(cfg.seed, _TAG_WQ), 1.0 / np.sqrt(H))
    Wuk = np.empty((n_q, MLA_NOPE, MLA_DC), np.uint16)
    _normal_bf16_into(Wuk, rng_for(cfg.seed, _TAG_WUK), 1.0 / np.sqrt(MLA_DC))
    Wdkv = np.empty((H, MLA_LAT), np.uint16)
    _normal_bf16_into(Wdkv, rng_for(cfg.seed, _TAG_WDKV), 1.0 / np.sqrt(H))
    Wuk_l = np.empty((L, n_q, MLA_NOPE, MLA_DC), np.uint16)
    Wuv_l = np.empty((L, n_q, MLA_NOPE, MLA_DC), np.uint16)
    for l in range(L):
        _normal_bf16_into(Wuk_l[l], rng_for(cfg.seed, _TAG_WUK_L, l), 1.0 / np.sqrt(MLA_DC))
        _normal_bf16_into(Wuv_l[l], rng_for(cfg.seed, _TAG_WUV_L, l), 1.0 / np.sqrt(MLA_DC))

    xs = np.empty((steps + 1, B, H), np.uint16)
    for b in range(B):
        r = rng_for(cfg.seed, _TAG_X, b)
        x = r.standard_normal(H)
        for t in range(steps + 1):
            if t > 0:
                x = _drift(x, r.standard_normal(H), cfg.rho[b], np.sqrt(H))
            xs[t, b] = to_bf16_bits(x.astype(np.float32))

    q_llm = np.empty((steps, L, B, n_q, MLA_QK), np.uint16)
    for b in range(B):
        r = rng_for(cfg.seed, _TAG_QLLM, b)
        q = r.standard_normal((L, n_q, MLA_QK))
        q *= np.sqrt(MLA_QK) / np.linalg.norm(q, axis=-1, keepdims=True)
        for t in range(steps):
            if t > 0:
                q = _drift(q, r.standard_normal((L, n_q, MLA_QK)), cfg.rho[b], np.sqrt(MLA_QK))
            q_llm[t, :, b] = to_bf16_bits(q.astype(np.float32))

    C = np.zeros((B, cap, MLA_LAT), np.uint16)
    Wq_f = bf16_bits_to_f32(Wq)
    Wuk_f = bf16_bits_to_f32(Wuk)
    hot = []
    for b in range(B):
        Lb = int(cfg.lens[b])
        _normal_bf16_into(C[b, :Lb], rng_for(cfg.seed, _TAG_KDLM, b))
        q0 = (bf16_bits_to_f32(xs[0, b]) @ Wq_f).reshape(n_q, MLA_QK)
        lat = np.einsum("hjc,hj->hc", Wuk_f, q0[:, :MLA_NOPE])
        u = np.concatenate([lat, q0[:, MLA_NOPE:]], axis=1).sum(axis=0)
        u /= np.linalg.norm(u)
        r = rng_for(cfg.seed, _TAG_HOT, b)
        lo, hi = cfg.n_sink, max(cfg.n_sink, Lb - cfg.n_recent)
        n_hot = min(int(cfg.hot[b]), hi - lo)
        pos = np.sort(r.choice(np.arange(lo, hi), size=n_hot, replace=False))
        rows = bf16_bits_to_f32(C[b, pos]) + np.float32(cfg.gamma * np.sqrt(n_q)) * u.astype(np.float32)
        C[b, pos] = to_bf16_bits(rows)
        hot.append(pos[None, :].astype(np.int64))
    return MlaInputs(cfg=cfg, Wq=Wq, Wuk=Wuk, Wdkv=Wdkv, C_dlm=C, hot=hot, x=xs, q_llm=q_llm, Wuk_llm=Wuk_l,
                     Wuv_llm=Wuv_l, lens=np.asarray(cfg.lens, np.int32))


def fill_mla_layer(cfg: Workload, b: int, layer: int, out: np.ndarray) -> None:
    """LLM latent rows of request b, one layer: u16 [rows][576] (the first
    rows of the layer's sequence, so any prefix agrees)."""
    _normal_bf16_into(out, rng_for(cfg.seed, _TAG_KV, b, layer))


def fill_mla_store(cfg: Workload, b: int, layer_lo: int, layer_hi: int, store: np.ndarray, store_layer0: int,
                   threads: Optional[int] = None) -> None:
    """``fill_mla_layer`` rows of layers [layer_lo, layer_hi) written into a
    position-major store u16 [rows][store_layers][576]."""
    rows = store.shape[0]

    def work(l):
        tmp = np.empty((rows, MLA_LAT), np.uint16)
        fill_mla_layer(cfg, b, l, tmp)
        store[:, l - store_layer0, :] = tmp

    layers = list(range(layer_lo, layer_hi))
    threads = threads or min(16, os.cpu_count() or 1)
    if threads <= 1 or len(layers) <= 1:
        for l in layers:
            work(l)
        return
    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, layers))


__all__ = ["Inputs", "make_inputs", "fill_llm_kv", "fill_llm_kv_store", "to_bf16_bits", "bf16_bits_to_f32",
           "rng_for", "MlaInputs", "make_mla_inputs", "fill_mla_layer", "fill_mla_store"]
