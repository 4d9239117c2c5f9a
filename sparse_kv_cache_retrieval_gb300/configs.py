"""The five synthetic decode workloads the hot path is checked and timed on.

Sources (page title, section):
  * "SpeContext: Enabling Efficient Long-context Reasoning with Speculative
    Context Sparsity in LLMs" (paperlayer.ai summary of arXiv 2512.00722v1):
    §7.1 (models: Llama3.1-8B / DeepSeek-R1-Distill-Llama-8B shapes),
    §7.3 (speed-up runs use a KV budget of 2048), §6.2 (layers offloaded to
    CPU DRAM, last layer first).
  * "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache" (marsggbo blog):
    §1 (32K context on Llama3.1-8B ~ 4 GB of KV), §5 (GQA / MQA rules),
    §6 (adjacent-step overlap above 80%), §7 (per-layer offload thresholds).
  * "SparseSpec-L" news post (a different paper): the "sink + recent + top-K"
    retained set; used here only for the forced sink/recent window.

Every field here is a size, a seed or a distribution parameter. Nothing in this
module computes any step of the method.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

GiB = 1 << 30
MLA_LATENT_ROW = 512 + 64      # latent + decoupled rope key, per position and layer
MLA_QK = 128 + 64              # per-head query: nope + rope values


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int                 # requests in the batch
    lens: tuple            # current context length of each request at step 0
    H: int                 # hidden size of the retrieval head input
    n_q: int               # query heads
    n_kv: int              # KV heads (GQA groups)
    d: int                 # head dimension
    budget: int            # KV budget per KV head (top-K size incl. forced set)
    n_layers: int          # LLM layers
    gpu_layers: tuple      # per request: layers [0, gpu_layers[b]) keep their full KV in HBM
    steps: int             # decode steps
    rho: tuple             # per-request drift factor of the head input and LLM queries
    hot: tuple             # per request: number of planted hot positions per KV head
    seed: int
    append: bool = False   # does every step append one token (new K row) to the context?
    cap: int = 0           # capacity (max context) of every per-request cache
    n_sink: int = 4
    n_recent: int = 64
    gamma: float = 8.0     # planted hot keys get + gamma*sqrt(G) along the group's query direction
    kv_bytes: Optional[int] = None   # GPU memory for the LLM KV: set = adaptive layer offload
    mla: bool = False      # MLA attention: one 576-value latent row per position (n_kv = 1, d = 128)
    layers_per_launch: int = 16   # attention/gather layer chunk of the step schedule
    front_after: str = "select"   # the next step's projection + key scan start after this step's
                                  # select, or after its last attention ("attention")
    host_store_copies: int = 0    # distinct LLM K/V contents in the batch: request b holds the K/V of
                                  # request b % copies (0: every request its own). Lets a batch whose
                                  # host stores would not fit in the box's memory share one pinned
                                  # store per distinct content; selections, loads and bytes moved
                                  # stay per request
    note: str = ""

    @property
    def G(self) -> int:
        return self.n_q // self.n_kv

    def host_layers(self, b: int) -> int:
        return self.n_layers - self.gpu_layers[b]

    def kv_source(self, b: int) -> int:
        """The request whose LLM K/V contents request b holds."""
        return b % self.host_store_copies if self.host_store_copies else b

    @property
    def row_elems(self) -> int:
        """bf16 values one position holds in one layer: K and V of every KV
        head, or one MLA latent row (512 latent + 64 rope values)."""
        return MLA_LATENT_ROW if self.mla else self.n_kv * 2 * self.d

    def kv_layer_bytes(self, length: int) -> int:
        """Bytes of one layer's KV for one request at the given length (bf16)."""
        return length * self.row_elems * 2

    def host_store_bytes(self) -> int:
        return sum(self.host_layers(b) * self.kv_layer_bytes(self.cap) for b in range(self.B))

    def hbm_kv_bytes(self) -> int:
        return sum(self.gpu_layers[b] * self.kv_layer_bytes(self.cap) for b in range(self.B))


def _split_by_threshold(lens, n_layers, n_kv, d, budget, allowance_bytes):
    """Per-request count of HBM-resident layers under a fixed HBM allowance.

    Reading of the blog §7 / summary §6.2 for a fixed threshold: every offloaded
    layer keeps a budget-sized workspace in HBM; requests, in order, each keep
    as many leading layers in HBM as the remaining allowance pays for (the last
    layers are the ones offloaded first).
    """
    per_row = n_kv * 2 * d * 2
    ws = budget * per_row
    remaining = allowance_bytes - len(lens) * n_layers * ws
    out = []
    for L in lens:
        extra = L * per_row - ws
        n = n_layers if extra <= 0 else max(0, min(n_layers, remaining // extra))
        remaining -= n * max(extra, 0)
        out.append(int(n))
    return tuple(out)


def _cfg3_lens(seed: int, B: int):
    import numpy as np
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    lens = rng.integers(8192, 16384, size=B, endpoint=True)
    rho = rng.uniform(0.7, 0.95, size=B)
    return tuple(int(v) for v in lens), tuple(float(r) for r in rho)


def _build() -> dict:
    # Schedules: the link-bound workloads whose select/diff/attention chain is
    # slowed by the next step's key scan running beside it (cfg2, cfg3) start
    # that scan after the step's last attention (measured on one GB300:
    # cfg2 135.1 vs 138.4 us/step, cfg3 1435 vs 1455); where the chain itself
    # is the bound (cfg1, cfg4b, MLA) the scan overlaps it (cfg1 27.4 vs 34.0,
    # cfg4b 521 vs 651, MLA 95.3 vs 106.8); cfg5 is indifferent (2781 vs 2779).
    cfgs = {}
    cfgs["cfg1"] = Workload(
        name="cfg1_b1_ctx4096_gqa32x8_budget512_2layers",
        B=1, lens=(4096,), H=4096, n_q=32, n_kv=8, d=128, budget=512, n_layers=2,
        gpu_layers=(0,), steps=8, rho=(0.9,), hot=(64,), seed=0, cap=4096,
        note="PR1 reference shape: 64 planted hot positions, sinks 0-3 and recent 64 forced")
    cfgs["cfg2"] = Workload(
        name="cfg2_b1_ctx32768_gqa32x8_budget2048_32layers_host",
        B=1, lens=(32768,), H=4096, n_q=32, n_kv=8, d=128, budget=2048, n_layers=32,
        gpu_layers=(0,), steps=64, rho=(0.9,), hot=(328,), seed=1, cap=32768, front_after="attention",
        note="Llama3.1-8B-shaped GQA; 32-layer KV (4 GiB) in pinned host; hot set 1%")
    lens3, rho3 = _cfg3_lens(2, 16)
    cap3 = max(lens3)
    cfgs["cfg3"] = Workload(
        name="cfg3_b16_ragged8k-16k_gqa32x8_budget1024_32layers_split",
        B=16, lens=lens3, H=4096, n_q=32, n_kv=8, d=128, budget=1024, n_layers=32,
        gpu_layers=_split_by_threshold(lens3, 32, 8, 128, 1024, 12 * GiB),
        steps=32, rho=rho3, hot=tuple(max(1, L // 100) for L in lens3), seed=2, cap=cap3, front_after="attention",
        note="ragged batch; HBM/host split per request from a 12 GiB HBM allowance")
    cfgs["cfg4a"] = Workload(
        name="cfg4a_b4_ctx2048+256_append_gqa32x8_budget2048_32layers_host",
        B=4, lens=(2048,) * 4, H=4096, n_q=32, n_kv=8, d=128, budget=2048, n_layers=32,
        gpu_layers=(0,) * 4, steps=256, rho=(0.9,) * 4, hot=(20,) * 4, seed=3, append=True,
        cap=2048 + 256, note="long reasoning phase A: one token appended per step")
    cfgs["cfg4b"] = Workload(
        name="cfg4b_b4_ctx131072+256_append_gqa32x8_budget2048_32layers_host",
        B=4, lens=(131072,) * 4, H=4096, n_q=32, n_kv=8, d=128, budget=2048, n_layers=32,
        gpu_layers=(0,) * 4, steps=256, rho=(0.9,) * 4, hot=(1310,) * 4, seed=3, append=True,
        cap=131072 + 256, note="long reasoning phase B: continued from a 128K prefilled state")
    # cfg5's 8 x 79 host layers are 158 GiB of K/V, more than the GPU machine's
    # host memory holds pinned beside everything else: requests b and b + 2
    # share their K/V contents, so two pinned stores of 19.75 GiB serve the
    # batch. Every request still selects, diffs and gathers its own positions
    # into its own slots, so the bytes moved per step are unchanged.
    cfgs["cfg5"] = Workload(
        name="cfg5_b8_ctx65536_gqa64x8_budget4096_80layers",
        B=8, lens=(65536,) * 8, H=8192, n_q=64, n_kv=8, d=128, budget=4096, n_layers=80,
        gpu_layers=(1,) * 8, steps=64, rho=(0.85,) * 8, hot=(327,) * 8, seed=4, cap=65536,
        host_store_copies=2,
        note="70B-shaped GQA; layer 0 in HBM, 79 layers in pinned host; hot set 0.5%; "
             "two distinct K/V contents (request b holds request b % 2's)")
    # (one KV head: 8 x 79 host layers are 20 GiB, every request keeps its own)
    cfgs["cfg5mqa"] = dataclasses.replace(
        cfgs["cfg5"], name="cfg5mqa_b8_ctx65536_mqa64x1_budget4096_80layers", n_kv=1, host_store_copies=0,
        note="MQA variant of cfg5: all 64 query heads form one group")
    # MLA (DeepSeek-V2-Lite shapes: hidden 2048, 16 heads, latent 512 + rope
    # 64, 27 layers): the cfg2 setting (32K context, budget 2048, every layer's
    # latent cache in pinned host memory) on a latent cache. Its gathers are
    # small (1152 B per load and layer, 88% reused), so one attention launch
    # over all 27 layers beats chunks that overlap gathers with attention
    # (measured 94.9 vs 108.2 us/step at 16 layers per launch)
    cfgs["mla"] = Workload(
        name="mla_b1_ctx32768_mla16_latent512_budget2048_27layers_host",
        B=1, lens=(32768,), H=2048, n_q=16, n_kv=1, d=128, budget=2048, n_layers=27,
        gpu_layers=(0,), steps=64, rho=(0.9,), hot=(328,), seed=6, cap=32768, mla=True, layers_per_launch=27,
        note="MLA variant: head-level selection over the latent cache, only selected latent rows "
             "loaded and up-projected; latent cache (27 layers, 0.95 GiB) in pinned host")
    # adaptive memory management on a growing context: 4 requests from 4096
    # positions, one token per step, GPU KV memory for 4127 positions of all
    # 32 layers per request, so the first threshold falls 32 steps in and a
    # further layer leaves every ~70-100 steps
    row4 = 2 * 8 * 128 * 2
    cfgs["c3"] = Workload(
        name="c3_b4_ctx4096+512_append_gqa32x8_budget2048_32layers_adaptive",
        B=4, lens=(4096,) * 4, H=4096, n_q=32, n_kv=8, d=128, budget=2048, n_layers=32,
        gpu_layers=(32,) * 4, steps=512, rho=(0.9,) * 4, hot=(41,) * 4, seed=5, append=True,
        cap=4096 + 512, kv_bytes=4 * 32 * 4127 * row4,
        note="progressive per-layer offload driven by the memory model's thresholds")
    return cfgs


CONFIGS = _build()


def scaled(cfg: Workload, *, B: Optional[int] = None, lens=None, n_layers: Optional[int] = None,
           steps: Optional[int] = None, cap: Optional[int] = None, budget: Optional[int] = None,
           H: Optional[int] = None, name_suffix: str = "_small") -> Workload:
    """A smaller copy of a workload (same structure) for tests the oracle finishes quickly."""
    B = cfg.B if B is None else B
    lens = tuple(cfg.lens[:B]) if lens is None else tuple(lens)
    n_layers = cfg.n_layers if n_layers is None else n_layers
    budget = cfg.budget if budget is None else budget
    base_cap = max(lens) + (cfg.steps if cfg.append else 0)
    cap = base_cap if cap is None else cap
    gpu = tuple(min(g, n_layers) for g in cfg.gpu_layers[:B])
    if len(gpu) < B:
        gpu = gpu + (0,) * (B - len(gpu))
    frac = [h / max(1, L) for h, L in zip(cfg.hot, cfg.lens)]
    frac = frac + [frac[-1]] * (B - len(frac))
    hot = tuple(max(1, int(round(f * L))) for f, L in zip(frac, lens))
    rho = tuple(cfg.rho[:B]) + (cfg.rho[-1],) * max(0, B - len(cfg.rho))
    return dataclasses.replace(cfg, name=cfg.name + name_suffix, B=B, lens=lens, n_layers=n_layers,
                               gpu_layers=gpu, steps=cfg.steps if steps is None else steps,
                               rho=rho, hot=hot, cap=cap, budget=budget,
                               H=cfg.H if H is None else H)


def describe(cfg: Workload) -> dict:
    return {
        "workload": cfg.name, "batch": cfg.B, "context": list(cfg.lens) if cfg.B <= 4 else
        [min(cfg.lens), max(cfg.lens)], "hidden": cfg.H, "heads_q": cfg.n_q, "heads_kv": cfg.n_kv,
        "head_dim": cfg.d, "budget": cfg.budget, "layers": cfg.n_layers,
        "host_layers": [cfg.host_layers(b) for b in range(cfg.B)] if cfg.B <= 4 else
        sum(cfg.host_layers(b) for b in range(cfg.B)),
        "sinks": cfg.n_sink, "recent": cfg.n_recent, "seed": cfg.seed,
        **({"attention": "mla", "latent_row": MLA_LATENT_ROW} if cfg.mla else {}),
        **({"host_store_copies": cfg.host_store_copies,
            "host_store_note": f"request b holds the LLM K/V contents of request b % {cfg.host_store_copies} "
                               "(shared pinned stores); selections, loads and bytes moved are per request"}
           if cfg.host_store_copies else {}),
    }


__all__ = ["Workload", "CONFIGS", "scaled", "describe", "GiB", "MLA_LATENT_ROW", "MLA_QK"]
