"""The decode step on CUDA streams: the retrieval head's projection and key
scan (stream C), select, diff and per layer chunk attention (stream A), and
the in-place gather of the next step's missing rows (stream B; two
alternating streams with gather_streams=2), for GQA caches or an MLA latent
cache, with head-level (the method) or batch-level selection.

Method ordering: "ASPLOS'26 | SpeContext 让小模型先圈出重要 KV Cache"
(marsggbo blog) §4 -- the retrieval head predicts the positions of step t+1
while the LLM runs step t on the sparse KV prepared at step t-1, and the
prefetcher moves only the missing rows on another CUDA stream; §6 -- only
S_now - S_last is loaded; "SpeContext: Enabling Efficient Long-context
Reasoning with Speculative Context Sparsity in LLMs" (paperlayer.ai summary)
§5.1 and §5.4 (in place). The pages omit the pipeline warm-up; here a
prologue runs the head once on the last prompt token and loads its whole
selection before the first decode step.

Ordering (per layer chunk c, step t, parity p = t % 2):
  C: wait select(t-1); project + key scan of x_{t+1}          (the "front")
  A: wait front(t); select -> selected[1-p]; diff(selected[1-p], slot_pos[p])
     -> slot_pos[1-p], loads[1-p]; for each chunk c: wait gather(c, t-1);
     attention(c, selected[p], slot_pos[p]); record attn(c, t)
  B: wait attn(c, t); gather(c, loads[1-p]) into the slots; record gather(c, t)
Inside a run of steps, the front of step t+1 is issued right after select(t)
(it only needs the scan scratch that select(t) has consumed and the length
select(t) has advanced), so it overlaps diff(t) and attention(t), or, with
front_after="attention", after step t's last attention. The in-place
overwrite of chunk c always follows the attention that reads the old rows,
and the next step's attention on c always follows it.

PyTorch provides device memory, pinned host memory, streams, events and CUDA
graphs; every step of the method runs in libspc's kernels.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Union

import numpy as np
import torch

from . import binding as spc
from .configs import MLA_LATENT_ROW, MLA_QK, Workload
from .synth import Inputs, MlaInputs, fill_llm_kv, fill_llm_kv_store, fill_mla_layer, fill_mla_store


def _dev_u16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device)


class DecodePipeline:
    """Device-resident state and the pipelined decode step for one workload.

    ``inputs`` comes from ``synth.make_inputs`` (``synth.make_mla_inputs`` for
    an MLA workload); ``n_layers`` may be smaller than the workload's to keep
    tests small. LLM KV of layers [0, gpu_layers[b]) lives in HBM (attention
    reads it by position); the other layers live in pinned host memory
    (``host_stores``) and are reached through budget-sized HBM slots. A
    position of one layer holds K and V rows of every KV head ([2][n_kv][d],
    GQA) or one 576-value latent row (MLA, n_kv = 1).
    """

    def __init__(self, cfg: Workload, inputs: Union[Inputs, MlaInputs], *, device: str = "cuda",
                 n_layers: Optional[int] = None, layers_per_launch: int = 16,
                 host_io: bool = False, timing: bool = False, fill_threads: Optional[int] = None,
                 gather_streams: int = 1, kv_bytes: Optional[int] = None,
                 offload_policy: str = "progressive", elastic: bool = True, front_after: Optional[str] = None,
                 retrieval: str = "head"):
        self.cfg = cfg
        self.inp = inputs
        self.dev = torch.device(device)
        self.L = cfg.n_layers if n_layers is None else n_layers
        self.B, self.H, self.n_q, self.n_kv, self.d = cfg.B, cfg.H, cfg.n_q, cfg.n_kv, cfg.d
        self.K, self.cap = cfg.budget, cfg.cap
        self.G = cfg.G
        self.mla = cfg.mla
        self.qdim = MLA_QK if self.mla else self.d           # per-head LLM query width
        self.scale = 1.0 / math.sqrt(self.qdim)
        self.gpu_layers = [min(int(g), self.L) for g in cfg.gpu_layers]
        self.host_io = host_io
        self.timing = timing
        self.timing_kinds = None        # with timing on: the kinds that get event pairs (None: all)
        dev = self.dev
        B, L, K, n_kv, d, cap = self.B, self.L, self.K, self.n_kv, self.d, self.cap

        # retrieval head (MLA: W_uk of the head, the latent down-projection
        # for appends and the head's latent cache in place of W_k / K_dlm)
        self.Wq = _dev_u16(inputs.Wq, dev)
        self.len = torch.from_numpy(inputs.lens.astype(np.int32)).to(dev)
        if self.mla:
            if kv_bytes is not None:
                raise ValueError("adaptive layer offload is implemented for GQA caches only")
            self.Wuk = _dev_u16(inputs.Wuk, dev)
            self.Wk = _dev_u16(inputs.Wdkv, dev)
            self.K_dlm = _dev_u16(inputs.C_dlm, dev)
            self.Wuk_llm = _dev_u16(inputs.Wuk_llm[:self.L], dev)
            self.Wuv_llm = _dev_u16(inputs.Wuv_llm[:self.L], dev)
            ws_bytes = spc.spc_mla_score_select_workspace_size(B, self.H, cap, K)
        else:
            self.Wk = _dev_u16(inputs.Wk, dev)
            self.K_dlm = _dev_u16(inputs.K_dlm, dev)
            ws_bytes = spc.spc_score_select_workspace_size(B, self.H, self.n_q, n_kv, d, cap, K)
        self.ws_score = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        n_steps = inputs.q_llm.shape[0]
        self.x_dev = _dev_u16(inputs.x, dev)                                  # [steps+1][B][H]
        self.q_dev = _dev_u16(inputs.q_llm[:, :L], dev)                       # [steps][L][B][n_q][qdim]
        self.n_steps = n_steps

        # selection state, double-buffered by step parity
        def i32(*shape, fill=0):
            return torch.full(shape, fill, dtype=torch.int32, device=dev)
        self.selected = i32(2, B, n_kv, K, fill=-1)
        self.slot_pos = i32(2, B, n_kv, K, fill=-1)
        self.load_slot = i32(2, B, n_kv, K)
        self.load_pos = i32(2, B, n_kv, K)
        self.n_load = i32(2, B, n_kv)
        self.no_resident = i32(B, n_kv, K, fill=-1)
        self.group_scores = torch.zeros(B, n_kv, cap, dtype=torch.float32, device=dev)
        self.selected_head = i32(2, B, n_kv, K, fill=-1)
        self.ws_batch = (torch.zeros(spc.spc_batch_select_workspace_size(B, cap, K), dtype=torch.uint8, device=dev)
                         if retrieval == "batch" else None)
        # attention output, double-buffered by step parity (the copy of step t's
        # output to the host may still run while step t+1 writes); `out` is the
        # buffer of the step issued last
        self.out_buf = torch.zeros(2, L, B, self.n_q, d, dtype=torch.float32, device=dev)
        self.out = self.out_buf[0]

        # adaptive memory management (C3, "ASPLOS'26 | SpeContext ..." §7):
        # context-length thresholds from the memory model; each request starts
        # with as many trailing layers offloaded as its context requires, and
        # maybe_offload() moves further layers as the context grows
        if offload_policy not in ("progressive", "static"):
            raise ValueError("offload_policy is 'progressive' or 'static'")
        # elastic=False is the comparison the pages measure elastic loading
        # against: every step reloads its whole selection (the diff sees no
        # resident slot)
        self.elastic = elastic
        # where the next step's projection and key scan (the front) start
        # inside a run of steps: right after this step's select ("select"),
        # or after its last attention ("attention"), so that they do not
        # compete with this step's diff and attention for the SMs and HBM
        front_after = cfg.front_after if front_after is None else front_after
        if front_after not in ("select", "attention"):
            raise ValueError("front_after is 'select' or 'attention'")
        self.front_after = front_after
        # retrieval="batch" is the alternative the pages compare head-level
        # retrieval with ([Blog] §5): one Top-K per request from the max over
        # all groups' scores, shared by every KV head. The head-level
        # selection of the same step is kept in selected_head for comparison;
        # record_scores keeps the group scores in head-level mode too
        if retrieval not in ("head", "batch"):
            raise ValueError("retrieval is 'head' or 'batch'")
        self.retrieval = retrieval
        self.record_scores = False
        self.adaptive = kv_bytes is not None
        self.kv_bytes = kv_bytes
        self.offload_policy = offload_policy
        self.thresholds = None
        self.offload_log: List[tuple] = []        # (step, request, layer) of every offload
        self._pending_free: List[torch.Tensor] = []
        if self.adaptive:
            self.thresholds = spc.spc_offload_thresholds(L, n_kv, d, B, K, int(kv_bytes))
            self.gpu_layers = [L - self._offload_count(self._kv_length(b, -1), 0) for b in range(B)]

        # LLM KV: per-layer HBM full caches, pinned host stores and HBM slots.
        # A request's host store and slots cover layers [store_base[b], L): its
        # host layers in the static split, every layer in the adaptive one (so
        # a layer can move without reallocating)
        self.hbm: List[List[Optional[torch.Tensor]]] = []
        self.host_stores: List[Optional[torch.Tensor]] = []
        self.slots: List[Optional[torch.Tensor]] = []
        self.store_base: List[int] = []
        self._store_dev: List[int] = []
        for b in range(B):
            ng = self.gpu_layers[b]
            s0 = 0 if self.adaptive else ng
            layers = []
            for l in range(ng):
                if self.mla:
                    buf = np.empty((cap, MLA_LATENT_ROW), np.uint16)
                    fill_mla_layer(cfg, b, l, buf)
                    layers.append(_dev_u16(buf, dev))
                else:
                    buf = np.empty((1, 2, n_kv, cap, d), np.uint16)
                    fill_llm_kv(cfg, b, l, buf, threads=fill_threads)
                    layers.append(_dev_u16(buf[0], dev))
                del buf
            self.hbm.append(layers)
            src = cfg.kv_source(b)
            if L - s0 > 0 and src != b and not self.adaptive and not self.mla and \
                    self.store_base[src] == s0 and self.gpu_layers[src] == ng:
                # request b holds request src's K/V contents: share its pinned
                # store (the gather still reads b's own positions into b's slots)
                self.host_stores.append(self.host_stores[src])
                self.slots.append(torch.zeros((L - s0, 2, n_kv, K, d), dtype=torch.int16, device=dev))
                self._store_dev.append(self._store_dev[src])
            elif L - s0 > 0:
                # position-major [cap][n_kv][layers][2][d] (MLA: [cap][layers][576]):
                # one (position, head) holds every stored layer's row(s) in one host page
                if self.mla:
                    hs = torch.empty((cap, L - s0, MLA_LATENT_ROW), dtype=torch.int16, pin_memory=True)
                    if L - ng > 0:
                        fill_mla_store(cfg, b, ng, L, hs.numpy().view(np.uint16), s0, threads=fill_threads)
                    sl = torch.zeros((L - s0, K, MLA_LATENT_ROW), dtype=torch.int16, device=dev)
                else:
                    hs = torch.empty((cap, n_kv, L - s0, 2, d), dtype=torch.int16, pin_memory=True)
                    if L - ng > 0:
                        fill_llm_kv_store(cfg, b, ng, L, hs.numpy().view(np.uint16), s0, threads=fill_threads)
                    sl = torch.zeros((L - s0, 2, n_kv, K, d), dtype=torch.int16, device=dev)
                self.host_stores.append(hs)
                self.slots.append(sl)
                self._store_dev.append(spc.spc_host_device_pointer(hs))
            else:
                self.host_stores.append(None)
                self.slots.append(None)
                self._store_dev.append(0)
            self.store_base.append(s0)
        self._slot_layer_bytes = K * cfg.row_elems * 2
        self.gviews = spc.to_device_bytes(self._gather_view_table(), dev)
        if self.adaptive:
            # the GPU's first access to each page of a pinned buffer pays for the
            # page's address translation over the link; an adaptive pipeline
            # writes its stores only when a layer moves, so read every page once
            # here (setup) instead of inside the first offload
            sink = torch.zeros(spc.spc_device_sm_count() * 4, dtype=torch.int32, device=dev)
            for b, hs in enumerate(self.host_stores):
                if hs is not None:
                    spc.spc_stream_read(self._store_dev[b], hs.numel() * 2 // 16 * 16, sink, sink.numel())
            torch.cuda.synchronize()
            del sink

        # attention views [L][B]
        table = np.concatenate([self._attn_view_row(l, b) for l in range(L) for b in range(B)])
        self.aviews = spc.to_device_bytes(table, dev)
        self.aview_stride = 32 * B

        # layer chunks, streams, events
        lc = max(1, min(layers_per_launch, L))
        self.chunks = [(l0, min(L, l0 + lc)) for l0 in range(0, L, lc)]
        # the workspace a launch needs is not monotone in its layer count (a
        # shorter chunk may split its segments over more CTAs): the largest
        # over the chunk lengths in use
        ws_attn = max((spc.spc_mla_decode_attn_workspace_size(l1 - l0, B, K) if self.mla else
                       spc.spc_sparse_decode_attn_workspace_size(l1 - l0, B, self.n_q, n_kv, d, K))
                      for l0, l1 in self.chunks)
        self.ws_attn = torch.zeros(ws_attn, dtype=torch.uint8, device=dev)
        # The gathers (B) get the highest priority: a gather CTA needs a whole
        # SM and waits for one to drain, and the next free SM should go to it
        # rather than to another attention CTA (the link is the step's bound;
        # on the 80-layer 70B-shaped workload 9.43 vs 9.91 ms/step). Select,
        # diff and attention (A) come next; the front (C) has a whole step of
        # slack, so its CTAs yield to both
        hi, lo = self._priorities()
        mid = hi + 1 if hi < lo else hi
        self.sA = torch.cuda.Stream(device=dev, priority=mid)
        self.sB = torch.cuda.Stream(device=dev, priority=hi)
        # gathers of consecutive layer chunks alternate over `gather_streams`
        # streams: with two, one launch's ramp-down overlaps the next one's
        # ramp-up; with one, the gathers never share the host link, so each
        # chunk's rows land as early as the link allows
        if gather_streams not in (1, 2):
            raise ValueError("gather_streams must be 1 or 2")
        self.sBs = [self.sB] + [torch.cuda.Stream(device=dev, priority=hi)
                                for _ in range(gather_streams - 1)]
        self.sC = torch.cuda.Stream(device=dev, priority=lo)
        self.e_front = torch.cuda.Event()
        self.e_sel = torch.cuda.Event()
        self._front_issued = None      # step whose front is in flight on stream C
        self._range_end = None         # end of the current run of steps (look-ahead bound)
        self.e_attn = [torch.cuda.Event() for _ in self.chunks]
        self.e_gath = [torch.cuda.Event() for _ in self.chunks]
        self._gather_pending = [False] * len(self.chunks)
        # host I/O: H2D of the LLM queries one step ahead (stream H), D2H of
        # each step's output and selection (stream D), per parity events
        self.sH = torch.cuda.Stream(device=dev, priority=hi)
        self.sD = torch.cuda.Stream(device=dev, priority=lo)
        self.e_q = [torch.cuda.Event(), torch.cuda.Event()]
        self.e_attn_end = [torch.cuda.Event(), torch.cuda.Event()]
        self.e_d2h = [torch.cuda.Event(), torch.cuda.Event()]
        self._reset_io_state()

        self.host_io = False
        if host_io:
            self.enable_host_io()
        self.h2d_bytes_per_step = (B * self.H + L * B * self.n_q * self.qdim) * 2
        self.d2h_bytes_per_step = L * B * self.n_q * d * 4 + B * n_kv * K * 4

        # optional timing events: (stream, kind, start, end) per launch
        self._timed: List[tuple] = []
        self._all_events: List[torch.cuda.Event] = []
        self._capturing = False
        self._prologue_done = False
        self._step_events: Optional[List[torch.cuda.Event]] = None

    # ------------------------------------------------------------------ layout
    def _gather_view_table(self) -> np.ndarray:
        host, slots, layer0, n_host, st0, stn = [], [], [], [], [], []
        for b in range(self.B):
            ng, s0 = self.gpu_layers[b], self.store_base[b]
            if self.slots[b] is not None and ng < self.L:
                host.append(self._store_dev[b])
                slots.append(self.slots[b].data_ptr() + (ng - s0) * self._slot_layer_bytes)
            else:
                host.append(0)
                slots.append(0)
            layer0.append(ng)
            n_host.append(self.L - ng)
            st0.append(s0)
            stn.append(self.L - s0)
        return spc.gather_views(host, slots, layer0, n_host, st0, stn)

    def _attn_view_row(self, l: int, b: int) -> np.ndarray:
        if l < self.gpu_layers[b]:
            base, rows, use = self.hbm[b][l], self.cap, 0
        else:
            base, rows, use = self.slots[b][l - self.store_base[b]], self.K, 1
        if self.mla:
            return spc.kv_views([base.data_ptr()], [0], [rows], [use])
        return spc.kv_views([base[0].data_ptr()], [base[1].data_ptr()], [rows], [use])

    def host_slots(self, b: int) -> Optional[torch.Tensor]:
        """Slots of request b's host layers, [L - gpu_layers[b]][2][n_kv][K][d]."""
        if self.slots[b] is None or self.gpu_layers[b] >= self.L:
            return None
        return self.slots[b][self.gpu_layers[b] - self.store_base[b]:]

    # ------------------------------------------------------------------ C3
    def _kv_length(self, b: int, t: int) -> int:
        """Context length of request b while step t runs (t = -1: the prompt):
        an appending workload adds one row per step."""
        n = int(self.inp.lens[b]) + (t + 1 if self.cfg.append and t >= 0 else 0)
        return min(n, self.cap)

    def _offload_count(self, length: int, n_off: int) -> int:
        """Offloaded layers a request of `length` positions needs. progressive:
        the rule of [Blog] §7 (while the length has reached the threshold of
        the current count, offload one more layer); static: nothing until the
        first threshold, then every layer at once."""
        thr = self.thresholds
        if self.offload_policy == "static":
            return self.L if length >= thr[0] else n_off
        while n_off < self.L and length >= thr[n_off]:
            n_off += 1
        return n_off

    def maybe_offload(self, t: int) -> int:
        """Before issuing step t: offload the layers the memory model asks for.
        Returns the number of layers moved. Each move waits for the GPU to
        drain (the view tables change), copies the layer's cache to the
        pinned host store, fills its budget workspace from the HBM cache
        with the slot map step t attends with, and repoints the views."""
        if not self.adaptive:
            return 0
        moved = 0
        for b in range(self.B):
            length = self._kv_length(b, t)
            target = self._offload_count(length, self.L - self.gpu_layers[b])
            while self.L - self.gpu_layers[b] < target:
                if self._capturing:
                    raise RuntimeError("an offload cannot be captured in a CUDA graph")
                if moved == 0:
                    torch.cuda.synchronize()
                    self._pending_free.clear()
                self._offload_layer(b, t % 2)
                self.offload_log.append((t, b, self.gpu_layers[b]))
                moved += 1
        return moved

    def _offload_layer(self, b: int, p: int) -> None:
        l = self.gpu_layers[b] - 1
        s0, sA = self.store_base[b], self.sA
        src = self.hbm[b][l]
        with torch.cuda.stream(sA):
            # every row of the layer up to the capacity: rows past the current
            # length stand for the K/V rows the LLM writes as the context grows
            # (the workloads prefill them), so the store is complete from here on
            spc.spc_store_layer(self._store_dev[b], src, self.n_kv, self.d, self.cap, self.cap, self.L - s0, l - s0,
                                stream=sA)
            host = [0] * self.B
            slots = [0] * self.B
            n_layers = [0] * self.B
            host[b] = src.data_ptr()
            slots[b] = self.slots[b][l - s0].data_ptr()
            n_layers[b] = 1
            fill_views = spc.to_device_bytes(spc.gather_views(host, slots, [l] * self.B, n_layers), self.dev)
            spc.spc_fill_slots(fill_views, l, l + 1, self.slot_pos[p], self.B, self.n_kv, self.d, self.cap,
                               self.K, stream=sA)
            self.gpu_layers[b] = l
            self.hbm[b][l] = None
            row = torch.from_numpy(self._attn_view_row(l, b).view(np.uint8).copy()).to(self.dev)
            off = l * self.aview_stride + b * 32
            self.aviews[off:off + 32].copy_(row)
            self.gviews.copy_(torch.from_numpy(self._gather_view_table().view(np.uint8).copy()).to(self.dev))
        # the copy and the fill read the old cache: keep it until the next drain
        self._pending_free.extend([src, fill_views])

    def kv_hbm_bytes(self) -> int:
        """GPU KV bytes the memory model charges now: full caches of HBM layers
        at the current length plus one budget workspace per offloaded layer."""
        tot = 0
        for b in range(self.B):
            n_off = self.L - self.gpu_layers[b]
            tot += ((self.L - n_off) * self._kv_length(b, -1) + n_off * self.K) * 2 * self.n_kv * self.d * 2
        return tot

    @staticmethod
    def _priorities():
        """(highest, lowest) stream priority of the device (lower is higher)."""
        try:
            lo, hi = torch.cuda.Stream.priority_range()
        except Exception:
            return 0, 0
        return hi, lo

    def _reset_io_state(self) -> None:
        self._q_issued = None                 # step whose query copy is in flight
        self._attn_end_rec = [False, False]   # e_attn_end[parity] recorded in this run
        self._d2h_pending = [False, False]    # e_d2h[parity] recorded in this run

    def enable_host_io(self) -> None:
        """Switch to end-to-end mode: every step copies its head input and LLM
        queries from pinned host memory and copies its attention output and
        selection back to pinned host memory. The head input goes with the
        front (stream C); the queries of step t+1 are copied while step t runs
        (stream H, double-buffered); outputs go back on stream D."""
        if self.host_io:
            return
        inputs, B, L, d, dev = self.inp, self.B, self.L, self.d, self.dev
        n_steps = self.n_steps
        self.x_host = torch.from_numpy(inputs.x.view(np.int16).copy()).pin_memory()
        self.q_host = torch.from_numpy(np.ascontiguousarray(inputs.q_llm[:, :L]).view(np.int16)).pin_memory()
        self.x_stage = torch.empty(B, self.H, dtype=torch.int16, device=dev)
        self.q_stage = torch.empty(2, L, B, self.n_q, self.qdim, dtype=torch.int16, device=dev)
        self.out_host = torch.empty((n_steps, L, B, self.n_q, d), dtype=torch.float32).pin_memory()
        self.sel_host = torch.empty((n_steps, B, self.n_kv, self.K), dtype=torch.int32).pin_memory()
        # transfers run as libspc copy kernels on the device-visible addresses
        # of the pinned buffers (a copy-engine transfer to or from host memory
        # inside a CUDA graph stalled every step)
        self._x_bytes = B * self.H * 2
        self._q_bytes = L * B * self.n_q * self.qdim * 2
        self._out_bytes = L * B * self.n_q * d * 4
        self._sel_bytes = B * self.n_kv * self.K * 4
        self._x_dev_host = spc.spc_host_device_pointer(self.x_host)
        self._q_dev_host = spc.spc_host_device_pointer(self.q_host)
        self._out_dev_host = spc.spc_host_device_pointer(self.out_host)
        self._sel_dev_host = spc.spc_host_device_pointer(self.sel_host)
        # the GPU's first write to each page of a pinned buffer pays for the
        # page's address translation over the link: touch the output buffers
        # once here, so the steps write to translated pages
        with torch.cuda.stream(self.sD):
            z = torch.zeros(max(self._out_bytes, self._sel_bytes, self._q_bytes, self._x_bytes) // 4 + 1,
                            dtype=torch.float32, device=dev)
            for t in range(n_steps):
                spc.spc_copy(self._out_dev_host + t * self._out_bytes, z, self._out_bytes, stream=self.sD)
                spc.spc_copy(self._sel_dev_host + t * self._sel_bytes, z, self._sel_bytes, stream=self.sD)
                spc.spc_copy(z, self._q_dev_host + t * self._q_bytes, self._q_bytes, stream=self.sD)
            for t in range(n_steps + 1):
                spc.spc_copy(z, self._x_dev_host + t * self._x_bytes, self._x_bytes, stream=self.sD)
        self.sD.synchronize()
        del z
        self.host_io = True

    # ------------------------------------------------------------------ pieces
    def _score_select(self, x, out_sel, append: int, stream, stages: int = 7, q_out=None, scores_out=None):
        c = self.cfg
        if self.mla:
            spc.spc_mla_score_select(x, self.Wq, self.Wuk, self.Wk, self.K_dlm, self.len, append, self.B, self.H,
                                     self.cap, self.K, c.n_sink, c.n_recent, scores_out, out_sel, self.ws_score,
                                     stream=stream, stages=stages)
            return
        spc.spc_score_select_stages(x, self.Wq, self.Wk, self.K_dlm, self.len, append, self.B, self.H,
                                    self.n_q, self.n_kv, self.d, self.cap, self.K, c.n_sink, c.n_recent,
                                    q_out, scores_out, out_sel, self.ws_score, stream=stream,
                                    stages=stages)

    def _select(self, pn, append: int, stream):
        """The select stage into selected[pn]: head-level, or (retrieval =
        "batch") head-level into selected_head[pn] and the batch-level
        selection from its group scores into selected[pn]."""
        if self.retrieval == "batch":
            self._score_select(self.x_dev[0], self.selected_head[pn], append, stream, 4, scores_out=self.group_scores)
            c = self.cfg
            spc.spc_batch_select(self.group_scores, self.len, self.B, self.n_kv, self.cap, self.K, c.n_sink,
                                 c.n_recent, self.selected[pn], self.ws_batch, stream=stream)
        else:
            self._score_select(self.x_dev[0], self.selected[pn], append, stream, 4,
                               scores_out=self.group_scores if self.record_scores else None)

    def _diff(self, pn, p, stream):
        prev = self.slot_pos[p] if self.elastic else self.no_resident
        spc.spc_elastic_diff(self.selected[pn], prev, self.slot_pos[pn], self.load_slot[pn],
                             self.load_pos[pn], self.n_load[pn], self.B, self.n_kv, self.K, self.cap,
                             stream=stream)

    def _gather(self, pn, l0, l1, stream):
        if self.mla:
            spc.spc_mla_gather(self.gviews, l0, l1, self.load_slot[pn], self.load_pos[pn], self.n_load[pn], self.B,
                               self.cap, self.K, stream=stream)
            return
        spc.spc_gather_kv(self.gviews, l0, l1, self.load_slot[pn], self.load_pos[pn], self.n_load[pn],
                          self.B, self.n_kv, self.d, self.cap, self.K, stream=stream)

    def _attn(self, q_layers, out, p, l0, l1, stream):
        views = self.aviews.data_ptr() + l0 * self.aview_stride
        if self.mla:
            spc.spc_mla_decode_attn(q_layers[l0].data_ptr(), self.Wuk_llm[l0].data_ptr(),
                                    self.Wuv_llm[l0].data_ptr(), views, self.selected[p], self.slot_pos[p], l1 - l0,
                                    self.B, self.K, self.scale, out[l0].data_ptr(), self.ws_attn, stream=stream)
            return
        spc.spc_sparse_decode_attn(q_layers[l0].data_ptr(), views, self.selected[p], self.slot_pos[p],
                                   l1 - l0, self.B, self.n_q, self.n_kv, self.d, self.K, self.scale,
                                   out[l0].data_ptr(), self.ws_attn, stream=stream)

    def _timing_event(self):
        # Inside a capture a timing event must be an external record node.
        # Every event a graph records stays referenced in self._timed for the
        # pipeline's lifetime: destroying an event a graph still records into
        # is undefined behaviour at launch.
        if self._capturing:
            return torch.cuda.Event(enable_timing=True, external=True)
        return torch.cuda.Event(enable_timing=True)

    def _is_timed(self, kind) -> bool:
        return self.timing and (self.timing_kinds is None or kind in self.timing_kinds)

    def _timed_call(self, kind, stream, fn):
        if not self._is_timed(kind):
            fn()
            return
        s, e = self._timing_event(), self._timing_event()
        self._all_events.extend((s, e))
        s.record(stream)
        fn()
        e.record(stream)
        self._timed.append((kind, s, e))

    # ------------------------------------------------------------------ steps
    def prologue(self) -> None:
        """Head on the last prompt token; load its whole selection (no append)."""
        sA = self.sA
        with torch.cuda.stream(sA):
            self.len.copy_(torch.from_numpy(self.inp.lens.astype(np.int32)))
            self.slot_pos[1].fill_(-1)
            self._score_select(self.x_dev[0], self.selected[0], 0, sA, 3)
            self._select(0, 0, sA)
            self._diff(0, 1, sA)
            self._gather(0, 0, self.L, sA)
        sA.synchronize()
        self._gather_pending = [False] * len(self.chunks)
        self._front_issued = None
        self._prologue_done = True

    def _front(self, t: int, after: Optional[torch.cuda.Event] = None) -> None:
        """Projection and key scan of step t (input x[t+1]) on stream C, after
        the select of step t-1 issued in this run (none before the first), and
        after `after` when given."""
        sC = self.sC
        append = 1 if self.cfg.append else 0
        if self._front_issued is not None:
            sC.wait_event(self.e_sel)
        else:
            sC.wait_stream(self.sA)
        if after is not None:
            sC.wait_event(after)
        pn = (t + 1) % 2
        if self.host_io:
            spc.spc_copy(self.x_stage, self._x_dev_host + (t + 1) * self._x_bytes, self._x_bytes, stream=sC)
            x = self.x_stage
        else:
            x = self.x_dev[t + 1]
        if self._is_timed("project") or self._is_timed("key_scan"):
            self._timed_call("project", sC, lambda: self._score_select(x, self.selected[pn], append, sC, 1))
            self._timed_call("key_scan", sC, lambda: self._score_select(x, self.selected[pn], append, sC, 2))
        else:
            self._score_select(x, self.selected[pn], append, sC, 3)
        self.e_front.record(sC)
        self._front_issued = t

    def _q_copy(self, t: int) -> None:
        """H2D copy of the LLM queries of step t into q_stage[t % 2] on stream
        H, after the attention of step t-2 (the buffer's last reader)."""
        sH, par = self.sH, t % 2
        if self._attn_end_rec[par]:
            sH.wait_event(self.e_attn_end[par])
        else:
            sH.wait_stream(self.sA)
        spc.spc_copy(self.q_stage[par], self._q_dev_host + t * self._q_bytes, self._q_bytes, stream=sH)
        self.e_q[par].record(sH)
        self._q_issued = t

    def step(self, t: int) -> None:
        """Issue decode step t (uses inputs x[t+1] and q_llm[t])."""
        sA = self.sA
        p, pn = t % 2, (t + 1) % 2
        append = 1 if self.cfg.append else 0
        lookahead = self._range_end is not None and t + 1 < self._range_end
        if self.adaptive:
            self.maybe_offload(t)
        if self._step_events is not None:
            ev = self._timing_event()
            self._all_events.append(ev)
            ev.record(sA)
            self._step_events.append(ev)
        if self._front_issued != t:
            self._front(t)
        if self.host_io and self._q_issued != t:
            self._q_copy(t)
        sA.wait_event(self.e_front)
        if self.host_io:
            if self._d2h_pending[p]:
                # step t-2's copies still read selected[pn] and out_buf[p]
                sA.wait_event(self.e_d2h[p])
            sA.wait_event(self.e_q[p])
            q_layers = self.q_stage[p]
        else:
            q_layers = self.q_dev[t]
        out_t = self.out_buf[p]
        self.out = out_t
        # the select stage reads only the front's scratch; x is not used
        self._timed_call("select", sA, lambda: self._select(pn, append, sA))
        self.e_sel.record(sA)
        if lookahead and t + 2 < len(self.inp.x) and self.front_after == "select":
            self._front(t + 1)
        self._timed_call("diff", sA, lambda: self._diff(pn, p, sA))
        for c, (l0, l1) in enumerate(self.chunks):
            if self._gather_pending[c]:
                sA.wait_event(self.e_gath[c])
            self._timed_call("attention", sA, lambda: self._attn(q_layers, out_t, p, l0, l1, sA))
            self.e_attn[c].record(sA)
            sg = self.sBs[c % len(self.sBs)]
            sg.wait_event(self.e_attn[c])
            self._timed_call("gather", sg, lambda: self._gather(pn, l0, l1, sg))
            self.e_gath[c].record(sg)
            self._gather_pending[c] = True
        self.e_attn_end[p].record(sA)
        self._attn_end_rec[p] = True
        if lookahead and t + 2 < len(self.inp.x) and self.front_after == "attention":
            self._front(t + 1, after=self.e_attn_end[p])
        if self.host_io:
            if lookahead and t + 1 < self.n_steps:
                self._q_copy(t + 1)
            sD = self.sD
            sD.wait_event(self.e_attn_end[p])
            spc.spc_copy(self._out_dev_host + t * self._out_bytes, out_t, self._out_bytes, stream=sD)
            spc.spc_copy(self._sel_dev_host + t * self._sel_bytes, self.selected[pn], self._sel_bytes, stream=sD)
            self.e_d2h[p].record(sD)
            self._d2h_pending[p] = True

    def _side_streams(self):
        return self.sBs + [self.sC, self.sH, self.sD]

    def join(self) -> None:
        for sg in self._side_streams():
            self.sA.wait_stream(sg)
        self._front_issued = None
        self._reset_io_state()

    def run(self, t0: int, n: int) -> None:
        self._range_end = t0 + n
        try:
            for t in range(t0, t0 + n):
                self.step(t)
        finally:
            self._range_end = None
        self.join()

    def capture_timed(self, t0: int, n: int):
        """capture() with a timing event recorded on stream A at the start of
        every step and after the last one; returns (graph, events). The
        pipeline keeps the events alive."""
        self._step_events = []
        try:
            g = self.capture(t0, n, _final_event=True)
        finally:
            evs, self._step_events = self._step_events, None
        return g, evs

    def capture(self, t0: int, n: int, _final_event: bool = False) -> torch.cuda.CUDAGraph:
        """A CUDA graph of steps [t0, t0+n) (both streams, forked and joined).

        Replay it on stream A (``with torch.cuda.stream(pipe.sA): g.replay()``).
        With timing on, the graph records external timing events that the
        pipeline keeps alive; read them after a replay."""
        g = torch.cuda.CUDAGraph()
        self.join()
        saved = list(self._gather_pending)
        self._gather_pending = [False] * len(self.chunks)
        self._capturing = True
        try:
            with torch.cuda.graph(g, stream=self.sA):
                for sg in self._side_streams():
                    sg.wait_stream(self.sA)
                self._front_issued = None
                self._reset_io_state()
                self._range_end = t0 + n
                for t in range(t0, t0 + n):
                    self.step(t)
                self.join()
                if _final_event and self._step_events is not None:
                    ev = self._timing_event()
                    self._all_events.append(ev)
                    ev.record(self.sA)
                    self._step_events.append(ev)
        finally:
            self._capturing = False
            self._range_end = None
        self._gather_pending = [False] * len(self.chunks)
        del saved
        return g

    def timed_summary(self) -> Dict[str, dict]:
        """Per kernel kind: launches and mean duration (ms) of the timed calls."""
        res: Dict[str, dict] = {}
        for kind, s, e in self._timed:
            r = res.setdefault(kind, {"launches": 0, "total_ms": 0.0})
            r["launches"] += 1
            r["total_ms"] += s.elapsed_time(e)
        for r in res.values():
            r["mean_ms"] = r["total_ms"] / max(1, r["launches"])
        return res

    def reset_timing(self) -> None:
        """Forget the recorded (kind, start, end) triples; the events stay alive."""
        self._timed = []

    # ------------------------------------------------------------------ accounting
    def loads_per_step(self, parity: int) -> np.ndarray:
        return self.n_load[parity].cpu().numpy()

    def key_scan_bytes(self, lens) -> int:
        row = MLA_LATENT_ROW if self.mla else self.n_kv * self.d
        return int(sum(int(L) for L in lens) * row * 2)


__all__ = ["DecodePipeline"]
