"""ctypes binding of libspc.so: the C entry points under the same names.

Marshalling only: tensors become device (or host) pointers, the stream
defaults to torch's current CUDA stream, a non-zero status raises SpcError.
Every computation runs in the library's CUDA kernels; if the library is
missing or cannot be loaded, the first call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspc.so")

SPC_OK = 0
STATUS_NAMES = {0: "SPC_OK", -1: "SPC_ERR_INVALID_ARG", -2: "SPC_ERR_SHAPE", -3: "SPC_ERR_CUDA",
                -4: "SPC_ERR_TIMEOUT", -5: "SPC_ERR_WORKSPACE", -6: "SPC_ERR_OVERFLOW"}

# struct layouts of include/spc.h (32 bytes each)
GATHER_VIEW_DTYPE = np.dtype([("host", "<u8"), ("slots", "<u8"), ("layer0", "<i4"),
                              ("n_layers", "<i4"), ("store_layer0", "<i4"), ("store_layers", "<i4")])
KV_VIEW_DTYPE = np.dtype([("k", "<u8"), ("v", "<u8"), ("rows", "<i8"), ("use_slots", "<i4"),
                          ("reserved", "<i4")])

_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "spc_status_string": (ctypes.c_char_p, [_I]),
    "spc_version": (_I, []),
    "spc_device_sm_count": (_I, []),
    "spc_score_select_workspace_size": (ctypes.c_size_t, [_I] * 7),
    "spc_score_select": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P,
                              _P, ctypes.c_size_t, _P]),
    "spc_score_select_stages": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P,
                                     _P, _P, ctypes.c_size_t, _P, _I]),
    "spc_elastic_diff": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "spc_gather_kv": (_I, [_P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "spc_sparse_decode_attn_workspace_size": (ctypes.c_size_t, [_I] * 6),
    "spc_sparse_decode_attn": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P,
                                    ctypes.c_size_t, _P]),
    "spc_sparse_decode_attn_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float,
                                            _P, _P]),
    "spc_host_device_pointer": (_I, [_P, ctypes.POINTER(ctypes.c_void_p)]),
    "spc_stream_read": (_I, [_P, ctypes.c_size_t, _P, _I, _P]),
    "spc_copy": (_I, [_P, _P, ctypes.c_size_t, _P]),
    "spc_fill_slots": (_I, [_P, _I, _I, _P, _I, _I, _I, _I, _I, _P]),
    "spc_store_layer": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "spc_offload_thresholds": (_I, [_I, _I, _I, _I, _I, ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)]),
    "spc_batch_select_workspace_size": (ctypes.c_size_t, [_I] * 3),
    "spc_batch_select": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, ctypes.c_size_t, _P]),
    "spc_mla_score_select_workspace_size": (ctypes.c_size_t, [_I] * 4),
    "spc_mla_score_select": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P,
                                  ctypes.c_size_t, _P, _I]),
    "spc_mla_gather": (_I, [_P, _I, _I, _P, _P, _P, _I, _I, _I, _P]),
    "spc_mla_decode_attn_workspace_size": (ctypes.c_size_t, [_I] * 3),
    "spc_mla_decode_attn": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, ctypes.c_float, _P, _P, ctypes.c_size_t,
                                 _P]),
}


class SpcError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}: "
                         f"{lib().spc_status_string(status).decode()}")


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(handle, name)
            f.restype = res
            f.argtypes = args
        _lib = handle
    return _lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return t.data_ptr()
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(t)}")


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int) -> None:
    if status != SPC_OK:
        raise SpcError(fn, status)


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


# ------------------------------------------------------------------ entry points
def spc_score_select_workspace_size(B, H, n_q, n_kv, d, cap, budget) -> int:
    return int(lib().spc_score_select_workspace_size(B, H, n_q, n_kv, d, cap, budget))


def spc_score_select(x, Wq, Wk, K_dlm, len, append, B, H, n_q, n_kv, d, cap, budget, n_sink,
                     n_recent, q_out, scores_out, selected, workspace, workspace_bytes=None,
                     stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    _check("spc_score_select", lib().spc_score_select(
        _ptr(x), _ptr(Wq), _ptr(Wk), _ptr(K_dlm), _ptr(len), int(append), B, H, n_q, n_kv, d, cap,
        budget, n_sink, n_recent, _ptr(q_out), _ptr(scores_out), _ptr(selected), _ptr(workspace),
        workspace_bytes, _stream(stream)))


SPC_STAGE_PROJECT, SPC_STAGE_SCAN, SPC_STAGE_SELECT = 1, 2, 4


def spc_score_select_stages(x, Wq, Wk, K_dlm, len, append, B, H, n_q, n_kv, d, cap, budget, n_sink,
                            n_recent, q_out, scores_out, selected, workspace, workspace_bytes=None,
                            stream=None, stages=7) -> None:
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    _check("spc_score_select_stages", lib().spc_score_select_stages(
        _ptr(x), _ptr(Wq), _ptr(Wk), _ptr(K_dlm), _ptr(len), int(append), B, H, n_q, n_kv, d, cap,
        budget, n_sink, n_recent, _ptr(q_out), _ptr(scores_out), _ptr(selected), _ptr(workspace),
        workspace_bytes, _stream(stream), int(stages)))


def spc_elastic_diff(selected, slot_pos_prev, slot_pos_next, load_slot, load_pos, n_load, B, n_kv,
                     budget, cap, stream=None) -> None:
    _check("spc_elastic_diff", lib().spc_elastic_diff(
        _ptr(selected), _ptr(slot_pos_prev), _ptr(slot_pos_next), _ptr(load_slot), _ptr(load_pos),
        _ptr(n_load), B, n_kv, budget, cap, _stream(stream)))


def spc_gather_kv(views, layer_lo, layer_hi, load_slot, load_pos, n_load, B, n_kv, d, cap, budget,
                  stream=None) -> None:
    _check("spc_gather_kv", lib().spc_gather_kv(
        _ptr(views), layer_lo, layer_hi, _ptr(load_slot), _ptr(load_pos), _ptr(n_load), B, n_kv, d,
        cap, budget, _stream(stream)))


def spc_sparse_decode_attn_workspace_size(n_layers, B, n_q, n_kv, d, budget) -> int:
    return int(lib().spc_sparse_decode_attn_workspace_size(n_layers, B, n_q, n_kv, d, budget))


def spc_sparse_decode_attn(q, views, selected, slot_pos, n_layers, B, n_q, n_kv, d, budget, scale,
                           out, workspace, workspace_bytes=None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    _check("spc_sparse_decode_attn", lib().spc_sparse_decode_attn(
        _ptr(q), _ptr(views), _ptr(selected), _ptr(slot_pos), n_layers, B, n_q, n_kv, d, budget,
        float(scale), _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream)))


SPC_ATTN_NOALLOC_SCRATCH_BYTES = 8 << 20


def spc_sparse_decode_attn_noalloc(q, views, selected, slot_pos, n_layers, B, n_q, n_kv, d, budget,
                                   scale, out, stream=None) -> None:
    """spc_sparse_decode_attn with the library's fixed scratch area instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    _check("spc_sparse_decode_attn_noalloc", lib().spc_sparse_decode_attn_noalloc(
        _ptr(q), _ptr(views), _ptr(selected), _ptr(slot_pos), n_layers, B, n_q, n_kv, d, budget,
        float(scale), _ptr(out), _stream(stream)))


def spc_host_device_pointer(host) -> int:
    out = ctypes.c_void_p()
    _check("spc_host_device_pointer", lib().spc_host_device_pointer(_ptr(host), ctypes.byref(out)))
    return int(out.value)


def spc_stream_read(src, nbytes, sink, n_blocks, stream=None) -> None:
    _check("spc_stream_read", lib().spc_stream_read(_ptr(src), nbytes, _ptr(sink), n_blocks,
                                                    _stream(stream)))


def spc_copy(dst, src, nbytes, stream=None) -> None:
    """Kernel copy between device memory and device-visible host addresses."""
    _check("spc_copy", lib().spc_copy(_ptr(dst), _ptr(src), int(nbytes), _stream(stream)))


def spc_fill_slots(views, layer_lo, layer_hi, slot_pos, B, n_kv, d, cap, budget, stream=None) -> None:
    _check("spc_fill_slots", lib().spc_fill_slots(_ptr(views), layer_lo, layer_hi, _ptr(slot_pos), B,
                                                  n_kv, d, cap, budget, _stream(stream)))


def spc_store_layer(store, src, n_kv, d, cap, rows, store_layers, layer, stream=None) -> None:
    _check("spc_store_layer", lib().spc_store_layer(_ptr(store), _ptr(src), n_kv, d, cap, rows, store_layers,
                                                    layer, _stream(stream)))


def spc_offload_thresholds(n_layers, n_kv, d, B, budget, kv_bytes) -> list:
    """Host-side memory model: n_layers + 1 context-length thresholds (the
    last one is INT64_MAX)."""
    out = (ctypes.c_int64 * (n_layers + 1))()
    _check("spc_offload_thresholds", lib().spc_offload_thresholds(n_layers, n_kv, d, B, budget,
                                                                  int(kv_bytes), out))
    return [int(v) for v in out]


def spc_batch_select_workspace_size(B, cap, budget) -> int:
    return int(lib().spc_batch_select_workspace_size(B, cap, budget))


def spc_batch_select(scores, len, B, n_kv, cap, budget, n_sink, n_recent, selected, workspace, workspace_bytes=None,
                     stream=None) -> None:
    """Batch-level selection: one Top-K per request from the max over groups,
    copied to every KV head."""
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    _check("spc_batch_select", lib().spc_batch_select(
        _ptr(scores), _ptr(len), B, n_kv, cap, budget, n_sink, n_recent, _ptr(selected), _ptr(workspace),
        workspace_bytes, _stream(stream)))


# ------------------------------------------------------------------ MLA variant
SPC_MLA_LATENT, SPC_MLA_ROPE, SPC_MLA_NOPE, SPC_MLA_V, SPC_MLA_HEADS = 512, 64, 128, 128, 16


def spc_mla_score_select_workspace_size(B, H, cap, budget) -> int:
    return int(lib().spc_mla_score_select_workspace_size(B, H, cap, budget))


def spc_mla_score_select(x, Wq, Wuk, Wdkv, C_dlm, len, append, B, H, cap, budget, n_sink, n_recent,
                         scores_out, selected, workspace, workspace_bytes=None, stream=None, stages=7) -> None:
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    _check("spc_mla_score_select", lib().spc_mla_score_select(
        _ptr(x), _ptr(Wq), _ptr(Wuk), _ptr(Wdkv), _ptr(C_dlm), _ptr(len), int(append), B, H, cap, budget,
        n_sink, n_recent, _ptr(scores_out), _ptr(selected), _ptr(workspace), workspace_bytes, _stream(stream),
        int(stages)))


def spc_mla_gather(views, layer_lo, layer_hi, load_slot, load_pos, n_load, B, cap, budget, stream=None) -> None:
    _check("spc_mla_gather", lib().spc_mla_gather(
        _ptr(views), layer_lo, layer_hi, _ptr(load_slot), _ptr(load_pos), _ptr(n_load), B, cap, budget,
        _stream(stream)))


def spc_mla_decode_attn_workspace_size(n_layers, B, budget) -> int:
    return int(lib().spc_mla_decode_attn_workspace_size(n_layers, B, budget))


def spc_mla_decode_attn(q, Wuk, Wuv, views, selected, slot_pos, n_layers, B, budget, scale, out, workspace,
                        workspace_bytes=None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    _check("spc_mla_decode_attn", lib().spc_mla_decode_attn(
        _ptr(q), _ptr(Wuk), _ptr(Wuv), _ptr(views), _ptr(selected), _ptr(slot_pos), n_layers, B, budget,
        float(scale), _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream)))


def spc_device_sm_count() -> int:
    return int(lib().spc_device_sm_count())


# ------------------------------------------------------------------ view tables
def gather_views(host_ptrs: Sequence[int], slot_ptrs: Sequence[int], layer0: Sequence[int],
                 n_layers: Sequence[int], store_layer0: Optional[Sequence[int]] = None,
                 store_layers: Optional[Sequence[int]] = None) -> np.ndarray:
    """spc_gather_view table. By default a request's store holds exactly its
    host layers (store_layer0 = layer0, store_layers = n_layers)."""
    v = np.zeros(len(host_ptrs), GATHER_VIEW_DTYPE)
    v["host"], v["slots"], v["layer0"], v["n_layers"] = host_ptrs, slot_ptrs, layer0, n_layers
    v["store_layer0"] = layer0 if store_layer0 is None else store_layer0
    v["store_layers"] = n_layers if store_layers is None else store_layers
    return v


def kv_views(k_ptrs, v_ptrs, rows, use_slots) -> np.ndarray:
    v = np.zeros(len(k_ptrs), KV_VIEW_DTYPE)
    v["k"], v["v"], v["rows"], v["use_slots"] = k_ptrs, v_ptrs, rows, use_slots
    return v


def to_device_bytes(arr: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).copy()).to(device)


__all__ = [n for n in dir() if n.startswith("spc_")] + [
    "SpcError", "lib", "gather_views", "kv_views", "to_device_bytes", "GATHER_VIEW_DTYPE",
    "KV_VIEW_DTYPE", "LIB_PATH", "SIGNATURES"]
