"""A bounded device-side wait that runs out: the attention kernel must record
SPC_ERR_TIMEOUT in its workspace status word, end by itself, and leave the
context usable, so that the next call on the same workspace matches the
oracle again.

The wait is made to run out without any GPU fault: the library's test build
(the same sources compiled with -DSPC_TEST_HOOKS into libspc_testhooks.so,
never into libspc.so) exports spc_test_starve_attention(calls, cycles), which
makes the next `calls` launches run with a producer warp that issues no copies
and publishes no stage, and with a wait limit of `cycles` clock cycles. Every
consumer warp's first wait then gives up, marks the warp dead (it runs its
loop without waiting, so every barrier is still reached) and the kernel
returns.
"""
import ctypes
import math
import time

import numpy as np
import pytest
import torch

import oracle.spc_oracle as O
from oracle.checks import ATTN_ATOL
from sparse_kv_cache_retrieval_gb300 import _build
from sparse_kv_cache_retrieval_gb300 import binding as spc

pytestmark = pytest.mark.gpu
DEV = "cuda"
SPC_ERR_TIMEOUT = -4


@pytest.fixture(scope="module")
def hooks():
    path = _build.build(test_hooks=True)
    lib = ctypes.CDLL(path)
    _P, _I = ctypes.c_void_p, ctypes.c_int
    lib.spc_test_starve_attention.restype = _I
    lib.spc_test_starve_attention.argtypes = [_I, ctypes.c_longlong]
    lib.spc_sparse_decode_attn.restype = _I
    lib.spc_sparse_decode_attn.argtypes = list(spc.SIGNATURES["spc_sparse_decode_attn"][1])
    lib.spc_sparse_decode_attn_workspace_size.restype = ctypes.c_size_t
    lib.spc_sparse_decode_attn_workspace_size.argtypes = [_I] * 6
    return lib


def _case(rng, L, B, n_q, n_kv, K):
    d = 128
    keep, kp, vp, rows, use = [], [], [], [], []
    for _ in range(L * B):
        bits = O.round_to_bf16(rng.standard_normal((2, n_kv, K, d)))
        t = torch.from_numpy(bits.view(np.int16)).to(DEV)
        keep.append((bits, t))
        kp.append(t[0].data_ptr()); vp.append(t[1].data_ptr()); rows.append(K); use.append(1)
    views = spc.to_device_bytes(spc.kv_views(kp, vp, rows, use), DEV)
    q = O.round_to_bf16(rng.standard_normal((L, B, n_q, d)) * 1.5)
    slot = np.full((B, n_kv, K), -1, np.int32)
    kept = []
    for b in range(B):
        kb = []
        for g in range(n_kv):
            m = int(rng.integers(K // 2, K + 1))
            s = np.sort(rng.choice(K, size=m, replace=False))
            slot[b, g, s] = rng.choice(100000, size=m, replace=False)
            kb.append(s)
        kept.append(kb)
    want = np.zeros((L, B, n_q, d))
    for l in range(L):
        for b in range(B):
            bits = keep[l * B + b][0]
            want[l, b] = O.sparse_attention(q[l, b], bits[0], bits[1], kept[b], 1 / math.sqrt(d))
    sel = torch.from_numpy(np.where(slot >= 0, slot, -1).astype(np.int32)).to(DEV)
    return keep, views, torch.from_numpy(q.view(np.int16)).to(DEV), sel, \
        torch.from_numpy(slot).to(DEV), want


def _call(lib, case, out, ws, L, B, n_q, n_kv, K):
    keep, views, q, sel, slot, _ = case
    st = torch.cuda.current_stream().cuda_stream
    return lib.spc_sparse_decode_attn(q.data_ptr(), views.data_ptr(), sel.data_ptr(), slot.data_ptr(), L, B, n_q,
                                      n_kv, 128, K, 1 / math.sqrt(128), out.data_ptr(), ws.data_ptr(),
                                      ws.numel(), st)


@pytest.mark.parametrize("L,B,n_q,n_kv,K", [
    (2, 1, 32, 8, 2048),     # clusters of several CTAs, split partials merged through the workspace
    (1, 2, 64, 1, 512),      # MQA: 64 heads on one KV head
])
def test_wait_that_runs_out_reports_timeout_and_the_next_call_recovers(hooks, L, B, n_q, n_kv, K):
    lib = hooks
    case = _case(np.random.default_rng(7 + n_q), L, B, n_q, n_kv, K)
    want = case[-1]
    ws = torch.zeros(lib.spc_sparse_decode_attn_workspace_size(L, B, n_q, n_kv, 128, K), dtype=torch.uint8,
                     device=DEV)
    status = ws[:4].view(torch.int32)
    out = torch.full((L, B, n_q, 128), 3.0, dtype=torch.float32, device=DEV)

    # a normal call: status 0, oracle parity
    assert _call(lib, case, out, ws, L, B, n_q, n_kv, K) == spc.SPC_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.abs(out.cpu().numpy() - want).max() <= ATTN_ATOL

    # a starved call: its waits give up after ~20 000 cycles (plus the
    # hardware's suspend hint of at most 10 ms per first wait)
    assert lib.spc_test_starve_attention(1, 20000) == spc.SPC_OK
    t0 = time.perf_counter()
    assert _call(lib, case, out, ws, L, B, n_q, n_kv, K) == spc.SPC_OK
    torch.cuda.synchronize()                       # the kernel ended by itself
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == SPC_ERR_TIMEOUT
    assert elapsed < 5.0, f"starved launch took {elapsed:.2f} s"

    # the context is usable: clear the status word, call again, parity holds
    status.zero_()
    out.fill_(3.0)
    assert _call(lib, case, out, ws, L, B, n_q, n_kv, K) == spc.SPC_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.abs(out.cpu().numpy() - want).max() <= ATTN_ATOL
