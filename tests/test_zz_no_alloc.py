"""The attention entry point that needs no caller workspace.

Some callers cannot allocate device memory -- code living under another
framework's memory manager (which has already reserved the device memory, so
an extra cudaMalloc fails or escapes its accounting) or a decode loop that
cannot afford cudaMalloc/cudaFree. spc_sparse_decode_attn_noalloc serves them
from a fixed scratch area inside the library. These checks call it through
the C ABI twice in a row, on different inputs, and compare each result with
the regular entry point's (same kernel, caller workspace), within the
attention tolerance the other tests use. A second call must not be disturbed
by what the first one left in the shared area. Both results are also held
to the CPU oracle's attention on the same rows.

This file is named to be collected last.
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


def _case(seed, L, B, n_q, n_kv, K, cap, use_slots):
    rng = np.random.default_rng(seed)
    d = 128
    keep, kp, vp, rows, use = [], [], [], [], []
    for _ in range(L * B):
        nrows = K if use_slots else cap
        kv = torch.from_numpy(rng.standard_normal((2, n_kv, nrows, d)).astype(np.float32)).to(DEV)
        kv = kv.to(torch.bfloat16).view(torch.int16).contiguous()
        keep.append(kv)
        kp.append(kv[0].data_ptr()); vp.append(kv[1].data_ptr()); rows.append(nrows); use.append(use_slots)
    views = spc.to_device_bytes(spc.kv_views(kp, vp, rows, use), DEV)
    q = torch.from_numpy(rng.standard_normal((L, B, n_q, d)).astype(np.float32)).to(DEV)
    q = q.to(torch.bfloat16).view(torch.int16).contiguous()
    sel = np.full((B, n_kv, K), -1, np.int32)
    slot = np.full((B, n_kv, K), -1, np.int32)
    for b in range(B):
        for g in range(n_kv):
            m = int(rng.integers(K // 2, K + 1))
            pos = np.sort(rng.choice(cap, size=m, replace=False))
            sel[b, g, :m] = pos
            slot[b, g, rng.choice(K, size=m, replace=False)] = pos
    return keep, views, q, torch.from_numpy(sel).to(DEV), torch.from_numpy(slot).to(DEV)


def _oracle(case, L, B, n_q, n_kv, use_slots):
    """The oracle's attention on the case's bits: the rows a view keeps are
    the slots holding a position (use_slots) or the selected positions."""
    keep, views, q, sel, slot = case
    qb = q.cpu().numpy().view(np.uint16)
    sel_h, slot_h = sel.cpu().numpy(), slot.cpu().numpy()
    want = np.zeros((L, B, n_q, 128), np.float64)
    for l in range(L):
        for b in range(B):
            kv = keep[l * B + b].cpu().numpy().view(np.uint16)
            rows = [np.nonzero(slot_h[b, g] >= 0)[0] if use_slots else sel_h[b, g][sel_h[b, g] >= 0]
                    for g in range(n_kv)]
            want[l, b] = O.sparse_attention(qb[l, b], kv[0], kv[1], rows, 1 / math.sqrt(128))
    return want


def _with_workspace(case, L, B, n_q, n_kv, K):
    keep, views, q, sel, slot = case
    out = torch.zeros(L, B, n_q, 128, dtype=torch.float32, device=DEV)
    ws = torch.zeros(spc.spc_sparse_decode_attn_workspace_size(L, B, n_q, n_kv, 128, K),
                     dtype=torch.uint8, device=DEV)
    spc.spc_sparse_decode_attn(q, views, sel, slot, L, B, n_q, n_kv, 128, K, 1 / math.sqrt(128), out, ws)
    return out


def _without_workspace(case, L, B, n_q, n_kv, K):
    keep, views, q, sel, slot = case
    out = torch.full((L, B, n_q, 128), 5.0, dtype=torch.float32, device=DEV)
    spc.spc_sparse_decode_attn_noalloc(q, views, sel, slot, L, B, n_q, n_kv, 128, K, 1 / math.sqrt(128), out)
    return out


@pytest.mark.parametrize("L,B,n_q,n_kv,K,cap,use_slots", [
    (1, 1, 32, 8, 2048, 4096, 1),     # one layer: several clusters per KV head merge through the scratch
    (4, 1, 32, 8, 2048, 4096, 1),     # the benchmark's launch shape
    (2, 2, 64, 8, 1000, 3000, 0),     # positions into a full cache
])
def test_noalloc_matches_the_workspace_entry_point_on_two_calls(L, B, n_q, n_kv, K, cap, use_slots):
    assert spc.spc_sparse_decode_attn_workspace_size(L, B, n_q, n_kv, 128, K) <= \
        spc.SPC_ATTN_NOALLOC_SCRATCH_BYTES
    first = _case(100 + L, L, B, n_q, n_kv, K, cap, use_slots)
    second = _case(200 + L, L, B, n_q, n_kv, K, cap, use_slots)
    got1 = _without_workspace(first, L, B, n_q, n_kv, K)
    got2 = _without_workspace(second, L, B, n_q, n_kv, K)
    torch.cuda.synchronize()
    for got, case in ((got1, first), (got2, second)):
        ref = _with_workspace(case, L, B, n_q, n_kv, K)
        torch.cuda.synchronize()
        err = (got - ref).abs()
        assert float(err.max()) <= ATTN_ATOL
        assert bool(torch.all(err <= 2e-5 + 1e-4 * ref.abs()))
        want = _oracle(case, L, B, n_q, n_kv, use_slots)
        e = np.abs(got.cpu().numpy() - want)
        assert e.max() <= ATTN_ATOL
        assert np.all(e <= 2e-5 + 1e-4 * np.abs(want)), f"max err vs oracle {e.max():.3g}"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 1023 layers x 64 requests x 64 KV heads need ~16 MB of merge counters,
    # more than the fixed area: refused before any launch
    L, B, n_q, n_kv, K = 1023, 64, 64, 64, 64
    assert spc.spc_sparse_decode_attn_workspace_size(L, B, n_q, n_kv, 128, K) > \
        spc.SPC_ATTN_NOALLOC_SCRATCH_BYTES
    fake = 0x10000
    with pytest.raises(spc.SpcError) as ei:
        spc.spc_sparse_decode_attn_noalloc(fake, fake, fake, fake, L, B, n_q, n_kv, 128, K, 0.1, fake,
                                           stream=0)
    assert ei.value.status == -5
