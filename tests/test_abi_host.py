"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function include/spc.h declares, and
reject bad arguments before touching the device: each call below returns
its error code from host validation, so no kernel is launched.
"""
import ctypes
import os
import re

import pytest

import __graft_entry__
from sparse_kv_cache_retrieval_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return B.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "spc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spc_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_hot_path_calls():
    names = declared_functions()
    for n in ("spc_score_select", "spc_elastic_diff", "spc_gather_kv", "spc_sparse_decode_attn"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in spc.h but not exported"
        assert n in B.SIGNATURES, f"{n} has no binding signature"


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, 42):
        assert lib.spc_status_string(code)


def test_workspace_sizes(lib):
    ws = B.spc_score_select_workspace_size(1, 4096, 32, 8, 128, 32768, 2048)
    # at least the fp32 logits of every query head over the capacity
    assert ws >= 32 * 32768 * 4
    assert B.spc_score_select_workspace_size(1, 4096, 32, 8, 64, 32768, 2048) == 0
    assert B.spc_score_select_workspace_size(1, 4096, 30, 8, 128, 32768, 2048) == 0
    assert B.spc_sparse_decode_attn_workspace_size(1, 1, 32, 8, 128, 2048) > 0
    assert B.spc_sparse_decode_attn_workspace_size(1, 1, 32, 8, 96, 2048) == 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def _score(lib, **kw):
    a = dict(x=FAKE, Wq=FAKE, Wk=FAKE, K=FAKE, len=FAKE, append=0, B=1, H=4096, n_q=32, n_kv=8,
             d=128, cap=4096, budget=512, n_sink=4, n_recent=64, q_out=None, scores=None,
             sel=FAKE, ws=FAKE, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.spc_score_select(a["x"], a["Wq"], a["Wk"], a["K"], a["len"], a["append"], a["B"],
                                a["H"], a["n_q"], a["n_kv"], a["d"], a["cap"], a["budget"],
                                a["n_sink"], a["n_recent"], a["q_out"], a["scores"], a["sel"],
                                a["ws"], a["ws_bytes"], a["stream"])


def test_score_select_rejects_bad_arguments(lib):
    assert _score(lib, x=None) == -1
    assert _score(lib, append=2) == -1
    assert _score(lib, append=1, Wk=None) == -1
    assert _score(lib, K=FAKE + 8) == -1                 # misaligned key cache
    assert _score(lib, d=64) == -2
    assert _score(lib, n_q=30) == -2                     # n_q % n_kv != 0
    assert _score(lib, n_q=24, n_kv=8) == -2             # G = 3 unsupported
    assert _score(lib, budget=8192) == -2                # budget > max
    assert _score(lib, budget=5000, cap=4096) == -2
    assert _score(lib, cap=300000) == -2                 # cap > max
    assert _score(lib, n_sink=500, n_recent=64) == -2    # forced set > budget
    assert _score(lib, B=0) == -2
    assert _score(lib, H=4095) == -2
    assert _score(lib, H=32776) == -2                   # H > max
    assert _score(lib) == -5                             # workspace too small
    assert lib.spc_score_select_stages(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1, 4096, 32, 8, 128, 4096,
                                       512, 4, 64, None, None, FAKE, FAKE, 1 << 40, None, 0) == -1


def test_diff_gather_attention_reject_bad_arguments(lib):
    assert lib.spc_elastic_diff(None, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 512, 4096, None) == -1
    assert lib.spc_elastic_diff(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 5000, 4096, None) == -2
    assert lib.spc_elastic_diff(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 512, 1 << 20, None) == -2
    assert lib.spc_gather_kv(None, 0, 1, FAKE, FAKE, FAKE, 1, 8, 128, 4096, 512, None) == -1
    assert lib.spc_gather_kv(FAKE, 0, 1, FAKE, FAKE, FAKE, 1, 8, 64, 4096, 512, None) == -2
    assert lib.spc_gather_kv(FAKE, 2, 1, FAKE, FAKE, FAKE, 1, 8, 128, 4096, 512, None) == -2
    assert lib.spc_gather_kv(FAKE, 0, 1, FAKE, FAKE, FAKE, 64, 32, 128, 4096, 512, None) == -2
    assert lib.spc_sparse_decode_attn(None, FAKE, FAKE, FAKE, 1, 1, 32, 8, 128, 512, 0.1, FAKE,
                                      FAKE, 1 << 30, None) == -1
    assert lib.spc_sparse_decode_attn(FAKE, FAKE, FAKE, FAKE, 1, 1, 32, 8, 128, 512, -1.0, FAKE,
                                      FAKE, 1 << 30, None) == -1
    assert lib.spc_sparse_decode_attn(FAKE, FAKE, FAKE, FAKE, 1, 1, 32, 8, 128, 512, 0.1, FAKE,
                                      FAKE, 0, None) == -5
    assert lib.spc_sparse_decode_attn(FAKE, FAKE, FAKE, FAKE, 1, 1, 48, 8, 128, 512, 0.1, FAKE,
                                      FAKE, 1 << 30, None) == -2
    assert lib.spc_stream_read(FAKE, 17, FAKE, 1, None) == -2
    assert lib.spc_stream_read(FAKE + 4, 16, FAKE, 1, None) == -1


def test_binding_raises_spc_error(lib):
    with pytest.raises(B.SpcError) as ei:
        B.spc_elastic_diff(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 5000, 4096, stream=0)
    assert ei.value.status == -2


def test_view_struct_layouts():
    assert B.GATHER_VIEW_DTYPE.itemsize == 32
    assert B.KV_VIEW_DTYPE.itemsize == 32
    v = B.kv_views([1, 2], [3, 4], [5, 6], [1, 0])
    raw = v.view(ctypes.c_uint64 * 4 if False else "u8").reshape(2, 4)
    assert raw[0, 0] == 1 and raw[0, 1] == 3 and raw[0, 2] == 5 and (raw[0, 3] & 0xFFFFFFFF) == 1


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "sparse_kv_cache_retrieval_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")) and f != "smoke.py":
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_offload_thresholds_through_the_abi_match_the_oracle(lib):
    # host-only entry point: the memory model of adaptive offloading, checked
    # against the oracle's definition on random shapes and on the workloads
    import numpy as np
    import oracle.spc_oracle as O
    rng = np.random.default_rng(5)
    cases = [(32, 8, 128, 4, 2048, 12 << 30), (32, 8, 128, 16, 1024, 12 << 30),
             (80, 8, 128, 8, 4096, 60 << 30), (80, 1, 128, 8, 4096, 20 << 30)]
    for _ in range(200):
        L, n_kv, B_, K = int(rng.integers(1, 90)), int(rng.integers(1, 9)), int(rng.integers(1, 17)), \
            int(rng.integers(1, 4097))
        row = 2 * n_kv * 128 * 2
        cases.append((L, n_kv, 128, B_, K, int(B_ * row * L * K * rng.uniform(1.0, 40.0))))
    for L, n_kv, d, B_, K, kv in cases:
        got = B.spc_offload_thresholds(L, n_kv, d, B_, K, kv)
        want = O.offload_thresholds(L, n_kv, d, B_, K, kv)
        assert got[:L] == want[:L]
        assert got[L] == 2 ** 63 - 1


def test_offload_thresholds_reject_memory_below_the_workspaces(lib):
    with pytest.raises(B.SpcError) as e:
        B.spc_offload_thresholds(32, 8, 128, 2, 2048, 2 * 32 * 2048 * 4096 - 1)
    assert e.value.status == -5
    assert lib.spc_offload_thresholds(32, 8, 128, 2, 2048, 1 << 40, None) == -1
    assert lib.spc_offload_thresholds(0, 8, 128, 2, 2048, 1 << 40, None) in (-1, -2)


def test_fill_slots_validates_before_launch(lib):
    assert lib.spc_fill_slots(None, 0, 1, FAKE, 1, 8, 128, 100, 64, None) == -1
    assert lib.spc_fill_slots(FAKE, 0, 1, FAKE, 1, 8, 64, 100, 64, None) == -2
    assert lib.spc_fill_slots(FAKE, 2, 1, FAKE, 1, 8, 128, 100, 64, None) == -2
    assert lib.spc_fill_slots(FAKE, 0, 1, FAKE, 1, 8, 128, 100, 5000, None) == -2


def _mla_score(lib, **kw):
    a = dict(x=FAKE, Wq=FAKE, Wuk=FAKE, Wd=FAKE, C=FAKE, len=FAKE, append=0, B=1, H=2048, cap=4096,
             budget=512, n_sink=4, n_recent=64, scores=None, sel=FAKE, ws=FAKE, ws_bytes=0, stream=None,
             stages=7)
    a.update(kw)
    return lib.spc_mla_score_select(a["x"], a["Wq"], a["Wuk"], a["Wd"], a["C"], a["len"], a["append"], a["B"],
                                    a["H"], a["cap"], a["budget"], a["n_sink"], a["n_recent"], a["scores"],
                                    a["sel"], a["ws"], a["ws_bytes"], a["stream"], a["stages"])


def test_mla_calls_validate_before_launch(lib):
    assert _mla_score(lib, x=None) == -1
    assert _mla_score(lib, Wuk=None) == -1
    assert _mla_score(lib, append=1, Wd=None) == -1
    assert _mla_score(lib, C=FAKE + 8) == -1             # misaligned latent cache
    assert _mla_score(lib, stages=0) == -1
    assert _mla_score(lib, H=2047) == -2
    assert _mla_score(lib, budget=8192) == -2
    assert _mla_score(lib, budget=600, cap=512) == -2
    assert _mla_score(lib, n_sink=500) == -2
    assert _mla_score(lib) == -5                         # workspace too small
    ws = B.spc_mla_score_select_workspace_size(1, 2048, 32768, 2048)
    assert ws >= 16 * 32768 * 4                          # fp32 logits of 16 heads
    assert lib.spc_mla_gather(None, 0, 1, FAKE, FAKE, FAKE, 1, 4096, 512, None) == -1
    assert lib.spc_mla_gather(FAKE, 2, 1, FAKE, FAKE, FAKE, 1, 4096, 512, None) == -2
    assert lib.spc_mla_gather(FAKE, 0, 1, FAKE, FAKE, FAKE, 65, 4096, 512, None) == -2
    assert lib.spc_mla_gather(FAKE, 0, 1, FAKE, FAKE, FAKE, 1, 4096, 5000, None) == -2
    wa = B.spc_mla_decode_attn_workspace_size(16, 1, 2048)
    assert wa >= 16 * 16 * 576 * 4                       # the absorbed queries at least
    assert B.spc_mla_decode_attn_workspace_size(16, 1, 5000) == 0
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 1, 2048, 0.07, FAKE, FAKE, wa, None]
    assert lib.spc_mla_decode_attn(None, *args[1:]) == -1
    bad = list(args); bad[9] = 0.0
    assert lib.spc_mla_decode_attn(*bad) == -1
    bad = list(args); bad[12] = wa - 1
    assert lib.spc_mla_decode_attn(*bad) == -5
    bad = list(args); bad[8] = 0
    assert lib.spc_mla_decode_attn(*bad) == -2
    bad = list(args); bad[11] = FAKE + 64
    assert lib.spc_mla_decode_attn(*bad) == -1           # workspace not 256-byte aligned


def test_batch_select_validates_before_launch(lib):
    args = [FAKE, FAKE, 2, 8, 4096, 512, 4, 64, FAKE, FAKE, 1 << 30, None]
    assert lib.spc_batch_select(None, *args[1:]) == -1
    bad = list(args); bad[3] = 0
    assert lib.spc_batch_select(*bad) == -2               # no KV head
    bad = list(args); bad[5] = 5000
    assert lib.spc_batch_select(*bad) == -2               # budget > cap
    bad = list(args); bad[6] = 500
    assert lib.spc_batch_select(*bad) == -2               # forced set > budget
    bad = list(args); bad[10] = 16
    assert lib.spc_batch_select(*bad) == -5               # workspace too small
    bad = list(args); bad[9] = FAKE + 64
    assert lib.spc_batch_select(*bad) == -1               # workspace misaligned
    assert B.spc_batch_select_workspace_size(2, 4096, 512) >= 2 * 4096 * 4


def test_header_is_plain_c99_and_links_against_the_library(lib, tmp_path):
    """include/spc.h is a C ABI: a C99 program that includes it compiles with
    warnings as errors and links against libspc.so."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_spc.c"
    src.write_text('#include "spc.h"\n#include <stdio.h>\n'
                   'int main(void) { printf("%s\\n", spc_status_string(SPC_ERR_SHAPE)); '
                   'return spc_version() > 0 ? 0 : 1; }\n')
    exe = tmp_path / "use_spc"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), B.LIB_PATH, "-Wl,-rpath," + os.path.dirname(B.LIB_PATH)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0 and "sizes" in run.stdout
