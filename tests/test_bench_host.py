"""Host-side pieces of bench.py (no GPU): the byte accounting per workload
family and the reference arm's oracle sample on the MLA workload."""
import json
import os
import subprocess
import sys

import bench
from sparse_kv_cache_retrieval_gb300.configs import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bytes_per_unit_follow_the_cache_layout():
    gqa, mla = CONFIGS["cfg2"], CONFIGS["mla"]
    assert bench.load_bytes(gqa) == 2 * 128 * 2            # K and V row of one KV head
    assert bench.load_bytes(mla) == 576 * 2                # one latent row
    assert bench.scan_row_bytes(gqa) == 256 and bench.scan_row_bytes(mla) == 1152
    # attention: kept rows, plus q/out; MLA also W_uk and W_uv of the layer
    assert bench.attn_bytes_per_layer(gqa, 10) == 10 * 512 + gqa.B * gqa.n_q * 128 * 6
    w = 2 * 16 * 128 * 512 * 2
    assert bench.attn_bytes_per_layer(mla, 10) == 10 * 1152 + w + mla.B * 16 * (192 * 2 + 128 * 4)
    assert bench.traffic_units(mla)["attention"] == ("mla_attention", 1152)
    assert bench.kernels_per_call(mla)["attention"] == 3
    assert bench.kernels_per_call(gqa, "batch")["select"] == 4


def test_roofline_kernel_is_the_largest_one_with_a_byte_model():
    k = {"gather": {"total_ms": 5.0}, "attention": {"total_ms": 3.0}, "select": {"total_ms": 1.0}}
    assert bench.roofline_kernel(k) == ("gather", "gather")
    # a latency-bound kernel leads the step: the largest modelled one is reported
    k = {"select": {"total_ms": 9.0}, "attention": {"total_ms": 3.0}, "key_scan": {"total_ms": 2.0}}
    assert bench.roofline_kernel(k) == ("select", "attention")
    assert bench.roofline_kernel({"select": {"total_ms": 1.0}}) == ("select", None)
    assert bench.roofline_kernel({}) == (None, None)


def test_traffic_is_none_for_an_unknown_source_hash():
    assert bench.ncu_traffic("no_such_kernel", 10) is None


def test_reference_arm_on_the_mla_workload_prints_one_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "mla",
           "--oracle-sample-steps", "1", "--oracle-sample-layers", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["attention"] == "mla"
