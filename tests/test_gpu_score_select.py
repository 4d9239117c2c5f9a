"""GPU parity of spc_score_select (projection, key scan, group score, Top-K)
against the CPU oracle, through the C ABI.

Bars (the stated ones): scores within 2e-3 relative; selections identical
except swaps whose oracle scores lie within 2e-3 of the oracle's K-th score;
appended key rows within 1 bf16 ulp (fp32 vs fp64 accumulation before the
one rounding).
"""
import numpy as np
import pytest
import torch

from oracle.checks import bf16_ulp_distance
from sparse_kv_cache_retrieval_gb300.configs import CONFIGS
from tests import swap_log
from tests.gpu_cases import ScoreRun, check_score_call, oracle_score, workload

pytestmark = pytest.mark.gpu


def _one_call(cfg, t=0, append=False):
    run = ScoreRun(cfg)
    K0 = run.inp.K_dlm.copy()
    gq, gs, gsel, glen, gK = run.call(t, int(append))
    oq, ok_new, oK, olens, os_all, osel = oracle_score(cfg, K0, run.inp.lens, run.inp.x[t],
                                                       run.inp.Wq, run.inp.Wk, append)
    swaps = check_score_call(cfg, gq, gs, gsel, glen, oq, olens, os_all, osel)
    assert run.status() == 0
    if append:
        for b in range(cfg.B):
            L0 = int(run.inp.lens[b])
            assert bf16_ulp_distance(gK[b, :, L0], ok_new[b]).max() <= 1
    return swaps


SMALL = [
    # (name, kwargs)
    ("gqa4_tiles_and_tail", dict(lens=(1000,), n_q=8, n_kv=2, H=512, budget=128)),
    ("mha_g1", dict(lens=(777,), n_q=4, n_kv=4, H=256, budget=96)),
    ("g2", dict(lens=(640,), n_q=8, n_kv=4, H=256, budget=80)),
    ("g8", dict(lens=(900,), n_q=16, n_kv=2, H=512, budget=100)),
    ("g16", dict(lens=(513,), n_q=16, n_kv=1, H=256, budget=72)),
    ("g32", dict(lens=(1100,), n_q=32, n_kv=1, H=256, budget=90)),
    ("g8_two_groups_ragged_tiles", dict(B=2, lens=(1025, 255), n_q=16, n_kv=2, H=256, budget=120)),
    ("mqa_g64", dict(lens=(1300,), n_q=64, n_kv=1, H=1024, budget=200)),
    ("ragged_batch", dict(B=3, lens=(1500, 129, 700), n_q=8, n_kv=2, H=256, budget=96)),
    ("batch17_over_16", dict(B=17, lens=tuple(200 + 37 * i for i in range(17)), n_q=8, n_kv=2, H=256,
                             budget=80)),
    ("batch5_hidden520_partial_stage", dict(B=5, lens=(300, 200, 450, 129, 260), n_q=8, n_kv=2, H=520,
                                            budget=96)),
    ("batch4_hidden8", dict(B=4, lens=(200, 150, 100, 250), n_q=8, n_kv=2, H=8, budget=96)),
    ("batch16_hidden8192_split16", dict(B=16, lens=tuple(150 + 11 * i for i in range(16)), n_q=8, n_kv=2,
                                        H=8192, budget=96)),
    ("len_le_budget_select_all", dict(lens=(50,), budget=96)),
    ("len_eq_budget", dict(lens=(96,), budget=96)),
    ("len_budget_plus_one", dict(lens=(97,), budget=96, cap=97)),
    ("len_tiny", dict(lens=(3,), budget=96)),
    ("len_zero", dict(lens=(0,), budget=96)),
    ("forced_only", dict(lens=(500,), budget=68)),
    ("no_forced", dict(lens=(500,), budget=50, n_sink=0, n_recent=0)),
    ("cap_multi_cta_cluster", dict(lens=(20000,), n_q=8, n_kv=2, H=256, budget=300, cap=20011)),
    # tensor-core scan (groups of 16+ heads), work split: more busy segments
    # (request, KV head) than SMs, so CTAs take consecutive runs of tiles across
    # segments, with empty requests among them
    ("g16_256_segments_runs_across_segments",
     dict(B=64, lens=tuple(0 if i % 9 == 0 else 40 + (53 * i) % 600 for i in range(64)), n_q=64, n_kv=4,
          H=256, budget=96)),
    # fewer requests than SMs: CTAs per request in proportion to its tiles,
    # interleaved over them; an empty and a one-position request
    ("mqa_g64_ragged_proportional_ctas", dict(B=5, lens=(3000, 0, 129, 1, 700), n_q=64, n_kv=1, H=1024,
                                              budget=96)),
    ("g32_two_kv_heads_ragged", dict(B=3, lens=(900, 128, 1), n_q=64, n_kv=2, H=512, budget=80)),
    # every request empty: no CTA has a tile
    ("g16_all_requests_empty", dict(B=2, lens=(0, 0), n_q=16, n_kv=1, H=256, budget=96)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[s[0] for s in SMALL])
def test_score_select_small(name, kw):
    cfg = workload(name=name, **kw)
    _one_call(cfg)


def test_all_equal_keys_over_a_long_context_ties_go_to_lower_positions():
    # every one of 20000 keys ties: the threshold bin holds far more keys than
    # one rank finishes alone, so the finer levels run over the whole cluster
    cfg = workload(name="ties_long", lens=(20000,), n_q=8, n_kv=2, H=256, budget=300, n_recent=64,
                   cap=20000)
    run = ScoreRun(cfg)
    run.K[:, :, :20000] = run.K[:, :, :1]
    gq, gs, gsel, glen, gK = run.call(0, 0)
    expect = list(range(4 + 232)) + list(range(20000 - 64, 20000))
    for g in range(2):
        assert gsel[0, g].tolist() == expect
    assert run.status() == 0


@pytest.mark.parametrize("B", [2, 6])
def test_score_select_append_grows_len_and_switches_from_select_all(B):
    # phase-A shape in miniature: len 120 -> 123 with budget 121 (B = 6 takes
    # the tensor-core projection, B = 2 the CUDA-core one)
    cfg = workload(name="append", lens=tuple(120 - 2 * (b % 2) for b in range(B)), B=B, n_q=8, n_kv=2,
                   H=256, budget=121, steps=3, append=True)
    run = ScoreRun(cfg)
    oK = run.inp.K_dlm.copy()
    olens = [int(v) for v in run.inp.lens]
    for t in range(1, 4):
        gq, gs, gsel, glen, gK = run.call(t, 1)
        oq, ok_new, oK, olens, os_all, osel = oracle_score(cfg, oK, olens, run.inp.x[t], run.inp.Wq,
                                                           run.inp.Wk, True)
        check_score_call(cfg, gq, gs, gsel, glen, oq, olens, os_all, osel)
        for b in range(cfg.B):
            assert bf16_ulp_distance(gK[b, :, olens[b] - 1], ok_new[b]).max() <= 1
    assert run.status() == 0


def test_tensor_core_scan_ragged_batch_with_append():
    # groups of 32 heads: the appended key row is part of the scanned context
    cfg = workload(name="tc_append", B=4, lens=(700, 0, 129, 1000), n_q=32, n_kv=1, H=256, budget=96,
                   append=True)
    _one_call(cfg, append=True)


def test_append_at_capacity_sets_overflow_and_keeps_len():
    cfg = workload(name="full", lens=(100,), n_q=8, n_kv=2, H=256, budget=96, cap=100, append=True)
    run = ScoreRun(cfg)
    run.call(0, 1)
    assert int(run.len.item()) == 100
    assert run.status() == -6


def test_all_equal_keys_ties_go_to_lower_positions():
    cfg = workload(name="ties", lens=(400,), n_q=8, n_kv=2, H=256, budget=80, n_recent=64)
    run = ScoreRun(cfg)
    run.K[:, :, :400] = run.K[:, :, :1]   # every row equal -> every score equal
    gq, gs, gsel, glen, gK = run.call(0, 0)
    expect = list(range(4 + 12)) + list(range(336, 400))  # sinks, the lowest others, recent 64
    for g in range(2):
        assert gsel[0, g].tolist() == expect
    assert np.allclose(gs[0, :, :400], 1.0 / 400, rtol=1e-5)


@pytest.mark.parametrize("key", ["cfg1", "cfg2", "cfg3", "cfg4a", "cfg4b", "cfg5", "cfg5mqa"])
def test_score_select_full_size_configs(key):
    """One call at every workload's full head shape and context, against the oracle."""
    cfg = CONFIGS[key]
    if key == "cfg5":
        cfg = cfg.__class__(**{**cfg.__dict__, "B": 2, "lens": cfg.lens[:2], "rho": cfg.rho[:2],
                               "hot": cfg.hot[:2], "gpu_layers": cfg.gpu_layers[:2]})
    swaps = _one_call(cfg, t=1 if cfg.append else 0, append=cfg.append)
    swap_log.record(f"score_select full size {key}", swaps, cfg.B * cfg.n_kv, 0)


def test_stages_one_by_one_equal_the_fused_call():
    cfg = workload(name="stages", B=2, lens=(900, 500), n_q=8, n_kv=2, H=256, budget=70, append=True,
                   steps=1)
    from sparse_kv_cache_retrieval_gb300 import binding as spc
    a, b = ScoreRun(cfg), ScoreRun(cfg)
    ga = a.call(1, 1)
    x = torch.from_numpy(np.ascontiguousarray(b.inp.x[1]).view(np.int16)).cuda()
    for st in (1, 2, 4):
        spc.spc_score_select_stages(x, b.Wq, b.Wk, b.K, b.len, 1, cfg.B, cfg.H, cfg.n_q, cfg.n_kv, 128,
                                    cfg.cap, cfg.budget, cfg.n_sink, cfg.n_recent, b.q, b.scores, b.sel,
                                    b.ws, stages=st)
    torch.cuda.synchronize()
    assert torch.equal(a.sel, b.sel) and torch.equal(a.len, b.len) and torch.equal(a.K, b.K)
    assert torch.equal(a.scores, b.scores)


def test_repeat_calls_are_deterministic():
    cfg = workload(name="det", lens=(3000,), n_q=8, n_kv=2, H=512, budget=200)
    run = ScoreRun(cfg)
    r1 = run.call(0, 0)
    r2 = run.call(0, 0)
    for u, v in zip(r1, r2):
        assert np.array_equal(u, v)
