"""Pins of the MLA oracle to facts outside itself.

The MLA head and attention reduce to ordinary attention when the up-projection
matrices only pick latent coordinates (each row of W_uk / W_uv a unit vector):
then a head's expanded keys and values are slices of the latent rows, and the
library's scaled_dot_product_attention on those slices (float64, CPU) must
agree. Closed forms cover the rope term and the logit scale, a single kept row
gives the up-projected row itself, and the mutation tests plant plausible
mistakes in copies of the oracle functions.
"""
import math

import numpy as np
import pytest
import torch

import oracle.mla_oracle as M
import oracle.spc_oracle as O

from test_oracle_pins import _bits, _is_valid_topk


def _picker(idx):
    """W [len(idx)][512] whose row j is the unit vector e_{idx[j]}: W c = c[idx]."""
    W = np.zeros((len(idx), M.D_C))
    W[np.arange(len(idx)), idx] = 1.0
    return _bits(W)


def _pickers(n_q, seed):
    """Per head a different set of 128 latent coordinates for W_uk and W_uv."""
    rng = np.random.default_rng(seed)
    uk = np.stack([_picker(rng.choice(M.D_C, M.D_NOPE, replace=False)) for _ in range(n_q)])
    uv = np.stack([_picker(rng.choice(M.D_C, M.D_V, replace=False)) for _ in range(n_q)])
    return uk, uv


def _picked(W_bits):
    """Latent coordinate picked by each row of a picker matrix."""
    return np.argmax(O.bf16_to_f64(W_bits), axis=1)


def check_mla_probs_vs_sdpa(prob_fn):
    """Picker W_uk: the weights equal SDPA(q_h, [C[:, picked] , C_rope], V = I)."""
    rng = np.random.default_rng(41)
    n_q, n = 4, 23
    C = O.round_to_bf16(rng.standard_normal((n, M.D_LAT)))
    uk, _ = _pickers(n_q, 43)
    q = rng.standard_normal((n_q, M.D_QK))
    P = prob_fn(q, C, uk, n)
    Cf = O.bf16_to_f64(C)
    for h in range(n_q):
        k = np.concatenate([Cf[:, _picked(uk[h])], Cf[:, M.D_C:]], axis=1)
        w = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[h]).view(1, 1, 1, M.D_QK), torch.from_numpy(k).view(1, 1, n, M.D_QK),
            torch.eye(n, dtype=torch.float64).view(1, 1, n, n))
        if not np.allclose(P[h], w.view(-1).numpy(), rtol=1e-12, atol=1e-15):
            return False
    return True


def check_mla_probs_rope_closed_form(prob_fn):
    """W_uk = 0, two rows: c_0 = 0, c_1 has rope value a in coordinate 0, the
    query's rope value b there: p_1 = 1 / (1 + exp(-a b / sqrt(192)))."""
    Wuk = np.zeros((1, M.D_NOPE, M.D_C), np.uint16)
    for a, b in [(1.0, 2.0), (4.0, -1.5), (0.5, 8.0)]:
        C = np.zeros((2, M.D_LAT))
        C[1, M.D_C] = a
        q = np.zeros((1, M.D_QK))
        q[0, M.D_NOPE] = b
        P = prob_fn(q, _bits(C), Wuk, 2)
        want = 1.0 / (1.0 + math.exp(-a * b / math.sqrt(M.D_QK)))
        if abs(P[0, 1] - want) > 1e-13:
            return False
    return True


def check_mla_attention_vs_sdpa(attn_fn):
    """Picker W_uk and W_uv, a subset of rows: each head equals SDPA over the
    sliced keys [C[r, picked_k], C[r, rope]] and values C[r, picked_v]."""
    rng = np.random.default_rng(47)
    n_q, n = 4, 31
    C = O.round_to_bf16(rng.standard_normal((n, M.D_LAT)))
    uk, uv = _pickers(n_q, 53)
    q = O.round_to_bf16(rng.standard_normal((n_q, M.D_QK)))
    rows = np.array([0, 3, 4, 11, 29, 30])
    scale = 1 / math.sqrt(M.D_QK)
    out = attn_fn(q, C, uk, uv, rows, scale)
    Cf = O.bf16_to_f64(C[rows])
    for h in range(n_q):
        k = np.concatenate([Cf[:, _picked(uk[h])], Cf[:, M.D_C:]], axis=1)
        v = Cf[:, _picked(uv[h])]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(O.bf16_to_f64(q[h])).view(1, 1, 1, M.D_QK),
            torch.from_numpy(k).view(1, 1, len(rows), M.D_QK), torch.from_numpy(v).view(1, 1, len(rows), M.D_V),
            scale=scale).view(-1).numpy()
        if not np.allclose(out[h], ref, rtol=1e-12, atol=1e-13):
            return False
    return True


def check_mla_attention_special(attn_fn):
    """One kept row: each head's output is that row up-projected by its W_uv
    (library matmul); no kept row: zeros."""
    rng = np.random.default_rng(59)
    n_q, n = 3, 9
    C = O.round_to_bf16(rng.standard_normal((n, M.D_LAT)))
    Wuk = O.round_to_bf16(rng.standard_normal((n_q, M.D_NOPE, M.D_C)) / 20)
    Wuv = O.round_to_bf16(rng.standard_normal((n_q, M.D_V, M.D_C)) / 20)
    q = O.round_to_bf16(rng.standard_normal((n_q, M.D_QK)))
    o = attn_fn(q, C, Wuk, Wuv, np.array([6]), 0.07)
    for h in range(n_q):
        want = np.matmul(O.bf16_to_f64(Wuv[h]), O.bf16_to_f64(C[6, :M.D_C]))
        if not np.allclose(o[h], want, rtol=1e-13, atol=1e-13):
            return False
    o = attn_fn(q, C, Wuk, Wuv, np.array([], np.int64), 0.07)
    return np.array_equal(o, np.zeros((n_q, M.D_V)))


def check_mla_projection_exact(project_fn):
    """Small-integer inputs: q and the new latent row equal integer arithmetic."""
    B, H, n_q = 2, 5, 2
    x = [[(3 * b + 2 * i) % 7 - 3 for i in range(H)] for b in range(B)]
    Wq = [[(5 * i + 3 * j) % 9 - 4 for j in range(n_q * M.D_QK)] for i in range(H)]
    Wd = [[(2 * i + 7 * j) % 5 - 2 for j in range(M.D_LAT)] for i in range(H)]
    q, c = project_fn(_bits(x), _bits(Wq), _bits(Wd), n_q)
    for b in range(B):
        for h in range(n_q):
            for j in range(M.D_QK):
                if q[b, h, j] != sum(x[b][i] * Wq[i][h * M.D_QK + j] for i in range(H)):
                    return False
        for j in range(M.D_LAT):
            ref = sum(x[b][i] * Wd[i][j] for i in range(H))
            if int(c[b, j]) != int(_bits([ref])[0]):
                return False
    return True


def test_mla_probabilities_vs_library_sdpa():
    assert check_mla_probs_vs_sdpa(M.mla_head_probabilities)


def test_mla_probabilities_rope_term_closed_form():
    assert check_mla_probs_rope_closed_form(M.mla_head_probabilities)


def test_mla_attention_vs_library_sdpa():
    assert check_mla_attention_vs_sdpa(M.mla_sparse_attention)


def test_mla_attention_special_cases():
    assert check_mla_attention_special(M.mla_sparse_attention)


def test_mla_projection_exact_integers():
    assert check_mla_projection_exact(M.mla_project)


def test_mla_absorbed_form_equals_expansion():
    """The identity the CUDA path relies on, checked on the oracle: scoring the
    query absorbed into the latent space, [W_uk^T q_nope ; q_rope] . c, and
    aggregating latents before W_uv give the literal expansion's result."""
    rng = np.random.default_rng(61)
    n_q, n = 3, 17
    C = O.round_to_bf16(rng.standard_normal((n, M.D_LAT)))
    Wuk = O.round_to_bf16(rng.standard_normal((n_q, M.D_NOPE, M.D_C)) / math.sqrt(M.D_C))
    Wuv = O.round_to_bf16(rng.standard_normal((n_q, M.D_V, M.D_C)) / math.sqrt(M.D_C))
    q = O.round_to_bf16(rng.standard_normal((n_q, M.D_QK)))
    rows = np.array([1, 2, 8, 16])
    scale = 1 / math.sqrt(M.D_QK)
    lit = M.mla_sparse_attention(q, C, Wuk, Wuv, rows, scale)
    Cf, qf = O.bf16_to_f64(C[rows]), O.bf16_to_f64(q)
    for h in range(n_q):
        qa = np.concatenate([O.bf16_to_f64(Wuk[h]).T @ qf[h, :M.D_NOPE], qf[h, M.D_NOPE:]])
        lg = Cf @ qa * scale
        w = np.exp(lg - lg.max())
        w /= w.sum()
        assert np.allclose(O.bf16_to_f64(Wuv[h]) @ (w @ Cf[:, :M.D_C]), lit[h], rtol=1e-11, atol=1e-12)


def test_mla_decode_state_chain_small():
    """A three-step growing chain: one valid selection per request, the slots
    hold exactly the selected latent rows, attention over the slots equals
    attention over the store rows by position."""
    rng = np.random.default_rng(67)
    B, n_q, cap, L, budget, H = 2, 4, 40, 3, 12, 16
    C_dlm = O.round_to_bf16(rng.standard_normal((B, cap, M.D_LAT)))
    stores = [O.round_to_bf16(rng.standard_normal((L, cap, M.D_LAT))) for _ in range(B)]
    st = M.MlaDecodeState(C_dlm, [30, 9], stores, [1, 0], budget, 2, 3)
    Wq = O.round_to_bf16(rng.standard_normal((H, n_q * M.D_QK)) / 4)
    Wuk = O.round_to_bf16(rng.standard_normal((n_q, M.D_NOPE, M.D_C)) / 20)
    Wd = O.round_to_bf16(rng.standard_normal((H, M.D_LAT)) / 4)
    Wuk_l = O.round_to_bf16(rng.standard_normal((L, n_q, M.D_NOPE, M.D_C)) / 20)
    Wuv_l = O.round_to_bf16(rng.standard_normal((L, n_q, M.D_V, M.D_C)) / 20)
    for t in range(3):
        x = O.round_to_bf16(rng.standard_normal((B, H)))
        _, _, _, ss, sel = st.score_select(x, Wq, Wuk, Wd, n_q, append=(t > 0))
        for b in range(B):
            assert _is_valid_topk(sel[b][0], ss[b][0], budget, 2, 3)
        st.diff_and_gather(sel)
        ql = O.round_to_bf16(rng.standard_normal((L, B, n_q, M.D_QK)))
        out = st.attention(ql, Wuk_l, Wuv_l, 1 / math.sqrt(M.D_QK))
        for b in range(B):
            h0 = st.host_layer0[b]
            held = st.slot_pos[b, 0]
            assert set(int(p) for p in held if p >= 0) == set(sel[b][0].tolist())
            for s_, p_ in enumerate(held):
                if p_ >= 0:
                    assert np.array_equal(st.slots[b][:, s_], stores[b][h0:, p_])
            for l in range(h0, L):
                live = np.nonzero(held >= 0)[0]
                via_slots = M.mla_sparse_attention(ql[l, b], st.slots[b][l - h0], Wuk_l[l], Wuv_l[l], live,
                                                   1 / math.sqrt(M.D_QK))
                assert np.allclose(via_slots, out[l, b], rtol=1e-12, atol=1e-13)
    assert st.lens == [32, 11]


def test_mla_planted_latent_rows_are_selected():
    """Latent rows shifted along the heads' summed absorbed query direction
    (8 standard deviations up) are the Top-K when they fit, for the one group
    of 16 heads; written out here from the query, not through the generator."""
    rng = np.random.default_rng(71)
    n_q, n, n_hot = 16, 1500, 30
    Wuk = O.round_to_bf16(rng.standard_normal((n_q, M.D_NOPE, M.D_C)) / math.sqrt(M.D_C))
    q = rng.standard_normal((n_q, M.D_QK))
    qa = np.concatenate([np.einsum("hjc,hj->hc", O.bf16_to_f64(Wuk), q[:, :M.D_NOPE]), q[:, M.D_NOPE:]], axis=1)
    u = qa.sum(0) / np.linalg.norm(qa.sum(0))
    C = rng.standard_normal((n, M.D_LAT))
    hot = np.sort(rng.choice(np.arange(4, n - 64), n_hot, replace=False))
    C[hot] += 8.0 * math.sqrt(n_q) * u
    P = M.mla_head_probabilities(q, O.round_to_bf16(C), Wuk, n)
    sel = O.select(O.group_scores(P, 1)[0], n_hot + 68, 4, 64)
    assert set(hot.tolist()) <= set(sel.tolist())


# ----------------------------------------------------------------- mutations
def _mut_probs_no_rope(q, C_bits, Wuk_bits, length):
    C = np.array(C_bits, copy=True)
    C[:, M.D_C:] = 0
    return M.mla_head_probabilities(q, C, Wuk_bits, length)


def _mut_probs_scale_128(q, C_bits, Wuk_bits, length):
    return M.mla_head_probabilities(q * math.sqrt(M.D_QK / M.D_NOPE), C_bits, Wuk_bits, length)


def _mut_probs_head0(q, C_bits, Wuk_bits, length):
    return M.mla_head_probabilities(q, C_bits, np.repeat(Wuk_bits[:1], Wuk_bits.shape[0], 0), length)


def _mut_attn_uk_for_uv(q_bits, C_bits, Wuk_bits, Wuv_bits, rows, scale):
    return M.mla_sparse_attention(q_bits, C_bits, Wuk_bits, Wuk_bits, rows, scale)


def _mut_attn_no_rope(q_bits, C_bits, Wuk_bits, Wuv_bits, rows, scale):
    C = np.array(C_bits, copy=True)
    C[:, M.D_C:] = 0
    return M.mla_sparse_attention(q_bits, C, Wuk_bits, Wuv_bits, rows, scale)


def _mut_attn_head0_uv(q_bits, C_bits, Wuk_bits, Wuv_bits, rows, scale):
    return M.mla_sparse_attention(q_bits, C_bits, Wuk_bits, np.repeat(Wuv_bits[:1], Wuv_bits.shape[0], 0),
                                  rows, scale)


def _mut_probs_rope_from_latent(q, C_bits, Wuk_bits, length):
    C = np.array(C_bits, copy=True)
    C[:, M.D_C:] = C[:, M.D_C - M.D_ROPE:M.D_C]      # rope key read from the latent's last 64 values
    return M.mla_head_probabilities(q, C, Wuk_bits, length)


def _mut_project_rope_first(x_bits, Wq_bits, Wdkv_bits, n_q):
    q, c = M.mla_project(x_bits, Wq_bits, Wdkv_bits, n_q)
    return np.concatenate([q[..., M.D_NOPE:], q[..., :M.D_NOPE]], axis=-1), c


MUTANTS = [
    ("rope key term dropped from the scores", [check_mla_probs_vs_sdpa, check_mla_probs_rope_closed_form],
     _mut_probs_no_rope),
    ("scores scaled by 1/sqrt(128)", [check_mla_probs_vs_sdpa, check_mla_probs_rope_closed_form],
     _mut_probs_scale_128),
    ("every head expands with head 0's W_uk", [check_mla_probs_vs_sdpa], _mut_probs_head0),
    ("values expanded with W_uk", [check_mla_attention_vs_sdpa, check_mla_attention_special], _mut_attn_uk_for_uv),
    ("rope key term dropped from attention", [check_mla_attention_vs_sdpa], _mut_attn_no_rope),
    ("every head's values use head 0's W_uv", [check_mla_attention_vs_sdpa, check_mla_attention_special],
     _mut_attn_head0_uv),
    ("query split rope-first", [check_mla_projection_exact], _mut_project_rope_first),
    ("rope key read from the latent's last values", [check_mla_probs_vs_sdpa, check_mla_probs_rope_closed_form],
     _mut_probs_rope_from_latent),
]


@pytest.mark.parametrize("name,checks,mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mla_pins_catch_planted_mistakes(name, checks, mutant):
    assert not all(chk(mutant) for chk in checks), f"no pin caught: {name}"
