"""Pins of the batch-level selection (the alternative to head-level retrieval
the pages compare against: every head's weights merged into one Top-K per
request, shared by all KV heads).

With one group it is the head-level selection itself (brute force over every
subset, as for `select`); with several groups, a hand-worked case where the
element-wise max and a mean disagree, and the symmetry and domination facts
that hold for a max.
"""
import numpy as np
import pytest

import oracle.spc_oracle as O

from test_oracle_pins import check_select_bruteforce


def check_batch_reduces_to_select(fn):
    return check_select_bruteforce(lambda s, budget, ns, nr: fn(np.asarray(s)[None, :], budget, ns, nr))


def check_batch_hand_example(fn):
    """Hand-worked cases, no forced set.
    (1) Two groups over 6 positions, budget 2: the element-wise max is
        [0, .6, 0, 0, .4, .5], so positions {1, 5} are kept.
    (2) Position 0 strong in one group (0.6), position 1 moderately strong in
        both (0.4, 0.4), budget 1: the max keeps position 0, where a mean
        (0.3 vs 0.4) or a sum (0.6 vs 0.8) would keep position 1."""
    s = np.array([[0.0, 0.6, 0.0, 0.0, 0.0, 0.0],
                  [0.0, 0.4, 0.0, 0.0, 0.4, 0.5]])
    if list(fn(s, 2, 0, 0)) != [1, 5]:
        return False
    s2 = np.array([[0.6, 0.4],
                   [0.0, 0.4]])
    return list(fn(s2, 1, 0, 0)) == [0]


def check_batch_symmetry_and_domination(fn):
    rng = np.random.default_rng(29)
    for _ in range(50):
        n_kv, n = int(rng.integers(2, 5)), int(rng.integers(20, 60))
        s = rng.random((n_kv, n)) ** 4
        budget = int(rng.integers(8, 20))
        got = list(fn(s, budget, 2, 3))
        if list(fn(s[::-1], budget, 2, 3)) != got:          # order of the groups is irrelevant
            return False
        if list(fn(np.vstack([s, s[:1] * 0.5]), budget, 2, 3)) != got:   # a dominated group changes nothing
            return False
        if list(fn(np.repeat(s[:1], n_kv, 0), budget, 2, 3)) != list(O.select(s[0], budget, 2, 3)):
            return False
    return True


def test_batch_level_with_one_group_is_the_head_level_selection():
    assert check_batch_reduces_to_select(O.batch_level_select)


def test_batch_level_hand_example():
    assert check_batch_hand_example(O.batch_level_select)


def test_batch_level_symmetry_and_domination():
    assert check_batch_symmetry_and_domination(O.batch_level_select)


def _mut_mean(s, budget, ns, nr):
    return O.select(np.asarray(s).mean(axis=0), budget, ns, nr)


def _mut_sum(s, budget, ns, nr):
    return O.select(np.asarray(s).sum(axis=0), budget, ns, nr)


def _mut_first_group(s, budget, ns, nr):
    return O.select(np.asarray(s)[0], budget, ns, nr)


MUTANTS = [
    ("mean over groups", [check_batch_hand_example], _mut_mean),
    ("sum over groups", [check_batch_hand_example, check_batch_symmetry_and_domination], _mut_sum),
    ("first group only", [check_batch_symmetry_and_domination], _mut_first_group),
]


@pytest.mark.parametrize("name,checks,mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_batch_level_pins_catch_planted_mistakes(name, checks, mutant):
    assert not all(chk(mutant) for chk in checks), f"no pin caught: {name}"
