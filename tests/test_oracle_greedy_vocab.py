"""Pins for oracle.greedy (golden hand-built trees) and oracle.vocab (closed forms)."""
import json
import math
import os

import numpy as np
import pytest

import synth
from oracle import greedy, vocab

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "greedy_cases.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_greedy_golden(case):
    acc, bonus = greedy.greedy_walk(case["parent"], case["tokens"], case["argmax"])
    assert acc == case["accepted"]
    assert bonus == case["bonus"]


def test_all_equal_row_closed_form():
    v = 1000
    x = np.full(v, 0.375, dtype=np.float32)
    m, lse, am = vocab.row_stats(x, 1.0)
    assert am == 0
    assert abs(lse - (0.375 + math.log(v))) < 1e-12
    # temperature divides the logits
    m2, lse2, _ = vocab.row_stats(x, 0.5)
    assert abs(lse2 - (0.75 + math.log(v))) < 1e-12


def test_two_value_row_is_logistic():
    x = np.array([0.0, 1.25, -3.0], dtype=np.float32)
    _, lse, am = vocab.row_stats(x)
    assert am == 1
    p1 = math.exp(1.25 - lse)
    # softmax over three logits written via pairwise logistic terms
    assert abs(p1 - 1.0 / (1.0 + math.exp(-1.25) + math.exp(-4.25))) < 1e-14


def test_ties_take_lowest_index_and_shift_invariance():
    x = np.array([1.0, 3.0, -2.0, 3.0, 3.0], dtype=np.float32)
    _, lse, am = vocab.row_stats(x)
    assert am == 1
    _, lse_s, am_s = vocab.row_stats(x + np.float32(5.0))
    assert am_s == 1 and abs(lse_s - (lse + 5.0)) < 1e-12


def test_drafted_probabilities_sum_to_one_over_all_tokens():
    g = synth.rng(11)
    n, v = 4, 37
    x = synth.normal(g, (n, v), std=math.sqrt(2))
    _, lse, _ = vocab.vocab_stats(x)
    # make node 1..v children of node 0 covering every token; their p sum to 1
    parent = np.array([-1] + [0] * v, dtype=np.int32)
    toks = np.array([0] + list(range(v)), dtype=np.int32)
    xx = np.concatenate([x[:1], np.zeros((v, v), dtype=np.float32)])
    _, lse2, _ = vocab.vocab_stats(xx)
    p = vocab.drafted_token_prob(xx, lse2, parent, toks)
    assert np.isnan(p[0])
    assert abs(np.sum(p[1:]) - 1.0) < 1e-12


def test_planted_argmax_is_found():
    g = synth.rng(12)
    n, v = 6, 501
    par = synth.random_parents(g, n, 3)
    tok = synth.distinct_child_tokens(g, par, v)
    x = synth.normal(g, (n, v), std=math.sqrt(2), bf16=True)
    xp = synth.plant_first_child_argmax(g, x, par, tok, 1.0, bf16=True)
    fc = synth.first_children(par)
    _, _, am = vocab.vocab_stats(xp)
    for u in range(n):
        if fc[u] >= 0:
            assert am[u] == tok[fc[u]]


def test_padded_rows_are_not_drafts():
    # padding rows (parent -1 after the last node) are no drafts: NaN drafted-token
    # probability, never walked; the walk equals that of the unpadded tree
    par = [-1, 0, 0, 1]
    tok = [5, 3, 4, 7]
    pad = par + [-1, -1]
    logits = np.zeros((6, 10))
    logits[0, 3] = 4.0
    logits[1, 7] = 4.0
    _, lse, am = vocab.vocab_stats(logits)
    p = vocab.drafted_token_prob(logits, lse, pad, tok + [0, 0])
    assert np.isnan(p[4:]).all() and np.isnan(p[0])
    assert np.allclose(p[1:4], vocab.drafted_token_prob(logits[:4], lse[:4], par, tok)[1:4])
    assert greedy.greedy_walk(pad, tok + [3, 3], am) == greedy.greedy_walk(par, tok, am[:4]) == ([1, 3], int(am[3]))
