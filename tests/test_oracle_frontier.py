"""Pins of oracle.frontier (CPU): hand-built rows and pools, closed forms, brute force."""
import itertools
import math

import numpy as np
import pytest

import synth
from oracle import frontier


def test_frontier_hand_built_with_ties():
    scores = [0.1, 0.5, 0.5, 0.9, 0.0, 0.5]
    assert frontier.frontier_topw(scores, 6, 3) == [3, 1, 2]
    assert frontier.frontier_topw(scores, 6, 10) == [3, 1, 2, 5, 0, 4]
    assert frontier.frontier_topw(scores, 3, 2) == [1, 2]  # only the first 3 count
    assert frontier.frontier_topw(scores, 0, 4) == []


def test_frontier_matches_brute_force_over_subsets():
    g = synth.rng(11)
    for _ in range(50):
        c = int(g.integers(1, 8))
        s = np.round(g.random(c), 1).astype(np.float32)  # coarse values: many ties
        w = int(g.integers(1, c + 1))
        got = frontier.frontier_topw(s, c, w)
        # brute force: the w-subset with the largest sum, then lowest positions, listed by (-s, pos)
        best = max(itertools.combinations(range(c), w),
                   key=lambda sub: (round(sum(float(s[i]) for i in sub), 6), [-i for i in sorted(sub)]))
        assert sorted(got) == sorted(best)
        assert got == sorted(got, key=lambda i: (-float(s[i]), i))


def test_children_hand_built_row():
    x = np.array([1.0, 3.0, 2.0, 3.0, -1.0])
    tok, p, s = frontier.attach_children(x, 0.5, 3)
    assert tok.tolist() == [1, 3, 2]  # the tie 3.0 / 3.0 goes to the lower token
    z = math.log(sum(math.exp(v) for v in x))
    np.testing.assert_allclose(p, np.exp(np.array([3.0, 3.0, 2.0]) - z).astype(np.float32), rtol=1e-7)
    assert np.array_equal(s, (np.float32(0.5) * p).astype(np.float32))


def test_children_logistic_closed_form_and_temperature():
    # two tokens: p(top) = 1 / (1 + exp(-(a - b) / T))
    for a, b, t in ((2.0, 0.0, 1.0), (2.0, 0.0, 2.0), (0.3, 0.1, 0.5)):
        tok, p, _ = frontier.attach_children(np.array([b, a]), 1.0, 1, temperature=t)
        assert tok.tolist() == [1]
        assert abs(float(p[0]) - 1.0 / (1.0 + math.exp(-(a - b) / t))) < 1e-7


def test_all_tokens_sum_to_one_and_scores_never_grow():
    g = synth.rng(12)
    x = g.standard_normal(200) * 2
    tok, p, s = frontier.attach_children(x, 0.8, 200)
    assert sorted(tok.tolist()) == list(range(200))
    assert abs(float(np.sum(p.astype(np.float64))) - 1.0) < 1e-5
    assert np.all(np.diff(p) <= 0) and np.all(s <= np.float32(0.8))


def test_expand_step_rows_are_independent():
    g = synth.rng(13)
    logits = g.standard_normal((4, 50))
    ps = np.array([1.0, 0.5, 0.25, 0.0], dtype=np.float32)
    tok, p, s = frontier.expand_step(logits, ps, 5)
    for r in range(4):
        t1, p1, s1 = frontier.attach_children(logits[r], ps[r], 5)
        assert np.array_equal(tok[r], t1) and np.array_equal(p[r], p1) and np.array_equal(s[r], s1)
    assert np.all(s[3] == 0)
