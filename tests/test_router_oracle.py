"""Pins of the router oracle (CPU): worked cases and independent forms.

The router: sigmoid scores plus a selection-only bias, stable top K (highest
first, ties to the lower expert index), weights from the raw scores divided by
their left-to-right sum plus 1e-20, times the scaling factor ("MoE Expert
Kernels", section 1; the Hy3 decode write-up, the router after its logits).
"""
import itertools
import math

import numpy as np

from oracle import router as R


def test_sigmoid_closed_forms():
    raw, choice = R.choice_scores(np.array([[0.0, 2.0, -2.0]]), np.zeros(3))
    assert raw[0, 0] == np.float32(0.5)
    assert abs(raw[0, 1] - 1 / (1 + math.exp(-2))) < 1e-7
    assert abs(raw[0, 1] + raw[0, 2] - 1.0) < 1e-6          # s(x) + s(-x) = 1
    assert np.array_equal(raw, choice)


def test_ties_go_to_the_lower_index():
    # All logits equal: every score ties, the first K experts win, in order.
    sel, p = R.router(np.zeros((2, 9)), np.zeros(9), K=4)
    assert sel.tolist() == [[0, 1, 2, 3]] * 2
    assert np.allclose(p, 0.25)
    # A tie between experts 5 and 2 at the top: 2 first.
    logits = np.array([[0.0, 0.0, 3.0, 0.0, 0.0, 3.0]])
    sel, _ = R.router(logits, np.zeros(6), K=3)
    assert sel.tolist() == [[2, 5, 0]]


def test_bias_steers_selection_not_weights():
    logits = np.array([[1.0, 0.9, -1.0, 0.0]])
    bias = np.array([0.0, 0.0, 2.0, 0.0])       # expert 2 is lifted above all
    sel, p = R.router(logits, bias, K=2)
    assert sel.tolist() == [[2, 0]]
    s2, s0 = 1 / (1 + math.exp(1.0)), 1 / (1 + math.exp(-1.0))
    # weights from the raw scores: s2 small, s0 large, despite the order
    assert abs(p[0, 0] - s2 / (s2 + s0)) < 1e-6
    assert abs(p[0, 1] - s0 / (s2 + s0)) < 1e-6


def test_normalisation_and_scaling():
    rng = np.random.default_rng(3)
    logits = rng.normal(size=(5, 16))
    sel, p = R.router(logits, rng.normal(0, 0.1, 16), K=6, scaling=2.5)
    assert np.allclose(p.sum(1), 2.5, atol=1e-12)
    assert (p > 0).all()


def test_k_equals_e_is_a_full_stable_sort():
    rng = np.random.default_rng(4)
    logits = rng.integers(-2, 3, size=(3, 7)).astype(np.float32)   # many ties
    sel, _ = R.router(logits, np.zeros(7), K=7)
    for t in range(3):
        keyed = sorted(range(7), key=lambda e: (-float(R.choice_scores(logits, np.zeros(7))[1][t, e]), e))
        assert sel[t].tolist() == keyed


def test_against_repeated_argmax_brute_force():
    # Independent form: K times take np.argmax (first maximum = lower index)
    # and knock the winner out.
    rng = np.random.default_rng(5)
    logits = rng.normal(size=(40, 12)).astype(np.float32)
    logits[::7, 3] = logits[::7, 8]          # planted exact ties
    bias = rng.normal(0, 0.2, 12).astype(np.float32)
    sel, p = R.router(logits, bias, K=5, scaling=1.7)
    raw, choice = R.choice_scores(logits, bias)
    for t in range(40):
        c = choice[t].astype(np.float64).copy()
        picks = []
        for _ in range(5):
            e = int(np.argmax(c))
            picks.append(e)
            c[e] = -np.inf
        assert sel[t].tolist() == picks
        s = raw[t, picks].astype(np.float64)
        assert np.allclose(p[t], s / (s.sum() + 1e-20) * 1.7, rtol=1e-14)


def test_every_subset_brute_force_tiny():
    # E = 5, K = 2: the chosen pair maximises the sum of choice scores among
    # all pairs, and is ordered highest first.
    rng = np.random.default_rng(6)
    for _ in range(20):
        logits = rng.normal(size=(1, 5))
        bias = rng.normal(0, 0.3, 5)
        sel, _ = R.router(logits, bias, K=2)
        _, choice = R.choice_scores(logits, bias)
        best = max(itertools.combinations(range(5), 2),
                   key=lambda c: (choice[0, c[0]] + choice[0, c[1]], -min(c)))
        assert set(sel[0].tolist()) == set(best)
        assert choice[0, sel[0, 0]] >= choice[0, sel[0, 1]]
