"""The oracle against the pages' printed values, closed forms and invariants.

Both oracle implementations (the float64 C loops and the numpy brute force)
must pass every pin; they are also cross-checked against each other.
"""
import numpy as np
import pytest

import oracle
from oracle import brute
import oracle_pins as pins


def c_impl(x, packed, scales, sel, p, ys):
    return oracle.expert_linear(x, packed, scales, sel, p, ys)


def brute_impl(x, packed, scales, sel, p, ys):
    sel = np.asarray(sel)
    E = np.asarray(packed).shape[0]
    valid = (sel >= 0) & (sel < E)
    p = np.where(valid, np.asarray(p, dtype=np.float64), 0.0)
    out = brute.expert_linear(x, packed, scales, np.where(valid, sel, 0), p, ys)
    return out, None, None


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_c_oracle(check):
    check(c_impl)


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_brute_oracle(check):
    check(brute_impl)


@pytest.mark.parametrize("seed", range(4))
def test_c_oracle_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    T, E, K, I, O = 5, 7, 3, 96, 11
    x = rng.standard_normal((T, I))
    packed = rng.integers(0, 256, (E, O, I // 32, 16), dtype=np.uint8)
    scales = rng.integers(110, 140, (E, O, I // 32), dtype=np.uint8)
    sel = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    p = rng.random((T, K))
    ys = rng.standard_normal((T, O))
    out, absm, bad = oracle.expert_linear(x, packed, scales, sel, p, ys)
    ref = brute.expert_linear(x, packed, scales, sel, p, ys)
    assert bad == 0
    assert np.all(np.abs(out - ref) <= 1e-12 * absm)


def test_row_subset_matches_full():
    rng = np.random.default_rng(3)
    T, E, K, I, O = 9, 4, 2, 64, 7
    x = rng.standard_normal((T, I))
    packed = rng.integers(0, 256, (E, O, I // 32, 16), dtype=np.uint8)
    scales = rng.integers(118, 136, (E, O, I // 32), dtype=np.uint8)
    sel = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    p = rng.random((T, K))
    ys = rng.standard_normal((T, O))
    full, fabs_, _ = oracle.expert_linear(x, packed, scales, sel, p, ys)
    rows = [8, 0, 3]
    sub, sabs, _ = oracle.expert_linear(x, packed, scales, sel, p, ys, rows=rows)
    assert np.array_equal(sub, full[rows]) and np.array_equal(sabs, fabs_[rows])


def test_decode_expert_matches_encoder():
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 16, size=(2, 3, 64))
    sb = rng.integers(100, 150, size=(2, 3, 2)).astype(np.uint8)
    packed = pins.encode(codes)
    want = pins.matrix_from_codes(codes, sb)
    for e in range(2):
        assert np.array_equal(oracle.decode_expert(packed, sb, e), want[e])
        assert np.array_equal(brute.dequantize(packed[e], sb[e]), want[e])
