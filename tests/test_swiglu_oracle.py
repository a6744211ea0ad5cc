"""Pins for the SwiGLU expert oracle (oracle/swiglu.py), on the CPU.

What pins it, other than itself:
  * closed forms built from the pages' fixed points: a group of 0x22 bytes
    decodes to 32 ones and scale byte s multiplies by 2^(s-127), so gate, up
    and down rows of known constant value give silu(g) u and the down sum in
    closed form (silu(1) = 1 / (1 + e^-1), silu(-1) = -1 / (1 + e));
  * a library routine: silu(v) against v * scipy.special.expit(v);
  * mathematics: |silu'| <= 1.1 everywhere, the bound the tolerance uses;
  * brute force on tiny inputs: dense matrices from the numpy decoder
    (oracle.brute, independent of the C oracle) and plain loops;
  * invariants: rows= selects rows of the full result, invalid ids add
    nothing and are counted, p = 0 returns the shared output;
  * the tolerance formula is an upper bound: perturbing g and u by up to
    tau1 Ag, tau1 Au (worst signs and random ones) and h by rho never moves
    the result further than ``tolerance`` allows.
The tests at the end plant plausible mistakes in a copy of the oracle and check that
one of these pins fails.
"""
import importlib.util
import os
import sys

import numpy as np
import pytest
import torch

import oracle.brute as brute
import oracle.swiglu as sw

sys.path.insert(0, os.path.dirname(__file__))
from oracle_pins import encode  # noqa: E402

SRC = sw.__file__


# ---------------------------------------------------------------- helpers --
def const_rows(E, R, I, byte, scale):
    """(E, R, I/32, 16) bytes all equal to `byte`, scales all `scale`."""
    packed = np.full((E, R, I // 32, 16), byte, dtype=np.uint8)
    scales = np.full((E, R, I // 32), scale, dtype=np.uint8)
    return packed, scales


def random_case(seed, T=3, E=3, K=2, I=64, F=32, O=5):
    rng = np.random.default_rng(seed)
    gcodes = rng.integers(0, 16, size=(E, 2 * F, I))
    dcodes = rng.integers(0, 16, size=(E, O, F))
    gu = encode(gcodes)
    gus = rng.integers(121, 127, size=(E, 2 * F, I // 32)).astype(np.uint8)
    dn = encode(dcodes)
    dns = rng.integers(122, 129, size=(E, O, F // 32)).astype(np.uint8)
    x = rng.standard_normal((T, I))
    sel = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    p = rng.random((T, K))
    ys = rng.standard_normal((T, O))
    return x, gu, gus, dn, dns, sel, p, ys


def dense_expert(x, gu, gus, dn, dns, sel, p, ys):
    """Brute force: decode every selected matrix densely, loop over tokens
    and slots."""
    T, K = sel.shape
    F = gu.shape[1] // 2
    out = np.array(ys, dtype=np.float64, copy=True)
    for t in range(T):
        for k in range(K):
            e = int(sel[t, k])
            Wgu = brute.dequantize(gu[e], gus[e])
            Wd = brute.dequantize(dn[e], dns[e])
            gate = Wgu[:F] @ x[t]
            up = Wgu[F:] @ x[t]
            h = np.array([gate[f] * float(1.0 / (1.0 + np.exp(-gate[f]))) * up[f]
                          for f in range(F)])
            out[t] += p[t, k] * (Wd @ h)
    return out


def _close(a, b, rel=1e-12):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    assert np.all(np.abs(a - b) <= rel * scale), (a, b)


# ------------------------------------------------------------------- pins --
def check_closed_form_gate_up(mod):
    # I = 32: a row of 0x22 bytes is 32 ones; scale 122 -> g = 1, scale 123 -> u = 2.
    E, T, I, F, O = 2, 2, 32, 32, 3
    gp, gs = const_rows(E, 2 * F, I, 0x22, 127)
    gs[:, :F] = 122
    gs[:, F:] = 123
    gp[1, :F] = 0xAA            # expert 1: gate rows of -1 -> g = -1
    dp, ds = const_rows(E, O, F, 0x22, 127)        # down rows of ones: sum over f
    x = np.ones((T, I))
    sel = np.array([[0], [1]])
    p = np.array([[0.5], [2.0]])
    ys = np.array([[1.0, -2.0, 0.25], [0.0, 3.0, -1.0]])
    r = mod.swiglu_expert(x, gp, gs, dp, ds, sel, p, ys)
    s1 = 1.0 / (1.0 + np.exp(-1.0))                # silu(1)
    sm1 = -1.0 / (1.0 + np.e)                      # silu(-1)
    _close(r["out"][0], ys[0] + 0.5 * F * s1 * 2.0)
    _close(r["out"][1], ys[1] + 2.0 * F * sm1 * 2.0)
    _close(r["g"][:, 0], [1.0, -1.0])
    _close(r["u"][:, 0], [2.0, 2.0])
    assert r["bad"] == 0


def check_silu_library(mod):
    special = pytest.importorskip("scipy.special")
    v = np.concatenate([np.linspace(-40, 40, 4001), [-700.0, -100.0, 0.0, 100.0, 700.0]])
    _close(mod.silu(v), v * special.expit(v), rel=1e-14)


def check_brute_force(mod):
    for seed in range(3):
        x, gu, gus, dn, dns, sel, p, ys = random_case(seed)
        r = mod.swiglu_expert(x, gu, gus, dn, dns, sel, p, ys)
        _close(r["out"], dense_expert(x, gu, gus, dn, dns, sel, p, ys), rel=1e-11)


def check_abs_terms(mod):
    x, gu, gus, dn, dns, sel, p, ys = random_case(7)
    r = mod.swiglu_expert(x, gu, gus, dn, dns, sel, p, ys)
    T, K = sel.shape
    F = gu.shape[1] // 2
    want = np.abs(ys).copy()
    for t in range(T):
        for k in range(K):
            e = sel[t, k]
            Wgu = brute.dequantize(gu[e], gus[e])
            g, u = Wgu[:F] @ x[t], Wgu[F:] @ x[t]
            h = g / (1 + np.exp(-g)) * u
            want[t] += abs(p[t, k]) * (np.abs(brute.dequantize(dn[e], dns[e])) @ np.abs(h))
    _close(r["abs_terms"], want, rel=1e-11)


def check_rows_and_invariants(mod):
    x, gu, gus, dn, dns, sel, p, ys = random_case(3, T=5)
    full = mod.swiglu_expert(x, gu, gus, dn, dns, sel, p, ys)
    rows = np.array([4, 0, 2])
    part = mod.swiglu_expert(x, gu, gus, dn, dns, sel, p, ys, rows=rows)
    _close(part["out"], full["out"][rows], rel=0)
    zero = mod.swiglu_expert(x, gu, gus, dn, dns, sel, np.zeros_like(p), ys)
    _close(zero["out"], ys, rel=0)
    # Invalid ids add nothing and are counted.
    bad_sel = sel.copy()
    bad_sel[1, 0] = -1
    bad_sel[3, 1] = gu.shape[0]
    r = mod.swiglu_expert(x, gu, gus, dn, dns, bad_sel, p, ys)
    assert r["bad"] == 2
    keep = p.copy()
    keep[1, 0] = 0.0
    keep[3, 1] = 0.0
    ref = mod.swiglu_expert(x, gu, gus, dn, dns, sel, keep, ys)
    _close(r["out"], ref["out"], rel=1e-14)


def check_tolerance_is_a_bound(mod):
    rng = np.random.default_rng(11)
    x, gu, gus, dn, dns, sel, p, ys = random_case(5, T=4, K=2, F=64)
    r = mod.swiglu_expert(x, gu, gus, dn, dns, sel, p, ys)
    T, K = sel.shape
    tau1, rho = 3e-2, 2.0 ** -9
    bound = mod.tolerance(r, 0.0, tau1, rho)
    g, u, ag, au = r["g"], r["u"], r["ag"], r["au"]
    trials = [(np.sign(g) * np.sign(u), np.ones_like(u)), (np.ones_like(g), np.ones_like(u)),
              (-np.ones_like(g), np.sign(u))]
    trials += [(rng.choice([-1.0, 1.0], g.shape), rng.choice([-1.0, 1.0], u.shape))
               for _ in range(20)]
    worst = 0.0
    for sg, su in trials:
        g2 = g + sg * tau1 * ag
        u2 = u + su * tau1 * au
        h2 = g2 / (1.0 + np.exp(-g2)) * u2
        h2 *= 1.0 + rho * rng.choice([-1.0, 1.0], h2.shape)
        out2 = np.array(ys, dtype=np.float64, copy=True)
        for t in range(T):
            for k in range(K):
                e = sel[t, k]
                out2[t] += p[t, k] * (brute.dequantize(dn[e], dns[e]) @ h2[t * K + k])
        err = np.abs(out2 - r["out"])
        assert np.all(err <= bound * (1 + 1e-12)), float(np.max(err / bound))
        worst = max(worst, float(np.max(err / bound)))
    assert worst > 0.05               # the bound is not vacuous on these inputs


def check_tolerance_terms_are_tight(mod):
    # Constant rows: g = 2.4 (near the largest slope of silu), u = 1.2, every
    # term positive (Ag = g, Au = u), down rows of ones. Perturbing with all
    # signs aligned moves the result by nearly the full bound, so each term
    # of the bound is needed: the slope and product terms (rho = 0, large
    # tau1) and the rounding term (tau1 = 0).
    I = F = 32
    gp, gs = const_rows(1, 2 * F, I, 0x22, 127)
    dp, ds = const_rows(1, 1, F, 0x22, 127)
    x = np.full((1, I), 2.4 / 32)
    gp2, gs2 = gp.copy(), gs.copy()
    r0 = mod.swiglu_expert(x, gp2, gs2, dp, ds, np.array([[0]]), np.ones((1, 1)),
                           np.zeros((1, 1)))
    assert abs(r0["g"][0, 0] - 2.4) < 1e-12
    # Up rows at half the gate rows' value: a scale byte one lower.
    gs2[:, F:] = 126
    r = mod.swiglu_expert(x, gp2, gs2, dp, ds, np.array([[0]]), np.ones((1, 1)),
                          np.zeros((1, 1)))
    g, u, ag, au = r["g"], r["u"], r["ag"], r["au"]
    assert abs(u[0, 0] - 1.2) < 1e-12 and np.allclose(ag, g) and np.allclose(au, u)
    for tau1, rho in ((0.3, 0.0), (0.0, 2.0 ** -9)):
        g2, u2 = g + tau1 * ag, u + tau1 * au
        h2 = g2 / (1.0 + np.exp(-g2)) * u2 * (1.0 + rho)
        err = float(np.sum(h2) - np.sum(r["h"]))
        bound = float(mod.tolerance(r, 0.0, tau1, rho)[0, 0])
        assert err <= bound * (1 + 1e-12), (tau1, rho, err, bound)
        assert err >= 0.9 * bound, (tau1, rho, err, bound)


def check_round_to_bf16_matches_torch(mod):
    # For float32 inputs one rounding to bf16 is what torch's conversion
    # (round to nearest, ties to even) does: normals over float32's whole
    # exponent range, subnormals, values that overflow, signs, ties.
    rng = np.random.default_rng(3)
    exps = rng.integers(-149, 128, size=20000)
    v = np.ldexp(rng.uniform(1.0, 2.0, size=exps.size), exps) * rng.choice([-1, 1], exps.size)
    v = np.concatenate([v, np.ldexp(np.arange(1, 1025, dtype=np.float64), -24)]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    got = mod.round_to_bf16(v.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def check_round_to_bf16_is_one_rounding(mod):
    # From the exact value, not through float32: 1 + 2^-8 + 2^-40 rounds up
    # (float32 first would make it the tie 1 + 2^-8, then 1.0).
    cases = [(1 + 2.0 ** -8 + 2.0 ** -40, 1 + 2.0 ** -7), (1 + 2.0 ** -8, 1.0),
             (1 + 3 * 2.0 ** -8, 1 + 2.0 ** -6), (-(1 + 2.0 ** -8 + 2.0 ** -40), -(1 + 2.0 ** -7)),
             ((2 - 2.0 ** -8) * 2.0 ** 127, np.inf),
             ((2 - 2.0 ** -8 - 2.0 ** -30) * 2.0 ** 127, (2 - 2.0 ** -7) * 2.0 ** 127),
             (2.0 ** -134, 0.0), (3 * 2.0 ** -134, 2.0 ** -132), (2.0 ** -133, 2.0 ** -133),
             (0.0, 0.0), (-np.inf, -np.inf)]
    for v, want in cases:
        got = float(mod.round_to_bf16(np.array([v]))[0])
        assert got == want, (v, got, want)


def check_h_round_feeds_the_down_projection(mod):
    # With h rounded, the result moves by exactly p Wd (round(h) - h), the
    # brute-force expert applied to the difference (its down stage only).
    x, gu, gus, dn, dns, sel, p, ys = random_case(11)
    a = mod.swiglu_expert(x, gu, gus, dn, dns, sel, p, ys)
    b = mod.swiglu_expert(x, gu, gus, dn, dns, sel, p, ys, h_round="bf16")
    np.testing.assert_array_equal(b["h"], a["h"])
    np.testing.assert_array_equal(b["h_used"], mod.round_to_bf16(a["h"]))
    assert np.any(b["h_used"] != a["h"])
    T, K = sel.shape
    moved = np.zeros_like(a["out"])
    for t in range(T):
        for k in range(K):
            Wd = brute.dequantize(dn[int(sel[t, k])], dns[int(sel[t, k])])
            j = t * K + k
            moved[t] += p[t, k] * (Wd @ (b["h_used"][j] - a["h"][j]))
    _close(b["out"] - a["out"], moved, rel=1e-9)


PINS = [check_closed_form_gate_up, check_tolerance_terms_are_tight, check_silu_library, check_brute_force, check_abs_terms,
        check_rows_and_invariants, check_tolerance_is_a_bound, check_round_to_bf16_matches_torch,
        check_round_to_bf16_is_one_rounding, check_h_round_feeds_the_down_projection]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(sw)


def test_silu_slope_is_below_the_bound():
    # silu'(v) = s (1 + v (1 - s)), s = sigmoid(v); its extremes are about
    # 1.0998 and -0.0998, near v = +-2.3994.
    v = np.linspace(-60, 60, 1_200_001)
    s = 1.0 / (1.0 + np.exp(-v))
    d = s * (1.0 + v * (1.0 - s))
    assert np.max(np.abs(d)) <= sw.SILU_SLOPE_MAX
    assert 1.099 < np.max(d) < 1.1 and -0.1 < np.min(d) < -0.099
    assert abs(v[np.argmax(d)] - 2.3994) < 1e-3


# -------------------------------------------------------------- mutations --
MUTATIONS = {
    "gate_up_swapped": ("g, u = gu[:, :F], gu[:, F:]", "u, g = gu[:, :F], gu[:, F:]"),
    "sigmoid_not_silu": ("return v / (1.0 + np.exp(-v))", "return 1.0 / (1.0 + np.exp(-v))"),
    "silu_sign": ("return v / (1.0 + np.exp(-v))", "return v / (1.0 + np.exp(v))"),
    "up_dropped": ("h = silu(g) * u", "h = silu(g)"),
    "h_round_ignored": ('h_used = round_to_bf16(h) if h_round == "bf16" else h', "h_used = h"),
    "bf16_truncates": ("np.rint(np.ldexp(x, -quantum_exp))", "np.trunc(np.ldexp(x, -quantum_exp))"),
    "gate_dropped": ("h = silu(g) * u", "h = silu(u) * u"),
    "weight_ignored": ("out += pk * d[j]", "out += d[j]"),
    "shared_dropped": ("out = ys.copy()", "out = np.zeros_like(ys)"),
    "slot_stride": ("j = np.arange(n) * K + k", "j = np.arange(n) + k * n"),
    "last_slot_dropped": ("for k in range(K):", "for k in range(K - 1):"),
    "gate_rows_half": ("F = gate_up_packed.shape[1] // 2", "F = gate_up_packed.shape[1] // 4"),
    "abs_terms_no_shared": ('"abs_terms": np.abs(ys) + s_h', '"abs_terms": s_h'),
    "slope_term_dropped": ("SILU_SLOPE_MAX * ag * np.abs(u) + np.abs(g) * au",
                           "np.abs(g) * au"),
    "second_order_dropped": ("+ SILU_SLOPE_MAX * tau1 * tau1 * terms[\"s_second\"])", ")"),
    "rho_dropped": ("          + rho * terms[\"s_h\"])", "          )"),
}


def _mutant(name, tmp_path):
    src = open(SRC).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"snippet for {name} not found exactly once"
    src = src.replace(old, new).replace("from .reference import", "from oracle.reference import")
    path = tmp_path / f"swiglu_{name}.py"
    path.write_text(src)
    spec = importlib.util.spec_from_file_location(f"swiglu_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    mod = _mutant(name, tmp_path)
    failed = []
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutation {name} passed every pin"
