"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Each ``check_*`` takes an implementation ``impl(x, packed, scales, sel, p,
y_shared) -> (out, abs_terms_or_None, bad_pairs)`` and raises AssertionError
when the implementation disagrees with:

  * values printed on the pages (tests/golden/page_examples.json): the 32.0
    worked example, the 0x21 decoding example, the E2M1 table, the scale
    factors for bytes 126/127/128, the output shapes;
  * closed forms: every table entry in both nibble positions, 2^(s-127) for
    every scale byte, per-(row, group) scales;
  * an independent encoder: codes and scale bytes chosen first, packed into
    bytes following the storage description (position 2j in the low nibble,
    2j+1 in the high one, group g in bytes [g, :]), so the expected matrix is
    known without decoding bytes; the expected result is then a library
    matmul, or exact rational arithmetic;
  * invariants: unselected experts cannot matter, p = 0 or K = 0 returns the
    shared output, relabelling experts changes nothing, scale + 1 doubles the
    routed part exactly, the result is linear in p, slot order is irrelevant,
    abs_terms equals the result when every term is non-negative.

The set is chosen so that each plausible slip in an oracle (nibble order,
bias sign, scale granularity, table entry, dropped term, wrong index, missing
weight) fails at least one check; tests/test_oracle_mutations.py plants those
slips in a copy of the oracle and confirms it.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "page_examples.json")))
TABLE = GOLDEN["e2m1_table"]["values"]


# ---------------------------------------------------------------- helpers --
def encode(codes: np.ndarray) -> np.ndarray:
    """Pack nibble codes (E, O, I) into bytes (E, O, I/32, 16).

    Storage description: each 32-value group is 16 bytes; byte j of group g
    holds input position 32g+2j in its low nibble and 32g+2j+1 in its high
    nibble.
    """
    E, O, I = codes.shape
    G = I // 32
    packed = np.zeros((E, O, G, 16), dtype=np.uint8)
    for i in range(I):
        g, within = divmod(i, 32)
        j, high = divmod(within, 2)
        packed[:, :, g, j] |= (codes[:, :, i].astype(np.uint8) << (4 * high))
    return packed


def matrix_from_codes(codes: np.ndarray, scale_bytes: np.ndarray) -> np.ndarray:
    """Dense float64 weights from chosen codes and scale bytes (no bytes)."""
    E, O, I = codes.shape
    vals = np.array(TABLE)[codes]
    factor = np.power(2.0, scale_bytes.astype(np.float64) - 127.0)  # (E,O,G)
    return vals * np.repeat(factor, 32, axis=2)


def one_hot(I: int, i: int) -> np.ndarray:
    x = np.zeros((1, I))
    x[0, i] = 1.0
    return x


def dyadic(rng, shape, bits=6):
    """Random values with few significant bits (exact in bf16 and float64)."""
    m = rng.integers(-(1 << bits), (1 << bits) + 1, size=shape)
    e = rng.integers(-4, 3, size=shape)
    return np.ldexp(m.astype(np.float64), e)


def single_group_case(byte_at_j0: int, scale: int, x: np.ndarray):
    packed = np.zeros((1, 1, 1, 16), dtype=np.uint8)
    packed[0, 0, 0, 0] = byte_at_j0
    scales = np.array([[[scale]]], dtype=np.uint8)
    return (x, packed, scales, np.array([[0]]), np.array([[1.0]]),
            np.zeros((x.shape[0], 1)))


def _close(a, b, rel=1e-12, scale=None):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    s = np.abs(b) if scale is None else np.asarray(scale)
    assert np.all(np.abs(a - b) <= rel * np.maximum(s, 1e-300)), (a, b)


# ----------------------------------------------------- values the pages print
def check_worked_example_32(impl):
    ex = GOLDEN["worked_example_32"]
    out, _, _ = impl(np.array(ex["latent_tokens"], float),
                     np.array(ex["packed_weights"], np.uint8),
                     np.array(ex["scale_bytes"], np.uint8),
                     np.array(ex["selected_experts"]),
                     np.array(ex["mixture_weights"], float),
                     np.array(ex["shared_output"], float))
    assert out.shape == (1, 1)
    assert out[0, 0] == ex["output"][0][0], out


def check_decode_0x21(impl):
    ex = GOLDEN["decode_0x21"]
    for s, (v0, v1) in ex["decoded_at_scale"].items():
        for pos, want in ((0, v0), (1, v1)):
            out, _, _ = impl(*single_group_case(ex["byte"], int(s), one_hot(32, pos)))
            assert out[0, 0] == want, (s, pos, out[0, 0], want)


def check_scale_factor_examples(impl):
    for s, f in GOLDEN["scale_factors"]["byte_to_factor"].items():
        out, _, _ = impl(*single_group_case(0x22, int(s), np.ones((1, 32))))
        # byte 0x22 is code 2 (1.0) in both nibbles; only position 0 and 1 set
        assert out[0, 0] == 2.0 * f, (s, out[0, 0])


def check_shape_examples(impl):
    rng = np.random.default_rng(11)
    for c in GOLDEN["shape_examples"]["cases"]:
        T, I = c["latent_tokens"]
        E, O, G, _ = c["packed_weights"]
        K = c["selected_experts"][1]
        sel = np.stack([rng.permutation(E)[:K] for _ in range(T)])
        out, _, _ = impl(rng.standard_normal((T, I)),
                         rng.integers(0, 256, (E, O, G, 16), dtype=np.uint8),
                         rng.integers(120, 130, (E, O, G), dtype=np.uint8),
                         sel, np.full((T, K), 1.0 / K),
                         rng.standard_normal(tuple(c["shared_output"])))
        assert tuple(out.shape) == tuple(c["output"]), out.shape


# ------------------------------------------------------------- closed forms
def check_every_table_entry_both_nibbles(impl):
    for code, want in enumerate(TABLE):
        out, _, _ = impl(*single_group_case(code, 127, one_hot(32, 0)))
        assert out[0, 0] == want, ("low", code, out[0, 0])
        out, _, _ = impl(*single_group_case(code << 4, 127, one_hot(32, 1)))
        assert out[0, 0] == want, ("high", code, out[0, 0])
        # the other nibble position must read zero (code 0)
        out, _, _ = impl(*single_group_case(code, 127, one_hot(32, 1)))
        assert out[0, 0] == 0.0, ("low leaks into high", code)


def check_every_scale_byte(impl):
    for s in range(256):
        out, _, _ = impl(*single_group_case(0x02, s, one_hot(32, 0)))
        assert out[0, 0] == np.ldexp(1.0, s - 127), (s, out[0, 0])


def check_scale_granularity(impl):
    # 3 rows x 3 groups, every (row, group) its own scale; byte 0x22 = 1.0, 1.0
    O, G = 3, 3
    scales = np.array([[[120, 127, 131], [125, 129, 122], [133, 118, 127]]],
                      dtype=np.uint8)
    packed = np.full((1, O, G, 16), 0x22, dtype=np.uint8)
    x = np.zeros((1, 32 * G))
    weights_of_group = [1.0, 10.0, 100.0]
    for g in range(G):
        x[0, 32 * g:32 * (g + 1)] = weights_of_group[g]
    out, _, _ = impl(x, packed, scales, np.array([[0]]), np.array([[1.0]]),
                     np.zeros((1, O)))
    want = [sum(32 * weights_of_group[g] * 2.0 ** (int(scales[0, o, g]) - 127)
                for g in range(G)) for o in range(O)]
    _close(out[0], want, 1e-15)


# ------------------------------------------------ independent encoder pins
def _encoded_case(seed, T=3, E=3, K=2, I=96, O=5):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(E, O, I))
    scale_bytes = rng.integers(119, 136, size=(E, O, I // 32)).astype(np.uint8)
    x = dyadic(rng, (T, I))
    y_shared = dyadic(rng, (T, O))
    sel = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    p = dyadic(rng, (T, K), bits=4) / 16.0
    return codes, scale_bytes, encode(codes), x, y_shared, sel, p


def check_encoded_matrix_matmul(impl):
    for seed in range(3):
        codes, sb, packed, x, ys, sel, p = _encoded_case(seed)
        W = matrix_from_codes(codes, sb)
        want = ys.copy()
        for t in range(x.shape[0]):
            for k in range(sel.shape[1]):
                want[t] += p[t, k] * (W[sel[t, k]] @ x[t])
        out, _, _ = impl(x, packed, sb, sel, p, ys)
        _close(out, want, 1e-12, scale=np.abs(want) + 1.0)


def check_encoded_exact_rational(impl):
    codes, sb, packed, x, ys, sel, p = _encoded_case(7, T=2, E=2, K=2, I=64, O=3)
    T, I = x.shape
    O = ys.shape[1]
    table = [Fraction(v) for v in TABLE]
    for t in range(T):
        for o in range(O):
            exact = Fraction(ys[t, o])
            mag = abs(Fraction(ys[t, o]))
            for k in range(sel.shape[1]):
                e = int(sel[t, k])
                pk = Fraction(p[t, k])
                for i in range(I):
                    w = table[codes[e, o, i]] * Fraction(2) ** (int(sb[e, o, i // 32]) - 127)
                    term = pk * w * Fraction(x[t, i])
                    exact += term
                    mag += abs(term)
            out, absm, _ = impl(x, packed, sb, sel, p, ys)
            assert abs(Fraction(out[t, o]) - exact) <= Fraction(1, 10**12) * mag, (t, o)
            if absm is not None:
                assert abs(Fraction(absm[t, o]) - mag) <= Fraction(1, 10**12) * mag


# --------------------------------------------------------------- invariants
def _random_case(seed, T=4, E=5, K=2, I=64, O=6):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, I)),
            rng.integers(0, 256, (E, O, I // 32, 16), dtype=np.uint8),
            rng.integers(118, 136, (E, O, I // 32), dtype=np.uint8),
            np.stack([rng.permutation(E)[:K] for _ in range(T)]),
            rng.random((T, K)), rng.standard_normal((T, O)))


def check_unselected_experts_do_not_matter(impl):
    x, packed, scales, sel, p, ys = _random_case(1, E=6, K=2)
    sel[:] = np.array([0, 2])          # experts 1, 3, 4, 5 never selected
    base, _, _ = impl(x, packed, scales, sel, p, ys)
    rng = np.random.default_rng(99)
    packed2, scales2 = packed.copy(), scales.copy()
    for e in (1, 3, 4, 5):
        packed2[e] = rng.integers(0, 256, packed2[e].shape, dtype=np.uint8)
        scales2[e] = rng.integers(0, 256, scales2[e].shape, dtype=np.uint8)
    out, _, _ = impl(x, packed2, scales2, sel, p, ys)
    assert np.array_equal(out, base)


def check_shared_path(impl):
    x, packed, scales, sel, p, ys = _random_case(2)
    out, absm, _ = impl(x, packed, scales, sel, np.zeros_like(p), ys)
    assert np.array_equal(out, ys)
    out, absm, _ = impl(x, packed, scales, sel[:, :0], p[:, :0], ys)
    assert np.array_equal(out, ys)
    if absm is not None:
        assert np.array_equal(absm, np.abs(ys))


def check_expert_relabelling(impl):
    x, packed, scales, sel, p, ys = _random_case(3)
    E = packed.shape[0]
    perm = np.random.default_rng(5).permutation(E)       # new id of expert e
    packed2 = np.empty_like(packed)
    scales2 = np.empty_like(scales)
    packed2[perm] = packed
    scales2[perm] = scales
    a, _, _ = impl(x, packed, scales, sel, p, ys)
    b, _, _ = impl(x, packed2, scales2, perm[sel], p, ys)
    assert np.array_equal(a, b)


def check_scale_plus_one_doubles(impl):
    x, packed, scales, sel, p, ys = _random_case(4)
    zero = np.zeros_like(ys)
    a, _, _ = impl(x, packed, scales, sel, p, zero)
    b, _, _ = impl(x, packed, scales + 1, sel, p, zero)
    assert np.array_equal(b, 2.0 * a)


def check_linear_in_p_and_slot_order(impl):
    x, packed, scales, sel, p, ys = _random_case(5, K=3, E=6)
    a, _, _ = impl(x, packed, scales, sel, p, ys)
    b, _, _ = impl(x, packed, scales, sel, 2.0 * p, ys)
    _close(b - ys, 2.0 * (a - ys), 1e-12, scale=np.abs(a - ys) + 1.0)
    order = [2, 0, 1]
    c, _, _ = impl(x, packed, scales, sel[:, order], p[:, order], ys)
    _close(c, a, 1e-12, scale=np.abs(a) + 1.0)
    # per-slot contributions add up: slot-by-slot sums equal the whole
    parts = sum(impl(x, packed, scales, sel[:, k:k + 1], p[:, k:k + 1],
                     np.zeros_like(ys))[0] for k in range(3))
    _close(parts + ys, a, 1e-12, scale=np.abs(a) + 1.0)


def check_abs_terms(impl):
    # All-positive inputs: abs_terms equals the result itself.
    rng = np.random.default_rng(6)
    T, E, K, I, O = 3, 4, 2, 64, 5
    codes = rng.integers(0, 8, size=(E, O, I))          # non-negative codes
    sb = rng.integers(120, 130, size=(E, O, I // 32)).astype(np.uint8)
    x = np.abs(dyadic(rng, (T, I)))
    ys = np.abs(dyadic(rng, (T, O)))
    sel = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    p = np.array([[0.25, 0.75]] * T)
    out, absm, _ = impl(x, encode(codes), sb, sel, p, ys)
    if absm is None:
        return
    _close(absm, out, 1e-14, scale=np.abs(out) + 1e-300)
    # with negative y_shared it is |y_shared| that enters
    out2, absm2, _ = impl(x, encode(codes), sb, sel, p, -ys)
    _close(absm2, absm, 1e-14, scale=absm)


def check_duplicate_pick_sums_slots(impl):
    x, packed, scales, sel, p, ys = _random_case(8, K=1)
    a, _, _ = impl(x, packed, scales, sel, np.ones_like(p), ys)
    b, _, _ = impl(x, packed, scales, np.concatenate([sel, sel], 1),
                   np.full((sel.shape[0], 2), 0.5), ys)
    _close(b, a, 1e-13, scale=np.abs(a) + 1.0)


def check_invalid_index_skipped(impl):
    x, packed, scales, sel, p, ys = _random_case(9, K=2)
    E = packed.shape[0]
    bad = sel.copy()
    bad[0, 1] = E          # out of range: the pair contributes nothing
    bad[2, 0] = -1
    out, _, nbad = impl(x, packed, scales, bad, p, ys)
    want, _, _ = impl(x, packed, scales, sel, np.where(bad == sel, p, 0.0), ys)
    assert np.array_equal(out, want)
    if nbad is not None:
        assert nbad == 2


ALL_CHECKS = [
    check_worked_example_32, check_decode_0x21, check_scale_factor_examples,
    check_shape_examples, check_every_table_entry_both_nibbles,
    check_every_scale_byte, check_scale_granularity,
    check_encoded_matrix_matmul, check_encoded_exact_rational,
    check_unselected_experts_do_not_matter, check_shared_path,
    check_expert_relabelling, check_scale_plus_one_doubles,
    check_linear_in_p_and_slot_order, check_abs_terms,
    check_duplicate_pick_sums_slots, check_invalid_index_skipped,
]
