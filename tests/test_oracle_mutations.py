"""Plant plausible mistakes in a copy of the C oracle; each must fail a pin.

The copy is compiled into a temporary directory; the committed oracle is
never touched. A mutation whose snippet is not found exactly once fails the
test, so the list stays in step with the source.
"""
import os

import pytest

import oracle.reference as ref
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(ref.__file__), "oracle.c")

MUTATIONS = {
    "high_nibble_first": [("(within % 2 == 0) ? (b & 0x0F)",
                           "(within % 2 == 1) ? (b & 0x0F)")],
    "all_low_then_all_high": [("int64_t j = within / 2;", "int64_t j = within % 16;"),
                              ("(within % 2 == 0) ? (b & 0x0F)",
                               "(within < 16) ? (b & 0x0F)")],
    "bias_wrong_sign": [("s - 127);", "127 - s);")],
    "bias_off_by_one": [("s - 127);", "s - 128);")],
    "one_scale_per_row": [("int s = scales[(e * O + o) * G + g];",
                           "int s = scales[(e * O + o) * G];")],
    "one_scale_per_matrix": [("int s = scales[(e * O + o) * G + g];",
                              "int s = scales[e * O * G];")],
    "scale_layout_swapped": [("int s = scales[(e * O + o) * G + g];",
                              "int s = scales[(o * 1 + e * 0) * G + g];")],
    "group_stride_wrong": [("int64_t g = i / 32;", "int64_t g = i / 64;")],
    "table_linear_misread": [("0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,",
                              "0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 3.0, 3.5,")],
    "table_sign_lost": [("-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,",
                         "0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,")],
    "shared_output_dropped": [("double y = y_shared[t * O + o];", "double y = 0.0;")],
    "mixture_weight_ignored": [("y += pk * dot;", "y += dot;")],
    "first_slot_expert_for_all": [("const int64_t e = sel[t * K + k];",
                                   "const int64_t e = sel[t * K];")],
    "last_slot_dropped": [("            for (int64_t k = 0; k < K; ++k) {",
                           "            for (int64_t k = 0; k + 1 < K; ++k) {")],
    "token_zero_for_all": [("const double term = w * x[t * I + i];",
                            "const double term = w * x[i];")],
    "abs_terms_without_shared": [("double a = fabs(y_shared[t * O + o]);",
                                  "double a = 0.0;")],
    "abs_terms_without_weight": [("mag += fabs(pk * term);", "mag += fabs(term);")],
    "invalid_index_not_counted": [("if (sel[t * K + k] < 0 || sel[t * K + k] >= E) ++bad;",
                                   "if (sel[t * K + k] < 0) ++bad;")],
}


def _impl_for(lib):
    def impl(x, packed, scales, sel, p, ys):
        return ref.expert_linear(x, packed, scales, sel, p, ys, lib=lib)
    return impl


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTATIONS[name]:
        assert src.count(old) == 1, f"snippet for {name} not unique: {old!r}"
        src = src.replace(old, new)
    mutant_c = tmp_path / "oracle_mutant.c"
    mutant_c.write_text(src)
    so = ref.build(force=True, src=str(mutant_c), out=str(tmp_path / "libmutant.so"))
    impl = _impl_for(ref.load(so))
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(impl)
        except (AssertionError, ValueError, IndexError):
            failed.append(check.__name__)
    assert failed, f"mutation {name} passed every pin"
