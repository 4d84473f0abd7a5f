"""Planted mistakes in the oracle must each fail at least one pin.

Each case copies oracle.c, replaces one exact piece of its text with a
plausible mistake (a dropped rounding, a wrong index, a dropped term, ...),
compiles the copy with gcc into a temporary directory and runs the pins of
tests/oracle_pins.py on it.  Nothing here touches the real oracle or a GPU.
"""
import os

import pytest

import oracle
import oracle_pins as P

PLANTS = {
    # the weights are not rounded to bf16 (the pages' exact-codes lane form)
    "exact_weights": (
        "wrow[k] = oracle_bf16_to_double(\n"
        "                oracle_dequant_one(q, jb->scales[n * G + j], jb->biases[n * G + j]));",
        "wrow[k] = oracle_bf16_to_double(jb->scales[n * G + j]) * (double)q +\n"
        "                oracle_bf16_to_double(jb->biases[n * G + j]);"),
    # fp32 rounding of s*q + b before the bf16 rounding (double rounding)
    "double_rounding": (
        "return bf16_round_pair(hi, lo);",
        "return oracle_bf16_from_double((double)(float)hi);"),
    # the midpoint tie-break by the sign of the TwoSum remainder is lost
    "midpoint_tiebreak": (
        "if (lo == 0.0 || isnan(hi) || isinf(hi)) return r;",
        "return r;"),
    # ties away from zero instead of to even
    "ties_away": ("double rounded = nearbyint(scaled);", "double rounded = round(scaled);"),
    # underflow loses the sign of zero
    "unsigned_zero": ("return (uint16_t)(sign | (u >> 16));",
                      "return (uint16_t)(r == 0.0 ? 0 : (sign | (u >> 16)));"),
    # subnormals flushed: the grid never gets finer than the smallest normal's
    "no_subnormals": ("#define BF16_MIN_ULP_EXP (-133)", "#define BF16_MIN_ULP_EXP (-126)"),
    # group index off by one along K
    "group_off_by_one": (
        "            int64_t j = k / jb->group;\n            wrow[k]",
        "            int64_t j = (k + 1) / jb->group; if (j >= G) j = G - 1;\n            wrow[k]"),
    # one bias per row instead of one per group
    "bias_per_row": (
        "oracle_dequant_one(q, jb->scales[n * G + j], jb->biases[n * G + j]));",
        "oracle_dequant_one(q, jb->scales[n * G + j], jb->biases[n * G]));"),
    # the first product of every sum is dropped
    "dropped_term": ("for (int64_t k = 0; k < K; ++k) acc += wrow[k]",
                     "for (int64_t k = 1; k < K; ++k) acc += wrow[k]"),
    # fp32 accumulation in place of the exact (double) sum
    "float_accumulation": ("            double acc = 0.0;\n            for (int64_t k = 0; k < K; ++k) acc",
                           "            float acc = 0.0f;\n            for (int64_t k = 0; k < K; ++k) acc"),
    # every output row reads activation row 0
    "wrong_x_row": ("const uint16_t* xr = jb->x + m * K;", "const uint16_t* xr = jb->x;"),
    # the bias enters with the wrong sign
    "bias_sign": ("double hi = p + bd;\n    double bv = hi - p;",
                  "double hi = p - bd;\n    double bv = hi - p;"),
    # embedding rows: the scale applied to the unrounded weight (one rounding instead of two)
    "embed_no_first_rounding": (
        "out[t * K + k] = has_scale ? oracle_bf16_from_double(oracle_bf16_to_double(w) * sc) : w;",
        "out[t * K + k] = has_scale ? oracle_bf16_from_double((oracle_bf16_to_double(scales[n * G + j]) * (double)q + "
        "oracle_bf16_to_double(biases[n * G + j])) * sc) : w;"),
    # embedding rows: the scale folded into the group's scale and bias
    "embed_scale_folded": (
        "uint16_t w = oracle_dequant_one(q, scales[n * G + j], biases[n * G + j]);",
        "uint16_t w = has_scale ? oracle_dequant_one(q, oracle_bf16_from_double(oracle_bf16_to_double(scales[n * G + j]) * sc), "
        "oracle_bf16_from_double(oracle_bf16_to_double(biases[n * G + j]) * sc)) : "
        "oracle_dequant_one(q, scales[n * G + j], biases[n * G + j]); if (has_scale) { out[t * K + k] = w; continue; }"),
    # exact-codes form: the bias times the group's sum of x is dropped
    "groupsum_bias_dropped": ("acc += s * sqx + b * sx;", "acc += s * sqx;"),
    # exact-codes form: the codes' products use the next row's codes
    "groupsum_wrong_code_row": ("double q = (double)codes[n * K + k];",
                                "double q = (double)codes[((n + 1) % N) * K + k];"),
    # the scale and bias patterns swapped
    "swapped_scale_bias": ("double sd = oracle_bf16_to_double(s);\n    double bd = oracle_bf16_to_double(b);",
                           "double sd = oracle_bf16_to_double(b);\n    double bd = oracle_bf16_to_double(s);"),
}


@pytest.mark.parametrize("name", sorted(PLANTS))
def test_plant_is_caught(name, tmp_path):
    old, new = PLANTS[name]
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"plant {name!r}: target text not found exactly once"
    mutated = tmp_path / "oracle.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_oracle(str(mutated), str(tmp_path / "liboracle_plant.so"))
    orc = oracle.Oracle(lib)
    failures = []
    for pin in P.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failures.append(pin.__name__)
    assert failures, f"planted mistake {name!r} passed every pin"
