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
    # supplied group sums: every activation row takes row 0's sums
    "given_sums_row0": ("acc += s * sqx + b * (double)xsums[m * G + j];", "acc += s * sqx + b * (double)xsums[j];"),
    # supplied group sums ignored: recomputed from x (the form the producer's sums replace)
    "given_sums_recomputed": (
        "                for (int64_t k = j * group; k < (j + 1) * group; ++k)\n"
        "                    sqx += (double)codes[n * K + k] * oracle_bf16_to_double(xr[k]);\n"
        "                acc += s * sqx + b * (double)xsums[m * G + j];",
        "                double sx = 0.0;\n"
        "                for (int64_t k = j * group; k < (j + 1) * group; ++k) {\n"
        "                    sqx += (double)codes[n * K + k] * oracle_bf16_to_double(xr[k]);\n"
        "                    sx += oracle_bf16_to_double(xr[k]); }\n"
        "                acc += s * sqx + b * sx;"),
    # GeGLU: each plant drops one rounding point of the bf16 chain, or changes a constant or an operand
    "geglu_cube_unrounded": ("uint16_t a = bf_round(bf(c1) * bf(c3));", "uint16_t a = bf_round(bf(c1) * (gv * gv * gv));"),
    "geglu_product_unrounded": ("uint16_t z = bf_round(gv + bf(a));", "uint16_t z = bf_round(gv + bf(c1) * bf(c3));"),
    "geglu_sum_unrounded": ("uint16_t u = bf_round(bf(c2) * bf(z));", "uint16_t u = bf_round(bf(c2) * (gv + bf(a)));"),
    "geglu_scaled_unrounded": ("const double tv = tanh(bf(u));", "const double tv = tanh(bf(c2) * bf(z));"),
    "geglu_tanh_unrounded": (
        "        h_lo[i] = geglu_tail(g, bf(t_lo), up[i]);\n        h_hi[i] = geglu_tail(g, bf(t_hi), up[i]);",
        "        h_lo[i] = geglu_tail(g, tv, up[i]);\n        h_hi[i] = geglu_tail(g, tv, up[i]);"),
    "geglu_one_plus_unrounded": ("    uint16_t r = bf_round(bf(p) * bf(e));", "    uint16_t r = bf_round(bf(p) * (1.0 + t));"),
    "geglu_gelu_unrounded": ("    return bf_round(bf(r) * bf(up));", "    return bf_round(bf(p) * bf(e) * bf(up));"),
    "geglu_constants_unrounded": (
        "    const uint16_t c1 = bf_round(0.044715);\n    const uint16_t c2 = bf_round(sqrt(2.0 / 3.14159265358979323846));",
        "    const uint16_t c1 = bf_round(0.044715) + 1;\n    const uint16_t c2 = bf_round(sqrt(2.0 / 3.14159265358979323846)) - 1;"),
    "geglu_half_dropped": ("    uint16_t p = bf_round(0.5 * bf(g));", "    uint16_t p = g;"),
    "geglu_up_ignored": ("    return bf_round(bf(r) * bf(up));", "    return r;"),
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
