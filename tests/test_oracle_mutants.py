"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each mutant is a copy of ``oracle/oracle.c`` with one plausible error (a
dropped term, a wrong sign, index or operand, a wrong rounding rule), built
into a temporary library; at least one pin must fail on it.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "eps_outside_sqrt": ("sqrt(ss / (double)H + (double)eps)", "(sqrt(ss / (double)H) + (double)eps)"),
    "sum_not_mean": ("sqrt(ss / (double)H + (double)eps)", "sqrt(ss + (double)eps)"),
    "eps_dropped": ("sqrt(ss / (double)H + (double)eps)", "sqrt(ss / (double)H)"),
    "weight_dropped": ("y[j] = r[j] * inv * orc_bf16_decode(weight[j]);", "y[j] = r[j] * inv;"),
    "sum_not_rounded": ("r[j] = orc_bf16_decode(rb);", "r[j] = sum;"),
    "residual_not_added": ("orc_bf16_decode(xt[j]) + orc_bf16_decode(residual[t * H + j])",
                           "orc_bf16_decode(xt[j])"),
    "scale_multiplied": ("double vj = yg[j] / s;", "double vj = yg[j] * s;"),
    "static_scale_multiplied": ("double vj = y[j] / s;", "double vj = y[j] * s;"),
    "amax_not_abs": ("if (fabs(yg[j]) > amax)\n                amax = fabs(yg[j]);",
                     "if (yg[j] > amax)\n                amax = yg[j];"),
    "amax_propagates_nan": ("if (fabs(yg[j]) > amax)\n                amax = fabs(yg[j]);",
                            "if (!(fabs(yg[j]) <= amax))\n                amax = fabs(yg[j]);"),
    "silu_exp_form": ("a[j] = g / (1.0 + exp(-g)) * u;", "a[j] = g * exp(g) / (1.0 + exp(g)) * u;"),
    "fp8_max_480": ("#define ORC_E4M3_MAX 448.0", "#define ORC_E4M3_MAX 480.0"),
    "scale_layout_transposed": ("scale[t * ngroups + g] = s32;", "scale[g * 1 + t * 1] = s32;"),
    "ties_away_from_zero": ("return nearbyint(m) * quantum;", "return round(m) * quantum;"),
    "truncating_rounding": ("return nearbyint(m) * quantum;", "return trunc(m) * quantum;"),
    "no_subnormals": ("if (e < emin)\n        e = emin;", "if (e < emin)\n        return 0.0 * v;"),
    "sign_of_zero_lost": ("if (r == 0.0)\n        return sign;", "if (r == 0.0)\n        return 0;"),
    "silu_sign": ("a[j] = g / (1.0 + exp(-g)) * u;", "a[j] = g / (1.0 + exp(g)) * u;"),
    "silu_gate_up_swapped": ("double g = orc_bf16_decode(row[j]);\n            double u = orc_bf16_decode(row[I + j]);",
                             "double g = orc_bf16_decode(row[I + j]);\n            double u = orc_bf16_decode(row[j]);"),
    "silu_up_dropped": ("a[j] = g / (1.0 + exp(-g)) * u;", "a[j] = g / (1.0 + exp(-g));"),
    "e4m3_bias_8": ("return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | mant));",
                    "return (uint8_t)(sign | (uint8_t)(((e + 8) << 3) | mant));"),
    "amax_floor_dropped": ("double a = amax > orc_amax_floor() ? amax : orc_amax_floor();",
                           "double a = amax;"),
    "bf16_decode_shift": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    "bf16_norm_eps_dropped": ("sqrt(mean + (double)eps)", "sqrt(mean)"),
    "bf16_norm_sum_not_mean": ("double mean = ss / (double)H;", "double mean = ss;"),
    "bf16_norm_weight_dropped": ("double yj = r[j] * inv * orc_bf16_decode(weight[j]);",
                                 "double yj = r[j] * inv;"),
    "bf16_norm_rounded_twice": ("double yj = r[j] * inv * orc_bf16_decode(weight[j]);",
                                "double yj = orc_bf16_decode(orc_bf16_encode(r[j] * inv))"
                                " * orc_bf16_decode(weight[j]);"),
    "bf16_norm_row_offset_dropped": ("r[j] = orc_bf16_decode(x[t * H + j]);",
                                     "r[j] = orc_bf16_decode(x[j]);"),
    "pad_tail_not_zero": ("out[t * Hp + j] = j < H ? orc_bf16_encode(yj) : 0;",
                          "out[t * Hp + j] = j < H ? orc_bf16_encode(yj) : 0x3F80;"),
    "pad_row_stride_unpadded": ("out[t * Hp + j] = j < H ? orc_bf16_encode(yj) : 0;",
                                "if (j < H) out[t * H + j] = orc_bf16_encode(yj);"),
    "pad_residual_not_added": ("uint16_t rb = orc_bf16_encode(orc_bf16_decode(xrow[j]) +\n"
                               "                                              orc_bf16_decode(residual[t * H + j]));",
                               "uint16_t rb = orc_bf16_encode(orc_bf16_decode(xrow[j]));"),
    "pad_eps_dropped": ("double scale = 1.0 / sqrt(sq / (double)H + (double)eps);",
                        "double scale = 1.0 / sqrt(sq / (double)H);"),
    "ue8m0_rounds_down": ("    while (ldexp(ORC_E4M3_MAX, e - 1) >= a)\n        --e;\n    return ldexp(1.0, e);",
                          "    while (ldexp(ORC_E4M3_MAX, e - 1) >= a)\n        --e;\n    return ldexp(1.0, e - 1);"),
    "ue8m0_ignored": ("float s32 = (flags & ORC_UE8M0) ? (float)ue8m0_scale(amax) : dynamic_scale(amax);",
                      "float s32 = dynamic_scale(amax);"),
    "ue8m0_wrong_floor": ("const double a = fmax(amax, orc_amax_floor());", "const double a = fmax(amax, 1e-8);"),
    "col_major_unpadded_stride": ("scale[g * ((T + 3) / 4 * 4) + t] = s32;", "scale[g * T + t] = s32;"),
    "e2m1_ties_away": ("    double r = isinf(a) ? 6.0 : round_to_precision(a, 2, 0);",
                       "    double r = isinf(a) ? 6.0 : ldexp(round(ldexp(a, 1)), -1);"),
    "e2m1_max_4": ("    if (r > 6.0)\n        r = 6.0;", "    if (r > 4.0)\n        r = 4.0;"),
    "nvfp4_block_scale_no_div6": ("uint8_t code = orc_e4m3_encode((double)gs * amax / 6.0);",
                                  "uint8_t code = orc_e4m3_encode((double)gs * amax);"),
    "nvfp4_nibbles_swapped": ("                q4[col / 2] = e;\n            else\n                q4[col / 2] = (uint8_t)(q4[col / 2] | (e << 4));",
                              "                q4[col / 2] = (uint8_t)(e << 4);\n            else\n                q4[col / 2] = (uint8_t)(q4[col / 2] | e);"),
    "nvfp4_global_scale_ignored": ("double vj = s > 0.0 ? yb[j] * (double)gs / s : 0.0;",
                                   "double vj = s > 0.0 ? yb[j] / s : 0.0;"),
    "nvfp4_amax_not_abs": ("            if (fabs(yb[j]) > amax)\n                amax = fabs(yb[j]);",
                           "            if (yb[j] > amax)\n                amax = yb[j];"),
    "nvfp4_zero_block_divided": ("double vj = s > 0.0 ? yb[j] * (double)gs / s : 0.0;",
                                 "double vj = yb[j] * (double)gs / s;"),
    "rope_sign": ("rot[a] = y[a] * c - y[b] * sn;", "rot[a] = y[a] * c + y[b] * sn;"),
    "rope_cos_sin_swapped": ("double c = (double)cs[i], sn = (double)cs[D / 2 + i];",
                             "double sn = (double)cs[i], c = (double)cs[D / 2 + i];"),
    "rope_neox_pairs_adjacent": ("int64_t b = is_neox ? i + D / 2 : 2 * i + 1;",
                                 "int64_t b = is_neox ? 2 * i + 1 : 2 * i + 1;\n"
                                 "                a = is_neox ? 2 * i : a;"),
    "qk_k_heads_use_q_weight": ("const uint16_t *w = h < Hq ? q_weight : k_weight;",
                                "const uint16_t *w = q_weight;"),
    "qk_position_ignored": ("const float *cs = cos_sin_cache + positions[t] * D;",
                            "const float *cs = cos_sin_cache;"),
    "qk_eps_dropped": ("double inv_rms = 1.0 / sqrt(sq / (double)D + (double)eps);",
                       "double inv_rms = 1.0 / sqrt(sq / (double)D);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / f"oracle_{name}.c"
    mutated.write_text(src.replace(old, new))
    lib_path = oracle.compile_source(str(mutated), str(tmp_path / f"lib_{name}.so"))
    orc = oracle.Oracle(oracle.load_library(lib_path))
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(orc)
        except Exception as exc:  # noqa: BLE001 - any failure counts as caught
            caught.append(f"{check.__name__}: {type(exc).__name__}")
    assert caught, f"no pin catches the planted mistake {name!r}"
