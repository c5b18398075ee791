"""Plant a mistake in a copy of the oracle's C source and require a pin to catch it.

Each mutant is a plausible slip (a wrong nibble order, sign, offset, rounding
rule, tie-break, dropped factor or transposed index).  The copy is compiled on
the CPU into a temporary directory and every pin runs against it; the test
passes only if at least one pin fails.  Mutants only change arithmetic or
in-bounds indexing, so a mutant cannot read or write out of bounds.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gq_oracle.c")

MUTANTS = {
    "nibble_order": ("out[2 + i] = (uint8_t)(q[i] | (q[i + QK / 2] << 4));",
                     "out[2 + i] = (uint8_t)((q[i] << 4) | q[i + QK / 2]);"),
    "q4_offset": ("s += (int32_t)(q4_code(b4, j) - 8) * (int32_t)q8_code(b8, j);",
                  "s += (int32_t)(q4_code(b4, j) - 7) * (int32_t)q8_code(b8, j);"),
    "q4_tie_break": ("if (a > amax) { amax = a; vmax = x[j]; }   /* strict: the first wins */\n    }\n    float d = vmax / -8.0f;",
                     "if (a >= amax) { amax = a; vmax = x[j]; }\n    }\n    float d = vmax / -8.0f;"),
    "q5_tie_break": ("if (a > amax) { amax = a; vmax = x[j]; }   /* strict: the first wins */\n    }\n    float d = vmax / -16.0f;",
                     "if (a >= amax) { amax = a; vmax = x[j]; }\n    }\n    float d = vmax / -16.0f;"),
    "q4_scale_sign": ("float d = vmax / -8.0f;", "float d = vmax / 8.0f;"),
    "q4_round_even": ("int v = (int)roundf(x[j] / d) + 8;", "int v = (int)rintf(x[j] / d) + 8;"),
    "q8_round_even": ("v = (int)roundf(x[j] / d);", "v = (int)rintf(x[j] / d);"),
    "q8_divisor": ("float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    "q4_codes_from_fp16_scale": ("int v = (int)roundf(x[j] / d) + 8;",
                                 "int v = (int)roundf(x[j] / oracle_f16_to_f32(oracle_f32_to_f16(d))) + 8;"),
    "q4_zero_block_code": ("q[j] = 8;", "q[j] = 0;"),
    "q4_high_nibble": ("uint8_t byte = blk[2 + (j % (QK / 2))];\n    return j < QK / 2 ? (byte & 0x0f) : (byte >> 4);",
                       "uint8_t byte = blk[2 + (j % (QK / 2))];\n    return j < QK / 2 ? (byte & 0x0f) : (byte & 0x0f);"),
    "q41_high_nibble": ("uint8_t byte = blk[4 + (j % (QK / 2))];\n    return j < QK / 2 ? (byte & 0x0f) : (byte >> 4);",
                        "uint8_t byte = blk[4 + (j % (QK / 2))];\n    return j < QK / 2 ? (byte & 0x0f) : (byte & 0x0f);"),
    "f16_ties_away": ("if (rem > half || (rem == half && (q & 1u))) q++;",
                      "if (rem >= half) q++;"),
    "f16_subnormal_scale": ("if (E == 0)       v = ldexpf((float)F, -24);",
                            "if (E == 0)       v = ldexpf((float)F, -25);"),
    "dropped_d8": ("acc += d4 * d8 * (double)block_dot(b4, b8);",
                   "acc += d4 * (double)block_dot(b4, b8);"),
    "transposed_dst": ("Q4_0_BYTES, wdata + m * nb * Q8_0_BYTES, nb,\n                              &dst[m * N + n], &T[m * N + n]);",
                       "Q4_0_BYTES, wdata + m * nb * Q8_0_BYTES, nb,\n                              &dst[n * M + m], &T[n * M + m]);"),
    "f16_reversed_k": ("double p = (double)oracle_f16_to_f32(w[k]) * (double)x[k];",
                       "double p = (double)oracle_f16_to_f32(w[k]) * (double)x[K - 1 - k];"),
    "q8w_dropped_dw": ("acc += dw * dx * (double)block_dot_q8_0(bw, bx);",
                       "acc += dx * (double)block_dot_q8_0(bw, bx);"),
    "q8w_shifted_lane": ("s += (int32_t)q8_code(bw, j) * (int32_t)q8_code(bx, j);",
                         "s += (int32_t)q8_code(bw, j) * (int32_t)q8_code(bx, (j + 1) % QK);"),
    "q5_offset": ("s += (int32_t)(q5_code(b5, j) - 16) * (int32_t)q8_code(b8, j);",
                  "s += (int32_t)(q5_code(b5, j) - 15) * (int32_t)q8_code(b8, j);"),
    "q5_fifth_bit_order": ("qh |= (uint32_t)((q[j] >> 4) & 1) << j;",
                           "qh |= (uint32_t)((q[j] >> 4) & 1) << (QK - 1 - j);"),
    "q5_scale_divisor": ("float d = vmax / -16.0f;", "float d = vmax / -15.0f;"),
    "q5_clamp": ("q[j] = v < 0 ? 0 : (v > 31 ? 31 : v);", "q[j] = v < 0 ? 0 : (v > 31 ? 15 : v);"),
    "q41_min_term_dropped": ("        acc += mn * d8 * (double)sums[1];\n", ""),
    "q41_divisor": ("float d = (hi - lo) / 15.0f;", "float d = (hi - lo) / 16.0f;"),
    "q41_offset_from_max": ("int v = (int)roundf((x[j] - lo) / d);", "int v = (int)roundf((x[j] - hi) / d) + 15;"),
    "kv_divisor": ("float s = amax / 127.0f;", "float s = amax / 128.0f;"),
    "kv_round_even": ("v = (int)roundf(xr[j] / s);", "v = (int)rintf(xr[j] / s);"),
    "kv_scale_through_fp16": ("float s = amax / 127.0f;\n        scale[r] = s;",
                              "float s = oracle_f16_to_f32(oracle_f32_to_f16(amax / 127.0f));\n        scale[r] = s;"),
    "attn_key_scale_dropped": ("p[t] = c * (double)ksb[t] * dot;", "p[t] = c * dot;"),
    "attn_value_scale_from_keys": ("double term = p[t] * (double)vsb[t] * (double)vb[t * D + j];",
                                   "double term = p[t] * (double)ksb[t] * (double)vb[t * D + j];"),
    "attn_values_from_keys": ("double term = p[t] * (double)vsb[t] * (double)vb[t * D + j];",
                              "double term = p[t] * (double)vsb[t] * (double)kb[t * D + j];"),
    "attn_group_map": ("int64_t hk = h / G;", "int64_t hk = h % Hkv;"),
    "attn_last_token_dropped": ("for (int64_t t = 0; t < L; t++) {\n                double dot = 0.0, adot = 0.0;",
                                "for (int64_t t = 0; t + 1 < L; t++) {\n                double dot = 0.0, adot = 0.0;"),
    "attn_no_max_shift": ("p[t] = exp(p[t] - m);", "p[t] = exp(p[t]);"),
    "attn_unnormalized": ("            for (int64_t t = 0; t < L; t++)\n                p[t] /= l;\n", ""),
    "attn_key_row_stride": ("double term = (double)qv[j] * (double)kb[t * D + j];",
                            "double term = (double)qv[j] * (double)kb[(t * D + j * 7) % (L * D)];"),
    "q8_abs_dropped": ("float a = fabsf(x[j]);\n        if (a > amax) amax = a;",
                       "float a = x[j];\n        if (a > amax) amax = a;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(before) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(before, after))
    lib = oracle.build(str(src), str(tmp_path / "libmutant.so"), force=True)
    o = oracle.Oracle(oracle.load(lib))
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
