"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case copies the oracle's C source, plants one plausible mistake by a
textual substitution (at every place the anchor text occurs), compiles the copy into a temporary library and runs
every pin check against it.  At least one pin must fail for every mutant;
the unmodified source must pass them all (tests/test_oracle_pins.py).
"""
import os

import pytest

import oracle
import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "qgemm_oracle.c")

MUTANTS = {
    "msb_first_bit_order": ("return (int)((v >> (bit % 8)) & ((1u << bits) - 1u));",
                            "return (int)((v >> (8 - bits - bit % 8)) & ((1u << bits) - 1u));"),
    "straddling_code_truncated": ("if (bit % 8 + bits > 8) /* the code continues into the next byte */\n"
                                  "        v |= (unsigned)row[bit / 8 + 1] << 8;", ""),
    "scales_transposed": ("float s = (float)oracle_half_to_double(scales[n * nb + b]);",
                          "float s = (float)oracle_half_to_double(scales[b * N + n]);"),
    "zero_point_sign": ("float d = (float)q - zpv;", "float d = zpv - (float)q;"),
    "midpoint_wrong": ("zpv = (float)(1 << (bits - 1));", "zpv = (float)((1 << bits) - 1);"),
    "block_index_mod": ("int64_t b = k / bs;", "int64_t b = k % nb;"),
    "codebook_reversed": ("float w = codebook[q] * absmax[n * nb + k / bs];",
                          "float w = codebook[15 - q] * absmax[n * nb + k / bs];"),
    "absmax_row_dropped": ("float w = codebook[q] * absmax[n * nb + k / bs];",
                           "float w = codebook[q] * absmax[k / bs];"),
    "half_exponent_bias": ("v = ldexp((double)(f + 1024), e - 25);", "v = ldexp((double)(f + 1024), e - 24);"),
    "half_subnormal_scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "bf16_shift": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    "activation_transposed": ("double a = load_elem(A, a_dtype, (size_t)(m * K + k));\n                double w = (double)oracle_weight_nbits",
                              "double a = load_elem(A, a_dtype, (size_t)(k * M + m));\n                double w = (double)oracle_weight_nbits"),
    "gate_up_swapped": ("double gate = swiglu_interleaved ? g[2 * i] : g[i];\n            double up = swiglu_interleaved ? g[2 * i + 1] : g[I + i];",
                        "double gate = swiglu_interleaved ? g[2 * i] : g[I + i];\n            double up = swiglu_interleaved ? g[2 * i + 1] : g[i];"),
    "silu_sign": ("return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    "fc2_bias_dropped": ("if (fc2_bias) acc += oracle_half_to_double(fc2_bias[(int64_t)e * H + r]);", ""),
    "fc1_bias_wrong_expert": ("if (fc1_bias) acc += oracle_half_to_double(fc1_bias[(int64_t)e * I2 + r]);",
                              "if (fc1_bias) acc += oracle_half_to_double(fc1_bias[r]);"),
    "slot_weight_dropped": ("y[r] += (double)weights[j] * acc;", "y[r] += acc;"),
    "expert_offset_by_slot": ("const uint8_t *w1 = fc1_w + (int64_t)e * I2 * fc1_row_bytes;",
                              "const uint8_t *w1 = fc1_w + (int64_t)j * I2 * fc1_row_bytes;"),
    "bad_id_not_reported": ("if (e < 0 || e >= num_experts) {\n            ++bad;\n            continue;\n        }",
                            "if (e < 0 || e >= num_experts) {\n            continue;\n        }"),
    "uniform_by_value": ("if (t[i] != t[0]) return 0;",
                         "if (oracle_half_to_double(t[i]) != oracle_half_to_double(t[0])) return 0;"),
    "uniform_accepts_nan": ("if (isnan(v)) return 0;", ""),
    "e4m3_exponent_bias": ("v = ldexp((double)(f + 8), e - 10);", "v = ldexp((double)(f + 8), e - 9);"),
    "e4m3_subnormal_scale": ("v = ldexp((double)f, -9);", "v = ldexp((double)f, -10);"),
    "e4m3_nan_missing": ("if (e == 15 && f == 7)\n        return NAN;", ""),
    "gather_negative_not_wrapped": ("if (row < 0)\n            row += V;", ""),
    "gather_bad_index_not_counted": ("++bad;\n            for (int64_t d = 0; d < D; ++d)",
                                     "for (int64_t d = 0; d < D; ++d)"),
    "gather_scale_by_position": ("scales[row * nb + d / bs]", "scales[i * nb + d / bs]"),
    "i8_truncates": ("float r = rintf(v[k] / s);", "float r = truncf(v[k] / s);"),
    "i8_rounds_half_up": ("float r = rintf(v[k] / s);", "float r = floorf(v[k] / s + 0.5f);"),
    "i8_scale_128": ("float s = a / 127.0f;", "float s = a / 128.0f;"),
    "dp4a_zero_point_sum_dropped": ("((double)dot - z * (double)sum)", "((double)dot)"),
    "dp4a_first_block_scale": ("acc += s * (double)sx[b] *", "acc += s * (double)sx[0] *"),
    "dp4a_h_not_requantized": ("oracle_quantize_i8_blocks(h, I, bs, q8, sx);", ""),
    "ragged_scales_not_offset": ("const uint16_t *se = scales + (int64_t)e * N * nb;", "const uint16_t *se = scales;"),
    "ragged_row_within_segment": ("load_elem(X, x_dtype, (size_t)(r * K + k))",
                                  "load_elem(X, x_dtype, (size_t)((r - off[e]) * K + k))"),
    "ragged_first_offset_unchecked": ("if (off[0] != 0)\n        return -1;", ""),
    "nested_offset_dropped": ("absmax[i] = v + offset;", "absmax[i] = v;"),
    "nested_scale_index": ("absmax2[i / nested_bs]", "absmax2[i % nested_bs]"),
    "nested_table_reversed": ("table256[qa[i]]", "table256[255 - qa[i]]"),
    "packed_zp_rows_unpadded": ("int64_t row_bytes = (nb * bits + 7) / 8;", "int64_t row_bytes = nb * bits / 8;"),
    "packed_zp_straddle_dropped": ("if (bit % 8 + bits > 8) /* the field continues into the next byte */\n"
                                   "                v |= (unsigned)row[bit / 8 + 1] << 8;", ""),
    "packed_zp_msb_first": ("out[n * nb + b] = (int32_t)((v >> (bit % 8))",
                            "out[n * nb + b] = (int32_t)((v >> ((8 - bits - bit % 8) & 7))"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    # the same mistake is planted at every occurrence (the fp and int8 QMoE
    # decodes share their slot loop's text)
    assert src.count(old) >= 1, "mutation anchor not found: %s" % name
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(force=True, src=str(msrc), out=str(tmp_path / "libmutant.so")))
    failed = []
    for check in P.ALL_CHECKS:
        try:
            check(lib)
        except (AssertionError, IndexError, ValueError):
            failed.append(check.__name__)
    assert failed, "no pin catches the planted mistake %r" % name
