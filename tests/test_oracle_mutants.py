"""Mutation tests: plant a plausible mistake in a copy of the oracle's C
source, build it on the CPU, and check that at least one pin catches it.
The oracle itself is never modified."""
import os

import pytest

import oracle as oracle_pkg
import oracle_pins

# (name, original snippet, mutated snippet)
MUTANTS = [
    ("round_ties_up",
     "return (fmodf(f, 2.0f) == 0.0f) ? f : f + 1.0f;", "return f + 1.0f;"),
    ("truncate_instead_of_round",
     "float t = round_half_even(v / scale);", "float t = truncf(v / scale);"),
    ("multiply_by_127_over_amax",
     "float t = round_half_even(v / scale);",
     "float t = round_half_even(v * (127.0f / amax));"),
    ("drop_last_k",
     "for (int64_t k = 0; k < K; ++k)\n                sum += (int64_t)a[k] * (int64_t)b[k];",
     "for (int64_t k = 0; k < K - 1; ++k)\n                sum += (int64_t)a[k] * (int64_t)b[k];"),
    ("transposed_weight",
     "sum += (int64_t)a[k] * (int64_t)b[k];",
     "sum += (int64_t)a[k] * (int64_t)wq[k * N + n];"),
    ("dequant_drops_weight_scale", "float scale = sx * sw;", "float scale = sx;"),
    ("dequant_other_order", "return a * scale;", "return (a * sx) * sw;"),
    ("argmax_last_tie", "if (y[m * N + n] > bv)", "if (y[m * N + n] >= bv)"),
    ("lm_head_last_tie", "if (best < 0 || y > bv)", "if (best < 0 || y >= bv)"),
    ("accept_no_bonus", "len[b] = (int32_t)(k + 1);", "len[b] = (int32_t)k;"),
    ("accept_out_short", "out[b * G + j] = (j <= k) ? t[b * G + j] : -1;",
     "out[b * G + j] = (j < k) ? t[b * G + j] : -1;"),
    ("accept_shifted_compare", "d[b * gamma + k] == t[b * G + k]",
     "d[b * gamma + k] == t[b * G + k + 1]"),
    ("bf16_ties_away", "(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)"),
    ("amax_ignores_smoothing",
     "float v = mul ? xr[k] * mul[k] : xr[k];\n            float a = fabsf(v);",
     "float v = xr[k];\n            float a = fabsf(v);"),
    ("linear_f64_in_float", "double sum = 0.0;", "float sum = 0.0f;"),
    ("exp_taylor_short", "for (int n = 6; n >= 0; --n) {", "for (int n = 6; n >= 2; --n) {"),
    ("exp_drops_ln2_lo", "r = r - k * QVO_LN2_LO;", "r = r;"),
    ("silu_sigmoid_sign", "float e = qvo_exp(-v);", "float e = qvo_exp(v);"),
    ("swiglu_gate_up_swapped", "a[k] = qvo_silu(row[k]) * row[F + k];",
     "a[k] = qvo_silu(row[F + k]) * row[k];"),
    ("rmsnorm_sum_not_mean", "float var = (float)(ss / (double)H);", "float var = (float)ss;"),
    ("rmsnorm_no_sqrt", "float sq = sqrtf(t);", "float sq = t;"),
    ("rmsnorm_ignores_weight", "x[k] = qvo_f32_to_bf16_rne(qvo_bf16_to_f32(g[k]) * u);",
     "x[k] = qvo_f32_to_bf16_rne(u);"),
    ("spec_keep_test_inverted", "if (lhs < rhs) continue;", "if (lhs > rhs) continue;"),
    ("spec_residual_q_minus_p", "x128[v] = a1 > a2 ? a1 - a2 : 0;", "x128[v] = a2 > a1 ? a2 - a1 : 0;"),
    ("spec_bonus_from_first_row", "int64_t row = b * G + gamma;", "int64_t row = b * G;"),
    ("spec_draw_inclusive", "if (acc > target) return (int32_t)v;\n    }\n    return (int32_t)(V - 1);\n}\nstatic int32_t draw_u128",
     "if (acc >= target) return (int32_t)v;\n    }\n    return (int32_t)(V - 1);\n}\nstatic int32_t draw_u128"),
    ("spec_same_draw_for_both", "(uint64_t)(2 * row + 1)) >> 40);\n            if (R > 0)",
     "(uint64_t)(2 * row)) >> 40);\n            if (R > 0)"),
    ("splitmix_constant", "0xBF58476D1CE4E5B9ull", "0xBF58476D1CE4E5B8ull"),
    ("tree_own_token", "acc[i] = (p >= 0 && p < i && acc[p] && db[i] == tb[p]) ? 1 : 0;",
     "acc[i] = (p >= 0 && p < i && acc[p] && db[i] == tb[i]) ? 1 : 0;"),
    ("tree_ignores_ancestors", "acc[i] = (p >= 0 && p < i && acc[p] && db[i] == tb[p]) ? 1 : 0;",
     "acc[i] = (p >= 0 && p < i && db[i] == tb[p]) ? 1 : 0;"),
    ("tree_ties_last", "if (acc[i] && depth[i] > depth[best]) best = i;",
     "if (acc[i] && depth[i] >= depth[best]) best = i;"),
    ("tree_bonus_from_parent", "out[b * N + D] = tb[best];", "out[b * N + D] = tb[pb[best] >= 0 ? pb[best] : 0];"),
    ("w4_scale_127", "float scale = amax / 7.0f;", "float scale = amax / 127.0f;"),
    ("w4_truncate", "float t = round_half_even(xr[k] / scale);", "float t = truncf(xr[k] / scale);"),
    ("w4_nibbles_swapped", "packed[r * (K / 2) + j] = (uint8_t)(lo | (hi << 4));",
     "packed[r * (K / 2) + j] = (uint8_t)(hi | (lo << 4));"),
    ("w4_unpack_unsigned", "return (int8_t)(n >= 8u ? (int)n - 16 : (int)n);", "return (int8_t)n;"),
    ("w4_unpack_high_first", "q[r * K + 2 * j] = nibble_value(byte & 0xFu);",
     "q[r * K + 2 * j] = nibble_value(byte >> 4);"),
    ("kl_reversed", "s += exp(lp) * (lp - lq);", "s += exp(lq) * (lq - lp);"),
    ("kl_no_normalisation", "const double lp = (double)ar[v] - ma - lza;", "const double lp = (double)ar[v] - ma;"),
    ("fidelity_last_tie", "if (ar[v] > ar[ia]) ia = v;", "if (ar[v] >= ar[ia]) ia = v;"),
    ("attention_not_causal", "const int64_t n = L + j + 1;", "const int64_t n = L + T;"),
    ("attention_heads_interleaved", "const int64_t kh = h / G;", "const int64_t kh = h % Hkv;"),
    ("attention_no_scale", "s[i] = scale * dot;", "s[i] = dot;"),
    ("attention_values_from_keys", "(Hq + Hkv + kh) * D;\n                        acc", "(Hq + kh) * D;\n                        acc"),
    ("residual_not_added",
     "hr[k] = qvo_f32_to_bf16_rne(qvo_bf16_to_f32(hr[k]) + qvo_bf16_to_f32(d[m * H + k]));",
     "hr[k] = hr[k];"),
]


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, orig, mut):
    with open(oracle_pkg.SOURCE) as f:
        src = f.read()
    assert src.count(orig) >= 1, f"snippet for {name} not found"
    bad = src.replace(orig, mut, 1)
    csrc = tmp_path / f"{name}.c"
    csrc.write_text(bad)
    lib = oracle_pkg.build(str(csrc), str(tmp_path / f"lib{name}.so"), force=True)
    o = oracle_pkg.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, OverflowError, ValueError) as e:  # noqa: PERF203
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {name}"
