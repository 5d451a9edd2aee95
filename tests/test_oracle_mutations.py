"""Plant one plausible mistake at a time in a copy of the oracle's C source
and check that the pins catch it. Nothing here touches a GPU."""

import os

import pytest

import oracle
import oracle_pins as pins

# (name, [(exact text in moe_oracle.c, replacement)])
MUTATIONS = [
    ("int4_nibble_order_swapped", [("const int code = (nibble & 1) ? (byte >> 4) : (byte & 15);",
                                    "const int code = (nibble & 1) ? (byte & 15) : (byte >> 4);")]),
    ("int4_two_per_byte_order", [("const size_t nibble = in_word / 2 + 4 * (in_word % 2);",
                                  "const size_t nibble = in_word;")]),
    ("int4_pairs_not_split", [("const size_t nibble = in_word / 2 + 4 * (in_word % 2);",
                               "const size_t nibble = (in_word % 4) * 2 + in_word / 4;")]),
    ("int4_code_offset", [("return bf16_val(bf16_round((double)(code - 8) * bf16_val(scale)));",
                           "return bf16_val(bf16_round((double)(code - 7) * bf16_val(scale)));")]),
    ("int4_dequant_unrounded", [("return bf16_val(bf16_round((double)(code - 8) * bf16_val(scale)));",
                                 "return (double)(code - 8) * bf16_val(scale);")]),
    ("int4_scale_row_major", [("return int4_dequant(code, m->gscale[(col / 128) * m->rows + row]);",
                               "return int4_dequant(code, m->gscale[row * (cols / 128) + col / 128]);")]),
    ("int4_scale_first_row", [("return int4_dequant(code, m->gscale[(col / 128) * m->rows + row]);",
                               "return int4_dequant(code, m->gscale[(col / 128) * m->rows]);")]),
    ("health_std_sample", [("h[0] = sqrt(var / (double)N);", "h[0] = sqrt(var / (double)(N - 1));")]),
    ("health_entropy_sign", [("ent -= p * log(p);", "ent += p * log(p);")]),
    ("gelu_grad_no_phi_term", [("return 0.5 * (1.0 + erf(v / sqrt(2.0))) + v * phi;",
                                "return 0.5 * (1.0 + erf(v / sqrt(2.0)));")]),
    ("softmax_jacobian_sign", [("dst[idx[(size_t)t * K + k]] += w[(size_t)t * K + k] * (dw_out[(size_t)t * K + k] - sdw);",
                                "dst[idx[(size_t)t * K + k]] += w[(size_t)t * K + k] * (sdw - dw_out[(size_t)t * K + k]);")]),
    ("aux_grad_not_centred", [("((double)demand[e] / TK - fp)", "((double)demand[e] / TK)")]),
    ("dW2_from_preactivation", [("dW2e[(size_t)c * f + j] += dO[c] * h[j];", "dW2e[(size_t)c * f + j] += dO[c] * a[j];")]),
    ("dx_without_shared_expert", [("double acc = dx_shared ? dx_shared[(size_t)t * d + i] : 0.0;", "double acc = 0.0;")]),
    ("dx_without_gate_term", [("acc += dst[e] * bf16_val(Wg[(size_t)e * d + i]);", "acc += 0.0 * dst[e];")]),
    ("z_grad_without_lse", [("+ g_z * 2.0 * beta / (double)T * lse * p;", "+ g_z * 2.0 * beta / (double)T * p;")]),
    ("dWg_from_wrong_row", [("dWg[(size_t)e * d + i] += g * bf16_val(x[(size_t)t * d + i]);",
                             "dWg[(size_t)e * d + i] += g * bf16_val(x[(size_t)e * d + i]);")]),
    ("health_drop_rate_inverted", [("h[1] = 1.0 - kept_all / TK;", "h[1] = kept_all / TK;")]),
    ("health_mean_weight_over_kept", [("mean_w[e] = demand[e] > 0 ? mean_w[e] / (double)demand[e] : 0.0;",
                                       "mean_w[e] = kept[e] > 0 ? mean_w[e] / (double)kept[e] : 0.0;")]),
    ("fp8_exponent_bias", [("v = ldexp(1.0 + (double)man / 8.0, ex - 7);", "v = ldexp(1.0 + (double)man / 8.0, ex - 8);")]),
    ("fp8_subnormal_as_normal", [("v = ldexp((double)man, -9);", "v = ldexp(1.0 + (double)man / 8.0, -7);")]),
    ("fp8_scale_first_row_only", [("* (double)m->scale[row];", "* (double)m->scale[0];")]),
    ("tie_break_flipped", [("return (a->e > b->e) - (a->e < b->e);",
                            "return (a->e < b->e) - (a->e > b->e);")]),
    ("weights_from_biased_logits", [("if (st[buf[k].e] > m)\n                m = st[buf[k].e];",
                                     "if (buf[k].u > m)\n                m = buf[k].u;"),
                                    ("z += exp(st[buf[k].e] - m);", "z += exp(buf[k].u - m);"),
                                    ("w[(size_t)t * K + k] = (float)(exp(st[buf[k].e] - m) / z);",
                                     "w[(size_t)t * K + k] = (float)(exp(buf[k].u - m) / z);")]),
    ("capacity_floor", [("double c = ceil(", "double c = floor(")]),
    ("capacity_off_by_one", [("if (p < C) {", "if (p <= C) {")]),
    ("gate_transposed", [("bf16_val(Wg[(size_t)e * d + j])", "bf16_val(Wg[(size_t)j * N + e])")]),
    ("bias1_dropped", [("acc += (double)b1e[j];", "acc += 0.0;")]),
    ("bias2_dropped", [("acc += (double)b2e[c];", "acc += 0.0;")]),
    ("gelu_sign", [("0.5 * v * (1.0 + erf(v / sqrt(2.0)))", "0.5 * v * (1.0 - erf(v / sqrt(2.0)))")]),
    ("hidden_not_rounded", [("h[j] = bf16_val(bf16_round(gelu_erf(acc)));", "h[j] = gelu_erf(acc);")]),
    ("w2_transposed", [("acc += h[j] * wval(W2e, (size_t)c, (size_t)j, (size_t)f);",
                        "acc += h[j] * wval(W2e, (size_t)j, (size_t)c, (size_t)d);")]),
    ("combine_weight_index", [("acc += (double)w[(size_t)t * K + k] *",
                               "acc += (double)w[(size_t)t * K + (K - 1 - k)] *")]),
    ("shared_not_added", [("double acc = z ? bf16_val(z[(size_t)t * d + c]) : 0.0;", "double acc = 0.0;")]),
    ("aux_f_over_T", [("acc += ((double)demand[e] / ((double)T * (double)K)) * P[e];",
                       "acc += ((double)demand[e] / ((double)T)) * P[e];")]),
    ("round_ties_away", [("nearbyint(ldexp(a, 7 - E))", "round(ldexp(a, 7 - E))")]),
    ("prob_not_normalised", [("P[e] += ex[e] / zn;", "P[e] += ex[e];")]),
    ("z_loss_not_squared", [("acc += lse * lse;", "acc += lse;")]),
    ("z_loss_no_max_shift", [("double lse = m + log(z);\n        acc += lse * lse;",
                              "double lse = log(z);\n        acc += lse * lse;")]),
    ("rank_major_ignored", [("const int outer = rank_major ? K : T, inner = rank_major ? T : K;",
                             "const int outer = T, inner = K; (void)rank_major;"),
                            ("const int t = rank_major ? b : a, k = rank_major ? a : b;",
                             "const int t = a, k = b;")]),
    ("kl_direction_swapped", [("acc += u * (log(u) - log(f));", "acc += f * (log(f) - log(u));")]),
    ("expert_backward_wrong_token", [("const uint16_t *xi = x + (size_t)tok[i] * d;",
                                      "const uint16_t *xi = x + (size_t)i * d;")]),
    ("expert_backward_bias_from_hidden", [("            bsum += g;\n            for (int j = 0; j < f; ++j)",
                                           "            bsum += g * hi[0];\n            for (int j = 0; j < f; ++j)")]),
    ("combine_backward_wrong_operand", [("dot += bf16_val(dy[(size_t)t * d + c]) * bf16_val(y_perm[(size_t)r * d + c]);",
                                         "dot += bf16_val(dy[(size_t)t * d + c]) * bf16_val(y_perm[(size_t)t * d + c]);")]),
    ("dispatch_priority_inverted", [("const int outer = rank_major ? K : T, inner = rank_major ? T : K;",
                                     "const int outer = rank_major ? T : K, inner = rank_major ? K : T;"),
                                    ("const int t = rank_major ? b : a, k = rank_major ? a : b;",
                                     "const int t = rank_major ? a : b, k = rank_major ? b : a;")]),
]


def _mutant(tmp_path, name, edits):
    with open(oracle.SOURCE) as fh:
        src = fh.read()
    for old, new in edits:
        assert src.count(old) == 1, f"{name}: mutation anchor not unique/absent: {old!r}"
        src = src.replace(old, new)
    path = os.path.join(tmp_path, f"{name}.c")
    with open(path, "w") as fh:
        fh.write(src)
    return oracle.Oracle(oracle.compile_source(path, os.path.join(tmp_path, f"lib{name}.so")))


@pytest.mark.parametrize("name,edits", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(tmp_path, name, edits):
    orc = _mutant(str(tmp_path), name, edits)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
