"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

Each mutant is the oracle's C source with one textual change (a dropped term,
a wrong sign or index, a transposed operand, a flipped tie-break ...), compiled
on the CPU into a temporary library. The real oracle is never modified.
"""

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "silu_dropped": ("a[i] = silu(gi) * ui;", "a[i] = gi * ui;"),
    "gate_up_swapped": ("a[i] = silu(gi) * ui;", "a[i] = silu(ui) * gi;"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "w2_transposed": ("acc += bf16_value(W2[h * I + i]) * a[i];",
                      "acc += bf16_value(W2[i * H + h]) * a[i];"),
    "up_rows_offset": ("ui += bf16_value(W1[(I + i) * H + h]) * xt[h];",
                       "ui += bf16_value(W1[(I + i - 1 + (i == 0)) * H + h]) * xt[h];"),
    "combine_unweighted": ("yt[h] += w * o[h];", "yt[h] += o[h];"),
    "normalize_dropped": ("if (normalize) w_out[j] /= chosen_sum;", ";"),
    "scale_dropped": ("w_out[j] *= scale;", ";"),
    "tie_to_higher_index": ("if (best < 0 || v[i] > v[best]) best = i;",
                            "if (best < 0 || v[i] >= v[best]) best = i;"),
    "bias_in_weights": ("w_out[j] = s[b];\n        chosen_sum += s[b];",
                        "w_out[j] = sel[b];\n        chosen_sum += sel[b];"),
    "bias_ignored": ("sel[e] = s[e] + (sel_bias ? (double)sel_bias[e] : 0.0);", "sel[e] = s[e];"),
    "sigmoid_sign": ("s[e] = 1.0 / (1.0 + exp(-s[e]));", "s[e] = 1.0 / (1.0 + exp(s[e]));"),
    "softmax_sign": ("s[e] = exp(s[e] - m);", "s[e] = exp(m - s[e]);"),
    "offset_dropped": ("if (logit_offset) l += (double)logit_offset[e];", ";"),
    "group_top1": ("for (int32_t n = 0; n < group_topn && n < gs; ++n) {",
                   "for (int32_t n = 0; n < 1 && n < gs; ++n) {"),
    "group_limit_ignored": ("for (int64_t e = 0; e < E; ++e) ok[e] = kept[e / gs];", ";"),
    "aux_no_E": ("*aux = (double)E * a;", "*aux = a;"),
    "aux_f_without_k": ("(double)c / ((double)T * (double)k)", "(double)c / (double)T"),
    "perm_unstable": ("for (int64_t s = 0; s < R; ++s) {\n            if (topk_idx[s] != e) continue;",
                      "for (int64_t s = R - 1; s >= 0; --s) {\n            if (topk_idx[s] != e) continue;"),
    "dropped_slot_kept": ("if (e < 0 || e >= E) {\n                        if (a_slot)",
                          "if (e < 0 || e >= E) { e = (e < 0) ? 0 : E - 1; } if (0) {\n                        if (a_slot)"),
    "router_weight_transposed": ("bf16_value(x_t[h]) * (double)w_r[e * H + h]",
                                 "bf16_value(x_t[h]) * (double)w_r[h * E + e]"),
    # backward
    "bwd_dsilu_as_sigmoid": ("const double dsilu = sg * (1.0 + g[i] * (1.0 - sg));",
                             "const double dsilu = sg;"),
    "bwd_dU_without_silu": ("const double dU = dA[i] * silu(g[i]);",
                            "const double dU = dA[i] * g[i];"),
    "bwd_dA_w2_transposed": ("acc += bf16_value(W2[h * I + i]) * dO[h];",
                             "acc += bf16_value(W2[i * H + h]) * dO[h];"),
    "bwd_dO_unweighted": ("dO[h] = w * dyt[h];", "dO[h] = dyt[h];"),
    "bwd_dx_gate_up_swapped": (
        "bf16_value(W1[i * H + h]) * dG + bf16_value(W1[(I + i) * H + h]) * dU",
        "bf16_value(W1[i * H + h]) * dU + bf16_value(W1[(I + i) * H + h]) * dG"),
    "bwd_dw2_a_reversed": ("DW2[h * I + i] += d * a_s[slot * I + i];",
                           "DW2[h * I + i] += d * a_s[slot * I + (I - 1 - i)];"),
    "bwd_dw1_wrong_token": ("const int64_t t = slot / k;", "const int64_t t = slot % T;"),
    "bwd_dtopk_weighted": ("dwt += dyt[h] * o[h];", "dwt += w * dyt[h] * o[h];"),
    "rbwd_softmax_norm_no_scale": ("(w[j] / scale) * sum_wdw", "w[j] * sum_wdw"),
    "rbwd_sigmoid_deriv_dropped": ("si * (1.0 - si) / S", "si / S"),
    "rbwd_softmax_plain_cross_dropped": ("dlt[e] = -scale * s[e] * sum_sdw;", "dlt[e] = 0.0;"),
    "rbwd_sigmoid_plain_no_scale": ("dlt[K[j]] += scale * si * (1.0 - si) * dw[j];",
                                    "dlt[K[j]] += si * (1.0 - si) * dw[j];"),
    "rbwd_dx_wr_transposed": ("acc += dlt[e] * (double)w_r[e * H + h];",
                              "acc += dlt[e] * (double)w_r[h * E + e];"),
    # MXFP8
    "mx_emax_7": ("int e = (p - 1) - 8;", "int e = (p - 1) - 7;"),
    "mx_truncate": ("const double m = rint((ldexp(a, -p) - 1.0) * 8.0);",
                    "const double m = floor((ldexp(a, -p) - 1.0) * 8.0);"),
    "mx_subnormal_step": ("const double m = rint(a * 512.0);", "const double m = rint(a * 256.0);"),
    "mx_amax_first_only": ("if (fabs(v[i]) > amax) amax = fabs(v[i]);", "if (i == 0) amax = fabs(v[i]);"),
    "mx_dequant_unscaled": ("return e4m3_value(codes[r * cols + c]) * e8m0_value(scales[r * (cols / 32) + c / 32]);",
                            "return e4m3_value(codes[r * cols + c]);"),
    "mx_block_index_off": ("e8m0_value(scales[r * (cols / 32) + c / 32]);",
                           "e8m0_value(scales[r * (cols / 32) + (c / 32 + 1) % (cols / 32)]);"),
    "mx_a_not_requantized": ("for (int64_t i = 0; i < I; ++i) aq[i] = e4m3_value(ac[i]) * e8m0_value(as[i / 32]);",
                             "for (int64_t i = 0; i < I; ++i) aq[i] = a[i];"),
    "mx_overflow_to_nan": ("if (a >= 448.0) return sign | 0x7E;", "if (a >= 448.0) return sign | 0x7F;"),
    # MXFP8 backward
    "mxb_forward_x_unquantized": ("xq[h] = mx_value(x_codes, x_scales, H, t, h);",
                                  "xq[h] = bf16_value(x[t * H + h]);"),
    "mxb_wa_unweighted": ("for (int64_t i = 0; i < I; ++i) wa_s[slot * I + i] = w * a[i];",
                          "for (int64_t i = 0; i < I; ++i) wa_s[slot * I + i] = a[i];"),
    "mxb_wgrad_a_unquantized": ("for (int r = 0; r < 32; ++r) qa[r * M + m] = cq[r];",
                                "for (int r = 0; r < 32; ++r) qa[r * M + m] = col[r];"),
    "mxb_wgrad_b_unquantized": ("for (int r = 0; r < 32; ++r) qb[r * N + c] = cq[r];",
                                "for (int r = 0; r < 32; ++r) qb[r * N + c] = col[r];"),
    "mxb_dy_weighted": ("ady[r * H + h] = bf16_value(dy[tok * H + h]);",
                        "ady[r * H + h] = topk_w[slot] * bf16_value(dy[tok * H + h]);"),
    "mxb_dw1_x_wrong_token": ("ax[r * H + h] = bf16_value(x[tok * H + h]);",
                              "ax[r * H + h] = bf16_value(x[((tok + 1) % T) * H + h]);"),
    "mxb_blocks_of_16": ("const int64_t n = (end - b0 < 32) ? end - b0 : 32;",
                         "const int64_t n = (end - b0 < 16) ? end - b0 : 16;"),
    "mxb_gate_up_up": ("gacc += mx_value(w1_codes, w1_scales, H, w1_row + i, h) * xq[h];",
                       "gacc += mx_value(w1_codes, w1_scales, H, w1_row + I + i, h) * xq[h];"),
    "rbwd_dwr_wrong_token": ("acc += dl[t * E + e] * bf16_value(x[t * H + h]);",
                             "acc += dl[t * E + e] * bf16_value(x[((t + 1) % T) * H + h]);"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation anchor for {name} not unique in the oracle source"
    src = tmp_path / f"mutant_{name}.c"
    src.write_text(source.replace(old, new))
    lib = oracle.compile_source(str(src), str(tmp_path / f"mutant_{name}.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
        except (ValueError, IndexError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"
