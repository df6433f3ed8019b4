"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

Each mutant is the oracle's C source with one textual change (a dropped term,
a wrong sign or index, a transposed operand, a flipped tie-break ...), compiled
on the CPU into a temporary library. The real oracle is never modified.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "silu_dropped": ("a[i] = silu(g) * u;", "a[i] = g * u;"),
    "gate_up_swapped": ("a[i] = silu(g) * u;", "a[i] = silu(u) * g;"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "w2_transposed": ("bf16_value(W2[h * I + i])", "bf16_value(W2[i * H + h])"),
    "up_rows_offset": ("W1[(I + i) * H + h]", "W1[(I + i - 1 + (i == 0)) * H + h]"),
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
