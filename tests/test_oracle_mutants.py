"""The pins must catch plausible mistakes in the oracle.

Each mutant is a copy of the oracle's C source with one planted mistake (a sign,
a dropped term, a wrong index, a transposed operand, an off-by-one), built with
gcc into a temporary directory.  Every mutant must fail at least one pin.  The
mistakes are planted only in these temporary copies, on the CPU.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

MUTANTS = {
    "softmax_sign": ("pt[e] = exp(l[e] - m) / s;", "pt[e] = exp(m - l[e]) / s;"),
    "lse_drops_max": ("lse[t] = m + log(s);", "lse[t] = log(s);"),
    "tie_to_higher_index": ("return (a->e < b->e) ? -1 : (a->e > b->e);",
                            "return (a->e > b->e) ? -1 : (a->e < b->e);"),
    "no_renormalise": ("gates[(size_t)t * k + s2] = pt[it[s2]] / denom;",
                       "gates[(size_t)t * k + s2] = pt[it[s2]];"),
    "bias_ignored": ("ord[e].key = pt[e] + (sel_bias ? (double)sel_bias[e] : 0.0);",
                     "ord[e].key = pt[e];"),
    "gap_wrong_index": ("ord[k - 1].key - ord[k].key", "ord[0].key - ord[k].key"),
    "offset_dropped": ("if (offset) acc += (double)offset[e];", "(void)offset;"),
    "capacity_floor": ("return (int64_t)ceil(", "return (int64_t)floor("),
    "capacity_without_k": ("ceil(c * (double)k * (double)T", "ceil(c * (double)T"),
    "capacity_off_by_one": ("kept_counts[e] < C", "kept_counts[e] <= C"),
    "offsets_from_precap_counts": ("offsets[e + 1] = offsets[e] + kept_counts[e];",
                                   "offsets[e + 1] = offsets[e] + counts[e];"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "gate_up_swapped": ("h[j] = silu(a) * b;", "h[j] = a * silu(b);"),
    "w2_transposed": ("bf16_val(w2[(size_t)o * Mw + j])", "bf16_val(w2[(size_t)j * d + o])"),
    "dropped_pairs_added": ("if (dropped[pq]) continue;", "if (0) continue;"),
    "shared_not_added": ("x + t * d, ws1, ws3, ws2, tmp);\n                for (int o = 0; o < d; ++o) yt[o] += tmp[o];",
                         "x + t * d, ws1, ws3, ws2, tmp);\n                for (int o = 0; o < d; ++o) yt[o] += 0.0 * tmp[o];"),
    "priority_offsets_precap": ("offsets[e + 1] = kept_counts[e] + offsets[e];",
                                "offsets[e + 1] = counts[e] + offsets[e];"),
    "zloss_not_squared": ("sz += lse[t] * lse[t];", "sz += lse[t];"),
    "f_over_T": ("oracle_losses_n(T, E, (double)k * (double)T,", "oracle_losses_n(T, E, (double)T,"),
    "balance_without_E": ("*L_bal = lambda * (double)E * sfp;", "*L_bal = lambda * sfp;"),
    "sigmoid_sign": ("pt[e] = 1.0 / (1.0 + exp(-l[e]));", "pt[e] = 1.0 / (1.0 + exp(l[e]));"),
    "no_renorm_ignored": ("if (flags & ORACLE_NO_RENORM) denom = 1.0;", "(void)0;"),
    "entropy_sign": ("if (q > 0.0) h -= q * log(q);", "if (q > 0.0) h += q * log(q);"),
    "importance_sample_variance": ("    var /= (double)E;", "    var /= (double)(E - 1);"),
    "alf_sign": ("const double diff = nbar - (double)counts[e];",
                 "const double diff = (double)counts[e] - nbar;"),
    "combine_drop_ignored": ("if (r < 0) continue;\n            double g", "if (r < 0) r = 0;\n            double g"),
    "priority_keeps_lowest": ("if (a->key > b->key) return -1;\n    if (a->key < b->key) return 1;\n    return (a->q",
                              "if (a->key < b->key) return -1;\n    if (a->key > b->key) return 1;\n    return (a->q"),
    "priority_ties_reversed": ("return (a->q < b->q) ? -1 : (a->q > b->q);",
                               "return (a->q > b->q) ? -1 : (a->q < b->q);"),
    "priority_wrong_score": ("list[m].key = p[(q / k) * (int64_t)E + e];",
                             "list[m].key = p[(q % k) * (int64_t)E + e];"),
    "priority_cut_off_by_one": ("for (int64_t j = C; j < m; ++j) dropped[list[j].q] = 1;",
                                "for (int64_t j = C + 1; j < m; ++j) dropped[list[j].q] = 1;"),
    "ec_rows_unsorted": ("qsort(rt, (size_t)r, sizeof(int32_t), i32_cmp);", "(void)i32_cmp;"),
    "ec_gate_transposed": ("row_gate[(size_t)e * r + j] = p[(size_t)rt[j] * E + e];",
                           "row_gate[(size_t)e * r + j] = p[(size_t)e * E + rt[j] % E];"),
    "ec_capacity_no_cap": ("return r < T ? r : T;", "return r;"),
    "ec_default_c": ("double cc = (c > 0.0) ? c : 1.0;", "double cc = c;"),
    "ec_shared_missing": ("oracle_swiglu_row(d, Ms, x + (size_t)t * d, ws1, ws3, ws2, tmp);\n                for (int o = 0; o < d; ++o) yt[o] += tmp[o];",
                          "oracle_swiglu_row(d, Ms, x + (size_t)t * d, ws1, ws3, ws2, tmp);\n                for (int o = 0; o < d; ++o) yt[o] += 0.0;"),
    "expert_rows_all_expert0": ("        size_t e = (size_t)expert[r];\n",
                                "        size_t e = 0; (void)expert;\n"),
    "expert_rows_w2_stride": ("w3 + e * M * d,\n                          w2 + e * d * M, out",
                              "w3 + e * M * d,\n                          w2 + e * d * d, out"),
    "expert_rows_w3_from_w1": ("x_rows + (size_t)r * d, w1 + e * M * d, w3 + e * M * d,",
                               "x_rows + (size_t)r * d, w1 + e * M * d, w1 + e * M * d,"),
    "combine_shared_missing": ("yt[o] += bf16_val(y_shared[(size_t)t * d + o]);", "yt[o] += 0.0;"),
    "router_wr_transposed": ("acc += bf16_val(wr[(size_t)e * d + i]) * bf16_val(x[(size_t)t * d + i]);",
                             "acc += bf16_val(wr[(size_t)i * E + e]) * bf16_val(x[(size_t)t * d + i]);"),
    "dispatch_rows_reversed": ("int r = offsets[e] + rank[q];", "int r = offsets[e + 1] - 1 - rank[q];"),
    "combine_gate_of_slot0": ("double g = gates[(size_t)t * k + s];", "double g = gates[(size_t)t * k];"),
    "P_over_E": ("P[e] = (T > 0) ? acc / (double)T : 0.0;", "P[e] = (T > 0) ? acc / (double)E : 0.0;"),
    "counts_after_capacity": ("            counts[e] += 1;\n            if (C < 0 || kept_counts[e] < C) {",
                              "            counts[e] += (C < 0 || kept_counts[e] < C);\n            if (C < 0 || kept_counts[e] < C) {"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/found"
    msrc = tmp_path / "moe_oracle_mut.c"
    msrc.write_text(src.replace(old, new))
    lib_path = str(tmp_path / "libmut.so")
    oracle.build(str(msrc), lib_path)
    lib = oracle.load(lib_path)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
