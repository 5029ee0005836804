"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check
that the pins catch each one.  The committed oracle is never modified."""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sv_oracle.c")

# (name, text in sv_oracle.c, replacement, expected number of occurrences)
MUTANTS = [
    ("accept_le", "if (u[k] < o.accept_prob[k])", "if (u[k] <= o.accept_prob[k])", 1),
    ("residual_no_clamp", "w[i] = d > 0.0 ? d : 0.0;", "w[i] = d;", 1),
    ("ratio_inverted", "double a = px / qx;", "double a = qx / px;", 1),
    ("accept_no_min", "o.accept_prob[k] = a < 1.0 ? a : 1.0;", "o.accept_prob[k] = a;", 1),
    ("temperature_times", "/ T;", "* T;", 3),
    ("cdf_le", "if (t < C)", "if (t <= C)", 1),
    ("correction_uses_rejecting_draw", "inverse_cdf(w_scratch, V, u[K], &Z)",
     "inverse_cdf(w_scratch, V, u[jstar], &Z)", 1),
    ("bonus_row_off_by_one", "const double *prow = P + (int64_t)jstar * V;",
     "const double *prow = P + (int64_t)(jstar > 0 ? jstar - 1 : 0) * V;", 1),
    ("onehot_keeps_x", "double qi = onehot ? (i == x ? 1.0 : 0.0) : q[i];",
     "double qi = onehot ? 0.0 : q[i];", 1),
    ("row_stride_K", "(b * (K + 1) + j) * (int64_t)V, V, J->T,",
     "(b * K + j) * (int64_t)V, V, J->T,", 1),
    ("no_stop_at_rejection", "jstar = k;\n            break;", "jstar = k;", 1),
    ("unnormalised_p", "p[i] /= s;", "p[i] /= 1.0;", 1),
    ("bf16_shift", "(uint32_t)h << 16", "(uint32_t)h << 15", 1),
    ("residual_q_next_row",
     "rejected && Q ? Q + (int64_t)jstar * V : NULL",
     "rejected && Q ? Q + (int64_t)(jstar + 1 < K ? jstar + 1 : jstar) * V : NULL", 1),
    ("u_upper_inclusive", "u[k] < 1.0)", "u[k] <= 1.0)", 1),
    ("p_of_draft_from_next_row", "double px = P[(int64_t)k * V + tok[k]];",
     "double px = P[(int64_t)(k + 1) * V + tok[k]];", 1),
    # top-k / top-p filtering
    ("filter_ties_high_id", "return (x->id > y->id) - (x->id < y->id);\n}\n\n/* One row",
     "return (x->id < y->id) - (x->id > y->id);\n}\n\n/* One row", 1),
    ("filter_topp_of_total_mass", "top_p * cum[nk - 1]", "top_p * cum[n - 1]", 1),
    ("filter_drops_crossing_id", "    return r + 1;\n}", "    return r > 0 ? r : 1;\n}", 1),
    ("filter_reach_strict", "cum[r] < tau", "cum[r] <= tau", 1),
    ("filter_topk_one_more", "top_k < n) ? top_k : n", "top_k < n) ? top_k + 1 : n", 1),
    ("filter_mass_without_temperature", "acc += exp(rank[r].z / T - m);",
     "acc += exp(rank[r].z - m);", 1),
    # LM head and bf16 rounding
    ("lm_w_transposed", "W[col * d + k]", "W[k * d + col]", 1),
    ("lm_k_reversed", "h[row * d + k]", "h[row * d + (d - 1 - k)]", 1),
    ("bf16_round_truncates", "nearbyint(ldexp(m, 8))", "trunc(ldexp(m, 8))", 1),
    ("bf16_round_ties_away", "nearbyint(ldexp(m, 8))", "round(ldexp(m, 8))", 1),
    ("bf16_round_seven_bits", "nearbyint(ldexp(m, 8))", "nearbyint(ldexp(m, 7))", 1),
    # tree verification
    ("tree_accept_uses_p", "double a = r[tok[c]] / qv[tok[c]];", "double a = pv[tok[c]] / qv[tok[c]];", 1),
    ("tree_residual_unnormalised", "r[i] /= Z;", "r[i] /= 1.0;", 1),
    ("tree_final_from_p", "w[i] = r[i];", "w[i] = pv[i];", 1),
    ("tree_final_uniform_of_depth", "y = inverse_cdf(w, V, u[0], &Z);", "y = inverse_cdf(w, V, u[len], &Z);", 1),
    ("tree_siblings_reversed", "for (int32_t c = v + 1; c < N; ++c) {", "for (int32_t c = N - 1; c > v; --c) {", 1),
    ("tree_accept_le", "if (u[c] < a) {", "if (u[c] <= a) {", 1),
    ("tree_parent_may_equal_node", "parent[i] >= i)", "parent[i] > i)", 1),
    ("tree_residual_from_p", "double d = r[i] - qv[i];", "double d = pv[i] - qv[i];", 1),
    ("tree_child_row_for_test", "const double *qv = Q + (int64_t)v * V;",
     "const double *qv = Q + (int64_t)(v + 1 < N ? v + 1 : v) * V;", 1),
]


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new, count):
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) == count, f"mutation site for {name} not found"
    mutant_src = tmp_path / f"mut_{name}.c"
    mutant_src.write_text(src.replace(old, new), encoding="utf-8")
    lib = oracle.compile_oracle(str(mutant_src), str(tmp_path / f"lib_{name}.so"))
    mut = oracle.load(lib)
    caught = None
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mut)
        except Exception as exc:  # AssertionError or a refused call
            caught = (pin.__name__, type(exc).__name__)
            break
    assert caught is not None, f"no pin caught mutant {name}"
