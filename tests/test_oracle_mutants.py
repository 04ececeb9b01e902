"""Plausible mistakes planted in copies of the oracle must fail at least one pin.

This shows the pins are strong enough to trust the oracle: each mutant is the
real oracle source with one textual change (a wrong sign, swapped operands, a
wrong index or column, a dropped term, an off-by-one in the inverse CDF), built
into a temporary library and run through the same checks, on the CPU.
"""
import functools

import pytest

import oracle
import oracle_pins as P

MUTANTS = {
    "residual_sign": ("double diff = p[v] - (double)q[v];", "double diff = (double)q[v] - p[v];"),
    "accept_operands_swapped": ("const double lhs = us * qs, rhs = p[xs];", "const double lhs = us * p[xs], rhs = qs;"),
    "sampling_uses_coin_column": ("const double us = (double)uniforms[2 * t + 1];",
                                  "const double us = (double)uniforms[2 * t + 0];"),
    "output_row_off_by_one": ("const int64_t t = tb + j;", "const int64_t t = tb + (j > 0 ? j - 1 : 0);"),
    "one_hot_residual_keeps_draft": ("r[xs] = 0.0;", "r[xs] = r[xs];"),
    "inverse_cdf_non_strict": ("if (C > theta) {", "if (C >= theta) {"),
    "temperature_dropped": ("p[v] = (l >= cut) ? exp((l - m) / temp) : 0.0;", "p[v] = (l >= cut) ? exp((l - m)) : 0.0;"),
    "top_k_off_by_one": ("cut = sorted[F->top_k - 1];", "cut = sorted[F->top_k];"),
    "top_p_cut_one_token_late": ("                    if (sorted[i] > cut)\n                        cut = sorted[i];",
                                 "                    if (i + 1 < V && sorted[i + 1] > cut)\n                        cut = sorted[i + 1];"),
    "top_p_normalised_over_all_tokens": ("for (int32_t i = 0; i < V && sorted[i] >= cut; ++i)\n                Sk += ",
                                         "for (int32_t i = 0; i < V; ++i)\n                Sk += "),
    "greedy_emits_draft": ("token = row_argmax(&L, t);", "token = (j < k) ? draft_ids[db + j] : row_argmax(&L, t);"),
    "count_includes_recovered": ("out_num_accepted[req] = (int32_t)j;", "out_num_accepted[req] = (int32_t)j + 1;"),
    "bonus_not_sampled_from_p": ("} else {\n                    for (int32_t v = 0; v < V; ++v)\n                        r[v] = p[v];\n                }",
                                 "} else {\n                    for (int32_t v = 0; v < V; ++v)\n                        r[v] = p[v];\n                    r[draft_ids[db + j - 1 > 0 ? db + j - 1 : 0]] = 0.0;\n                }"),
    "greedy_tie_last_index": ("if (l > bv) {", "if (l >= bv) {"),
    "degenerate_residual_ignored": ("if (Z > 0.0) {", "if (1) {"),
    # the near-boundary report that excuses GPU mismatches
    "sampling_margin_one_side_only": ("*margin = a < b ? a : b;", "*margin = b;"),
    "acceptance_margin_unscaled": ("if (big > 0.0 && fabs(lhs - rhs) / big < margin_accept)\n                    margin_accept = fabs(lhs - rhs) / big;",
                                   "if (big > 0.0 && fabs(lhs - rhs) < margin_accept)\n                    margin_accept = fabs(lhs - rhs);"),
}

# smaller statistical checks keep the mutant run short
FAST_CHECKS = [
    functools.partial(P.check_output_distribution, N=200_000),
    functools.partial(P.check_acceptance_rate, N=100_000),
    P.check_residual_mass,
    functools.partial(P.check_accepted_length, N=100_000),
    P.check_exact_enumeration, P.check_q_equals_p, P.check_disjoint_supports, P.check_one_hot_draft,
    P.check_greedy_worked_chain, P.check_rollback_arithmetic, P.check_greedy_ties_and_bonus, P.check_zero_drafts,
    P.check_extreme_uniforms, P.check_row_statistics, P.check_invalid_inputs, P.check_degenerate_residual,
    P.check_top_k_top_p, P.check_margins_and_flags,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / f"mutant_{name}.c"
    path.write_text(src.replace(old, new))
    impl = oracle.Oracle(oracle.build(force=True, src=str(path), out=str(tmp_path / f"mutant_{name}.so")))
    failures = []
    for check in FAST_CHECKS:
        try:
            ok, msg = check(impl=impl)
        except Exception as e:  # a crash in a check also counts as detection
            ok, msg = False, f"raised {type(e).__name__}: {e}"
        if not ok:
            failures.append(msg)
            break
    assert failures, f"mutant {name} passed every pin"
