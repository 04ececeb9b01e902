"""Pins of the closed forms against the tables the pages print."""
import json
import os

import pytest

from oracle import closed_forms as cf


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_speedup_table_matches_page(golden_dir):
    g = _load(golden_dir, "speedup_tables.json")
    for row in g["speedup"]:
        for k in (3, 5, 7):
            assert round(cf.speedup(row["alpha"], row["c"], k), 2) == pytest.approx(row[f"k{k}"], abs=1e-9), (row, k)
        assert round(cf.speedup_bound(row["alpha"]), 2) == pytest.approx(row["bound"], abs=1e-9)


def test_tau_table_matches_page(golden_dir):
    g = _load(golden_dir, "speedup_tables.json")
    for row in g["tau"]:
        got = round(cf.speedup_tau(row["tau"], row["r"]), row["digits"])
        assert got == pytest.approx(row["speedup"], abs=1e-9), row


def test_expected_accepted_sum_equals_closed_form():
    # The page's sum form and its simplification (E[tokens] - 1) must agree.
    for alpha in (0.0, 0.1, 0.25, 0.5, 0.75, 0.9, 0.999):
        for k in range(0, 10):
            assert cf.expected_accepted(alpha, k) == pytest.approx(cf.expected_tokens_per_step(alpha, k) - 1.0,
                                                                   rel=1e-12, abs=1e-12)


def test_expected_tokens_limits():
    assert cf.expected_tokens_per_step(1.0, 5) == 6.0
    assert cf.expected_tokens_per_step(0.0, 5) == 1.0
    # bound 1/(1-alpha) is the k -> infinity limit
    assert cf.expected_tokens_per_step(0.75, 200) == pytest.approx(cf.speedup_bound(0.75), rel=1e-12)


def test_metrics_worked_example(golden_dir):
    g = _load(golden_dir, "metrics_example.json")
    proposed = g["verify_count"] * g["drafts_per_step"]
    assert cf.accept_rate(g["accepted"], proposed) == pytest.approx(g["accept_rate"])
    assert cf.accept_length(g["completion_tokens"], g["verify_count"]) == pytest.approx(g["accept_length"])
    # completion = accepted drafts + one bonus/recovered per verify
    assert g["completion_tokens"] == g["accepted"] + g["verify_count"]


def test_rollback_arithmetic(golden_dir):
    g = _load(golden_dir, "rollback.json")
    for c in g["cases"]:
        assert cf.tokens_advanced(c["num_accepted"]) == c["advance"]


def test_acceptance_counters_reproduce_metrics_example(golden_dir):
    """Ten verify steps of K=4 drafts with 25 accepted give alpha 0.625 and tau 3.5."""
    g = _load(golden_dir, "metrics_example.json")
    acc = [4, 4, 4, 3, 3, 2, 2, 2, 1, 0]
    assert sum(acc) == g["accepted"] and len(acc) == g["verify_count"]
    cu = [g["drafts_per_step"] * i for i in range(len(acc) + 1)]
    c = cf.acceptance_counters(cu, acc)
    alpha, tau = cf.rate_and_length(c)
    assert alpha == pytest.approx(g["accept_rate"]) and tau == pytest.approx(g["accept_length"])
    assert c[2] + c[3] == g["completion_tokens"]
    # per-position counts: position i is accepted in every request that accepted more than i drafts
    assert c[4:8] == [9, 8, 5, 3] and c[0] == 10


def test_acceptance_counters_skip_invalid_and_count_zero_draft_requests():
    # k = 0, 3, 2, 6; request 0 verifies without drafting, request 2 is invalid
    c = cf.acceptance_counters([0, 0, 3, 5, 11], [0, 2, -1, 4])
    assert c[:4] == [2, 9, 6, 3]
    assert c[4:9] == [2, 2, 1, 1, 0]
