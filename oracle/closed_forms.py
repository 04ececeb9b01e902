"""Closed forms of speculative decoding that the pages state, in plain Python.

TEST INFRASTRUCTURE (and benchmark-report context).  These are pinned against the
tables the pages print (``tests/golden/speedup_tables.json``) and used as
expected values by the oracle's statistical tests.
"""
from __future__ import annotations


def expected_tokens_per_step(alpha: float, k: int) -> float:
    """E[tokens per step] = (1 - alpha^(k+1)) / (1 - alpha) under i.i.d. acceptance alpha.

    "第12章 投机解码：以小博大" §12.5.1: the accepted drafts plus the one bonus or
    recovered token.  At alpha = 1 the limit is k + 1.
    """
    if alpha == 1.0:
        return float(k + 1)
    return (1.0 - alpha ** (k + 1)) / (1.0 - alpha)


def expected_accepted(alpha: float, k: int) -> float:
    """E[accepted drafts] = sum_{i<k} alpha^i (1 - alpha) i + alpha^k k  ("以小博大" §12.5.1).

    Written as the page's sum, not its simplification, so that the test that
    compares it with ``expected_tokens_per_step - 1`` checks the algebra.
    """
    return sum(alpha ** i * (1.0 - alpha) * i for i in range(k)) + alpha ** k * k


def speedup(alpha: float, c: float, k: int) -> float:
    """(1 - alpha^(k+1)) / ((1 - alpha)(1 + c k)): "以小博大" §12.5.3 (Leviathan et al. Thm 3.8)."""
    return expected_tokens_per_step(alpha, k) / (1.0 + c * k)


def speedup_bound(alpha: float) -> float:
    """Upper bound 1 / (1 - alpha), the c = 0, k -> infinity limit ("以小博大" §12.5.4)."""
    return 1.0 / (1.0 - alpha)


def speedup_tau(tau: float, r: float) -> float:
    """tau / (1 + r): accept length over relative draft cost ("投机解码端到端深挖" §1.3)."""
    return tau / (1.0 + r)


def accept_rate(num_accepted: int, num_proposed: int) -> float:
    """spec_accept_rate alpha = correct drafts / proposed drafts, bonus excluded ("投机解码端到端深挖" §13)."""
    return num_accepted / num_proposed


def accept_length(completion_tokens: int, verify_count: int) -> float:
    """spec_accept_length tau = completion tokens / verify count, bonus included ("投机解码端到端深挖" §13)."""
    return completion_tokens / verify_count


def tokens_advanced(num_accepted: int) -> int:
    """Position advance of one step: accepted drafts + 1 ("以小博大" §12.3.4; "投机解码端到端深挖" §8.1)."""
    return num_accepted + 1


def acceptance_counters(cu_num_draft, num_accepted, max_spec_len: int = 32) -> list[int]:
    """Acceptance counters of one batch, by plain loops.

    [0] requests that drafted at least one token (vLLM spec_decode_num_drafts),
    [1] draft tokens proposed (num_draft_tokens), [2] drafts accepted (num_accepted_tokens),
    [3] verify steps (one per request), [4 + i] requests whose draft at position i was
    accepted (num_accepted_tokens_per_pos).  "第12章 投机解码：以小博大" §12.7.5 names the
    counters; "投机解码端到端深挖" §13 defines alpha and tau from them.  Requests reported
    invalid (accepted = -1) are skipped.
    """
    c = [0] * (4 + max_spec_len)
    for r in range(len(num_accepted)):
        a = int(num_accepted[r])
        if a < 0:
            continue
        k = int(cu_num_draft[r + 1]) - int(cu_num_draft[r])
        c[0] += 1 if k > 0 else 0
        c[1] += k
        c[2] += a
        c[3] += 1
        for i in range(min(a, max_spec_len)):
            c[4 + i] += 1
    return c


def rate_and_length(counters) -> tuple[float, float]:
    """alpha = accepted / proposed; tau = (accepted + verifies) / verifies (the bonus counts in tau)."""
    return accept_rate(counters[2], counters[1]), accept_length(counters[2] + counters[3], counters[3])
