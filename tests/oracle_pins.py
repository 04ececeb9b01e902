"""Checks that pin the CPU oracle to what the pages and the mathematics fix.

Each check returns ``(ok, message)`` and takes the oracle build to run (``impl``),
so that ``test_oracle_pins.py`` asserts them on the real oracle and
``test_oracle_mutants.py`` shows that copies of the oracle with planted mistakes
fail at least one of them.  None of the checks re-types the oracle's formulas:
they compare its outputs with the exactness theorem (output distribution = p),
with A = sum min(p, q), with library routines (scipy softmax / logsumexp, numpy
argmax / cumsum / searchsorted), with exact enumeration of outcomes, or with the
pages' worked examples.
"""
from __future__ import annotations

import itertools
import json
import os

import numpy as np
from scipy import special, stats

import oracle
from oracle import closed_forms as cf

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Dyadic draft distributions: exact in float32 and summing to exactly 1, so the
# exactness identity holds to 1e-12 (it needs sum q = sum p).
Q4 = [np.array([0.5, 0.25, 0.125, 0.125]), np.array([0.125, 0.125, 0.25, 0.5]), np.array([0.25, 0.5, 0.0, 0.25])]
Q8 = np.array([0.25, 0.125, 0.125, 0.0625, 0.0625, 0.125, 0.1875, 0.0625])


def _p_from_logits(l32: np.ndarray, temp: float) -> np.ndarray:
    """Target distribution the oracle should use, by a library routine."""
    return special.softmax(l32.astype(np.float64) / np.float64(np.float32(temp)), axis=-1)


def _iid_batch(N, K, l_row, temp, q_row, draw_q, seed):
    """N i.i.d. requests of K drafts sharing one target row and one draft row (stride-0 views)."""
    rng = np.random.default_rng(seed)
    V = l_row.shape[0]
    ids = rng.choice(V, size=N * K, p=draw_q).astype(np.int32)
    u = rng.random((N * (K + 1), 2), dtype=np.float32)
    cu = (np.arange(N + 1) * K).astype(np.int32)
    temps = np.full(N, temp, np.float32)
    return ids, u, cu, temps


def _run_iid(impl, N, K, l_row, temp, q_row, draw_q, seed):
    ids, u, cu, temps = _iid_batch(N, K, l_row, temp, q_row, draw_q, seed)
    V = l_row.shape[0]
    res = oracle.reject_sample(l_row, ids, cu, u, temps, q_row, logits_row_stride=0,
                               q_row_stride=None if q_row is None else 0, vocab=V, num_rows=N * (K + 1), impl=impl)
    return res


def check_output_distribution(impl=None, N=1_000_000, cases=None):
    """(a) Every emitted position's token is distributed as p (chi-square, Bonferroni over all tests)."""
    cases = cases or [(1, True, 1.0), (3, True, 0.7), (3, False, 1.0), (3, True, 1.3)]
    base = np.array([0.4, -0.3, 1.2, 0.1, -1.0, 0.6, 0.0, -0.5], dtype=np.float32)
    ntests = sum(K + 1 for K, _, _ in cases)
    for ci, (K, explicit, temp) in enumerate(cases):
        l = (base * np.float32(1.7)).astype(np.float32)
        p = _p_from_logits(l, temp)
        q = Q8.astype(np.float32)
        res = _run_iid(impl, N, K, l, temp, q if explicit else None, Q8, seed=100 + ci)
        tok = res.tokens.reshape(N, K + 1)
        acc = res.num_accepted
        for m in range(K + 1):
            sel = acc >= m
            obs = np.bincount(tok[sel, m], minlength=8)
            if obs.shape[0] != 8 or (tok[sel, m] < 0).any():
                return False, f"case {ci} pos {m}: token out of range"
            pval = stats.chisquare(obs, p * sel.sum()).pvalue
            if not pval > 1e-4 / ntests:
                return False, f"case {ci} (K={K}, explicit={explicit}, T={temp}) pos {m}: chi-square p={pval:.3g}"
    return True, "ok"


def check_acceptance_rate(impl=None, N=400_000):
    """(b) Per-position acceptance rate equals A = sum min(p, q) (explicit q) or sum q_draw p (one-hot q)."""
    l = np.array([0.9, -0.4, 0.3, 0.2, -1.2, 0.5, 0.1, -0.2], dtype=np.float32)
    for ci, (explicit, temp) in enumerate([(True, 1.0), (True, 0.6), (False, 1.0)]):
        p = _p_from_logits(l, temp)
        A = np.minimum(p, Q8).sum() if explicit else (Q8 * p).sum()
        K = 3
        res = _run_iid(impl, N, K, l, temp, Q8.astype(np.float32) if explicit else None, Q8, seed=200 + ci)
        acc = res.num_accepted
        for m in range(K):
            reached = (acc >= m).sum()
            rate = (acc >= m + 1).sum() / reached
            sig = np.sqrt(A * (1 - A) / reached)
            if abs(rate - A) > 5 * sig:
                return False, f"case {ci} pos {m}: acceptance {rate:.5f} vs A={A:.5f} (5 sigma {5 * sig:.5f})"
    return True, "ok"


def check_residual_mass(impl=None):
    """(c) At a rejection the residual mass Z = sum max(0, p - q) equals 1 - A to 1e-12."""
    rng = np.random.default_rng(300)
    for V in (2, 5, 8, 100, 1000):
        for trial in range(5):
            # dyadic q with sum exactly 1: integer weights over a power of two
            w = rng.integers(0, 64, size=V).astype(np.float64)
            w[rng.integers(0, V)] += 1
            tot = 2 ** int(np.ceil(np.log2(w.sum())))
            w[np.argmax(w)] += tot - w.sum()
            q = (w / tot).astype(np.float32)
            l = (rng.standard_normal(V) * 1.5).astype(np.float32)
            temp = float(rng.choice([0.5, 1.0, 1.7]))
            p = _p_from_logits(l, temp)
            over = np.nonzero(q.astype(np.float64) > p * 1.01)[0]
            if over.size == 0:
                continue
            x = int(over[0])
            res = oracle.reject_sample(l[None, :], np.array([x], np.int32), np.array([0, 1], np.int32),
                                       np.array([[0.999999, 0.5], [0.5, 0.5]], np.float32),
                                       np.array([temp], np.float32), q[None, :], logits_row_stride=0, vocab=V,
                                       num_rows=2, debug=True, impl=impl)
            if res.num_accepted[0] != 0:
                return False, f"V={V}: draft with q > p/0.999999 was accepted"
            A = np.minimum(p, q.astype(np.float64)).sum()
            if abs(res.z[0] - (1.0 - A)) > 1e-12:
                return False, f"V={V}: Z={res.z[0]!r} vs 1-A={1 - A!r}"
    return True, "ok"


def check_accepted_length(impl=None, N=400_000):
    """(d) Mean tokens per step matches (1 - a^(K+1)) / (1 - a) under i.i.d. acceptance a = A."""
    l = np.array([0.2, 0.1, 0.8, -0.3, 0.4, -0.6, 0.9, 0.0], dtype=np.float32)
    for ci, (K, temp) in enumerate([(1, 1.0), (3, 0.9), (5, 1.0), (8, 1.2)]):
        p = _p_from_logits(l, temp)
        A = np.minimum(p, Q8).sum()
        res = _run_iid(impl, N, K, l, temp, Q8.astype(np.float32), Q8, seed=400 + ci)
        steps = res.num_accepted.astype(np.float64) + 1
        want = cf.expected_tokens_per_step(A, K)
        sig = steps.std() / np.sqrt(N)
        if abs(steps.mean() - want) > 5 * sig:
            return False, f"K={K}: mean {steps.mean():.5f} vs closed form {want:.5f} (5 sigma {5 * sig:.5f})"
        emitted = (res.tokens.reshape(N, K + 1) >= 0).sum(axis=1)
        if not np.array_equal(emitted, res.num_accepted + 1):
            return False, f"K={K}: emitted tokens != accepted + 1"
    return True, "ok"


def _enumerate(impl, K, V, ls, temp, qs, explicit):
    """Exact outcome probabilities of one step with position-dependent p_i, q_i (V <= 4, K <= 2).

    The test computes the cells of the uniforms (accept / reject interval of each
    coin, residual CDF intervals of the sampling draw) from p and q, queries the
    oracle at every cell's midpoint, and weights the oracle's emitted sequence by
    the cell's probability.  Returns {emitted tuple: probability}.
    """
    ps = [_p_from_logits(li, temp) for li in ls]
    leaves = []  # (draft seq, uniforms [(K+1), 2], weight)
    for xs in itertools.product(range(V), repeat=K):
        wx = np.prod([qs[i][x] for i, x in enumerate(xs)])
        if wx == 0:
            continue
        # position j = first rejection (K = all accepted)
        for j in range(K + 1):
            w = wx
            coins = []
            ok = True
            for i in range(min(j + 1, K)):
                x = xs[i]
                a = min(1.0, ps[i][x] / qs[i][x]) if explicit else ps[i][x]
                if i < j:
                    coins.append(a / 2)
                    w *= a
                else:
                    coins.append((a + 1) / 2)
                    w *= 1 - a
                if w == 0:
                    ok = False
                    break
            if not ok:
                continue
            if j < K:
                if explicit:
                    r = np.maximum(0.0, ps[j] - qs[j])
                else:
                    r = ps[j].copy()
                    r[xs[j]] = 0.0
            else:
                r = ps[K]
            Z = r.sum()
            C = np.cumsum(r) / Z
            for v in range(V):
                if r[v] <= 0:
                    continue
                lo = C[v - 1] if v > 0 else 0.0
                u = np.zeros((K + 1, 2), np.float32)
                u[: len(coins), 0] = coins
                u[:, 1] = 0.5
                u[j, 1] = (lo + C[v]) / 2
                leaves.append((xs, u, w * (r[v] / Z)))
    n = len(leaves)
    logits = np.stack([np.stack(ls) for _ in range(n)]).reshape(n * (K + 1), V).astype(np.float32)
    ids = np.array([lf[0] for lf in leaves], np.int32).reshape(-1)
    u = np.concatenate([lf[1] for lf in leaves])
    cu = (np.arange(n + 1) * K).astype(np.int32)
    q = None
    if explicit:
        q = np.stack([np.stack(qs) for _ in range(n)]).reshape(n * K, V).astype(np.float32)
    res = oracle.reject_sample(logits, ids, cu, u, np.full(n, temp, np.float32), q, impl=impl)
    tok = res.tokens.reshape(n, K + 1)
    probs = {}
    for i, lf in enumerate(leaves):
        j = int(res.num_accepted[i])
        if j < 0 or j > K:
            return None, ps
        seq = tuple(int(t) for t in tok[i, : j + 1])
        probs[seq] = probs.get(seq, 0.0) + lf[2]
    return probs, ps


def check_exact_enumeration(impl=None):
    """(e) Step output followed by fresh draws from p is exactly an independent p-sequence (to 1e-12)."""
    V, K = 4, 2
    ls = [np.array([0.3, -0.2, 1.1, 0.05], np.float32), np.array([-0.5, 0.7, 0.2, 0.4], np.float32),
          np.array([1.0, 0.1, -0.3, 0.6], np.float32)]
    for explicit in (True, False):
        for temp in (1.0, 0.8):
            probs, ps = _enumerate(impl, K, V, ls, temp, [Q4[0], Q4[1]], explicit)
            if probs is None:
                return False, "accepted count out of range"
            total = sum(probs.values())
            if abs(total - 1.0) > 1e-12:
                return False, f"explicit={explicit} T={temp}: outcome probabilities sum to {total!r}"
            for y in itertools.product(range(V), repeat=K + 1):
                lhs = 0.0
                for m in range(1, K + 2):
                    pm = probs.get(tuple(y[:m]), 0.0)
                    lhs += pm * np.prod([ps[i][y[i]] for i in range(m, K + 1)])
                rhs = np.prod([ps[i][y[i]] for i in range(K + 1)])
                if abs(lhs - rhs) > 1e-12:
                    return False, f"explicit={explicit} T={temp} y={y}: {lhs!r} != {rhs!r}"
    return True, "ok"


def check_q_equals_p(impl=None):
    """q = p: every draft is accepted and the bonus is numpy's inverse CDF of p."""
    rng = np.random.default_rng(500)
    B, K, V, temp = 64, 4, 1000, 0.9
    l = (rng.standard_normal((B * (K + 1), V)) * 2).astype(np.float32)
    p = _p_from_logits(l, temp)
    q = p.reshape(B, K + 1, V)[:, :K].reshape(B * K, V).astype(np.float32)
    ids = np.array([rng.choice(V, p=qq / qq.sum()) for qq in q.astype(np.float64)], np.int32)
    u = rng.random((B * (K + 1), 2), dtype=np.float32)
    u[:, 0] *= np.float32(0.999)
    cu = (np.arange(B + 1) * K).astype(np.int32)
    res = oracle.reject_sample(l, ids, cu, u, np.full(B, temp, np.float32), q, impl=impl)
    if not (res.num_accepted == K).all():
        return False, "q = p but a draft was rejected"
    tok = res.tokens.reshape(B, K + 1)
    if not np.array_equal(tok[:, :K].reshape(-1), ids):
        return False, "accepted drafts not emitted in order"
    for b in range(B):
        row = b * (K + 1) + K
        c = np.cumsum(p[row])
        want = int(np.searchsorted(c, float(u[row, 1]) * c[-1], side="right"))
        if tok[b, K] != want and not (res.flags[b] & oracle.NEAR_SAMPLE):
            return False, f"request {b}: bonus {tok[b, K]} != searchsorted {want}"
    return True, "ok"


def check_disjoint_supports(impl=None):
    """Disjoint supports: every draft is rejected and the recovered token is numpy's inverse CDF of p."""
    rng = np.random.default_rng(600)
    B, K, V, temp = 64, 3, 512, 1.1
    l = (rng.standard_normal((B * (K + 1), V)) * 2).astype(np.float32)
    l[:, 1::2] = -np.inf  # p lives on even tokens
    qw = rng.random((B * K, V))
    qw[:, 0::2] = 0.0  # q lives on odd tokens
    q = (qw / qw.sum(axis=1, keepdims=True)).astype(np.float32)
    ids = np.array([rng.choice(V, p=qq / qq.sum()) for qq in q.astype(np.float64)], np.int32)
    u = rng.random((B * (K + 1), 2), dtype=np.float32)
    cu = (np.arange(B + 1) * K).astype(np.int32)
    res = oracle.reject_sample(l, ids, cu, u, np.full(B, temp, np.float32), q, impl=impl)
    if not (res.num_accepted == 0).all():
        return False, "disjoint supports but a draft was accepted"
    tok = res.tokens.reshape(B, K + 1)
    for b in range(B):
        row = b * (K + 1)
        c = np.cumsum(_p_from_logits(l[row], temp))
        want = int(np.searchsorted(c, float(u[row, 1]) * c[-1], side="right"))
        if tok[b, 0] != want and not (res.flags[b] & oracle.NEAR_SAMPLE):
            return False, f"request {b}: recovered {tok[b, 0]} != {want}"
        if (tok[b, 1:] != -1).any():
            return False, f"request {b}: rows after the rejection not padded with -1"
    return True, "ok"


def check_one_hot_draft(impl=None):
    """One-hot q: accept iff u < p(x*); on rejection the recovered token is the inverse CDF of p with x* removed."""
    rng = np.random.default_rng(700)
    B, K, V, temp = 200, 1, 64, 1.0
    l = (rng.standard_normal((B * (K + 1), V)) * 1.0).astype(np.float32)
    p = _p_from_logits(l, temp)
    ids = np.array([rng.choice(V, p=p[b * 2]) if b % 2 else rng.integers(0, V) for b in range(B)], np.int32)
    u = rng.random((B * (K + 1), 2), dtype=np.float32)
    cu = (np.arange(B + 1) * K).astype(np.int32)
    res = oracle.reject_sample(l, ids, cu, u, np.full(B, temp, np.float32), None, impl=impl)
    for b in range(B):
        row = b * 2
        x = ids[b]
        ps = p[row][x]
        if abs(float(u[row, 0]) - ps) < 1e-9:
            continue
        accepted = float(u[row, 0]) < ps
        if accepted != (res.num_accepted[b] == 1):
            return False, f"request {b}: u={u[row, 0]} p(x*)={ps} accepted={res.num_accepted[b]}"
        if not accepted:
            r = p[row].copy()
            r[x] = 0.0
            c = np.cumsum(r)
            want = int(np.searchsorted(c, float(u[row, 1]) * c[-1], side="right"))
            if res.tokens[row] != want and not (res.flags[b] & oracle.NEAR_SAMPLE):
                return False, f"request {b}: recovered {res.tokens[row]} != {want}"
    return True, "ok"


def _greedy_rows(argmaxes, V, rng):
    rows = (rng.standard_normal((len(argmaxes), V))).astype(np.float32)
    for i, a in enumerate(argmaxes):
        rows[i, a] = rows[i].max() + 1.0
    return rows


def check_greedy_worked_chain(impl=None):
    """The pages' chain example: drafts A,B,C vs target argmax A,B,X -> emit A,B,X; 2 correct, accept_lens 3."""
    with open(os.path.join(GOLDEN, "greedy_chain.json")) as f:
        g = json.load(f)
    V = g["vocab"]
    rng = np.random.default_rng(800)
    l = _greedy_rows(g["target_argmax"], V, rng)
    K = len(g["drafts"])
    for temp in (0.0, -1.0):
        res = oracle.reject_sample(l, np.array(g["drafts"], np.int32), np.array([0, K], np.int32),
                                   rng.random((K + 1, 2), dtype=np.float32), np.array([temp], np.float32),
                                   None, impl=impl)
        if res.tokens.tolist() != g["expected_tokens"]:
            return False, f"T={temp}: tokens {res.tokens.tolist()} != {g['expected_tokens']}"
        if res.num_accepted[0] != g["expected_num_accepted"]:
            return False, f"num_accepted {res.num_accepted[0]}"
        if int((res.tokens >= 0).sum()) != g["expected_accept_lens"]:
            return False, "accept_lens"
    return True, "ok"


def check_rollback_arithmetic(impl=None):
    """k=5 with 5 / 3 / 0 matching drafts advances 6 / 4 / 1 positions (accepted + 1)."""
    with open(os.path.join(GOLDEN, "rollback.json")) as f:
        g = json.load(f)
    K, V = g["k"], 32
    rng = np.random.default_rng(900)
    for c in g["cases"]:
        am = rng.integers(0, V, size=K + 1)
        l = _greedy_rows(am, V, rng)
        drafts = am[:K].copy()
        n = c["num_accepted"]
        if n < K:
            drafts[n] = (am[n] + 1) % V
        res = oracle.reject_sample(l, drafts.astype(np.int32), np.array([0, K], np.int32),
                                   rng.random((K + 1, 2), dtype=np.float32), np.array([0.0], np.float32), None,
                                   impl=impl)
        if res.num_accepted[0] != n or int((res.tokens >= 0).sum()) != c["advance"]:
            return False, f"case {c}: accepted {res.num_accepted[0]}, emitted {(res.tokens >= 0).sum()}"
    return True, "ok"


def check_greedy_ties_and_bonus(impl=None):
    """Greedy: ties go to the lowest index (numpy argmax); all-accepted requests emit the argmax bonus."""
    rng = np.random.default_rng(1000)
    B, K, V = 50, 4, 300
    # coarse bf16-like values: many ties at the maximum
    l = np.round(rng.standard_normal((B * (K + 1), V)) * 2).astype(np.float32)
    am = np.argmax(l, axis=1)
    ids = am.reshape(B, K + 1)[:, :K].reshape(-1).astype(np.int32)
    res = oracle.reject_sample(l, ids, (np.arange(B + 1) * K).astype(np.int32),
                               rng.random((B * (K + 1), 2), dtype=np.float32), np.zeros(B, np.float32), None,
                               debug=True, impl=impl)
    if not np.array_equal(res.row_argmax, am):
        return False, "row argmax differs from numpy's first-occurrence argmax"
    if not (res.num_accepted == K).all():
        return False, "drafts equal to the argmax were rejected"
    if not np.array_equal(res.tokens.reshape(B, K + 1)[:, K], am.reshape(B, K + 1)[:, K]):
        return False, "bonus is not the argmax of the last row"
    return True, "ok"


def check_zero_drafts(impl=None):
    """k = 0 emits exactly one token: argmax (greedy) or the inverse CDF of p."""
    rng = np.random.default_rng(1100)
    B, V = 40, 200
    l = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    u = rng.random((B, 2), dtype=np.float32)
    temps = np.where(np.arange(B) % 2 == 0, 0.0, 0.75).astype(np.float32)
    res = oracle.reject_sample(l, np.zeros(0, np.int32), np.zeros(B + 1, np.int32), u, temps, None, impl=impl)
    if not (res.num_accepted == 0).all():
        return False, "k=0 request reports accepted drafts"
    for b in range(B):
        if temps[b] <= 0:
            want = int(np.argmax(l[b]))
        else:
            c = np.cumsum(_p_from_logits(l[b], float(temps[b])))
            want = int(np.searchsorted(c, float(u[b, 1]) * c[-1], side="right"))
        if res.tokens[b] != want and not (res.flags[b] & oracle.NEAR_SAMPLE):
            return False, f"request {b}: token {res.tokens[b]} != {want}"
    return True, "ok"


def check_extreme_uniforms(impl=None):
    """u = 0 picks the first token with mass; the largest float32 below 1 picks the last; masked tokens never."""
    V = 16
    l = np.full((2, V), -np.inf, np.float32)
    l[:, 3:12] = np.linspace(-1, 1, 9, dtype=np.float32)
    u = np.array([[0.0, 0.0], [0.0, np.nextafter(np.float32(1), np.float32(0))]], np.float32)
    res = oracle.reject_sample(l, np.zeros(0, np.int32), np.zeros(3, np.int32), u, np.ones(2, np.float32), None,
                               impl=impl)
    if res.tokens.tolist() != [3, 11]:
        return False, f"extreme uniforms gave {res.tokens.tolist()} (want [3, 11])"
    # one-hot draft at a masked token: p(x*) = 0 is rejected even at u = 0
    res = oracle.reject_sample(l, np.array([0], np.int32), np.array([0, 1], np.int32), u, np.ones(1, np.float32),
                               None, impl=impl)
    if res.num_accepted[0] != 0 or res.tokens[0] != 3:
        return False, f"masked draft: accepted={res.num_accepted[0]} token={res.tokens[0]}"
    return True, "ok"


def check_row_statistics(impl=None):
    """Debug row statistics against library routines (max, logsumexp, softmax, argmax); bf16 widening."""
    from speculative_decoding_rejection_spec_gb300 import workloads as W
    for name in ("tiny",):
        w = W.generate(name)
        res = oracle.reject_sample_workload(w, debug=True, impl=impl)
        l = W.logits_as_f32(w).astype(np.float64)
        temp = float(w["temperature"][0])
        if not np.array_equal(res.row_max, l.max(axis=1)):
            return False, "row max"
        temp = np.float64(np.float32(temp))
        want_s = np.exp(special.logsumexp(l / temp, axis=1) - l.max(axis=1) / temp)
        if np.max(np.abs(res.row_sum / want_s - 1)) > 1e-12:
            return False, "row sum"
        rows = np.arange(w["T"])
        req = np.repeat(np.arange(w["B"]), np.diff(w["cu_num_draft"]) + 1)
        drows = rows[(rows - (w["cu_num_draft"][req] + req)) < np.diff(w["cu_num_draft"])[req]]
        p = special.softmax(l[drows] / temp, axis=1)
        want_p = p[np.arange(drows.size), w["draft_ids"]]
        if np.max(np.abs(res.p_draft / want_p - 1)) > 1e-12:
            return False, "p(x*)"
    # bf16 rows widen exactly
    rng = np.random.default_rng(1200)
    x = (rng.standard_normal((3, 77)) * 4).astype(np.float32)
    bits = W.f32_to_bf16_bits(x)
    res = oracle.reject_sample(bits, np.zeros(2, np.int32), np.array([0, 2], np.int32),
                               rng.random((3, 2), dtype=np.float32), np.ones(1, np.float32), None, debug=True,
                               impl=impl)
    if not np.array_equal(res.row_max, W.bf16_bits_to_f32(bits).astype(np.float64).max(axis=1)):
        return False, "bf16 row max"
    return True, "ok"


def check_invalid_inputs(impl=None):
    """Invalid requests report -1 and the bad-input flag; valid neighbours are unaffected."""
    V = 10
    rng = np.random.default_rng(1300)
    cu = np.array([0, 2, 2 + 33, 2 + 33 + 1], np.int32)  # request 1 has k = 33 > 32
    B = 3
    T = int(cu[-1]) + B
    l = rng.standard_normal((T, V)).astype(np.float32)
    ids = rng.integers(0, V, size=T - B).astype(np.int32)
    ids[-1] = V  # request 2 has an out-of-range draft id
    res = oracle.reject_sample(l, ids, cu, rng.random((T, 2), dtype=np.float32), np.ones(B, np.float32), None,
                               impl=impl)
    if res.num_accepted.tolist()[1:] != [-1, -1] or res.num_accepted[0] < 0:
        return False, f"num_accepted {res.num_accepted.tolist()}"
    if not (res.flags[1] & oracle.BAD_INPUT and res.flags[2] & oracle.BAD_INPUT) or res.flags[0] & oracle.BAD_INPUT:
        return False, "flags"
    res = oracle.reject_sample(l[:T - 1], ids, cu, rng.random((T, 2), dtype=np.float32), np.ones(B, np.float32),
                               None, impl=impl)
    if res.status != 1 or not (res.num_accepted == -1).all():
        return False, "T != cu[B] + B not reported"
    res = oracle.reject_sample(l, ids, np.array([0, 3, 1, 36], np.int32), rng.random((T, 2), dtype=np.float32),
                               np.ones(B, np.float32), None, impl=impl)
    if res.status != 1 or not (res.num_accepted == -1).all() or (res.tokens != -2).any():
        return False, "decreasing cu not reported as a layout error"
    return True, "ok"


def check_degenerate_residual(impl=None):
    """An empty residual (p = q exactly, draft with q(x*) = p(x*) = 0) falls back to a draw from p, flagged."""
    V = 6
    l = np.full((2, V), -np.inf, np.float32)
    l[:, 2] = 0.0  # p is one-hot at token 2
    q = np.zeros((1, V), np.float32)
    q[0, 2] = 1.0  # q equals p exactly
    res = oracle.reject_sample(l, np.array([4], np.int32), np.array([0, 1], np.int32),
                               np.array([[0.0, 0.3], [0.5, 0.5]], np.float32), np.ones(1, np.float32), q,
                               impl=impl)
    if res.num_accepted[0] != 0:
        return False, "draft with p(x*) = q(x*) = 0 was accepted"
    if res.tokens[0] != 2 or not (res.flags[0] & oracle.DEGENERATE):
        return False, f"degenerate residual gave token {res.tokens[0]} flags {res.flags[0]}"
    return True, "ok"


def _filtered(p, top_k, top_p):
    """Kept set of the top-k / top-p restriction by library routines (numpy sort / cumsum)."""
    order = np.argsort(-p, kind="stable")
    keep = np.ones_like(p, dtype=bool)
    if 0 < top_k < p.size:
        keep &= p >= p[order[top_k - 1]]
    if 0 < top_p < 1:
        pk = np.where(keep, p, 0.0)
        pk = pk / pk.sum()
        srt = np.sort(pk)[::-1]
        n = int(np.searchsorted(np.cumsum(srt), top_p))  # first index where the cumulative reaches top_p
        keep &= pk >= srt[min(n, srt.size - 1)]
    q = np.where(keep, p, 0.0)
    return q / q.sum()


def check_top_k_top_p(impl=None, N=300_000):
    """Top-k / top-p: every emitted position is distributed as the renormalised restricted p
    (chi-square), and the special cases top-k = 1 and a tiny top-p give the argmax."""
    base = np.array([0.4, -0.3, 1.2, 0.1, -1.0, 0.6, 0.0, -0.5], dtype=np.float32)
    cases = [(3, 1.0, 1.0), (0, 0.8, 0.9), (5, 0.6, 0.7), (8, 0.5, 1.0), (2, 0.3, 1.3), (5, 0.8, 1.3), (3, 0.7, 1.0)]
    ntests = 2 * len(cases)
    for ci, (tk, tp, temp) in enumerate(cases):
        l = (base * np.float32(1.7)).astype(np.float32)
        pf = _filtered(_p_from_logits(l, temp), tk, tp)
        K = 1
        ids, u, cu, temps = _iid_batch(N, K, l, temp, Q8, Q8, seed=900 + ci)
        res = oracle.reject_sample(l, ids, cu, u, temps, Q8.astype(np.float32), logits_row_stride=0, q_row_stride=0,
                                   vocab=8, num_rows=N * (K + 1), impl=impl, top_k=np.full(N, tk, np.int32),
                                   top_p=np.full(N, tp, np.float32))
        tok = res.tokens.reshape(N, K + 1)
        for m in range(K + 1):
            sel = res.num_accepted >= m
            obs = np.bincount(tok[sel, m], minlength=8)
            if obs.shape[0] != 8:
                return False, "token out of range"
            exp_ = pf * sel.sum()
            if (obs[exp_ == 0] > 0).any():
                return False, f"case {ci}: a filtered-out token was emitted at position {m}"
            nz = exp_ > 0
            if nz.sum() > 1:
                pval = stats.chisquare(obs[nz], exp_[nz]).pvalue
                if not pval > 1e-4 / ntests:
                    return False, f"case {ci} (top_k={tk}, top_p={tp}) pos {m}: chi-square p={pval:.3g}"
    rng = np.random.default_rng(950)
    l = (rng.standard_normal((20, 300)) * 2).astype(np.float32)
    am = np.argmax(l, axis=1)
    for tk, tp in ((1, 1.0), (0, 1e-9)):
        res = oracle.reject_sample(l, np.zeros(0, np.int32), np.zeros(21, np.int32),
                                   rng.random((20, 2), dtype=np.float32), np.ones(20, np.float32), None, impl=impl,
                                   top_k=np.full(20, tk, np.int32), top_p=np.full(20, tp, np.float32))
        if not np.array_equal(res.tokens, am):
            return False, f"top_k={tk} top_p={tp} should give the argmax"
    # filters off (k >= V, p = 1) change nothing
    w = None
    res0 = oracle.reject_sample(l, np.zeros(0, np.int32), np.zeros(21, np.int32),
                                np.full((20, 2), 0.37, np.float32), np.ones(20, np.float32), None, impl=impl)
    res1 = oracle.reject_sample(l, np.zeros(0, np.int32), np.zeros(21, np.int32),
                                np.full((20, 2), 0.37, np.float32), np.ones(20, np.float32), None, impl=impl,
                                top_k=np.full(20, 300, np.int32), top_p=np.ones(20, np.float32))
    if not np.array_equal(res0.tokens, res1.tokens):
        return False, "disabled filters changed the result"
    return True, "ok"


def _expected_margins(l32, temps, cu, ids, u, q):
    """Per request, by numpy / scipy routines: the visited positions' smallest relative
    acceptance margin |u*q* - p*| / max(p*, u*q*), the output row's sampling margin
    min(theta - C(v-1), C(v) - theta) / Z with C = cumsum(residual), v = searchsorted(C,
    theta, side='right'), theta = u_s * Z, and whether that row is an explicit-q residual."""
    B = len(cu) - 1
    out = []
    for r in range(B):
        k = int(cu[r + 1] - cu[r])
        tb, db = int(cu[r]) + r, int(cu[r])
        p_rows = special.softmax(l32[tb:tb + k + 1].astype(np.float64) / np.float64(np.float32(temps[r])), axis=1)
        acc_m, j = np.inf, k
        for i in range(k):
            x = int(ids[db + i])
            qs = np.float64(q[db + i, x]) if q is not None else 1.0
            lhs, rhs = np.float64(u[tb + i, 0]) * qs, p_rows[i, x]
            big = max(lhs, rhs)
            if big > 0:
                acc_m = min(acc_m, abs(lhs - rhs) / big)
            if not lhs < rhs:
                j = i
                break
        p = p_rows[j]
        explicit = q is not None and j < k
        if j < k:
            res = np.maximum(p - q[db + j].astype(np.float64), 0.0) if q is not None else p.copy()
            if q is None:
                res[int(ids[db + j])] = 0.0
        else:
            res = p
        C = np.cumsum(res)
        Z = C[-1]
        theta = np.float64(u[tb + j, 1]) * Z
        v = int(np.searchsorted(C, theta, side="right"))
        lo = C[v - 1] if v > 0 else 0.0
        smp = min(theta - lo, C[v] - theta) / Z
        out.append((j, acc_m, smp, explicit, smp * Z))
    return out


def check_margins_and_flags(impl=None):
    """The oracle's near-boundary report, which decides which GPU requests may differ: its
    margins against an independent numpy recomputation (1e-12), and its flags against the bands
    applied to those margins, on 8- and 16-token rows with decisions planted near a boundary."""
    rng = np.random.default_rng(1500)
    for V, explicit in ((8, True), (16, True), (8, False), (16, False)):
        B = 48
        ks = rng.integers(0, 4, size=B)
        cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
        T = int(cu[-1]) + B
        l32 = (rng.standard_normal((T, V)) * 1.5).astype(np.float32)
        temps = rng.choice([0.7, 1.0, 1.3], size=B).astype(np.float32)
        q = None
        if explicit:
            q = rng.random((T - B, V)) ** 2
            q = (q / q.sum(axis=1, keepdims=True)).astype(np.float32)
        ids = np.array([rng.choice(V, p=(q[d] / q[d].sum()) if q is not None else None) for d in range(T - B)],
                       np.int32)
        u = rng.random((T, 2)).astype(np.float32)
        # plant near-boundary decisions: for every third request, position 0's coin a relative
        # 3e-6 from p / q (inside the 1e-5 band); for every fourth, the output row's draw a
        # relative 2e-6 from a CDF boundary
        pre = _expected_margins(l32, temps, cu, ids, u, q)
        for r in range(B):
            tb, db, k = int(cu[r]) + r, int(cu[r]), int(ks[r])
            if r % 3 == 0 and k > 0:
                p0 = special.softmax(l32[tb].astype(np.float64) / np.float64(temps[r]))
                x = int(ids[db])
                qs = float(q[db, x]) if q is not None else 1.0
                target = p0[x] / qs * (1 + (3e-6 if r % 2 else -3e-6))
                if target < 1:
                    u[tb, 0] = np.float32(target)
        mid = _expected_margins(l32, temps, cu, ids, u, q)
        for r in range(B):
            if r % 4 == 1:
                j = mid[r][0]
                tb, db, k = int(cu[r]) + r, int(cu[r]), int(ks[r])
                p = special.softmax(l32[tb + j].astype(np.float64) / np.float64(temps[r]))
                res = p if j == k else (np.maximum(p - q[db + j], 0.0) if q is not None else p.copy())
                if q is None and j < k:
                    res[int(ids[db + j])] = 0.0
                C = np.cumsum(res)
                b = min(V - 2, int(rng.integers(0, V - 1)))
                if C[-1] > 0 and 0 < C[b] < C[-1]:
                    u[tb + j, 1] = np.float32(C[b] / C[-1] * (1 + 2e-6))
        want = _expected_margins(l32, temps, cu, ids, u, q)
        res = oracle.reject_sample(l32, ids, cu, u, temps, q, debug=True, impl=impl)
        near_acc = near_smp = 0
        for r, (j, am, sm, expl, sabs) in enumerate(want):
            if res.num_accepted[r] != j:
                return False, f"V={V} request {r}: accepted {res.num_accepted[r]}, expected {j}"
            got_a, got_s = float(res.margin[r, 0]), float(res.margin[r, 1])
            if (np.isinf(am) != np.isinf(got_a)) or (np.isfinite(am) and abs(got_a - am) > 1e-12):
                return False, f"V={V} request {r}: acceptance margin {got_a} vs {am}"
            if abs(got_s - sm) > 1e-12:
                return False, f"V={V} request {r}: sampling margin {got_s} vs {sm}"
            f = int(res.flags[r])
            if bool(f & oracle.NEAR_ACCEPT) != (am <= 1e-5):
                return False, f"V={V} request {r}: acceptance flag {f} for margin {am}"
            if bool(f & oracle.NEAR_SAMPLE) != (sm <= 1e-5):
                return False, f"V={V} request {r}: sampling flag {f} for margin {sm}"
            if bool(f & oracle.NEAR_SAMPLE_ABS) != (expl and sabs <= 2e-6):
                return False, f"V={V} request {r}: absolute flag {f} for margin {sabs}"
            near_acc += am <= 1e-5
            near_smp += sm <= 1e-5
        if near_acc < 3 or near_smp < 3:
            return False, f"V={V}: too few planted near-boundary decisions ({near_acc}, {near_smp})"
    return True, "ok"


ALL_CHECKS = [
    check_output_distribution, check_acceptance_rate, check_residual_mass, check_accepted_length,
    check_exact_enumeration, check_q_equals_p, check_disjoint_supports, check_one_hot_draft,
    check_greedy_worked_chain, check_rollback_arithmetic, check_greedy_ties_and_bonus, check_zero_drafts,
    check_extreme_uniforms, check_row_statistics, check_invalid_inputs, check_degenerate_residual,
    check_top_k_top_p, check_margins_and_flags,
]
