"""Pins of the n-gram proposer oracle: the page's example and an independent KMP search."""
import json
import os

import numpy as np

from oracle import ngram


def test_docstring_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "ngram_example.json")))
    assert ngram.propose(g["context"], g["min_n"], g["max_n"], g["k"]) == g["expected"]


def test_longest_n_first_and_limits():
    ctx = [5, 6, 7, 9, 6, 7, 1, 5, 6, 7]
    # n=3 pattern [5,6,7] occurs at 0 -> propose what follows it
    assert ngram.propose(ctx, 1, 3, 2) == [9, 6]
    # only n=2 allowed: pattern [6,7] first occurs at 1
    assert ngram.propose(ctx, 2, 2, 3) == [9, 6, 7]
    # max_model_len caps k; k <= 0 gives nothing
    assert ngram.propose(ctx, 1, 3, 5, max_model_len=11) == [9]
    assert ngram.propose(ctx, 1, 3, 5, max_model_len=10) is None
    # no earlier occurrence of any suffix
    assert ngram.propose([1, 2, 3, 4], 1, 2, 3) is None
    # the occurrence may not overlap the final pattern: [1,1,1] with n=1 matches s=0 (follows: [1,1])
    assert ngram.propose([1, 1, 1], 1, 1, 5) == [1, 1]
    assert ngram.propose([1, 1], 2, 2, 5) is None


def _kmp_first(text, pattern):
    """Leftmost start of `pattern` in `text` by Knuth-Morris-Pratt (textbook failure function)."""
    n = len(pattern)
    fail = [0] * n
    q = 0
    for i in range(1, n):
        while q and pattern[i] != pattern[q]:
            q = fail[q - 1]
        if pattern[i] == pattern[q]:
            q += 1
        fail[i] = q
    q = 0
    for i, x in enumerate(text):
        while q and x != pattern[q]:
            q = fail[q - 1]
        if x == pattern[q]:
            q += 1
        if q == n:
            return i - n + 1
    return -1


def test_brute_force_agrees_with_kmp_on_random_contexts():
    rng = np.random.default_rng(3)
    for trial in range(3000):
        L = int(rng.integers(1, 40))
        ctx = [int(x) for x in rng.integers(0, int(rng.integers(2, 6)), size=L)]
        min_n, max_n, k = 1, int(rng.integers(1, 6)), int(rng.integers(1, 6))
        want = None
        for n in range(max_n, min_n - 1, -1):
            if 2 * n > L:
                continue
            s = _kmp_first(ctx[:L - n], ctx[L - n:])
            if s >= 0:
                want = ctx[s + n:s + n + k]
                break
        assert ngram.propose(ctx, min_n, max_n, k) == want, (ctx, max_n, k)
