"""Plain CPU oracle of the n-gram (prompt-lookup) draft proposer.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"第12章 投机解码：以小博大" §12.4.4: for n from max_n down to min_n, take the last n tokens of
the context as the pattern, find its first (leftmost) earlier occurrence, and propose the
tokens that follow it, at most k of them (fewer when the context ends first); the longest
n that matches wins; no match gives no proposal.  "Earlier" means the occurrence lies
wholly before the final n tokens, i.e. it starts at s <= L - 2n (the page's search stops
comparing at index L - n).  k is first capped by max_model_len - L.

This is the definition written out as a brute-force search; the page computes the same
with a KMP scan.
"""
from __future__ import annotations


def propose(context: list[int], min_n: int, max_n: int, k: int, max_model_len: int | None = None) -> list[int] | None:
    L = len(context)
    if max_model_len is not None:
        k = min(k, max_model_len - L)
    if k <= 0:
        return None
    for n in range(max_n, min_n - 1, -1):
        if n <= 0 or 2 * n > L:
            continue
        pattern = context[L - n:]
        for s in range(0, L - 2 * n + 1):
            if context[s:s + n] == pattern:
                return context[s + n:s + n + k]
    return None


def propose_batch(tokens, cu_tokens, min_n: int, max_n: int, k: int, max_model_len: int | None = None):
    """Per request r the context tokens[cu[r]:cu[r+1]]; returns (drafts [B, k] padded with -1, counts [B])."""
    import numpy as np
    B = len(cu_tokens) - 1
    out = np.full((B, max(k, 0)), -1, dtype=np.int32)
    cnt = np.zeros(B, dtype=np.int32)
    for r in range(B):
        ctx = [int(x) for x in tokens[cu_tokens[r]:cu_tokens[r + 1]]]
        p = propose(ctx, min_n, max_n, k, max_model_len)
        if p:
            out[r, :len(p)] = p
            cnt[r] = len(p)
    return out, cnt
