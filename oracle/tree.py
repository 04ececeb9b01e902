"""Plain CPU oracle of greedy tree verification.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"投机解码（Speculative Decoding）端到端深挖" §6.2 and §7.1: starting at the root, take the
target argmax at the current node; if one of the current node's children carries that
token, accept it and continue from it; otherwise stop.  The token emitted after the last
accepted node is the target argmax there (the bonus).  Readings: node 0 of each request
is the root (parent -1), every other node's parent precedes it; among children carrying
the argmax token the lowest node index wins; argmax ties go to the lowest token index.
"""
from __future__ import annotations

import numpy as np


def verify_batch(logits_f64: np.ndarray, parent, node_tokens, cu_nodes):
    """logits_f64: [N, V] target logits (float64 view of the fp32 / bf16 values).

    Returns (tokens [N] with each request's accepted tokens then the bonus, -1 padded;
    num_accepted [B]; last_node [B] local index; -1 counts for invalid trees).
    """
    N = logits_f64.shape[0]
    V = logits_f64.shape[1]
    B = len(cu_nodes) - 1
    out = np.full(N, -1, np.int32)
    acc = np.zeros(B, np.int32)
    last = np.zeros(B, np.int32)
    for r in range(B):
        n0, n1 = int(cu_nodes[r]), int(cu_nodes[r + 1])
        n = n1 - n0
        par = [int(x) for x in parent[n0:n1]]
        tok = [int(x) for x in node_tokens[n0:n1]]
        ok = n >= 1 and par[0] == -1 and all(0 <= par[i] < i for i in range(1, n)) and \
            all(0 <= tok[i] < V for i in range(1, n))
        if not ok:
            acc[r] = -1
            last[r] = -1
            continue
        cur, a = 0, 0
        while True:
            am = int(np.argmax(logits_f64[n0 + cur]))  # first index of the maximum
            child = next((i for i in range(1, n) if par[i] == cur and tok[i] == am), None)
            out[n0 + a] = am
            if child is None:
                break
            a += 1
            cur = child
        acc[r] = a
        last[r] = cur
    return out, acc, last
