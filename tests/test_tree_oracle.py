"""Pins of the greedy tree-verification oracle."""
import json
import os

import numpy as np

import oracle
from oracle import tree


def _rows_with_argmax(am, V, rng):
    x = rng.standard_normal((len(am), V))
    for i, a in enumerate(am):
        x[i, a] = x[i].max() + 1.0
    return x


def test_page_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tree_greedy_example.json")))
    x = _rows_with_argmax(g["target_argmax"], g["vocab"], np.random.default_rng(0))
    out, acc, last = tree.verify_batch(x, g["parent"], g["node_tokens"], [0, len(g["parent"])])
    assert out.tolist() == g["expected_tokens"]
    assert acc[0] == g["expected_num_accepted"] and last[0] == g["expected_last_node"]


def test_chain_tree_equals_chain_greedy_sampler():
    """A tree whose nodes form one chain is the chain case: same tokens as the greedy sampler."""
    rng = np.random.default_rng(1)
    V, B, K = 50, 40, 6
    x = np.round(rng.standard_normal((B * (K + 1), V)) * 2).astype(np.float32)  # ties present
    am = np.argmax(x, axis=1)
    drafts = np.where(rng.random((B, K)) < 0.7, am.reshape(B, K + 1)[:, :K], rng.integers(0, V, (B, K)))
    cu_draft = (np.arange(B + 1) * K).astype(np.int32)
    ref = oracle.reject_sample(x, drafts.reshape(-1).astype(np.int32), cu_draft,
                               rng.random((B * (K + 1), 2), dtype=np.float32), np.zeros(B, np.float32), None)
    parent = np.tile(np.arange(-1, K), B)
    toks = np.concatenate([np.concatenate([[0], d]) for d in drafts])
    out, acc, last = tree.verify_batch(x.astype(np.float64), parent, toks, np.arange(B + 1) * (K + 1))
    assert np.array_equal(acc, ref.num_accepted)
    assert np.array_equal(out, ref.tokens)
    assert np.array_equal(last, acc)


def test_first_matching_sibling_and_invalid_trees():
    V = 8
    rng = np.random.default_rng(2)
    # root has two children with the same token 3; the lower node index is taken
    x = _rows_with_argmax([3, 4, 5, 6], V, rng)
    out, acc, last = tree.verify_batch(x, [-1, 0, 0, 2], [0, 3, 3, 4], [0, 4])
    assert acc[0] == 1 and last[0] == 1 and out[:2].tolist() == [3, 4]
    # a parent that does not precede its child, a token outside the vocabulary
    out, acc, last = tree.verify_batch(np.vstack([x, x]), [-1, 2, 0, 0, -1, 0, 0, 0], [0, 1, 2, 3, 0, 1, 9, 2],
                                       [0, 4, 8])
    assert acc.tolist() == [-1, -1]
