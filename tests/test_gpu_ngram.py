"""GPU n-gram proposer against the CPU oracle (exact)."""
import json
import os

import numpy as np
import pytest

from oracle import ngram
from speculative_decoding_rejection_spec_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    import __graft_entry__ as G
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.build()
    binding.load()


def _run(contexts, min_n, max_n, k, max_model_len=0):
    import torch
    cu = np.zeros(len(contexts) + 1, np.int64)
    cu[1:] = np.cumsum([len(c) for c in contexts])
    tokens = np.concatenate([np.asarray(c, np.int32) for c in contexts]) if cu[-1] else np.zeros(1, np.int32)
    d, n = binding.ngram_propose(torch.from_numpy(tokens).cuda(), torch.from_numpy(cu).cuda(), min_n, max_n, k,
                                 max_model_len)
    want_d, want_n = ngram.propose_batch(tokens, cu, min_n, max_n, k, max_model_len if max_model_len > 0 else None)
    return d.cpu().numpy(), n.cpu().numpy(), want_d, want_n


def test_docstring_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "ngram_example.json")))
    d, n, wd, wn = _run([g["context"]], g["min_n"], g["max_n"], g["k"])
    assert n[0] == 3 and d[0, :3].tolist() == g["expected"] and d[0, 3] == -1


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_contexts_match_oracle(seed):
    rng = np.random.default_rng(seed)
    contexts = []
    for r in range(300):
        L = int(rng.integers(0, 3000 if r % 10 == 0 else 200))
        vocab = int(rng.integers(2, 50))
        contexts.append(rng.integers(0, vocab, size=L).tolist())
    for (mn, mx, k, mml) in [(1, 3, 4, 0), (2, 8, 5, 0), (3, 5, 8, 150), (1, 1, 1, 0)]:
        d, n, wd, wn = _run(contexts, mn, mx, k, mml)
        assert np.array_equal(n, wn) and np.array_equal(d, wd), (mn, mx, k, mml)


def test_long_repetitive_context():
    # code-like context: a template repeated with small edits, 40k tokens
    rng = np.random.default_rng(7)
    base = rng.integers(0, 32000, size=500)
    ctx = np.concatenate([np.where(rng.random(500) < 0.05, rng.integers(0, 32000, 500), base) for _ in range(80)])
    d, n, wd, wn = _run([ctx.tolist()] * 4, 3, 8, 5)
    assert np.array_equal(n, wn) and np.array_equal(d, wd) and (n > 0).all()
