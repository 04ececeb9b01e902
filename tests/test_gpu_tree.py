"""GPU greedy tree verification against the CPU oracle (exact: every decision is an argmax)."""
import json
import os

import numpy as np
import pytest

from oracle import tree
from speculative_decoding_rejection_spec_gb300 import binding, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    import __graft_entry__ as G
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.build()
    binding.load()


def _random_trees(B, V, seed, max_nodes=64, topk=4, depth=6, dtype="bf16"):
    """EAGLE-style draft trees: up to `topk` children per node, up to `depth` levels, bounded node
    budget; children copy the parent's target argmax with some probability so walks go deep."""
    rng = np.random.default_rng(seed)
    parents, toks, cu = [], [], [0]
    rows = []
    for r in range(B):
        par, tk, lvl = [-1], [0], [0]
        i = 0
        while i < len(par) and len(par) < max_nodes:
            if lvl[i] < depth:
                for _ in range(int(rng.integers(1, topk + 1))):
                    if len(par) >= max_nodes:
                        break
                    par.append(i)
                    tk.append(-1)  # filled below
                    lvl.append(lvl[i] + 1)
            i += 1
        n = len(par)
        x = (rng.standard_normal((n, V)) * 3).astype(np.float32)
        if dtype == "bf16":
            x = W.bf16_bits_to_f32(W.f32_to_bf16_bits(x))
        am = np.argmax(x, axis=1)
        for j in range(1, n):
            tk[j] = int(am[par[j]]) if rng.random() < 0.5 else int(rng.integers(0, V))
        parents += par
        toks += tk
        cu.append(cu[-1] + n)
        rows.append(x)
    return np.vstack(rows), np.array(parents, np.int32), np.array(toks, np.int32), np.array(cu, np.int32)


def _run(x, parent, toks, cu, dtype):
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(W.f32_to_bf16_bits(x).view(np.int16)).cuda().view(torch.bfloat16)
    else:
        t = torch.from_numpy(x).cuda()
    out, acc, last, ws = binding.tree_verify_greedy(t, torch.from_numpy(parent).cuda(), torch.from_numpy(toks).cuda(),
                                                     torch.from_numpy(cu).cuda())
    st = binding.last_device_error(ws)
    return out.cpu().numpy(), acc.cpu().numpy(), last.cpu().numpy(), st


def test_page_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tree_greedy_example.json")))
    rng = np.random.default_rng(0)
    x = rng.standard_normal((len(g["parent"]), g["vocab"])).astype(np.float32)
    for i, a in enumerate(g["target_argmax"]):
        x[i, a] = x[i].max() + 1
    out, acc, last, st = _run(x, np.array(g["parent"], np.int32), np.array(g["node_tokens"], np.int32),
                              np.array([0, len(g["parent"])], np.int32), "f32")
    assert out.tolist() == g["expected_tokens"] and acc[0] == g["expected_num_accepted"]
    assert last[0] == g["expected_last_node"] and st[0] == 0


@pytest.mark.parametrize("dtype,V", [("bf16", 128256), ("f32", 32000), ("bf16", 1001)])
def test_random_trees_match_oracle(dtype, V):
    x, parent, toks, cu = _random_trees(48, V, seed=V, dtype=dtype)
    out, acc, last, st = _run(x, parent, toks, cu, dtype)
    wout, wacc, wlast = tree.verify_batch(x.astype(np.float64), parent, toks, cu)
    assert st[0] == 0
    assert np.array_equal(acc, wacc) and np.array_equal(last, wlast) and np.array_equal(out, wout)
    assert acc.max() >= 3  # the walks do go deep


def test_malformed_trees_are_reported():
    x, parent, toks, cu = _random_trees(4, 500, seed=3, dtype="f32")
    parent = parent.copy()
    toks = toks.copy()
    parent[cu[1] + 2] = 5 if cu[2] - cu[1] > 6 else cu[2] - cu[1]  # parent not preceding its child
    toks[cu[3] + 1] = 500  # token outside the vocabulary
    out, acc, last, st = _run(x, parent, toks, cu, "f32")
    wout, wacc, wlast = tree.verify_batch(x.astype(np.float64), parent, toks, cu)
    assert acc[1] == -1 and acc[3] == -1 and np.array_equal(acc, wacc)
    assert st[0] == 5 and st[1] & binding.DEVERR_TREE and st[2] == 1
