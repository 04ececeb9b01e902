"""The seeded input generators: shapes, determinism and the structure each workload promises."""
import numpy as np

from oracle import ngram as ong, tree as otree
from speculative_decoding_rejection_spec_gb300 import workloads as W

SMALL_TREE = dict(B=6, max_nodes=20, topk=3, depth=4, V=300, dtype="bf16", sigma=3.0, lead=30.0, p_follow=0.5,
                  seed=3)


def test_tree_structure_and_planted_argmax():
    w = W.generate_tree(SMALL_TREE)
    cu, par = w["cu_nodes"], w["parent"]
    assert cu[0] == 0 and cu[-1] == w["N"] == w["logits"].shape[0] and w["logits"].shape[1] == w["V"]
    lg = W.bf16_bits_to_f32(w["logits"])
    for r in range(w["B"]):
        p = par[cu[r]:cu[r + 1]]
        assert p[0] == -1 and all(0 <= p[i] < i for i in range(1, len(p)))
        assert len(p) <= SMALL_TREE["max_nodes"]
    # the planted lead is each row's strict maximum, so a child that copies it matches the argmax
    top2 = np.sort(lg, axis=1)[:, -2:]
    assert (top2[:, 1] == 30.0).all() and (top2[:, 0] < 30.0).all()
    # some children follow their parent's lead: the walks of the oracle go below the root
    tok, acc, last = otree.verify_batch(lg.astype(np.float64), par, w["node_tokens"], cu)
    assert acc.max() >= 1


def test_tree_generator_is_deterministic():
    a, b = W.generate_tree(SMALL_TREE), W.generate_tree(SMALL_TREE)
    for k in ("logits", "parent", "node_tokens", "cu_nodes"):
        assert np.array_equal(a[k], b[k])
    c = W.generate_tree(SMALL_TREE, seed=4)
    assert not np.array_equal(a["logits"], c["logits"])


def test_ngram_contexts_have_repeats():
    spec = dict(B=16, L=512, vocab=1000, span=(4, 32), p_copy=0.3, min_n=2, max_n=4, k=6, seed=7)
    g = W.generate_ngram(spec)
    assert g["tokens"].shape == (16 * 512,) and g["cu_tokens"][-1] == 16 * 512
    assert g["tokens"].min() >= 0 and g["tokens"].max() < 1000
    assert np.array_equal(g["tokens"], W.generate_ngram(spec)["tokens"])
    drafts, counts = ong.propose_batch(g["tokens"], g["cu_tokens"], 2, 4, 6)
    assert (counts > 0).any()  # copied spans make some suffixes reappear
