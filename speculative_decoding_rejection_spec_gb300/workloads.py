"""Seeded synthetic inputs for the rejection sampler.

This module only draws inputs: target logits, draft distributions, draft tokens,
ragged draft counts, uniforms and temperatures.  It contains none of the
sampler's own arithmetic (no acceptance test, no residual, no inverse CDF of the
target).  Both the CUDA path and the CPU oracle read exactly the arrays it
returns.

Layout of a workload (request-major, the flattened ragged layout of
"第12章 投机解码：以小博大" §12.3.5):

* ``cu_num_draft`` int32 [B+1], cu[0] = 0; request r has k_r = cu[r+1] - cu[r] drafts;
* ``logits`` [T, V], T = cu[B] + B; request r owns target rows cu[r]+r .. cu[r+1]+r
  (k_r verify rows followed by its bonus row).  float32, or uint16 holding bf16
  bits (round-to-nearest-even from float32);
* ``draft_ids`` int32 [T-B]; request r's drafts are rows cu[r] .. cu[r+1]-1;
* ``draft_probs`` float32 [T-B, V] or None (one-hot draft);
* ``uniforms`` float32 [T, 2] in [0, 1): column 0 is the acceptance coin of a
  verify row, column 1 the sampling draw of the output row;
* ``temperature`` float32 [B]; values <= 0 select the greedy path.

Random streams are keyed by (seed, component, block of rows) through numpy's
SeedSequence, so the arrays do not depend on how many threads generate them.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROWS_PER_BLOCK = 16

# The five synthetic workloads (sizes, distributions and seeds as specified for this sampler).
CONFIGS = {
    # B=4, K=3, V=1000, fp32 ~N(0, 2^2); draft logits = target + N(0, 0.5^2), softmaxed to q; T=1.0
    "tiny": dict(B=4, K=3, V=1000, dtype="f32", sigma=2.0, temperature=1.0, draft="noisy_q", q_sigma=0.5,
                 q_temperature=1.0, seed=0),
    # B=64, K=5, V=32000, bf16 ~N(0, 3^2), T=0, no draft probs; draft = argmax w.p. 0.7 else uniform token
    "greedy": dict(B=64, K=5, V=32000, dtype="bf16", sigma=3.0, temperature=0.0, draft="argmax_mix", p_match=0.7,
                   seed=1),
    # B=32, K=5, V=128256, fp32 ~N(0, 2.5^2), T=0.8; q = softmax((logits + N(0, 1)) / 0.8); ids ~ q
    "probabilistic": dict(B=32, K=5, V=128256, dtype="f32", sigma=2.5, temperature=0.8, draft="noisy_q",
                          q_sigma=1.0, q_temperature=0.8, seed=2),
    # B=256, K ~ U{0..7}, V=151936, bf16 ~N(0, 2^2), T=1.0, no draft probs; ids ~ target softmax w.p. 0.6
    "deterministic": dict(B=256, K="ragged", K_max=7, V=151936, dtype="bf16", sigma=2.0, temperature=1.0,
                          draft="target_mix", p_match=0.6, seed=3),
    # B in {128, 512, 1024}, K=8, V=128256, bf16 ~N(0, 2^2), one logit per row +8, T=0.7;
    # q = softmax(logits + N(0, 0.7^2)) (temperature 1 for the draft); ids ~ q
    "large-128": dict(B=128, K=8, V=128256, dtype="bf16", sigma=2.0, boost=8.0, temperature=0.7, draft="noisy_q",
                      q_sigma=0.7, q_temperature=1.0, seed=4),
    "large-512": dict(B=512, K=8, V=128256, dtype="bf16", sigma=2.0, boost=8.0, temperature=0.7, draft="noisy_q",
                      q_sigma=0.7, q_temperature=1.0, seed=4),
    "large-1024": dict(B=1024, K=8, V=128256, dtype="bf16", sigma=2.0, boost=8.0, temperature=0.7, draft="noisy_q",
                       q_sigma=0.7, q_temperature=1.0, seed=4),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); returns the raw uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((b + (((b >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bits to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def logits_as_f32(w: dict) -> np.ndarray:
    """The target logits of a workload as the float32 values both sides read."""
    return bf16_bits_to_f32(w["logits"]) if w["dtype"] == "bf16" else w["logits"]


def _rng(seed: int, component: int, block: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(entropy=seed, spawn_key=(component, block)))


def _draft_counts(spec: dict, seed: int) -> np.ndarray:
    B = spec["B"]
    K = spec["K"]
    if isinstance(K, str):  # ragged: uniform in 0..K_max
        ks = _rng(seed, 0).integers(0, spec["K_max"] + 1, size=B)
    elif np.ndim(K) == 1:
        ks = np.asarray(K)
    else:
        ks = np.full(B, int(K))
    return ks.astype(np.int32)


def generate(spec: dict | str, seed: int | None = None, threads: int | None = None, **overrides) -> dict:
    """Build one workload from a named config or a spec dict (fields as in CONFIGS).

    Extra fields accepted by the spec:
      ``K`` an int, "ragged" (with ``K_max``) or a per-request sequence;
      ``draft``: "noisy_q" (explicit q = softmax((l + N(0, q_sigma^2)) / q_temperature), ids ~ q),
                 "target_q" (explicit q equal to the target's tempered distribution, ids ~ q),
                 "argmax_mix" (no q; argmax w.p. p_match else a uniform token),
                 "target_mix" (no q; a draw from softmax(l) w.p. p_match else a uniform token),
                 "uniform" (no q; uniform tokens);
      ``boost``: add this to one uniformly chosen logit per row;
      ``temperature``: a scalar or a per-request sequence;
      ``top_k`` / ``top_p``: optional target filters, scalars or per-request sequences.
    """
    name = spec if isinstance(spec, str) else spec.get("name", "custom")
    spec = dict(CONFIGS[spec]) if isinstance(spec, str) else dict(spec)
    spec.update(overrides)
    name = spec.get("name", name)
    seed = int(spec.get("seed", 0) if seed is None else seed)
    B, V = int(spec["B"]), int(spec["V"])
    ks = _draft_counts(spec, seed)
    assert ks.shape == (B,)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ks)
    T = int(cu[-1]) + B
    ND = T - B
    row_req = np.repeat(np.arange(B), ks + 1)           # request of each target row
    row_pos = np.arange(T) - (cu[:-1] + np.arange(B))[row_req]  # position i within the request
    is_draft_row = row_pos < ks[row_req]
    draft_row_of = np.where(is_draft_row, np.arange(T) - row_req, -1)  # d = t - r on verify rows

    dtype = spec.get("dtype", "f32")
    sigma = float(spec.get("sigma", 1.0))
    boost = spec.get("boost")
    draft = spec.get("draft", "noisy_q")
    explicit_q = draft in ("noisy_q", "target_q")
    temps = np.broadcast_to(np.asarray(spec.get("temperature", 1.0), dtype=np.float32), (B,)).copy()

    logits = np.empty((T, V), dtype=np.uint16 if dtype == "bf16" else np.float32)
    draft_probs = np.empty((ND, V), dtype=np.float32) if explicit_q else None
    draft_ids = np.zeros(ND, dtype=np.int32)

    nblocks = (T + ROWS_PER_BLOCK - 1) // ROWS_PER_BLOCK

    def make_block(b: int) -> None:
        lo, hi = b * ROWS_PER_BLOCK, min(T, (b + 1) * ROWS_PER_BLOCK)
        rng = _rng(seed, 1, b)
        x = (rng.standard_normal((hi - lo, V)) * sigma).astype(np.float32)
        if boost is not None:
            hot = rng.integers(0, V, size=hi - lo)
            x[np.arange(hi - lo), hot] += np.float32(boost)
        if dtype == "bf16":
            logits[lo:hi] = f32_to_bf16_bits(x)
            x = bf16_bits_to_f32(logits[lo:hi])
        else:
            logits[lo:hi] = x
        # Draft side for the verify rows of this block.
        rows = np.nonzero(is_draft_row[lo:hi])[0]
        if rows.size == 0:
            return
        drng = _rng(seed, 2, b)
        d_idx = draft_row_of[lo:hi][rows]
        xl = x[rows].astype(np.float64)
        if explicit_q:
            if draft == "noisy_q":
                z = (xl + drng.standard_normal(xl.shape) * float(spec.get("q_sigma", 1.0)))
                z /= float(spec.get("q_temperature", 1.0))
            else:  # draft distribution identical to the tempered target
                z = xl / temps[row_req[lo:hi][rows]][:, None].astype(np.float64)
            z -= z.max(axis=1, keepdims=True)
            e = np.exp(z)
            q = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
            draft_probs[d_idx] = q
            c = np.cumsum(q.astype(np.float64), axis=1)
            u = drng.random(rows.size) * c[:, -1]
            ids = np.array([np.searchsorted(c[i], u[i], side="right") for i in range(rows.size)])
            draft_ids[d_idx] = np.minimum(ids, V - 1)
        else:
            uni = drng.integers(0, V, size=rows.size)
            if draft == "uniform":
                draft_ids[d_idx] = uni
                return
            pm = float(spec.get("p_match", 0.5))
            match = drng.random(rows.size) < pm
            if draft == "argmax_mix":
                pick = np.argmax(xl, axis=1)
            elif draft == "target_mix":  # Gumbel-max draw from softmax(l) (temperature 1)
                g = -np.log(-np.log(drng.random(xl.shape) + 1e-300) + 1e-300)
                pick = np.argmax(xl + g, axis=1)
            else:
                raise ValueError(f"unknown draft mode {draft!r}")
            draft_ids[d_idx] = np.where(match, pick, uni)

    workers = threads if threads is not None else min(32, os.cpu_count() or 1)
    if workers <= 1 or nblocks <= 1:
        for b in range(nblocks):
            make_block(b)
    else:
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(make_block, range(nblocks)))

    uniforms = _rng(seed, 3).random((T, 2), dtype=np.float32)
    out = dict(name=name, dtype=dtype, B=B, T=T, V=V, logits=logits, draft_probs=draft_probs, draft_ids=draft_ids,
               cu_num_draft=cu, uniforms=uniforms, temperature=temps, spec=spec)
    # optional top-k / top-p on the target (scalars or per-request sequences)
    if spec.get("top_k") is not None:
        out["top_k"] = np.broadcast_to(np.asarray(spec["top_k"], dtype=np.int32), (B,)).copy()
    if spec.get("top_p") is not None:
        out["top_p"] = np.broadcast_to(np.asarray(spec["top_p"], dtype=np.float32), (B,)).copy()
    return out


def total_drafts(w: dict) -> int:
    """Number of verified draft positions, sum_r k_r."""
    return int(w["cu_num_draft"][-1])


# ---------------------------------------------------------------------------------------
# Draft trees (greedy tree verification) and n-gram contexts
# ---------------------------------------------------------------------------------------

# EAGLE-style draft trees: up to `topk` children per node, up to `depth` levels, at most
# `max_nodes` nodes per request (root included), one target row per node.
TREE_CONFIGS = {
    "tree-64x64": dict(B=64, max_nodes=64, topk=4, depth=6, V=128256, dtype="bf16", sigma=3.0, lead=30.0,
                       p_follow=0.5, seed=21),
    "tree-256x64": dict(B=256, max_nodes=64, topk=4, depth=6, V=128256, dtype="bf16", sigma=3.0, lead=30.0,
                        p_follow=0.5, seed=22),
}


def generate_tree(spec: dict | str, seed: int | None = None) -> dict:
    """Draft trees with one target row per node.

    Each node row is N(0, sigma^2) with one planted lead token set to ``lead`` (10 sigma:
    the row's largest logit by construction); a child's token is its parent's lead token
    with probability ``p_follow``, else uniform, so walks go several levels deep.  Nodes are
    in topological order with node 0 of each request its root (parent -1, token 0).
    """
    if isinstance(spec, str):
        spec = TREE_CONFIGS[spec]
    spec = dict(spec)
    seed = spec["seed"] if seed is None else seed
    rng = np.random.default_rng(np.random.SeedSequence([seed, 7]))
    B, V = spec["B"], spec["V"]
    parents, toks, cu = [], [], [0]
    for _ in range(B):
        par, lvl = [-1], [0]
        i = 0
        while i < len(par) and len(par) < spec["max_nodes"]:
            if lvl[i] < spec["depth"]:
                for _c in range(int(rng.integers(1, spec["topk"] + 1))):
                    if len(par) >= spec["max_nodes"]:
                        break
                    par.append(i)
                    lvl.append(lvl[i] + 1)
            i += 1
        parents.append(np.array(par, np.int32))
        cu.append(cu[-1] + len(par))
    N = cu[-1]
    lead = rng.integers(0, V, size=N).astype(np.int32)
    node_tokens = np.zeros(N, np.int32)
    for r in range(B):
        base = cu[r]
        par = parents[r]
        for j in range(1, len(par)):
            follow = rng.random() < spec["p_follow"]
            node_tokens[base + j] = lead[base + par[j]] if follow else int(rng.integers(0, V))
    bf16 = spec["dtype"] == "bf16"
    logits = np.empty((N, V), np.uint16 if bf16 else np.float32)

    def fill(b0):
        b1 = min(N, b0 + ROWS_PER_BLOCK)
        x = (_rng(seed, 40, b0 // ROWS_PER_BLOCK).standard_normal((b1 - b0, V)) * spec["sigma"]).astype(np.float32)
        x[np.arange(b1 - b0), lead[b0:b1]] = spec["lead"]
        logits[b0:b1] = f32_to_bf16_bits(x) if bf16 else x

    with ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
        list(ex.map(fill, range(0, N, ROWS_PER_BLOCK)))
    parent = np.concatenate(parents).astype(np.int32)
    return dict(logits=logits, parent=parent, node_tokens=node_tokens, cu_nodes=np.array(cu, np.int32), B=B, N=N,
                V=V, dtype=spec["dtype"], spec=spec)


# Token contexts for the n-gram proposer: random tokens with planted repeats of earlier spans,
# so that the final n-gram often occurs earlier in the context.
NGRAM_CONFIGS = {
    "ngram-1024x4096": dict(B=1024, L=4096, vocab=32000, span=(4, 64), p_copy=0.3, min_n=2, max_n=5, k=8, seed=31),
}


def generate_ngram(spec: dict | str, seed: int | None = None) -> dict:
    """B contexts of L tokens: spans of fresh tokens, and with probability ``p_copy`` copies
    of an earlier span of the same context."""
    if isinstance(spec, str):
        spec = NGRAM_CONFIGS[spec]
    spec = dict(spec)
    seed = spec["seed"] if seed is None else seed
    rng = np.random.default_rng(np.random.SeedSequence([seed, 9]))
    B, L = spec["B"], spec["L"]
    lo, hi = spec["span"]
    out = np.empty(B * L, np.int32)
    for r in range(B):
        ctx = np.empty(L, np.int32)
        n = 0
        while n < L:
            m = int(min(L - n, rng.integers(lo, hi + 1)))
            if n > hi and rng.random() < spec["p_copy"]:
                s = int(rng.integers(0, n - m + 1))
                ctx[n:n + m] = ctx[s:s + m]
            else:
                ctx[n:n + m] = rng.integers(0, spec["vocab"], size=m)
            n += m
        out[r * L:(r + 1) * L] = ctx
    cu = (np.arange(B + 1, dtype=np.int64) * L)
    return dict(tokens=out, cu_tokens=cu, B=B, L=L, min_n=spec["min_n"], max_n=spec["max_n"], k=spec["k"], spec=spec)
