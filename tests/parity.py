"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle, compare.

Comparison rule: accepted counts and tokens must match the oracle exactly on every
request the oracle does not flag.  A request is flagged when one of its decisions
came within the oracle's near-boundary band (acceptance within 1e-5 relative of
u * q(x*) = p(x*); the sampling threshold within 1e-5 * Z of a CDF boundary, or
within 2e-6 absolute on an explicit-q residual row), when its residual was empty, or
when a row it visited was not finite.  Flagged requests are counted, never excused
silently.  How many are flagged depends on the workload (with V = 151936 most of the
mass sits in tokens narrower than 1e-5), so the tests bound what matters: how many
flagged requests actually differ, and how close to a boundary each of them was (the
oracle's margins; the fp32 path's error is far below the band).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle
from speculative_decoding_rejection_spec_gb300 import binding


@dataclass
class Compared:
    n: int
    flagged: int
    mismatched: int        # unflagged requests that differ (must be 0)
    mismatched_flagged: int
    detail: str
    worst_margin: float    # largest oracle margin among mismatched requests (0 if none)


def dtype_code(w):
    return binding.BF16 if w["dtype"] == "bf16" else binding.F32


def run_gpu(w, debug=False, device_tensors=None, buffers=None):
    import torch
    d = device_tensors or binding.to_device(w)
    buf = buffers or binding.make_buffers(w["B"], w["T"], w["V"], dtype_code(w), d["draft_probs"] is not None)
    dbg = {} if debug else None
    if w.get("top_k") is not None or w.get("top_p") is not None:
        tk = None if w.get("top_k") is None else torch.from_numpy(w["top_k"]).cuda()
        tp = None if w.get("top_p") is None else torch.from_numpy(w["top_p"]).cuda()
        tok, acc = binding.sample_filtered(**d, top_k=tk, top_p=tp, buffers=buf, debug=dbg)
    else:
        tok, acc = binding.sample(**d, buffers=buf, debug=dbg)
    st, bits, first = binding.last_device_error(buf.workspace)
    torch.cuda.synchronize()
    out = dict(tokens=tok.cpu().numpy().copy(), acc=acc.cpu().numpy().copy(), status=st, bits=bits, first=first)
    if debug:
        out.update({k: v.cpu().numpy() for k, v in dbg.items()})
    return out


def compare(w, gpu, ref) -> Compared:
    cu = w["cu_num_draft"]
    B = w["B"]
    flagged = (ref.flags & (oracle.NEAR_ANY | oracle.NONFINITE)) != 0
    mism = 0
    mism_f = 0
    first = ""
    worst = 0.0
    for r in range(B):
        lo, hi = int(cu[r]) + r, int(cu[r + 1]) + r + 1
        same = gpu["acc"][r] == ref.num_accepted[r] and np.array_equal(gpu["tokens"][lo:hi], ref.tokens[lo:hi])
        if not same:
            if ref.margin is not None:
                m_acc, m_smp, m_topp = (float(x) for x in ref.margin[r, :3])
                if w.get("draft_probs") is not None and 0 <= ref.num_accepted[r] < cu[r + 1] - cu[r]:
                    m_smp *= float(ref.z[r])  # explicit-q residual: the fp32 error is absolute, not relative to Z
                worst = max(worst, min(m_acc, m_smp, m_topp))
            if flagged[r]:
                mism_f += 1
            else:
                mism += 1
                if not first:
                    first = (f"request {r}: gpu acc {gpu['acc'][r]} tokens {gpu['tokens'][lo:hi].tolist()} | "
                             f"oracle acc {ref.num_accepted[r]} tokens {ref.tokens[lo:hi].tolist()} "
                             f"flags {ref.flags[r]}")
    return Compared(n=B, flagged=int(flagged.sum()), mismatched=mism, mismatched_flagged=mism_f, detail=first,
                    worst_margin=worst)


# Largest relative margin at which the fp32 path may still decide differently from the
# fp64 oracle: well inside the 1e-5 band, several times the path's worst fp32 error.
MISMATCH_MARGIN = 2e-6


def assert_parity(w, gpu=None, ref=None, max_mismatch_frac=0.01):
    gpu = gpu if gpu is not None else run_gpu(w)
    ref = ref if ref is not None else oracle.reject_sample_workload(w, debug=True)
    c = compare(w, gpu, ref)
    msg = (f"{w['name']}: {c.n} requests, {c.flagged} flagged, {c.mismatched_flagged} flagged mismatches, "
           f"worst margin {c.worst_margin:.3g}")
    print(msg)
    assert c.mismatched == 0, f"{msg}; {c.mismatched} UNFLAGGED mismatches; first: {c.detail}"
    assert c.mismatched_flagged <= max(2, int(max_mismatch_frac * c.n)), msg
    assert c.worst_margin <= MISMATCH_MARGIN, msg
    return c, gpu, ref


def assert_rowstats(w, gpu, ref):
    """Per-row probabilities from the diagnostic entry point against the oracle (1e-5 relative)."""
    B, T = w["B"], w["T"]
    cu = w["cu_num_draft"]
    valid_req = ref.num_accepted >= 0
    rows = np.concatenate([np.arange(cu[r] + r, cu[r + 1] + r + 1) for r in range(B) if valid_req[r]]
                          ) if valid_req.any() else np.zeros(0, int)
    finite = np.isfinite(ref.row_max[rows])
    rows = rows[finite]
    assert np.array_equal(gpu["row_max"][rows].astype(np.float64), ref.row_max[rows]), "row max"
    assert np.array_equal(gpu["row_argmax"][rows], ref.row_argmax[rows]), "row argmax"
    s_ref = ref.row_sum[rows]
    s_gpu = gpu["row_sum"][rows].astype(np.float64)
    pos = s_ref > 0
    rel = np.abs(s_gpu[pos] / s_ref[pos] - 1)
    assert (rel <= 1e-5).all(), f"row sum: max rel err {rel.max():.3g}"
    assert (s_gpu[~pos] == 0).all()
    drows = np.concatenate([np.arange(cu[r], cu[r + 1]) for r in range(B) if valid_req[r]]
                           ) if valid_req.any() else np.zeros(0, int)
    if drows.size:
        p_ref = ref.p_draft[drows]
        p_gpu = gpu["p_draft"][drows].astype(np.float64)
        err = np.abs(p_gpu - p_ref)
        ok = err <= 1e-5 * p_ref + 1e-37
        assert ok.all(), f"p(x*): worst {np.max(err / np.maximum(p_ref, 1e-300)):.3g} rel"
    same_j = valid_req & (gpu["acc"] == ref.num_accepted)  # Z belongs to the output row j
    zr = ref.z[same_j]
    zg = gpu["z"][same_j].astype(np.float64)
    explicit = w.get("draft_probs") is not None
    tol = 1e-5 * zr + (2e-6 if explicit else 0.0)
    bad = np.abs(zg - zr) > tol
    assert not bad.any(), f"Z: gpu {zg[bad][:4]} oracle {zr[bad][:4]}"


def assert_both_paths(w, ref=None, max_mismatch_frac=0.01, rowstats=True):
    """The production call (the pass that reads rows up to each first rejection, in clusters of
    blocks for small batches) and the diagnostic call (the full pass over every row, with the
    per-row probabilities) both against the oracle, and against each other: they take every
    decision with the same arithmetic, so their outputs must be identical."""
    ref = ref if ref is not None else oracle.reject_sample_workload(w, debug=True)
    full = run_gpu(w, debug=True)
    assert full["status"] == 0 or full["status"] == 5, full["status"]
    c, _, _ = assert_parity(w, full, ref, max_mismatch_frac=max_mismatch_frac)
    if rowstats:
        assert_rowstats(w, full, ref)
    prod = run_gpu(w)
    assert prod["status"] == full["status"] and prod["bits"] == full["bits"]
    assert_parity(w, prod, ref, max_mismatch_frac=max_mismatch_frac)
    assert_same_unflagged(w, prod, full, ref)
    return c, prod, full, ref


def assert_same_unflagged(w, a, b, ref=None):
    """Two GPU runs of the same batch agree on every request the oracle does not flag.  The two
    passes take every decision with the same arithmetic except the draw's search inside the
    located chunk (the first-rejection pass sums the chunk in 256 segments by a whole block,
    the full pass in 32 segments by one warp), so they may differ only on draws the oracle
    flags as within the near-boundary band."""
    ref = ref if ref is not None else oracle.reject_sample_workload(w, debug=True)
    flagged = (ref.flags & (oracle.NEAR_ANY | oracle.NONFINITE)) != 0
    cu = w["cu_num_draft"]
    diff = []
    for r in range(w["B"]):
        lo, hi = int(cu[r]) + r, int(cu[r + 1]) + r + 1
        if a["acc"][r] != b["acc"][r] or not np.array_equal(a["tokens"][lo:hi], b["tokens"][lo:hi]):
            diff.append(r)
    bad = [r for r in diff if not flagged[r]]
    assert not bad, f"{w['name']}: the two passes differ on unflagged requests {bad[:5]}"
    return diff
