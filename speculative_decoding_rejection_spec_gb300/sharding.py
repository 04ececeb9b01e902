"""Splitting a batch across GPUs by contiguous request ranges.

Requests are independent, so a batch shards by request with no exchange step: each
rank takes a contiguous range of requests, whose target rows, draft rows, uniforms
and temperatures are contiguous slices of the flattened layout, and re-bases
cu_num_draft to start at 0.  Outputs concatenate back in rank order.
"""
from __future__ import annotations

import numpy as np


def request_range(B: int, rank: int, world: int) -> tuple[int, int]:
    """[r0, r1) of the requests rank `rank` of `world` handles (sizes differ by at most one)."""
    base, extra = divmod(B, world)
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


def shard_workload(w: dict, rank: int, world: int) -> dict:
    """The sub-batch of requests [r0, r1) as a workload of its own (host arrays, views where possible)."""
    cu = w["cu_num_draft"]
    r0, r1 = request_range(w["B"], rank, world)
    d0, d1 = int(cu[r0]), int(cu[r1])
    t0, t1 = d0 + r0, d1 + r1
    out = dict(w)
    out.update(name=f"{w['name']}[{r0}:{r1}]", B=r1 - r0, T=t1 - t0,
               logits=w["logits"][t0:t1], draft_ids=w["draft_ids"][d0:d1],
               draft_probs=None if w.get("draft_probs") is None else w["draft_probs"][d0:d1],
               cu_num_draft=(cu[r0:r1 + 1] - cu[r0]).astype(np.int32), uniforms=w["uniforms"][t0:t1],
               temperature=w["temperature"][r0:r1], shard=(r0, r1, t0, t1))
    return out
