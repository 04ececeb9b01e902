"""Multi-process (gloo, world size 2, CPU) check of the request sharding used for N > 1.

Each rank runs the CPU oracle on its contiguous range of requests; the gathered shard
results must equal the unsharded run exactly (requests are independent, nothing is
exchanged on the data path).
"""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_rejection_spec_gb300 import sharding, workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, spec, q):
    import torch
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.generate(spec)
    part = sharding.shard_workload(w, rank, world)
    res = oracle.reject_sample_workload(part)
    tok = [None] * world
    acc = [None] * world
    dist.all_gather_object(tok, res.tokens.tolist())
    dist.all_gather_object(acc, res.num_accepted.tolist())
    t = torch.tensor([float(part["T"])])
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    if rank == 0:
        q.put((sum(tok, []), sum(acc, []), float(t.item())))
    dist.barrier()
    dist.destroy_process_group()


def test_request_range_partition():
    for B in (0, 1, 5, 64, 1023):
        for world in (1, 2, 3, 8):
            spans = [sharding.request_range(B, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == B
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def test_sharded_oracle_equals_unsharded_world2():
    import oracle
    spec = dict(B=37, K="ragged", K_max=6, V=3001, dtype="bf16", sigma=2.0, temperature=0.9, draft="noisy_q",
                q_sigma=0.5, seed=77)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world = 2
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, spec, q)) for r in range(world)]
    for p in procs:
        p.start()
    tok, acc, T = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = W.generate(spec)
    ref = oracle.reject_sample_workload(w)
    assert T == w["T"]
    assert np.array_equal(np.array(tok, np.int32), ref.tokens)
    assert np.array_equal(np.array(acc, np.int32), ref.num_accepted)
