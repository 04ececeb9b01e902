"""Acceptance counters on the GPU against the oracle's counters (exact integers)."""
import numpy as np
import pytest

import oracle
from oracle import closed_forms as cf
from speculative_decoding_rejection_spec_gb300 import binding, workloads as W

import parity as PT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    import __graft_entry__ as G
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.build()
    binding.load()


def test_metrics_worked_example_and_accumulation():
    import torch
    acc = torch.tensor([4, 4, 4, 3, 3, 2, 2, 2, 1, 0], dtype=torch.int32, device="cuda")
    cu = torch.arange(0, 44, 4, dtype=torch.int32, device="cuda")
    counters = torch.zeros(binding.METRIC_COUNT, dtype=torch.int64, device="cuda")
    binding.metrics_update(cu, acc, counters)
    alpha, tau = binding.accept_rate_and_length(counters.cpu().tolist())
    assert alpha == pytest.approx(0.625) and tau == pytest.approx(3.5)
    binding.metrics_update(cu, acc, counters)  # cumulative
    c = counters.cpu().tolist()
    assert c == [2 * x for x in cf.acceptance_counters(cu.cpu().tolist(), acc.cpu().tolist())]


@pytest.mark.parametrize("name", ["deterministic", "large-128"])
def test_metrics_of_sampler_outputs_match_oracle(name):
    import torch
    w = W.generate(name)
    gpu = PT.run_gpu(w)
    ref = oracle.reject_sample_workload(w)
    counters = torch.zeros(binding.METRIC_COUNT, dtype=torch.int64, device="cuda")
    binding.metrics_update(torch.from_numpy(w["cu_num_draft"]).cuda(), torch.from_numpy(gpu["acc"]).cuda(), counters)
    got = counters.cpu().tolist()
    want = cf.acceptance_counters(w["cu_num_draft"], ref.num_accepted)
    # equal unless a flagged near-boundary draw went the other way (then within that draw's count)
    diff = np.abs(np.array(got) - np.array(want))
    assert diff.sum() <= 2 * int((gpu["acc"] != ref.num_accepted).sum()) * 33, (got, want)
    assert got == cf.acceptance_counters(w["cu_num_draft"], gpu["acc"])


@pytest.mark.parametrize("name,filters", [("deterministic", None), ("large-128", None), ("large-128", (50, 0.9)),
                                          ("greedy", None), ("tiny", None)])
def test_counters_fused_into_the_call(name, filters):
    """spec_reject_sample_ex with counters: the finalize pass adds exactly what
    spec_reject_metrics_update computes from the call's outputs (and the oracle's counters on them)."""
    import torch
    w = W.generate(name) if filters is None else W.generate(name, top_k=filters[0], top_p=filters[1])
    d = binding.to_device(w, "cuda")
    kw = {}
    if filters is not None:
        kw = dict(top_k=torch.from_numpy(w["top_k"]).cuda(), top_p=torch.from_numpy(w["top_p"]).cuda())
    fused = torch.zeros(binding.METRIC_COUNT, dtype=torch.int64, device="cuda")
    fused[:] = 7  # accumulates onto what is there
    tok, acc = binding.sample_ex(**d, counters=fused, **kw)
    separate = torch.full((binding.METRIC_COUNT,), 7, dtype=torch.int64, device="cuda")
    binding.metrics_update(d["cu_num_draft"], acc, separate)
    assert fused.cpu().tolist() == separate.cpu().tolist()
    want = [x + 7 for x in cf.acceptance_counters(w["cu_num_draft"], acc.cpu().numpy())]
    assert fused.cpu().tolist() == want
    # the same tokens as the call without counters
    ref_tok, ref_acc = binding.sample_ex(**d, **kw)
    assert torch.equal(tok, ref_tok) and torch.equal(acc, ref_acc)


def test_counters_skip_invalid_requests():
    import torch
    w = W.generate("tiny")
    ids = w["draft_ids"].copy()
    ids[0] = w["V"] + 5  # request 0 invalid
    w = dict(w, draft_ids=ids)
    d = binding.to_device(w, "cuda")
    fused = torch.zeros(binding.METRIC_COUNT, dtype=torch.int64, device="cuda")
    tok, acc = binding.sample_ex(**d, counters=fused)
    a = acc.cpu().numpy()
    assert a[0] == -1
    assert fused.cpu().tolist() == cf.acceptance_counters(w["cu_num_draft"], a)
