"""Top-k / top-p on the target distribution: CUDA path against the oracle."""
import numpy as np
import pytest

import oracle
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


def _check(w, max_mismatch_frac=0.01):
    ref = oracle.reject_sample_workload(w, debug=True)
    gpu = PT.run_gpu(w, debug=True)
    assert gpu["status"] == 0
    c, _, _ = PT.assert_parity(w, gpu, ref, max_mismatch_frac=max_mismatch_frac)
    # restricted normaliser and p'(x*) within 1e-5 relative on sampled rows
    B = w["B"]
    cu = w["cu_num_draft"]
    # sampled requests whose top-p cut was not a near-boundary decision (a cut one token apart
    # changes the normaliser by that token's mass)
    samp = [r for r in range(B) if w["temperature"][r] > 0 and ref.num_accepted[r] >= 0
            and not (ref.flags[r] & oracle.NEAR_TOPP)]
    rows = np.concatenate([np.arange(cu[r] + r, cu[r + 1] + r + 1) for r in samp]) if samp else np.zeros(0, int)
    s_ref, s_gpu = ref.row_sum[rows], gpu["row_sum"][rows].astype(np.float64)
    assert np.all(np.abs(s_gpu / s_ref - 1) <= 1e-5), np.max(np.abs(s_gpu / s_ref - 1))
    drows = np.concatenate([np.arange(cu[r], cu[r + 1]) for r in samp]) if samp else np.zeros(0, int)
    p_ref, p_gpu = ref.p_draft[drows], gpu["p_draft"][drows].astype(np.float64)
    assert np.all(np.abs(p_gpu - p_ref) <= 1e-5 * p_ref + 1e-37)
    return c, gpu, ref


@pytest.mark.parametrize("name,tk,tp", [
    ("large-128", 50, 0.9), ("large-128", 0, 0.95), ("large-128", 2000, 1.0),
    ("deterministic", 0, 0.9), ("deterministic", 100, 0.99),
    ("probabilistic", 1000, 0.8), ("tiny", 20, 0.7), ("greedy", 5, 0.5),
])
def test_configs_with_filters(name, tk, tp):
    w = W.generate(name, top_k=tk, top_p=tp)
    _check(w)


def test_mixed_per_request_filters_and_special_values():
    B = 48
    rng = np.random.default_rng(5)
    tk = rng.choice([0, 1, 5, 40, 7000, 20000], size=B).astype(np.int32)
    tp = rng.choice([1.0, 0.5, 0.9, 1e-6, 0.999], size=B).astype(np.float32)
    temps = np.where(np.arange(B) % 5 == 0, 0.0, 0.8).astype(np.float32)
    w = W.generate(dict(B=B, K="ragged", K_max=6, V=20011, dtype="bf16", sigma=2.0, temperature=temps,
                        draft="noisy_q", q_sigma=0.5, top_k=tk, top_p=tp, seed=17), name="mixed-filters")
    c, gpu, ref = _check(w)
    # top-k = 1 (or a tiny top-p) keeps only the maximum (all tokens tied with it): the drawn
    # token of those sampled requests carries the row maximum
    lg = W.logits_as_f32(w)
    cu = w["cu_num_draft"]
    for r in range(B):
        if w["temperature"][r] > 0 and (tk[r] == 1 or tp[r] < 1e-3):
            t = cu[r] + r + gpu["acc"][r]
            assert lg[t, gpu["tokens"][t]] == lg[t].max()


def test_filters_off_give_the_unfiltered_result():
    w = W.generate("large-128")
    a = PT.run_gpu(w)
    w2 = dict(w, top_k=np.zeros(w["B"], np.int32), top_p=np.ones(w["B"], np.float32))
    b = PT.run_gpu(w2)
    assert np.array_equal(a["tokens"], b["tokens"]) and np.array_equal(a["acc"], b["acc"])


def test_profiled_entry_with_filters_matches_filtered_entry():
    import torch
    w = W.generate("large-128", top_k=50, top_p=0.9)
    a = PT.run_gpu(w)
    dev = torch.device("cuda", 0)
    d = binding.to_device(w, dev)
    dt = binding.BF16 if w["dtype"] == "bf16" else binding.F32
    buf = binding.make_buffers(w["B"], w["T"], w["V"], dt, d["draft_probs"] is not None, dev)
    nk = binding.num_kernels(w["B"], d["draft_probs"] is not None, True)
    assert nk == 3 + (d["draft_probs"] is not None)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
    stream = torch.cuda.current_stream()
    for e in ev:
        e.record(stream)
    binding.sample_profiled(d, buf, ev, stream, torch.from_numpy(w["top_k"]).to(dev),
                            torch.from_numpy(w["top_p"]).to(dev))
    torch.cuda.synchronize()
    assert np.array_equal(buf.out_tokens.cpu().numpy(), a["tokens"])
    assert np.array_equal(buf.out_num_accepted.cpu().numpy(), a["acc"])
    assert all(ev[i].elapsed_time(ev[i + 1]) >= 0 for i in range(nk))
