"""The entry point for callers that cannot allocate device memory.

Some callers of this library are not allowed to allocate: a plugin inside a host
inference engine that only receives its inputs and outputs, or a serving loop that
must not call cudaMalloc between steps.  spec_reject_sample_noalloc() runs the same
kernels with their scratch in a fixed device array inside the library.  Here it must
give exactly the results of the ordinary entry point, on two calls in a row (the
second call reuses the array the first one left behind).
"""
import numpy as np
import pytest

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


def _both(w):
    import torch
    d = binding.to_device(w)
    ref_tok, ref_acc = binding.sample(**d)
    ref_tok, ref_acc = ref_tok.clone(), ref_acc.clone()
    tok = torch.full((w["T"],), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((w["B"],), -7, dtype=torch.int32, device="cuda")
    err = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    binding.sample_noalloc(**d, out_tokens=tok, out_num_accepted=acc, device_error_word=err)
    torch.cuda.synchronize()
    return ref_tok.cpu().numpy(), ref_acc.cpu().numpy(), tok.cpu().numpy(), acc.cpu().numpy(), err.cpu().numpy()


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    # batches back to back: explicit draft probabilities (fp32 logits), one-hot drafts with a
    # mixed greedy / sampled bf16 batch, and 128 requests of the large-batch workload (rows
    # split over clusters of blocks; its queue counter lives in the shared scratch too)
    cases = [W.generate("probabilistic", B=12),
             W.generate(dict(B=40, K="ragged", K_max=8, V=20011, dtype="bf16", sigma=2.0, draft="target_mix",
                             p_match=0.7, temperature=np.where(np.arange(40) % 4 == 0, 0.0, 0.8), seed=5)),
             W.generate("large-128")]
    for w in cases:
        ref_tok, ref_acc, tok, acc, err = _both(w)
        assert np.array_equal(tok, ref_tok), w["name"]
        assert np.array_equal(acc, ref_acc), w["name"]
        assert err[0] == 0


def test_noalloc_reports_device_errors_then_clears_them():
    w = W.generate(dict(B=3, K=[1, 2, 1], V=300, dtype="f32", draft="uniform", seed=9))
    w["draft_ids"][1] = 300  # request 1: draft id out of range
    ref_tok, ref_acc, tok, acc, err = _both(w)
    assert np.array_equal(acc, ref_acc) and acc[1] == -1
    assert err[0] == binding.DEVERR_DRAFT_ID and err[1] == 1
    # the next call through the same scratch starts from a clean error word
    w2 = W.generate(dict(B=70, K=3, V=5000, dtype="bf16", sigma=2.0, temperature=0.9, draft="noisy_q", seed=10))
    ref_tok, ref_acc, tok, acc, err = _both(w2)
    assert np.array_equal(tok, ref_tok) and np.array_equal(acc, ref_acc)
    assert err[0] == 0
