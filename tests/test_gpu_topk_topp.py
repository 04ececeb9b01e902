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


@pytest.mark.parametrize("B", [128, 48])
def test_profiled_entry_with_filters_matches_filtered_entry(B):
    import torch
    w = W.generate("large-128", B=B, top_k=50, top_p=0.9)
    a = PT.run_gpu(w)
    dev = torch.device("cuda", 0)
    d = binding.to_device(w, dev)
    dt = binding.BF16 if w["dtype"] == "bf16" else binding.F32
    buf = binding.make_buffers(w["B"], w["T"], w["V"], dt, d["draft_probs"] is not None, dev)
    nk = binding.num_kernels(w["B"], d["draft_probs"] is not None, True, dt)
    # bf16 rows: 64 requests or more take the first-rejection pass, fewer the full pass
    assert nk == (2 if B >= 64 else 3 + (d["draft_probs"] is not None))
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


# ---------------------------------------------------------------------------- cuts in the first-rejection pass

FLAT = dict(K=6, V=32000, dtype="bf16", sigma=0.3, temperature=1.0, draft="target_mix", p_match=0.8)


@pytest.mark.parametrize("name,over,tk,tp", [
    ("large-128", {}, 50, 0.9),          # cut inside the 512-key window, explicit q
    ("large-128", {}, 0, 0.95),          # top-p alone
    ("large-128", {}, 2000, 1.0),
    ("deterministic", {}, 0, 0.9),       # one-hot drafts, ragged k
    ("deterministic", {}, 100, 0.99),
    ("greedy", {}, 5, 0.5),              # greedy requests take no cut
    # flat rows (sigma 0.3): the window's 512 keys hold about 40% of the tokens and of the mass
    (dict(FLAT, B=80, seed=61), {}, 0, 0.9),        # the top-p key lies below the window
    (dict(FLAT, B=72, seed=62), {}, 20000, 0.95),   # top-k below it too: two radix selects
    (dict(FLAT, B=64, seed=63, draft="noisy_q", q_sigma=0.3), {}, 700, 0.5),  # inside it
])
def test_first_rejection_pass_with_filters_equals_full_pass(name, over, tk, tp):
    """bf16 calls with cuts on 64 or more requests take the first-rejection pass, which cuts each
    row as it reaches it; the diagnostic entry runs the full pass (K1, K1F, K2, K3) over every
    row.  The cut key and the chunk partials come from the same integer sums, so the two
    agree on every request the oracle does not flag (the draws search inside the located chunk
    in different segment shapes), and they match the oracle."""
    w = W.generate(name, top_k=tk, top_p=tp, **over) if isinstance(name, str) else \
        W.generate(dict(name, top_k=tk, top_p=tp), name="flat-filters")
    assert binding.reads_to_first_rejection(w["B"], True, binding.BF16)
    lazy = PT.run_gpu(w)
    full = PT.run_gpu(w, debug=True)
    assert lazy["status"] == 0 and full["status"] == 0
    PT.assert_same_unflagged(w, lazy, full)
    PT.assert_parity(w, lazy)


def test_first_rejection_pass_mixed_filters_strided_rows():
    """Per-request cuts with special values, greedy requests, and rows further apart than V with
    a ragged last chunk (V not a multiple of 8, row stride a multiple of 8)."""
    import torch
    B = 96
    rng = np.random.default_rng(23)
    tk = rng.choice([0, 1, 5, 40, 7000, 20000], size=B).astype(np.int32)
    tp = rng.choice([1.0, 0.5, 0.9, 1e-6, 0.999], size=B).astype(np.float32)
    temps = np.where(np.arange(B) % 5 == 0, 0.0, 0.8).astype(np.float32)
    w = W.generate(dict(B=B, K="ragged", K_max=6, V=20011, dtype="bf16", sigma=2.0, temperature=temps,
                        draft="noisy_q", q_sigma=0.5, top_k=tk, top_p=tp, seed=29), name="mixed-filters-strided")
    d = binding.to_device(w)
    big = torch.zeros((w["T"], 20016), dtype=torch.bfloat16, device="cuda")
    big[:, :20011] = d["target_logits"]
    d["target_logits"] = big[:, :20011]
    lazy = PT.run_gpu(w, device_tensors=d)
    full = PT.run_gpu(w, debug=True, device_tensors=d)
    assert lazy["status"] == 0
    PT.assert_same_unflagged(w, lazy, full)
    PT.assert_parity(w, lazy)


def test_first_rejection_pass_with_filters_fp32_takes_full_pass():
    """fp32 rows with cuts keep the full pass (the cut in the first-rejection pass is bf16 only)."""
    assert not binding.reads_to_first_rejection(128, True, binding.F32)
    assert binding.reads_to_first_rejection(128, False, binding.F32)
    assert binding.num_kernels(128, True, True, binding.F32) == 4


def test_first_rejection_pass_with_filters_on_negative_rows():
    """Rows whose every logit is negative (the window's order keys below 0x8000 + 512, where a
    token's key offset comes from its signed magnitude), with cuts inside and below the window."""
    for seed, tk, tp in [(71, 50, 0.9), (72, 0, 0.95), (73, 20000, 1.0)]:
        w = W.generate(dict(FLAT, B=64, seed=seed, top_k=tk, top_p=tp), name="negative-rows")
        x = W.logits_as_f32(w) - np.float32(4.0)
        w["logits"] = W.f32_to_bf16_bits(x)
        assert W.logits_as_f32(w).max() < 0
        lazy = PT.run_gpu(w)
        full = PT.run_gpu(w, debug=True)
        assert lazy["status"] == 0
        PT.assert_same_unflagged(w, lazy, full)
        PT.assert_parity(w, lazy)


def test_first_rejection_pass_with_filters_device_errors_per_request():
    """k > 32 and an out-of-range draft id on a batch that takes the cut mode invalidate only their
    request (the same error word as the full pass); the rest match the full pass on every
    request the oracle does not flag."""
    B = 72
    ks = [3] * B
    ks[7] = 33
    w = W.generate(dict(B=B, K=ks, V=4096, dtype="bf16", sigma=2.0, temperature=0.9, draft="noisy_q", q_sigma=0.5,
                        top_k=20, top_p=0.8, seed=131), name="bad-cut")
    cu = w["cu_num_draft"]
    w["draft_ids"][cu[50] + 1] = w["V"] + 2
    lazy = PT.run_gpu(w)
    full = PT.run_gpu(w, debug=True)
    for g in (lazy, full):
        assert g["status"] == 5 and g["bits"] == (binding.DEVERR_SPEC_LEN | binding.DEVERR_DRAFT_ID)
        assert g["first"] == 7 and g["acc"][7] == -1 and g["acc"][50] == -1
    for r in (7, 50):
        assert (lazy["tokens"][cu[r] + r:cu[r + 1] + r + 1] == -1).all()
    PT.assert_same_unflagged(w, lazy, full)


# ---------------------------------------------------------------------------- host-buffer entry with cuts

@pytest.mark.parametrize("name,tk,tp,pinned", [
    ("large-128", 50, 0.9, True),         # bf16, 128 requests: rows read in place, each reached row cut
    ("large-128", 0, 0.95, False),        # pageable: copied, then the cut mode on the device copy
    ("deterministic", 100, 0.99, True),   # one-hot drafts
    ("probabilistic", 1000, 0.8, True),   # fp32 with cuts: logits copied, full pass with the cut kernel
])
def test_host_entry_with_filters_and_counters(name, tk, tp, pinned):
    """spec_reject_sample_host_ex: the device filtered entry's tokens and counts bit for bit, the
    acceptance counters added onto the caller's host array, and (pinned bf16, >= 64 requests)
    only the rows up to each output row copied to the arena."""
    import torch
    from oracle import closed_forms as cf
    w = W.generate(name, top_k=tk, top_p=tp)
    dev = PT.run_gpu(w)
    has_q = w["draft_probs"] is not None

    def host(a):
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        return t.pin_memory() if pinned else t.clone()

    keys = ["logits", "draft_ids", "cu_num_draft", "uniforms", "temperature", "top_k", "top_p"]
    keys += ["draft_probs"] if has_q else []
    h = {k: host(w[k]) for k in keys}
    h["out_tokens"] = torch.full((w["T"],), -7, dtype=torch.int32)
    h["out_num_accepted"] = torch.full((w["B"],), -7, dtype=torch.int32)
    h["counters"] = torch.full((binding.METRIC_COUNT,), 3, dtype=torch.int64)
    ptrs = {k: v.data_ptr() for k, v in h.items()}
    dt = PT.dtype_code(w)
    arena = torch.full((binding.host_arena_size(w["B"], w["T"], w["V"], dt, has_q),), 0xA5, dtype=torch.uint8,
                       device="cuda")
    binding.sample_host_ptrs(ptrs, w["T"], w["V"], w["B"], dt, arena)
    tok, acc = h["out_tokens"].numpy(), h["out_num_accepted"].numpy()
    assert np.array_equal(tok, dev["tokens"]) and np.array_equal(acc, dev["acc"])
    assert h["counters"].tolist() == [x + 3 for x in cf.acceptance_counters(w["cu_num_draft"], acc)]
    if pinned and w["dtype"] == "bf16" and w["B"] >= 64:
        es, T, B, V = 2, w["T"], w["B"], w["V"]
        base = (-arena.data_ptr()) % 256
        rows = arena[base:base + es * T * V].view(T, es * V)
        got = set(torch.nonzero((rows != 0xA5).any(dim=1)).flatten().cpu().numpy().tolist())
        cu = w["cu_num_draft"]
        assert got == {int(cu[r]) + r + i for r in range(B) for i in range(int(acc[r]) + 1)}


def test_first_rejection_pass_with_filters_many_tied_maxima():
    """300 tokens of the first chunk tied with each row's maximum: more than an 8-bit per-chunk
    count holds, so the cut takes the 512-key path; top-k keeps every tied token (ties kept), and
    the result is the full pass's and the oracle's."""
    w = W.generate(dict(B=64, K=3, V=8192, dtype="bf16", sigma=2.0, boost=4.0, temperature=0.8, draft="noisy_q",
                        q_sigma=0.5, top_k=50, top_p=0.9, seed=141), name="tied-maxima")
    bits = w["logits"]
    for t in range(w["T"]):
        bits[t, :300] = bits[t].view(np.int16).max()  # positive maxima: the largest bits
    assert (W.logits_as_f32(w)[:, :300] == W.logits_as_f32(w).max(axis=1, keepdims=True)).all()
    lazy = PT.run_gpu(w)
    full = PT.run_gpu(w, debug=True)
    assert lazy["status"] == 0
    PT.assert_same_unflagged(w, lazy, full)
    PT.assert_parity(w, lazy)


@pytest.mark.parametrize("tk,tp", [(20, 0.9), (0, 0.95), (3000, 1.0)])
def test_first_rejection_pass_with_filters_low_chunks(tk, tp):
    """Rows whose last six chunks lie far below the maximum (logits lowered by 20): the cut's count
    passes skip chunks whose maximum is below their window; the result is the full pass's and
    the oracle's."""
    w = W.generate(dict(B=64, K=4, V=32768, dtype="bf16", sigma=2.0, temperature=0.9, draft="noisy_q",
                        q_sigma=0.5, top_k=tk, top_p=tp, seed=151), name="low-chunks")
    x = W.logits_as_f32(w).copy()
    x[:, 2 * 4096:] -= np.float32(20.0)
    w["logits"] = W.f32_to_bf16_bits(x)
    lazy = PT.run_gpu(w)
    full = PT.run_gpu(w, debug=True)
    assert lazy["status"] == 0
    PT.assert_same_unflagged(w, lazy, full)
    PT.assert_parity(w, lazy)


@pytest.mark.gpu
def test_first_rejection_pass_with_filters_is_deterministic():
    """The same batch gives the same bits on every call, although which of the cut's windows a
    block tries first depends on the rows it happened to take before (the request queue's order
    changes from call to call): a row whose cut lies inside the widest window and keeps at most
    256 tokens always draws from its listed kept tokens, whichever window found the cut.  Per
    request cuts at several depths make the blocks' window choices differ between calls."""
    import torch
    B = 320
    rng = np.random.default_rng(41)
    tk = rng.choice([0, 20, 50, 200, 3000], size=B).astype(np.int32)
    tp = rng.choice([1.0, 0.5, 0.8, 0.9, 0.95], size=B).astype(np.float32)
    w = W.generate(dict(B=B, K=6, V=32768, dtype="bf16", sigma=2.0, boost=8.0, temperature=0.7, draft="noisy_q",
                        q_sigma=0.7, q_temperature=1.0, top_k=tk, top_p=tp, seed=43), name="mixed-depth-cuts")
    d = binding.to_device(w)
    kt, kp = torch.from_numpy(tk).cuda(), torch.from_numpy(tp).cuda()
    buf = binding.make_buffers(w["B"], w["T"], w["V"], binding.BF16, True)
    first = None
    for _ in range(6):
        tokens, acc = binding.sample_filtered(**d, top_k=kt, top_p=kp, buffers=buf)
        got = (tokens.cpu().numpy().copy(), acc.cpu().numpy().copy())
        if first is None:
            first = got
        assert np.array_equal(got[0], first[0]) and np.array_equal(got[1], first[1])
    lazy = {"tokens": first[0], "acc": first[1], "status": 0}
    PT.assert_parity(w, lazy)


@pytest.mark.gpu
def test_first_rejection_pass_with_filters_largest_vocab():
    """Cuts on rows of 530000 bf16 tokens (130 chunks: past what a kept-token list can name, so
    the output rows draw from the whole row) and of 262143 tokens (64 chunks, the most the
    128-key count takes per chunk), with top-k small enough for the kept-token draw elsewhere."""
    for V, seed in ((530000, 51), (262143, 52)):
        w = W.generate(dict(B=64, K=2, V=V, dtype="bf16", sigma=2.0, boost=8.0, temperature=0.7, draft="noisy_q",
                            q_sigma=0.7, q_temperature=1.0, top_k=20, top_p=0.9, seed=seed), name=f"cut-V{V}")
        assert binding.reads_to_first_rejection(w["B"], True)
        lazy = PT.run_gpu(w)
        assert lazy["status"] == 0
        PT.assert_parity(w, lazy)
