"""CUDA path against the CPU oracle, element by element, through the C ABI (needs a GB300)."""
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


# ---------------------------------------------------------------------------- the five workloads

SMALL = ["tiny", "greedy", "probabilistic", "deterministic", "large-128"]


@pytest.mark.parametrize("name", SMALL)
def test_config_parity_and_rowstats(name):
    w = W.generate(name)
    c, prod, full, ref = PT.assert_both_paths(w)
    assert full["status"] == 0, full
    if name == "greedy":
        assert c.flagged == 0  # every greedy decision is an exact comparison


@pytest.mark.parametrize("name", ["large-512", "large-1024"])
def test_full_size_parity(name):
    """Full-size large-batch workloads, in the launch configuration the benchmark times."""
    w = W.generate(name)
    gpu = PT.run_gpu(w)
    assert gpu["status"] == 0
    PT.assert_parity(w, gpu, oracle.reject_sample_workload(w, debug=True))


def test_full_size_parity_with_filters():
    """The filtered benchmark's workload at full size (large-1024, top-k 50, top-p 0.9), in the
    launch configuration it times: the cut mode of the first-rejection pass."""
    w = W.generate("large-1024", top_k=50, top_p=0.9)
    assert binding.reads_to_first_rejection(w["B"], True, binding.BF16)
    gpu = PT.run_gpu(w)
    assert gpu["status"] == 0
    PT.assert_parity(w, gpu, oracle.reject_sample_workload(w, debug=True))


@pytest.mark.parametrize("name", ["greedy", "probabilistic", "deterministic", "large-128"])
def test_config_parity_unaligned_rows(name):
    """The same workloads with the logits one element off a 16-byte boundary, which sends the
    row-statistics pass through its register-staged kernel instead of the TMA ring."""
    import torch
    w = W.generate(name)
    d = binding.to_device(w)
    t = d["target_logits"]
    buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
    view = buf[1:1 + t.numel()].view(t.shape)
    view.copy_(t)
    assert view.data_ptr() % 16 != 0
    d["target_logits"] = view
    gpu = PT.run_gpu(w, device_tensors=d)
    assert gpu["status"] == 0
    PT.assert_parity(w, gpu, oracle.reject_sample_workload(w, debug=True))


def test_production_entry_matches_diagnostic_entry():
    w = W.generate("probabilistic", B=8)
    a = PT.run_gpu(w)
    b = PT.run_gpu(w, debug=True)
    PT.assert_same_unflagged(w, a, b)


def test_deterministic_repeat():
    w = W.generate("large-128")
    d = binding.to_device(w)
    a = PT.run_gpu(w, device_tensors=d)
    b = PT.run_gpu(w, device_tensors=d)
    assert np.array_equal(a["tokens"], b["tokens"]) and np.array_equal(a["acc"], b["acc"])


# ---------------------------------------------------------------------------- edge cases

def _mixed_k(B, seed):
    rng = np.random.default_rng(seed)
    k = rng.integers(0, 33, size=B)
    k[:4] = [0, 32, 0, 32]
    return k


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("draft", ["noisy_q", "target_mix"])
def test_ragged_k_zero_and_max_odd_vocab(dtype, draft):
    """k in 0..32 (k = 0 and k = 32 present), V = 5003 (odd: misaligned rows, vector tails)."""
    w = W.generate(dict(B=24, K=_mixed_k(24, 5), V=5003, dtype=dtype, sigma=1.0, temperature=1.0, draft=draft,
                        q_sigma=0.3, p_match=0.9, seed=21), name=f"ragged-{dtype}-{draft}")
    PT.assert_both_paths(w, max_mismatch_frac=0.05)


@pytest.mark.parametrize("V", [1, 7, 1001, 4096, 4097, 12289])
def test_vocab_edges(V):
    """Vocabularies from 1 to several chunks with ragged tails, both dtypes, both draft kinds."""
    for dtype in ("f32", "bf16"):
        for draft in ("noisy_q", "uniform"):
            w = W.generate(dict(B=6, K=3, V=V, dtype=dtype, sigma=1.5, temperature=0.9, draft=draft, seed=V),
                           name=f"V{V}-{dtype}-{draft}")
            PT.assert_both_paths(w, max_mismatch_frac=0.2)


def test_q_equals_p_accepts_everything():
    w = W.generate(dict(B=32, K=6, V=3000, dtype="f32", sigma=2.0, temperature=0.8, draft="target_q", seed=31),
                   name="q=p")
    w["uniforms"][:, 0] *= np.float32(0.999)  # fp32 rounding of q vs p cannot flip a decision
    c, gpu, ref = PT.assert_parity(w)
    assert (gpu["acc"] == 6).all()


def test_disjoint_supports_reject_at_zero():
    w = W.generate(dict(B=16, K=4, V=2048, dtype="f32", sigma=2.0, temperature=1.0, draft="noisy_q", seed=41),
                   name="disjoint")
    w["logits"][:, 1::2] = -np.inf
    q = np.random.default_rng(3).random(w["draft_probs"].shape)
    q[:, 0::2] = 0
    w["draft_probs"][:] = (q / q.sum(axis=1, keepdims=True)).astype(np.float32)
    w["draft_ids"][:] = np.random.default_rng(4).integers(0, 1024, size=w["draft_ids"].shape) * 2 + 1
    c, gpu, ref = PT.assert_parity(w)
    assert (gpu["acc"] == 0).all()
    assert (gpu["tokens"].reshape(16, 5)[:, 0] % 2 == 0).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_hot_target_and_masked_logits(dtype):
    w = W.generate(dict(B=20, K=5, V=3001, dtype=dtype, sigma=2.0, temperature=1.0, draft="uniform", seed=51),
                   name="masked")
    neg = np.float32(-np.inf)
    rng = np.random.default_rng(5)
    lg = W.logits_as_f32(w).copy()
    lg[rng.random(lg.shape) < 0.3] = neg          # 30 % masked tokens
    hot_rows = rng.random(lg.shape[0]) < 0.3       # some rows one-hot
    hot = rng.integers(0, 3001, size=lg.shape[0])
    lg[hot_rows] = neg
    lg[hot_rows, hot[hot_rows]] = 0.0
    # half of the drafts of one-hot rows hit the hot token
    rows = np.arange(w["T"])
    req = np.repeat(np.arange(w["B"]), 6)
    drow = rows - req
    isd = (rows - (w["cu_num_draft"][req] + req)) < 5
    sel = isd & hot_rows & (rng.random(w["T"]) < 0.5)
    w["draft_ids"][drow[sel]] = hot[sel]
    w["logits"][:] = W.f32_to_bf16_bits(lg) if dtype == "bf16" else lg
    PT.assert_both_paths(w)


def test_mixed_greedy_and_sampled_explicit_q():
    temps = np.where(np.arange(40) % 2 == 0, -1.0, 0.7)
    temps[::5] = 0.0
    w = W.generate(dict(B=40, K="ragged", K_max=8, V=7000, dtype="bf16", sigma=2.5, temperature=temps,
                        draft="noisy_q", q_sigma=0.5, seed=61), name="mixed")
    PT.assert_both_paths(w)


def test_greedy_bf16_ties_lowest_index():
    w = W.generate(dict(B=64, K=5, V=9000, dtype="bf16", sigma=1.0, temperature=0.0, draft="argmax_mix",
                        p_match=0.8, seed=71), name="ties")
    lg = np.round(W.logits_as_f32(w) * 2) / 2  # coarse values: many ties at the maximum
    w["logits"][:] = W.f32_to_bf16_bits(lg.astype(np.float32))
    am = np.argmax(lg, axis=1)
    rows = np.arange(w["T"])
    req = np.repeat(np.arange(w["B"]), 6)
    isd = (rows - (w["cu_num_draft"][req] + req)) < 5
    w["draft_ids"][:] = am[isd]
    c, prod, full, ref = PT.assert_both_paths(w)
    assert c.flagged == 0
    assert (prod["acc"] == 5).all()


def test_zero_uniforms():
    w = W.generate(dict(B=16, K=4, V=3000, dtype="f32", sigma=2.0, temperature=1.0, draft="noisy_q", seed=81),
                   name="u0")
    w["uniforms"][::3] = 0.0
    PT.assert_parity(w, max_mismatch_frac=0.05)


def test_strided_logits_rows():
    """Rows further apart than V (a padded or sliced logits buffer)."""
    import torch
    w = W.generate(dict(B=8, K=4, V=1001, dtype="bf16", sigma=2.0, temperature=0.9, draft="noisy_q", seed=91),
                   name="strided")
    d = binding.to_device(w)
    big = torch.zeros((w["T"], 1024 + 40), dtype=torch.bfloat16, device="cuda")
    big[:, 8:8 + 1001] = d["target_logits"]
    d["target_logits"] = big[:, 8:8 + 1001]
    qbig = torch.zeros((w["T"] - w["B"], 1100), dtype=torch.float32, device="cuda")
    qbig[:, 3:3 + 1001] = d["draft_probs"]
    d["draft_probs"] = qbig[:, 3:3 + 1001]
    gpu = PT.run_gpu(w, device_tensors=d)
    PT.assert_parity(w, gpu)


def test_single_request_and_empty_batch():
    import torch
    w = W.generate(dict(B=1, K=7, V=2000, dtype="f32", sigma=2.0, temperature=1.0, draft="noisy_q", seed=101),
                   name="single")
    PT.assert_parity(w)
    # B = 0, T = 0: nothing to do, no device error
    z = torch.zeros(0, device="cuda")
    e = binding.make_buffers(0, 0, 10, binding.F32, False)
    tok, acc = binding.sample(torch.zeros((0, 10), device="cuda"), torch.zeros(0, dtype=torch.int32, device="cuda"),
                              torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros((0, 2), device="cuda"),
                              z, buffers=e)
    assert binding.last_device_error(e.workspace)[0] == 0


# ---------------------------------------------------------------------------- invalid device input

def _run_raw(w):
    d = binding.to_device(w)
    buf = binding.make_buffers(w["B"], w["T"], w["V"], PT.dtype_code(w), d["draft_probs"] is not None)
    tok, acc = binding.sample(**d, buffers=buf)
    st, bits, first = binding.last_device_error(buf.workspace)
    return tok.cpu().numpy(), acc.cpu().numpy(), st, bits, first


def test_device_errors_per_request():
    w = W.generate(dict(B=5, K=[2, 33, 3, 1, 4], V=500, dtype="f32", sigma=1.0, temperature=1.0, draft="noisy_q",
                        seed=111), name="bad")
    w["draft_ids"][w["cu_num_draft"][3]] = 500  # request 3: id out of range
    ref = oracle.reject_sample_workload(w)
    tok, acc, st, bits, first = _run_raw(w)
    assert st == 5 and bits == (binding.DEVERR_SPEC_LEN | binding.DEVERR_DRAFT_ID) and first == 1
    assert acc[1] == -1 and acc[3] == -1 and (ref.num_accepted[[1, 3]] == -1).all()
    assert np.array_equal(tok, ref.tokens) and np.array_equal(acc, ref.num_accepted)


@pytest.mark.parametrize("which", ["cu0", "decreasing", "total"])
def test_device_errors_layout(which):
    w = W.generate(dict(B=4, K=3, V=300, dtype="f32", sigma=1.0, temperature=1.0, draft="uniform", seed=121),
                   name="layout")
    if which == "cu0":
        w["cu_num_draft"][0] = 1
    elif which == "decreasing":
        w["cu_num_draft"][2] = 1
    else:
        w["cu_num_draft"][-1] -= 1
    tok, acc, st, bits, first = _run_raw(w)
    assert st == 5 and bits & binding.DEVERR_LAYOUT and first == -1
    assert (acc == -1).all()
    ref = oracle.reject_sample_workload(w)
    assert ref.status == 1 and (ref.num_accepted == -1).all()


@pytest.mark.parametrize("draft", ["noisy_q", "uniform"])
def test_first_rejection_pass_device_errors_per_request(draft):
    """The same per-request errors on a batch that takes the first-rejection pass (B >= 64):
    k > 32 and an out-of-range draft id invalidate only their request; the rest match the full
    pass on every request the oracle does not flag."""
    B = 70
    ks = [3] * B
    ks[5] = 33
    w = W.generate(dict(B=B, K=ks, V=500, dtype="f32", sigma=1.0, temperature=1.0, draft=draft, seed=112),
                   name="bad-many")
    w["draft_ids"][w["cu_num_draft"][40] + 1] = -3  # request 40: id out of range
    tok, acc, st, bits, first = _run_raw(w)
    assert st == 5 and bits == (binding.DEVERR_SPEC_LEN | binding.DEVERR_DRAFT_ID) and first == 5
    assert acc[5] == -1 and acc[40] == -1
    cu = w["cu_num_draft"]
    for r in (5, 40):
        assert (tok[cu[r] + r:cu[r + 1] + r + 1] == -1).all()
    full = PT.run_gpu(w, debug=True)
    PT.assert_same_unflagged(w, dict(tokens=tok, acc=acc), full)
    # the diagnostic entry's error word holds the same per-request errors (its extra argmax
    # pass over every row does not reset it)
    assert full["status"] == 5 and full["bits"] == bits and full["first"] == 5
    ref = oracle.reject_sample_workload(w)
    assert (ref.num_accepted[[5, 40]] == -1).all()


@pytest.mark.parametrize("which", ["cu0", "decreasing", "total"])
def test_first_rejection_pass_device_errors_layout(which):
    w = W.generate(dict(B=80, K=3, V=300, dtype="f32", sigma=1.0, temperature=1.0, draft="uniform", seed=122),
                   name="layout-many")
    if which == "cu0":
        w["cu_num_draft"][0] = 1
    elif which == "decreasing":
        w["cu_num_draft"][20] = w["cu_num_draft"][19] - 1
    else:
        w["cu_num_draft"][-1] -= 1
    tok, acc, st, bits, first = _run_raw(w)
    assert st == 5 and bits & binding.DEVERR_LAYOUT and first == -1
    assert (acc == -1).all()


# ---------------------------------------------------------------------------- host-buffer entry point

def test_host_entry_matches_device_entry():
    import torch
    for name in ("tiny", "greedy"):
        w = W.generate(name)
        dev = PT.run_gpu(w)
        arena = torch.empty(binding.host_arena_size(w["B"], w["T"], w["V"], PT.dtype_code(w),
                                                    w["draft_probs"] is not None), dtype=torch.uint8, device="cuda")
        tok, acc = binding.sample_host(w["logits"], w["draft_ids"], w["cu_num_draft"], w["uniforms"],
                                       w["temperature"], w["draft_probs"], arena)
        assert np.array_equal(tok, dev["tokens"]) and np.array_equal(acc, dev["acc"])


@pytest.mark.parametrize("name", ["tiny", "large-128", "deterministic"])
def test_host_entry_reads_pinned_inputs_in_place(name):
    """Pinned inputs are read in place by the kernels: below 64 requests the draft probabilities
    (the rows the residual pass needs are staged into the arena), from 64 requests the target
    logits too (the first-rejection pass reads rows over the host link and keeps a device copy
    of exactly those rows, and of the draft row of each explicit-q rejection, for its residual
    pass and draw).  The result is the device entry's, bit for bit."""
    import torch
    w = W.generate(name)
    dev = PT.run_gpu(w)
    has_q = w["draft_probs"] is not None

    def pinned(a):
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()

    keys = ["logits", "draft_ids", "cu_num_draft", "uniforms", "temperature"] + (["draft_probs"] if has_q else [])
    host = {k: pinned(w[k]) for k in keys}
    host["out_tokens"] = torch.full((w["T"],), -7, dtype=torch.int32).pin_memory()
    host["out_num_accepted"] = torch.full((w["B"],), -7, dtype=torch.int32).pin_memory()
    ptrs = {k: v.data_ptr() for k, v in host.items()}
    dt = PT.dtype_code(w)
    arena = torch.full((binding.host_arena_size(w["B"], w["T"], w["V"], dt, has_q),), 0xA5, dtype=torch.uint8,
                       device="cuda")
    binding.sample_host_ptrs(ptrs, w["T"], w["V"], w["B"], dt, arena)
    tok, acc = host["out_tokens"].numpy(), host["out_num_accepted"].numpy()
    assert np.array_equal(tok, dev["tokens"]) and np.array_equal(acc, dev["acc"])
    # the arena holds the logits copy first, then the q copy (256-byte aligned regions)
    es = 2 if w["dtype"] == "bf16" else 4
    base = (-arena.data_ptr()) % 256
    T, B, V = w["T"], w["B"], w["V"]
    lbytes = es * T * V
    q0 = base + ((lbytes + 255) // 256) * 256
    nd = T - B
    cu = w["cu_num_draft"]
    ks = np.diff(cu)

    def rows_written(region, n, width):
        r = region.view(n, width)
        return r, set(torch.nonzero((r != 0xA5).any(dim=1)).flatten().cpu().numpy().tolist())

    def same_bytes(r, rows, src):
        idx = sorted(rows)
        want = torch.from_numpy(np.ascontiguousarray(src.view(np.uint8).reshape(len(src), -1)[idx])).cuda()
        return torch.equal(r[torch.tensor(idx, device="cuda")], want)

    # rejecting requests with explicit q (temperature > 0): their draft row at the output position
    rej = [int(cu[r]) + int(acc[r]) for r in range(B)
           if has_q and w["temperature"][r] > 0 and 0 <= acc[r] < ks[r]]
    if B >= 64:
        # exactly the target rows up to each request's output row were read (and copied)
        want = {int(cu[r]) + r + i for r in range(B) for i in range(int(acc[r]) + 1)}
        lr, got = rows_written(arena[base:base + lbytes], T, es * V)
        assert got == want, (len(got), len(want))
        assert same_bytes(lr, got, w["logits"])
        if has_q:
            qr, gq = rows_written(arena[q0:q0 + 4 * nd * V], nd, 4 * V)
            assert gq == set(rej) and same_bytes(qr, gq, w["draft_probs"])
    else:
        assert bool((arena[base:base + lbytes] != 0xA5).any())  # copied whole
        if has_q:  # only the rows for the residual pass were staged, each equal to its row of q
            qr, gq = rows_written(arena[q0:q0 + 4 * nd * V], nd, 4 * V)
            assert 0 < len(gq) <= B and gq == set(rej)
            assert same_bytes(qr, gq, w["draft_probs"])


# ---------------------------------------------------------------------------- rows read up to the first rejection

@pytest.mark.parametrize("name,over", [("tiny", dict(B=96)), ("greedy", {}), ("probabilistic", dict(B=80)),
                                       ("deterministic", {}), ("large-128", {})])
def test_first_rejection_pass_equals_full_pass(name, over):
    """Calls without cuts or diagnostics read each request's rows only up
    to its first rejection (KL); the diagnostic entry still runs the full pass over every row
    (K1, K2, K3).  Both take every decision with the same arithmetic and differ only in how the
    draw searches inside the located chunk (a block's 256 segments against a warp's 32), so the
    outputs agree on every request the oracle does not flag (fp32 and bf16 rows, explicit and
    one-hot drafts, greedy requests), and the first-rejection pass matches the oracle."""
    w = W.generate(name, **over)
    lazy = PT.run_gpu(w)
    full = PT.run_gpu(w, debug=True)
    PT.assert_same_unflagged(w, lazy, full)
    PT.assert_parity(w, lazy)


def test_first_rejection_pass_long_chains_and_counters():
    """Requests that accept every draft walk all k + 1 rows (up to 32 drafts), and the counters
    added inside the pass match the standalone update."""
    import torch
    B, K = 72, 32
    w = W.generate(dict(B=B, K=K, V=5003, dtype="bf16", sigma=2.0, temperature=0.9, draft="target_q", seed=44),
                   name="long-chains")
    lazy = PT.run_gpu(w)
    full = PT.run_gpu(w, debug=True)
    PT.assert_same_unflagged(w, lazy, full)
    PT.assert_parity(w, lazy)
    assert (lazy["acc"] == K).any()  # q = p accepts every draft
    d = binding.to_device(w, "cuda")
    ctr = torch.zeros(binding.METRIC_COUNT, dtype=torch.int64, device="cuda")
    tok, acc = binding.sample_ex(**d, counters=ctr)
    from oracle import closed_forms as cf
    assert ctr.cpu().tolist() == cf.acceptance_counters(w["cu_num_draft"], acc.cpu().numpy())


# ---------------------------------------------------------------------------- requests split over clusters

@pytest.mark.parametrize("name,over,blocks", [
    ("large-128", {}, 2),                                                   # 128 requests, 32 chunks per row
    ("probabilistic", {}, 4),                                               # 32 fp32 requests, 63 chunks
    ("wide", dict(B=24, K=4, V=262144, dtype="bf16", sigma=2.0, temperature=0.9, draft="noisy_q", q_sigma=0.7,
                  q_temperature=1.0, seed=131), 8),                         # 24 requests, 64 chunks
    ("wide-onehot", dict(B=20, K=6, V=262144, dtype="bf16", sigma=2.0, temperature=1.0, draft="target_mix",
                         p_match=0.6, seed=132), 8),
])
def test_cluster_per_request_parity(name, over, blocks):
    """Batches too small to fill the GPU one block per request split each request's rows and
    residual pass over a thread-block cluster; the outputs match the oracle and, on every request
    the oracle does not flag, the full pass."""
    import torch
    w = W.generate(name, **over) if name in W.CONFIGS else W.generate(over, name=name)
    got = binding.blocks_per_request(w["B"], w["V"], PT.dtype_code(w))
    if torch.cuda.get_device_properties(0).multi_processor_count >= 148:
        assert got == blocks, got
    PT.assert_both_paths(w, rowstats=False)


def test_first_rejection_pass_branches_b72():
    """Every branch of the first-rejection pass in one batch of 72 requests, against the oracle:
    k in 0..32 (0 and 32 present), greedy and sampled requests mixed, one-hot drafts with bf16
    rows of V = 12289 (ragged last chunk), and explicit draft probabilities with fp32 rows of
    V = 4097."""
    temps = np.where(np.arange(72) % 3 == 0, 0.0, 0.8).astype(np.float32)
    for dtype, V, draft in (("bf16", 12289, "target_mix"), ("f32", 4097, "noisy_q")):
        w = W.generate(dict(B=72, K=_mixed_k(72, 141), V=V, dtype=dtype, sigma=1.5, temperature=temps, draft=draft,
                            p_match=0.8, q_sigma=0.3, seed=142), name=f"branches-{dtype}")
        c, prod, full, ref = PT.assert_both_paths(w, max_mismatch_frac=0.05, rowstats=False)
        assert (prod["acc"][temps == 0] >= 0).all()


# ---------------------------------------------------------------------------- graph capture

@pytest.mark.parametrize("name,over", [("probabilistic", {}), ("large-128", {}), ("tiny", {}),
                                       ("greedy", dict(B=16))])
def test_call_replays_from_a_cuda_graph(name, over):
    """After one eager call on the device (which fills the launch-shape cache), the call can be
    captured into a CUDA graph (the layout check, then the first-rejection pass as a
    programmatic dependent launch, in clusters of blocks for small batches) and replayed; each
    replay gives the eager call's outputs."""
    import torch
    w = W.generate(name, **over)
    d = binding.to_device(w)
    buf = binding.make_buffers(w["B"], w["T"], w["V"], PT.dtype_code(w), d["draft_probs"] is not None)
    tok, acc = binding.sample(**d, buffers=buf)
    ref_tok, ref_acc = tok.cpu().numpy().copy(), acc.cpu().numpy().copy()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            binding.sample(**d, buffers=buf)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        buf.out_tokens.fill_(-7)
        buf.out_num_accepted.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(buf.out_tokens.cpu().numpy(), ref_tok)
        assert np.array_equal(buf.out_num_accepted.cpu().numpy(), ref_acc)
    assert binding.last_device_error(buf.workspace)[0] == 0


def test_launch_shapes():
    """The launch shape each benchmark workload takes on this GPU (host logic with the device's
    occupancy): large batches one block per request, with the last requests in a chained second
    launch of two blocks each; small batches in clusters of blocks."""
    import torch
    if torch.cuda.get_device_properties(0).multi_processor_count < 148:
        pytest.skip("shapes checked on a GB300-sized GPU")
    shapes = {}
    for name in ("large-1024", "large-512", "large-128", "probabilistic", "deterministic", "greedy", "tiny"):
        spec = W.CONFIGS[name]
        dt = binding.BF16 if spec["dtype"] == "bf16" else binding.F32
        has_q = spec["draft"] in ("noisy_q", "target_q")
        shapes[name] = (binding.blocks_per_request(spec["B"], spec["V"], dt),
                        binding.launches_per_call(spec["B"], spec["V"], has_q, False, dt))
    assert shapes["large-1024"] == (1, 3), shapes
    assert shapes["large-512"] == (1, 2) and shapes["deterministic"] == (1, 2), shapes
    assert shapes["large-128"] == (2, 2) and shapes["probabilistic"] == (4, 2), shapes
    assert shapes["greedy"] == (1, 2) and shapes["tiny"] == (1, 2), shapes
    # with top-k / top-p: bf16 batches of at least 64 requests take the first-rejection pass, large
    # ones with their last requests in a chained launch of the 16-warp build; fp32 the full pass
    cut = {n: binding.launches_per_call(W.CONFIGS[n]["B"], W.CONFIGS[n]["V"], True, True,
                                        binding.BF16 if W.CONFIGS[n]["dtype"] == "bf16" else binding.F32)
           for n in ("large-1024", "large-512", "large-128", "probabilistic")}
    assert cut == {"large-1024": 3, "large-512": 2, "large-128": 2, "probabilistic": 4}, cut
