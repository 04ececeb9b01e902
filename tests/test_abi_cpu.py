"""The C-ABI library without a GPU: it loads, exports every declared symbol, and its
host-side checks reject bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import __graft_entry__ as G
from speculative_decoding_rejection_spec_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_reject.h")


@pytest.fixture(scope="module")
def lib():
    G.build()
    return binding.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_(?:reject|ngram|tree)_\w+)\s*\(", src)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    assert set(binding.EXPORTED) <= set(names), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"


def test_status_strings(lib):
    for st in range(7):
        assert binding.status_string(st)
    assert binding.status_string(3) == "workspace too small"
    assert lib.spec_reject_version() >= 100


def test_workspace_size_monotone_and_rejects_bad_sizes(lib):
    small = binding.workspace_size(4, 16, 1000, binding.F32, True)
    big = binding.workspace_size(1024, 9216, 128256, binding.BF16, True)
    assert 0 < small < big
    assert binding.workspace_size(1024, 9216, 128256, binding.BF16, False) <= big
    for bad in [(-1, 4, 10), (1, -1, 10), (1, 1, 0), (1, 1, 2 ** 21)]:
        assert lib.spec_reject_workspace_size(bad[0], bad[1], bad[2], 0, 0) == 0


def _call(lib, **kw):
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: the host checks fail first
    args = dict(logits=fake, dtype=0, T=8, V=100, stride=100, q=None, qstride=0, ids=fake, cu=fake, B=2,
                uni=fake, temp=fake, tok=fake, acc=fake, ws=fake, wsb=1 << 20, stream=None)
    args.update(kw)
    return lib.spec_reject_sample(args["logits"], args["dtype"], args["T"], args["V"], args["stride"], args["q"],
                                  args["qstride"], args["ids"], args["cu"], args["B"], args["uni"], args["temp"],
                                  args["tok"], args["acc"], args["ws"], args["wsb"], args["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(logits=None), 1), (dict(cu=None), 1), (dict(ws=None), 1), (dict(ids=None), 1), (dict(uni=None), 1),
    (dict(temp=None), 1), (dict(tok=None), 1), (dict(acc=None), 1),
    (dict(dtype=7), 1), (dict(V=0), 1), (dict(T=1, B=2), 1), (dict(B=-1), 1), (dict(stride=50), 1),
    (dict(q=ctypes.c_void_p(4096), qstride=10), 1), (dict(V=2 ** 21, stride=2 ** 21), 2),
    (dict(logits=ctypes.c_void_p(4098)), 1), (dict(cu=ctypes.c_void_p(4098)), 1),
    (dict(wsb=16), 3),
])
def test_host_checks(lib, kw, status):
    assert _call(lib, **kw) == status


def test_host_entry_checks(lib):
    P = ctypes.c_void_p
    fake = P(4096)
    st = lib.spec_reject_sample_host(fake, 0, 8, 100, None, fake, fake, 2, fake, fake, fake, fake, fake, 16, None)
    assert st == 3
    st = lib.spec_reject_sample_host(fake, 0, 8, 100, None, fake, None, 2, fake, fake, fake, fake, fake, 1 << 30,
                                     None)
    assert st == 1
    assert lib.spec_reject_last_device_error(None, None, None, None) == 1


def test_kernel_counts_per_call_kind(lib):
    """Which pass a call takes, from the host logic alone: without top-k / top-p every batch of
    at least one request takes the first-rejection pass (2 launches); with them, 64 or more
    requests on bf16 rows; otherwise the full pass (K1, K2, plus the cut with filters, plus the
    residual pass with draft probabilities)."""
    for dt in (binding.F32, binding.BF16):
        for q in (False, True):
            assert binding.num_kernels(64, q, False, dt) == 2
            assert binding.num_kernels(1, q, False, dt) == 2
            assert binding.num_kernels(0, q, False, dt) == 2 + q
            assert binding.num_kernels(0, q, True, dt) == 3 + q
            assert binding.num_kernels(63, q, True, dt) == 3 + q
        assert binding.reads_to_first_rejection(1024, False, dt)
        assert binding.reads_to_first_rejection(1, False, dt)
        assert not binding.reads_to_first_rejection(63, True, dt)
    assert binding.num_kernels(64, True, True, binding.BF16) == 2
    assert binding.num_kernels(64, True, True, binding.F32) == 4
    assert binding.reads_to_first_rejection(64, True, binding.BF16)
    assert not binding.reads_to_first_rejection(64, True, binding.F32)


def test_host_arena_size(lib):
    """The host-buffer entry's arena holds a logits region, a q region, the small arrays and the
    sampler's workspace; it grows with each of them and rejects bad sizes."""
    a = binding.host_arena_size(1024, 9216, 128256, binding.BF16, True)
    b = binding.host_arena_size(1024, 9216, 128256, binding.BF16, False)
    c = binding.host_arena_size(1024, 9216, 128256, binding.F32, True)
    assert a > 2 * 9216 * 128256 + 4 * 8192 * 128256
    assert b < a < c
    assert b >= 2 * 9216 * 128256 + binding.workspace_size(1024, 9216, 128256, binding.BF16, False)
    assert lib.spec_reject_host_arena_size(-1, 4, 10, 0, 0) == 0


def test_host_entry_with_options_checks(lib):
    """spec_reject_sample_host_ex rejects what spec_reject_sample_host rejects, before any copy."""
    P = ctypes.c_void_p
    fake = P(4096)
    args = [fake, 0, 8, 100, None, fake, fake, 2, fake, fake, fake, fake, fake]
    assert lib.spec_reject_sample_host_ex(*args, 16, None, fake, fake, fake) == 3  # arena too small
    bad = list(args)
    bad[6] = None  # cu_num_draft
    assert lib.spec_reject_sample_host_ex(*bad, 1 << 30, None, None, None, None) == 1


def test_noalloc_capacity_and_oversized_batches(lib):
    """The fixed scratch of spec_reject_sample_noalloc holds the workspace of 3376 requests of
    K = 8 drafts over V = 128256 bf16 logits with draft probabilities (30384 target rows), and
    not of one request more; a larger batch is refused with SPEC_ERR_WORKSPACE after the
    argument checks and before any CUDA call (no device needed)."""
    cap = 8 << 20
    size = lambda B: lib.spec_reject_workspace_size(B, 9 * B, 128256, binding.BF16, 1)
    assert size(3376) <= cap < size(3377)
    fake = ctypes.c_void_p(4096)
    for B in (3377, 40000):
        st = lib.spec_reject_sample_noalloc(fake, binding.BF16, 9 * B, 128256, 128256, fake, 128256, fake, fake, B,
                                            fake, fake, fake, fake, None, None)
        assert st == 3 and binding.status_string(st) == "workspace too small"
    # argument errors come first, as in spec_reject_sample
    st = lib.spec_reject_sample_noalloc(None, binding.BF16, 9 * 40000, 128256, 128256, None, 0, None, None, 40000,
                                        None, None, None, None, None, None)
    assert st == lib.spec_reject_sample(None, binding.BF16, 9 * 40000, 128256, 128256, None, 0, None, None, 40000,
                                        None, None, None, None, None, 0, None) == 1
    st = lib.spec_reject_sample_noalloc(fake, binding.BF16, 8, 2000000, 2000000, None, 0, fake, fake, 2,
                                        fake, fake, fake, fake, None, None)
    assert st == 2  # V above SPEC_REJECT_MAX_VOCAB: unsupported, as spec_reject_sample reports it
