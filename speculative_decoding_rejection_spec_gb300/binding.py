"""Thin ctypes binding of ``libspecreject.so`` (declared in ``include/spec_reject.h``).

Argument marshalling only: every step of the sampler runs in the library's CUDA
kernels.  Tensors must already live on the GPU (the ``*_host`` form takes host
arrays and does its own copies inside the library).  There is no CPU fallback:
if the library is missing or a call fails, these functions raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libspecreject.so")

F32, BF16 = 0, 1
MAX_SPEC_LEN = 32
DEVERR_LAYOUT, DEVERR_SPEC_LEN, DEVERR_DRAFT_ID, DEVERR_TIMEOUT, DEVERR_TREE = 1, 2, 4, 8, 16

EXPORTED = [
    "spec_reject_workspace_size", "spec_reject_sample", "spec_reject_last_device_error",
    "spec_reject_host_arena_size", "spec_reject_sample_host", "spec_reject_debug_rowstats",
    "spec_reject_status_string", "spec_reject_version", "spec_reject_sample_profiled", "spec_reject_num_kernels",
    "spec_reject_sample_noalloc", "spec_reject_metrics_update", "spec_ngram_propose",
    "spec_tree_workspace_size", "spec_tree_verify_greedy", "spec_reject_sample_filtered", "spec_reject_sample_ex",
    "spec_reject_sample_host_ex", "spec_reject_blocks_per_request", "spec_reject_launches_per_call",
]


class Options(ctypes.Structure):
    """spec_reject_options (device pointers; None = off)."""
    _fields_ = [("top_k", ctypes.c_void_p), ("top_p", ctypes.c_void_p), ("counters", ctypes.c_void_p),
                ("row_sum", ctypes.c_void_p), ("p_draft", ctypes.c_void_p)]
METRIC_NUM_DRAFTS, METRIC_NUM_DRAFT_TOKENS, METRIC_NUM_ACCEPTED_TOKENS, METRIC_NUM_VERIFIES = 0, 1, 2, 3
METRIC_ACCEPTED_PER_POS = 4
METRIC_COUNT = 4 + MAX_SPEC_LEN

_lib = None


class SpecRejectError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


def load():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBRARY):
        raise RuntimeError(f"{LIBRARY} is missing: build it with __graft_entry__.build() "
                           "(the sampler has no CPU fallback)")
    lib = ctypes.CDLL(LIBRARY)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.spec_reject_workspace_size.restype = sz
    lib.spec_reject_workspace_size.argtypes = [i32, i64, i32, ctypes.c_int, ctypes.c_int]
    sample_args = [P, ctypes.c_int, i64, i32, i64, P, i64, P, P, i32, P, P, P, P, P, sz, P]
    lib.spec_reject_sample.restype = ctypes.c_int
    lib.spec_reject_sample.argtypes = sample_args
    lib.spec_reject_debug_rowstats.restype = ctypes.c_int
    lib.spec_reject_debug_rowstats.argtypes = sample_args + [P, P, P, P, P]
    lib.spec_reject_last_device_error.restype = ctypes.c_int
    lib.spec_reject_last_device_error.argtypes = [P, P, P, P]
    lib.spec_reject_host_arena_size.restype = sz
    lib.spec_reject_host_arena_size.argtypes = [i32, i64, i32, ctypes.c_int, ctypes.c_int]
    lib.spec_reject_sample_host.restype = ctypes.c_int
    lib.spec_reject_sample_host.argtypes = [P, ctypes.c_int, i64, i32, P, P, P, i32, P, P, P, P, P, sz, P]
    lib.spec_reject_sample_host_ex.restype = ctypes.c_int
    lib.spec_reject_sample_host_ex.argtypes = [P, ctypes.c_int, i64, i32, P, P, P, i32, P, P, P, P, P, sz, P, P, P, P]
    lib.spec_reject_status_string.restype = ctypes.c_char_p
    lib.spec_reject_status_string.argtypes = [ctypes.c_int]
    lib.spec_reject_version.restype = ctypes.c_int
    lib.spec_reject_sample_profiled.restype = ctypes.c_int
    lib.spec_reject_sample_profiled.argtypes = sample_args + [P, P, P, ctypes.c_int]
    lib.spec_reject_sample_noalloc.restype = ctypes.c_int
    lib.spec_reject_sample_noalloc.argtypes = [P, ctypes.c_int, i64, i32, i64, P, i64, P, P, i32, P, P, P, P, P, P]
    lib.spec_reject_metrics_update.restype = ctypes.c_int
    lib.spec_reject_metrics_update.argtypes = [P, P, i32, P, P]
    lib.spec_ngram_propose.restype = ctypes.c_int
    lib.spec_ngram_propose.argtypes = [P, P, i32, i32, i32, i32, i64, P, P, P]
    lib.spec_tree_workspace_size.restype = sz
    lib.spec_tree_workspace_size.argtypes = [i64, i32, i32, ctypes.c_int]
    lib.spec_tree_verify_greedy.restype = ctypes.c_int
    lib.spec_tree_verify_greedy.argtypes = [P, ctypes.c_int, i64, i32, i64, P, P, P, i32, P, P, P, P, sz, P]
    lib.spec_reject_sample_filtered.restype = ctypes.c_int
    lib.spec_reject_sample_filtered.argtypes = [P, ctypes.c_int, i64, i32, i64, P, i64, P, P, i32, P, P, P, P, P, P,
                                                P, sz, P, P, P]
    lib.spec_reject_sample_ex.restype = ctypes.c_int
    lib.spec_reject_sample_ex.argtypes = sample_args + [P]
    lib.spec_reject_blocks_per_request.restype = ctypes.c_int
    lib.spec_reject_blocks_per_request.argtypes = [ctypes.c_int, ctypes.c_int32, ctypes.c_int32]
    lib.spec_reject_launches_per_call.restype = ctypes.c_int
    lib.spec_reject_launches_per_call.argtypes = [ctypes.c_int, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
                                                  ctypes.c_int]
    lib.spec_reject_num_kernels.restype = ctypes.c_int
    lib.spec_reject_num_kernels.argtypes = [ctypes.c_int, ctypes.c_int32, ctypes.c_int, ctypes.c_int]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().spec_reject_status_string(int(status)).decode()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"target logits must be float32 or bfloat16, got {t.dtype}")


def workspace_size(B: int, T: int, V: int, dtype_code: int, has_draft_probs: bool) -> int:
    n = load().spec_reject_workspace_size(int(B), int(T), int(V), int(dtype_code), int(bool(has_draft_probs)))
    if n == 0:
        raise ValueError("invalid sizes for spec_reject_workspace_size")
    return int(n)


def host_arena_size(B: int, T: int, V: int, dtype_code: int, has_draft_probs: bool) -> int:
    n = load().spec_reject_host_arena_size(int(B), int(T), int(V), int(dtype_code), int(bool(has_draft_probs)))
    if n == 0:
        raise ValueError("invalid sizes for spec_reject_host_arena_size")
    return int(n)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _row_stride(t) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit stride along the vocabulary")
    return int(t.stride(0)) if t.shape[0] > 1 else int(t.shape[1])


@dataclass
class Buffers:
    """Device buffers of one call, reusable across calls of the same shape."""
    out_tokens: object
    out_num_accepted: object
    workspace: object


def make_buffers(B: int, T: int, V: int, dtype_code: int, has_draft_probs: bool, device=None) -> Buffers:
    import torch
    dev = device if device is not None else torch.device("cuda")
    return Buffers(out_tokens=torch.empty(T, dtype=torch.int32, device=dev),
                   out_num_accepted=torch.empty(B, dtype=torch.int32, device=dev),
                   workspace=torch.empty(workspace_size(B, T, V, dtype_code, has_draft_probs), dtype=torch.uint8,
                                         device=dev))


def sample(target_logits, draft_ids, cu_num_draft, uniforms, temperature, draft_probs=None, *,
           buffers: Buffers | None = None, stream=None, debug: dict | None = None):
    """Run the rejection sampler on device tensors; returns (out_tokens [T], out_num_accepted [B]).

    target_logits: float32 / bfloat16 [T, V]; draft_probs: float32 [T - B, V] or None;
    draft_ids int32 [T - B]; cu_num_draft int32 [B + 1]; uniforms float32 [T, 2];
    temperature float32 [B].  With ``debug`` (a dict), the diagnostic entry point also
    fills debug['row_max'], ['row_sum'], ['row_argmax'], ['p_draft'], ['z'] (device tensors).
    """
    import torch
    lib = load()
    T, V = int(target_logits.shape[0]), int(target_logits.shape[1])
    B = int(cu_num_draft.shape[0]) - 1
    dt = _dtype_code(target_logits)
    if buffers is None:
        buffers = make_buffers(B, T, V, dt, draft_probs is not None, target_logits.device)
    for name, t, want in (("draft_ids", draft_ids, torch.int32), ("cu_num_draft", cu_num_draft, torch.int32),
                          ("uniforms", uniforms, torch.float32), ("temperature", temperature, torch.float32)):
        if t.dtype != want or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous {want} tensor")
    qs = 0
    if draft_probs is not None:
        if draft_probs.dtype != torch.float32:
            raise TypeError("draft_probs must be float32")
        qs = _row_stride(draft_probs)
    args = [_ptr(target_logits), dt, T, V, _row_stride(target_logits), _ptr(draft_probs), qs, _ptr(draft_ids),
            _ptr(cu_num_draft), B, _ptr(uniforms), _ptr(temperature), _ptr(buffers.out_tokens),
            _ptr(buffers.out_num_accepted), _ptr(buffers.workspace), int(buffers.workspace.numel()),
            _stream(stream)]
    if debug is None:
        st = lib.spec_reject_sample(*args)
        what = "spec_reject_sample"
    else:
        dev = target_logits.device
        debug.update(row_max=torch.full((T,), float("nan"), device=dev),
                     row_sum=torch.full((T,), float("nan"), device=dev),
                     row_argmax=torch.full((T,), -1, dtype=torch.int32, device=dev),
                     p_draft=torch.full((max(T - B, 0),), float("nan"), device=dev),
                     z=torch.full((B,), float("nan"), device=dev))
        st = lib.spec_reject_debug_rowstats(*args, _ptr(debug["row_max"]), _ptr(debug["row_sum"]),
                                            _ptr(debug["row_argmax"]), _ptr(debug["p_draft"]), _ptr(debug["z"]))
        what = "spec_reject_debug_rowstats"
    if st != 0:
        raise SpecRejectError(st, what)
    return buffers.out_tokens, buffers.out_num_accepted


def sample_profiled(d: dict, buffers: Buffers, events: list, stream=None, top_k=None, top_p=None):
    """``sample`` plus CUDA events recorded between the kernels (see spec_reject_sample_profiled).

    ``events`` are torch.cuda.Event(enable_timing=True) objects that have been recorded once
    (so that their handles exist).  ``top_k`` / ``top_p`` are optional device tensors as in
    ``sample_filtered``.
    """
    lib = load()
    t = d["target_logits"]
    T, V = int(t.shape[0]), int(t.shape[1])
    B = int(d["cu_num_draft"].shape[0]) - 1
    q = d.get("draft_probs")
    handles = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    st = lib.spec_reject_sample_profiled(
        _ptr(t), _dtype_code(t), T, V, _row_stride(t), _ptr(q), 0 if q is None else _row_stride(q),
        _ptr(d["draft_ids"]), _ptr(d["cu_num_draft"]), B, _ptr(d["uniforms"]), _ptr(d["temperature"]),
        _ptr(buffers.out_tokens), _ptr(buffers.out_num_accepted), _ptr(buffers.workspace),
        int(buffers.workspace.numel()), _stream(stream), _ptr(top_k), _ptr(top_p), handles, len(events))
    if st != 0:
        raise SpecRejectError(st, "spec_reject_sample_profiled")


def sample_noalloc(target_logits, draft_ids, cu_num_draft, uniforms, temperature, draft_probs=None, *,
                   out_tokens, out_num_accepted, device_error_word=None, stream=None):
    """``sample`` without a workspace: the library's fixed device scratch array is used.

    For callers that cannot allocate device memory.  The caller still provides the
    outputs (and optionally a device int32[2] for the error word).  Calls that overlap
    on the GPU share the one scratch array and race.
    """
    T, V = int(target_logits.shape[0]), int(target_logits.shape[1])
    B = int(cu_num_draft.shape[0]) - 1
    q = draft_probs
    st = load().spec_reject_sample_noalloc(
        _ptr(target_logits), _dtype_code(target_logits), T, V, _row_stride(target_logits), _ptr(q),
        0 if q is None else _row_stride(q), _ptr(draft_ids), _ptr(cu_num_draft), B, _ptr(uniforms),
        _ptr(temperature), _ptr(out_tokens), _ptr(out_num_accepted), _ptr(device_error_word), _stream(stream))
    if st != 0:
        raise SpecRejectError(st, "spec_reject_sample_noalloc")
    return out_tokens, out_num_accepted


def metrics_update(cu_num_draft, out_num_accepted, counters, stream=None):
    """Accumulate one call's acceptance counters into ``counters`` (device int64 [METRIC_COUNT])."""
    B = int(cu_num_draft.shape[0]) - 1
    st = load().spec_reject_metrics_update(_ptr(cu_num_draft), _ptr(out_num_accepted), B, _ptr(counters),
                                           _stream(stream))
    if st != 0:
        raise SpecRejectError(st, "spec_reject_metrics_update")
    return counters


def accept_rate_and_length(counters) -> tuple[float, float]:
    """(alpha, tau) from accumulated counters (host copy)."""
    c = [int(x) for x in counters]
    return (c[METRIC_NUM_ACCEPTED_TOKENS] / max(c[METRIC_NUM_DRAFT_TOKENS], 1),
            (c[METRIC_NUM_ACCEPTED_TOKENS] + c[METRIC_NUM_VERIFIES]) / max(c[METRIC_NUM_VERIFIES], 1))


def ngram_propose(tokens, cu_tokens, min_n: int, max_n: int, k: int, max_model_len: int = 0, stream=None,
                  out=None, num=None):
    """n-gram draft proposals for a batch of contexts (device int32 tokens, int64 offsets [B + 1]).

    Returns (drafts int32 [B, k] padded with -1, counts int32 [B]); ``out`` / ``num`` may be
    given to reuse device buffers.
    """
    import torch
    B = int(cu_tokens.shape[0]) - 1
    if out is None:
        out = torch.empty((B, k), dtype=torch.int32, device=tokens.device)
    if num is None:
        num = torch.empty(B, dtype=torch.int32, device=tokens.device)
    st = load().spec_ngram_propose(_ptr(tokens), _ptr(cu_tokens), B, int(min_n), int(max_n), int(k),
                                   int(max_model_len), _ptr(out), _ptr(num), _stream(stream))
    if st != 0:
        raise SpecRejectError(st, "spec_ngram_propose")
    return out, num


def tree_verify_greedy(target_logits, parent, node_tokens, cu_nodes, stream=None, buffers=None):
    """Greedy tree verification on device tensors.

    Returns (out_tokens [N], out_num_accepted [B], out_last_node [B], workspace); passing that
    tuple back as ``buffers`` reuses it.
    """
    import torch
    N, V = int(target_logits.shape[0]), int(target_logits.shape[1])
    B = int(cu_nodes.shape[0]) - 1
    dt = _dtype_code(target_logits)
    dev = target_logits.device
    n_ws = load().spec_tree_workspace_size(N, B, V, dt)
    if n_ws == 0:
        raise ValueError("invalid sizes for spec_tree_workspace_size")
    if buffers is not None:
        out, acc, last, ws = buffers
    else:
        ws = torch.empty(n_ws, dtype=torch.uint8, device=dev)
        out = torch.empty(N, dtype=torch.int32, device=dev)
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        last = torch.empty(B, dtype=torch.int32, device=dev)
    st = load().spec_tree_verify_greedy(_ptr(target_logits), dt, N, V, _row_stride(target_logits), _ptr(parent),
                                        _ptr(node_tokens), _ptr(cu_nodes), B, _ptr(out), _ptr(acc), _ptr(last),
                                        _ptr(ws), n_ws, _stream(stream))
    if st != 0:
        raise SpecRejectError(st, "spec_tree_verify_greedy")
    return out, acc, last, ws


def num_kernels(B: int, has_draft_probs: bool, has_filters: bool = False, dtype: int = BF16) -> int:
    """Kernels one call of B requests launches (16-byte-aligned rows in device memory)."""
    return int(load().spec_reject_num_kernels(int(dtype), int(B), int(bool(has_draft_probs)),
                                              int(bool(has_filters))))


def blocks_per_request(B: int, V: int, dtype: int = BF16) -> int:
    """Blocks (a thread-block cluster) per request of an unfiltered call on the current device."""
    return int(load().spec_reject_blocks_per_request(int(dtype), int(B), int(V)))


def launches_per_call(B: int, V: int, has_draft_probs: bool, has_filters: bool = False, dtype: int = BF16) -> int:
    """Kernel launches of one call on the current device (stages, plus the chained second launch of
    the first-rejection pass for large batches)."""
    return int(load().spec_reject_launches_per_call(int(dtype), int(B), int(V), int(bool(has_draft_probs)),
                                                    int(bool(has_filters))))


def reads_to_first_rejection(B: int, has_filters: bool = False, dtype: int = BF16) -> bool:
    """Whether a call of B requests takes the pass that reads rows up to each first rejection."""
    return all(int(load().spec_reject_num_kernels(int(dtype), int(B), q, int(bool(has_filters)))) == 2
               for q in (0, 1))


def sample_filtered(target_logits, draft_ids, cu_num_draft, uniforms, temperature, draft_probs=None, *,
                    top_k=None, top_p=None, buffers: Buffers | None = None, stream=None, debug: dict | None = None):
    """``sample`` with per-request top-k (int32 [B]) / top-p (float32 [B]) on the target; either may be None.

    With ``debug`` (a dict) also fills debug['row_sum'] (restricted normaliser per row) and
    debug['p_draft'] (p'(x*) per draft row).
    """
    import torch
    T, V = int(target_logits.shape[0]), int(target_logits.shape[1])
    B = int(cu_num_draft.shape[0]) - 1
    dt = _dtype_code(target_logits)
    if buffers is None:
        buffers = make_buffers(B, T, V, dt, draft_probs is not None, target_logits.device)
    qs = 0 if draft_probs is None else _row_stride(draft_probs)
    rs = pdr = None
    if debug is not None:
        rs = torch.full((T,), float("nan"), device=target_logits.device)
        pdr = torch.full((max(T - B, 0),), float("nan"), device=target_logits.device)
        debug.update(row_sum=rs, p_draft=pdr)
    st = load().spec_reject_sample_filtered(
        _ptr(target_logits), dt, T, V, _row_stride(target_logits), _ptr(draft_probs), qs, _ptr(draft_ids),
        _ptr(cu_num_draft), B, _ptr(uniforms), _ptr(temperature), _ptr(top_k), _ptr(top_p),
        _ptr(buffers.out_tokens), _ptr(buffers.out_num_accepted), _ptr(buffers.workspace),
        int(buffers.workspace.numel()), _stream(stream), _ptr(rs), _ptr(pdr))
    if st != 0:
        raise SpecRejectError(st, "spec_reject_sample_filtered")
    return buffers.out_tokens, buffers.out_num_accepted


def sample_ex(target_logits, draft_ids, cu_num_draft, uniforms, temperature, draft_probs=None, *, top_k=None,
              top_p=None, counters=None, buffers: Buffers | None = None, stream=None, debug: dict | None = None):
    """``sample`` with options: top-k / top-p as ``sample_filtered`` and ``counters`` (device int64
    [METRIC_COUNT]) to which this call's acceptance counters are added inside the finalize pass."""
    import torch
    T, V = int(target_logits.shape[0]), int(target_logits.shape[1])
    B = int(cu_num_draft.shape[0]) - 1
    dt = _dtype_code(target_logits)
    if buffers is None:
        buffers = make_buffers(B, T, V, dt, draft_probs is not None, target_logits.device)
    qs = 0 if draft_probs is None else _row_stride(draft_probs)
    rs = pdr = None
    if debug is not None:
        rs = torch.full((T,), float("nan"), device=target_logits.device)
        pdr = torch.full((max(T - B, 0),), float("nan"), device=target_logits.device)
        debug.update(row_sum=rs, p_draft=pdr)
    opts = Options(_ptr(top_k), _ptr(top_p), _ptr(counters), _ptr(rs), _ptr(pdr))
    st = load().spec_reject_sample_ex(
        _ptr(target_logits), dt, T, V, _row_stride(target_logits), _ptr(draft_probs), qs, _ptr(draft_ids),
        _ptr(cu_num_draft), B, _ptr(uniforms), _ptr(temperature), _ptr(buffers.out_tokens),
        _ptr(buffers.out_num_accepted), _ptr(buffers.workspace), int(buffers.workspace.numel()), _stream(stream),
        ctypes.byref(opts))
    if st != 0:
        raise SpecRejectError(st, "spec_reject_sample_ex")
    return buffers.out_tokens, buffers.out_num_accepted


def last_device_error(workspace, stream=None):
    """(status, error_bits, first_bad_request) of the last call that used ``workspace`` (synchronises)."""
    bits = ctypes.c_int32(0)
    first = ctypes.c_int32(0)
    st = load().spec_reject_last_device_error(_ptr(workspace), _stream(stream), ctypes.byref(bits),
                                              ctypes.byref(first))
    if st not in (0, 5):
        raise SpecRejectError(st, "spec_reject_last_device_error")
    return int(st), int(bits.value), int(first.value)


def sample_host(logits: np.ndarray, draft_ids: np.ndarray, cu_num_draft: np.ndarray, uniforms: np.ndarray,
                temperature: np.ndarray, draft_probs: np.ndarray | None, arena, *, out_tokens: np.ndarray | None = None,
                out_num_accepted: np.ndarray | None = None, stream=None):
    """Host-buffer entry point: host arrays in, host arrays out; copies happen inside the library.

    ``logits`` is float32 or uint16 (bf16 bits) [T, V], C-contiguous (pinned memory copies fastest);
    ``arena`` a device tensor of at least ``host_arena_size`` bytes.
    """
    T, V = logits.shape
    B = cu_num_draft.shape[0] - 1
    dt = BF16 if logits.dtype == np.uint16 else F32
    for a in (logits, draft_ids, cu_num_draft, uniforms, temperature) + (() if draft_probs is None else (draft_probs,)):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("host arrays must be C-contiguous")
    if out_tokens is None:
        out_tokens = np.empty(T, np.int32)
    if out_num_accepted is None:
        out_num_accepted = np.empty(B, np.int32)
    hp = lambda a: None if a is None else ctypes.c_void_p(a.ctypes.data)
    st = load().spec_reject_sample_host(hp(logits), dt, T, V, hp(draft_probs), hp(draft_ids), hp(cu_num_draft), B,
                                        hp(uniforms), hp(temperature), hp(out_tokens), hp(out_num_accepted),
                                        _ptr(arena), int(arena.numel()), _stream(stream))
    if st != 0:
        raise SpecRejectError(st, "spec_reject_sample_host")
    return out_tokens, out_num_accepted


def sample_host_ptrs(ptrs: dict, T: int, V: int, B: int, dtype_code: int, arena, stream=None):
    """Same as ``sample_host`` but with raw host addresses (e.g. of pinned torch tensors).

    Optional ``ptrs`` keys ``top_k`` (int32 [B]), ``top_p`` (float32 [B]) and ``counters``
    (int64 [METRIC_COUNT], added to) take ``spec_reject_sample_host_ex``."""
    base = (ptrs["logits"], dtype_code, T, V, ptrs.get("draft_probs"), ptrs["draft_ids"], ptrs["cu_num_draft"], B,
            ptrs["uniforms"], ptrs["temperature"], ptrs["out_tokens"], ptrs["out_num_accepted"], _ptr(arena),
            int(arena.numel()), _stream(stream))
    if any(ptrs.get(k) is not None for k in ("top_k", "top_p", "counters")):
        st = load().spec_reject_sample_host_ex(*base, ptrs.get("top_k"), ptrs.get("top_p"), ptrs.get("counters"))
        what = "spec_reject_sample_host_ex"
    else:
        st = load().spec_reject_sample_host(*base)
        what = "spec_reject_sample_host"
    if st != 0:
        raise SpecRejectError(st, what)


def to_device(w: dict, device="cuda"):
    """Copy a synthetic workload (host numpy arrays) to device tensors for ``sample``."""
    import torch
    dev = torch.device(device)
    if w["dtype"] == "bf16":
        logits = torch.from_numpy(w["logits"].view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        logits = torch.from_numpy(w["logits"]).to(dev)
    q = None if w.get("draft_probs") is None else torch.from_numpy(w["draft_probs"]).to(dev)
    return dict(target_logits=logits, draft_probs=q,
                draft_ids=torch.from_numpy(w["draft_ids"]).to(dev),
                cu_num_draft=torch.from_numpy(w["cu_num_draft"]).to(dev),
                uniforms=torch.from_numpy(w["uniforms"]).to(dev),
                temperature=torch.from_numpy(w["temperature"]).to(dev))
