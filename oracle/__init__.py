"""Plain fp64 CPU oracle of the verify-side rejection sampler.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product library never
loads it, and the oracle shares no code with the CUDA path: its arithmetic lives
in ``reject_oracle.c`` (double precision, libm ``exp``, sums in index order) and
its closed forms in ``closed_forms.py``.

The method it follows is the speculative-sampling acceptance rule of
"第12章 投机解码：以小博大" §12.2.1 (accept x* with probability min(1, p/q), resample
the recovered token from max(0, p - q) on rejection), the bonus token of §12.3.2,
the one-hot draft of §12.2.3 / §12.9 and the greedy degenerate form of §12.2.4.
Every function of ``reject_oracle.c`` cites the passage it implements.

Parity status: every part of the oracle is pinned by tests that do not re-type
its formulas (``tests/test_oracle_pins.py``): a chi-square test of the output
distribution, the acceptance rate against A = sum min(p, q), the residual-mass
identity, the accepted-length closed form, exact enumeration of outcomes on tiny
vocabularies, library-routine special cases and the pages' worked examples; and
``tests/test_oracle_mutants.py`` shows that plausible mistakes planted in a copy
of the oracle fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "reject_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

# Per-request flags (the OF_* values of reject_oracle.c).
NEAR_ACCEPT = 1
NEAR_SAMPLE = 2
NEAR_SAMPLE_ABS = 4
DEGENERATE = 8
BAD_INPUT = 16
NONFINITE = 32
NEAR_TOPP = 64
NEAR_ANY = NEAR_ACCEPT | NEAR_SAMPLE | NEAR_SAMPLE_ABS | DEGENERATE | NEAR_TOPP

MAX_SPEC_LEN = 32


def build(force: bool = False, src: str = SOURCE, out: str = LIBRARY) -> str:
    """Compile the oracle source into a shared library with gcc.

    OpenMP over requests; no fast-math and no FMA contraction, so x86-64 and
    aarch64 hosts round every operation the same way.
    """
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               src, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, out)
    return out


class Oracle:
    """One loaded build of the oracle library (the default one, or a test's variant)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        lib.oracle_reject_sample.restype = ctypes.c_int
        lib.oracle_reject_sample.argtypes = [
            P, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64,  # logits, dtype, T, V, stride
            P, ctypes.c_int64, P, P, ctypes.c_int32,  # q, q stride, draft ids, cu, B
            P, P,  # uniforms, temperature
            P, P, P,  # out tokens, out accepted, out flags
            P, P, P, P, P, P,  # dbg row max / sum / argmax, p draft, z, margins
            ctypes.c_int,  # nthreads
            P, P,  # top_k, top_p (optional)
        ]
        lib.oracle_max_threads.restype = ctypes.c_int
        self.lib = lib

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())


_default: Oracle | None = None


def _load() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def max_threads() -> int:
    return _load().max_threads()


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class OracleResult:
    tokens: np.ndarray        # int32 [T]
    num_accepted: np.ndarray  # int32 [B]
    flags: np.ndarray         # uint32 [B]
    status: int               # 0, or 1 when the batch is inconsistent as a whole
    row_max: np.ndarray | None = None
    row_sum: np.ndarray | None = None
    row_argmax: np.ndarray | None = None
    p_draft: np.ndarray | None = None
    z: np.ndarray | None = None
    margin: np.ndarray | None = None  # [B, 3]: acceptance margin (relative), sampling margin / Z, top-p margin


def reject_sample(logits: np.ndarray, draft_ids: np.ndarray, cu_num_draft: np.ndarray, uniforms: np.ndarray,
                  temperature: np.ndarray, draft_probs: np.ndarray | None = None, *, dtype: str | None = None,
                  vocab: int | None = None, logits_row_stride: int | None = None, q_row_stride: int | None = None,
                  debug: bool = False, nthreads: int = 0, num_rows: int | None = None,
                  impl: Oracle | None = None, top_k: np.ndarray | None = None,
                  top_p: np.ndarray | None = None) -> OracleResult:
    """Run the oracle on host arrays.

    ``logits`` is float32 [T, V] or uint16 (raw bf16 bits) [T, V].  With an
    explicit ``logits_row_stride`` any buffer works (stride 0 makes every row
    alias row 0; pass ``num_rows`` and ``vocab`` then).  ``draft_probs`` is
    float32 [T-B, V] (or strided the same way) or None for a one-hot draft.
    ``uniforms`` is float32 [T, 2]; ``temperature`` float32 [B].
    """
    if logits_row_stride is None:
        logits = np.ascontiguousarray(logits)
    if dtype is None:
        dtype = "bf16" if logits.dtype == np.uint16 else "f32"
    if dtype == "bf16":
        assert logits.dtype == np.uint16
        dcode = 1
    else:
        assert logits.dtype == np.float32
        dcode = 0
    V = int(vocab if vocab is not None else logits.shape[-1])
    stride = int(logits_row_stride if logits_row_stride is not None else V)
    cu = np.ascontiguousarray(cu_num_draft, dtype=np.int32)
    B = cu.shape[0] - 1
    T = int(num_rows if num_rows is not None else logits.shape[0])
    ids = np.ascontiguousarray(draft_ids, dtype=np.int32)
    u = np.ascontiguousarray(uniforms, dtype=np.float32)
    temp = np.ascontiguousarray(temperature, dtype=np.float32)
    assert u.size >= 2 * T and temp.size >= B
    q = None
    qs = 0
    if draft_probs is not None:
        q = draft_probs if q_row_stride is not None else np.ascontiguousarray(draft_probs, dtype=np.float32)
        assert q.dtype == np.float32
        qs = int(q_row_stride if q_row_stride is not None else V)
    tokens = np.full(T, -2, dtype=np.int32)
    acc = np.zeros(max(B, 0), dtype=np.int32)
    flags = np.zeros(max(B, 0), dtype=np.uint32)
    dbg = {}
    if debug:
        dbg = dict(row_max=np.full(T, np.nan), row_sum=np.full(T, np.nan), row_argmax=np.full(T, -1, np.int32),
                   p_draft=np.full(max(T - B, 0), np.nan), z=np.full(B, np.nan),
                   margin=np.full((max(B, 0), 3), np.inf))
    if ids.size == 0:
        ids = np.zeros(1, dtype=np.int32)
    tk = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32)
    tp = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float32)
    status = (impl or _load()).lib.oracle_reject_sample(
        _ptr(logits), dcode, T, V, stride, _ptr(q), qs, _ptr(ids), _ptr(cu), B, _ptr(u), _ptr(temp),
        _ptr(tokens), _ptr(acc), _ptr(flags), _ptr(dbg.get("row_max")), _ptr(dbg.get("row_sum")),
        _ptr(dbg.get("row_argmax")), _ptr(dbg.get("p_draft")), _ptr(dbg.get("z")), _ptr(dbg.get("margin")),
        int(nthreads), _ptr(tk), _ptr(tp))
    return OracleResult(tokens=tokens, num_accepted=acc, flags=flags, status=int(status), **dbg)


def reject_sample_workload(w: dict, debug: bool = False, nthreads: int = 0, num_requests: int | None = None,
                           impl: Oracle | None = None) -> OracleResult:
    """Run the oracle on a workload dict from the synthetic input generator.

    ``num_requests`` restricts the run to the first requests (their rows form a
    prefix of the flattened layout): the bounded sample the CPU baseline times.
    """
    cu = w["cu_num_draft"]
    q = w.get("draft_probs")
    tk, tp = w.get("top_k"), w.get("top_p")
    if num_requests is not None and num_requests < cu.shape[0] - 1:
        B = int(num_requests)
        cu = cu[: B + 1]
        nd = int(cu[-1])
        T = nd + B
        return reject_sample(w["logits"][:T], w["draft_ids"][:nd], cu, w["uniforms"][:T], w["temperature"][:B],
                             None if q is None else q[:nd], debug=debug, nthreads=nthreads, impl=impl,
                             top_k=None if tk is None else tk[:B], top_p=None if tp is None else tp[:B])
    return reject_sample(w["logits"], w["draft_ids"], cu, w["uniforms"], w["temperature"], q, debug=debug,
                         nthreads=nthreads, impl=impl, top_k=tk, top_p=tp)
