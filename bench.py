"""Benchmark of the batched rejection sampler on one GB300 (or N replicas).

One step = one spec_reject_sample() call over a whole synthetic batch (every kernel of
the path: the layout check, then the pass that reads each request's target rows up to
its output row, decides, runs the residual pass of explicit-q rejections and draws the
output token), inputs resident in HBM.

Default workload: the large-batch sweep point B=1024, K=8, V=128256, bf16 target
logits, explicit fp32 draft probabilities, temperature 0.7 (2.36 GB of logits +
4.2 GB of draft probabilities per step: larger than L2, so no flush is needed).
Exactly --steps calls are timed with CUDA events; SM clocks and clock-event reasons are
read through NVML every 0.5 ms during that region (`clocks`), and again over half a
second of the same calls right after it (`clocks_window`: a 20-step region lasts a few
milliseconds, too few samples to show a throttle).

The JSON line also carries `per_config`: the other workloads of the target's list
(tiny, greedy, probabilistic, deterministic, large-128, large-512) and the cut mode
(large-1024 and large-512 with top-k 50 / top-p 0.9, large-1024 with top-p 0.9 alone),
each timed for about half a second of calls in the same run (L2 flushed before every
call when the inputs are smaller than twice L2), with its dominant kernel's roofline
fraction.

Prints one JSON line.  `--impl reference` times the CPU oracle instead (a bounded
sample of the same workload on the host cores).

`--path tree | ngram | counters` times the other entry points on their own synthetic
workloads instead (greedy tree verification, the n-gram proposer, the acceptance
counters), one JSON line each with the same keys.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft positions/sec and achieved HBM GB/s vs ~8 TB/s peak (1 GB300)"
UNIT = "draft positions/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCE = os.path.join(ROOT, "speculative_decoding_rejection_spec_gb300", "csrc", "spec_reject.cu")
KERNEL_COMMON = os.path.join(ROOT, "speculative_decoding_rejection_spec_gb300", "csrc", "common.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def source_sha(full=False):
    """Hash of the kernel code: by default the shared device code (common.cuh) and the kernel
    file up to the end of the row-statistics kernel (K1 and everything it can use are defined
    before that point; later code cannot change it), with full=True both files whole.  Comments
    and blank space are left out (they compile to nothing), so a recorded traffic figure stays
    valid until the code itself changes."""
    import re
    parts = []
    for path, whole in ((KERNEL_COMMON, True), (KERNEL_SOURCE, full)):
        with open(path, "rb") as f:
            src = f.read()
        cut = -1 if whole else src.find(b"// K1F: top-k / top-p cut")
        parts.append((src if cut < 0 else src[:cut]).decode())
    code = "\n".join(parts)
    code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
    code = re.sub(r"//[^\n]*", " ", code)
    code = " ".join(code.split())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def traffic_for(workload):
    """DRAM bytes per launch of the row-statistics kernel on this workload from the committed
    ncu summary, only if it was taken on the current kernel source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    e = d.get("rowstats", {})
    if e.get("source_sha") != source_sha():
        return None
    return e.get("dram_bytes_per_launch", {}).get(workload)


def traffic_lazy_for(workload):
    """DRAM bytes per launch of KL on this workload from the committed ncu summary, only if it
    was taken on the current kernel source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    e = d.get("lazy", {})
    if e.get("source_sha") != source_sha(full=True):
        return None
    return e.get("dram_bytes_per_launch", {}).get(workload)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


class NvmlClocks:
    """SM clock and clock-event reasons read through NVML (libnvidia-ml, reading only) every
    half millisecond from a thread during the timed region: timed regions of a few milliseconds
    are too short for nvidia-smi's 50 ms sampling."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, torch_device):
        import ctypes
        self.ok = False
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            uuid = getattr(__import__("torch").cuda.get_device_properties(torch_device), "uuid", None)
            found = False
            if uuid is not None:
                sid = str(uuid)
                sid = sid if sid.startswith("GPU-") else "GPU-" + sid
                found = lib.nvmlDeviceGetHandleByUUID(sid.encode(), ctypes.byref(h)) == 0
            if not found and lib.nvmlDeviceGetHandleByIndex_v2(torch_device.index or 0, ctypes.byref(h)) != 0:
                return
            self.lib, self.h, self.ct = lib, h, ctypes
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 else None
            self.ok = True
        except OSError:
            pass

    def _one(self):
        clk, rs = self.ct.c_uint(), self.ct.c_ulonglong()
        a = self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(clk))
        b = self.lib.nvmlDeviceGetCurrentClocksEventReasons(self.h, self.ct.byref(rs))
        return (float(clk.value) if a == 0 else None), (int(rs.value) if b == 0 else 0)

    def start(self):
        import threading
        self.samples, self.stop_flag = [], False

        def run():
            while not self.stop_flag:
                self.samples.append(self._one())
                time.sleep(0.0005)
        if self.ok:
            self.th = threading.Thread(target=run, daemon=True)
            self.th.start()

    def stop(self):
        if not self.ok:
            return None
        self.stop_flag = True
        self.th.join()
        self.samples.append(self._one())
        sm = [c for c, _ in self.samples if c is not None]
        reasons = sorted({n for _, r in self.samples for bit, n in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "source": "NVML, every 0.5 ms"}


def clock_sampler(dev):
    """NVML sampling where libnvidia-ml can be loaded, else nvidia-smi every 50 ms."""
    n = NvmlClocks(dev)
    return n if n.ok else ClockSampler(dev.index or 0)


def cpu_baseline(w, target_s=8.0):
    """The oracle as it stands on the host cores, on the first requests of the workload."""
    import oracle
    cores = oracle.max_threads()
    n = 8
    while True:
        n = min(n, w["B"])
        t0 = time.perf_counter()
        oracle.reject_sample_workload(w, num_requests=n)
        dt = time.perf_counter() - t0
        if dt > target_s / 4 or n >= w["B"]:
            break
        n = min(w["B"], max(n * 2, int(n * (target_s / 2) / max(dt, 1e-3))))
    positions = int(w["cu_num_draft"][n])
    return {"value": positions / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {w['B']} requests ({positions} draft positions), {dt:.2f} s wall"}


def run_reference(args, w, meta):
    """--impl reference: the CPU oracle on bounded samples of the same workload."""
    import oracle
    rank, world, _ = dist_env()
    if rank != 0:
        return
    n = 8
    t0 = time.perf_counter()
    oracle.reject_sample_workload(w, num_requests=n)
    dt = time.perf_counter() - t0
    # each step a bounded sample sized so that the whole run stays within a few minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(min(w["B"], max(8, n * budget / max(dt, 1e-3))))
    for _ in range(args.warmup):
        oracle.reject_sample_workload(w, num_requests=n)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.reject_sample_workload(w, num_requests=n)
        times.append(time.perf_counter() - t0)
    positions = int(w["cu_num_draft"][n])
    value = positions / statistics.mean(times)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": meta,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"first {n} of {w['B']} requests per step ({positions} draft positions)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def time_calls(fn, steps, warmup, dev):
    """Per-call CUDA-event times (ms) of fn on the current stream, with clocks sampled."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = clock_sampler(dev)
    sampler.start()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    return start.elapsed_time(stop) / steps, [a.elapsed_time(b) for a, b in ev], clocks


def time_graph(fn, steps, warmup, dev, per_graph=20):
    """Device time per call (ms) of fn replayed from a CUDA graph of per_graph calls, with clocks
    sampled: for calls of a few microseconds the Python binding, not the kernel, would set the
    pace of eager calls."""
    import torch
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(max(warmup, 3)):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            fn()
    reps = max(1, steps // per_graph)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    sampler = clock_sampler(dev)
    sampler.start()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(reps):
        g.replay()
    stop.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    return start.elapsed_time(stop) / (reps * per_graph), reps * per_graph, clocks


def bounded(fn, n0, nmax, target_s):
    """Grow a sample size n until fn(n) takes about target_s / 2 .. target_s seconds."""
    n = n0
    while True:
        n = min(n, nmax)
        t0 = time.perf_counter()
        fn(n)
        dt = time.perf_counter() - t0
        if dt > target_s / 4 or n >= nmax:
            return n, dt
        n = min(nmax, max(n * 2, int(n * (target_s / 2) / max(dt, 1e-3))))


def bench_other_path(args):
    """--path tree | ngram | counters on one GPU (rank 0 of a replica run)."""
    import torch
    import __graft_entry__ as G
    from speculative_decoding_rejection_spec_gb300 import binding, workloads as W
    G.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, peak_kind = peaks()
    line = {"n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "data": "synthetic"}
    if args.path == "tree":
        name = args.workload if args.workload in W.TREE_CONFIGS else "tree-64x64"
        w = W.generate_tree(name)
        bf16 = w["dtype"] == "bf16"
        lg = torch.from_numpy(w["logits"].view(np.int16) if bf16 else w["logits"]).to(dev)
        if bf16:
            lg = lg.view(torch.bfloat16)
        par = torch.from_numpy(w["parent"]).to(dev)
        tok = torch.from_numpy(w["node_tokens"]).to(dev)
        cu = torch.from_numpy(w["cu_nodes"]).to(dev)
        buf = binding.tree_verify_greedy(lg, par, tok, cu)
        ms, per, clocks = time_calls(lambda: binding.tree_verify_greedy(lg, par, tok, cu, buffers=buf), args.steps,
                                     args.warmup, dev)
        es = 2 if bf16 else 4
        nbytes = w["N"] * w["V"] * es
        acc = buf[1].cpu().numpy()
        line.update(metric="verified tree nodes/s (greedy tree verification)", unit="tree nodes/s",
                    value=w["N"] / (ms / 1e3), ms_per_step=ms, dtype="bf16" if bf16 else "f32",
                    config={"workload": f"{name}: B={w['B']} trees, N={w['N']} nodes, V={w['V']} "
                                        f"{w['dtype']} logits, topk<= {w['spec']['topk']}, depth<= {w['spec']['depth']}",
                            "l2": "inputs larger than L2 (no flush)" if nbytes > 129e6 else "L2-resident inputs"},
                    mean_accepted_depth=float(acc.mean()), gpu_launches=2 * args.steps, clocks=clocks)
        achieved = nbytes / (statistics.mean(per) / 1e3) / 1e9
        line["roofline"] = {"bound": "hbm", "kernel": "whole call (argmax pass over every node row + tree walk)",
                            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                            "frac": round(achieved / peak, 4), "peak_kind": peak_kind, "traffic": None,
                            "algorithmic_bytes_per_launch": nbytes}
        if not args.no_cpu:
            from oracle import tree as otree
            x64 = (W.bf16_bits_to_f32(w["logits"]) if bf16 else w["logits"])

            def run(n):
                e = int(w["cu_nodes"][n])
                otree.verify_batch(x64[:e].astype(np.float64), w["parent"][:e], w["node_tokens"][:e],
                                   w["cu_nodes"][:n + 1])
            n, dt = bounded(run, 2, w["B"], 10.0)
            nodes = int(w["cu_nodes"][n])
            line["cpu_baseline"] = {"value": nodes / dt, "unit": "tree nodes/s", "cores": 1, "kind": "oracle",
                                    "sample": f"first {n} of {w['B']} trees ({nodes} nodes), {dt:.2f} s wall"}
    elif args.path == "ngram":
        name = args.workload if args.workload in W.NGRAM_CONFIGS else "ngram-1024x4096"
        g = W.generate_ngram(name)
        toks = torch.from_numpy(g["tokens"]).to(dev)
        cu = torch.from_numpy(g["cu_tokens"]).to(dev)
        out = torch.empty((g["B"], g["k"]), dtype=torch.int32, device=dev)
        num = torch.empty(g["B"], dtype=torch.int32, device=dev)
        call = lambda: binding.ngram_propose(toks, cu, g["min_n"], g["max_n"], g["k"], out=out, num=num)
        eager_ms, _, _ = time_calls(call, args.steps, args.warmup, dev)
        ms, launches, clocks = time_graph(call, args.steps, args.warmup, dev)
        nbytes = g["B"] * g["L"] * 4
        achieved = nbytes / (ms / 1e3) / 1e9
        line.update(metric="n-gram proposals/s (one proposal per context)", unit="proposals/s",
                    value=g["B"] / (ms / 1e3), ms_per_step=ms, dtype="int32",
                    config={"workload": f"{name}: B={g['B']} contexts of L={g['L']} tokens, n={g['min_n']}..{g['max_n']}, "
                                        f"k={g['k']}", "l2": "L2-resident inputs (16 MB)"},
                    hit_rate=float((num.cpu().numpy() > 0).mean()), context_tokens_per_s=g["B"] * g["L"] / (ms / 1e3),
                    gpu_launches=launches, clocks=clocks, timing="CUDA graph of 20 calls, replayed",
                    eager_ms_per_call=round(eager_ms, 4))
        line["roofline"] = {"bound": "hbm", "kernel": "ngram_kernel (block per context, candidate starts in parallel)",
                            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                            "frac": round(achieved / peak, 4), "peak_kind": peak_kind, "traffic": None,
                            "algorithmic_bytes_per_launch": nbytes}
        if not args.no_cpu:
            from oracle import ngram as ong

            def run(n):
                ong.propose_batch(g["tokens"][:n * g["L"]], g["cu_tokens"][:n + 1], g["min_n"], g["max_n"], g["k"])
            n, dt = bounded(run, 8, g["B"], 10.0)
            line["cpu_baseline"] = {"value": n / dt, "unit": "proposals/s", "cores": 1, "kind": "oracle",
                                    "sample": f"first {n} of {g['B']} contexts, {dt:.2f} s wall"}
    else:  # counters
        name = args.workload if args.workload in W.CONFIGS else "large-1024"
        spec = W.CONFIGS[name]
        B = spec["B"]
        rng = np.random.default_rng(5)
        ks = np.full(B, spec["K"], np.int32) if spec["K"] != "ragged" else rng.integers(0, spec["K_max"] + 1, B)
        cu_h = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
        acc_h = rng.integers(0, np.maximum(ks, 0) + 1).astype(np.int32)
        cu = torch.from_numpy(cu_h).to(dev)
        acc = torch.from_numpy(acc_h).to(dev)
        ctr = torch.zeros(binding.METRIC_COUNT, dtype=torch.int64, device=dev)
        call = lambda: binding.metrics_update(cu, acc, ctr)
        eager_ms, _, _ = time_calls(call, args.steps, args.warmup, dev)
        ms, launches, clocks = time_graph(call, args.steps, args.warmup, dev)
        nbytes = (2 * B + 1) * 4
        achieved = nbytes / (ms / 1e3) / 1e9
        line.update(metric="requests counted/s (acceptance counters update)", unit="requests/s",
                    value=B / (ms / 1e3), ms_per_step=ms, dtype="int64",
                    config={"workload": f"{name}: B={B} requests", "l2": "L2-resident inputs"},
                    gpu_launches=launches, clocks=clocks, timing="CUDA graph of 20 calls, replayed",
                    eager_ms_per_call=round(eager_ms, 4))
        line["roofline"] = {"bound": "hbm", "kernel": "metrics_kernel (launch-bound: a few KB per call)",
                            "achieved": round(achieved, 3), "peak": peak, "unit": "GB/s",
                            "frac": round(achieved / peak, 6), "peak_kind": peak_kind, "traffic": None,
                            "algorithmic_bytes_per_launch": nbytes}
        # the fused form: the same counters added inside the sampler's finalize pass
        wl = W.generate("large-128")
        dd = binding.to_device(wl, dev)
        bufs = binding.make_buffers(wl["B"], wl["T"], wl["V"], binding.BF16, dd["draft_probs"] is not None, dev)
        plain_ms, _, _ = time_calls(lambda: binding.sample_ex(**dd, buffers=bufs), args.steps, args.warmup, dev)
        fused_ms, _, _ = time_calls(lambda: binding.sample_ex(**dd, counters=ctr, buffers=bufs), args.steps,
                                    args.warmup, dev)
        line["fused"] = {"workload": "large-128 sampler call", "call_ms_without_counters": round(plain_ms, 4),
                         "call_ms_with_counters": round(fused_ms, 4), "extra_launches": 0}
        if not args.no_cpu:
            from oracle import closed_forms as cf
            n, dt = bounded(lambda n: [cf.acceptance_counters(cu_h, acc_h) for _ in range(n)], 1, 10 ** 6, 4.0)
            line["cpu_baseline"] = {"value": n * B / dt, "unit": "requests/s", "cores": 1, "kind": "oracle",
                                    "sample": f"{n} updates of {B} requests, {dt:.2f} s wall"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large-1024")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the other workloads' figures")
    ap.add_argument("--top-k", type=int, default=None, help="top-k on the target, every request")
    ap.add_argument("--top-p", type=float, default=None, help="top-p on the target, every request")
    ap.add_argument("--path", default="sample", choices=["sample", "tree", "ngram", "counters"],
                    help="entry point to time: the sampler (default) or one of the other calls")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    from speculative_decoding_rejection_spec_gb300 import workloads as W
    rank, world, local = dist_env()
    if args.impl == "reference" and rank != 0:
        return  # the reference arm runs on rank 0 only
    if args.path != "sample":
        if rank == 0 and args.impl == "ours":
            bench_other_path(args)
        return
    spec = W.CONFIGS[args.workload]
    meta = {"workload": f"{args.workload}: B={spec['B']} K={spec['K']} V={spec['V']} {spec['dtype']} logits, "
                        f"{'explicit fp32 draft probs' if spec['draft'] in ('noisy_q', 'target_q') else 'one-hot drafts'}"
                        f", temperature {spec['temperature']}",
            "B_per_gpu": spec["B"], "V": spec["V"], "logits_dtype": spec["dtype"],
            "l2": "inputs larger than L2 (no flush)", "rng": "numpy PCG64, seeded"}
    filtered = args.top_k is not None or args.top_p is not None
    if filtered:
        meta["workload"] += f", top-k {args.top_k}, top-p {args.top_p}"
    # each rank draws its own batch (independent requests: weak scaling, no data-path collective)
    w = W.generate(args.workload, seed=spec["seed"] + 1000 * rank, top_k=args.top_k, top_p=args.top_p)
    if args.impl == "reference":
        run_reference(args, w, meta)
        return

    import torch
    import __graft_entry__ as G
    from speculative_decoding_rejection_spec_gb300 import binding
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    G.build()
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    peak, peak_kind = peaks()

    m = measure(w, dev, args.steps, args.warmup, tk_tp=(args.top_k, args.top_p), barrier=world > 1)
    if world > 1:
        t = torch.tensor([m["total_ms"]], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        m["total_ms"] = float(t.item())
    ms = m["total_ms"] / args.steps
    positions = W.total_drafts(w)
    value = positions * world / (ms / 1e3)
    workload_key = args.workload + (f"+k{args.top_k}+p{args.top_p}" if filtered else "")
    roofline = roofline_of(m, peak, peak_kind, workload_key)

    meta["l2"] = m["l2"]
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": meta,
            "hbm_gbs_effective": round(m["alg_bytes"] / (ms / 1e3) / 1e9, 1),
            "stage_ms": [round(x, 4) for x in m["stage_ms"]], "stages": m["stages"],
            "roofline": roofline, "gpu_launches": m["launches"] * args.steps, "clocks": m["clocks"],
            "clocks_window": m["clocks_window"],
            "rows_read_per_step": m["rows_read"], "rows_total": int(w["T"]),
            "blocks_per_request": m["blocks_per_request"]}

    if not args.no_e2e:
        line["e2e"] = e2e(w, dev, args)
    if rank == 0 and world == 1 and not args.no_per_config and not filtered:
        line["per_config"] = per_config(args, dev, peak, peak_kind)
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def q_bytes_per_rejection(w, cut_in_first_rejection_pass):
    """Draft-probability bytes one rejection needs: the whole row of q, except where the
    first-rejection pass cuts with a top-k of at most 256 tokens on every request: the residual
    has mass at the kept tokens only, and the pass reads q there alone (a 32-byte sector per kept
    token; ties at the cut key aside, at most top-k of them)."""
    tk = w.get("top_k")
    if cut_in_first_rejection_pass and tk is not None and (tk > 0).all() and int(tk.max()) <= 256:
        return 32 * int(tk.max())
    return w["V"] * 4


def measure(w, dev, steps, warmup, tk_tp=(None, None), barrier=False, min_seconds=0.0):
    """One sampler call per step over workload w (inputs resident in HBM).  Times `steps` plain
    calls with CUDA events on the launching stream (at least `min_seconds` of them when that is
    set), then the same number of calls through the stage-event entry for each kernel's own
    time.  Returns the times, the call's algorithmic bytes (rows read up to each output row,
    the draft rows of explicit-q rejections, the small arrays) and the launch shape."""
    import torch
    from speculative_decoding_rejection_spec_gb300 import binding
    d = binding.to_device(w, dev)
    has_q = d["draft_probs"] is not None
    dt = binding.BF16 if w["dtype"] == "bf16" else binding.F32
    buf = binding.make_buffers(w["B"], w["T"], w["V"], dt, has_q, dev)
    tk = None if w.get("top_k") is None else torch.from_numpy(w["top_k"]).to(dev)
    tp = None if w.get("top_p") is None else torch.from_numpy(w["top_p"]).to(dev)
    filtered = tk is not None or tp is not None
    nk = binding.num_kernels(w["B"], has_q, filtered, dt)
    launches = binding.launches_per_call(w["B"], w["V"], has_q, filtered, dt)
    lazy = binding.reads_to_first_rejection(w["B"], filtered, dt)
    stream = torch.cuda.current_stream()
    call = lambda: binding.sample_profiled(d, buf, [], stream, tk, tp)
    for _ in range(warmup):
        call()
    st, bits, _ = binding.last_device_error(buf.workspace)
    if st != 0:
        raise SystemExit(f"device input error bits {bits}")
    torch.cuda.synchronize()
    # inputs smaller than twice the L2 cache: flush it before every timed call (a write of a
    # buffer larger than L2, outside the events), so that no call reads what the last one left
    in_bytes = sum(t.numel() * t.element_size() for t in d.values() if t is not None)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev) if in_bytes < 2 * l2 else None
    if min_seconds > 0:  # enough calls to fill the requested time
        t0 = time.perf_counter()
        for _ in range(5):
            call()
        torch.cuda.synchronize()
        per = (time.perf_counter() - t0) / 5
        steps = max(steps, min(20000, int(min_seconds / max(per, 1e-6))))
    clocks = clock_sampler(dev)
    if barrier:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    if flush is None:
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            call()
        stop.record(stream)
        torch.cuda.synchronize()
        total_ms = start.elapsed_time(stop)
    else:
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in pairs:
            flush.zero_()
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize()
        total_ms = sum(a.elapsed_time(b) for a, b in pairs)
    clk = clocks.stop()
    if barrier:
        torch.distributed.barrier()
    clk_window = None
    if min_seconds <= 0:
        # a few-step timed region lasts milliseconds, a handful of clock samples: the same call
        # repeated for half a second right after it, outside the timed region, samples the clocks
        # the kernels run at (reported beside the timed region's own samples)
        window = clock_sampler(dev)
        window.start()
        t0, n = time.perf_counter(), 0
        while time.perf_counter() - t0 < 0.5:
            for _ in range(20):
                if flush is not None:
                    flush.zero_()
                call()
            n += 20
            torch.cuda.synchronize()
        clk_window = window.stop()
        if clk_window is not None:
            clk_window["calls"] = n
            clk_window["seconds"] = round(time.perf_counter() - t0, 3)
    # per-kernel times: the same calls with an event after each kernel
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(min(steps, 200))]
    for row in ev:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    for row in ev:
        if flush is not None:
            flush.zero_()
        binding.sample_profiled(d, buf, row, stream, tk, tp)
    torch.cuda.synchronize()
    stage_ms = [statistics.mean(row[i].elapsed_time(row[i + 1]) for row in ev) for i in range(nk)]

    es = 2 if w["dtype"] == "bf16" else 4
    acc = buf.out_num_accepted.cpu().numpy()
    ks = np.diff(w["cu_num_draft"])
    valid = acc >= 0
    rejecting = int((valid & (acc < ks)).sum()) if has_q else 0
    small = 8 * (w["T"] - w["B"]) + 12 * w["T"] + 4 * (2 * w["B"] + 1)
    q_row_bytes = q_bytes_per_rejection(w, lazy and filtered)
    if lazy:
        rows_read = int((acc[valid] + 1).sum())
        stages = ["layout_check", "rows_to_first_rejection"]
        dom = 1
        dom_bytes = rows_read * w["V"] * es + rejecting * q_row_bytes + small
        bpr = binding.blocks_per_request(w["B"], w["V"], dt) if not filtered else 1
        dom_name = ("KL: lazy_kernel (request queue; rows streamed through warp-private TMA rings up to the first "
                    "rejection; residual pass and draw in the same block" +
                    (f"; each request split over a cluster of {bpr} blocks" if bpr > 1 else "") +
                    (("; the last requests in a chained second launch (" +
                      ("16-warp blocks" if filtered else "two blocks each") + "), timed with the first")
                     if launches > nk else "") + ")")
        if filtered:
            dom_name += ("; each reached row cut in the block (key-offset counts of marked tokens), the output row "
                         "drawn from its kept tokens")
        alg = dom_bytes
    else:
        rows_read = int(w["T"])
        stages = (["rowstats"] + (["topk_topp_cut"] if filtered else []) + ["finalize"] + (["residual"] if has_q else []))
        dom = 0
        dom_bytes = w["T"] * w["V"] * es + 4 * (w["T"] - w["B"])
        dom_name = "row statistics (K1: rowstats_wr_kernel, warp-private TMA pipelines)"
        bpr = 0
        alg = w["T"] * w["V"] * es + rejecting * w["V"] * 4 + small
    out = {"total_ms": total_ms, "steps": steps, "stage_ms": stage_ms, "stages": stages, "dom": dom,
           "l2": ("L2 flushed before every call (inputs smaller than twice L2)" if flush is not None
                  else "inputs larger than twice L2 (no flush)"),
           "dom_bytes": dom_bytes, "dom_name": dom_name, "alg_bytes": alg, "rows_read": rows_read,
           "kernels": nk, "launches": launches, "clocks": clk, "clocks_window": clk_window, "lazy": lazy,
           "blocks_per_request": bpr}
    del d, buf
    torch.cuda.empty_cache()
    return out


def roofline_of(m, peak, peak_kind, workload_key):
    dom_ms = m["stage_ms"][m["dom"]]
    achieved = m["dom_bytes"] / (dom_ms / 1e3) / 1e9
    traffic = traffic_lazy_for(workload_key) if m["lazy"] else traffic_for(workload_key)
    return {"bound": "hbm", "kernel": m["dom_name"], "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_kind": peak_kind, "traffic": traffic,
            "algorithmic_bytes_per_launch": m["dom_bytes"], "ms_per_launch": round(dom_ms, 4),
            "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4)}


PER_CONFIG = ["tiny", "greedy", "probabilistic", "deterministic", "large-128", "large-512"]
# the same measurement with top-k / top-p on the target (every request): (workload, top-k, top-p)
PER_CONFIG_CUT = [("large-1024", 50, 0.9), ("large-512", 50, 0.9), ("large-1024", None, 0.9)]


def per_config(args, dev, peak, peak_kind):
    """The other workloads of the target's config list, measured in the same run (each for
    about half a second of calls): step time, the dominant kernel and its roofline fraction."""
    from speculative_decoding_rejection_spec_gb300 import workloads as W
    out = {}
    runs = [(n, n, None, None) for n in PER_CONFIG]
    runs += [(n + (f"+k{tk}" if tk else "") + (f"+p{tp}" if tp else ""), n, tk, tp) for n, tk, tp in PER_CONFIG_CUT]
    base = {}
    for key, name, tk, tp in runs:
        if name not in base:  # one draw of each workload; the cuts only add their per-request arrays
            base.clear()
            base[name] = W.generate(name)
        w = dict(base[name])
        B = w["B"]
        if tk is not None:
            w["top_k"] = np.full(B, tk, dtype=np.int32)
        if tp is not None:
            w["top_p"] = np.full(B, tp, dtype=np.float32)
        m = measure(w, dev, 20, max(args.warmup, 3), tk_tp=(tk, tp), min_seconds=0.5)
        ms = m["total_ms"] / m["steps"]
        rf = roofline_of(m, peak, peak_kind, key)
        out[key] = {"ms_per_step": round(ms, 5), "value": W.total_drafts(w) / (ms / 1e3), "unit": UNIT,
                     "steps": m["steps"], "kernel": rf["kernel"], "kernel_ms": rf["ms_per_launch"],
                     "algorithmic_bytes": m["dom_bytes"], "achieved_gbs": rf["achieved"], "frac": rf["frac"],
                     "frac_of_nominal_8tbs": rf["frac_of_nominal_8tbs"], "traffic": rf["traffic"],
                     "rows_read": m["rows_read"], "rows_total": int(w["T"]),
                     "blocks_per_request": m["blocks_per_request"], "stage_ms": [round(x, 4) for x in m["stage_ms"]],
                     "l2": m["l2"], "clocks": m["clocks"]}
    return out


def e2e(w, dev, args):
    """Same metric through the host-buffer entry point: pinned host inputs copied to the
    device, the sampler run, the outputs copied back, every step."""
    import torch
    from speculative_decoding_rejection_spec_gb300 import binding
    has_q = w["draft_probs"] is not None
    dt = binding.BF16 if w["dtype"] == "bf16" else binding.F32

    def pinned(a):
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()
        return t

    host = {"logits": pinned(w["logits"]), "draft_ids": pinned(w["draft_ids"]),
            "cu_num_draft": pinned(w["cu_num_draft"]), "uniforms": pinned(w["uniforms"]),
            "temperature": pinned(w["temperature"])}
    if has_q:
        host["draft_probs"] = pinned(w["draft_probs"])
    filtered = w.get("top_k") is not None or w.get("top_p") is not None
    for k in ("top_k", "top_p"):  # cuts go through spec_reject_sample_host_ex
        if w.get(k) is not None:
            host[k] = pinned(w[k])
    host["out_tokens"] = torch.empty(w["T"], dtype=torch.int32).pin_memory()
    host["out_num_accepted"] = torch.empty(w["B"], dtype=torch.int32).pin_memory()
    ptrs = {k: v.data_ptr() for k, v in host.items()}
    arena = torch.empty(binding.host_arena_size(w["B"], w["T"], w["V"], dt, has_q), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    steps = max(3, min(args.steps, 10))
    for _ in range(2):
        binding.sample_host_ptrs(ptrs, w["T"], w["V"], w["B"], dt, arena, stream)
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        binding.sample_host_ptrs(ptrs, w["T"], w["V"], w["B"], dt, arena, stream)
    stop.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(stop) / steps
    # bytes that cross the host link per step (the algorithmic ones): the small inputs are copied;
    # pinned draft probabilities are read in place (one 32-byte sector per q(x*) gather and the
    # row at each rejecting request's first rejection); pinned target logits of a batch that
    # takes the first-rejection pass are read in place too, only the rows up to each output row
    from speculative_decoding_rejection_spec_gb300 import binding as _b
    acc = host["out_num_accepted"].numpy()
    ks = np.diff(w["cu_num_draft"])
    logits_in_place = _b.reads_to_first_rejection(w["B"], filtered, dt)
    h2d = sum(v.numel() * v.element_size() for k, v in host.items()
              if not k.startswith("out_") and k != "draft_probs" and not (k == "logits" and logits_in_place))
    es = 2 if w["dtype"] == "bf16" else 4
    notes = []
    if logits_in_place:
        rows = int((acc[acc >= 0] + 1).sum())
        h2d += rows * w["V"] * es
        notes.append(f"target logits read in place from pinned memory: {rows} of {w['T']} rows")
    if has_q:
        rejecting = int(((acc >= 0) & (acc < ks)).sum())
        qb = q_bytes_per_rejection(w, logits_in_place and filtered)
        h2d += rejecting * qb + 32 * (w["T"] - w["B"])
        what = "rows" if qb == w["V"] * 4 else f"x {qb} bytes at the kept tokens"
        notes.append(f"draft probabilities read in place: {rejecting} {what} + {w['T'] - w['B']} gathers")
    q_note = "; ".join(notes) if notes else None
    d2h = 4 * (w["T"] + w["B"])
    from speculative_decoding_rejection_spec_gb300 import workloads as W
    out = {"value": W.total_drafts(w) / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h), "ms_per_step": ms, "steps": steps}
    if q_note:
        out["note"] = q_note
    return out


if __name__ == "__main__":
    main()
