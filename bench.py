#!/usr/bin/env python
"""Benchmark of fused exact attention (forward + backward) on GB300.

One step is one pass of the whole path over one batch: fa_fwd (O, L) then
fa_bwd (D preprocess, fused key-block backward, dQ conversion) on seeded
synthetic inputs already resident in HBM. Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long8k]
  python bench.py --impl reference ...   # the fp64 CPU oracle on a sample

Multi-GPU (torchrun, one rank per GPU): every rank runs an independent
replica of the workload (heads are independent; no data exchange), the
timing is the maximum over ranks and the value is the total over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd and fwd+bwd TFLOP/s on 1 GB300; % of dense BF16 tensor peak"
DEFAULT_WORKLOAD = "sparse16k"   # the largest configuration: B2 H16 N16384 d128, 128x128 tile mask
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-targets", action="store_true",
                    help="skip the measurement of the other N >= 4096 workloads (the line's 'targets')")
    ap.add_argument("--spin-up-s", type=float, default=0.5,
                    help="untimed calls after the warm-up steps until the GPU has been busy this long (0: none), "
                         "so that the clocks have settled before the timed region")
    ap.add_argument("--table", action="store_true",
                    help="measure every workload (times, TFLOP/s, errors vs the oracle on sampled heads); "
                         "prints one JSON object per workload instead of the benchmark line")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def describe(w):
    mask = "causal" if w.causal else ("key padding U{%d..%d}" % w.kv_len_range if w.kv_len_range else
                                       ("128x128 tile mask, diagonal + %.1f%% of other tiles" % (100 * w.block_density)
                                        if w.block_density else "no mask"))
    ks = ", K rows x%g" % w.k_scale if w.k_scale != 1.0 else ""
    return f"{w.name}: attention fwd+bwd, B={w.B} H={w.H} N={w.N} d={w.d} {w.dtype}, {mask}{ks}"


# ------------------------------------------------------------------ clocks
# NVML clocks-event-reason bits (nvml.h, nvmlClocksEventReason*): read-only
# queries; nothing here changes a GPU setting.
_NVML_REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
                 0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """Samples the SM clock, power and clock-event reasons of one GPU while
    the timed region runs: through NVML (libnvidia-ml, every 5 ms) when it
    can be loaded, else through `nvidia-smi -lms 20`."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None, period_s=0.005):
        self.uuid = uuid
        self.period = period_s
        self.rows = []      # (time, sm_mhz, max_mhz, power_w, set of reasons)
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()
        self.source = None

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        if self.uuid:
            rc = lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h))
        else:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h))
        if rc != 0:
            return None
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons_fn

    def start(self):
        nv = None
        try:
            nv = self._nvml()
        except OSError:
            nv = None
        if nv is not None:
            import ctypes
            lib, h, reasons_fn = nv
            self.source = "nvml every %g ms" % (1e3 * self.period)
            mx = ctypes.c_uint()
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))   # 1 = NVML_CLOCK_SM

            def poll():
                c, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
                while not self.stop_flag.is_set():
                    ok = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(c)) == 0
                    lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
                    reasons_fn(h, ctypes.byref(rs))
                    if ok:
                        names = {n for bit, n in _NVML_REASONS.items() if rs.value & bit}
                        self.rows.append((time.time(), float(c.value), float(mx.value), pw.value / 1e3, names))
                    time.sleep(self.period)

            self.thread = threading.Thread(target=poll, daemon=True)
            self.thread.start()
            time.sleep(0.05)
            return
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20"]
        if self.uuid:
            cmd[1:1] = ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.source = "nvidia-smi -lms 20"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        def reader():
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in self.proc.stdout:
                r = [c.strip() for c in line.split(",")]
                if len(r) < 10 or num(r[2]) is None:
                    continue
                rs = {n for k, n in enumerate(names) if r[6 + k].lower().startswith("active")}
                self.rows.append((time.time(), num(r[2]), num(r[3]), num(r[4]) or 0.0, rs))

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        time.sleep(0.6)

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t_begin, t_end):
        rows = [r for r in self.rows if t_begin <= r[0] <= t_end]
        if not rows:
            rows = self.rows[-3:]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        reasons = set()
        for r in rows:
            reasons |= r[4]
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": rows[0][2],
                "sm_mhz_min": min(r[1] for r in rows), "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r[3] for r in rows), "source": self.source}


# ------------------------------------------------------------------ helpers
# source files each profiled kernel is compiled from (its .cu plus the shared
# headers); a recorded DRAM-traffic figure stays valid while their code (the
# text without `//` comments and blank lines) is unchanged
KERNEL_SOURCES = {
    "fa_fwd_kernel": ["fa_fwd.cu"],
    "fa_fwd_fp8_kernel": ["fa_fwd_fp8.cu", "fa_fp8.h"],
    "fa_bwd_kernel": ["fa_bwd.cu"],
    "fa_fwd_t1_kernel": ["fa_fwd_t1.cu"],
    "fa_decode_split_kernel": ["fa_decode.cu", "fa_decode.h"],
}
SHARED_HEADERS = ["fa_common.cuh", "fa_launch.h", "sm103_ptx.cuh", "tmap.h"]


def kernel_source_sha(kernel: str):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "io_aware_exact_tiled_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES.get(kernel, []) + SHARED_HEADERS):
        h.update(f.encode())
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if
    the kernel sources have not changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(kernel, {}).get(workload)
        if e and e.get("source_sha") == kernel_source_sha(kernel):
            return e["dram_bytes_per_launch"]
    except (ValueError, KeyError, TypeError):
        return None
    return None


def oracle_sample(w, x, budget_s=12.0, max_heads=8):
    """Time the fp64 CPU oracle (forward + backward) on whole heads of the
    workload until about `budget_s` seconds have been spent."""
    import oracle
    from io_aware_exact_tiled_gb300 import accounting as acc
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    done, flop, t_used = [], 0.0, 0.0
    kl = None if x.kv_len is None else x.kv_len.cpu()
    bm = None if x.blockmask is None else x.blockmask.cpu()
    q, k, v, do = (t.cpu() for t in (x.q, x.k, x.v, x.do))
    for (b, h) in heads[:max_heads]:
        qs, ks, vs, dos = (t[b:b + 1, h:h + 1] for t in (q, k, v, do))
        kls = None if kl is None else kl[b:b + 1]
        t0 = time.perf_counter()
        oracle.forward(qs, ks, vs, x.scale, causal=x.causal, kv_len=kls, blockmask=bm)
        oracle.backward(qs, ks, vs, dos, x.scale, causal=x.causal, kv_len=kls, blockmask=bm)
        t_used += time.perf_counter() - t0
        pb = acc.pairs_per_batch(w.N, w.causal, None if kl is None else kl.tolist(),
                                 None if bm is None else bm.numpy(), w.B)[b]
        flop += 14.0 * w.d * pb
        done.append((b, h))
        if t_used >= budget_s:
            break
    return flop, t_used, done


# ------------------------------------------------------------------ reference arm
def oracle_rows(w, x, R):
    """Time the oracle on the last R query rows of head (0, 0) (the rows with
    the most visible keys under a causal mask); returns (flops, seconds)."""
    import numpy as np
    import oracle
    from oracle.attention import visible
    kl = None if x.kv_len is None else x.kv_len[:1]
    bm = None if x.blockmask is None else x.blockmask
    rows = (w.N - R, w.N)
    q, k, v, do = (t[:1, :1] for t in (x.q, x.k, x.v, x.do))   # head (0, 0)
    t0 = time.perf_counter()
    oracle.forward(q, k, v, x.scale, causal=x.causal, kv_len=kl, blockmask=bm, rows=rows)
    oracle.backward(q, k, v, do, x.scale, causal=x.causal, kv_len=kl, blockmask=bm, rows=rows)
    t = time.perf_counter() - t0
    vis = visible(w.N, x.causal, None if kl is None else int(kl[0]), bm, np.arange(*rows))
    return 14.0 * w.d * float(vis.sum()), t


def run_reference(args, rank, world):
    if rank != 0:
        return
    from io_aware_exact_tiled_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    x = W.make_inputs(w, seed=0)
    # size each step so that warm-up + timed steps stay within a few minutes
    budget = min(5.0, 150.0 / max(1, args.steps + args.warmup))
    f1, t1 = oracle_rows(w, x, 128)
    R = int(min(w.N, max(128, 128 * math.floor(budget / max(t1, 1e-6)))))
    times, flops = [], []
    for i in range(args.warmup + args.steps):
        f, t = oracle_rows(w, x, R)
        if i >= args.warmup:
            times.append(t)
            flops.append(f)
    total_t = sum(times)
    value = sum(flops) / total_t / 1e12
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(w), "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": bool(w.causal),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: fp64 NumPy forward + backward of the last {R} query rows of head "
                                   f"(0, 0) (N={w.N}, d={w.d}) on the host cores (BLAS threads = all cores; exp "
                                   f"single-threaded)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ per-workload table
# heads on which the table's CPU baseline times the oracle (other workloads: head (0, 0))
TABLE_HEADS = {"long4k": [(0, 0), (0, 31)], "long8k": [(0, 0), (0, 31)], "sparse16k": [(0, 0), (1, 15)]}


def run_table(args):
    """Kernel and call times of every workload. Agreement with the oracle is
    checked by the GPU parity tests; here the oracle is only timed, as each
    row's CPU baseline (unless --no-cpu-baseline)."""
    import torch

    import io_aware_exact_tiled_gb300 as fa
    from io_aware_exact_tiled_gb300 import accounting as acc
    from io_aware_exact_tiled_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    peaks, _ = load_peaks()
    peak = float(peaks["bf16_tflops"])
    ev = lambda: torch.cuda.Event(enable_timing=True)
    for name, w in W.WORKLOADS.items():
        x = W.make_inputs(w, seed=0)
        q, k, v, do = (t.to(dev) for t in (x.q, x.k, x.v, x.do))
        bm = None if x.blockmask is None else x.blockmask.to(dev)
        kl = None if x.kv_len is None else x.kv_len.to(dev)
        kw = dict(scale=x.scale, causal=x.causal, blockmask=bm, kv_len=kl)
        B, H, N, d = q.shape
        fwd_flop, bwd_flop = acc.flops(B, H, N, d, x.causal, None if kl is None else x.kv_len.tolist(),
                                       None if bm is None else x.blockmask.numpy())
        o, lse = fa.forward(q, k, v, **kw)
        ws_f = fa.workspace(fa.fwd_workspace_size(B, H, N, d), dev)
        ws_b = fa.workspace(fa.bwd_workspace_size(B, H, N, d), dev) if w.backward else None
        row = {"workload": describe(w)}

        def timed(fn, reps=20):
            """(mean ms per call, mean ms of the main kernel per call)."""
            for _ in range(3):
                fn()
            pairs = [(ev(), ev()) for _ in range(reps)]
            for a, b in pairs:  # materialise the event handles
                a.record()
                b.record()
            c0, c1 = ev(), ev()
            torch.cuda.synchronize()
            c0.record()
            for i in range(reps):
                fa.set_timing_events(*pairs[i])
                fn()
            c1.record()
            fa.set_timing_events(None, None)
            torch.cuda.synchronize()
            return c0.elapsed_time(c1) / reps, sum(a.elapsed_time(b) for a, b in pairs) / reps

        fcall, fker = timed(lambda: fa.forward(q, k, v, out=o, lse=lse, ws=ws_f, **kw))
        row["fwd"] = {"call_ms": fcall, "kernel_ms": fker, "tflops": fwd_flop / (fker * 1e-3) / 1e12,
                      "pct_peak": 100 * fwd_flop / (fker * 1e-3) / 1e12 / peak}
        if w.backward:
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            bcall, bker = timed(lambda: fa.backward(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, ws=ws_b, **kw))
            row["bwd"] = {"call_ms": bcall, "kernel_ms": bker, "tflops_call": bwd_flop / (bcall * 1e-3) / 1e12,
                          "tflops_kernel": bwd_flop / (bker * 1e-3) / 1e12,
                          "pct_peak_kernel": 100 * bwd_flop / (bker * 1e-3) / 1e12 / peak}
        if not args.no_cpu_baseline:
            row["cpu_baseline"] = table_cpu_baseline(w, x, TABLE_HEADS.get(name, [(0, 0)]))
        print(json.dumps(row), flush=True)


def table_cpu_baseline(w, x, heads):
    """The fp64 oracle, forward and backward, timed on whole heads."""
    import oracle
    from io_aware_exact_tiled_gb300 import accounting as acc
    kl = x.kv_len
    pairs = acc.pairs_per_batch(w.N, w.causal, None if kl is None else kl.tolist(),
                                None if x.blockmask is None else x.blockmask.numpy(), w.B)
    t0 = time.perf_counter()
    for b, h in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        kls = None if kl is None else kl[b:b + 1]
        oracle.forward(x.q[sl], x.k[sl], x.v[sl], x.scale, causal=x.causal, kv_len=kls, blockmask=x.blockmask)
        if w.backward:
            oracle.backward(x.q[sl], x.k[sl], x.v[sl], x.do[sl], x.scale, causal=x.causal, kv_len=kls,
                            blockmask=x.blockmask)
    t = time.perf_counter() - t0
    flop = sum((14.0 if w.backward else 4.0) * w.d * pairs[b] for b, _ in heads)
    return {"value": flop / t / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "seconds_per_head": t / len(heads),
            "sample": f"fp64 NumPy {'forward + backward' if w.backward else 'forward'} of heads {heads}"}


# ------------------------------------------------------------------ decoding and packed batches
L2_FLUSH_BYTES = 512 << 20   # > the 129 MB L2: written between timed steps, outside their events


class L2Flush:
    """Writes a 512 MiB device buffer, so that no step finds the previous
    step's data in L2. Runs between timed steps, outside their events."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.i = 0

    def __call__(self):
        self.i += 1
        self.buf.fill_(self.i & 0xFF)

    describe = "a 512 MiB L2-flush write between timed steps, outside their CUDA events"


def timed_steps(fns, K, fa, flush=None):
    """Run K steps; a step calls every function of `fns` in order (each
    returns the number of kernels it launched). Each step is bracketed by its
    own CUDA events on the current stream and each call's main kernel by the
    library's timing events; `flush` runs between steps, outside the events.
    The whole loop sits between barriers over the ranks of a replica run.
    Returns (sum of the step durations in ms, [mean main-kernel ms per
    function], kernels launched)."""
    import torch

    from io_aware_exact_tiled_gb300 import replicas
    ev = lambda: torch.cuda.Event(enable_timing=True)
    steps = [(ev(), ev()) for _ in range(K)]
    kern = [[(ev(), ev()) for _ in range(K)] for _ in fns]
    for a, b in steps + [p for row in kern for p in row]:   # materialise the event handles
        a.record()
        b.record()
    torch.cuda.synchronize()
    replicas.barrier()
    torch.cuda.synchronize()
    n = 0
    for i in range(K):
        steps[i][0].record()
        for j, fn in enumerate(fns):
            fa.set_timing_events(*kern[j][i])
            n += fn()
        steps[i][1].record()
        fa.set_timing_events(None, None)
        if flush is not None:
            flush()
    torch.cuda.synchronize()
    replicas.barrier()
    total = sum(a.elapsed_time(b) for a, b in steps)
    return total, [sum(a.elapsed_time(b) for a, b in row) / K for row in kern], n


SPIN_UP_S = 0.5


def spin_up(fn, seconds=None, min_calls=3):
    """Untimed calls (beyond the warm-up steps) until the GPU has been busy
    for about `seconds` (default: the --spin-up-s option), so that its clocks
    have settled under load before the timed region starts; none when it is
    0 (deterministic launch counts, e.g. under a profiler)."""
    import torch
    seconds = SPIN_UP_S if seconds is None else min(seconds, SPIN_UP_S)
    if seconds <= 0:
        return
    t0 = time.time()
    n = 0
    while n < min_calls or time.time() - t0 < seconds:
        fn()
        n += 1
        if n % 8 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()


def e2e_simple(host_in, dev_in, host_out, dev_out, compute, K, flops_or_bytes, unit, scale=1e12):
    """End to end through the public API, one stream: every step copies its
    inputs in from pinned host memory, runs `compute` and copies its results
    back to pinned host memory. Returns the contract's e2e object."""
    import torch
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def step():
        for dst, src in zip(dev_in, host_in):
            dst.copy_(src, non_blocking=True)
        compute()
        for dst, src in zip(host_out, dev_out):
            dst.copy_(src, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    e0.record()
    for _ in range(K):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    return {"value": flops_or_bytes / (ms * 1e-3) / scale, "unit": unit,
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host_in),
            "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in host_out), "ms_per_step": ms,
            "pipeline": "one stream: copies in, compute, copies out, every step"}


def pinned_like(t):
    import torch
    return torch.empty(t.shape, dtype=t.dtype).pin_memory()


def _emit(line, rank, world, dev):
    """Print a workload's JSON line. In a replica run every rank did the same
    work: the line reports the whole job (the slowest rank's step time, the
    work of all ranks) and only rank 0 prints it."""
    from io_aware_exact_tiled_gb300 import replicas
    if world > 1:
        ms_max = replicas.max_over_ranks([line["ms_per_step"]], dev)[0]
        line["value"] = line["value"] * world * line["ms_per_step"] / ms_max
        line["ms_per_step"] = ms_max
        line["n_gpus"] = world
    if rank == 0:
        print(json.dumps(line), flush=True)
    replicas.finish()


def _clock_uuid(dev):
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return None


def _timed_with_clocks(fns, K, fa, flush, dev, rank):
    """timed_steps with the clock sampler running on rank 0; returns
    (step ms total, kernel ms list, launches, clocks summary)."""
    sampler = ClockSampler(_clock_uuid(dev))
    if rank == 0:
        sampler.start()
    wall0 = time.time()
    ms, ker, n = timed_steps(fns, K, fa, flush)
    wall1 = time.time()
    sampler.stop()
    return ms, ker, n, sampler.summary(wall0, wall1)


def run_decode(args, rank, world):
    """Split-key decoding: one step = fa_decode (split kernel + merge) for
    every (request, head) of the workload; value = cache bytes read per
    second (K and V of the valid entries; q, o and lse are added to the
    algorithmic bytes of the roofline)."""
    import torch

    import io_aware_exact_tiled_gb300 as fa
    from io_aware_exact_tiled_gb300 import workloads as W
    w = W.DECODE_WORKLOADS[args.workload]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    fa.load()
    x = W.make_decode_workload(w, seed=rank, device="cuda")
    q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
    cl = x.cache_len.to(dev)
    B, H, Nq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    ws = fa.workspace(fa.load().fa_decode_workspace_size(B, H, Nq, w.Nk, d, 0), dev)
    valid = int(x.cache_len.sum())
    cache_bytes = 2 * valid * H * d * 2
    io_bytes = 2 * q.numel() * q.element_size() + lse.numel() * 4
    flush = L2Flush(dev)

    def step():
        fa.decode(q, k, v, cache_len=cl, scale=x.scale, out=o, lse=lse, ws=ws)
        return fa.last_launch_count()

    for _ in range(max(3, args.warmup)):
        step()
    spin_up(step)
    ms, (ker_ms,), launches, clocks = _timed_with_clocks([step], args.steps, fa, flush, dev, rank)
    if fa.get_status(ws) != 0:
        raise RuntimeError("device status word reports a timed-out wait")
    ms_step = ms / args.steps
    value = cache_bytes / (ms_step * 1e-3) / 1e9
    peaks, src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    achieved = (cache_bytes + io_bytes) / (ker_ms * 1e-3) / 1e9
    e2e = None
    if not args.no_e2e:
        hq = x.q.cpu().pin_memory()
        ho, hl = pinned_like(o), pinned_like(lse)
        qd = torch.empty_like(q)
        e2e = e2e_simple([hq], [qd], [ho, hl], [o, lse],
                         lambda: fa.decode(qd, k, v, cache_len=cl, scale=x.scale, out=o, lse=lse, ws=ws),
                         max(3, min(args.steps, 50)), cache_bytes, "GB/s", 1e9)
        e2e["note"] = "the cache stays resident in HBM; q in, o and lse out per step"
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        from oracle import decode as DEC
        # two requests of the workload's shape and length range, decoded
        # repeatedly until about 10 s of CPU time is spent
        xs = W.make_decode(2, H, Nq, w.Nk, d, w.len_range, seed=0)
        t_used, nb, byt = 0.0, 0, 0
        while t_used < 10.0 and nb < 400:
            b = nb % 2
            t0 = time.perf_counter()
            DEC.decode_forward(xs.q[b:b + 1], xs.k[b:b + 1], xs.v[b:b + 1], xs.scale, xs.cache_len[b:b + 1])
            t_used += time.perf_counter() - t0
            nb += 1
            byt += 2 * int(xs.cache_len[b]) * H * d * 2
        cpu = {"value": byt / t_used / 1e9, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 NumPy decode of {nb} request-steps (all {H} heads, Nk={w.Nk}, cache_len "
                         f"U{{{w.len_range[0]}..{w.len_range[1]}}}) ({t_used:.1f} s)"}
    line = {
        "metric": "decode: KV-cache bytes read per second (split-key decoding)", "value": value, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) q and cache)",
        "config": {"workload": f"{w.name}: decode, B={B} H={H} Nq={Nq} Nk={w.Nk} d={d}, cache_len "
                               f"U{{{w.len_range[0]}..{w.len_range[1]}}}",
                   "l2": "cache larger than L2 (%d MiB of K+V allocated), and %s"
                         % (2 * k.numel() * 2 >> 20, L2Flush.describe)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": recorded_traffic("fa_decode_split_kernel", w.name),
                     "algorithmic_bytes": cache_bytes + io_bytes, "kernel": "fa_decode_split_kernel",
                     "peak_source": f"{src} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"},
        "split_kernel_ms": ker_ms, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "clocks": clocks,
    }
    _emit(line, rank, world, dev)


def run_packed(args, rank, world):
    """Packed variable-length batch: one step = fa_fwd_varlen + fa_bwd_varlen."""
    import torch

    import io_aware_exact_tiled_gb300 as fa
    from io_aware_exact_tiled_gb300 import binding as fb
    from io_aware_exact_tiled_gb300 import workloads as W
    w = W.PACKED_WORKLOADS[args.workload]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    fa.load()
    x = W.make_packed_workload(w, seed=rank, device="cuda")
    q, k, v, do = (t.to(dev) for t in (x.q, x.k, x.v, x.do))
    cu = x.cu_seqlens.to(dev)
    total, H, d = q.shape
    B = len(x.lens)
    o = torch.empty_like(q)
    lse = torch.empty((H, total), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_f = fa.workspace(256, dev)
    ws_b = fa.workspace(fb.load().fa_bwd_varlen_workspace_size(B, H, total, d), dev)
    pairs_of = lambda n: n * n / 2 if w.causal else n * n
    pairs = sum(pairs_of(n) for n in x.lens) * H
    fwd_flop, bwd_flop = 4.0 * d * pairs, 10.0 * d * pairs
    kw = dict(scale=x.scale, causal=w.causal)
    flush = L2Flush(dev)

    def fwd():
        fa.forward_varlen(q, k, v, cu, x.max_seqlen, out=o, lse=lse, ws=ws_f, **kw)
        return fa.last_launch_count()

    def bwd():
        fa.backward_varlen(q, k, v, o, lse, do, cu, x.max_seqlen, dq=dq, dk=dk, dv=dv, ws=ws_b, **kw)
        return fa.last_launch_count()

    for _ in range(max(3, args.warmup)):
        fwd()
        bwd()
    spin_up(lambda: (fwd(), bwd()))
    ms, (f_ker, b_ker), n, clocks = _timed_with_clocks([fwd, bwd], args.steps, fa, flush, dev, rank)
    if fa.get_status(ws_f) != 0 or fa.get_status(ws_b) != 0:
        raise RuntimeError("device status word reports an error")
    ms_step = ms / args.steps
    value = (fwd_flop + bwd_flop) / (ms_step * 1e-3) / 1e12
    peaks, src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    fwd_tf, bwd_tf = fwd_flop / (f_ker * 1e-3) / 1e12, bwd_flop / (b_ker * 1e-3) / 1e12
    e2e = None
    if not args.no_e2e:
        hin = [x.q.cpu().pin_memory(), x.k.cpu().pin_memory(), x.v.cpu().pin_memory(), x.do.cpu().pin_memory()]
        din = [torch.empty_like(t) for t in (q, k, v, do)]
        dout = [o, lse, dq, dk, dv]
        hout = [pinned_like(t) for t in dout]

        def compute():
            qd, kd, vd, dod = din
            fa.forward_varlen(qd, kd, vd, cu, x.max_seqlen, out=o, lse=lse, ws=ws_f, **kw)
            fa.backward_varlen(qd, kd, vd, o, lse, dod, cu, x.max_seqlen, dq=dq, dk=dk, dv=dv, ws=ws_b, **kw)

        e2e = e2e_simple(hin, din, hout, dout, compute, max(3, min(args.steps, 20)), fwd_flop + bwd_flop,
                         "TFLOP/s")
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        from oracle import varlen as VL
        xs = W.make_packed_workload(w, seed=0)
        cuh = xs.cu_seqlens.tolist()
        t_used, flop, done = 0.0, 0.0, []
        for b in range(B):
            for h in range(H):
                s, e = cuh[b], cuh[b + 1]
                one = torch.tensor([0, e - s], dtype=torch.int32)
                sub = lambda t: t[s:e][:, h:h + 1]
                t0 = time.perf_counter()
                VL.forward_varlen(sub(xs.q), sub(xs.k), sub(xs.v), one, xs.scale, causal=w.causal)
                VL.backward_varlen(sub(xs.q), sub(xs.k), sub(xs.v), sub(xs.do), one, xs.scale, causal=w.causal)
                t_used += time.perf_counter() - t0
                flop += 14.0 * d * pairs_of(e - s)
                done.append((b, h))
                if t_used >= 10.0:
                    break
            if t_used >= 10.0:
                break
        cpu = {"value": flop / t_used / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 NumPy forward + backward of {len(done)} (sequence, head) pairs of the packed "
                         f"batch, starting at sequence 0 head 0 ({t_used:.1f} s)"}
    line = {
        "metric": "packed variable-length attention fwd+bwd TFLOP/s", "value": value, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), packed)",
        "config": {"workload": f"{w.name}: B={B} sequences, lengths U{{{w.len_range[0]}..{w.len_range[1]}}} "
                               f"(total {total} tokens), H={H} d={d}, causal={w.causal}",
                   "l2": L2Flush.describe},
        "fwd": {"kernel_ms": f_ker, "tflops": fwd_tf, "pct_peak": 100 * fwd_tf / peak},
        "bwd": {"kernel_ms": b_ker, "tflops": bwd_tf, "pct_peak": 100 * bwd_tf / peak},
        "roofline": {"bound": "tensor", "achieved": bwd_tf, "peak": peak, "unit": "TFLOP/s", "frac": bwd_tf / peak,
                     "traffic": None, "kernel": "fa_bwd_kernel (packed)",
                     "peak_source": f"{src} bf16 dense burst"},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": n, "clocks": clocks,
    }
    _emit(line, rank, world, dev)


def run_fp8(args, rank, world):
    """FP8 forward (rotation + block quantisation + attention) on a dense
    workload's shape: one step = one fa_fwd_fp8 call (all its kernels)."""
    import torch

    import io_aware_exact_tiled_gb300 as fa
    from io_aware_exact_tiled_gb300 import accounting as acc
    from io_aware_exact_tiled_gb300 import workloads as W
    base = args.workload[: -len("_fp8")]
    w = W.WORKLOADS[base]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    fa.load()
    x = W.make_inputs(w, seed=rank, device="cuda")
    q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
    signs = W.make_signs(w.d, seed=rank).to(dev)
    B, H, N, d = q.shape
    kl = None if x.kv_len is None else x.kv_len.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    ws = fa.workspace(fa.load().fa_fwd_fp8_workspace_size(B, H, N, d), dev)
    fwd_flop, _ = acc.flops(B, H, N, d, x.causal, None if kl is None else x.kv_len.tolist(), None)
    flush = L2Flush(dev)

    def step():
        fa.forward_fp8(q, k, v, signs, scale=x.scale, causal=x.causal, kv_len=kl, out=o, lse=lse, ws=ws)
        return fa.last_launch_count()

    for _ in range(max(3, args.warmup)):
        step()
    spin_up(step)
    ms, (ker_ms,), launches, clocks = _timed_with_clocks([step], args.steps, fa, flush, dev, rank)
    if fa.get_status(ws) != 0:
        raise RuntimeError("device status word reports an error")
    ms_step = ms / args.steps
    peaks, src = load_peaks()
    peak8 = 2.0 * float(peaks["bf16_tflops"])
    ker_tf = fwd_flop / (ker_ms * 1e-3) / 1e12
    e2e = None
    if not args.no_e2e:
        hin = [x.q.cpu().pin_memory(), x.k.cpu().pin_memory(), x.v.cpu().pin_memory()]
        din = [torch.empty_like(t) for t in (q, k, v)]
        hout = [pinned_like(o), pinned_like(lse)]
        e2e = e2e_simple(hin, din, hout, [o, lse],
                         lambda: fa.forward_fp8(*din, signs, scale=x.scale, causal=x.causal, kv_len=kl, out=o,
                                                lse=lse, ws=ws),
                         max(3, min(args.steps, 20)), fwd_flop, "TFLOP/s")
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        from oracle import fp8 as F8
        xs = W.make_inputs(w, seed=0)
        s_cpu = W.make_signs(w.d, seed=0).numpy()
        t, f, heads = 0.0, 0.0, []
        for (bb, hh) in [(bb, hh) for bb in range(B) for hh in range(H)]:
            kls = None if xs.kv_len is None else xs.kv_len[bb:bb + 1]
            t0 = time.perf_counter()
            F8.fp8_forward(xs.q[bb:bb + 1, hh:hh + 1], xs.k[bb:bb + 1, hh:hh + 1], xs.v[bb:bb + 1, hh:hh + 1],
                           xs.scale, s_cpu, causal=xs.causal, kv_len=kls)
            t += time.perf_counter() - t0
            f += acc.flops(1, 1, N, d, x.causal, None if kls is None else kls.tolist(), None)[0]
            heads.append((bb, hh))
            if t >= 10.0:
                break
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 NumPy FP8 forward (the oracle's definition) of {len(heads)} whole head(s) "
                         f"from (0, 0) on ({t:.1f} s)"}
    line = {
        "metric": "FP8 attention forward TFLOP/s (Hadamard rotation + block-quantised E4M3)",
        "value": fwd_flop / (ms_step * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate; bf16 in and out)", "data": "synthetic (seeded N(0,1))",
        "config": {"workload": describe(w) + ", FP8 forward only", "l2": L2Flush.describe},
        "attention_kernel": {"ms": ker_ms, "tflops": ker_tf},
        "quantisation_ms": ms_step - ker_ms,
        "roofline": {"bound": "tensor", "achieved": ker_tf, "peak": peak8, "unit": "TFLOP/s", "frac": ker_tf / peak8,
                     "traffic": recorded_traffic("fa_fwd_fp8_kernel", args.workload), "kernel": "fa_fwd_fp8_kernel",
                     "peak_source": f"{src} bf16 dense burst x 2 (nominal FP8 / BF16 ratio 4.5 / 2.25)"},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
    }
    _emit(line, rank, world, dev)


def run_dropout(args, rank, world, p_drop: float = 0.1):
    """Attention fwd + bwd with fused dropout (rate 0.1) on a dense workload's
    shape: one step = fa_fwd_dropout + fa_bwd_dropout."""
    import torch

    import io_aware_exact_tiled_gb300 as fa
    from io_aware_exact_tiled_gb300 import accounting as acc
    from io_aware_exact_tiled_gb300 import workloads as W
    w = W.WORKLOADS[args.workload[: -len("_dropout")]]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    fa.load()
    x = W.make_inputs(w, seed=rank, device="cuda")
    q, k, v, do = (t.to(dev) for t in (x.q, x.k, x.v, x.do))
    kl = None if x.kv_len is None else x.kv_len.to(dev)
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_f = fa.workspace(256, dev)
    ws_b = fa.workspace(fa.bwd_workspace_size(B, H, N, d), dev)
    fwd_flop, bwd_flop = acc.flops(B, H, N, d, x.causal, None if kl is None else x.kv_len.tolist(), None)
    kw = dict(scale=x.scale, causal=x.causal, kv_len=kl)
    seed = 1234 + rank
    flush = L2Flush(dev)

    def fwd():
        fa.forward_dropout(q, k, v, p_drop, seed, out=o, lse=lse, ws=ws_f, **kw)
        return fa.last_launch_count()

    def bwd():
        fa.backward_dropout(q, k, v, o, lse, do, p_drop, seed, dq=dq, dk=dk, dv=dv, ws=ws_b, **kw)
        return fa.last_launch_count()

    for _ in range(max(3, args.warmup)):
        fwd()
        bwd()
    spin_up(lambda: (fwd(), bwd()))
    ms, (f_ker, b_ker), n, clocks = _timed_with_clocks([fwd, bwd], args.steps, fa, flush, dev, rank)
    if fa.get_status(ws_f) != 0 or fa.get_status(ws_b) != 0:
        raise RuntimeError("device status word reports an error")
    ms_step = ms / args.steps
    peaks, src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    fwd_tf, bwd_tf = fwd_flop / (f_ker * 1e-3) / 1e12, bwd_flop / (b_ker * 1e-3) / 1e12
    e2e = None
    if not args.no_e2e:
        hin = [x.q.cpu().pin_memory(), x.k.cpu().pin_memory(), x.v.cpu().pin_memory(), x.do.cpu().pin_memory()]
        din = [torch.empty_like(t) for t in (q, k, v, do)]
        dout = [o, lse, dq, dk, dv]
        hout = [pinned_like(t) for t in dout]

        def compute():
            qd, kd, vd, dod = din
            fa.forward_dropout(qd, kd, vd, p_drop, seed, out=o, lse=lse, ws=ws_f, **kw)
            fa.backward_dropout(qd, kd, vd, o, lse, dod, p_drop, seed, dq=dq, dk=dk, dv=dv, ws=ws_b, **kw)

        e2e = e2e_simple(hin, din, hout, dout, compute, max(3, min(args.steps, 20)), fwd_flop + bwd_flop,
                         "TFLOP/s")
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        from oracle import dropout as DR
        from oracle.attention import visible
        import numpy as np
        xs = W.make_inputs(w, seed=0)
        kls = None if xs.kv_len is None else xs.kv_len[:1]
        t, f, done = 0.0, 0.0, 0
        # query rows of head (0, 0) from the last (the most visible keys under
        # a causal mask) backwards, 1024 at a time, until about 10 s are spent
        for r1 in range(N, 0, -1024):
            rows = (max(0, r1 - 1024), r1)
            t0 = time.perf_counter()
            DR.forward(xs.q[:1, :1], xs.k[:1, :1], xs.v[:1, :1], xs.scale, p_drop, 1234, causal=xs.causal,
                       kv_len=kls, rows=rows)
            DR.backward(xs.q[:1, :1], xs.k[:1, :1], xs.v[:1, :1], xs.do[:1, :1], xs.scale, p_drop, 1234,
                        causal=xs.causal, kv_len=kls, rows=rows)
            t += time.perf_counter() - t0
            vis = visible(N, xs.causal, None if kls is None else int(kls[0]), None, np.arange(*rows))
            f += 14.0 * d * float(vis.sum())
            done += rows[1] - rows[0]
            if t >= 10.0:
                break
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 NumPy dropout forward + backward of the last {done} query rows of head (0, 0) "
                         f"({t:.1f} s)"}
    line = {
        "metric": f"attention fwd+bwd with fused dropout (p = {p_drop}) TFLOP/s", "unit": "TFLOP/s",
        "value": (fwd_flop + bwd_flop) / (ms_step * 1e-3) / 1e12, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1))",
        "config": {"workload": describe(w) + f", dropout p = {p_drop} (Philox-4x32-10 masks)",
                   "l2": L2Flush.describe},
        "fwd": {"kernel_ms": f_ker, "tflops": fwd_tf, "pct_peak": 100 * fwd_tf / peak},
        "bwd": {"kernel_ms": b_ker, "tflops": bwd_tf, "pct_peak": 100 * bwd_tf / peak},
        "roofline": {"bound": "tensor", "achieved": bwd_tf, "peak": peak, "unit": "TFLOP/s", "frac": bwd_tf / peak,
                     "traffic": None, "kernel": "fa_bwd_kernel (dropout)", "peak_source": f"{src} bf16 dense burst"},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": n, "clocks": clocks,
    }
    _emit(line, rank, world, dev)


# ------------------------------------------------------------------ our arm
TARGET_WORKLOADS = ("long4k", "long8k", "sparse16k")   # the N >= 4096, d = 128 configs


class DenseCase:
    """Device buffers and step functions of one dense workload."""

    def __init__(self, w, dev, seed):
        import torch

        import io_aware_exact_tiled_gb300 as fa
        from io_aware_exact_tiled_gb300 import accounting as acc
        from io_aware_exact_tiled_gb300 import workloads as W
        self.w = w
        x = W.make_inputs(w, seed=seed, device="cuda")
        self.x = x
        self.q, self.k, self.v, self.do = (t.to(dev) for t in (x.q, x.k, x.v, x.do))
        self.bm = None if x.blockmask is None else x.blockmask.to(dev)
        self.kl = None if x.kv_len is None else x.kv_len.to(dev)
        B, H, N, d = self.q.shape
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = (torch.empty_like(self.q) for _ in range(3))
        self.ws_f = fa.workspace(256, dev)
        self.ws_b = fa.workspace(fa.bwd_workspace_size(B, H, N, d), dev)
        self.kw = dict(scale=x.scale, causal=x.causal, blockmask=self.bm, kv_len=self.kl)
        self.fwd_flop, self.bwd_flop = acc.flops(B, H, N, d, x.causal,
                                                 None if self.kl is None else x.kv_len.tolist(),
                                                 None if self.bm is None else x.blockmask.cpu().numpy())
        self.fa = fa

    def fwd(self):
        self.fa.forward(self.q, self.k, self.v, out=self.o, lse=self.lse, ws=self.ws_f, **self.kw)
        return self.fa.last_launch_count()

    def bwd(self):
        self.fa.backward(self.q, self.k, self.v, self.o, self.lse, self.do, dq=self.dq, dk=self.dk, dv=self.dv,
                         ws=self.ws_b, **self.kw)
        return self.fa.last_launch_count()

    def check_status(self):
        if self.fa.get_status(self.ws_f) != 0 or self.fa.get_status(self.ws_b) != 0:
            raise RuntimeError("device status word reports a timed-out wait")


def target_row(case, ms_step, fwd_ms, bwd_ms, peak):
    fwd_tf = case.fwd_flop / (fwd_ms * 1e-3) / 1e12
    bwd_tf = case.bwd_flop / (bwd_ms * 1e-3) / 1e12
    return {"workload": describe(case.w), "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "step_ms": ms_step,
            "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
            "fwd_pct_peak": 100 * fwd_tf / peak, "bwd_pct_peak": 100 * bwd_tf / peak,
            "step_tflops": (case.fwd_flop + case.bwd_flop) / (ms_step * 1e-3) / 1e12,
            "fwd_meets_60pct": fwd_tf >= 0.6 * peak, "bwd_meets_45pct": bwd_tf >= 0.45 * peak}


def main():
    global SPIN_UP_S
    args = parse()
    SPIN_UP_S = args.spin_up_s
    if args.table:
        return run_table(args)
    from io_aware_exact_tiled_gb300 import replicas
    rank, world, local = replicas.env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    from io_aware_exact_tiled_gb300 import workloads as W_
    if world > 1:
        # replica run: one process per GPU under torchrun
        import torch
        torch.cuda.set_device(local)
        replicas.init("nccl", world)
    if args.workload in W_.DECODE_WORKLOADS:
        return run_decode(args, rank, world)
    if args.workload in W_.PACKED_WORKLOADS:
        return run_packed(args, rank, world)
    if args.workload.endswith("_fp8") and args.workload[:-4] in W_.WORKLOADS:
        return run_fp8(args, rank, world)
    if args.workload.endswith("_dropout") and args.workload[: -len("_dropout")] in W_.WORKLOADS:
        return run_dropout(args, rank, world)

    import torch

    import io_aware_exact_tiled_gb300 as fa
    from io_aware_exact_tiled_gb300 import workloads as W

    if world > 1:
        torch.cuda.set_device(local)
    replicas.init("nccl", world)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load()
    peaks, peaks_src = load_peaks()
    peak = float(peaks["bf16_tflops"])

    w = W.WORKLOADS[args.workload]
    case = DenseCase(w, dev, seed=rank)
    q, k, v, do, o, lse = case.q, case.k, case.v, case.do, case.o, case.lse
    B, H, N, d = q.shape
    fwd_flop, bwd_flop = case.fwd_flop, case.bwd_flop
    flush = L2Flush(dev)

    for _ in range(max(3, args.warmup)):
        case.fwd()
        case.bwd()
    torch.cuda.synchronize()
    case.check_status()
    spin_up(lambda: (case.fwd(), case.bwd()))

    # the timed region: K steps, each bracketed by its own events, the main
    # kernels by the library's events, an L2 flush between steps
    K = args.steps
    ms, (fwd_ms, bwd_ms), launches, clocks = _timed_with_clocks([case.fwd, case.bwd], K, fa, flush, dev, rank)
    case.check_status()
    # the slowest rank's times; every rank did the same work
    ms, fwd_ms, bwd_ms = replicas.max_over_ranks([ms, fwd_ms, bwd_ms], dev)
    ms_step = ms / K
    total_flop = (fwd_flop + bwd_flop) * world
    value = replicas.whole_job_rate(fwd_flop + bwd_flop, ms_step * 1e-3, world) / 1e12

    # ---------------- end to end through the public API with host buffers
    # Every step copies its inputs in from pinned host memory, runs forward
    # and backward through the public API and copies O, L, dQ, dK, dV back.
    # The copies run on their own streams with two sets of device buffers, so
    # step k + 1's inputs travel in and step k - 1's results travel out while
    # step k computes (the way an input pipeline feeds a training step).
    e2e = None
    if not args.no_e2e:
        ev = lambda: torch.cuda.Event(enable_timing=True)
        kw, ws_f, ws_b = case.kw, case.ws_f, case.ws_b
        hq, hk, hv, hdo = (t.cpu().pin_memory() for t in (q, k, v, do))
        nbuf = 2
        din = [tuple(torch.empty_like(t) for t in (q, k, v, do)) for _ in range(nbuf)]
        dout = [(torch.empty_like(q), torch.empty_like(lse), torch.empty_like(q), torch.empty_like(k),
                 torch.empty_like(v)) for _ in range(nbuf)]
        hout = [(torch.empty_like(hq).pin_memory(), torch.empty(lse.shape, dtype=torch.float32).pin_memory(),
                 torch.empty_like(hq).pin_memory(), torch.empty_like(hk).pin_memory(),
                 torch.empty_like(hv).pin_memory()) for _ in range(nbuf)]
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [ev() for _ in range(nbuf)]
        ev_cmp = [ev() for _ in range(nbuf)]
        ev_out = [ev() for _ in range(nbuf)]
        started = [False] * nbuf

        def e2e_step(kstep):
            bi = kstep % nbuf
            qd, kd, vd, dod = din[bi]
            o_, l_, dq_, dk_, dv_ = dout[bi]
            with torch.cuda.stream(s_in):
                if started[bi]:
                    s_in.wait_event(ev_cmp[bi])  # step k - 2 has finished reading these inputs
                for dst, src in ((qd, hq), (kd, hk), (vd, hv), (dod, hdo)):
                    dst.copy_(src, non_blocking=True)
                ev_in[bi].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[bi])
                if started[bi]:
                    s_cmp.wait_event(ev_out[bi])  # step k - 2's results have been copied out
                fa.forward(qd, kd, vd, out=o_, lse=l_, ws=ws_f, **kw)
                fa.backward(qd, kd, vd, o_, l_, dod, dq=dq_, dk=dk_, dv=dv_, ws=ws_b, **kw)
                ev_cmp[bi].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[bi])
                for dst, src in zip(hout[bi], dout[bi]):
                    dst.copy_(src, non_blocking=True)
                ev_out[bi].record(s_out)
            started[bi] = True

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        K2 = max(3, min(K, 30))
        e0, e1 = ev(), ev()
        replicas.barrier()
        e0.record(s_in)
        for i in range(K2):
            e2e_step(3 + i)
        e1.record(s_out)  # after the last step's results are copied out
        torch.cuda.synchronize()
        ems = replicas.max_over_ranks([e0.elapsed_time(e1)], dev)[0]
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
        d2h = sum(t.numel() * t.element_size() for t in hout[0])
        e2e = {"value": total_flop / (ems / K2 * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems / K2,
               "pipeline": "copies in / compute / copies out on three streams, two device buffer sets"}
        # the last step's results are the ones a caller would read
        assert torch.equal(hout[(3 + K2 - 1) % nbuf][0].view(torch.int16),
                           dout[(3 + K2 - 1) % nbuf][0].cpu().view(torch.int16))
        del din, dout, hout

    # ---------------- the other N >= 4096, d = 128 configurations, same protocol
    targets = None
    if world == 1 and not args.no_targets:
        targets = {w.name: target_row(case, ms_step, fwd_ms, bwd_ms, peak)}
        Kt = max(5, min(K, 50))
        for name in TARGET_WORKLOADS:
            if name == w.name:
                continue
            c2 = DenseCase(W.WORKLOADS[name], dev, seed=0)
            for _ in range(3):
                c2.fwd()
                c2.bwd()
            spin_up(lambda: (c2.fwd(), c2.bwd()), seconds=0.2)
            ms2, (f2, b2), _ = timed_steps([c2.fwd, c2.bwd], Kt, fa, flush)
            c2.check_status()
            targets[name] = target_row(c2, ms2 / Kt, f2, b2, peak)
            targets[name]["steps"] = Kt
            del c2
            torch.cuda.empty_cache()

    if rank != 0:
        replicas.finish()
        return

    fwd_tf = fwd_flop / (fwd_ms * 1e-3) / 1e12
    bwd_tf = bwd_flop / (bwd_ms * 1e-3) / 1e12
    # bf16 [B, H, N, d] forwards without dropout run fa_fwd_t1_kernel
    dominant = "fa_bwd_kernel" if bwd_ms >= fwd_ms else "fa_fwd_t1_kernel"
    dom_tf = bwd_tf if dominant == "fa_bwd_kernel" else fwd_tf
    roofline = {"bound": "tensor", "achieved": dom_tf, "peak": peak, "unit": "TFLOP/s", "frac": dom_tf / peak,
                "traffic": recorded_traffic(dominant, args.workload), "kernel": dominant,
                "peak_source": f"{peaks_src} bf16 dense burst (MEASURED_PEAKS.json bf16_tflops)"
                if peaks_src == "measured" else "fallback 1.9 PFLOP/s bf16 burst"}

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        xs = W.make_inputs(w, seed=0)
        f, t, heads = oracle_sample(w, xs)
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 NumPy forward + backward of {len(heads)} whole head(s) {heads} of the workload "
                         f"({t:.1f} s; BLAS threads = all cores, exp single-threaded)"}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q, K, V, dO in bf16)",
        "config": {"workload": describe(w), "B": B, "H": H, "N": N, "d": d, "causal": bool(case.x.causal),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (Q, K, V, O, dO = %d MiB each vs 129 MB L2), and %s"
                         % (q.numel() * q.element_size() >> 20, L2Flush.describe)},
        "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "pct_peak": 100 * fwd_tf / peak},
        "bwd": {"ms": bwd_ms, "tflops": bwd_tf, "pct_peak": 100 * bwd_tf / peak,
                "note": "fa_bwd_kernel alone; the D preprocess and dQ conversion kernels are in ms_per_step"},
        "pct_peak_step": 100 * value / world / peak,
        "targets": targets,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "peak_memory_bytes": torch.cuda.max_memory_allocated(dev),
    }
    print(json.dumps(line), flush=True)
    replicas.finish()


if __name__ == "__main__":
    main()
