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
DEFAULT_WORKLOAD = "long8k"
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
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 100 ms."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd[1:1] = ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t0 = None

        def reader():
            for line in self.proc.stdout:
                self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        time.sleep(0.6)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_begin, t_end):
        rows = [r for (t, r) in self.rows if t_begin <= t <= t_end + 0.05 and len(r) >= 10]
        if not rows:
            rows = [r for (_, r) in self.rows if len(r) >= 10][-3:]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for k, name in enumerate(names):
                if r[6 + k].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][3]), "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max((num(r[4]) or 0.0) for r in rows)}


# ------------------------------------------------------------------ helpers
# source files each profiled kernel is compiled from (its .cu plus the shared
# headers); a recorded DRAM-traffic figure stays valid while they are unchanged
KERNEL_SOURCES = {
    "fa_fwd_kernel": ["fa_fwd.cu"],
    "fa_fwd_fp8_kernel": ["fa_fwd_fp8.cu", "fa_fp8.h"],
    "fa_bwd_kernel": ["fa_bwd.cu"],
    "fa_fwd_q1_kernel": ["fa_fwd_q1.cu"],
    "fa_decode_split_kernel": ["fa_decode.cu", "fa_decode.h"],
}
SHARED_HEADERS = ["fa_common.cuh", "fa_launch.h", "sm103_ptx.cuh", "tmap.h"]


def kernel_source_sha(kernel: str):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "io_aware_exact_tiled_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES.get(kernel, []) + SHARED_HEADERS):
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
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
        "config": {"workload": describe(w)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: fp64 NumPy forward + backward of the last {R} query rows of head "
                                   f"(0, 0) (N={w.N}, d={w.d}) on the host cores (BLAS threads = all cores; exp "
                                   f"single-threaded)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ per-workload table
TABLE_HEADS = {"tiny": None, "bert": None, "gpt2": None, "long4k": [(0, 0), (0, 31)],
               "long8k": [(0, 0), (0, 31)], "sparse16k": [(0, 0), (1, 15)]}


def run_table(args):
    import numpy as np
    import torch

    import io_aware_exact_tiled_gb300 as fa
    import oracle
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
        g = {"o": o.float().cpu().numpy(), "lse": lse.cpu().numpy()}
        if w.backward:
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            bcall, bker = timed(lambda: fa.backward(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, ws=ws_b, **kw))
            row["bwd"] = {"call_ms": bcall, "kernel_ms": bker, "tflops_call": bwd_flop / (bcall * 1e-3) / 1e12,
                          "tflops_kernel": bwd_flop / (bker * 1e-3) / 1e12,
                          "pct_peak_kernel": 100 * bwd_flop / (bker * 1e-3) / 1e12 / peak}
            g.update(dq=dq.float().cpu().numpy(), dk=dk.float().cpu().numpy(), dv=dv.float().cpu().numpy())
        heads = TABLE_HEADS.get(name)
        okw = dict(causal=x.causal, kv_len=x.kv_len, blockmask=x.blockmask, heads=heads)
        t0 = time.perf_counter()
        O, L = oracle.forward(x.q, x.k, x.v, x.scale, **okw)
        sel = (slice(None),) if heads is None else tuple(np.array(ix) for ix in zip(*heads))
        err = {"o_maxabs": float(np.abs(g["o"][sel] - O[sel]).max()),
               "lse_maxabs": float(np.nanmax(np.where(np.isneginf(L[sel]) & np.isneginf(g["lse"][sel]), 0.0,
                                                      np.abs(g["lse"][sel] - L[sel]))))}
        if w.backward:
            dQ, dK, dV = oracle.backward(x.q, x.k, x.v, x.do, x.scale, **okw)
            for n, ref in (("dq", dQ), ("dk", dK), ("dv", dV)):
                err[n + "_rel"] = float(np.linalg.norm(g[n][sel] - ref[sel]) / np.linalg.norm(ref[sel]))
        t_oracle = time.perf_counter() - t0
        nheads = B * H if heads is None else len(heads)
        row["errors"] = err
        row["errors_on"] = "all heads" if heads is None else f"heads {heads}"
        row["oracle_cpu_s_per_head"] = t_oracle / nheads
        row["oracle_cores"] = os.cpu_count()
        print(json.dumps(row), flush=True)


# ------------------------------------------------------------------ decoding and packed batches
def _timed_loop(fn, K, ev, fa):
    """Run fn K times with the library's main-kernel events, between barriers
    over the ranks of a replica run; returns (total ms, mean main-kernel ms,
    launches)."""
    import torch

    from io_aware_exact_tiled_gb300 import replicas
    pairs = [(ev(), ev()) for _ in range(K)]
    for a, b in pairs:
        a.record()
        b.record()
    t0, t1 = ev(), ev()
    torch.cuda.synchronize()
    replicas.barrier()
    n = 0
    t0.record()
    for i in range(K):
        fa.set_timing_events(*pairs[i])
        n += fn()
    t1.record()
    fa.set_timing_events(None, None)
    torch.cuda.synchronize()
    replicas.barrier()
    return t0.elapsed_time(t1), sum(a.elapsed_time(b) for a, b in pairs) / K, n


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
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def step():
        fa.decode(q, k, v, cache_len=cl, scale=x.scale, out=o, lse=lse, ws=ws)
        return fa.last_launch_count()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler()
    sampler.start()
    wall0 = time.time()
    ms, ker_ms, launches = _timed_loop(step, args.steps, ev, fa)
    wall1 = time.time()
    sampler.stop()
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
        ho = torch.empty_like(hq).pin_memory()
        hl = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
        qd = torch.empty_like(q)

        def e2e_step():
            qd.copy_(hq, non_blocking=True)
            fa.decode(qd, k, v, cache_len=cl, scale=x.scale, out=o, lse=lse, ws=ws)
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)
            return 0

        for _ in range(3):
            e2e_step()
        e_ms, _, _ = _timed_loop(e2e_step, max(3, min(args.steps, 50)), ev, fa)
        e_step = e_ms / max(3, min(args.steps, 50))
        e2e = {"value": cache_bytes / (e_step * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": hq.numel() * 2, "d2h_bytes_per_step": ho.numel() * 2 + hl.numel() * 4,
               "ms_per_step": e_step, "note": "the cache stays resident in HBM; q in, o and lse out per step"}
    cpu = None
    if not args.no_cpu_baseline:
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
                   "l2": "cache larger than L2 (%d MiB of K+V allocated)" % (2 * k.numel() * 2 >> 20)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": recorded_traffic("fa_decode_split_kernel", w.name),
                     "algorithmic_bytes": cache_bytes + io_bytes, "kernel": "fa_decode_split_kernel",
                     "peak_source": f"{src} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"},
        "split_kernel_ms": ker_ms, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "clocks": sampler.summary(wall0, wall1),
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
    pairs = sum((n * n / 2 if w.causal else n * n) for n in x.lens) * H
    fwd_flop, bwd_flop = 4.0 * d * pairs, 10.0 * d * pairs
    ev = lambda: torch.cuda.Event(enable_timing=True)
    kw = dict(scale=x.scale, causal=w.causal)

    def fwd():
        fa.forward_varlen(q, k, v, cu, x.max_seqlen, out=o, lse=lse, ws=ws_f, **kw)
        return fa.last_launch_count()

    def bwd():
        fa.backward_varlen(q, k, v, o, lse, do, cu, x.max_seqlen, dq=dq, dk=dk, dv=dv, ws=ws_b, **kw)
        return fa.last_launch_count()

    for _ in range(max(3, args.warmup)):
        fwd()
        bwd()
    torch.cuda.synchronize()
    sampler = ClockSampler()
    sampler.start()
    wall0 = time.time()
    f_ms, f_ker, nf = _timed_loop(fwd, args.steps, ev, fa)
    b_ms, b_ker, nb = _timed_loop(bwd, args.steps, ev, fa)
    wall1 = time.time()
    sampler.stop()
    if fa.get_status(ws_f) != 0 or fa.get_status(ws_b) != 0:
        raise RuntimeError("device status word reports an error")
    ms_step = (f_ms + b_ms) / args.steps
    value = (fwd_flop + bwd_flop) / (ms_step * 1e-3) / 1e12
    peaks, src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    fwd_tf, bwd_tf = fwd_flop / (f_ker * 1e-3) / 1e12, bwd_flop / (b_ker * 1e-3) / 1e12
    line = {
        "metric": "packed variable-length attention fwd+bwd TFLOP/s", "value": value, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), packed)",
        "config": {"workload": f"{w.name}: B={B} sequences, lengths U{{{w.len_range[0]}..{w.len_range[1]}}} "
                               f"(total {total} tokens), H={H} d={d}, causal={w.causal}"},
        "fwd": {"kernel_ms": f_ker, "tflops": fwd_tf, "pct_peak": 100 * fwd_tf / peak},
        "bwd": {"kernel_ms": b_ker, "tflops": bwd_tf, "pct_peak": 100 * bwd_tf / peak},
        "roofline": {"bound": "tensor", "achieved": bwd_tf, "peak": peak, "unit": "TFLOP/s", "frac": bwd_tf / peak,
                     "traffic": None, "kernel": "fa_bwd_kernel (packed)",
                     "peak_source": f"{src} bf16 dense burst"},
        "cpu_baseline": None, "e2e": None, "gpu_launches": nf + nb, "clocks": sampler.summary(wall0, wall1),
    }
    _emit(line, rank, world, dev)


def run_fp8(args, rank, world):
    """FP8 forward (rotation + block quantisation + attention) on a dense
    workload's shape: one step = one fa_fwd_fp8 call (all five kernels)."""
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
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def step():
        fa.forward_fp8(q, k, v, signs, scale=x.scale, causal=x.causal, kv_len=kl, out=o, lse=lse, ws=ws)
        return fa.last_launch_count()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler()
    sampler.start()
    wall0 = time.time()
    ms, ker_ms, launches = _timed_loop(step, args.steps, ev, fa)
    wall1 = time.time()
    sampler.stop()
    if fa.get_status(ws) != 0:
        raise RuntimeError("device status word reports an error")
    ms_step = ms / args.steps
    peaks, src = load_peaks()
    peak8 = 2.0 * float(peaks["bf16_tflops"])
    ker_tf = fwd_flop / (ker_ms * 1e-3) / 1e12
    line = {
        "metric": "FP8 attention forward TFLOP/s (Hadamard rotation + block-quantised E4M3)",
        "value": fwd_flop / (ms_step * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate; bf16 in and out)", "data": "synthetic (seeded N(0,1))",
        "config": {"workload": describe(w) + ", FP8 forward only"},
        "attention_kernel": {"ms": ker_ms, "tflops": ker_tf},
        "quantisation_ms": ms_step - ker_ms,
        "roofline": {"bound": "tensor", "achieved": ker_tf, "peak": peak8, "unit": "TFLOP/s", "frac": ker_tf / peak8,
                     "traffic": recorded_traffic("fa_fwd_fp8_kernel", args.workload), "kernel": "fa_fwd_fp8_kernel",
                     "peak_source": f"{src} bf16 dense burst x 2 (nominal FP8 / BF16 ratio 4.5 / 2.25)"},
        "cpu_baseline": None, "e2e": None, "gpu_launches": launches, "clocks": sampler.summary(wall0, wall1),
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
    ev = lambda: torch.cuda.Event(enable_timing=True)
    kw = dict(scale=x.scale, causal=x.causal, kv_len=kl)
    seed = 1234 + rank

    def fwd():
        fa.forward_dropout(q, k, v, p_drop, seed, out=o, lse=lse, ws=ws_f, **kw)
        return fa.last_launch_count()

    def bwd():
        fa.backward_dropout(q, k, v, o, lse, do, p_drop, seed, dq=dq, dk=dk, dv=dv, ws=ws_b, **kw)
        return fa.last_launch_count()

    for _ in range(max(3, args.warmup)):
        fwd()
        bwd()
    torch.cuda.synchronize()
    sampler = ClockSampler()
    sampler.start()
    wall0 = time.time()
    f_ms, f_ker, nf = _timed_loop(fwd, args.steps, ev, fa)
    b_ms, b_ker, nb = _timed_loop(bwd, args.steps, ev, fa)
    wall1 = time.time()
    sampler.stop()
    if fa.get_status(ws_f) != 0 or fa.get_status(ws_b) != 0:
        raise RuntimeError("device status word reports an error")
    ms_step = (f_ms + b_ms) / args.steps
    peaks, src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    fwd_tf, bwd_tf = fwd_flop / (f_ker * 1e-3) / 1e12, bwd_flop / (b_ker * 1e-3) / 1e12
    line = {
        "metric": f"attention fwd+bwd with fused dropout (p = {p_drop}) TFLOP/s", "unit": "TFLOP/s",
        "value": (fwd_flop + bwd_flop) / (ms_step * 1e-3) / 1e12, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1))",
        "config": {"workload": describe(w) + f", dropout p = {p_drop} (Philox-4x32-10 masks)"},
        "fwd": {"kernel_ms": f_ker, "tflops": fwd_tf, "pct_peak": 100 * fwd_tf / peak},
        "bwd": {"kernel_ms": b_ker, "tflops": bwd_tf, "pct_peak": 100 * bwd_tf / peak},
        "roofline": {"bound": "tensor", "achieved": bwd_tf, "peak": peak, "unit": "TFLOP/s", "frac": bwd_tf / peak,
                     "traffic": None, "kernel": "fa_bwd_kernel (dropout)", "peak_source": f"{src} bf16 dense burst"},
        "cpu_baseline": None, "e2e": None, "gpu_launches": nf + nb, "clocks": sampler.summary(wall0, wall1),
    }
    _emit(line, rank, world, dev)


# ------------------------------------------------------------------ our arm
def main():
    args = parse()
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
    from io_aware_exact_tiled_gb300 import accounting as acc
    from io_aware_exact_tiled_gb300 import workloads as W

    if world > 1:
        torch.cuda.set_device(local)
    replicas.init("nccl", world)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load()

    w = W.WORKLOADS[args.workload]
    x = W.make_inputs(w, seed=rank, device="cuda")
    q, k, v, do = (t.to(dev) for t in (x.q, x.k, x.v, x.do))
    bm = None if x.blockmask is None else x.blockmask.to(dev)
    kl = None if x.kv_len is None else x.kv_len.to(dev)
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_f = fa.workspace(256, dev)
    ws_b = fa.workspace(fa.bwd_workspace_size(B, H, N, d), dev)
    kw = dict(scale=x.scale, causal=x.causal, blockmask=bm, kv_len=kl)
    fwd_flop, bwd_flop = acc.flops(B, H, N, d, x.causal, None if kl is None else x.kv_len.tolist(),
                                   None if bm is None else x.blockmask.numpy())
    launches = [0]

    def step():
        fa.forward(q, k, v, out=o, lse=lse, ws=ws_f, **kw)
        launches[0] += fa.last_launch_count()
        fa.backward(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, ws=ws_b, **kw)
        launches[0] += fa.last_launch_count()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if fa.get_status(ws_f) != 0 or fa.get_status(ws_b) != 0:
        raise RuntimeError("device status word reports a timed-out wait")

    # per-kernel events (the library records them around its main kernels)
    K = args.steps
    ev = lambda: torch.cuda.Event(enable_timing=True)
    fb_ev = [(ev(), ev()) for _ in range(K)]
    bb_ev = [(ev(), ev()) for _ in range(K)]
    for a, b in fb_ev + bb_ev:   # materialise the event handles
        a.record()
        b.record()
    t_start, t_stop = ev(), ev()
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    if rank == 0:
        sampler.start()
    replicas.barrier()
    torch.cuda.synchronize()
    launches[0] = 0
    wall0 = time.time()
    t_start.record()
    for i in range(K):
        fa.set_timing_events(*fb_ev[i])
        fa.forward(q, k, v, out=o, lse=lse, ws=ws_f, **kw)
        launches[0] += fa.last_launch_count()
        fa.set_timing_events(*bb_ev[i])
        fa.backward(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, ws=ws_b, **kw)
        launches[0] += fa.last_launch_count()
    t_stop.record()
    fa.set_timing_events(None, None)
    torch.cuda.synchronize()
    wall1 = time.time()
    replicas.barrier()
    sampler.stop()
    st_f, st_b = fa.get_status(ws_f), fa.get_status(ws_b)
    if st_f != 0 or st_b != 0:
        raise RuntimeError("device status word reports a timed-out wait")
    ms = t_start.elapsed_time(t_stop)
    fwd_ms = sum(a.elapsed_time(b) for a, b in fb_ev) / K
    bwd_ms = sum(a.elapsed_time(b) for a, b in bb_ev) / K
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
        assert torch.equal(hout[(3 + K2 - 1) % nbuf][0].view(torch.int16), dout[(3 + K2 - 1) % nbuf][0].cpu().view(torch.int16))

    if rank != 0:
        replicas.finish()
        return

    peaks, peaks_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    fwd_tf = fwd_flop / (fwd_ms * 1e-3) / 1e12
    bwd_tf = bwd_flop / (bwd_ms * 1e-3) / 1e12
    dominant = "fa_bwd_kernel" if bwd_ms >= fwd_ms else "fa_fwd_kernel"
    dom_tf = bwd_tf if dominant == "fa_bwd_kernel" else fwd_tf
    roofline = {"bound": "tensor", "achieved": dom_tf, "peak": peak, "unit": "TFLOP/s", "frac": dom_tf / peak,
                "traffic": recorded_traffic(dominant, args.workload), "kernel": dominant,
                "peak_source": f"{peaks_src} bf16 dense burst (MEASURED_PEAKS.json bf16_tflops)"
                if peaks_src == "measured" else "fallback 1.9 PFLOP/s bf16 burst"}
    clocks = sampler.summary(wall0, wall1)

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
        "config": {"workload": describe(w), "B": B, "H": H, "N": N, "d": d, "causal": bool(x.causal),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (Q, K, V, O, dO = %d MiB each vs 129 MB L2)"
                         % (q.numel() * q.element_size() >> 20)},
        "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "pct_peak": 100 * fwd_tf / peak},
        "bwd": {"ms": bwd_ms, "tflops": bwd_tf, "pct_peak": 100 * bwd_tf / peak,
                "note": "fa_bwd_kernel alone; the D preprocess and dQ conversion kernels are in ms_per_step"},
        "pct_peak_step": 100 * value / world / peak,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches[0],
        "clocks": clocks,
        "peak_memory_bytes": torch.cuda.max_memory_allocated(dev),
    }
    print(json.dumps(line), flush=True)
    replicas.finish()


if __name__ == "__main__":
    main()
