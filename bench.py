#!/usr/bin/env python
"""Benchmark of the k-quant weight matmul on GB300.

Headline (one JSON line on stdout): decode weight GB/s of the Q4_K x Q8_1
matvec on W[4096, 11008] and W[11008, 4096] (x fp32 N(0,1), Q8_1 quantisation
fused). A step is one decode sweep over 8 rotated weight copies of each shape
(16 launches, 406 MB of weights: larger than the 129 MB L2, so no flush is
needed). Extra keys report the prefill GEMMs (N = 64, 512, 2048; Q4_K and Q6_K)
and the MoE grouped GEMM as TFLOP/s, each call timed cold (L2 flushed between
calls: a 256 MB write, then a 256 MB read so no dirty flush data is left).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas; the path is not sharded), timing is the max over ranks, and the
value is the sum over ranks. ``--impl reference`` times the CPU oracle on
bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DECODE_SHAPES = [(4096, 11008), (11008, 4096)]
DECODE_COPIES = 8
Q4K_ROW = lambda K: (K // 256) * 144          # noqa: E731
METRIC = "Q4_K matmul: decode weight GB/s, prefill TFLOP/s, % of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------
def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-sections", action="store_true", help="skip the prefill/MoE sections")
    p.add_argument("--section-iters", type=int, default=10)
    p.add_argument("--only", default=None,
                   help="profiling aid: run only 'decode' or one section (prefill_*/moe_*/decode_*/mma_rate) and print its numbers")
    p.add_argument("--eager", action="store_true", help="launch the decode step eagerly instead of as a CUDA graph")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class Dist:
    def __init__(self, n_gpus):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s, p in zip(sm, power) if p is not None] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


def traffic_for(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if the
    kernel source is unchanged since the capture (else None): (read + write,
    read, write)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None, None, None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or sources_digest(e["sources"]) != e["sources_sha256_16"]:
        return None, None, None
    return e["dram_bytes_per_launch"], e.get("dram_read_bytes_per_launch"), e.get("dram_write_bytes_per_launch")


def sources_digest(sources) -> str:
    """First 16 hex digits of the SHA-256 of the listed files, concatenated."""
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------
# CPU oracle timing (spawned, single-threaded, never after a CUDA fork)
# ----------------------------------------------------------------------------
def _oracle_decode_sample(rows: int, reps: int, min_seconds: float):
    """Runs the oracle matvec on the first `rows` rows of each decode shape;
    returns (weight bytes, seconds)."""
    import numpy as np
    from oracle import kq_oracle as ora
    from quantized_weight_matmul_q4_gb300 import synthetic as syn
    data = []
    for (M, K) in DECODE_SHAPES:
        rng = np.random.default_rng(M)
        W = syn.q4_k_weights(rng, rows, K)
        x = syn.activations(rng, K, 1)
        data.append((W, x, K))
    nbytes = 0
    t0 = time.perf_counter()
    done = 0
    while done < reps or time.perf_counter() - t0 < min_seconds:
        for W, x, K in data:
            ora.matmul("q4_k", W, x, W.shape[0], K)
            nbytes += W.nbytes
        done += 1
        if done >= 2000:
            break
    return nbytes, time.perf_counter() - t0


def _oracle_worker_init():
    # one thread per worker process (set before numpy loads)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    os.environ["CUDA_VISIBLE_DEVICES"] = ""


def _oracle_worker(args):
    rows, reps, min_seconds = args
    return _oracle_decode_sample(rows, reps, min_seconds)


class OraclePool:
    """`procs` single-threaded oracle processes, started once with the spawn
    method (never a fork of a process that has used CUDA)."""

    def __init__(self, procs: int):
        import multiprocessing as mp
        self.procs = procs
        self.pool = mp.get_context("spawn").Pool(procs, initializer=_oracle_worker_init)
        self.pool.map(_oracle_worker, [(8, 1, 0.0)] * procs)  # imports and first calls

    def gbs(self, rows: int, reps: int, min_seconds: float):
        """Every process runs the sample at once: GB/s of weights summed over the
        processes, over the longest process's timed loop; and that time."""
        res = self.pool.map(_oracle_worker, [(rows, reps, min_seconds)] * self.procs)
        secs = max(r[1] for r in res)
        return sum(r[0] for r in res) / secs / 1e9, secs

    def close(self):
        self.pool.close()
        self.pool.join()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_baseline(rows: int, min_seconds: float) -> dict:
    """The oracle as it stands on the host: all cores (one single-threaded
    process per core) and one thread."""
    cores = host_cores()
    pool = OraclePool(cores)
    try:
        gbs_all, secs_all = pool.gbs(rows, 2, min_seconds)
    finally:
        pool.close()
    one = OraclePool(1)
    try:
        gbs_one, secs_one = one.gbs(rows, 2, min_seconds)
    finally:
        one.close()
    return {"value": round(gbs_all, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"oracle matvec on the first {rows} rows of each decode shape, repeated for about "
                      f"{min_seconds:.0f} s in each of {cores} single-threaded processes at once "
                      f"(longest loop {secs_all:.1f} s), and in one process alone ({secs_one:.1f} s)",
            "single_thread": {"value": round(gbs_one, 4), "unit": "GB/s", "cores": 1}}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def run_ours(args, dist):
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_matmul_q4_gb300 as kq
    from quantized_weight_matmul_q4_gb300 import synthetic as syn

    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    pk, pk_kind = peaks()

    # ---- decode inputs: 8 independent weight copies per shape ----------------
    # Both shapes' x (and y) are views of one buffer, so the end-to-end leg
    # moves each step's inputs and results with one copy each way.
    wls = [syn.make_workload(name, copies=DECODE_COPIES) for name in ("decode_q4k_4096x11008", "decode_q4k_11008x4096")]
    x_all = torch.empty(sum(wl["K"] for wl in wls), dtype=torch.float32, device=dev)
    y_all = torch.empty(sum(wl["M"] for wl in wls), dtype=torch.float32, device=dev)
    sets = []
    xo = yo = 0
    for wl in wls:
        Ws = [torch.from_numpy(w).to(dev) for w in wl["W"]]
        x = x_all[xo:xo + wl["K"]]
        x.copy_(torch.from_numpy(wl["X"][0]))
        y = y_all[yo:yo + wl["M"]]
        xo += wl["K"]
        yo += wl["M"]
        sets.append((wl["M"], wl["K"], Ws, x, y, wl["X"][0]))
    w_bytes_step = sum(W.numel() for s in sets for W in s[2])
    alg_bytes_launch = [M * Q4K_ROW(K) + 4 * K + 4 * M for (M, K) in DECODE_SHAPES]
    calls_step = DECODE_COPIES * len(sets)
    launches_step = calls_step  # one kernel per call (x is quantised inside the matvec kernel)

    # The step's calls in order; each also asks L2 to prefetch the weights of
    # the call after it (kq_matvec_prefetch), as a decode loop that knows its
    # next layer's matrix would. Every weight byte is still read from HBM once
    # per step; results are identical to kq_matvec's.
    calls = [(M, K, Ws[c], x, y) for c in range(DECODE_COPIES) for (M, K, Ws, x, y, _) in sets]

    def step():
        for i, (M, K, W, x, y) in enumerate(calls):
            kq.kq_matvec_prefetch(kq.KQ_Q4_K, W, x, M, K, W_next=calls[(i + 1) % len(calls)][2], y=y)

    if args.only and args.only != "decode":
        res = run_sections(args, kq, syn, torch, dev, stream, pk, only=args.only)
        print(json.dumps({"only": args.only, **res}), flush=True)
        return None

    clocks = ClockSampler(dist.local)
    clocks.start()
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    # The decode sweep is launch-bound when driven from Python, so it is
    # captured once in a CUDA graph and replayed (the library's calls allocate
    # nothing and never synchronise, so they capture as they are).
    run = step
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
        run = graph.replay
        for _ in range(max(3, args.warmup)):
            run()
        torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    ms_local = e0.elapsed_time(e1)
    ms_total = dist.max(ms_local)
    ms_step = ms_total / args.steps
    code = kq.kq_get_device_error()
    if code:
        raise RuntimeError(f"device error {code} during the decode bench")

    # ---- end to end: pinned host x in, y out, through the public API ---------
    hx = torch.from_numpy(np.concatenate([s[5] for s in sets])).pin_memory()
    hy = torch.empty(y_all.numel(), dtype=torch.float32).pin_memory()

    def step_e2e():
        x_all.copy_(hx, non_blocking=True)
        step()
        hy.copy_(y_all, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        step_e2e()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        step_e2e()
    e1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    ms_e2e = dist.max(e0.elapsed_time(e1)) / args.steps

    # ---- sections: prefill GEMMs and MoE, each call timed with L2 flushed ----
    sections = {}
    if not args.no_sections and not args.only:
        sections = run_sections(args, kq, syn, torch, dev, stream, pk)
    clk = clocks.stop()

    avg_launch_s = ms_step / 1e3 / calls_step
    traffic, traffic_read, traffic_write = traffic_for("matvec_q4k_lanerow_kernel")
    achieved = statistics.mean(alg_bytes_launch) / avg_launch_s / 1e9
    value = dist.world * w_bytes_step / (ms_step / 1e3) / 1e9
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": dist.world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u8 weights (Q4_K), int8 activations (Q8_1), i32 dots, f32 accumulate",
        "data": "synthetic (seeded; Q4_K fields per the workload distributions, x ~ N(0,1))",
        "config": {
            "workload": "decode matvec N=1, Q4_K W[4096,11008] and W[11008,4096], Q8_1 quant fused",
            "step": "16 kq_matvec_prefetch launches (kq_matvec plus an L2 prefetch of the next call's weights): 8 rotated weight copies x 2 shapes"
                    + ("" if args.eager else ", replayed as one CUDA graph"),
            "l2": "inputs larger than L2 (8 weight copies per shape, 406 MB of weights)",
            "parallelism": f"replicas x{dist.world}",
            "sections": "prefill/MoE calls: each captured once as a CUDA graph and replayed with L2 flushed "
                        "before every replay (256 MB written, then another 256 MB read, so the flush's dirty "
                        "lines are written back before the timed region); ms_eager: the same call launched eagerly",
        },
        "roofline": {
            "kernel": "matvec_q4k_lanerow_kernel",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": pk["hbm_gbs"],
            "unit": "GB/s",
            "frac": round(achieved / pk["hbm_gbs"], 4),
            "peak_source": f"{pk_kind} (copy bandwidth)",
            "traffic": traffic,
            "traffic_read": traffic_read,
            "traffic_write": traffic_write,
            "traffic_note": "dram bytes per launch from profiles/ncu_traffic.json (steady state); the writes "
                            "are L2 write-backs of other kernels' lines, the kernel itself writes only y",
            "algorithmic_bytes_per_launch": statistics.mean(alg_bytes_launch),
            "duration": "mean time per kq_matvec_prefetch launch over the timed region (launches PDL-chained in a CUDA graph)",
        },
        "e2e": {
            "value": round(dist.world * w_bytes_step / (ms_e2e / 1e3) / 1e9, 2),
            "unit": "GB/s",
            "h2d_bytes_per_step": hx.numel() * hx.element_size(),
            "d2h_bytes_per_step": hy.numel() * hy.element_size(),
            "ms_per_step": round(ms_e2e, 5),
        },
        "gpu_launches": launches_step * args.steps,
        "clocks": clk,
        "sections": sections,
    }
    return out


def _timed_calls(fn, iters, warm, flush, torch, stream):
    """Device time (ms) of one fn() call, L2 flushed before each: the call is
    captured once as a CUDA graph and replayed (mean, min over iters), and the
    same is measured for eager calls (mean), which adds host launch latency."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()

    def timed(call):
        times = []
        for _ in range(iters):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(torch.cuda.current_stream())
            call()
            b.record(torch.cuda.current_stream())
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        return times

    eager = timed(fn)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize()
    graph = timed(g.replay)
    return statistics.mean(graph), min(graph), statistics.mean(eager)


# Decode sweeps of other weight formats: name -> (workloads, weight copies).
# Copies of each matrix make the swept weights larger than L2.
DECODE_SECTIONS = {
    "decode_tq4_1s_18944x3584_3584x18944": (("decode_tq4_1s_18944x3584", "decode_tq4_1s_3584x18944"), 4),
    "decode_q6k_4096x11008_11008x4096": (("decode_q6k_4096x11008", "decode_q6k_11008x4096"), 4),
    "decode_q5k_4096x11008_11008x4096": (("decode_q5k_4096x11008", "decode_q5k_11008x4096"), 4),
}


def _decode_sweep(kq, syn, torch, dev, stream, names, copies, reps, pk):
    """One decode call per weight copy and shape, captured as a CUDA graph and
    replayed `reps` times back to back (weights larger than L2, so no flush).
    Returns the section's numbers: algorithmic GB/s = (weights + x + y bytes)
    / device time."""
    sets = []
    for name in names:
        wl = syn.make_workload(name, copies=copies)
        Ws = [torch.from_numpy(w).to(dev) for w in wl["W"]]
        x = torch.from_numpy(wl["X"][0]).to(dev)
        y = torch.empty(wl["M"], dtype=torch.float32, device=dev)
        sets.append((wl["wtype"], wl["M"], wl["K"], Ws, x, y))

    # The step's calls in order; as in the headline decode step each call names
    # the next call's weights for an L2 prefetch (kq_matvec_prefetch), except
    # for TQ4_1S, whose ring refills were slower beside the prefetch.
    order = [(c, st) for c in range(copies) for st in sets]

    def step():
        for i, (c, (wt, M, K, Ws, x, y)) in enumerate(order):
            if wt == "tq4_1s":
                kq.kq_matvec(wt, Ws[c], x, M, K, y=y)
            else:
                c2, st2 = order[(i + 1) % len(order)]
                kq.kq_matvec_prefetch(wt, Ws[c], x, M, K, W_next=st2[3][c2], y=y)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    nbytes = sum(copies * (Ws[0].numel() + 4 * K + 4 * M) for (_, M, K, Ws, _, _) in sets)
    launches = copies * len(sets)
    gbs = nbytes / (ms / 1e3) / 1e9
    if kq.kq_get_device_error():
        raise RuntimeError("device error during a decode section")
    return {"ms_per_sweep": round(ms, 4), "launches_per_sweep": launches,
            "us_per_launch": round(1e3 * ms / launches, 2),
            "weight_mb_per_sweep": round(sum(copies * Ws[0].numel() for (_, _, _, Ws, _, _) in sets) / 1e6, 1),
            "gbs": round(gbs, 1), "frac_hbm_peak": round(gbs / pk["hbm_gbs"], 4)}


def _mma_rate(torch, pk):
    """Issue rate of tcgen05 kind::f16 MMAs (M = 128, K = 16, fp32 accumulator)
    on every SM, with A read from shared memory or from tensor memory, for
    N = 64, 128, 256 (the measurement aid libkqprobe.so)."""
    import ctypes
    from quantized_weight_matmul_q4_gb300.build import PROBE_LIB_PATH
    L = ctypes.CDLL(PROBE_LIB_PATH)
    L.kqprobe_mma.restype = ctypes.c_int
    L.kqprobe_mma.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                              ctypes.c_void_p]
    nsm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    cyc = torch.zeros(nsm, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream()
    iters = 8192
    out = {}
    for kind, where in ((0, "a_smem"), (2, "a_tmem")):
        for n in (64, 128, 256):
            for _ in range(2):
                rc = L.kqprobe_mma(kind, n, iters, ctypes.c_void_p(cyc.data_ptr()), nsm, ctypes.c_void_p(s.cuda_stream))
                if rc != 0:
                    raise RuntimeError(f"kqprobe_mma failed ({rc})")
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            L.kqprobe_mma(kind, n, iters, ctypes.c_void_p(cyc.data_ptr()), nsm, ctypes.c_void_p(s.cuda_stream))
            b.record(s)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            c = cyc.cpu().tolist()
            if min(c) <= 0:
                raise RuntimeError("kqprobe_mma: a wait gave up")
            tf = 2.0 * 128 * n * 16 * iters * nsm / (ms / 1e3) / 1e12
            out[f"{where}_n{n}"] = {"cycles_per_mma": round(statistics.median(c) / iters, 1),
                                    "tflops": round(tf, 1), "frac_bf16_peak": round(tf / pk["bf16_tflops"], 4)}
    return out


def section_ncu():
    """Per-section ncu figures (the capture each section's kernels were profiled
    at), from profiles/ncu_sections.json; `current` says whether the section's
    listed sources still hash to the captured ones."""
    path = os.path.join(ROOT, "profiles", "ncu_sections.json")
    if not os.path.exists(path):
        return {}
    with open(path) as f:
        d = json.load(f)
    return {k: dict(v, current=sources_digest(v["sources"]) == v["sources_sha256_16"]) for k, v in d["sections"].items()}


def run_sections(args, kq, syn, torch, dev, stream, pk, only=None):
    # L2 flush between timed calls: write 256 MB (> L2), then read another
    # 256 MB, so L2 holds only clean lines when the call starts (the write-back
    # of the dirty flush data is paid before the timed region, not inside it).
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(64 << 20, dtype=torch.int32, device=dev)

    def flush():
        flush_w.zero_()
        flush_r.sum()
    res = {}
    if only is None or only == "mma_rate":
        res["mma_rate_f16_m128"] = _mma_rate(torch, pk)
    if only == "mma_rate":
        return res
    for name, (names, copies) in DECODE_SECTIONS.items():
        if only is None or only == name:
            res[name] = _decode_sweep(kq, syn, torch, dev, stream, names, copies, 20, pk)
    if only in DECODE_SECTIONS:
        return res
    iters = max(3, args.section_iters)
    gemm_names = ["smalln_q4k_4096x11008_n4", "prefill_q4k_4096x4096_n64", "prefill_q4k_4096x4096_n512",
                  "prefill_q4k_14336x4096_n2048", "prefill_q6k_4096x14336_n2048",
                  "prefill_q5k_14336x4096_n2048"]
    moe_names = ["moe_q4k_128x768x2048_t1024_top8", "moe_q6k_128x768x2048_t1024_top8"]
    if only is not None:
        if only not in gemm_names + moe_names + list(DECODE_SECTIONS):
            raise SystemExit(f"unknown section {only!r}")
        gemm_names = [n for n in gemm_names if n == only]
        moe_names = [n for n in moe_names if n == only]
    for name in gemm_names:
        wl = syn.make_workload(name)
        M, K, N = wl["M"], wl["K"], wl["N"]
        W = torch.from_numpy(wl["W"][0]).to(dev)
        X = torch.from_numpy(wl["X"]).to(dev)
        Y = torch.empty((N, M), dtype=torch.float32, device=dev)
        ws = torch.empty(kq.kq_workspace_bytes(kq.KQ_OP_GEMM, wl["wtype"], M, K, N), dtype=torch.uint8, device=dev)
        fn = lambda: kq.kq_gemm(wl["wtype"], W, X, M, K, Y=Y, ws=ws)  # noqa: E731
        ms, ms_min, ms_eager = _timed_calls(fn, iters, 2, flush, torch, stream)
        flops = 2.0 * M * N * K
        wbytes = W.numel() + X.numel() * 4 + Y.numel() * 4
        tf = flops / (ms / 1e3) / 1e12
        res[name] = {"ms": round(ms, 4), "ms_min": round(ms_min, 4), "ms_eager": round(ms_eager, 4),
                     "tflops": round(tf, 1),
                     "frac_bf16_peak": round(tf / pk["bf16_tflops"], 4),
                     "alg_gbs": round(wbytes / (ms / 1e3) / 1e9, 1),
                     "frac_hbm_peak": round(wbytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)}
        del W, X, Y, ws
    for moe_name in moe_names:
        wl = syn.make_workload(moe_name)
        E, M, K, T, top_k = wl["n_experts"], wl["M"], wl["K"], wl["T"], wl["top_k"]
        W = torch.from_numpy(wl["W"][0]).to(dev)
        X = torch.from_numpy(wl["X"]).to(dev)
        ids = torch.from_numpy(wl["ids"]).to(dev)
        Y = torch.empty((T, top_k, M), dtype=torch.float32, device=dev)
        ws = torch.empty(kq.kq_workspace_bytes(kq.KQ_OP_MOE, wl["wtype"], M, K, T, E, top_k), dtype=torch.uint8,
                         device=dev)
        fn = lambda: kq.kq_moe_grouped_gemm(wl["wtype"], W, E, ids, X, M, K, Y=Y, ws=ws)  # noqa: E731
        ms, ms_min, ms_eager = _timed_calls(fn, iters, 2, flush, torch, stream)
        flops = 2.0 * M * K * T * top_k
        nbytes = W.numel() + X.numel() * 4 + Y.numel() * 4 + ids.numel() * 4
        tf = flops / (ms / 1e3) / 1e12
        res[moe_name] = {
            "ms": round(ms, 4), "ms_min": round(ms_min, 4), "ms_eager": round(ms_eager, 4), "tflops": round(tf, 1),
            "frac_bf16_peak": round(tf / pk["bf16_tflops"], 4),
            "alg_gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
            "frac_hbm_peak": round(nbytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)}
        del W, X, ids, Y, ws
    if kq.kq_get_device_error():
        raise RuntimeError("device error during the sections")
    for name, fig in section_ncu().items():
        if name in res:
            res[name]["ncu"] = fig
    return res


# ----------------------------------------------------------------------------
def run_reference(args):
    """The CPU oracle, as it stands, on bounded samples of the decode workload,
    on every host core (one single-threaded oracle process per core)."""
    cores = host_cores()
    rows = 256
    vals = []
    pool = OraclePool(cores)
    try:
        for _ in range(args.warmup):
            pool.gbs(rows, 1, 0.0)
        t_all = 0.0
        for _ in range(args.steps):
            gbs, s = pool.gbs(rows, 1, 0.0)
            vals.append(gbs)
            t_all += s
    finally:
        pool.close()
    v = statistics.mean(vals)
    sample = (f"oracle matvec on the first {rows} rows of each decode shape per step, "
              f"{cores} single-threaded processes at once")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(v, 4),
        "unit": "GB/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_all / max(1, args.steps) * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 oracle (fp32 Q8_1 quantisation)",
        "data": "synthetic (seeded)",
        "config": {"workload": "decode matvec N=1, Q4_K W[4096,11008] and W[11008,4096], Q8_1 quant fused",
                   "parallelism": "cpu oracle"},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return
    dist = Dist(args.gpus)
    out = run_ours(args, dist)
    if out is None:
        dist.close()
        return
    if dist.rank == 0 and not args.only:
        out["cpu_baseline"] = oracle_baseline(512, 8.0)
        print(json.dumps(out), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
