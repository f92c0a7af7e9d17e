#!/usr/bin/env python3
"""Benchmark of the persistent micro-op dispatcher on one node.

A step is one pass of the dispatch path over one seeded synthetic descriptor
stream: every descriptor is committed to the ring, executed by the resident
executor and completed. The default workload is the variable-shape
element-wise stream (100,000 descriptors over add/mul/ReLU/GELU in fp32 and
bf16, sizes log-uniform in 256..65,536, 30 % chained, inputs sliced from a
768 MiB N(0,1) pool, larger than L2).

Timed region (per rank): barrier, device synchronize, launch of the
persistent executor (its one launch), K steps, stop (the kernel ends),
device synchronize, barrier. CUDA events on the executor's stream bracket the
kernel; the roofline uses them. `e2e` repeats the run with the stream's input
buffers and its outputs in pinned host memory, copied in and out every step.

`--impl reference` times the CPU oracle (the only other arm: the method has
no reference implementation to install) on a bounded sample of the same
workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c2]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "micro-ops/sec and p50 submit-to-complete latency (μs); HBM GB/s vs roofline"
UNIT = "micro-ops/s"

WORKLOADS = {
    "c1": ("smallest stream: 1,000 fp32 add/mul/ReLU on 4,096 elements", dict()),
    "c2": ("variable-shape element-wise stream: 100,000 descriptors, add/mul/ReLU/GELU x fp32/bf16, "
           "n log-uniform 256..65,536, 30% chained", dict()),
    "c2l": ("large element-wise ops: 4,000 descriptors, n log-uniform 65,536..1,048,576", dict()),
    "c3": ("row-op stream: 50,000 softmax/LayerNorm/sum/max/min, bf16 [1..64, 1024|2048|4096]", dict()),
    "c4": ("decode attention: 2,000 steps of RoPE -> KV write -> SDPA, B 1..8, 32x128, L 128..4096", dict()),
    "c5": ("mixed pipeline: synthetic 32-layer decoder, 7 chained ops per layer, hidden 4096", dict()),
}


def make_stream(name: str, tokens: int):
    from workloads import streams as S
    if name == "c5":
        return S.stream_c5(n_tokens=tokens)
    return S.STREAMS[name]()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9 or not parts[0].isdigit() or int(parts[0]) != self.idx:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if sm:
            out = {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                   "samples": len(sm)}
        return out


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per descriptor of
# the executor kernel, from one ncu capture of a bounded run of each stream
# (``--profile-run --profile-desc N``: the stream's first N descriptors in the
# ring before the single launch), and the digest of the device sources the
# capture was taken on. A launch's traffic is that figure times the
# descriptors it processed, reported only while the sources are unchanged.
TRAFFIC_SOURCES = ("persistent_micro_dispatch_gb300/csrc/gpuos_device.cu",
                   "persistent_micro_dispatch_gb300/csrc/gpuos_internal.h")
TRAFFIC = {
    "c2": dict(bytes=249_464_832, descs=4096, sources="5daa6d1650495ac2"),
    "c2l": dict(bytes=998_394_368, descs=400, sources="5daa6d1650495ac2"),
    "c3": dict(bytes=400_407_296, descs=2048, sources="5daa6d1650495ac2"),
    "c4": dict(bytes=30_850_434_000, descs=600, sources="5daa6d1650495ac2"),
    "c5": dict(bytes=493_723_136, descs=224, sources="5daa6d1650495ac2"),
}


def sources_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def launch_traffic(workload: str, descs: int):
    """DRAM bytes of one executor launch that processed `descs` descriptors,
    scaled from the stream's capture; None once the kernel has changed."""
    t = TRAFFIC.get(workload)
    if t is None or sources_digest() != t["sources"]:
        return None
    return t["bytes"] / t["descs"] * descs


def measured_peak_gbs():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(p))["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# multi-rank helpers (replicas: one executor per GPU, no data-path collective)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(units: float, seconds: float, world: int):
    """Whole-job throughput: units summed over ranks / the slowest rank's time."""
    if world <= 1:
        return units, seconds
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([units, seconds], dtype=torch.float64, device=dev)
    u = t[:1].clone()
    s = t[1:].clone()
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    dist.all_reduce(s, op=dist.ReduceOp.MAX)
    return float(u.item()), float(s.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------
_ORACLE_SAMPLES: dict = {}


def oracle_rate(workload: str, budget_s: float):
    """Oracle ops/s on a bounded sample of the workload (single thread): the
    sample stream's descriptors in ticket order, cycled until `budget_s` of
    CPU work has been spent (a repeated pass does the same work)."""
    from oracle.interp import Machine
    from workloads import streams as S
    samples = {
        "c1": (lambda: S.stream_c1(), "the stream itself"),
        "c2": (lambda: S.stream_c2(n_desc=20000, pool_elems=1 << 22), "its generator, 2^22-element input pool"),
        "c2l": (lambda: S.stream_c2l(n_desc=200, pool_elems=1 << 23), "its generator, 2^23-element input pool"),
        "c3": (lambda: S.stream_c3(n_desc=5000, pool_elems=1 << 22), "its generator, 2^22-element input pool"),
        "c4": (lambda: S.stream_c4(n_steps=40), "its generator, 40 decode steps"),
        "c5": (lambda: S.stream_c5(n_tokens=1), "its generator, one token"),
    }
    if workload not in _ORACLE_SAMPLES:
        _ORACLE_SAMPLES[workload] = samples[workload][0]()
    s = _ORACLE_SAMPLES[workload]
    m = Machine(s)  # fresh host copies of the sample's buffers
    n = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 <= budget_s:
        m.apply(n % len(s.ops))
        n += 1
    dt = time.perf_counter() - t0
    sample = (f"{n} descriptors ({n / len(s.ops):.1f} passes) over a {len(s.ops)}-descriptor "
              f"{workload} sample ({samples[workload][1]})")
    return n / dt, n, dt, sample


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    budget = max(2.0, min(20.0, 120.0 / max(1, args.steps)))
    for _ in range(args.warmup):
        oracle_rate(args.workload, 1.0)
    rates = []
    t_all = 0.0
    for _ in range(args.steps):
        r, n, dt, sample = oracle_rate(args.workload, budget)
        rates.append(r)
        t_all += dt
    value = float(np.median(rates))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_all / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOADS[args.workload][0], "arm": "CPU oracle"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# co-running GEMM (hybrid execution: large GEMMs keep the normal launch path)
# ---------------------------------------------------------------------------
class Gemm:
    """An 8192^3 bf16 torch.matmul looped on its own stream, operands
    N(0, 0.02). Warmed up (its kernel loaded) before any executor is
    resident."""

    N = 8192

    def __init__(self, device_index: int):
        import torch
        dev = f"cuda:{device_index}"
        g = torch.Generator(device=dev).manual_seed(5)
        self.a = (torch.randn(self.N, self.N, device=dev, generator=g) * 0.02).to(torch.bfloat16)
        self.b = (torch.randn(self.N, self.N, device=dev, generator=g) * 0.02).to(torch.bfloat16)
        self.c = torch.empty_like(self.a)
        self.stream = torch.cuda.Stream()
        with torch.cuda.stream(self.stream):
            torch.matmul(self.a, self.b, out=self.c)
        torch.cuda.synchronize()
        self.events = []
        self.alone_tflops = None

    def flops(self, n):
        return 2.0 * self.N ** 3 * n

    def measure_alone(self, n):
        import torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        with torch.cuda.stream(self.stream):
            for _ in range(n):
                torch.matmul(self.a, self.b, out=self.c)
        e1.record(self.stream)
        e1.synchronize()
        return self.flops(n) / (e0.elapsed_time(e1) / 1e3) / 1e12

    def enqueue(self, n):
        import torch
        first = torch.cuda.Event(enable_timing=True)
        first.record(self.stream)
        self.events = [first]
        with torch.cuda.stream(self.stream):
            for _ in range(n):
                torch.matmul(self.a, self.b, out=self.c)
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(self.stream)
                self.events.append(ev)

    def progress(self):
        return sum(1 for ev in self.events[1:] if ev.query())

    def report(self, done_while_resident, kern_ms):
        """TFLOP/s of the GEMMs that completed while the executor was
        resident (a bounded wait lets the rest finish afterwards)."""
        t0 = time.perf_counter()
        while not self.events[-1].query() and time.perf_counter() - t0 < 120:
            time.sleep(0.01)
        out = {"alone_tflops": self.alone_tflops, "gemms_done_while_executor_resident": done_while_resident,
               "gemms_enqueued": len(self.events) - 1, "executor_kernel_ms": kern_ms}
        if done_while_resident:
            ms = self.events[0].elapsed_time(self.events[done_while_resident])
            out["corun_tflops"] = self.flops(done_while_resident) / (ms / 1e3) / 1e12
            out["gemm_slowdown"] = out["alone_tflops"] / out["corun_tflops"]
        return out


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def pct(x, q):
    return float(np.percentile(x, q)) if len(x) else None


def producers_sweep(G, cfg_kw) -> int:
    """Aggregate submission throughput of T concurrent host threads, each
    committing NOP descriptors in batches of 16 through one ring (the page's
    ring-contention question). The single-thread line without the
    multi-producer path (plain SPSC ring) is the reference."""
    import threading
    per_thread = 20_000
    batch = 16
    nop = G.make_descs(batch)
    rows = []
    for T, mp in [(1, 0), (1, 1), (2, 1), (4, 1), (8, 1), (16, 1), (32, 1), (64, 1)]:
        ex = G.Executor(**cfg_kw, multi_producer=mp)
        try:
            go = threading.Barrier(T + 1)

            def work():
                go.wait()
                for _ in range(per_thread // batch):
                    ex.submit_batch(nop)

            th = [threading.Thread(target=work) for _ in range(T)]
            for t in th:
                t.start()
            go.wait()
            t0 = time.perf_counter()
            for t in th:
                t.join()
            t_sub = time.perf_counter() - t0
            ex.sync(timeout_ms=60_000)
            t_all = time.perf_counter() - t0
            st = ex.stats()
        finally:
            ex.shutdown()
        n = T * (per_thread // batch) * batch
        assert st["completed"] >= n, st
        rows.append({"threads": T, "multi_producer": mp, "descriptors": n,
                     "submit_per_s": n / t_sub, "complete_per_s": n / t_all})
    print(json.dumps({"metric": "host submission throughput vs producer threads (NOP batches of 16)",
                      "unit": "descriptors/s", "rows": rows}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c2", choices=sorted(WORKLOADS))
    ap.add_argument("--tokens", type=int, default=20, help="tokens per step of the c5 workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-eager", action="store_true")
    ap.add_argument("--profile-run", action="store_true",
                    help="one bounded executor run (ring filled before launch) for profilers; no JSON")
    ap.add_argument("--profile-desc", type=int, default=0,
                    help="profile run: descriptors (0 = the workload's own, capped at the ring size)")
    ap.add_argument("--pool-log2", type=int, default=0, help="profile run: log2 of the input pool elements")
    ap.add_argument("--warps", type=int, default=0, help="executor warps per block (0 = default)")
    ap.add_argument("--stage-bytes", type=int, default=16384, help="shared-memory staging per warp (0 = none)")
    ap.add_argument("--blocks", type=int, default=0, help="executor blocks (0 = one per SM)")
    ap.add_argument("--spin-polls", type=int, default=0, help="idle polls before backoff sleeps (0 = default)")
    ap.add_argument("--backoff-max-ns", type=int, default=0, help="longest idle sleep (0 = default)")
    ap.add_argument("--producers-sweep", action="store_true",
                    help="host-thread contention curve: T threads submitting NOP batches (multi_producer=1); "
                         "prints its own JSON line")
    ap.add_argument("--ring-device", action="store_true",
                    help="ring in device memory (managed, host-accessible) instead of pinned host memory")
    ap.add_argument("--graph", action="store_true",
                    help="also time the eager launches captured into a CUDA graph (replay, and re-capture per step)")
    ap.add_argument("--corun-gemm", action="store_true",
                    help="loop a normally launched 8192^3 bf16 GEMM on a second stream during the timed region")
    args = ap.parse_args()
    os.environ.setdefault("GPUOS_DEBUG", "1")
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    torch.cuda.set_device(local)
    from persistent_micro_dispatch_gb300 import build as pkg_build
    pkg_build.build()
    from persistent_micro_dispatch_gb300 import gpuos as G
    from workloads import streams as S
    from workloads.device import DeviceStream, warm_torch

    cfg_kw = dict(device=local, idle_exit_ms=20000, stage_bytes=args.stage_bytes, blocks=args.blocks)
    if args.warps:
        cfg_kw["warps_per_block"] = args.warps
    if args.spin_polls:
        cfg_kw["spin_polls"] = args.spin_polls
    if args.backoff_max_ns:
        cfg_kw["backoff_max_ns"] = args.backoff_max_ns
    if args.ring_device:
        cfg_kw["ring_in_device_mem"] = 1
    if args.profile_run and args.profile_desc and args.workload in ("c2", "c2l", "c3"):
        kw = dict(n_desc=args.profile_desc)
        if args.pool_log2:
            kw["pool_elems"] = 1 << args.pool_log2
        s = S.STREAMS[args.workload](**kw)
    elif args.profile_run and args.profile_desc and args.workload == "c4":
        s = S.stream_c4(n_steps=max(1, args.profile_desc // 3))
    elif args.profile_run and args.profile_desc and args.workload == "c5":
        s = S.stream_c5(n_tokens=max(1, args.profile_desc // 224))
    else:
        s = make_stream(args.workload, args.tokens)
    n_ops = len(s.ops)
    step_bytes = S.stream_bytes(s)
    ds = DeviceStream(s, device=f"cuda:{local}")
    descs = ds.descs()
    warm_torch(f"cuda:{local}")
    torch.cuda.synchronize()

    if args.producers_sweep:
        return producers_sweep(G, cfg_kw)
    if args.profile_run:
        # bounded run with the ring filled before the single launch: the
        # kernel ends on its own after len(descs) completions (replayable)
        nprof = min(n_ops, 4096)
        ex = G.Executor(**cfg_kw, deferred_start=1, exit_after=nprof)
        ex.submit_batch(descs[:nprof])
        ex.start()
        rc = ex.sync(timeout_ms=120_000, raise_on_error=False)
        ex.shutdown()
        print(f"profile run: {nprof} descriptors, sync rc={rc}", flush=True)
        return 0

    # ---- warm-up executor: warm-up steps, clock calibration, isolated latency
    ex = G.Executor(**cfg_kw)
    for _ in range(args.warmup):
        ex.submit_batch(descs)
        ex.sync(timeout_ms=600_000)
    off_lo, off_hi, min_rtt, rtts = ex.calibrate(300)
    off = (off_lo + off_hi) // 2
    rng = np.random.default_rng(0)
    iso_idx = rng.choice(n_ops, size=min(300, n_ops), replace=False)
    iso_rtt = []
    base = ex.stats()["submitted"]
    iso_hist = ex.set_history(base, len(iso_idx))
    for j in iso_idx:
        d1 = descs[j:j + 1].copy()
        d1["dep"] = 0  # isolated: no dependency on ops of another pass
        t0 = G.host_now_ns()
        t = ex.submit(d1)
        ex.sync(t)
        iso_rtt.append(G.host_now_ns() - t0)
    ex.sync()
    rc_sd = ex.shutdown()
    if rc_sd != G.OK:
        print(f"warm-up executor shutdown: {G.strerror(rc_sd)}", file=sys.stderr)

    gemm = None
    if args.corun_gemm:
        gemm = Gemm(local)
        gemm.alone_tflops = gemm.measure_alone(20)

    # ---- timed region: one launch of the persistent executor, K steps
    ex = G.Executor(**cfg_kw, deferred_start=1)
    hist = ex.set_history(0, args.steps * n_ops)
    xs = torch.cuda.ExternalStream(ex.stream)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    torch.cuda.synchronize()
    barrier(world)
    clocks.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    ev0.record(xs)
    ex.start()
    ev1.record(xs)  # completes when the executor kernel ends
    if gemm is not None:
        gemm.enqueue(40)
    submit_ns = 0
    for step in range(args.steps):
        a = time.perf_counter_ns()
        ex.submit_batch(descs)
        submit_ns += time.perf_counter_ns() - a
        ex.sync(timeout_ms=600_000)
    gemm_progress = None
    if gemm is not None:
        gemm_progress = gemm.progress()  # GEMMs finished while the executor was resident
    ex.stop()
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(world)
    clk = clocks.stop()
    wall = t1 - t0
    kern_ms = ev0.elapsed_time(ev1)
    st = ex.stats()
    tprof = ex.tile_profile()
    ex.shutdown()
    units, secs = aggregate(n_ops * args.steps, kern_ms / 1e3, world)
    value = units / secs

    # latencies of the timed tickets (device clock corrected by the offset)
    h = hist[hist["ticket"] != np.iinfo(np.uint64).max]
    commit = h["t_commit_host_ns"].astype(np.int64) + off
    lat_us = (h["t_done_dev_ns"].astype(np.int64) - commit) / 1e3
    disp_us = (h["t_dispatch_dev_ns"].astype(np.int64) - commit) / 1e3
    ih = iso_hist
    iso_disp_us = (ih["t_dispatch_dev_ns"].astype(np.int64) - ih["t_commit_host_ns"].astype(np.int64) - off) / 1e3
    iso_dev_us = (ih["t_done_dev_ns"].astype(np.int64) - ih["t_dispatch_dev_ns"].astype(np.int64)) / 1e3
    busy_ns = int(h["t_done_dev_ns"].max()) - int(h["t_dispatch_dev_ns"].min()) if len(h) else 0

    # per op kind: device time from tile-0 start to completion, and bandwidth
    kinds = {}
    if len(h):
        opn = np.array([s.ops[int(t) % n_ops].op for t in h["ticket"]])
        dur = (h["t_done_dev_ns"].astype(np.int64) - h["t_start_dev_ns"].astype(np.int64)) / 1e3
        # dispatch gap of a dependent op: its last dependency done -> its tile 0 started
        tix = h["ticket"].astype(np.int64)
        jj = tix % n_ops
        t_done = h["t_done_dev_ns"].astype(np.int64)
        last_dep = np.full(len(h), -1, dtype=np.int64)
        for k in range(2):
            offk = np.array([(j - o.deps[k]) if len(o.deps) > k else 0 for j, o in enumerate(s.ops)],
                            dtype=np.int64)[jj]
            dep_t = tix - offk
            idx = np.clip(np.searchsorted(tix, dep_t), 0, len(tix) - 1)
            ok = (offk > 0) & (tix[idx] == dep_t)
            last_dep = np.where(ok, np.maximum(last_dep, t_done[idx]), last_dep)
        gap = np.where(last_dep >= 0, (h["t_start_dev_ns"].astype(np.int64) - last_dep) / 1e3, np.nan)
        per_op_bytes = np.array([S.sdpa_bytes(o, s.buffers[o.aux0.buf].data[o.aux0.off:o.aux0.off + o.dims[0]])
                                 if o.op == "sdpa" else S.op_bytes(o) for o in s.ops], dtype=np.float64)
        byts = per_op_bytes[(h["ticket"] % n_ops).astype(np.int64)]
        for k in sorted(set(opn.tolist())):
            m = opn == k
            kinds[k] = {"n": int(m.sum()), "dur_us_p50": float(np.median(dur[m])),
                        "gbs_p50": float(np.median(byts[m] / np.maximum(dur[m], 1e-3) / 1e3))}
            gk = gap[m & ~np.isnan(gap)]
            if gk.size:
                kinds[k]["dep_gap_us_p50"] = float(np.median(gk))
            if k in tprof:  # mean device time per tile: in the op, finishing, waiting for inputs
                tp = tprof[k]
                kinds[k].update(tiles_per_op=tp["tiles"] / max(1, int(m.sum())), tile_body_us=tp["body_us"],
                                tile_finish_us=tp["finish_us"], tile_dep_us=tp["dep_us"])
    peak, peak_kind = measured_peak_gbs()
    achieved = step_bytes * args.steps / (kern_ms / 1e3) / 1e9
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": kern_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload][0], "descriptors_per_step": n_ops,
                   "algorithmic_bytes_per_step": step_bytes, "l2": "inputs larger than L2 (768 MiB pool)"
                   if args.workload in ("c2", "c2l") else "inputs and caches larger than L2",
                   "parallelism": f"replicas x{world}", "ring_entries": int(ex.config.ring_entries),
                   "warps_per_block": int(st["warps_per_block"]), "blocks": int(st["blocks"])},
        "gpu_launches": 1,
        "latency_us": {
            "submit_to_complete_p50": pct(lat_us, 50), "submit_to_complete_p99": pct(lat_us, 99),
            "submit_to_dispatch_p50": pct(disp_us, 50),
            "isolated_roundtrip_p50": pct(np.array(iso_rtt) / 1e3, 50),
            "isolated_roundtrip_p99": pct(np.array(iso_rtt) / 1e3, 99),
            "isolated_submit_to_dispatch_p50": pct(iso_disp_us, 50),
            "isolated_dispatch_to_done_p50": pct(iso_dev_us, 50),
            "clock_offset_uncertainty": (off_hi - off_lo) / 2e3,
            "nop_roundtrip_min": min_rtt / 1e3, "nop_roundtrip_p50": float(np.median(rtts)) / 1e3,
            "host_submit_ns_per_desc": submit_ns / (args.steps * n_ops),
        },
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": launch_traffic(args.workload, n_ops * args.steps),
                     "peak_kind": peak_kind,
                     "kernel": "gpuos_executor_kernel", "kernel_ms": kern_ms,
                     "device_busy_ms": busy_ns / 1e6},
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
        "op_kinds": kinds,
        "executor": {k: st[k] for k in ("tiles", "idle_polls", "sleeps", "dep_waits", "regs_per_thread",
                                        "static_smem_bytes", "seq_body_ns", "seq_mirror_ns", "seq_publish_ns", "seq_batches", "host_wait_ns")},
        "wall_s": wall,
    }

    if gemm is not None:
        result["corun_gemm"] = gemm.report(gemm_progress, kern_ms)

    # ---- eager baseline: same op bodies, one cudaLaunchKernel per descriptor
    if not args.no_eager:
        es = torch.cuda.Stream()
        for _ in range(max(1, args.warmup)):
            G.eager_run(descs, es.cuda_stream, args.stage_bytes)
        es.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(es)
        for _ in range(args.steps):
            G.eager_run(descs, es.cuda_stream, args.stage_bytes)
        e1.record(es)
        e1.synchronize()
        eg_ms = e0.elapsed_time(e1)
        # isolated latency, measured like the executor's isolated round trip:
        # the same sampled ops, one launch each, then a wait for it (host clock)
        eg_rtt = []
        for j in iso_idx:
            d1 = descs[j:j + 1].copy()
            d1["dep"] = 0
            t0 = G.host_now_ns()
            G.eager_run(d1, es.cuda_stream, args.stage_bytes)
            es.synchronize()
            eg_rtt.append(G.host_now_ns() - t0)
        result["eager"] = {"value": n_ops * args.steps / (eg_ms / 1e3), "unit": UNIT,
                           "ms_per_step": eg_ms / args.steps, "launches_per_step": n_ops,
                           "isolated_roundtrip_p50": pct(np.array(eg_rtt) / 1e3, 50),
                           "isolated_roundtrip_p99": pct(np.array(eg_rtt) / 1e3, 99)}

    # ---- CUDA Graphs baseline: the eager launches of one step captured once
    # and replayed (stable shapes), and captured + instantiated anew every
    # step (what shapes that change every step cost)
    if args.graph:
        gs = torch.cuda.Stream()
        G.eager_run(descs, gs.cuda_stream, args.stage_bytes)  # kernel attributes set outside capture
        gs.synchronize()
        c0 = time.perf_counter()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            G.eager_run(descs, gs.cuda_stream, args.stage_bytes)
        cap_s = time.perf_counter() - c0
        graph.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(gs):
            e0.record()
            for _ in range(args.steps):
                graph.replay()
            e1.record()
        e1.synchronize()
        rep_ms = e0.elapsed_time(e1) / args.steps
        result["cuda_graph"] = {"replay_value": n_ops / (rep_ms / 1e3), "unit": UNIT, "replay_ms_per_step": rep_ms,
                                "capture_instantiate_ms": cap_s * 1e3,
                                "recapture_value": n_ops / (rep_ms / 1e3 + cap_s)}
        del graph
        torch.cuda.synchronize()

    # ---- end to end: host buffers, copies inside the timed region
    if not args.no_e2e:
        in_idx = [i for i, b in enumerate(s.buffers) if b.data is not None]
        out_idx = sorted({o_ref.buf for o in s.ops for o_ref in (o.out, o.aux1 if o.op == "kv_write" else None)
                          if o_ref is not None} - set(in_idx))
        host_in = [torch.from_numpy(np.ascontiguousarray(s.buffers[i].data).view(np.uint8)).pin_memory() for i in in_idx]
        host_out = [torch.empty(ds.bufs[i].numel(), dtype=torch.uint8).pin_memory() for i in out_idx]
        h2d = sum(t.numel() for t in host_in)
        d2h = sum(t.numel() for t in host_out)
        cs = torch.cuda.Stream()
        # device-wide synchronisation only while no executor is resident: a
        # resident persistent kernel never lets it return
        torch.cuda.synchronize()
        ex = G.Executor(**cfg_kw)
        barrier(world)
        a = time.perf_counter()
        for _ in range(args.steps):
            with torch.cuda.stream(cs):
                for i, t in zip(in_idx, host_in):
                    ds.bufs[i].copy_(t, non_blocking=True)
            cs.synchronize()
            ex.submit_batch(descs)
            ex.sync(timeout_ms=600_000)
            with torch.cuda.stream(cs):
                for i, t in zip(out_idx, host_out):
                    t.copy_(ds.bufs[i], non_blocking=True)
            cs.synchronize()
        b = time.perf_counter()
        ex.shutdown()
        torch.cuda.synchronize()
        eu, esec = aggregate(n_ops * args.steps, b - a, world)
        result["e2e"] = {"value": eu / esec, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": 1e3 * (b - a) / args.steps}

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    if not args.no_cpu and rank == 0 and world == 1:
        r, n, dt, sample = oracle_rate(args.workload, 12.0)
        result["cpu_baseline"] = {"value": r, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                                  "seconds": dt, "host_cores": os.cpu_count()}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
