#!/usr/bin/env python3
"""Benchmark of the persistent micro-op dispatcher on one node.

A step is one pass of the dispatch path over one seeded synthetic descriptor
stream: every descriptor is committed to the ring, executed by the resident
executor and completed. The headline workload is the variable-shape
element-wise stream (100,000 descriptors over add/mul/ReLU/GELU in fp32 and
bf16, sizes log-uniform in 256..65,536, 30 % chained, inputs sliced from a
768 MiB N(0,1) pool, larger than L2).

Timed region (per rank): barrier, device synchronize, launch of the
persistent executor (its one launch), K steps, stop (the kernel ends),
device synchronize, barrier. CUDA events on the executor's stream bracket the
kernel; the roofline uses them. `e2e` repeats the run with the stream's input
buffers and its outputs in pinned host memory, copied in and out every step.

The same JSON line carries, under `streams`, every other workload measured
the same way (fewer steps): the smallest stream, large element-wise ops (the
>= 64 K-element roofline gate), row ops, decode attention and the mixed
pipeline at 500 tokens, each beside its eager baseline; under `corun_gemm`,
an 8192^3 bf16 GEMM looping on a second stream while the executor runs the
mixed pipeline on 8..152 SMs; under `cuda_graph`, the eager launches of one
step captured into a CUDA graph and replayed.

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
    "c1": "smallest stream: 1,000 fp32 add/mul/ReLU on 4,096 elements",
    "c2": ("variable-shape element-wise stream: 100,000 descriptors, add/mul/ReLU/GELU x fp32/bf16, "
           "n log-uniform 256..65,536, 30% chained"),
    "c2l": "large element-wise ops: 4,000 descriptors, n log-uniform 65,536..1,048,576",
    "c3": "row-op stream: 50,000 softmax/LayerNorm/sum/max/min, bf16 [1..64, 1024|2048|4096]",
    "c4": "decode attention: 2,000 steps of RoPE -> KV write -> SDPA, B 1..8, 32x128, L 128..4096",
    "c5": "mixed pipeline: synthetic 32-layer decoder, 7 chained ops per layer, hidden 4096, 500 tokens",
}
L2_NOTE = {
    "c1": "L2-resident (43 MB of operands, as the stream is defined)",
    "c2": "inputs larger than L2 (768 MiB pool)",
    "c2l": "inputs larger than L2 (768 MiB pool)",
    "c3": "inputs larger than L2 (256 MiB pool)",
    "c4": "inputs and caches larger than L2 (512 MiB of caches)",
    "c5": "inputs and caches larger than L2 (2 GiB of caches)",
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
    "c2": dict(bytes=251_875_840, descs=4096, sources="59f0042f3e66b557"),
    "c2l": dict(bytes=1_089_941_760, descs=400, sources="59f0042f3e66b557"),
    "c3": dict(bytes=417_755_392, descs=2048, sources="59f0042f3e66b557"),
    "c4": dict(bytes=31_051_235_584, descs=600, sources="59f0042f3e66b557"),
    "c5": dict(bytes=492_626_176, descs=224, sources="59f0042f3e66b557"),
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


def descriptors_per_step(workload: str, tokens: int) -> int:
    return {"c1": 1000, "c2": 100_000, "c2l": 4000, "c3": 50_000, "c4": 6000}.get(workload, tokens * 32 * 7)


def run_reference(args, world, rank):
    """The CPU oracle arm. Each step is a bounded sample of the workload
    (about `budget` seconds of CPU work); `value` is its median ops/s.
    `ms_per_step` is what one full step of the workload (all its
    descriptors) takes at that rate; the sampling budget is reported apart."""
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
    n_step = descriptors_per_step(args.workload, args.tokens)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * n_step / value,
        "sample_budget_ms_per_step": 1e3 * t_all / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOADS[args.workload], "arm": "CPU oracle",
                                        "descriptors_per_step": n_step},
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

    def start_loop(self, max_queued: int = 40):
        """Keep GEMMs queued on the GEMM stream from a host thread (at most
        max_queued not yet finished) until stop_loop()."""
        import threading
        import torch
        self.events = []
        self._stop = threading.Event()

        def loop():
            with torch.cuda.stream(self.stream):
                while not self._stop.is_set():
                    done = sum(1 for ev in self.events[-max_queued:] if ev.query()) if self.events else 0
                    pending = min(len(self.events), max_queued) - done
                    if pending >= max_queued // 2:
                        time.sleep(0.0005)
                        continue
                    for _ in range(max_queued // 2):
                        torch.matmul(self.a, self.b, out=self.c)
                        ev = torch.cuda.Event(enable_timing=True)
                        ev.record(self.stream)
                        self.events.append(ev)

        first = torch.cuda.Event(enable_timing=True)
        first.record(self.stream)
        self.first = first
        self._th = threading.Thread(target=loop, daemon=True)
        self._th.start()

    def stop_loop(self):
        self._stop.set()
        self._th.join()

    def report(self, ev_end):
        """TFLOP/s of the GEMMs that finished before the executor ended
        (`ev_end`, an event on the executor's stream), timed from the first
        GEMM's start event to the last such GEMM's event."""
        t0 = time.perf_counter()
        while self.events and not self.events[-1].query() and time.perf_counter() - t0 < 120:
            time.sleep(0.01)
        end_ms = self.first.elapsed_time(ev_end)
        times = [self.first.elapsed_time(ev) for ev in self.events]
        k = sum(1 for x in times if x <= end_ms)
        out = {"gemms_done_while_executor_resident": k, "gemms_enqueued": len(self.events),
               "gemm_tflops": self.flops(k) / (times[k - 1] / 1e3) / 1e12 if k else 0.0}
        return out


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def pct(x, q):
    return float(np.percentile(x, q)) if len(x) else None


def producers_sweep(local: int) -> int:
    """Aggregate submission throughput of T concurrent host threads, each
    committing NOP descriptors in batches of 16 through one ring (the page's
    ring-contention question). The threads are native (the library's
    measurement program, C ABI only): Python threads would serialise on the
    interpreter lock around every call and measure that instead. The
    single-thread line on the single-producer ring is the reference."""
    from persistent_micro_dispatch_gb300 import build as pkg_build
    exe = pkg_build.PRODUCERS
    r = subprocess.run([exe, "64", "20000", "16", str(local)], stdout=subprocess.PIPE, text=True, timeout=600)
    line = r.stdout.strip().splitlines()[-1] if r.stdout.strip() else "{}"
    print(line, flush=True)
    return r.returncode


def isolated_latency(G, ex, descs, n_ops, n=300):
    """Calibrate the clocks, then time n isolated descriptors (one in the
    ring at a time). Returns the offset bounds, NOP round trips and the
    per-descriptor records / host round trips."""
    off_lo, off_hi, min_rtt, rtts = ex.calibrate(1000)
    rng = np.random.default_rng(0)
    iso_idx = rng.choice(n_ops, size=min(n, n_ops), replace=False)
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
    return dict(off_lo=off_lo, off_hi=off_hi, min_rtt=min_rtt, rtts=rtts, iso_idx=iso_idx,
                iso_rtt=np.array(iso_rtt), iso_hist=iso_hist.copy())


def timed_executor(G, descs, cfg_kw, steps, gemm=None, history=True):
    """One launch of the executor around `steps` passes over `descs`:
    returns the kernel time (CUDA events on its own stream), the completion
    records of the last step, stats, tile profile and host submit time."""
    import torch
    n_ops = len(descs)
    ex = G.Executor(**cfg_kw, deferred_start=1)
    # completion records of the last timed step (its latency statistics and
    # per-op-kind table): keeping all K steps' records is host work of its
    # own, 56 bytes written per descriptor into a large array
    hist = ex.set_history((steps - 1) * n_ops, n_ops) if history else None
    xs = torch.cuda.ExternalStream(ex.stream)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(xs)
    ex.start()
    ev1.record(xs)  # completes when the executor kernel ends
    if gemm is not None:
        gemm.start_loop()
    submit_ns = 0
    for _ in range(steps):
        a = time.perf_counter_ns()
        ex.submit_batch(descs)
        submit_ns += time.perf_counter_ns() - a
        ex.sync(timeout_ms=600_000)
    ex.stop()
    if gemm is not None:
        gemm.stop_loop()
    ev1.synchronize()
    kern_ms = ev0.elapsed_time(ev1)
    gemm_report = gemm.report(ev1) if gemm is not None else None
    st = ex.stats()
    tprof = ex.tile_profile()
    ex.shutdown()
    return dict(kern_ms=kern_ms, hist=hist, stats=st, tprof=tprof, submit_ns=submit_ns,
                gemm=gemm_report, config=ex.config)


def op_kind_table(s, h, n_ops, tprof, passes):
    """Per op kind: p50 duration (tile 0 start -> completion), bandwidth,
    the dependency gap (from the records in `h`, one pass over the stream)
    and the per-tile device times (the tile profile covers all `passes`
    passes of the launch)."""
    from workloads import streams as S
    kinds = {}
    if not len(h):
        return kinds
    opn = np.array([s.ops[int(t) % n_ops].op for t in h["ticket"]])
    dur = (h["t_done_dev_ns"].astype(np.int64) - h["t_start_dev_ns"].astype(np.int64)) / 1e3
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
    byts = per_op_bytes[jj]
    for k in sorted(set(opn.tolist())):
        m = opn == k
        kinds[k] = {"n": int(m.sum()), "dur_us_p50": float(np.median(dur[m])),
                    "gbs_p50": float(np.median(byts[m] / np.maximum(dur[m], 1e-3) / 1e3))}
        gk = gap[m & ~np.isnan(gap)]
        if gk.size:
            kinds[k]["dep_gap_us_p50"] = float(np.median(gk))
        if k in tprof:
            tp = tprof[k]
            kinds[k].update(tiles_per_op=tp["tiles"] / max(1, passes * int(m.sum())), tile_body_us=tp["body_us"],
                            tile_finish_us=tp["finish_us"], tile_dep_us=tp["dep_us"])
    return kinds


def eager_rate(G, descs, steps, warmup, stage_bytes):
    import torch
    es = torch.cuda.Stream()
    for _ in range(max(1, warmup)):
        G.eager_run(descs, es.cuda_stream, stage_bytes)
    es.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(es)
    for _ in range(steps):
        G.eager_run(descs, es.cuda_stream, stage_bytes)
    e1.record(es)
    e1.synchronize()
    ms = e0.elapsed_time(e1)
    return len(descs) * steps / (ms / 1e3), ms / steps, es


def graph_rate(G, descs, steps, stage_bytes):
    """The eager launches of one step captured once into a CUDA graph and
    replayed (stable shapes), and the cost of capturing and instantiating
    it anew every step (shapes that change every step)."""
    import torch
    gs = torch.cuda.Stream()
    G.eager_run(descs, gs.cuda_stream, stage_bytes)  # kernel attributes set outside capture
    gs.synchronize()
    c0 = time.perf_counter()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        G.eager_run(descs, gs.cuda_stream, stage_bytes)
    graph.replay()
    torch.cuda.synchronize()
    cap_s = time.perf_counter() - c0
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(gs):
        e0.record()
        for _ in range(steps):
            graph.replay()
        e1.record()
    e1.synchronize()
    rep_ms = e0.elapsed_time(e1) / steps
    del graph
    torch.cuda.synchronize()
    n = len(descs)
    return {"replay_value": n / (rep_ms / 1e3), "unit": UNIT, "replay_ms_per_step": rep_ms,
            "capture_instantiate_ms": cap_s * 1e3, "recapture_value": n / (rep_ms / 1e3 + cap_s)}


def latency_block(h, off, lo):
    """Submit->complete and submit->dispatch of timed tickets (device clock
    corrected by the offset midpoint; the dispatch upper bound uses the
    offset's lower end, which no true offset is below)."""
    commit = h["t_commit_host_ns"].astype(np.int64)
    lat_us = (h["t_done_dev_ns"].astype(np.int64) - commit - off) / 1e3
    disp_us = (h["t_dispatch_dev_ns"].astype(np.int64) - commit - off) / 1e3
    disp_up = (h["t_dispatch_dev_ns"].astype(np.int64) - commit - lo) / 1e3
    return {"submit_to_complete_p50": pct(lat_us, 50), "submit_to_complete_p99": pct(lat_us, 99),
            "submit_to_dispatch_p50": pct(disp_us, 50), "submit_to_dispatch_p50_upper": pct(disp_up, 50)}


def stream_phase(G, name, args, cfg_kw, local, peak, gemm=None):
    """Measure one more workload: warm-up executor (calibration), one timed
    executor launch over `stream_steps` passes, the eager baseline and, for
    the mixed pipeline, the GEMM co-run curve."""
    import torch
    from workloads import streams as S
    from workloads.device import DeviceStream
    t_gen = time.perf_counter()
    s = make_stream(name, args.tokens if name == "c5" else 0)
    n_ops = len(s.ops)
    step_bytes = S.stream_bytes(s)
    ds = DeviceStream(s, device=f"cuda:{local}")
    descs = ds.descs()
    torch.cuda.synchronize()
    gen_s = time.perf_counter() - t_gen
    K = args.stream_steps
    if name == "c1":
        # a step of the smallest stream lasts tens of microseconds: over a
        # few steps the launch and the stop of the single executor launch
        # (included in the timed region) would outweigh the steps themselves
        K = max(K, args.c1_steps)
    if name == "c1" and not args.ring_entries:
        cfg_kw = dict(cfg_kw, ring_entries=4096)  # as the smallest stream is defined
    ex = G.Executor(**cfg_kw)
    for _ in range(args.stream_warmup):
        ex.submit_batch(descs)
        ex.sync(timeout_ms=600_000)
    off_lo, off_hi, _, _ = ex.calibrate(300)
    ex.shutdown()
    off = (off_lo + off_hi) // 2
    r = timed_executor(G, descs, cfg_kw, K)
    kern_ms = r["kern_ms"]
    value = n_ops * K / (kern_ms / 1e3)
    achieved = step_bytes * K / (kern_ms / 1e3) / 1e9
    h = r["hist"][r["hist"]["ticket"] != np.iinfo(np.uint64).max]
    out = {"workload": WORKLOADS[name], "descriptors_per_step": n_ops, "steps": K, "warmup": args.stream_warmup,
           "value": value, "unit": UNIT, "ms_per_step": kern_ms / K, "algorithmic_bytes_per_step": step_bytes,
           "l2": L2_NOTE[name],
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                        "frac": achieved / peak, "traffic": launch_traffic(name, n_ops * K)},
           "latency_us": latency_block(h, off, off_lo),
           "clock_offset_uncertainty_us": (off_hi - off_lo) / 2e3,
           "host_submit_ns_per_desc": r["submit_ns"] / (K * n_ops),
           "executor": {k: r["stats"][k] for k in ("seq_body_ns", "seq_mirror_ns", "seq_publish_ns",
                                                    "seq_batches", "host_wait_ns", "dep_waits")},
           "op_kinds": op_kind_table(s, h, n_ops, r["tprof"], K), "generate_and_upload_s": gen_s}
    if name == "c4":
        out["decode_steps_per_s"] = value / 3
    if name == "c5":
        out["tokens_per_s"] = value / (7 * 32)
    if not args.no_eager:
        ev, ems, _ = eager_rate(G, descs, K, 1, args.stage_bytes)
        out["eager"] = {"value": ev, "unit": UNIT, "ms_per_step": ems, "launches_per_step": n_ops}
        out["executor_vs_eager"] = value / ev
    if name in ("c1", "c4") and not args.no_graph:
        out["cuda_graph"] = graph_rate(G, descs, max(K, 3), args.stage_bytes)
    if name == "c5" and gemm is not None:
        out["corun_gemm"] = corun_curve(G, descs, cfg_kw, gemm, args)
    del ds
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def corun_curve(G, descs, cfg_kw, gemm, args):
    """The mixed pipeline on B executor blocks (one per SM) while the GEMM
    loops on a second stream: GEMM TFLOP/s over the GEMMs that completed
    while the executor was resident, and the executor's own rate."""
    n_ops = len(descs)
    rows = []
    for B in [int(x) for x in args.corun_blocks.split(",") if x]:
        kw = dict(cfg_kw)
        kw["blocks"] = B
        r = timed_executor(G, descs, kw, 1, gemm=gemm, history=False)
        rows.append({"executor_blocks": B, "executor_ops_per_s": n_ops / (r["kern_ms"] / 1e3),
                     "executor_kernel_ms": r["kern_ms"], **r["gemm"]})
    return {"gemm": "torch.matmul bf16 8192^3, operands N(0, 0.02), second stream",
            "alone_tflops": gemm.alone_tflops, "curve": rows}


# An operator that did not exist when the executor was launched, compiled
# at run time: out[i] = a[i] * 2 (fp32), tiles split like the built-in
# element-wise ops so it can serve under a built-in id's tile count.
_HANDOFF_OP_SRC = r'''
__device__ int op_twice(const gpuos_devdesc *d, uint32_t tile)
{
    const uint32_t n = d->dims[0], lane = threadIdx.x & 31u;
    const uint32_t nt = d->ntiles ? d->ntiles : 1u;
    const uint32_t te = ((n + nt - 1u) / nt + 255u) / 256u * 256u;
    const float *a = reinterpret_cast<const float *>(d->a);
    float *o = reinterpret_cast<float *>(d->out);
    const unsigned long long start = (unsigned long long)tile * te;
    const unsigned long long end = start + te < n ? start + te : n;
    for (unsigned long long i = start + lane; i < end; i += 32) o[i] = a[i] * 2.0f;
    return GPUOS_ST_OK;
}
__device__ gpuos_op_fn op_twice_ptr = op_twice;
'''


def handoff_measure(G, local, cfg_kw):
    """Operator injection into a running executor (the page's dynamic
    operator table, §3 Q2): the smallest stream runs, an operator compiled
    with NVRTC after the launch is registered (a hand-off: drain, the kernel
    leaves, the module set is linked again, the kernel relaunches at the
    next ticket), and the stream runs again. Reports the call's host time,
    the time spent linking (while the old executor still runs), the
    executor's downtime (stop request to the new kernel running) and the
    operator's own dispatch-to-done time."""
    import torch
    from workloads import streams as S
    from workloads.device import DeviceStream
    s = S.stream_c1()
    ds = DeviceStream(s, device=f"cuda:{local}")
    d = ds.descs()
    t0 = time.perf_counter()
    img = G.compile_op(_HANDOFF_OP_SRC, "twice.cu")
    compile_s = time.perf_counter() - t0
    n = 4096
    x = torch.randn(n, device=f"cuda:{local}")
    y = torch.zeros(n, device=f"cuda:{local}")
    torch.cuda.synchronize()
    op = G.make_descs(1)
    op["op_id"] = 90
    op["dtype"] = G.F32
    op["a"], op["out"] = x.data_ptr(), y.data_ptr()
    op["dims"][0, 0] = n
    op["ntiles"] = 4
    ex = G.Executor(**cfg_kw)
    try:
        hist = ex.set_history(0, 2 * len(d) + 1)
        ex.submit_batch(d)
        ex.sync(timeout_ms=60_000)
        a = time.perf_counter()
        ex.register_op(90, img, "op_twice_ptr")
        call_s = time.perf_counter() - a
        ex.submit_batch(d)
        ex.submit(op)
        ex.sync(timeout_ms=60_000)
        st = ex.stats()
    finally:
        ex.shutdown()
    ok = bool(torch.equal(y, x * 2.0))
    m = len(d)
    op_us = (int(hist["t_done_dev_ns"][2 * m]) - int(hist["t_dispatch_dev_ns"][2 * m])) / 1e3
    return {"compile_s": compile_s, "register_call_s": call_s, "handoffs": int(st["handoffs"]),
            "link_ms": st["handoff_link_ns"] / 1e6, "executor_down_ms": st["handoff_down_ns"] / 1e6,
            "op_dispatch_to_done_us": op_us, "result_ok": ok, "errors": int(st["errors"]),
            "version": int(st["version"])}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c2", choices=sorted(WORKLOADS))
    ap.add_argument("--tokens", type=int, default=500, help="tokens per step of the c5 workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-eager", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-handoff", action="store_true")
    ap.add_argument("--streams", default="c1,c2l,c3,c4,c5",
                    help="other workloads measured into the same line ('' = none)")
    ap.add_argument("--stream-steps", type=int, default=3, help="timed steps of each other workload")
    ap.add_argument("--c1-steps", type=int, default=200, help="timed steps of the smallest stream, at least")
    ap.add_argument("--stream-warmup", type=int, default=3, help="warm-up steps of each other workload")
    ap.add_argument("--corun-blocks", default="8,19,38,76,152",
                    help="executor blocks of the GEMM co-run curve (mixed pipeline); '' = none")
    ap.add_argument("--profile-run", action="store_true",
                    help="one bounded executor run (ring filled before launch) for profilers; no JSON")
    ap.add_argument("--profile-desc", type=int, default=0,
                    help="profile run: descriptors (0 = the workload's own, capped at the ring size)")
    ap.add_argument("--profile-idle-ms", type=int, default=0,
                    help="profile run: leave by the idle watchdog after this long instead of after the last "
                         "completion (the executor polls an empty ring until then)")
    ap.add_argument("--gemm-alone", type=int, default=0,
                    help="only run this many 8192^3 bf16 GEMMs and print their TFLOP/s (for profilers)")
    ap.add_argument("--pool-log2", type=int, default=0, help="profile run: log2 of the input pool elements")
    ap.add_argument("--warps", type=int, default=0, help="executor warps per block (0 = default)")
    ap.add_argument("--stage-bytes", type=int, default=16384, help="shared-memory staging per warp (0 = none)")
    ap.add_argument("--blocks", type=int, default=0, help="executor blocks (0 = one per SM)")
    ap.add_argument("--sequencers", type=int, default=0, help="sequencer warps (0 = the library's default)")
    ap.add_argument("--ring-entries", type=int, default=0, help="ring slots (0 = the library's default, 8192)")
    ap.add_argument("--spin-polls", type=int, default=0, help="idle polls before backoff sleeps (0 = default)")
    ap.add_argument("--backoff-max-ns", type=int, default=0, help="longest idle sleep (0 = default)")
    ap.add_argument("--producers-sweep", action="store_true",
                    help="host-thread contention curve: T threads submitting NOP batches (multi_producer=1); "
                         "prints its own JSON line")
    ap.add_argument("--ring-device", action="store_true",
                    help="ring in device memory (managed, host-accessible) instead of pinned host memory")
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
    if args.gemm_alone:
        gemm = Gemm(local)
        print(json.dumps({"gemm_alone_tflops": gemm.measure_alone(args.gemm_alone), "gemms": args.gemm_alone}))
        return 0
    from persistent_micro_dispatch_gb300 import build as pkg_build
    pkg_build.build()
    from persistent_micro_dispatch_gb300 import gpuos as G
    from workloads import streams as S
    from workloads.device import DeviceStream, warm_torch

    cfg_kw = dict(device=local, idle_exit_ms=20000, stage_bytes=args.stage_bytes, blocks=args.blocks)
    if args.warps:
        cfg_kw["warps_per_block"] = args.warps
    if args.sequencers:
        cfg_kw["sequencers"] = args.sequencers
    if args.ring_entries:
        cfg_kw["ring_entries"] = args.ring_entries
    elif args.workload == "c1":
        cfg_kw["ring_entries"] = 4096  # as the smallest stream is defined
    if args.spin_polls:
        cfg_kw["spin_polls"] = args.spin_polls
    if args.backoff_max_ns:
        cfg_kw["backoff_max_ns"] = args.backoff_max_ns
    if args.ring_device:
        cfg_kw["ring_in_device_mem"] = 1
    if args.profile_run and args.profile_desc and args.workload in ("c1", "c2", "c2l", "c3"):
        kw = dict(n_desc=args.profile_desc)
        if args.pool_log2 and args.workload != "c1":
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
        return producers_sweep(local)
    if args.profile_run:
        # bounded run with the ring filled before the single launch: the
        # kernel ends on its own after len(descs) completions (replayable),
        # or, with --profile-idle-ms, by its idle watchdog after polling an
        # empty ring for that long
        nprof = min(n_ops, 4096)
        if args.profile_idle_ms:
            kw = dict(cfg_kw, idle_exit_ms=args.profile_idle_ms)
            ex = G.Executor(**kw, deferred_start=1)
        else:
            ex = G.Executor(**cfg_kw, deferred_start=1, exit_after=nprof)
        ex.submit_batch(descs[:nprof])
        ex.start()
        rc = ex.sync(timeout_ms=120_000, raise_on_error=False)
        if args.profile_idle_ms:
            # no library call meanwhile: each one counts as host activity
            # and restarts the executor's idle clock
            time.sleep(args.profile_idle_ms / 1e3 + 0.5)
        ex.shutdown()
        print(f"profile run: {nprof} descriptors, sync rc={rc}", flush=True)
        return 0

    peak, peak_kind = measured_peak_gbs()
    # GEMM of the co-run curve: loaded and measured alone before any
    # executor is resident (a kernel first loaded beside a resident executor
    # waits for the device to go idle)
    others = [x for x in args.streams.split(",") if x and x != args.workload]
    gemm = None
    if "c5" in others and args.corun_blocks:
        gemm = Gemm(local)
        gemm.alone_tflops = gemm.measure_alone(20)

    # ---- warm-up executor: warm-up steps, clock calibration, isolated latency
    ex = G.Executor(**cfg_kw)
    for _ in range(args.warmup):
        ex.submit_batch(descs)
        ex.sync(timeout_ms=600_000)
    iso = isolated_latency(G, ex, descs, n_ops)
    rc_sd = ex.shutdown()
    if rc_sd != G.OK:
        print(f"warm-up executor shutdown: {G.strerror(rc_sd)}", file=sys.stderr)
    off_lo, off_hi = iso["off_lo"], iso["off_hi"]
    off = (off_lo + off_hi) // 2

    # ---- timed region: one launch of the persistent executor, K steps
    clocks = ClockSampler(local)
    torch.cuda.synchronize()
    barrier(world)
    clocks.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    r = timed_executor(G, descs, cfg_kw, args.steps)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(world)
    clk = clocks.stop()
    wall = t1 - t0
    kern_ms = r["kern_ms"]
    st = r["stats"]
    units, secs = aggregate(n_ops * args.steps, kern_ms / 1e3, world)
    value = units / secs

    h = r["hist"][r["hist"]["ticket"] != np.iinfo(np.uint64).max]
    ih = iso["iso_hist"]
    ih_commit = ih["t_commit_host_ns"].astype(np.int64)
    iso_disp_us = (ih["t_dispatch_dev_ns"].astype(np.int64) - ih_commit - off) / 1e3
    iso_disp_up = (ih["t_dispatch_dev_ns"].astype(np.int64) - ih_commit - off_lo) / 1e3
    iso_dev_us = (ih["t_done_dev_ns"].astype(np.int64) - ih["t_dispatch_dev_ns"].astype(np.int64)) / 1e3
    busy_ns = int(h["t_done_dev_ns"].max()) - int(h["t_dispatch_dev_ns"].min()) if len(h) else 0
    achieved = step_bytes * args.steps / (kern_ms / 1e3) / 1e9
    lat = latency_block(h, off, off_lo)
    lat.update({
        "isolated_roundtrip_p50": pct(iso["iso_rtt"] / 1e3, 50),
        "isolated_roundtrip_p99": pct(iso["iso_rtt"] / 1e3, 99),
        "isolated_submit_to_dispatch_p50": pct(iso_disp_us, 50),
        "isolated_submit_to_dispatch_p50_upper": pct(iso_disp_up, 50),
        "isolated_dispatch_to_done_p50": pct(iso_dev_us, 50),
        "clock_offset_uncertainty": (off_hi - off_lo) / 2e3,
        "nop_roundtrip_min": iso["min_rtt"] / 1e3, "nop_roundtrip_p50": float(np.median(iso["rtts"])) / 1e3,
        "host_submit_ns_per_desc": r["submit_ns"] / (args.steps * n_ops),
    })
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": kern_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "descriptors_per_step": n_ops,
                   "algorithmic_bytes_per_step": step_bytes, "l2": L2_NOTE[args.workload],
                   "parallelism": f"replicas x{world}", "ring_entries": int(r["config"].ring_entries),
                   "warps_per_block": int(st["warps_per_block"]), "blocks": int(st["blocks"])},
        "gpu_launches": 1,
        "latency_us": lat,
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": launch_traffic(args.workload, n_ops * args.steps),
                     "peak_kind": peak_kind,
                     "kernel": "gpuos_executor_kernel", "kernel_ms": kern_ms,
                     "device_busy_ms_last_step": busy_ns / 1e6},
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
        "op_kinds": op_kind_table(s, h, n_ops, r["tprof"], args.steps),
        "executor": {k: st[k] for k in ("tiles", "idle_polls", "sleeps", "dep_waits", "regs_per_thread",
                                        "static_smem_bytes", "seq_body_ns", "seq_mirror_ns", "seq_publish_ns",
                                        "seq_batches", "host_wait_ns")},
        "wall_s": wall,
    }

    # ---- eager baseline: same op bodies, one cudaLaunchKernel per descriptor
    if not args.no_eager:
        ev, ems, es = eager_rate(G, descs, args.steps, args.warmup, args.stage_bytes)
        # isolated latency, measured like the executor's isolated round trip:
        # the same sampled ops, one launch each, then a wait for it (host clock)
        eg_rtt = []
        for j in iso["iso_idx"]:
            d1 = descs[j:j + 1].copy()
            d1["dep"] = 0
            ta = G.host_now_ns()
            G.eager_run(d1, es.cuda_stream, args.stage_bytes)
            es.synchronize()
            eg_rtt.append(G.host_now_ns() - ta)
        result["eager"] = {"value": ev, "unit": UNIT, "ms_per_step": ems, "launches_per_step": n_ops,
                           "isolated_roundtrip_p50": pct(np.array(eg_rtt) / 1e3, 50),
                           "isolated_roundtrip_p99": pct(np.array(eg_rtt) / 1e3, 99)}

    # ---- CUDA Graphs baseline on the headline workload
    if not args.no_graph:
        result["cuda_graph"] = graph_rate(G, descs, args.steps, args.stage_bytes)

    # ---- end to end: host buffers, copies inside the timed region
    if not args.no_e2e:
        in_idx = [i for i, b in enumerate(s.buffers) if b.data is not None]
        out_idx = sorted({o_ref.buf for o in s.ops for o_ref in (o.out, o.aux1 if o.op == "kv_write" else None)
                          if o_ref is not None} - set(in_idx))
        host_in = [torch.from_numpy(np.ascontiguousarray(s.buffers[i].data).view(np.uint8)).pin_memory() for i in in_idx]
        host_out = [torch.empty(ds.bufs[i].numel(), dtype=torch.uint8).pin_memory() for i in out_idx]
        h2d = sum(t.numel() for t in host_in)
        d2h = sum(t.numel() for t in host_out)
        # two sets of device buffers, used by alternate steps: the copy of a
        # step's results back to the host overlaps the next step's input copy
        # and run (copy engines run both directions at once), and a set is
        # reused only once its previous results have left
        ds2 = DeviceStream(s, device=f"cuda:{local}")
        sets = [(ds, descs), (ds2, ds2.descs())]
        cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
        out_done = [None, None]
        # device-wide synchronisation only while no executor is resident: a
        # resident persistent kernel never lets it return
        torch.cuda.synchronize()
        ex = G.Executor(**cfg_kw)
        barrier(world)
        a = time.perf_counter()
        for k in range(args.steps):
            dsk, dk = sets[k % 2]
            with torch.cuda.stream(cin):
                for i, t in zip(in_idx, host_in):
                    dsk.bufs[i].copy_(t, non_blocking=True)
            cin.synchronize()
            if out_done[k % 2] is not None:
                out_done[k % 2].synchronize()  # this set's previous results have left
            ex.submit_batch(dk)
            ex.sync(timeout_ms=600_000)
            with torch.cuda.stream(cout):
                for i, t in zip(out_idx, host_out):
                    t.copy_(dsk.bufs[i], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cout)
            out_done[k % 2] = ev
        cout.synchronize()
        b = time.perf_counter()
        ex.shutdown()
        torch.cuda.synchronize()
        del sets, ds2
        eu, esec = aggregate(n_ops * args.steps, b - a, world)
        result["e2e"] = {"value": eu / esec, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": 1e3 * (b - a) / args.steps}
        del host_in, host_out

    # ---- operator injection into the running executor (hand-off)
    if not args.no_handoff:
        result["handoff"] = handoff_measure(G, local, cfg_kw)

    # ---- the other workloads, measured the same way (rank 0's GPU only
    # matters for the line; every rank runs them so the ranks stay aligned)
    if others:
        del ds
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        result["streams"] = {}
        for name in others:
            result["streams"][name] = stream_phase(G, name, args, cfg_kw, local, peak, gemm=gemm)

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    if not args.no_cpu and rank == 0 and world == 1:
        rr, n, dt, sample = oracle_rate(args.workload, 12.0)
        result["cpu_baseline"] = {"value": rr, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                                  "seconds": dt, "host_cores": os.cpu_count()}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
