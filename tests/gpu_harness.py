"""Shared helpers of the GPU tests: build once, run a stream through the
persistent executor (or the eager path) and compare with the oracle."""
from __future__ import annotations

import os
import random
from typing import Iterable, List, Optional

import numpy as np
import pytest

from oracle.interp import Machine
from tests.parity import Report, compare_op, operand_accesses, writers_of
from workloads.streams import NPTYPE, Stream, op_accesses


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


_built = False


def ensure_built():
    global _built
    if not _built:
        from persistent_micro_dispatch_gb300 import build
        build.build()
        _built = True


def run_executor(ds, descs: np.ndarray, timeout_ms: int = 120_000, **cfg):
    """Submit every descriptor to a fresh executor, wait, return (stats, records)."""
    from persistent_micro_dispatch_gb300 import gpuos as G
    from workloads.device import warm_torch
    warm_torch()
    ex = G.Executor(**cfg)
    try:
        hist = ex.set_history(0, len(descs))
        ex.submit_batch(descs)
        rc = ex.sync(timeout_ms=timeout_ms, raise_on_error=False)
        st = ex.stats()
    finally:
        sd = ex.shutdown()
    assert sd == G.OK, f"shutdown: {G.strerror(sd)}"
    assert rc == G.OK, f"sync: {G.strerror(rc)}; stats={st}"
    return st, hist


def final_output_ops(s: Stream, candidates: Iterable[int]) -> List[int]:
    """Ops whose written ranges no later op writes (comparable at the end)."""
    out = []
    for j in candidates:
        if not any(i > j for (b, lo, hi, w) in operand_accesses(s, s.ops[j]) if w for i in writers_of(s, b, lo, hi)):
            out.append(j)
    return out


def compare_stream(s: Stream, ds, mach: Machine, indices: Iterable[int]) -> Report:
    """Compare ops against an oracle machine that has already run the whole
    stream (every op's inputs must still hold what the op read)."""
    rep = Report()
    for j in indices:
        compare_op(rep, s, j, ds.read, mach)
    return rep


class TimedView:
    """GPU results as they stood right after a given op. A buffer written only
    by KV writes (row copies, compared byte for byte against a replay of
    every KV write by check_kv_copies) is rebuilt from its initial contents
    and the GPU's own k/v rows, up to and including the op being compared;
    every other range is read as it stands at the end of the run."""

    def __init__(self, s: Stream, ds):
        self.s, self.ds = s, ds
        kv = {r.buf for o in s.ops if o.op == "kv_write" for r in (o.out, o.aux1)}
        other = {b for o in s.ops if o.op != "kv_write" for (b, lo, hi, w) in op_accesses(s, o) if w}
        self.replayed = {b for b in kv - other if s.buffers[b].data is not None}
        self.cur = {b: s.buffers[b].data.copy() for b in self.replayed}
        self.at = 0  # ops [0, at) applied to the replayed buffers
        if self.replayed:
            # the k/v rows a replayed KV write copies must be final (no later
            # writer), so that reading them at the end gives what it copied
            for j, o in enumerate(s.ops):
                if o.op == "kv_write" and o.out.buf in self.replayed:
                    B, H, D = o.dims[:3]
                    for ref in (o.a, o.b):
                        later = [i for i in writers_of(s, ref.buf, ref.off, ref.off + B * H * D) if i > j]
                        assert not later, f"k/v rows of KV write {j} are rewritten by op {later[0]}"

    def timed(self, b: int) -> bool:
        return b in self.replayed

    def advance(self, j: int) -> None:
        """State right after op j (ops are visited in increasing order)."""
        assert j + 1 >= self.at, "TimedView moves forward only"
        while self.at <= j:
            o = self.s.ops[self.at]
            if o.op == "kv_write" and o.out.buf in self.replayed:
                B, H, D, Lc = o.dims[:4]
                lens = self.s.buffers[o.aux0.buf].data[o.aux0.off:o.aux0.off + B]
                for src, dst in ((o.a, o.out), (o.b, o.aux1)):
                    rows = self.ds.read(src, B * H * D).reshape(B, H, D)
                    c = self.cur[dst.buf][dst.off:dst.off + B * H * Lc * D].reshape(B, H, Lc, D)
                    for bb in range(B):
                        c[bb, :, int(lens[bb]) - 1] = rows[bb]
            self.at += 1

    def __call__(self, ref, n, dtype=None):
        if ref.buf in self.replayed:
            v = self.cur[ref.buf][ref.off:ref.off + n]
            return v.copy() if dtype is None else v.view(NPTYPE[dtype]).copy()
        return self.ds.read(ref, n, dtype)


def comparable_ops(s: Stream, view: TimedView, candidates: Iterable[int]) -> List[int]:
    """Ops whose outputs can be read as they stood right after the op: every
    written range is final or lies in a buffer the view rebuilds."""
    out = []
    for j in candidates:
        if not any(i > j for (b, lo, hi, w) in operand_accesses(s, s.ops[j]) if w and not view.timed(b)
                   for i in writers_of(s, b, lo, hi)):
            out.append(j)
    return out


def compare_in_order(s: Stream, ds, targets: Optional[Iterable[int]] = None, skip: Iterable[int] = ()):
    """Run the oracle op by op and compare each checked op with the GPU's
    result as it stood right after that op (``TimedView``).

    targets: ops to check (default: every comparable op). With targets, the
    oracle applies only the targets and everything they depend on, and every
    comparable op it applies is checked too, so that each producer a
    consumer's tolerance widens from has been checked first. skip: ops the
    oracle leaves out (the caller's claim that nothing else reads their
    outputs). Returns (report, machine)."""
    view = TimedView(s, ds)
    mach = Machine(s)
    mach._op_index = {id(op): k for k, op in enumerate(s.ops)}
    skip = set(skip)
    targets = None if targets is None else set(targets)
    if targets is None:
        order = [j for j in range(len(s.ops)) if j not in skip]
    else:
        # the targets and everything they depend on (through skipped ops
        # too, which are themselves not applied)
        need, seen = set(), set()
        stack = list(targets)
        while stack:
            k = stack.pop()
            if k in seen:
                continue
            seen.add(k)
            if k not in skip or k in targets:
                need.add(k)
            if s.ops[k].fence:
                stack.extend(range(k))
            stack.extend(s.ops[k].deps)
        order = sorted(need)
    check = set(comparable_ops(s, view, order))
    if targets is not None:
        missing = set(targets) - check
        assert not missing, f"targets not comparable: {sorted(missing)[:5]}"
    rep = Report()
    for j in order:
        mach.apply(j, keep=j in check)
        if j in check:
            view.advance(j)
            compare_op(rep, s, j, view, mach)
    return rep, mach


def check_canaries(s: Stream, ds, names=("out", "out_f32", "out_bf16")) -> None:
    """Bytes of output arenas that no op writes must still hold the canary."""
    for i, b in enumerate(s.buffers):
        if b.name not in names or b.data is not None:
            continue
        written = np.zeros(b.nelem, dtype=bool)
        for o in s.ops:
            for (bb, lo, hi, w) in op_accesses(s, o):
                if bb == i and w:
                    written[lo:hi] = True
        raw = ds.read_buf(i).view(np.uint8).reshape(b.nelem, -1)
        unw = raw[~written]
        assert np.all(unw == b.fill), f"canary overwritten in {b.name}: {np.count_nonzero(unw != b.fill)} bytes"


def sample(indices: List[int], k: int, seed: int = 0) -> List[int]:
    rng = random.Random(seed)
    if len(indices) <= k:
        return list(indices)
    return sorted(rng.sample(indices, k))


def check_kv_copies(s, ds):
    """Replay every KV write with the GPU's own (rotated) k/v rows on the
    initial caches: the GPU caches must equal the result byte for byte."""
    caches = {}
    for o in s.ops:
        if o.op != "kv_write":
            continue
        for ref in (o.out, o.aux1):
            if ref.buf not in caches:
                caches[ref.buf] = s.buffers[ref.buf].data.copy()
        B, H, D, Lc = o.dims[:4]
        lens = s.buffers[o.aux0.buf].data[o.aux0.off:o.aux0.off + B]
        k = ds.read(o.a, B * H * D).reshape(B, H, D)
        v = ds.read(o.b, B * H * D).reshape(B, H, D)
        K4 = caches[o.out.buf][o.out.off:o.out.off + B * H * Lc * D].reshape(B, H, Lc, D)
        V4 = caches[o.aux1.buf][o.aux1.off:o.aux1.off + B * H * Lc * D].reshape(B, H, Lc, D)
        for b in range(B):
            K4[b, :, lens[b] - 1] = k[b]
            V4[b, :, lens[b] - 1] = v[b]
    assert caches, "no KV write in the stream"
    for i, want in caches.items():
        assert np.array_equal(ds.read_buf(i), want), s.buffers[i].name
