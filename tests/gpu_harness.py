"""Shared helpers of the GPU tests: build once, run a stream through the
persistent executor (or the eager path) and compare with the oracle."""
from __future__ import annotations

import os
import random
from typing import Iterable, List, Optional

import numpy as np
import pytest

from oracle.interp import Machine
from tests.parity import Report, compare_op
from workloads.streams import Stream, op_accesses


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
    last_writer = {}
    for j, o in enumerate(s.ops):
        for (b, lo, hi, w) in op_accesses(s, o):
            if w:
                last_writer.setdefault(b, []).append((lo, hi, j))
    out = []
    for j in candidates:
        o = s.ops[j]
        ok = True
        for (b, lo, hi, w) in op_accesses(s, o):
            if not w:
                continue
            for (l2, h2, k) in last_writer.get(b, []):
                if k > j and l2 < hi and lo < h2:
                    ok = False
                    break
            if not ok:
                break
        if ok:
            out.append(j)
    return out


def compare_stream(s: Stream, ds, mach: Machine, indices: Iterable[int]) -> Report:
    rep = Report()
    for j in indices:
        compare_op(rep, s, j, ds.read, mach)
    return rep


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
