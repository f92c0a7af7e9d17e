"""Sequential interpreter over a descriptor stream -- TEST INFRASTRUCTURE ONLY.

Applies each descriptor of a ``workloads.streams.Stream`` to host copies of
its buffers, in ticket order, calling the C definitions in ``oracle.c``.
Dependencies are not needed for the meaning of a stream: sequential order is
the specification, and the GPU must reproduce it ("GPUOS: A GPU Operating
System Primitive for Transparent Operation Fusion", §2 and §3 Q2: the host
writes descriptors into a ring and the device executes what they describe).

For every op it applies, the interpreter can keep the exact (unrounded,
double) result next to the rounded value it stores, so that tests can judge
bf16 outputs against the exact value.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, Iterable, List, Optional, Set

import numpy as np

from oracle import build as _build
from workloads.streams import ESIZE, NPTYPE, Op, Stream

_lib = None

_DT = {"f32": 0, "bf16": 1}
_P = C.c_void_p
_L = C.c_long
_D = C.c_double


def lib():
    """Load (building if needed) the C oracle."""
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build.build())
        _lib.orc_bf16_from_double.restype = C.c_uint16
        _lib.orc_bf16_from_double.argtypes = [_D]
        _lib.orc_bf16_to_double.restype = _D
        _lib.orc_bf16_to_double.argtypes = [C.c_uint16]
        _lib.orc_store.argtypes = [C.c_int, _P, _P, _L]
        for f in ("orc_add", "orc_mul"):
            getattr(_lib, f).argtypes = [C.c_int, _P, _P, _P, _L]
        for f in ("orc_relu", "orc_gelu"):
            getattr(_lib, f).argtypes = [C.c_int, _P, _P, _L]
        _lib.orc_softmax.argtypes = [_P, _L, _L, _P]
        _lib.orc_layernorm.argtypes = [_P, _P, _P, _L, _L, _D, _P]
        _lib.orc_rowreduce.argtypes = [C.c_int, _P, _L, _L, _P]
        _lib.orc_rope.argtypes = [_P, _P, _P, _L, _L, _L, _D, _P, _P]
        _lib.orc_rope.restype = C.c_int
        _lib.orc_kv_write.argtypes = [_P, _P, _P, _L, _L, _L, _L, _P, _P]
        _lib.orc_kv_write.restype = C.c_int
        _lib.orc_sdpa.argtypes = [_P, _P, _P, _P, _L, _L, _L, _L, _D, _P]
        _lib.orc_sdpa.restype = C.c_int
        _lib.orc_vecmat.argtypes = [_P, _P, _L, _L, _P]
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def bf16_round(x) -> np.ndarray:
    """Round doubles to bf16 bit patterns with the oracle's rounding."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.size, dtype=np.uint16)
    lib().orc_store(1, _ptr(x), _ptr(out), x.size)
    return out.reshape(x.shape)


class Machine:
    """Host copies of a stream's buffers plus an in-order op applier."""

    def __init__(self, stream: Stream, lazy_outputs: bool = False):
        self.s = stream
        self.buf: List[np.ndarray] = [b.materialize() for b in stream.buffers]
        # exact[j] = {"out": double array, ...} for ops applied with keep=True
        self.exact: Dict[int, Dict[str, np.ndarray]] = {}
        self.status: Dict[int, int] = {}

    # -- views ------------------------------------------------------------
    def view(self, ref, n: int, dtype: Optional[str] = None) -> np.ndarray:
        b = self.buf[ref.buf]
        if dtype is not None and NPTYPE[dtype] != b.dtype:
            b = b.view(NPTYPE[dtype])
        return b[ref.off:ref.off + n]

    # -- one op -------------------------------------------------------------
    def apply(self, j: int, keep: bool = False) -> None:
        o: Op = self.s.ops[j]
        L = lib()
        d = o.dims
        st = 0
        ex: Dict[str, np.ndarray] = {}
        if o.op in ("add", "mul", "relu", "gelu"):
            n = d[0]
            dt = _DT[o.dtype]
            a = self.view(o.a, n)
            out = np.empty(n, dtype=np.float64)
            if o.op in ("add", "mul"):
                b = self.view(o.b, n)
                getattr(L, "orc_" + o.op)(dt, _ptr(a), _ptr(b), _ptr(out), n)
            else:
                getattr(L, "orc_" + o.op)(dt, _ptr(a), _ptr(out), n)
            L.orc_store(dt, _ptr(out), _ptr(self.view(o.out, n)), n)
            ex["out"] = out
        elif o.op in ("softmax", "layernorm"):
            R, H = d[:2]
            x = self.view(o.a, R * H)
            out = np.empty(R * H, dtype=np.float64)
            if o.op == "softmax":
                L.orc_softmax(_ptr(x), R, H, _ptr(out))
            else:
                L.orc_layernorm(_ptr(x), _ptr(self.view(o.b, H)), _ptr(self.view(o.aux0, H)), R, H,
                                float(o.fparam[0]), _ptr(out))
            L.orc_store(1, _ptr(out), _ptr(self.view(o.out, R * H)), R * H)
            ex["out"] = out
        elif o.op in ("rowsum", "rowmax", "rowmin"):
            R, H = d[:2]
            x = self.view(o.a, R * H)
            out = np.empty(R, dtype=np.float64)
            L.orc_rowreduce(("rowsum", "rowmax", "rowmin").index(o.op), _ptr(x), R, H, _ptr(out))
            odt = 0 if o.op == "rowsum" else 1
            L.orc_store(odt, _ptr(out), _ptr(self.view(o.out, R)), R)
            ex["out"] = out
        elif o.op == "rope":
            B, H, D = d[:3]
            n = B * H * D
            q, k = self.view(o.a, n), self.view(o.b, n)
            lens = self.view(o.aux0, B)
            qo = np.empty(n, dtype=np.float64)
            ko = np.empty(n, dtype=np.float64)
            st = L.orc_rope(_ptr(q), _ptr(k), _ptr(lens), B, H, D, float(o.fparam[0]), _ptr(qo), _ptr(ko))
            if st == 0:
                L.orc_store(1, _ptr(qo), _ptr(q), n)
                L.orc_store(1, _ptr(ko), _ptr(k), n)
            ex["a"], ex["b"] = qo, ko
        elif o.op == "kv_write":
            B, H, D, Lc = d[:4]
            n = B * H * D
            st = L.orc_kv_write(_ptr(self.view(o.a, n)), _ptr(self.view(o.b, n)), _ptr(self.view(o.aux0, B)),
                                B, H, D, Lc, _ptr(self.view(o.out, B * H * Lc * D)),
                                _ptr(self.view(o.aux1, B * H * Lc * D)))
        elif o.op == "sdpa":
            B, H, D, Lc = d[:4]
            n = B * H * D
            out = np.empty(n, dtype=np.float64)
            st = L.orc_sdpa(_ptr(self.view(o.a, n)), _ptr(self.view(o.b, B * H * Lc * D)),
                            _ptr(self.view(o.aux1, B * H * Lc * D)), _ptr(self.view(o.aux0, B)),
                            B, H, D, Lc, float(o.fparam[0]), _ptr(out))
            if st == 0:
                L.orc_store(1, _ptr(out), _ptr(self.view(o.out, n)), n)
            ex["out"] = out
        elif o.op == "vecmat":
            K, N = d[:2]
            out = np.empty(N, dtype=np.float64)
            L.orc_vecmat(_ptr(self.view(o.a, K)), _ptr(self.view(o.b, K * N)), K, N, _ptr(out))
            L.orc_store(1, _ptr(out), _ptr(self.view(o.out, N)), N)
            ex["out"] = out
        elif o.op == "nop":
            pass
        else:
            raise ValueError(o.op)
        self.status[j] = st
        if keep:
            self.exact[j] = ex

    # -- many ops -------------------------------------------------------------
    def run(self, keep: Optional[Iterable[int]] = None, upto: Optional[int] = None,
            skip: Optional[Iterable[int]] = None) -> None:
        """Apply ops 0..upto-1 in order; keep exact results for ``keep``.

        ``skip`` names ops whose outputs no later op reads (the caller's
        claim); leaving them out does not change any other op's result."""
        keep_set: Set[int] = set(keep) if keep is not None else set()
        skip_set: Set[int] = set(skip) if skip is not None else set()
        n = len(self.s.ops) if upto is None else upto
        for j in range(n):
            if j in skip_set and j not in keep_set:
                continue
            self.apply(j, keep=j in keep_set)

    def run_closure(self, targets: Iterable[int]) -> List[int]:
        """Apply, in ticket order, ``targets`` and every op they depend on.

        Valid for streams that pass the hazard checker: every producer of a
        value that a target reads is among its (transitive) dependencies.
        Returns the applied op indices.
        """
        need: Set[int] = set()
        stack = list(targets)
        while stack:
            k = stack.pop()
            if k in need:
                continue
            need.add(k)
            if self.s.ops[k].fence:
                stack.extend(range(k))
            stack.extend(self.s.ops[k].deps)
        tset = set(targets)
        order = sorted(need)
        for j in order:
            self.apply(j, keep=j in tset)
        return order


def esize(dtype: str) -> int:
    return ESIZE[dtype]
