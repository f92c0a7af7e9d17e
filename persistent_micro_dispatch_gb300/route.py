"""Routing of eligible PyTorch ops to the persistent executor (hybrid execution).

GPUOS page, §3 Q2 (PyTorch integration): a dispatch hook intercepts every op
and a four-dimensional filter decides where it runs; ops that fail it (large
GEMMs, anything the operator library lacks) keep PyTorch's normal launch
path. The filter here:

1. operation type: add, mul (same-shape tensors), ReLU, exact GELU, softmax
   over the last dim (bf16); contiguous CUDA tensors, fp32 or bf16;
2. tensor size: at most ``max_elems`` elements (small tensors gain most);
3. execution context: an op signature (aten op, dtype, shape) is routed only
   once it has been seen ``min_calls`` times (inner-loop ops first);
4. current load: a submission that finds the ring full (no free slot at
   once) falls back to the normal launch.

The executor must leave room on the SMs for the ordinary kernels (the
page's executor takes one block per SM and a few per cent of its threads):
the default configuration (12 warps, 197 KB of staging per SM) fills every
SM, and an ordinary kernel launched beside it would wait until it leaves.
Use for instance ``Executor(warps_per_block=4)`` (a third of the registers,
75 KB of shared memory per SM) or ``blocks`` below the SM count. And every
kernel the program launches the normal way must have been loaded before the
executor starts (run it once, or set CUDA_MODULE_LOADING=EAGER): with lazy
module loading its first launch loads its module, and a module load waits for
the device to go idle, which it never does while the executor is resident.

Ordering with the rest of PyTorch: a routed op that reads the output of
another routed op depends on its ticket (the executor orders them); before
the first routed op after ordinary kernels, the current stream is
synchronised (their outputs may be its inputs); an ordinary op that reads a
routed op's output first waits for that ticket on the host. Tensors a routed
op touches stay referenced until its ticket completes. The computation of a
routed op is the library's own CUDA kernel: this module only marshals
arguments, as the ctypes binding does.
"""
from __future__ import annotations

import weakref
from typing import Dict, Optional, Tuple

import numpy as np
import torch
from torch.utils._python_dispatch import TorchDispatchMode

from . import gpuos as G

aten = torch.ops.aten

_EW = {aten.add.Tensor: "add", aten.mul.Tensor: "mul", aten.relu.default: "relu", aten.gelu.default: "gelu"}


class GpuosRouting(TorchDispatchMode):
    """``with GpuosRouting(executor): ...`` routes eligible ops to ``executor``."""

    def __init__(self, executor: G.Executor, max_elems: int = 1 << 20, min_calls: int = 2):
        super().__init__()
        self.ex = executor
        self.max_elems = max_elems
        self.min_calls = min_calls
        self.calls: Dict[Tuple, int] = {}
        # id(output tensor) -> (weak reference to it, ticket of the routed op
        # that writes it); tensors compare element-wise, so they are looked up
        # by identity
        self.pending: Dict[int, Tuple[weakref.ref, int]] = {}
        self.keep: list = []  # (ticket, tensors) kept alive until the ticket completes
        self.stream_dirty = True
        self.routed = 0
        self.fallback = 0

    # -- filter ---------------------------------------------------------------
    def _eligible(self, func, args, kwargs) -> Optional[Tuple[str, list]]:
        if func in _EW:
            name = _EW[func]
            if name in ("add", "mul"):
                if len(args) < 2 or not isinstance(args[1], torch.Tensor):
                    return None
                if kwargs.get("alpha", 1) != 1 or (len(args) > 2 and args[2] != 1):
                    return None
                a, b = args[0], args[1]
                if a.shape != b.shape or a.dtype != b.dtype:
                    return None
                ts = [a, b]
            elif name == "gelu":
                if kwargs.get("approximate", "none") != "none" or (len(args) > 1 and args[1] != "none"):
                    return None
                ts = [args[0]]
            else:
                ts = [args[0]]
            if ts[0].dtype not in (torch.float32, torch.bfloat16):
                return None
        elif func == aten._softmax.default:
            x, dim, half_to_float = args[0], args[1], args[2]
            if half_to_float or x.dtype != torch.bfloat16 or x.dim() < 1 or dim not in (-1, x.dim() - 1):
                return None
            name, ts = "softmax", [x]
        else:
            return None
        for t in ts:
            if not (t.is_cuda and t.is_contiguous()) or t.numel() == 0 or t.numel() > self.max_elems:
                return None
            if t.data_ptr() % 16:
                return None
        key = (func, ts[0].dtype, tuple(ts[0].shape))
        n = self.calls.get(key, 0) + 1
        self.calls[key] = n
        if n < self.min_calls:
            return None
        return name, ts

    # -- ordering helpers -------------------------------------------------------
    def _ticket_of(self, t: torch.Tensor) -> Optional[int]:
        e = self.pending.get(id(t))
        if e is None:
            return None
        if e[0]() is not t:  # a freed tensor's id reused
            del self.pending[id(t)]
            return None
        return e[1]

    def _wait_inputs(self, args, kwargs) -> None:
        """An ordinary op about to run: wait for routed producers of its inputs."""
        for a in list(args) + list(kwargs.values()):
            for t in (a if isinstance(a, (list, tuple)) else [a]):
                if isinstance(t, torch.Tensor):
                    tk = self._ticket_of(t)
                    if tk is not None:
                        self.ex.sync(tk)
                        del self.pending[id(t)]

    def _harvest(self) -> None:
        if len(self.keep) > 256:
            last = self.keep[-1][0]
            self.ex.sync(last)
            self.keep.clear()

    def drain(self) -> None:
        """Wait for every routed op (call before reading results elsewhere)."""
        self.ex.sync()
        self.pending.clear()
        self.keep.clear()

    # -- dispatch --------------------------------------------------------------
    def __torch_dispatch__(self, func, types, args=(), kwargs=None):
        kwargs = kwargs or {}
        sel = self._eligible(func, args, kwargs)
        if sel is not None:
            name, ts = sel
            x = ts[0]
            out = torch.empty_like(x)
            d = G.make_descs(1)
            d["op_id"] = G.OP[name]
            d["dtype"] = G.BF16 if x.dtype == torch.bfloat16 else G.F32
            d["a"] = x.data_ptr()
            if len(ts) > 1:
                d["b"] = ts[1].data_ptr()
            d["out"] = out.data_ptr()
            if name == "softmax":
                H = x.shape[-1]
                d["dims"][0, 0], d["dims"][0, 1] = x.numel() // H, H
            else:
                d["dims"][0, 0] = x.numel()
            deps = [tk + 1 for tk in (self._ticket_of(t) for t in ts) if tk is not None][:2]
            for i, v in enumerate(deps):
                d["dep"][0, i] = v
            if self.stream_dirty:
                torch.cuda.current_stream().synchronize()
                self.stream_dirty = False
            rc, ticket = self._try(d)
            if rc == G.OK:
                self.pending[id(out)] = (weakref.ref(out), ticket)
                self.keep.append((ticket, ts + [out]))
                self.routed += 1
                self._harvest()
                return out
            # ring full (current load): the normal launch path
        self.fallback += 1
        self._wait_inputs(args, kwargs)
        self.stream_dirty = True
        return func(*args, **kwargs)

    def _try(self, d: np.ndarray) -> Tuple[int, int]:
        import ctypes as C
        t = C.c_uint64()
        rc = G.lib().gpuos_submit(self.ex._ctx, np.ascontiguousarray(d).ctypes.data, C.byref(t), 0)
        return rc, t.value

    def __exit__(self, *exc):
        r = super().__exit__(*exc)
        self.drain()
        return r
