"""Routing of eligible PyTorch ops to the persistent executor (hybrid execution).

GPUOS page, §3 Q2 (PyTorch integration): a dispatch hook intercepts every op
and a four-dimensional filter decides where it runs; ops that fail it (large
GEMMs, anything the operator library lacks) keep PyTorch's normal launch
path. The filter here:

1. operation type: element-wise ops, small reductions and (not here) cache
   updates first, as the page ranks them: add, mul (same-shape tensors),
   ReLU, exact GELU (fp32 or bf16), softmax over the last dim (bf16), and
   the row reductions over the last dim of a bf16 tensor that the operator
   library returns in PyTorch's own dtype: amax and amin (bf16 out) and sum
   with dtype=float32 (fp32 out; a bf16 sum would return bf16, which the
   library's fp32 row sum does not). LayerNorm is not routed: aten's
   native_layer_norm also returns the row statistics, which the library's
   LayerNorm does not produce. Contiguous CUDA tensors only;
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
synchronised (their outputs may be its inputs); an ordinary op that touches
the storage of a routed op's output first waits for that ticket on the host
(read after write), and an ordinary op that may write (an in-place or out=
op) to the storage of a routed op's input first waits for the last routed
op that reads it (write after read). Storages are matched, so views count.
Tensors a routed op touches stay referenced until its ticket completes, so
a matched storage cannot be a freed one reused. The computation of a
routed op is the library's own CUDA kernel: this module only marshals
arguments, as the ctypes binding does.
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import numpy as np
import torch
from torch.utils._python_dispatch import TorchDispatchMode

from . import gpuos as G

aten = torch.ops.aten

_EW = {aten.add.Tensor: "add", aten.mul.Tensor: "mul", aten.relu.default: "relu", aten.gelu.default: "gelu"}
_RED = {aten.amax.default: "rowmax", aten.amin.default: "rowmin", aten.sum.dim_IntList: "rowsum"}


def _storage(t: torch.Tensor) -> int:
    return t.untyped_storage().data_ptr()


class GpuosRouting(TorchDispatchMode):
    """``with GpuosRouting(executor): ...`` routes eligible ops to ``executor``."""

    def __init__(self, executor: G.Executor, max_elems: int = 1 << 20, min_calls: int = 2):
        super().__init__()
        self.ex = executor
        self.max_elems = max_elems
        self.min_calls = min_calls
        self.calls: Dict[Tuple, int] = {}
        # storage of a routed op's output -> ticket of the routed op that
        # writes it; storage of a routed op's input -> ticket of the last
        # routed op that reads it
        self.pending: Dict[int, int] = {}
        self.readers: Dict[int, int] = {}
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
        elif func in _RED:
            x = args[0]
            dims = args[1] if len(args) > 1 else kwargs.get("dim")
            keepdim = args[2] if len(args) > 2 else kwargs.get("keepdim", False)
            if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or x.dim() < 1:
                return None
            dims = [dims] if isinstance(dims, int) else list(dims or [])
            if len(dims) != 1 or dims[0] not in (-1, x.dim() - 1):
                return None
            name = _RED[func]
            if name == "rowsum":
                dt = args[3] if len(args) > 3 else kwargs.get("dtype")
                if dt != torch.float32:
                    return None
            ts = [x]
            self._keepdim = bool(keepdim)
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
        return self.pending.get(_storage(t))

    def _wait_inputs(self, func, args, kwargs) -> None:
        """An ordinary op about to run: wait for routed producers of the
        storages it touches and, if it may write, for routed readers of
        them."""
        mutable = bool(getattr(getattr(func, "_schema", None), "is_mutable", True))
        for a in list(args) + list(kwargs.values()):
            for t in (a if isinstance(a, (list, tuple)) else [a]):
                if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
                    continue
                st = _storage(t)
                tk = self.pending.pop(st, None)
                if tk is not None:
                    self.ex.sync(tk)
                if mutable:
                    tk = self.readers.pop(st, None)
                    if tk is not None:
                        self.ex.sync(tk)

    def _harvest(self) -> None:
        if len(self.keep) > 256:
            # everything routed so far has completed: no storage needs a
            # wait any more, and none is referenced past this point
            self.ex.sync()
            self.keep.clear()
            self.pending.clear()
            self.readers.clear()

    def drain(self) -> None:
        """Wait for every routed op (call before reading results elsewhere)."""
        self.ex.sync()
        self.pending.clear()
        self.readers.clear()
        self.keep.clear()

    # -- dispatch --------------------------------------------------------------
    def __torch_dispatch__(self, func, types, args=(), kwargs=None):
        kwargs = kwargs or {}
        sel = self._eligible(func, args, kwargs)
        if sel is not None:
            name, ts = sel
            x = ts[0]
            if name in ("rowsum", "rowmax", "rowmin"):
                shape = tuple(x.shape[:-1]) + ((1,) if self._keepdim else ())
                out = torch.empty(shape, dtype=torch.float32 if name == "rowsum" else x.dtype, device=x.device)
            else:
                out = torch.empty_like(x)
            d = G.make_descs(1)
            d["op_id"] = G.OP[name]
            d["dtype"] = G.BF16 if x.dtype == torch.bfloat16 else G.F32
            d["a"] = x.data_ptr()
            if len(ts) > 1:
                d["b"] = ts[1].data_ptr()
            d["out"] = out.data_ptr()
            if name in ("softmax", "rowsum", "rowmax", "rowmin"):
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
                self.pending[_storage(out)] = ticket
                for t_in in ts:
                    self.readers[_storage(t_in)] = ticket
                self.keep.append((ticket, ts + [out]))
                self.routed += 1
                self._harvest()
                return out
            # ring full (current load): the normal launch path
        self.fallback += 1
        self._wait_inputs(func, args, kwargs)
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
