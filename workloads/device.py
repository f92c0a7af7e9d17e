"""Materialise a ``Stream`` on the GPU and turn its ops into descriptors.

Harness code for tests and the benchmark: buffers become torch device
tensors (raw bytes), ops become ``gpuos_desc`` records pointing into them.
It holds no arithmetic of the ops.
"""
from __future__ import annotations

from typing import List, Optional

import numpy as np
import torch

from persistent_micro_dispatch_gb300 import gpuos as G
from workloads.streams import ESIZE, NPTYPE, Stream


class DeviceStream:
    def __init__(self, stream: Stream, device: str = "cuda"):
        self.s = stream
        self.device = device
        self.bufs: List[torch.Tensor] = []
        for b in stream.buffers:
            if b.data is not None:
                host = torch.from_numpy(np.ascontiguousarray(b.data).view(np.uint8))
                self.bufs.append(host.to(device))
            else:
                self.bufs.append(torch.full((b.nbytes,), b.fill, dtype=torch.uint8, device=device))
        self.ptrs = [t.data_ptr() for t in self.bufs]

    def ptr(self, ref) -> int:
        if ref is None:
            return 0
        return self.ptrs[ref.buf] + ref.off * ESIZE[self.s.buffers[ref.buf].dtype]

    def descs(self, indices: Optional[List[int]] = None, rel_deps: bool = True) -> np.ndarray:
        """gpuos_desc records of the stream's ops (deps as backward distances)."""
        ops = self.s.ops if indices is None else [self.s.ops[i] for i in indices]
        idx = range(len(self.s.ops)) if indices is None else indices
        d = np.zeros(len(ops), dtype=G.DESC_DTYPE)
        for k, (j, o) in enumerate(zip(idx, ops)):
            r = d[k]
            r["op_id"] = G.OP[o.op]
            r["dtype"] = G.DTYPE.get(o.dtype, G.BF16)
            flags = G.FLAG_DEP_REL if rel_deps else 0
            if o.fence:
                flags |= G.FLAG_FENCE
            r["flags"] = flags
            for f in ("a", "b", "out", "aux0", "aux1", "aux2"):
                r[f] = self.ptr(getattr(o, f))
            dims = list(o.dims) + [0] * (6 - len(o.dims))
            r["dims"] = dims
            fp = list(o.fparam) + [0.0] * (2 - len(o.fparam))
            r["fparam"] = fp
            assert len(o.deps) <= 2
            deps = [j - i for i in o.deps] + [0] * (2 - len(o.deps))
            r["dep"] = deps
            r["user"] = j
        return d

    def read(self, ref, n: int, dtype: Optional[str] = None) -> np.ndarray:
        """Copy n elements at ``ref`` back to the host."""
        bdt = self.s.buffers[ref.buf].dtype
        dt = dtype or bdt
        es = ESIZE[dt]
        off = ref.off * ESIZE[bdt]
        raw = self.bufs[ref.buf][off:off + n * es].cpu().numpy()
        return raw.view(NPTYPE[dt])

    def read_buf(self, i: int) -> np.ndarray:
        return self.bufs[i].cpu().numpy().view(NPTYPE[self.s.buffers[i].dtype])


def warm_torch(device: str = "cuda") -> None:
    """Run every torch kernel the harness uses once before the executor starts
    (a kernel first loaded while the persistent executor is resident may wait
    for the device to go idle)."""
    x = torch.full((1024,), 7, dtype=torch.uint8, device=device)
    y = torch.zeros(1024, dtype=torch.uint8, device=device)
    y.copy_(x)
    _ = x[:16].cpu()
    h = torch.from_numpy(np.zeros(64, np.uint8)).to(device)
    torch.cuda.synchronize()
    del x, y, h
