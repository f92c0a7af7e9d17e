"""Hybrid execution: eligible PyTorch ops routed to the executor (GPU).

The routing mode sends add/mul/ReLU/GELU, softmax and the row reductions
(amax, amin, float32 sum) on small contiguous CUDA tensors to the persistent
executor and leaves everything else (a matmul, a full reduction, an in-place
update) to PyTorch. Every routed result is checked against the CPU oracle
at the parity bar; the in-place update of a tensor a routed op still reads
must not reach that op (write after read)."""
import numpy as np
import pytest

from tests.gpu_harness import ensure_built, need_gpu
from tests.parity import ulp_bf16

pytestmark = pytest.mark.gpu


def _bits(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16).copy()
    return t.contiguous().cpu().numpy().copy()


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class Oracle:
    """The oracle's op definitions on host copies (double, then the output
    dtype's rounding)."""

    def __init__(self):
        from oracle.interp import lib
        self.L = lib()

    def ew(self, op, dt, a, b=None):
        n = a.size
        ex = np.empty(n, np.float64)
        if b is None:
            getattr(self.L, "orc_" + op)(dt, a.ctypes.data, ex.ctypes.data, n)
        else:
            getattr(self.L, "orc_" + op)(dt, a.ctypes.data, b.ctypes.data, ex.ctypes.data, n)
        out = np.empty(n, np.float32 if dt == 0 else np.uint16)
        self.L.orc_store(dt, ex.ctypes.data, out.ctypes.data, n)
        return out, ex

    def softmax(self, x, R, H):
        ex = np.empty(R * H, np.float64)
        self.L.orc_softmax(x.ctypes.data, R, H, ex.ctypes.data)
        return ex

    def rowreduce(self, kind, x, R, H):
        ex = np.empty(R, np.float64)
        self.L.orc_rowreduce(kind, x.ctypes.data, R, H, ex.ctypes.data)
        out = np.empty(R, np.float32 if kind == 0 else np.uint16)
        self.L.orc_store(0 if kind == 0 else 1, ex.ctypes.data, out.ctypes.data, R)
        return out, ex


def test_routed_ops_match_the_oracle_and_mix_with_normal_launches():
    torch = need_gpu()
    ensure_built()
    from persistent_micro_dispatch_gb300 import gpuos as G
    from persistent_micro_dispatch_gb300.route import GpuosRouting
    from workloads.device import warm_torch

    warm_torch()
    # keep the caching allocator supplied before the executor is resident
    pool = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    del pool
    g = torch.Generator(device="cuda").manual_seed(9)
    a, b, c = (torch.randn(4096, device="cuda", generator=g) for _ in range(3))
    s = (torch.randn(8, 1024, device="cuda", generator=g) * 2).to(torch.bfloat16)
    x0 = torch.randn(4096, device="cuda", generator=g)
    # every kernel the routed program launches the normal way is loaded now:
    # with lazy module loading a first launch loads its module, and a module
    # load waits for the device to go idle, which it never does while the
    # executor is resident
    _ = torch.relu(a + b) * c
    _ = torch.nn.functional.gelu(_)
    _ = torch.softmax(s, dim=-1), s.amax(-1), s.amin(-1), s.sum(-1, dtype=torch.float32)
    ref_m = float(a @ b)
    _ = _[0].float().sum()
    xw = x0.clone()
    xw.add_(1.0)
    xs = [x0.clone() for _ in range(4)]
    # (no device-wide synchronize once the executor is resident: it would
    # wait for a kernel that does not end)
    torch.cuda.synchronize()
    # an executor that leaves room on every SM for the ordinary kernels of the
    # same program (4 warps); the default one fills the SMs and ordinary
    # kernels would wait for it
    ex = G.Executor(warps_per_block=4)
    try:
        with GpuosRouting(ex, min_calls=2) as r:
            outs = []
            for k in range(4):
                y = torch.relu(a + b) * c
                gl = torch.nn.functional.gelu(y)
                p = torch.softmax(s, dim=-1)
                mx, mn = s.amax(-1), s.amin(-1)
                sm = s.sum(-1, dtype=torch.float32)
                m = a @ b              # not eligible: PyTorch's own kernel
                tot = gl.sum()         # reads a routed output: waits for it first
                rl = torch.relu(xs[k])  # routed from the second call on...
                xs[k].add_(1.0)         # ...and this in-place update waits for it
                outs.append((y, gl, p, mx, mn, sm, m, tot, rl))
        routed, fallback = r.routed, r.fallback
    finally:
        ex.shutdown()
    torch.cuda.synchronize()
    assert routed >= 24 and fallback >= 12, (routed, fallback)  # calls 2..4 of 9 eligible ops route

    O = Oracle()
    A, B, Cc, X0 = _bits(a), _bits(b), _bits(c), _bits(x0)
    sb = _bits(s).reshape(-1)
    ys, _ = O.ew("add", 0, A, B)
    ys, _ = O.ew("relu", 0, ys)
    y_want, _ = O.ew("mul", 0, ys, Cc)
    _, g_exact = O.ew("gelu", 0, y_want)
    p_exact = O.softmax(sb, 8, 1024)
    mx_want, _ = O.rowreduce(1, sb, 8, 1024)
    mn_want, _ = O.rowreduce(2, sb, 8, 1024)
    _, sm_exact = O.rowreduce(0, sb, 8, 1024)
    rl_want, _ = O.ew("relu", 0, X0)
    for k, (y, gl, p, mx, mn, sm, m, tot, rl) in enumerate(outs):
        assert np.array_equal(_bits(y).view(np.uint32), y_want.view(np.uint32))  # fp32 add, ReLU, mul: exact
        ge = np.abs(_bits(gl).astype(np.float64) - g_exact)
        if k == 0:
            # the first pass is PyTorch's own GELU (routing starts at the
            # second call of a signature): 0.5 x (1 + erf(x / sqrt 2)) loses
            # relative accuracy in the negative tail, where 1 + erf cancels
            assert (ge <= 1e-6 + 1e-4 * np.abs(g_exact)).all(), ge.max()
        else:
            # routed passes: the parity bar (the library's GELU uses erfc)
            bound = 1e-5 * np.maximum(np.abs(g_exact), 1e-3 * np.sqrt(np.mean(g_exact ** 2)))
            assert (ge <= bound).all(), (k, ge.max())
        pe = np.abs(_f64(_bits(p).reshape(-1)) - p_exact)
        assert (pe <= np.maximum(2e-2, ulp_bf16(p_exact))).all(), pe.max()
        assert np.array_equal(_bits(mx), mx_want) and np.array_equal(_bits(mn), mn_want)
        se = np.abs(_bits(sm).astype(np.float64) - sm_exact)
        assert (se <= 2e-2 + 1e-5 * np.abs(sm_exact)).all(), se.max()
        assert np.array_equal(_bits(rl).view(np.uint32), rl_want.view(np.uint32))  # relu of the old x
        assert abs(float(m) - ref_m) <= 1e-3 * max(1.0, abs(ref_m))
        assert abs(float(tot) - float(g_exact.sum())) <= 1e-3 * max(1.0, abs(float(g_exact.sum())))
    for xk in xs:
        assert torch.equal(xk, xw)
