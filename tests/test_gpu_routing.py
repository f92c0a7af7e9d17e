"""Hybrid execution: eligible PyTorch ops routed to the executor (GPU).

The routing mode sends add/mul/ReLU/GELU/softmax on small contiguous CUDA
tensors to the persistent executor and leaves everything else (a matmul, a
reduction) to PyTorch; results must equal PyTorch's own."""
import numpy as np
import pytest

from tests.gpu_harness import ensure_built, need_gpu

pytestmark = pytest.mark.gpu


def test_routed_ops_match_pytorch_and_mix_with_normal_launches():
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
    s = torch.randn(8, 1024, device="cuda", generator=g).to(torch.bfloat16)
    # the references also load every kernel the routed program launches the
    # normal way: with lazy module loading a first launch loads its module,
    # and a module load waits for the device to go idle, which it never does
    # while the executor is resident
    ref_y = torch.relu(a + b) * c
    ref_g = torch.nn.functional.gelu(ref_y)
    ref_p = torch.softmax(s, dim=-1)
    ref_m = float(a @ b)
    ref_tot = float(ref_g.sum())
    torch.cuda.synchronize()
    # an executor that leaves room on every SM for the ordinary kernels of the
    # same program (4 warps: 21.5K of 64K registers, 75 KB of shared memory);
    # the default one fills the SMs and ordinary kernels would wait for it
    ex = G.Executor(warps_per_block=4)
    try:
        with GpuosRouting(ex, min_calls=2) as r:
            outs = []
            for _ in range(4):
                y = torch.relu(a + b) * c
                gl = torch.nn.functional.gelu(y)
                p = torch.softmax(s, dim=-1)
                m = a @ b              # not eligible: PyTorch's own kernel
                tot = gl.sum()         # reads a routed output: waits for it first
                outs.append((y, gl, p, m, tot))
        routed, fallback = r.routed, r.fallback
    finally:
        ex.shutdown()
    torch.cuda.synchronize()
    assert routed >= 12 and fallback >= 8, (routed, fallback)  # calls 2..4 of 5 eligible ops route
    for y, gl, p, m, tot in outs:
        assert torch.equal(y, ref_y)  # add, mul, ReLU: exact in fp32
        assert torch.allclose(gl, ref_g, rtol=1e-5, atol=1e-6)
        assert (p.float() - ref_p.float()).abs().max().item() <= 2e-2
        assert abs(float(m) - ref_m) <= 1e-3 * max(1.0, abs(ref_m))
        assert abs(float(tot) - ref_tot) <= 1e-3 * max(1.0, abs(ref_tot))
