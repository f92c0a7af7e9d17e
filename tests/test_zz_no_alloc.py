"""gpuos_sdpa_noalloc: decode attention that allocates nothing (GPU).

Callers that run beside a resident persistent executor (where cudaFree, or a
cudaMalloc that must grow the heap, waits for an idle device that never
comes) or under a memory budget fixed up front cannot hand the attention a
freshly allocated workspace. This entry point keeps its split-K scratch in a
fixed array inside the library. The test calls it twice in a row through the
C ABI and checks each output against the workspace-based entry point
(gpuos_eager_run with a GPUOS_OP_SDPA descriptor) and against the CPU
oracle's decode attention, within the bf16 rule the parity tests use; it also
checks the size limit.
"""
import numpy as np
import pytest

from tests.gpu_harness import ensure_built, need_gpu
from tests.parity import ulp_bf16

pytestmark = pytest.mark.gpu


def _bf16_f64(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32).__lshift__(16).view(np.float32) \
        .astype(np.float64)


def _oracle_sdpa(q, K, V, lens_list, B, H, D, Lcap, scale):
    """The oracle's decode attention (double, unrounded) on host copies."""
    import torch
    from oracle.interp import lib as orc_lib
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16).copy()  # noqa: E731
    qh, Kh, Vh = bits(q), bits(K), bits(V)
    lens = np.array(lens_list, np.int32)
    out = np.empty(B * H * D, np.float64)
    rc = orc_lib().orc_sdpa(qh.ctypes.data, Kh.ctypes.data, Vh.ctypes.data, lens.ctypes.data, B, H, D, Lcap,
                            float(scale), out.ctypes.data)
    assert rc == 0
    return out


def _workspace_path(G, q, K, V, lens, out, ws, B, H, D, Lcap, Lmax, scale, stream):
    d = G.make_descs(1)
    d["op_id"] = G.OP["sdpa"]
    d["dtype"] = G.BF16
    d["a"], d["b"], d["aux1"], d["aux0"], d["out"], d["aux2"] = (q.data_ptr(), K.data_ptr(), V.data_ptr(),
                                                                lens.data_ptr(), out.data_ptr(), ws.data_ptr())
    d["dims"][0, :6] = (B, H, D, Lcap, Lmax, B * H)
    d["fparam"][0, 0] = scale
    G.eager_run(d, stream)


def test_sdpa_noalloc_matches_workspace_path_on_two_calls():
    torch = need_gpu()
    ensure_built()
    from persistent_micro_dispatch_gb300 import gpuos as G

    B, H, D, Lcap = 3, 32, 128, 2048
    scale = 1.0 / np.sqrt(D)
    g = torch.Generator(device="cuda").manual_seed(123)
    q = torch.randn(B * H * D, device="cuda", generator=g).to(torch.bfloat16)
    K = torch.randn(B * H * Lcap * D, device="cuda", generator=g).to(torch.bfloat16)
    V = torch.randn(B * H * Lcap * D, device="cuda", generator=g).to(torch.bfloat16)
    ws = torch.zeros(G.sdpa_workspace_bytes(B, H, D, Lcap), dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    # two calls in a row with different lengths (one, several and many chunks)
    for lens_list in ([1500, 7, 513], [700, 2048, 1]):
        lens = torch.tensor(lens_list, dtype=torch.int32, device="cuda")
        Lmax = max(lens_list)
        ref = torch.zeros(B * H * D, dtype=torch.bfloat16, device="cuda")
        got = torch.full((B * H * D,), 7.0, dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        _workspace_path(G, q, K, V, lens, ref, ws, B, H, D, Lcap, Lmax, scale, st.cuda_stream)
        rc = G.sdpa_noalloc(q.data_ptr(), K.data_ptr(), V.data_ptr(), lens.data_ptr(), got.data_ptr(),
                            B, H, D, Lcap, Lmax, scale, st.cuda_stream)
        assert rc == G.OK, G.strerror(rc)
        st.synchronize()
        r = _bf16_f64(ref)
        x = _bf16_f64(got)
        # against the workspace-based entry point
        assert np.all(np.abs(x - r) <= np.maximum(2e-2, ulp_bf16(r))), np.abs(x - r).max()
        # against the oracle's exact value
        exact = _oracle_sdpa(q, K, V, lens_list, B, H, D, Lcap, scale)
        assert np.all(np.abs(x - exact) <= np.maximum(2e-2, ulp_bf16(exact))), np.abs(x - exact).max()


def test_sdpa_noalloc_rejects_sizes_beyond_its_scratch():
    torch = need_gpu()
    ensure_built()
    from persistent_micro_dispatch_gb300 import gpuos as G

    buf = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(9, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    # 9 requests x 32 heads > 256
    assert G.sdpa_noalloc(p, p, p, lens.data_ptr(), p, 9, 32, 128, 4096, 64, 0.1, 0) == G.ETOOBIG
    # more than 4096 rows
    assert G.sdpa_noalloc(p, p, p, lens.data_ptr(), p, 1, 32, 128, 8192, 5000, 0.1, 0) == G.ETOOBIG
    assert "fixed scratch" in G.strerror(G.ETOOBIG)
