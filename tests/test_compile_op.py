"""Run-time operator compilation (NVRTC) on the host: no GPU needed.

The library prefixes the operator ABI header and compiles for sm_103a as a
relocatable image; the GPU side (linking and running it) is covered by
tests/test_gpu_protocol.py::test_runtime_compiled_op_injection."""
import pytest

from tests.gpu_harness import ensure_built


@pytest.fixture(scope="module")
def G():
    ensure_built()
    from persistent_micro_dispatch_gb300 import gpuos
    return gpuos


def test_header_describes_the_128_byte_descriptor(G):
    h = G.op_header()
    assert "struct gpuos_devdesc" in h and "sizeof(gpuos_devdesc) == 128" in h
    assert "gpuos_op_fn" in h


def test_compile_produces_a_relocatable_elf_image(G):
    src = r'''
    __device__ int op_twice(const gpuos_devdesc *d, uint32_t tile)
    {
        float *o = reinterpret_cast<float *>(d->out);
        const float *a = reinterpret_cast<const float *>(d->a);
        const uint32_t i = tile * 32u + (threadIdx.x & 31u);
        if (i < d->dims[0]) o[i] = 2.0f * a[i];
        return GPUOS_ST_OK;
    }
    __device__ gpuos_op_fn op_twice_ptr = op_twice;
    '''
    try:
        img = G.compile_op(src, "twice.cu")
    except G.GpuosError as e:
        if e.code == G.ECUDA:
            pytest.skip("libnvrtc not available here")
        raise
    assert img[:4] == b"\x7fELF" and len(img) > 1000


def test_compile_error_returns_the_log(G):
    with pytest.raises(G.GpuosError) as ei:
        G.compile_op("__device__ int broken( {", "broken.cu")
    if ei.value.code == G.ECUDA:
        pytest.skip("libnvrtc not available here")
    assert ei.value.code == G.ECOMPILE
    assert "broken.cu" in str(ei.value)
