"""The baselines the benchmark times are checked against the oracle too (GPU).

The eager baseline launches the executor's op bodies as ordinary kernels,
one launch per descriptor; the CUDA-graph baseline captures those launches
once and replays them ("GPUOS: A GPU Operating System Primitive for
Transparent Operation Fusion", §3 Q3, Table 2 and "vs CUDA Graphs"). Their
outputs must meet the same parity bar as the executor's.
"""
import numpy as np
import pytest

from tests.gpu_harness import check_kv_copies, compare_in_order, ensure_built, need_gpu
from workloads import streams as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    ensure_built()


def _eager(s, graph: bool):
    import torch
    from persistent_micro_dispatch_gb300 import gpuos as G
    from workloads.device import DeviceStream
    S.check_hazards(s)
    ds = DeviceStream(s)
    descs = ds.descs()
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    if graph:
        # kernel attributes (dynamic shared memory) are set on a first,
        # uncaptured launch of a descriptor of every kind; its outputs are
        # then reset to the stream's initial contents before the capture
        kinds = {}
        for j, o in enumerate(s.ops):
            kinds.setdefault(o.op, j)
        G.eager_run(descs[sorted(kinds.values())], st.cuda_stream, 16384)
        st.synchronize()
        del ds
        ds = DeviceStream(s)
        descs = ds.descs()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            G.eager_run(descs, st.cuda_stream, 16384)
        g.replay()
        torch.cuda.synchronize()
        del g
    else:
        G.eager_run(descs, st.cuda_stream, 16384)
        st.synchronize()
    return ds


@pytest.mark.parametrize("graph", [False, True])
def test_c1_baseline_bit_exact(graph):
    s = S.stream_c1()
    ds = _eager(s, graph)
    rep, _ = compare_in_order(s, ds)
    assert rep.ok(), "\n".join(rep.failures)
    assert rep.exact == len(s.ops)


def test_c2_baseline_small():
    """3,000 variable-shape element-wise descriptors launched eagerly (the
    eager path's own 4,096-element tiles, not the executor's), every output
    against the oracle."""
    s = S.stream_c2(n_desc=3000, pool_elems=1 << 22)
    ds = _eager(s, False)
    rep, _ = compare_in_order(s, ds)
    assert rep.ok(), "\n".join(rep.failures)


@pytest.mark.parametrize("graph", [False, True])
def test_mixed_small_baseline_every_op_kind(graph):
    s = S.stream_mixed_small()
    ds = _eager(s, graph)
    rep, _ = compare_in_order(s, ds)
    assert rep.ok(), "\n".join(rep.failures)
    check_kv_copies(s, ds)


@pytest.mark.parametrize("graph", [False, True])
def test_decode_attention_baseline(graph):
    """Five decode steps at full shapes, replayed as one graph."""
    s = S.stream_c4(n_steps=5)
    ds = _eager(s, graph)
    rep, _ = compare_in_order(s, ds)
    assert rep.ok(), "\n".join(rep.failures)
    check_kv_copies(s, ds)
    assert np.isfinite(rep.max_abs)
