"""The routing filter's host logic (CPU): which aten calls it declines,
before any tensor is handed to the executor. Acceptance needs CUDA tensors
and is covered by the GPU routing test."""
import pytest

torch = pytest.importorskip("torch")

from persistent_micro_dispatch_gb300.route import GpuosRouting  # noqa: E402

aten = torch.ops.aten


@pytest.fixture
def r():
    return GpuosRouting(executor=None, max_elems=1 << 10, min_calls=2)


def test_declines_ops_outside_the_library(r):
    x = torch.ones(8)
    assert r._eligible(aten.sub.Tensor, (x, x), {}) is None
    assert r._eligible(aten.mm.default, (x.view(2, 4), x.view(4, 2)), {}) is None


def test_declines_host_tensors_and_unsupported_forms(r):
    x = torch.ones(8)
    for _ in range(3):  # past min_calls, still declined: not CUDA tensors
        assert r._eligible(aten.add.Tensor, (x, x), {}) is None
    assert r._eligible(aten.add.Tensor, (x, x), {"alpha": 2}) is None          # scaled add
    assert r._eligible(aten.add.Tensor, (x, torch.ones(4)), {}) is None        # broadcast
    assert r._eligible(aten.add.Tensor, (x, x.double()), {}) is None           # mixed dtypes
    assert r._eligible(aten.add.Tensor, (x, 1.0), {}) is None                  # scalar operand
    assert r._eligible(aten.gelu.default, (x,), {"approximate": "tanh"}) is None
    assert r._eligible(aten._softmax.default, (x.view(2, 4), 0, False), {}) is None  # not the last dim
    assert r._eligible(aten._softmax.default, (x.view(2, 4).bfloat16(), -1, True), {}) is None  # half_to_float
    assert r._eligible(aten._softmax.default, (x.view(2, 4), -1, False), {}) is None  # fp32 softmax
    assert r._eligible(aten.relu.default, (torch.ones(8, dtype=torch.int32),), {}) is None


def test_call_counts_are_kept_per_signature(r):
    x = torch.ones(8)
    r._eligible(aten.relu.default, (x,), {})
    r._eligible(aten.relu.default, (x,), {})
    r._eligible(aten.relu.default, (torch.ones(16),), {})
    # host tensors are declined before counting, so nothing is counted
    assert r.calls == {}
