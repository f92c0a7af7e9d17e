"""The seeded synthetic streams follow the stated input recipe (CPU): op
mixes, size distributions, chaining, lengths, dependencies, seeds and pool
sizes, and every stream's declared dependencies order all its conflicting
accesses."""
import inspect
import math

import numpy as np
import pytest

from workloads import streams as S

L2_BYTES = 129 * 10**6


def _ops(s, name):
    return [o for o in s.ops if o.op == name]


def test_seeds_and_pool_sizes_of_the_full_streams():
    seeds = {k: inspect.signature(f).parameters["seed"].default for k, f in S.STREAMS.items()}
    assert seeds == {"c1": 1, "c2": 2, "c3": 3, "c4": 4, "c5": 5, "c2l": 6}
    for k, esize in (("c2", 4), ("c2l", 4), ("c3", 2)):
        pool = inspect.signature(S.STREAMS[k]).parameters["pool_elems"].default
        assert pool * esize > 2 * L2_BYTES, k  # inputs larger than L2


def test_c1_recipe():
    s = S.stream_c1()
    assert len(s.ops) == 1000
    assert {o.op for o in s.ops} == {"add", "mul", "relu"}
    assert all(o.dtype == "f32" and o.dims == (4096,) and not o.deps for o in s.ops)
    S.check_hazards(s)


def test_c2_recipe():
    s = S.stream_c2(n_desc=20000, pool_elems=1 << 22)
    n = len(s.ops)
    kinds = {k: len(_ops(s, k)) / n for k in ("add", "mul", "relu", "gelu")}
    assert sum(kinds.values()) == 1.0 and all(abs(v - 0.25) < 0.02 for v in kinds.values())
    chained = [i for i, o in enumerate(s.ops) if o.deps]
    assert abs(len(chained) / n - 0.30) < 0.015
    for i in chained:
        o, p = s.ops[i], s.ops[i - 1]
        assert o.deps == (i - 1,) and o.a == p.out and o.dtype == p.dtype and o.dims[0] <= p.dims[0]
    free = [o for o in s.ops if not o.deps]
    sizes = np.array([o.dims[0] for o in free])
    assert sizes.min() >= 256 and sizes.max() <= 65536
    # log-uniform: ln n uniform on [ln 256, ln 65536]
    ln = np.log(sizes)
    assert abs(ln.mean() - (math.log(256) + math.log(65536)) / 2) < 0.05
    assert abs(ln.std() - (math.log(65536) - math.log(256)) / math.sqrt(12)) < 0.05
    assert abs(np.mean([o.dtype == "bf16" for o in free]) - 0.5) < 0.02
    assert all(o.a.off % 256 == 0 and (o.b is None or o.b.off % 256 == 0) for o in free)
    S.check_hazards(s)


def test_c2l_recipe():
    s = S.stream_c2l(n_desc=500, pool_elems=1 << 21)
    sizes = np.array([o.dims[0] for o in s.ops])
    assert sizes.min() >= 65536 and sizes.max() <= 1 << 20
    assert not any(o.deps for o in s.ops)
    S.check_hazards(s)


def test_c3_recipe():
    s = S.stream_c3(n_desc=5000, pool_elems=1 << 22)
    n = len(s.ops)
    for k in ("softmax", "layernorm", "rowsum", "rowmax", "rowmin"):
        assert abs(len(_ops(s, k)) / n - 0.2) < 0.02, k
    R = np.array([o.dims[0] for o in s.ops])
    H = np.array([o.dims[1] for o in s.ops])
    assert R.min() == 1 and R.max() == 64 and set(H.tolist()) == {1024, 2048, 4096}
    for o in _ops(s, "layernorm"):
        assert o.b is not None and o.aux0 is not None and o.fparam == (1e-5,)
    S.check_hazards(s)


def test_c4_recipe():
    d = {k: v.default for k, v in inspect.signature(S.stream_c4).parameters.items()}
    assert (d["n_steps"], d["B_max"], d["H"], d["D"], d["Lcap"], d["L_lo"]) == (2000, 8, 32, 128, 4096, 128)
    steps = 200
    s = S.stream_c4(n_steps=steps, Lcap=1024)  # a shorter cache keeps the test quick
    assert [o.op for o in s.ops] == ["rope", "kv_write", "sdpa"] * steps
    lens = s.buffers[s.buf_index("lens")].data
    assert lens.min() >= 128 and lens.max() <= 1024
    for t in range(steps):
        r, kv, at = s.ops[3 * t:3 * t + 3]
        B = r.dims[0]
        assert 1 <= B <= 8 and r.dims[1:] == (32, 128)
        assert kv.deps == ((3 * t,) if t == 0 else (3 * t, 3 * t - 1))
        assert at.deps == (3 * t + 1,)
        assert at.dims[4] == int(lens[r.aux0.off:r.aux0.off + B].max())
        assert at.fparam[0] == pytest.approx(1 / math.sqrt(128))
    S.check_hazards(s)


def test_c5_recipe():
    d = {k: v.default for k, v in inspect.signature(S.stream_c5).parameters.items()}
    assert (d["n_layers"], d["hidden"], d["Lcap"], d["vm"], d["L_lo"], d["walk"]) == (32, 4096, 4096, 1024, 256, 32)
    tokens, layers = 40, 3  # fewer layers and a shorter cache keep the test quick
    s = S.stream_c5(n_tokens=tokens, n_layers=layers, Lcap=1024)
    chain = ["layernorm", "vecmat", "rope", "kv_write", "sdpa", "gelu", "add"]
    assert [o.op for o in s.ops] == chain * layers * tokens
    for j, o in enumerate(s.ops):
        assert o.deps == ((j - 1,) if j else ())
    lens = s.buffers[s.buf_index("lens")].data.astype(int)
    assert lens.min() >= 256 and lens.max() <= 1024
    assert np.abs(np.diff(lens)).max() <= 32 and np.abs(np.diff(lens)).max() > 0
    for o in _ops(s, "sdpa"):
        assert o.dims[4] == lens[o.aux0.off]  # attention covers the token's length
    S.check_hazards(s)


def test_hazard_checker_rejects_an_undeclared_conflict():
    s = S.stream_c2(n_desc=2000, pool_elems=1 << 20)
    i = next(i for i, o in enumerate(s.ops) if o.deps)
    s.ops[i].deps = ()
    with pytest.raises(AssertionError):
        S.check_hazards(s)
