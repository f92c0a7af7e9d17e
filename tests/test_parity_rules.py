"""The comparison rules the GPU parity tests apply (CPU). Candidate results
are held on the host: the oracle's own final buffers, which must pass, and
copies of them with one planted error each, which must fail (bit-exact ops
by one bit, tolerance ops just past their bound) or pass (just inside it)."""
import numpy as np
import pytest

from oracle.interp import Machine
from tests.gpu_harness import final_output_ops
from tests.parity import Report, compare_op
from workloads import streams as S


@pytest.fixture(scope="module")
def state():
    s = S.stream_mixed_small()
    m = Machine(s)
    m.run(keep=range(len(s.ops)))
    return s, m


class HostCandidate:
    """Candidate results on the host (a copy of the oracle's final buffers)."""

    def __init__(self, m):
        self.buf = [b.copy() for b in m.buf]

    def read(self, ref, n):
        return self.buf[ref.buf][ref.off:ref.off + n].copy()


def _compare(s, m, cand, idx):
    rep = Report()
    for j in idx:
        compare_op(rep, s, j, cand.read, m)
    return rep


def _first(s, pred):
    idx = final_output_ops(s, range(len(s.ops)))
    return next(j for j in idx if pred(s.ops[j]))


def _set_bf16(cand, ref, k, value):
    cand.buf[ref.buf][ref.off + k] = S.f32_to_bf16_bits(np.array([value], np.float32))[0]


def test_oracle_results_pass_against_themselves(state):
    s, m = state
    idx = final_output_ops(s, range(len(s.ops)))
    rep = _compare(s, m, HostCandidate(m), idx)
    assert rep.ok(), rep.failures
    assert rep.exact > 0 and rep.tol > 0


def test_bit_exact_op_rejects_one_flipped_bit(state):
    s, m = state
    j = _first(s, lambda o: o.op == "add" and o.dtype == "f32" and o.dims[0] > 0)
    cand = HostCandidate(m)
    o = s.ops[j]
    cand.buf[o.out.buf].view(np.uint32)[o.out.off + 5] ^= 1
    rep = _compare(s, m, cand, [j])
    assert not rep.ok() and "bit-exact" in rep.failures[0]


def test_bf16_tolerance_is_two_hundredths_absolute(state):
    s, m = state
    j = _first(s, lambda o: o.op == "softmax")
    o = s.ops[j]
    r = m.exact[j]["out"]
    k = int(np.argmin(np.abs(r)))  # a small value: its bf16 ulp is far below 2e-2
    for delta, ok in ((0.012, True), (0.03, False)):
        cand = HostCandidate(m)
        _set_bf16(cand, o.out, k, r[k] + delta)
        assert _compare(s, m, cand, [j]).ok() == ok, delta


def test_bf16_tolerance_widens_to_one_ulp_for_large_values():
    # exact values just above grid points of magnitude 5 and 10 (bf16 ulp
    # 2^-5 and 2^-4): the grid neighbour above is more than 2e-2 but at
    # most one ulp away and passes; two steps below fails
    from tests.parity import check_bf16
    o = S.Op("layernorm")
    r = np.array([5.001, -10.002, 0.25])
    ulp = np.array([2.0 ** -5, 2.0 ** -4, 2.0 ** -9])
    near = np.array([5.0 + ulp[0], -10.0 - ulp[1], 0.25 + 0.015])
    far = np.array([5.0 - 2 * ulp[0], -10.0 + 2 * ulp[1], 0.25])
    bits = lambda v: S.f32_to_bf16_bits(v.astype(np.float32))
    assert (np.abs(near - r)[:2] > 2e-2).all() and (np.abs(near - r)[:2] <= ulp[:2]).all()
    rep = Report()
    assert check_bf16(rep, 0, o, bits(near), r)
    assert rep.ulp_branch == 2
    assert not check_bf16(Report(), 0, o, bits(far), r)


def test_fp32_tolerance_is_relative(state):
    s, m = state
    j = _first(s, lambda o: o.op == "gelu" and o.dtype == "f32")
    o = s.ops[j]
    r = m.exact[j]["out"]
    k = int(np.argmax(np.abs(r)))
    for rel, ok in ((5e-6, True), (3e-5, False)):
        cand = HostCandidate(m)
        cand.buf[o.out.buf][o.out.off + k] = np.float32(r[k] * (1 + rel))
        assert _compare(s, m, cand, [j]).ok() == ok, rel


def test_kv_cache_rows_are_compared_bit_exactly(state):
    s, m = state
    j = _first(s, lambda o: o.op == "kv_write" and o.dims[2] == 128)
    o = s.ops[j]
    B, H, D, Lc = o.dims[:4]
    p = int(m.view(o.aux0, B)[0]) - 1
    cand = HostCandidate(m)
    cand.buf[o.out.buf][o.out.off + p * D + 3] ^= 1  # (b=0, h=0) row, one bit of one element
    assert not _compare(s, m, cand, [j]).ok()


def test_row_max_is_exact_and_row_sum_within_bound(state):
    s, m = state
    j = _first(s, lambda o: o.op == "rowmax")
    o = s.ops[j]
    cand = HostCandidate(m)
    cand.buf[o.out.buf][o.out.off] ^= 1
    assert not _compare(s, m, cand, [j]).ok()
    j = _first(s, lambda o: o.op == "rowsum")
    o = s.ops[j]
    r = m.exact[j]["out"]
    for delta, ok in ((0.015, True), (0.05, False)):
        cand = HostCandidate(m)
        cand.buf[o.out.buf][o.out.off] = np.float32(r[0] + delta)
        assert _compare(s, m, cand, [j]).ok() == ok, delta


def _chain_stream():
    """bf16 GELU feeding a bf16 add (the add's input comes from an op whose
    own result is only within tolerance)."""
    rng = np.random.default_rng(21)
    s = S.Stream("chain")
    n = 512
    ix = s.add_buf("x", "bf16", n, S.f32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32)))
    iy = s.add_buf("y", "bf16", n, S.f32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32)))
    ig = s.add_buf("g", "bf16", n)
    iz = s.add_buf("z", "bf16", n)
    s.ops.append(S.Op("gelu", "bf16", a=S.Ref(ix), out=S.Ref(ig), dims=(n,)))
    s.ops.append(S.Op("add", "bf16", a=S.Ref(ig), b=S.Ref(iy), out=S.Ref(iz), dims=(n,), deps=(0,)))
    S.check_hazards(s)
    return s


def test_rounding_carried_along_a_chain_is_allowed_and_errors_are_not():
    s = _chain_stream()
    m = Machine(s)
    m.run(keep=range(len(s.ops)))
    f32 = lambda bits: S.bf16_bits_to_f32(bits)  # noqa: E731
    g_ref, y, z_ref = s.ops[1].a, s.ops[1].b, s.ops[1].out
    # a candidate whose GELU rounded one element the other way (one bf16
    # ulp, within tolerance), and whose add is exact on that input
    exact = m.exact[0]["out"]
    yv = f32(m.buf[y.buf])
    for k in np.argsort(-np.abs(exact)):
        if abs(exact[k]) >= 2.0:  # keep the bf16 ulp <= 2^-7
            continue
        cand = HostCandidate(m)
        g = cand.buf[g_ref.buf]
        gk = float(f32(g[k:k + 1])[0])
        # the grid neighbour on the other side of the exact value (within one ulp)
        g[k] = g[k] + 1 if (exact[k] > gk) == (gk >= 0) else g[k] - 1
        z = S.f32_to_bf16_bits(f32(g) + yv)
        if z[k] != m.buf[z_ref.buf][k]:  # the perturbation reaches the add's result
            break
    assert z[k] != m.buf[z_ref.buf][k]
    assert abs(float(f32(g[k:k + 1])[0]) - exact[k]) <= 2.0 ** -7
    cand.buf[z_ref.buf][:] = z
    rep = _compare(s, m, cand, [0, 1])
    assert rep.ok(), rep.failures
    # the same candidate with a wrong sum on another element
    k2 = (k + 7) % z.size
    cand.buf[z_ref.buf][k2] = S.f32_to_bf16_bits(np.array([float(f32(z[k2:k2 + 1])[0]) + 0.1], np.float32))[0]
    assert not _compare(s, m, cand, [0, 1]).ok()


# ---- widening only from checked producers ------------------------------------------
class HostDS:
    """Host stand-in for a device stream: reads from given final buffers."""

    def __init__(self, s, bufs):
        self.s, self.buf = s, bufs

    def read(self, ref, n, dtype=None):
        v = self.buf[ref.buf]
        if dtype is not None:
            v = v.view(S.NPTYPE[dtype])
        return v[ref.off:ref.off + n].copy()


def _perturbed_chain_candidate():
    """The chain stream with a candidate whose GELU result is one bf16 ulp
    off on one element (within tolerance) and whose add is exact on it."""
    s = _chain_stream()
    m = Machine(s)
    m.run(keep=range(len(s.ops)))
    f32 = S.bf16_bits_to_f32
    g_ref, y, z_ref = s.ops[1].a, s.ops[1].b, s.ops[1].out
    cand = HostCandidate(m)
    g = cand.buf[g_ref.buf]
    exact = m.exact[0]["out"]
    k = int(np.argmin(np.abs(np.abs(exact) - 0.5)))
    gk = float(f32(g[k:k + 1])[0])
    g[k] = g[k] + 1 if (exact[k] > gk) == (gk >= 0) else g[k] - 1
    cand.buf[z_ref.buf][:] = S.f32_to_bf16_bits(f32(g) + f32(m.buf[y.buf]))
    return s, m, cand


def test_widening_needs_the_producer_checked_first():
    s, m, cand = _perturbed_chain_candidate()
    rep = _compare(s, m, cand, [1])  # the consumer alone
    assert not rep.ok() and "widening from an unchecked producer" in rep.failures[0]
    rep = _compare(s, m, cand, [0, 1])  # producer first
    assert rep.ok(), rep.failures


def test_widening_from_a_failed_producer_is_refused():
    s, m, cand = _perturbed_chain_candidate()
    g_ref = s.ops[0].out
    cand.buf[g_ref.buf][3] ^= 0x0100  # the producer itself now fails
    rep = _compare(s, m, cand, [0, 1])
    assert len(rep.failures) >= 2 and any("unchecked producer" in f for f in rep.failures)


def test_widening_from_an_input_rewritten_later_is_refused():
    """op 1 reads g after op 0 wrote it; op 2 rewrites g. At the end g no
    longer holds what op 1 read, so op 1 cannot widen from it."""
    rng = np.random.default_rng(5)
    s = S.Stream("rewrite")
    n = 256
    ix = s.add_buf("x", "bf16", n, S.f32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32)))
    iy = s.add_buf("y", "bf16", n, S.f32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32)))
    ig = s.add_buf("g", "bf16", n)
    iz = s.add_buf("z", "bf16", n)
    s.ops.append(S.Op("gelu", "bf16", a=S.Ref(ix), out=S.Ref(ig), dims=(n,)))
    s.ops.append(S.Op("add", "bf16", a=S.Ref(ig), b=S.Ref(iy), out=S.Ref(iz), dims=(n,), deps=(0,)))
    s.ops.append(S.Op("relu", "bf16", a=S.Ref(iy), out=S.Ref(ig), dims=(n,), deps=(1,)))
    S.check_hazards(s)
    full = Machine(s)
    full.run()
    bufs = [b.copy() for b in full.buf]
    bufs[iy][0] ^= 1  # differs from the oracle on an input op 1 reads...
    bufs[ig][0] ^= 1  # ...and on the rewritten buffer
    from tests.gpu_harness import compare_in_order
    rep, _ = compare_in_order(s, HostDS(s, bufs), targets=[1])
    assert not rep.ok()


def _nudged(s, bufs):
    """The outputs of every bf16 op judged by tolerance, moved by one bf16
    ulp on every fifth element below 2 in magnitude (still within the
    bound): downstream ops then see inputs that differ from the oracle's, as
    the GPU's do, and must widen from their checked producers."""
    tol_ops = ("softmax", "layernorm", "gelu", "sdpa", "vecmat", "rope")
    for o in s.ops:
        if o.op not in tol_ops or o.dtype != "bf16":
            continue
        refs = [(o.a, o.dims[0] * o.dims[1] * o.dims[2]), (o.b, o.dims[0] * o.dims[1] * o.dims[2])] \
            if o.op == "rope" else [(o.out, None)]
        for ref, n in refs:
            if n is None:
                d = o.dims
                if o.op in ("softmax", "layernorm"):
                    n = d[0] * d[1]
                elif o.op == "gelu":
                    n = d[0]
                elif o.op == "vecmat":
                    n = d[1]
                else:
                    n = d[0] * d[1] * d[2]
            v = bufs[ref.buf][ref.off:ref.off + n]
            small = np.abs(S.bf16_bits_to_f32(v)) < 2.0
            idx = np.nonzero(small)[0][::5]
            v[idx] ^= 1
    return bufs


@pytest.mark.parametrize("nudge", [False, True])
@pytest.mark.parametrize("make", [S.stream_mixed_small, lambda: S.stream_c4(n_steps=3),
                                  lambda: S.stream_c5(n_tokens=1, n_layers=2)])
def test_in_order_comparison_passes_the_oracle_own_results(make, nudge):
    """Op by op against the GPU's result as it stood right after the op: the
    oracle's own final buffers, given as the candidate, pass every op (KV
    caches rebuilt from the candidate's k/v rows)."""
    from tests.gpu_harness import compare_in_order
    s = make()
    full = Machine(s)
    full.run()
    bufs = [b.copy() for b in full.buf]
    for i, b in enumerate(s.buffers):
        if b.name.startswith("sdpa_ws"):  # the GPU leaves partials in its scratch
            bufs[i].view(np.uint8)[:] = 0x3C
    if nudge:
        bufs = _nudged(s, bufs)
    rep, _ = compare_in_order(s, HostDS(s, bufs))
    assert rep.ok(), rep.failures
    assert rep.checked >= len([o for o in s.ops if o.op != "nop"]) // 2
