"""Pins for the CPU oracle: each definition checked against something other
than itself (closed forms, textbook constants, special cases, independent
IEEE arithmetic, brute force on tiny inputs). CPU only.

The GPUOS pages ("GPUOS: A GPU Operating System Primitive for Transparent
Operation Fusion", §3 Q2, "Operator library") list the ops but print no
worked example, so the pins come from the mathematics of each op.
"""
import ctypes as C
import json
import math
import os

import numpy as np
import pytest

from oracle.interp import Machine, bf16_round, lib
from workloads import streams as S

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))
P = lambda a: a.ctypes.data  # noqa: E731


def bf(x):
    return S.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def unbf(b):
    return S.bf16_bits_to_f32(b).astype(np.float64)


# ---- number format -----------------------------------------------------------------
def test_bf16_rounding_known_patterns():
    """Hand-derived bf16 patterns: ties to even, subnormals, overflow."""
    for x, bits in GOLD["bf16_patterns"]["value"]:
        assert int(lib().orc_bf16_from_double(x)) == bits, (x, bits)
        assert int(lib().orc_bf16_from_double(-x)) == bits ^ 0x8000


def test_bf16_rounding_matches_integer_rne_on_binary32():
    """Oracle rounding (frexp/nearbyint on doubles) equals the integer
    round-half-even trick on binary32 bit patterns for binary32 inputs."""
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32),
                        (rng.standard_normal(20000) * 1e-38).astype(np.float32),
                        (rng.standard_normal(20000) * 1e30).astype(np.float32)])
    want = S.f32_to_bf16_bits(x)
    got = bf16_round(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_widening_exact():
    for bits in (0x3F80, 0xC020, 0x0001, 0x7F7F, 0x8000):
        assert lib().orc_bf16_to_double(bits) == float(S.bf16_bits_to_f32(np.array([bits], np.uint16))[0])


# ---- element-wise ------------------------------------------------------------------
def _ew(name, dtype, a, b=None):
    n = a.size
    out = np.empty(n, np.float64)
    dt = 0 if dtype == "f32" else 1
    if b is None:
        getattr(lib(), "orc_" + name)(dt, P(a), P(out), n)
    else:
        getattr(lib(), "orc_" + name)(dt, P(a), P(b), P(out), n)
    return out


def _store(dtype, x):
    if dtype == "f32":
        r = np.empty(x.size, np.float32)
        lib().orc_store(0, P(x), P(r), x.size)
        return r
    return bf16_round(x)


@pytest.mark.parametrize("op,npop", [("add", np.add), ("mul", np.multiply)])
def test_add_mul_fp32_equal_ieee_binary32(op, npop):
    """fp32 add/mul after rounding equal the hardware binary32 operation."""
    rng = np.random.default_rng(1)
    a = rng.standard_normal(100000).astype(np.float32)
    b = rng.standard_normal(100000).astype(np.float32)
    a[:6] = [0.0, -0.0, 1e-38, 3e38, 1.0, 2.0 ** -24]
    b[:6] = [-0.0, -0.0, -1e-38, 3e38, 2.0 ** -24, 1.0]
    got = _store("f32", _ew(op, "f32", a, b))
    want = npop(a, b)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("op,npop", [("add", np.add), ("mul", np.multiply)])
def test_add_mul_bf16_equal_binary32_then_rne(op, npop):
    """bf16 add/mul equal binary32 arithmetic followed by integer RNE."""
    rng = np.random.default_rng(2)
    a = bf(rng.standard_normal(100000))
    b = bf(rng.standard_normal(100000))
    got = _store("bf16", _ew(op, "bf16", a, b))
    want = S.f32_to_bf16_bits(npop(S.bf16_bits_to_f32(a), S.bf16_bits_to_f32(b)))
    assert np.array_equal(got, want)


def test_add_mul_identities():
    rng = np.random.default_rng(3)
    a = rng.standard_normal(1000).astype(np.float32)
    z = np.zeros_like(a)
    one = np.ones_like(a)
    assert np.array_equal(_store("f32", _ew("add", "f32", a, z)), a)
    assert np.array_equal(_store("f32", _ew("mul", "f32", a, one)), a)
    assert np.all(_store("f32", _ew("add", "f32", a, -a)) == 0)


def test_relu_special_values():
    a = np.array([-2.0, -0.0, 0.0, 1e-45, 3.5, -1e-45], np.float32)
    got = _store("f32", _ew("relu", "f32", a))
    assert got.view(np.uint32).tolist() == np.array([0, 0, 0, 1e-45, 3.5, 0], np.float32).view(np.uint32).tolist()


def test_gelu_textbook_values():
    """GELU(x) = x Phi(x): Phi(1), Phi(-1), Phi(2) from normal tables."""
    a = np.array([1.0, -1.0, 2.0, 0.0], np.float32)
    got = _ew("gelu", "f32", a)
    assert abs(got[0] - GOLD["phi_1"]["value"]) < 1e-15
    assert abs(got[1] + GOLD["phi_minus_1"]["value"]) < 1e-15
    assert abs(got[2] - 2 * GOLD["phi_2"]["value"]) < 1e-15
    assert got[3] == 0.0


def test_gelu_odd_part_and_limits():
    """GELU(x) - GELU(-x) = x (since Phi(x) + Phi(-x) = 1); GELU(x)->x, ->0."""
    rng = np.random.default_rng(4)
    a = (rng.standard_normal(5000) * 3).astype(np.float32)
    g = _ew("gelu", "f32", a)
    gm = _ew("gelu", "f32", -a)
    assert np.max(np.abs(g - gm - a.astype(np.float64))) < 1e-14
    big = np.array([10.0, 20.0, -10.0, -40.0], np.float32)
    gb = _ew("gelu", "f32", big)
    assert abs(gb[0] - 10.0) < 1e-20 and gb[1] == 20.0
    assert -1e-20 < gb[2] <= 0.0 and gb[3] == 0.0


def test_gelu_negative_tail_relative_accuracy():
    """Deep in the negative tail GELU(x) = x Phi(x) is tiny but not zero; the
    oracle must keep relative accuracy there (1 + erf cancels in double).
    Reference: SciPy's normal CDF (ndtr), an independent library routine."""
    sp = pytest.importorskip("scipy.special")
    a = np.array([-4.0, -6.0, -8.0, -9.0, -10.0, -12.0, -20.0, -30.0], np.float32)
    got = _ew("gelu", "f32", a)
    want = a.astype(np.float64) * sp.ndtr(a.astype(np.float64))
    assert np.all(want < 0)
    assert np.max(np.abs(got / want - 1.0)) < 1e-12


# ---- row ops -----------------------------------------------------------------------
def _softmax(x, R, H):
    out = np.empty(R * H, np.float64)
    lib().orc_softmax(P(x), R, H, P(out))
    return out.reshape(R, H)


def test_softmax_rows_sum_to_one_and_shift_invariance():
    rng = np.random.default_rng(5)
    R, H = 7, 1024
    xf = (rng.standard_normal((R, H)) * 2).astype(np.float32)
    x = bf(xf)
    y = _softmax(x, R, H)
    assert np.max(np.abs(y.sum(1) - 1.0)) < 1e-12
    assert np.all(y > 0)
    # adding a constant that keeps values exactly representable: +8 on values
    # that are multiples of 2^-4 with |x| < 8 stays exact in bf16
    xs = np.round(unbf(x) * 16) / 16
    xs = np.clip(xs, -7.9, 7.9)
    y1 = _softmax(bf(xs), R, H)
    y2 = _softmax(bf(xs + 8.0), R, H)
    assert np.max(np.abs(y1 - y2)) < 1e-15


def test_softmax_closed_forms():
    y = _softmax(bf([0.0, 1.0]), 1, 2)[0]
    assert abs(y[0] - GOLD["logistic_minus_1"]["value"]) < 1e-15
    assert abs(y[1] - GOLD["logistic_1"]["value"]) < 1e-15
    c = _softmax(bf(np.full(4096, 1.5)), 1, 4096)
    assert np.all(c == 1.0 / 4096)


def _ln(x, g, b, R, H, eps):
    out = np.empty(R * H, np.float64)
    lib().orc_layernorm(P(x), P(g), P(b), R, H, eps, P(out))
    return out.reshape(R, H)


def test_layernorm_closed_form_1234():
    got = _ln(bf([1, 2, 3, 4]), bf([1] * 4), bf([0] * 4), 1, 4, 0.0)[0]
    assert np.max(np.abs(got - np.array(GOLD["layernorm_1234"]["value"]))) < 1e-15


def test_layernorm_normalises_and_constant_row_gives_beta():
    rng = np.random.default_rng(6)
    R, H = 5, 2048
    x = bf(rng.standard_normal((R, H)) * 2)
    xd = unbf(x).reshape(R, H)
    y = _ln(x, bf(np.ones(H)), bf(np.zeros(H)), R, H, 1e-5)
    var = xd.var(axis=1)
    assert np.max(np.abs(y.mean(1))) < 1e-12
    assert np.max(np.abs(y.var(1) - var / (var + 1e-5))) < 1e-12
    beta = bf(rng.standard_normal(H) * 0.1)
    yc = _ln(bf(np.full(H, 3.0)), bf(rng.standard_normal(H)), beta, 1, H, 1e-5)[0]
    assert np.array_equal(yc, unbf(beta))
    # gamma scales, beta shifts
    g = bf(np.full(H, 2.0))
    y2 = _ln(x, g, bf(np.full(H, 0.5)), R, H, 1e-5)
    assert np.max(np.abs(y2 - (2 * y + 0.5))) < 1e-12


def test_row_reductions_against_fsum_and_builtins():
    rng = np.random.default_rng(7)
    R, H = 9, 4096
    x = bf(rng.standard_normal((R, H)) * 2)
    xd = unbf(x).reshape(R, H)
    for kind, f in ((0, math.fsum), (1, max), (2, min)):
        out = np.empty(R, np.float64)
        lib().orc_rowreduce(kind, P(x), R, H, P(out))
        for r in range(R):
            want = f(xd[r].tolist())
            if kind == 0:
                assert abs(out[r] - want) <= 1e-12 * max(1.0, abs(want))
            else:
                assert out[r] == want


# ---- RoPE --------------------------------------------------------------------------
def _rope(q, k, lens, B, H, D, theta):
    qo = np.empty(B * H * D, np.float64)
    ko = np.empty(B * H * D, np.float64)
    st = lib().orc_rope(P(q), P(k), P(lens), B, H, D, theta, P(qo), P(ko))
    return st, qo.reshape(B, H, D), ko.reshape(B, H, D)


def test_rope_position_zero_is_identity_and_norms_preserved():
    rng = np.random.default_rng(8)
    B, H, D = 3, 4, 128
    q = bf(rng.standard_normal(B * H * D))
    k = bf(rng.standard_normal(B * H * D))
    st, qo, ko = _rope(q, k, np.array([1, 1, 1], np.int32), B, H, D, 10000.0)
    assert st == 0
    assert np.array_equal(qo.reshape(-1), unbf(q)) and np.array_equal(ko.reshape(-1), unbf(k))
    lens = np.array([5, 777, 4096], np.int32)
    st, qo, ko = _rope(q, k, lens, B, H, D, 10000.0)
    qd = unbf(q).reshape(B, H, D)
    n_in = qd[..., :64] ** 2 + qd[..., 64:] ** 2
    n_out = qo[..., :64] ** 2 + qo[..., 64:] ** 2
    assert np.max(np.abs(n_in - n_out)) < 1e-12


def test_rope_unit_vectors_pairing_and_angle():
    """A unit vector on dim i only mixes with dim i+D/2, rotated by
    p * theta^(-2i/D); at p = 1, i = 0 the angle is exactly 1 rad."""
    B, H, D = 1, 1, 128
    for i, p in ((0, 1), (3, 100), (63, 4095)):
        x = np.zeros(D, np.float32)
        x[i] = 1.0
        st, qo, _ = _rope(bf(x), bf(x), np.array([p + 1], np.int32), B, H, D, 10000.0)
        y = qo[0, 0]
        others = np.delete(y, [i, i + 64])
        assert np.all(others == 0)
        phi = p * math.exp(-2.0 * i / D * math.log(10000.0))
        assert abs(y[i] - math.cos(phi)) < 1e-12 and abs(y[i + 64] - math.sin(phi)) < 1e-12
    x = np.zeros(D, np.float32)
    x[0] = 1.0
    _, qo, _ = _rope(bf(x), bf(x), np.array([2], np.int32), 1, 1, D, 10000.0)
    assert abs(qo[0, 0, 0] - GOLD["cos_1"]["value"]) < 1e-15
    assert abs(qo[0, 0, 64] - GOLD["sin_1"]["value"]) < 1e-15


def test_rope_composes_positions():
    """Rotating by p1 then by p2 equals rotating by p1 + p2 (on exact values:
    the second rotation is applied in double to the first's exact output)."""
    rng = np.random.default_rng(9)
    D = 128
    x = bf(rng.standard_normal(D))
    _, y1, _ = _rope(x, x, np.array([11], np.int32), 1, 1, D, 10000.0)  # p = 10
    _, y12, _ = _rope(x, x, np.array([31], np.int32), 1, 1, D, 10000.0)  # p = 30
    i = np.arange(64)
    phi2 = 20 * np.exp(-2.0 * i / D * np.log(10000.0))
    a, b = y1[0, 0, :64], y1[0, 0, 64:]
    r0 = a * np.cos(phi2) - b * np.sin(phi2)
    r1 = b * np.cos(phi2) + a * np.sin(phi2)
    assert np.max(np.abs(r0 - y12[0, 0, :64])) < 1e-12
    assert np.max(np.abs(r1 - y12[0, 0, 64:])) < 1e-12


# ---- KV write ----------------------------------------------------------------------
def test_kv_write_places_rows_and_leaves_others():
    rng = np.random.default_rng(10)
    B, H, D, Lc = 3, 2, 8, 16
    k = bf(rng.standard_normal(B * H * D))
    v = bf(rng.standard_normal(B * H * D))
    Kc = bf(rng.standard_normal(B * H * Lc * D))
    Vc = bf(rng.standard_normal(B * H * Lc * D))
    K0, V0 = Kc.copy(), Vc.copy()
    lens = np.array([1, 9, 16], np.int32)
    assert lib().orc_kv_write(P(k), P(v), P(lens), B, H, D, Lc, P(Kc), P(Vc)) == 0
    K4, V4 = Kc.reshape(B, H, Lc, D), Vc.reshape(B, H, Lc, D)
    mask = np.zeros((B, H, Lc, D), bool)
    for b in range(B):
        p = lens[b] - 1
        assert np.array_equal(K4[b, :, p], k.reshape(B, H, D)[b])
        assert np.array_equal(V4[b, :, p], v.reshape(B, H, D)[b])
        mask[b, :, p] = True
    assert np.array_equal(K4[~mask], K0.reshape(B, H, Lc, D)[~mask])
    assert np.array_equal(V4[~mask], V0.reshape(B, H, Lc, D)[~mask])
    bad = np.array([1, 17, 3], np.int32)
    assert lib().orc_kv_write(P(k), P(v), P(bad), B, H, D, Lc, P(Kc), P(Vc)) == -1


# ---- SDPA --------------------------------------------------------------------------
def _sdpa(q, K, V, lens, B, H, D, Lc, scale):
    out = np.empty(B * H * D, np.float64)
    st = lib().orc_sdpa(P(q), P(K), P(V), P(lens), B, H, D, Lc, scale, P(out))
    return st, out.reshape(B, H, D)


def test_sdpa_length_one_returns_first_value_row():
    rng = np.random.default_rng(12)
    B, H, D, Lc = 2, 3, 16, 8
    q, K, V = (bf(rng.standard_normal(n)) for n in (B * H * D, B * H * Lc * D, B * H * Lc * D))
    st, o = _sdpa(q, K, V, np.array([1, 1], np.int32), B, H, D, Lc, 0.25)
    assert st == 0
    assert np.array_equal(o, unbf(V).reshape(B, H, Lc, D)[:, :, 0])


def test_sdpa_identical_keys_average_values():
    rng = np.random.default_rng(13)
    B, H, D, Lc, L = 1, 2, 8, 8, 6
    q = bf(rng.standard_normal(B * H * D))
    krow = bf(rng.standard_normal(D))
    K = np.tile(krow, B * H * Lc)
    V = bf(rng.standard_normal(B * H * Lc * D))
    _, o = _sdpa(q, K, V, np.array([L], np.int32), B, H, D, Lc, 0.3)
    Vd = unbf(V).reshape(B, H, Lc, D)
    assert np.max(np.abs(o - Vd[:, :, :L].mean(axis=2))) < 1e-14


def test_sdpa_two_key_closed_form():
    """q.K0 = 0 and q.K1 = 1 with scale 1: weights 1/(1+e) and e/(1+e)."""
    D = 4
    q = bf([1, 0, 0, 0])
    K = bf([0, 1, 0, 0, 1, 0, 0, 0])
    V = bf([1, 2, 3, 4, -1, 0, 2, 8])
    _, o = _sdpa(q, K, V, np.array([2], np.int32), 1, 1, D, 2, 1.0)
    w0, w1 = GOLD["logistic_minus_1"]["value"], GOLD["logistic_1"]["value"]
    want = w0 * np.array([1, 2, 3, 4.0]) + w1 * np.array([-1, 0, 2, 8.0])
    assert np.max(np.abs(o[0, 0] - want)) < 1e-14


def test_sdpa_brute_force_tiny_heads():
    """B=1, H=2, D=4, L<=8 against an explicit double loop with math.exp."""
    rng = np.random.default_rng(14)
    B, H, D, Lc = 1, 2, 4, 8
    for L in range(1, 9):
        q, K, V = (bf(rng.standard_normal(n)) for n in (B * H * D, B * H * Lc * D, B * H * Lc * D))
        _, o = _sdpa(q, K, V, np.array([L], np.int32), B, H, D, Lc, 0.5)
        qd, Kd, Vd = unbf(q).reshape(H, D), unbf(K).reshape(H, Lc, D), unbf(V).reshape(H, Lc, D)
        for h in range(H):
            s = [0.5 * sum(qd[h, d] * Kd[h, t, d] for d in range(D)) for t in range(L)]
            w = [math.exp(x - max(s)) for x in s]
            z = math.fsum(w)
            for d in range(D):
                ref = math.fsum(w[t] * Vd[h, t, d] for t in range(L)) / z
                assert abs(o[0, h, d] - ref) < 1e-13


def test_sdpa_rejects_bad_length():
    q = bf(np.zeros(4))
    K = bf(np.zeros(8))
    assert _sdpa(q, K, K, np.array([3], np.int32), 1, 1, 4, 2, 1.0)[0] == -1
    assert _sdpa(q, K, K, np.array([0], np.int32), 1, 1, 4, 2, 1.0)[0] == -1


# ---- vecmat ------------------------------------------------------------------------
def test_vecmat_identity_and_integer_exact():
    rng = np.random.default_rng(15)
    K = N = 64
    x = bf(rng.standard_normal(K))
    eye = bf(np.eye(K))  # keep the operands alive across the C call
    out = np.empty(N, np.float64)
    lib().orc_vecmat(P(x), P(eye), K, N, P(out))
    assert np.array_equal(out, unbf(x))
    K, N = 37, 19
    xi = rng.integers(-8, 9, K)
    Wi = rng.integers(-8, 9, (K, N))
    xb, Wb = bf(xi), bf(Wi)
    out = np.empty(N, np.float64)
    lib().orc_vecmat(P(xb), P(Wb), K, N, P(out))
    want = [sum(int(xi[k]) * int(Wi[k, n]) for k in range(K)) for n in range(N)]
    assert out.tolist() == [float(w) for w in want]


# ---- interpreter -------------------------------------------------------------------
def test_interpreter_sequential_semantics_on_a_chain():
    """A chained element-wise stream: each consumer sees its producer's
    rounded output; the closure runner reproduces the full run."""
    s = S.stream_elementwise("t", 200, 256, 4096, 0.5, 1 << 16, seed=21)
    S.check_hazards(s)
    full = Machine(s)
    full.run()
    chained = [j for j, o in enumerate(s.ops) if o.deps]
    assert len(chained) > 50
    for j in chained[:20]:
        o, p = s.ops[j], s.ops[s.ops[j].deps[0]]
        assert o.a.buf == p.out.buf and o.a.off == p.out.off
    part = Machine(s)
    targets = chained[-5:]
    part.run_closure(targets)
    for j in targets:
        o = s.ops[j]
        n = o.dims[0]
        assert np.array_equal(part.view(o.out, n), full.view(o.out, n))


def test_hazard_checker_rejects_missing_dependency():
    s = S.stream_elementwise("t", 50, 256, 1024, 0.5, 1 << 14, seed=22)
    S.check_hazards(s)
    j = next(j for j, o in enumerate(s.ops) if o.deps)
    s.ops[j].deps = ()
    with pytest.raises(AssertionError):
        S.check_hazards(s)


def test_c4_and_c5_streams_are_hazard_free():
    S.check_hazards(S.stream_c4(n_steps=6, B_max=2, Lcap=256, L_lo=8))
    S.check_hazards(S.stream_c5(n_tokens=2, n_layers=2, hidden=256, H=2, D=128, Lcap=128, vm=64, L_lo=16))
