"""Parity of the persistent executor with the CPU oracle on the five seeded
streams (GPU). Small cases compare every op; full-size cases compare sampled
ops, recomputed by the oracle from the same seeded inputs.

Bar: bit-exact for copy/order/exact-IEEE ops, 1e-5 relative for fp32,
2e-2 absolute (or one bf16 ulp of the exact value) for bf16 outputs.
"""
import numpy as np
import pytest

from oracle.interp import Machine
from tests.gpu_harness import (check_canaries, check_kv_copies, compare_in_order, compare_stream, ensure_built,
                               final_output_ops, need_gpu, run_executor, sample)
from workloads import streams as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    ensure_built()


def _run_and_compare(s, check=None, sample_k=None, cfg=None, skip=None, seed=0):
    """Run the stream on the executor, then compare with the oracle op by op
    (each op against the GPU's result as it stood right after it). check /
    sample_k pick target ops (the oracle then applies them and what they
    depend on, and checks every comparable op it applies)."""
    from workloads.device import DeviceStream
    S.check_hazards(s)
    ds = DeviceStream(s)
    descs = ds.descs()
    st, hist = run_executor(ds, descs, **(cfg or {}))
    assert np.all(hist["status"] == 0), f"device status: {np.unique(hist['status'])}"
    assert st["completed"] == len(s.ops)
    targets = check
    if sample_k is not None:
        targets = sample(final_output_ops(s, range(len(s.ops))), sample_k, seed)
    rep, mach = compare_in_order(s, ds, targets=targets, skip=skip or ())
    print(f"{s.name}: {rep.summary()} stats={st}")
    assert rep.ok(), "\n".join(rep.failures)
    return s, ds, rep, st, hist


def test_c1_smallest_stream_bit_exact():
    """1,000 fp32 add/mul/ReLU on 4,096-element tensors: every output bit-exact."""
    s, ds, rep, st, hist = _run_and_compare(S.stream_c1())
    assert rep.exact == len(s.ops)
    check_canaries(s, ds)


@pytest.mark.parametrize("stage_bytes", [16384, 0])
def test_c2_variable_elementwise_small(stage_bytes):
    """3,000 descriptors over {add, mul, ReLU, GELU} x {fp32, bf16}, 30 % chained,
    with shared-memory (TMA bulk copy) staging and with the register path."""
    s, ds, rep, st, hist = _run_and_compare(S.stream_c2(n_desc=3000, pool_elems=1 << 22),
                                            cfg=dict(stage_bytes=stage_bytes))
    check_canaries(s, ds)


@pytest.mark.parametrize("stage_bytes", [16384, 0])
def test_c2l_large_ops_small(stage_bytes):
    s, ds, rep, st, hist = _run_and_compare(S.stream_c2l(n_desc=40, pool_elems=1 << 23),
                                            cfg=dict(stage_bytes=stage_bytes))
    check_canaries(s, ds)


def test_c3_row_ops_small():
    s, ds, rep, st, hist = _run_and_compare(S.stream_c3(n_desc=1500, pool_elems=1 << 22))
    check_canaries(s, ds, names=("out_bf16", "out_f32"))


def test_c4_decode_small_and_kv_copy_bit_exact():
    """20 decode steps at full shapes (B<=8, 32x128, caches of 4,096 rows)."""
    s, ds, rep, st, hist = _run_and_compare(S.stream_c4(n_steps=20))
    check_kv_copies(s, ds)


@pytest.mark.parametrize("stage_bytes", [16384, 0])
def test_c4_decode_wide_length_spread(stage_bytes):
    """Decode steps whose requests' lengths run from 1 to 4,096 rows in one
    op (the attention body shortens its chunks from the lengths, so a step
    mixes single-row requests, requests of one chunk and requests of many),
    staged and register paths; every output against the oracle."""
    s = S.stream_c4(n_steps=16, L_lo=1, seed=41)
    lens = s.buffers[s.buf_index("lens")].data
    for o in s.ops:
        if o.op == "sdpa" and o.dims[0] >= 2:
            lens[o.aux0.off] = 1        # a one-row request beside long ones
            lens[o.aux0.off + 1] = 33   # and one just past a 32-row chunk
    s, ds, rep, st, hist = _run_and_compare(s, cfg=dict(stage_bytes=stage_bytes))
    check_kv_copies(s, ds)


@pytest.mark.parametrize("stage_bytes", [16384, 0])
def test_elementwise_sizes_around_tile_boundaries(stage_bytes):
    """add/mul/ReLU/GELU in fp32 and bf16 at sizes around the tile sizes
    (1,024 for a GELU with a dependency, 16,384 and 32,768 elements, and
    their multiples), aligned and at odd element offsets (the scalar path),
    some with a dependency (a GELU then keeps its finer tiles); every output
    against the oracle."""
    rng = np.random.default_rng(45)
    s = S.Stream("ew_bounds", meta=dict(seed=45))
    n_pool = 1 << 20
    pf = s.add_buf("pool_f32", "f32", n_pool, S._pool(rng, n_pool, "f32"))
    pb = s.add_buf("pool_bf16", "bf16", n_pool, S._pool(rng, n_pool, "bf16"))
    sizes = [1, 255, 256, 257, 1023, 1025, 2049, 16383, 16384, 16385, 32767, 32768, 32769, 65539, 262147]
    total = {"f32": 0, "bf16": 0}
    plan = []
    for dt in ("f32", "bf16"):
        for op in ("add", "mul", "relu", "gelu"):
            for k, n in enumerate(sizes):
                off = 0 if k % 3 else 1  # every third at an odd element offset
                plan.append((dt, op, n, off, k % 4 == 1))
                total[dt] += n + 64
    of = s.add_buf("out_f32", "f32", total["f32"])
    ob = s.add_buf("out_bf16", "bf16", total["bf16"])
    top = {"f32": 0, "bf16": 0}
    for dt, op, n, off, chained in plan:
        src, dst = (pf, of) if dt == "f32" else (pb, ob)
        a_off = int(rng.integers(0, n_pool - n - 2)) // 256 * 256 + off
        b_off = int(rng.integers(0, n_pool - n - 2)) // 256 * 256
        o = top[dt] + off
        top[dt] += n + 64
        deps = (len(s.ops) - 1,) if chained and s.ops else ()
        bref = S.Ref(src, b_off) if op in ("add", "mul") else None
        s.ops.append(S.Op(op, dt, a=S.Ref(src, a_off), b=bref, out=S.Ref(dst, o), dims=(n,), deps=deps))
    _run_and_compare(s, cfg=dict(stage_bytes=stage_bytes))


def test_row_ops_many_rows():
    """Row ops of thousands of rows (about a thousand helper warps each,
    every helper taking further rows from the descriptor's counter and
    copying the next one while it works on the current one), including a
    LayerNorm whose gamma and beta stay in the staging buffer; every output
    against the oracle."""
    rng = np.random.default_rng(44)
    s = S.Stream("rows_many", meta=dict(seed=44))
    x1 = s.add_buf("x1", "bf16", 4096 * 1024, S._pool(rng, 4096 * 1024, "bf16", std=2.0))
    x2 = s.add_buf("x2", "bf16", 2048 * 2048, S._pool(rng, 2048 * 2048, "bf16", std=2.0))
    g = s.add_buf("gamma", "bf16", 2048, S._pool(rng, 2048, "bf16", std=0.1, mean=1.0))
    b = s.add_buf("beta", "bf16", 2048, S._pool(rng, 2048, "bf16", std=0.1))
    ob = s.add_buf("out_bf16", "bf16", 4096 * 1024 + 2048 * 2048 + 8192)
    of = s.add_buf("out_f32", "f32", 4096)
    s.ops.append(S.Op("softmax", "bf16", a=S.Ref(x1, 0), out=S.Ref(ob, 0), dims=(4096, 1024)))
    s.ops.append(S.Op("layernorm", "bf16", a=S.Ref(x2, 0), b=S.Ref(g, 0), aux0=S.Ref(b, 0),
                      out=S.Ref(ob, 4096 * 1024), dims=(2048, 2048), fparam=(1e-5,)))
    s.ops.append(S.Op("rowmax", "bf16", a=S.Ref(x1, 0), out=S.Ref(ob, 4096 * 1024 + 2048 * 2048), dims=(4096, 1024)))
    s.ops.append(S.Op("rowsum", "bf16", a=S.Ref(x1, 0), out=S.Ref(of, 0), dims=(4096, 1024)))
    _run_and_compare(s)


def test_decode_attention_many_requests():
    """One attention op over 40 requests of one head (more than 32, so the
    op body's prefix over the requests' chunk counts runs in two rounds),
    lengths from 1 to 1,024 rows; every output against the oracle."""
    import math
    rng = np.random.default_rng(43)
    s = S.Stream("sdpa_many", meta=dict(seed=43))
    B, H, D, Lc = 40, 1, 128, 1024
    iq = s.add_buf("q", "bf16", B * H * D, S._pool(rng, B * H * D, "bf16"))
    iK = s.add_buf("Kc", "bf16", B * H * Lc * D, S._pool(rng, B * H * Lc * D, "bf16"))
    iV = s.add_buf("Vc", "bf16", B * H * Lc * D, S._pool(rng, B * H * Lc * D, "bf16"))
    lens = rng.integers(1, Lc + 1, size=B).astype(np.int32)
    lens[0], lens[1], lens[33] = 1, Lc, 33
    il = s.add_buf("lens", "i32", B, lens)
    io = s.add_buf("out_bf16", "bf16", B * H * D)
    ws = s.add_buf("sdpa_ws", "u8", S.sdpa_workspace_bytes(B, H, D, Lc), fill=0)
    s.ops.append(S.Op("sdpa", "bf16", a=S.Ref(iq, 0), b=S.Ref(iK, 0), aux1=S.Ref(iV, 0), aux0=S.Ref(il, 0),
                      out=S.Ref(io, 0), aux2=S.Ref(ws, 0), dims=(B, H, D, Lc, int(lens.max()), B * H),
                      fparam=(1.0 / math.sqrt(D),)))
    _run_and_compare(s)


@pytest.mark.parametrize("stage_bytes", [16384, 0])
def test_mixed_small_every_op_kind(stage_bytes):
    """Every op kind at small, ragged sizes (tails, 1-row and 8-column tiles,
    ragged head groups, multi-chunk attention), staged and register paths."""
    s, ds, rep, st, hist = _run_and_compare(S.stream_mixed_small(), cfg=dict(stage_bytes=stage_bytes))
    check_kv_copies(s, ds)


def test_c5_mixed_pipeline_small():
    """3 tokens of the 32-layer synthetic decoder at hidden 4,096."""
    s, ds, rep, st, hist = _run_and_compare(S.stream_c5(n_tokens=3))
    check_kv_copies(s, ds)


def test_gelu_fp32_error_bound_sweep():
    """The GPU's GELU evaluates erfc by the Numerical Recipes Chebyshev fit
    (fractional error < 1.2e-7) in fp32. Over x in [-12, 12] (and special
    values) its relative error against the oracle's double GELU must stay
    within the fit's bound plus fp32 rounding, which grows with the
    conditioning of erfc(|x|/sqrt 2), about x^2 ulps of the argument."""
    from workloads.device import DeviceStream
    n = (1 << 20) + 37
    x = np.linspace(-12.0, 12.0, n - 37).astype(np.float32)
    special = np.array([0.0, -0.0, 1e-30, -1e-30, 1e-7, -1e-7, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0, 3.0, -3.0,
                        0.4769363, -0.4769363, 5.0, -5.0, 8.0, -8.0, 10.0, -10.0, 12.0, -12.0, 0.70710678,
                        -0.70710678, 1.4142135, -1.4142135, 2.5, -2.5, 6.0, -6.0, 4.0, -4.0, 1.5, -1.5,
                        3.5], np.float32)
    xs = np.concatenate([x, special])
    s = S.Stream("gelu_sweep")
    ia = s.add_buf("x", "f32", n, xs)
    io = s.add_buf("out", "f32", n)
    s.ops.append(S.Op("gelu", "f32", a=S.Ref(ia, 0), out=S.Ref(io, 0), dims=(n,)))
    ds = DeviceStream(s)
    st, hist = run_executor(ds, ds.descs())
    assert np.all(hist["status"] == 0)
    got = ds.read(S.Ref(io, 0), n).astype(np.float64)
    mach = Machine(s)
    mach.run(keep=[0])
    ref = mach.exact[0]["out"]
    xd = xs.astype(np.float64)
    bound = (6e-7 + 1.2e-7 * xd * xd) * np.abs(ref) + 1e-37
    err = np.abs(got - ref)
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, [(float(xd[i]), float(got[i]), float(ref[i])) for i in bad[:5]]
    # and the parity rule the streams use
    rep = compare_stream(s, ds, mach, [0])
    assert rep.ok(), "\n".join(rep.failures)


@pytest.mark.slow
def test_c2_full_sampled():
    """Full C2 (100,000 descriptors); 400 sampled ops recomputed by the oracle."""
    _run_and_compare(S.stream_c2(), sample_k=400, seed=2)


@pytest.mark.slow
def test_c2l_full_sampled():
    _run_and_compare(S.stream_c2l(), sample_k=60, seed=6)


@pytest.mark.slow
def test_c3_full_sampled():
    _run_and_compare(S.stream_c3(), sample_k=400, seed=3)


@pytest.mark.slow
def test_c4_full_sampled():
    """Full C4 (2,000 steps). The oracle replays every RoPE and KV write and
    evaluates SDPA only for 12 sampled steps (no op reads an SDPA output)."""
    s = S.stream_c4()
    sd = [j for j, o in enumerate(s.ops) if o.op == "sdpa"]
    keep = sample(sd, 12, seed=4)
    _run_and_compare(s, check=keep, skip=sd)


@pytest.mark.slow
def test_largest_elementwise_op_sampled():
    """One bf16 add of 2^31 + 1000 elements (three 4 GiB tensors): 64-bit
    element offsets past 2^32 bytes, 262,145 tiles over the capped helper
    count and the tile counter. Windows at the start, around 2^31 and at
    the ragged end are compared with the oracle's add on the same windows;
    the executor runs alone on this descriptor."""
    import torch
    from oracle.interp import lib as orc_lib
    from persistent_micro_dispatch_gb300 import gpuos as G
    n = (1 << 31) + 1000
    g = torch.Generator(device="cuda").manual_seed(31)
    a = torch.randn(n, device="cuda", generator=g, dtype=torch.bfloat16)
    b = torch.randn(n, device="cuda", generator=g, dtype=torch.bfloat16)
    out = torch.full((n,), 7.0, device="cuda", dtype=torch.bfloat16)
    torch.cuda.synchronize()
    d = G.make_descs(1)
    d["op_id"] = G.OP["add"]
    d["dtype"] = G.BF16
    d["a"], d["b"], d["out"] = a.data_ptr(), b.data_ptr(), out.data_ptr()
    d["dims"][0, 0] = n
    ex = G.Executor()
    try:
        ex.submit(d)
        ex.sync(timeout_ms=120_000)
    finally:
        assert ex.shutdown() == G.OK
    L = orc_lib()
    for lo in (0, 1 << 20, (1 << 31) - 4096, 1 << 31, n - 5000):
        hi = min(n, lo + 8192)
        av = a[lo:hi].view(torch.int16).cpu().numpy().view(np.uint16).copy()
        bv = b[lo:hi].view(torch.int16).cpu().numpy().view(np.uint16).copy()
        got = out[lo:hi].view(torch.int16).cpu().numpy().view(np.uint16)
        exact = np.empty(hi - lo, np.float64)
        want = np.empty(hi - lo, np.uint16)
        L.orc_add(1, av.ctypes.data, bv.ctypes.data, exact.ctypes.data, hi - lo)
        L.orc_store(1, exact.ctypes.data, want.ctypes.data, hi - lo)
        assert np.array_equal(got, want), (lo, int(np.count_nonzero(got != want)))
