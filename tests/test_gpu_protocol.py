"""Ring, table and failure-handling protocol of the executor (GPU).

Every failure here is made on the host or with a bounded device wait: no
test faults, traps or hangs the GPU.
"""
import time

import numpy as np
import pytest

from oracle.interp import Machine
from tests.gpu_harness import compare_stream, ensure_built, need_gpu
from workloads import streams as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    ensure_built()
    from workloads.device import warm_torch
    warm_torch()


def G():
    from persistent_micro_dispatch_gb300 import gpuos
    return gpuos


def _c1_small(n_desc=1000, n=4096, seed=11):
    from workloads.device import DeviceStream
    s = S.stream_c1(n_desc=n_desc, n=n, seed=seed)
    return s, DeviceStream(s)


def _check_all(s, ds):
    m = Machine(s)
    m.run(keep=range(len(s.ops)))
    rep = compare_stream(s, ds, m, range(len(s.ops)))
    assert rep.ok(), "\n".join(rep.failures)
    return rep


@pytest.mark.parametrize("sequencers", [1, 2, 4])
def test_ring_wraps_many_times_small_ring(sequencers):
    """1,000 descriptors through a 64-entry ring (15 laps), bit-exact; with
    several sequencer warps the 64-ticket windows are taken in turn."""
    s, ds = _c1_small()
    ex = G().Executor(ring_entries=64, sequencers=sequencers)
    try:
        ex.submit_batch(ds.descs())
        ex.sync(timeout_ms=30_000)
        st = ex.stats()
    finally:
        assert ex.shutdown() == 0
    assert st["completed"] == 1000 and st["errors"] == 0
    rep = _check_all(s, ds)
    assert rep.exact == 1000


def test_deferred_start_fills_ring_then_wraps():
    s, ds = _c1_small(n_desc=300)
    d = ds.descs()
    ex = G().Executor(ring_entries=64, deferred_start=1)
    try:
        ex.submit_batch(d[:64])
        # the ring is full and nothing runs yet: the next submit cannot wait
        assert ex.try_submit(d[64:65], timeout_us=0) == G().EAGAIN
        ex.start()
        ex.submit_batch(d[64:])
        ex.sync(timeout_ms=30_000)
    finally:
        assert ex.shutdown() == 0
    _check_all(s, ds)


def test_stop_stream_and_tile_profile():
    """The executor's own stream brackets its single launch (an event recorded
    after it completes only when the kernel ends), stop drains the ring and
    ends the kernel (exit reason 1), and the tile profile counts every tile
    of every descriptor once, per op kind, as the host's tiling rule gives
    them; the results match the oracle."""
    import torch
    from workloads.device import DeviceStream
    s = S.stream_elementwise("ew_profile", 300, 256, 65536, 0.30, 1 << 22, 21)
    ds = DeviceStream(s)
    d = ds.descs()
    expected = {}
    for i, o in enumerate(s.ops):
        expected[o.op] = expected.get(o.op, 0) + G().op_ntiles(d[i:i + 1])
    ex = G().Executor(deferred_start=1)
    try:
        sp = ex.stream
        assert sp != 0
        xs = torch.cuda.ExternalStream(sp)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(xs)
        ex.start()
        e1.record(xs)
        ex.submit_batch(d)
        ex.sync(timeout_ms=30_000)
        assert not e1.query()  # still resident: the event waits for the kernel's end
        assert ex.stop() == 0
        e1.synchronize()
        assert e0.elapsed_time(e1) > 0.0
        st = ex.stats()
        prof = ex.tile_profile()
    finally:
        assert ex.shutdown() == 0
    assert st["completed"] == len(s.ops) and st["errors"] == 0 and st["exit_reason"] == 1
    assert {k: v["tiles"] for k, v in prof.items()} == expected
    assert all(v["body_us"] > 0.0 and v["finish_us"] >= 0.0 and v["dep_us"] >= 0.0 for v in prof.values())
    _check_all(s, ds)


def _big_add(n):
    import torch
    a = torch.ones(n, dtype=torch.float32, device="cuda")
    b = torch.ones(n, dtype=torch.float32, device="cuda")
    c = torch.empty(n, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    d = G().make_descs(1)
    d["op_id"] = G().OP["add"]
    d["dtype"] = G().F32
    d["a"], d["b"], d["out"] = a.data_ptr(), b.data_ptr(), c.data_ptr()
    d["dims"][0, 0] = n
    return d, (a, b, c)


def test_full_ring_returns_eagain_and_recovers():
    """One worker warp busy with a long op: the 64-entry ring fills and a
    submit with a short timeout returns EAGAIN; everything completes later."""
    g = G()
    big, keep = _big_add(1 << 26)
    nop = g.make_descs(1)
    ex = g.Executor(ring_entries=64, blocks=1, warps_per_block=2)
    try:
        ex.submit(big)
        for _ in range(63):
            ex.submit(nop)
        t0 = time.perf_counter()
        rc = ex.try_submit(nop, timeout_us=2000)
        assert rc == g.EAGAIN
        assert time.perf_counter() - t0 < 1.0
        ex.submit(nop, timeout_us=30_000_000)  # waits for a slot, then succeeds
        ex.sync(timeout_ms=60_000)
        st = ex.stats()
    finally:
        assert ex.shutdown() == 0
    assert st["completed"] == 65 and st["errors"] == 0
    assert float(keep[2][-1].item()) == 2.0


def test_fence_wait_times_out_with_status():
    """A FENCE behind a long op with a 20 ms device wait bound completes with
    GPUOS_ST_DEP_TIMEOUT; sync reports EDEVICE; the executor stays usable."""
    g = G()
    big, keep = _big_add(1 << 26)
    nop = g.make_descs(1)
    fence = g.make_descs(1)
    fence["flags"] = g.FLAG_FENCE
    ex = g.Executor(blocks=1, warps_per_block=2, dep_timeout_ms=20)
    try:
        ex.submit(big)
        t = ex.submit(fence)
        rc = ex.sync(timeout_ms=60_000, raise_on_error=False)
        assert rc == g.EDEVICE
        assert ex.query(t).status == g.ST_DEP_TIMEOUT
        t2 = ex.submit(nop)
        assert ex.sync(t2, timeout_ms=10_000, raise_on_error=False) == g.OK
    finally:
        ex.shutdown()


@pytest.mark.parametrize("sequencers", [1, 4])
def test_fence_orders_after_all_earlier(sequencers):
    """A FENCE descriptor starts only after every earlier one completed."""
    g = G()
    big, keep = _big_add(1 << 24)
    nop = g.make_descs(1)
    fence = g.make_descs(1)
    fence["flags"] = g.FLAG_FENCE
    ex = g.Executor(sequencers=sequencers)
    try:
        base = ex.stats()["submitted"]
        h = ex.set_history(base, 3)
        ex.submit(big)
        ex.submit(nop)
        ex.submit(fence)
        ex.sync(timeout_ms=30_000)
    finally:
        ex.shutdown()
    # the fenced descriptor is published (and starts) after both completed
    assert h["t_publish_dev_ns"][2] >= h["t_done_dev_ns"][0]
    assert h["t_start_dev_ns"][2] >= h["t_done_dev_ns"][1]


@pytest.mark.parametrize("sequencers", [1, 4])
def test_fence_cuts_batches_at_any_position(sequencers):
    """FENCE descriptors anywhere in a full ring (a sequencer takes up to 128
    descriptors a batch, read in two halves of 64; with four sequencers each
    takes every fourth window of 128 tickets): each one is published and
    starts only after every earlier descriptor completed, including at the
    half, batch and window boundaries."""
    g = G()
    big, keep = _big_add(1 << 20)
    n = 300
    d = g.make_descs(n)
    d[:] = big[0]
    fences = [1, 63, 64, 65, 127, 128, 129, 191, 192, 255, 299]
    for i in fences:
        d["flags"][i] = g.FLAG_FENCE
    ex = g.Executor(ring_entries=512, deferred_start=1, sequencers=sequencers)
    try:
        h = ex.set_history(0, n)
        ex.submit_batch(d)
        ex.start()
        ex.sync(timeout_ms=30_000)
    finally:
        assert ex.shutdown() == 0
    assert (h["status"] == 0).all() and (h["ticket"] == np.arange(n)).all()
    done = h["t_done_dev_ns"]
    for i in fences:
        assert h["t_publish_dev_ns"][i] >= done[:i].max(), i
        assert h["t_start_dev_ns"][i] >= done[:i].max(), i
    assert bool((keep[2] == 2.0).all())


def test_device_bounds_checks_return_status():
    """Descriptors that pass the host checks but carry bad positions or
    lengths in device memory complete with GPUOS_ST_BAD_ARGS."""
    import torch
    g = G()
    B, H, D, Lc = 2, 4, 128, 64
    q = torch.zeros(B * H * D, dtype=torch.bfloat16, device="cuda")
    K = torch.zeros(B * H * Lc * D, dtype=torch.bfloat16, device="cuda")
    V = torch.zeros_like(K)
    o = torch.zeros_like(q)
    lens = torch.tensor([0, 70], dtype=torch.int32, device="cuda")  # 0: pos -1; 70 > Lcap
    ws = torch.zeros(g.sdpa_workspace_bytes(B, H, D, Lc), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    kv = g.make_descs(1)
    kv["op_id"] = g.OP["kv_write"]
    kv["a"], kv["b"], kv["aux0"], kv["out"], kv["aux1"] = q.data_ptr(), q.data_ptr(), lens.data_ptr(), K.data_ptr(), V.data_ptr()
    kv["dims"][0, :4] = (B, H, D, Lc)
    sd = g.make_descs(1)
    sd["op_id"] = g.OP["sdpa"]
    sd["a"], sd["b"], sd["aux1"], sd["aux0"], sd["out"], sd["aux2"] = (q.data_ptr(), K.data_ptr(), V.data_ptr(),
                                                                      lens.data_ptr(), o.data_ptr(), ws.data_ptr())
    sd["dims"][0, :6] = (B, H, D, Lc, Lc, B * H)
    sd["fparam"][0, 0] = 0.1
    bad = g.make_descs(1)
    bad["op_id"] = 200  # not registered: rejected on the host, no ticket used
    ex = g.Executor()
    try:
        assert ex.try_submit(bad) == g.EINVAL
        t1 = ex.submit(kv)
        t2 = ex.submit(sd)
        assert ex.sync(timeout_ms=10_000, raise_on_error=False) == g.EDEVICE
        assert ex.query(t1).status == g.ST_BAD_ARGS
        assert ex.query(t2).status == g.ST_BAD_ARGS
        st = ex.stats()
        assert st["errors"] == 2 and st["submitted"] == 2
    finally:
        ex.shutdown()
    assert int(ws.view(torch.int32)[: B * H].abs().sum().item()) == 0  # counters left zero


def test_dependency_on_future_ticket_rejected():
    g = G()
    nop = g.make_descs(1)
    nop["dep"][0, 0] = 5  # absolute ticket + 1 of a descriptor not yet submitted
    ex = g.Executor()
    try:
        assert ex.try_submit(nop) == g.EINVAL
    finally:
        ex.shutdown()


def _ext_image():
    return open(G().EXT_CUBIN, "rb").read()


def test_hot_swap_under_load_every_result_old_or_new():
    """Swap op ADD for the injected subtract while 3,000 adds are in flight;
    each descriptor's output is a+b or a-b according to the table version it
    recorded; swapping back restores add. Bit-exact against the oracle
    (a - b = a + (-b) exactly)."""
    g = G()
    from workloads.device import DeviceStream
    s = S.stream_c1(n_desc=3000, n=4096, seed=12)
    for o in s.ops:
        o.op = "add"
        if o.b is None:
            o.b = S.Ref(s.buf_index("b"), o.a.off)
    ds = DeviceStream(s)
    d = ds.descs()
    ex = g.Executor(deferred_start=1)
    try:
        ex.load_module(_ext_image())  # modules load before the executor is resident
        ex.start()
        hist = ex.set_history(0, len(d))
        ex.submit_batch(d[:1000])
        ex.register_op(g.OP["add"], _ext_image(), "gpuos_ext_sub_ptr")  # version 1
        ex.submit_batch(d[1000:2000])
        ex.alias_op(g.OP["add"], g.OP["mul"])  # version 2: mul
        ex.submit_batch(d[2000:])
        ex.sync(timeout_ms=30_000)
        st = ex.stats()
    finally:
        ex.shutdown()
    assert st["version"] == 2
    ver = hist["version"]
    assert set(np.unique(ver)) <= {0, 1, 2}
    assert (ver[:1000] <= 1).all() and (ver[2000:] == 2).all()
    assert (ver == 1).sum() > 0
    m = Machine(s)
    bi = s.buf_index("b")
    for j, o in enumerate(s.ops):
        if ver[j] == 1:
            m.buf[bi][o.b.off:o.b.off + o.dims[0]] *= -1  # oracle: a + (-b)
            m.apply(j)
            m.buf[bi][o.b.off:o.b.off + o.dims[0]] *= -1
        elif ver[j] == 2:
            o.op = "mul"
            m.apply(j)
            o.op = "add"
        else:
            m.apply(j)
    for j, o in enumerate(s.ops):
        n = o.dims[0]
        assert np.array_equal(ds.read(o.out, n).view(np.uint32), m.view(o.out, n).view(np.uint32)), (j, ver[j])


def test_user_op_registration():
    """An injected op under a new id (64) with a caller-set tile count."""
    import torch
    g = G()
    n = 5000
    x = torch.randn(n, dtype=torch.float32, device="cuda")
    y = torch.zeros(n, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    d = g.make_descs(1)
    d["op_id"] = 64
    d["dtype"] = g.F32
    d["a"], d["out"] = x.data_ptr(), y.data_ptr()
    d["dims"][0, 0] = n
    d["fparam"][0, 0] = 2.5
    d["ntiles"] = (n + 1023) // 1024
    ex = g.Executor(deferred_start=1)
    try:
        ex.load_module(_ext_image())
        ex.start()
        assert ex.try_submit(d) == g.EINVAL  # not registered yet
        ex.register_op(64, _ext_image(), "gpuos_ext_scale_ptr")
        ex.submit(d)
        ex.sync(timeout_ms=10_000)
    finally:
        ex.shutdown()
    xs = x.cpu().numpy()
    want = (xs.astype(np.float64) * np.float32(2.5)).astype(np.float32)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_register_op_rejects_bad_symbol_and_unloaded_image():
    g = G()
    ex = g.Executor(deferred_start=1)
    try:
        ex.load_module(_ext_image())
        ex.start()
        with pytest.raises(g.GpuosError) as e:
            ex.register_op(64, _ext_image(), "no_such_symbol")
        assert e.value.code == g.EINVAL
        with pytest.raises(g.GpuosError) as e:
            ex.register_op(20, _ext_image(), "gpuos_ext_sub_ptr")  # reserved id
        assert e.value.code == g.EINVAL
        # an image that does not link is refused before anything stops
        t0 = time.perf_counter()
        with pytest.raises(g.GpuosError) as e:
            ex.register_op(64, b"\x7fELF" + b"\0" * 256, "gpuos_ext_scale_ptr")
        assert e.value.code == g.EINVAL and time.perf_counter() - t0 < 5.0
        assert ex.stats()["running"] == 1
    finally:
        ex.shutdown()


def test_idle_watchdog_ends_executor():
    """With no host activity for idle_exit_ms the kernel leaves by itself."""
    g = G()
    ex = g.Executor(idle_exit_ms=300)
    try:
        time.sleep(1.5)
        st = ex.stats()
        assert st["running"] == 0 and st["exit_reason"] == 2
        assert ex.try_submit(g.make_descs(1)) == g.ESTOPPED
    finally:
        ex.shutdown()


def test_exit_after_bounded_run():
    s, ds = _c1_small(n_desc=200)
    g = G()
    ex = g.Executor(deferred_start=1, exit_after=200)
    try:
        ex.submit_batch(ds.descs())
        ex.start()
        ex.sync(timeout_ms=30_000)
        t0 = time.perf_counter()
        while ex.stats()["running"] and time.perf_counter() - t0 < 10:
            time.sleep(0.01)
        st = ex.stats()
        assert st["running"] == 0 and st["exit_reason"] == 3
    finally:
        ex.shutdown()
    _check_all(s, ds)


def test_calibration_bounds_and_record_order():
    g = G()
    ex = g.Executor()
    try:
        lo, hi, rtt, rtts = ex.calibrate(100)
        assert lo <= hi and 0 < rtt < 200_000
        base = ex.stats()["submitted"]
        h = ex.set_history(base, 50)
        for _ in range(50):
            ex.sync(ex.submit(g.make_descs(1)))
    finally:
        ex.shutdown()
    assert (h["t_dispatch_dev_ns"] <= h["t_publish_dev_ns"]).all()
    assert (h["t_publish_dev_ns"] <= h["t_start_dev_ns"]).all()
    assert (h["t_start_dev_ns"] <= h["t_done_dev_ns"]).all()


def test_eager_path_matches_executor_bitwise():
    """The eager baseline runs the same op bodies: identical outputs."""
    import torch
    g = G()
    from workloads.device import DeviceStream
    s = S.stream_mixed_small()
    ds1 = DeviceStream(s)
    ds2 = DeviceStream(s)
    ex = g.Executor()
    try:
        ex.submit_batch(ds1.descs())
        ex.sync(timeout_ms=30_000)
    finally:
        ex.shutdown()
    st = torch.cuda.Stream()
    g.eager_run(ds2.descs(), st.cuda_stream, stage_bytes=16384)
    st.synchronize()
    for i, b in enumerate(s.buffers):
        if b.name in ("sdpa_ws",):
            continue
        assert np.array_equal(ds1.read_buf(i).view(np.uint8), ds2.read_buf(i).view(np.uint8)), b.name


def test_multi_producer_threads_share_the_ring():
    """Eight host threads submit concurrently (multi_producer = 1) through a
    256-entry ring (many laps): each thread's descriptors (C1 ops on its own
    slice of the stream) get unique tickets, every op runs once, every
    output is bit-exact, and the completion count matches."""
    import threading
    s, ds = _c1_small(n_desc=2000)
    descs = ds.descs()
    ex = G().Executor(ring_entries=256, multi_producer=1)
    T = 8
    firsts = [[] for _ in range(T)]
    errors = []

    def producer(k):
        try:
            mine = descs[k::T]
            for i in range(0, len(mine), 5):  # batches of 5 and single submits
                chunk = mine[i:i + 5]
                if i % 2 == 0:
                    firsts[k].append((ex.submit_batch(chunk), len(chunk)))
                else:
                    for d in chunk:
                        firsts[k].append((ex.submit(d), 1))
        except Exception as e:  # reported below
            errors.append(e)

    try:
        th = [threading.Thread(target=producer, args=(k,)) for k in range(T)]
        for t in th:
            t.start()
        for t in th:
            t.join(timeout=120)
        assert not errors, errors
        ex.sync(timeout_ms=60_000)
        st = ex.stats()
    finally:
        assert ex.shutdown() == 0
    tickets = sorted(t0 + j for f in firsts for (t0, n) in f for j in range(n))
    assert tickets == list(range(len(descs)))  # unique, no gaps
    assert st["completed"] == len(descs) and st["errors"] == 0 and st["submitted"] == len(descs)
    rep = _check_all(s, ds)
    assert rep.exact == len(descs)


def test_multi_producer_needs_started_executor():
    g = G()
    ex = g.Executor(deferred_start=1, multi_producer=1)
    try:
        d = g.make_descs(1)
        assert ex.try_submit(d) == g.EINVAL
        ex.start()
        assert ex.try_submit(d) == g.OK
        ex.sync(timeout_ms=10_000)
    finally:
        assert ex.shutdown() == 0


_NEG_SRC = r'''
/* out[i] = -a[i] (fp32). Tiles split n like the built-in element-wise ops:
 * ntiles ranges of round_up(ceil(n / ntiles), 256) elements, so the op can
 * also stand in for a built-in id, whose tile count the library computes. */
__device__ int op_neg(const gpuos_devdesc *d, uint32_t tile)
{
    const uint32_t n = d->dims[0], lane = threadIdx.x & 31u;
    const uint32_t nt = d->ntiles ? d->ntiles : 1u;
    const uint32_t te = ((n + nt - 1u) / nt + 255u) / 256u * 256u;
    const float *a = reinterpret_cast<const float *>(d->a);
    float *o = reinterpret_cast<float *>(d->out);
    const unsigned long long start = (unsigned long long)tile * te;
    const unsigned long long end = start + te < n ? start + te : n;
    for (unsigned long long i = start + lane; i < end; i += 32) o[i] = -a[i];
    return GPUOS_ST_OK;
}
__device__ gpuos_op_fn op_neg_ptr = op_neg;
'''


def test_runtime_compiled_op_injection():
    """An op compiled at run time (NVRTC) is linked into the executor and
    installed under a new id; results are bit-exact, and swapping the
    built-in id 1 (add) to it later changes what id 1 computes. (Results are
    read after shutdown: a pageable device-to-host copy on PyTorch's stream
    waits while the executor is resident.)"""
    import torch
    g = G()
    img = g.compile_op(_NEG_SRC, "neg.cu")
    n = 10_000
    x = torch.randn(n, dtype=torch.float32, device="cuda")
    y = torch.zeros(n, dtype=torch.float32, device="cuda")
    z1 = torch.zeros(n, dtype=torch.float32, device="cuda")
    z2 = torch.zeros(n, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    d = g.make_descs(3)
    d["op_id"] = [70, 1, 1]
    d["dtype"] = g.F32
    d["a"] = x.data_ptr()
    d["b"] = x.data_ptr()
    d["out"] = [y.data_ptr(), z1.data_ptr(), z2.data_ptr()]
    d["dims"][:, 0] = n
    d["ntiles"][0] = (n + 1023) // 1024
    ex = g.Executor(deferred_start=1)
    try:
        ex.load_module(img)
        ex.start()
        ex.register_op(70, img, "op_neg_ptr")
        ex.submit_batch(d[:2])
        ex.sync(timeout_ms=10_000)
        ex.register_op(1, img, "op_neg_ptr")  # now id 1 runs the compiled op
        ex.submit(d[2:3])
        ex.sync(timeout_ms=10_000)
        st = ex.stats()
    finally:
        ex.shutdown()
    assert st["errors"] == 0 and st["version"] == 2
    xs = x.cpu().numpy()
    assert np.array_equal(y.cpu().numpy(), -xs)
    assert np.array_equal(z1.cpu().numpy(), xs + xs)  # id 1 was still add
    assert np.array_equal(z2.cpu().numpy(), -xs)


@pytest.mark.parametrize("sequencers", [1, 2, 3, 4])
def test_chains_across_windows_with_many_helpers(sequencers):
    """A strict chain of large ops (every descriptor waits for the one
    before it, 512 helper warps each) across many 128-ticket
    windows: with several sequencers a later window may be ready first, and
    the work queue must still hand out entries in ticket order, or waiting
    helpers would hold every worker. Every result equals the oracle's."""
    import torch
    from workloads.device import DeviceStream
    s = S.Stream("chain_windows")
    n = 1 << 21
    rng = np.random.default_rng(17)
    ix = s.add_buf("x", "f32", n, rng.standard_normal(n, dtype=np.float32))
    # |y| in [0.5, 1): the products shrink, the sums grow by at most 1 a step
    yv = (rng.uniform(0.5, 1.0, n) * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    iy = s.add_buf("y", "f32", n, yv)
    steps = 300
    iz = s.add_buf("z", "f32", n * 2)
    for j in range(steps):
        src = S.Ref(ix) if j == 0 else S.Ref(iz, ((j - 1) % 2) * n)
        dst = S.Ref(iz, (j % 2) * n)
        deps = () if j == 0 else (j - 1,)
        op = ("add", "mul", "relu")[j % 3]
        if op == "relu":
            s.ops.append(S.Op("relu", "f32", a=src, out=dst, dims=(n,), deps=deps))
        else:
            s.ops.append(S.Op(op, "f32", a=src, b=S.Ref(iy), out=dst, dims=(n,), deps=deps))
    S.check_hazards(s)
    ds = DeviceStream(s)
    ex = G().Executor(sequencers=sequencers)
    try:
        h = ex.set_history(0, steps)
        ex.submit_batch(ds.descs())
        ex.sync(timeout_ms=60_000)
    finally:
        assert ex.shutdown() == 0
    assert (h["status"] == 0).all()
    torch.cuda.synchronize()
    m = Machine(s)
    m.run()
    last = s.ops[-1].out
    assert np.array_equal(ds.read(last, n).view(np.uint32), m.view(last, n).view(np.uint32))


def test_operator_compiled_after_launch_enters_by_handoff():
    """Operators that did not exist when the executor was launched: each new
    module enters by a hand-off (drain, the kernel leaves, the module set is
    linked again, the kernel relaunches at the next ticket). Descriptors
    before and after every hand-off and flip run with the entry of the
    version they recorded; results are bit-exact against the oracle's add
    and mul and the exact negation. Earlier bindings survive a second
    hand-off (the table is rebuilt with the new module's addresses)."""
    import torch
    g = G()
    from workloads.device import DeviceStream
    s = S.stream_c1(n_desc=3000, n=4096, seed=13)
    for o in s.ops:
        o.op = "add"
        if o.b is None:
            o.b = S.Ref(s.buf_index("b"), o.a.off)
    ds = DeviceStream(s)
    d = ds.descs()
    neg = g.compile_op(_NEG_SRC, "neg.cu")
    n = 5000
    x = torch.randn(n, dtype=torch.float32, device="cuda")
    y = torch.zeros(n, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    sc = g.make_descs(1)
    sc["op_id"] = 64
    sc["dtype"] = g.F32
    sc["a"], sc["out"] = x.data_ptr(), y.data_ptr()
    sc["dims"][0, 0] = n
    sc["fparam"][0, 0] = 2.5
    sc["ntiles"] = (n + 1023) // 1024
    ex = g.Executor()  # launched with the built-in ops only
    times = []
    try:
        hist = ex.set_history(0, len(d) + 1)
        ex.submit_batch(d[:1000])                      # version 0: add
        t0 = time.perf_counter()
        ex.register_op(g.OP["add"], neg, "op_neg_ptr")  # hand-off, version 1: id 1 = neg
        times.append(time.perf_counter() - t0)
        ex.submit_batch(d[1000:2000])
        t0 = time.perf_counter()
        ex.register_op(64, _ext_image(), "gpuos_ext_scale_ptr")  # second hand-off, version 2
        times.append(time.perf_counter() - t0)
        ex.submit_batch(d[2000:2500])                   # id 1 still neg
        ex.submit(sc)
        # a flip applies to descriptors sequenced after it, not to those
        # submitted after it: wait until these have run, so that the
        # versions asserted below are fixed
        ex.sync(timeout_ms=30_000)
        ex.alias_op(g.OP["add"], g.OP["mul"])           # version 3: id 1 = mul
        ex.submit_batch(d[2500:])
        ex.sync(timeout_ms=30_000)
        st = ex.stats()
    finally:
        assert ex.shutdown() == 0
    print(f"hand-off times (s): {times}; last: link {st['handoff_link_ns'] / 1e6:.2f} ms, "
          f"executor down {st['handoff_down_ns'] / 1e6:.2f} ms")
    assert st["errors"] == 0 and st["version"] == 3
    assert st["handoffs"] == 2
    # the executor is down only for the drain, the exit and the relaunch (the
    # link runs while the old executor still serves)
    assert 0 < st["handoff_down_ns"] < 100_000_000 and st["handoff_down_ns"] < st["handoff_link_ns"]
    # tickets: d[:2500] are 0..2499, the scale op 2500, d[2500:] 2501..3000
    ver = np.concatenate([hist["version"][:2500], hist["version"][2501:]])
    assert hist["version"][2500] == 2
    assert (ver[:1000] == 0).all() and (ver[1000:2000] == 1).all() and (ver[2000:2500] == 2).all()
    assert (ver[2500:] == 3).all()
    # the relaunched kernel picked up where the old one stopped
    assert hist["t_dispatch_dev_ns"][1000] >= hist["t_done_dev_ns"][:1000].max()
    assert hist["t_dispatch_dev_ns"][2000] >= hist["t_done_dev_ns"][1000:2000].max()
    m = Machine(s)
    for j, o in enumerate(s.ops):
        if ver[j] == 3:
            o.op = "mul"
            m.apply(j)
            o.op = "add"
        elif ver[j] == 0:
            m.apply(j)
    for j, o in enumerate(s.ops):
        nn = o.dims[0]
        got = ds.read(o.out, nn)
        if ver[j] in (1, 2):
            want = -ds.read(o.a, nn)
        else:
            want = m.view(o.out, nn)
        assert np.array_equal(got.view(np.uint32), np.asarray(want, np.float32).view(np.uint32)), (j, ver[j])
    xs = x.cpu().numpy()
    want = (xs.astype(np.float64) * np.float32(2.5)).astype(np.float32)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert max(times) < 10.0


def test_handoff_needs_a_single_producer():
    g = G()
    ex = g.Executor(multi_producer=1)
    try:
        with pytest.raises(g.GpuosError) as e:
            ex.load_module(_ext_image())
        assert e.value.code == g.EBUSY
        assert ex.stats()["running"] == 1
    finally:
        ex.shutdown()

