"""The C-ABI library builds, loads and exports every symbol include/gpuos.h
declares; host-only entry points behave without a GPU (CPU)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def G():
    from persistent_micro_dispatch_gb300 import build
    build.build()
    from persistent_micro_dispatch_gb300 import gpuos
    gpuos.lib()
    return gpuos


def header_symbols():
    txt = open(os.path.join(ROOT, "include", "gpuos.h")).read()
    return sorted(set(re.findall(r"GPUOS_API\s+[\w\s\*]+?\b(gpuos_\w+)\s*\(", txt)))


def test_header_declares_the_ring_protocol_verbs():
    syms = header_symbols()
    for v in ("gpuos_init", "gpuos_submit", "gpuos_register_op", "gpuos_sync", "gpuos_shutdown"):
        assert v in syms
    assert len(syms) >= 17


def test_library_exports_every_declared_symbol(G):
    lib = C.CDLL(G.LIB_PATH)
    for name in header_symbols():
        assert hasattr(lib, name), name
    assert set(header_symbols()) == set(G.API), "binding and header disagree"


def test_only_public_symbols_exported(G):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", G.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == set(header_symbols())


def test_descriptor_layout_matches_header(G):
    assert G.DESC_DTYPE.itemsize == 128
    off = {n: G.DESC_DTYPE.fields[n][1] for n in G.DESC_DTYPE.names}
    assert off["dep"] == 8 and off["a"] == 24 and off["dims"] == 72 and off["fparam"] == 96
    assert off["user"] == 104 and off["ticket"] == 112 and off["seq"] == 120
    assert C.sizeof(G.Config) == 72 and C.sizeof(G.Record) == 56


def test_default_config(G):
    c = G.default_config()
    assert c.ring_entries == 8192 and c.warps_per_block == 12 and c.tq_entries == 0
    assert c.idle_exit_ms > 0 and c.dep_timeout_ms > 0


def _desc(G, op, dtype=1, dims=(), ptr=0x1000, **kw):
    d = G.make_descs(1)
    d["op_id"] = G.OP[op] if isinstance(op, str) else op
    d["dtype"] = dtype
    dd = list(dims) + [0] * (6 - len(dims))
    d["dims"] = dd
    for f in ("a", "b", "out", "aux0", "aux1", "aux2"):
        d[f] = kw.get(f, ptr)
    if "dep" in kw:
        d["dep"] = kw["dep"]
    return d


def test_elementwise_tiling_over_sizes(G):
    """The element-wise tile count over many sizes, against the rule stated
    as a loop: start at the op's smallest tile (16384 elements; a GELU with
    a dependency 1024, see test_tiling_rule), double it while it is below
    the dtype's largest tile (fp32
    16384, bf16 32768) and would cut n into more than 16 tiles; the count is
    ceil(n / tile), and an empty op has one tile."""
    rng = np.random.default_rng(5)
    ns = sorted(set(list(range(0, 300)) + [k * m + e for k in range(1, 22) for m in (1024, 4096, 65536)
                                           for e in (-1, 0, 1) if k * m + e >= 0]
                    + rng.integers(1, 1 << 31, size=300).tolist()))
    for op in ("add", "mul", "relu", "gelu"):
        for dt in (0, 1):
            tmin = 16384
            tmax = 16384 if dt == 0 else 32768
            for n in ns:
                te = min(tmin, tmax)
                while te < tmax and te * 16 < n:
                    te *= 2
                want = max(1, -(-n // te))
                if want > 0xFFFFFFFF:
                    continue
                assert G.op_ntiles(_desc(G, op, dt, (n,))) == want, (op, dt, n)


def test_tiling_rule(G):
    # element-wise: te = smallest power of two >= n/16 within [16384 (a GELU with a dependency:
    # 1024), 16384 | 32768]
    assert G.op_ntiles(_desc(G, "add", 0, (4096,))) == 1          # te 16384
    assert G.op_ntiles(_desc(G, "gelu", 0, (4096,))) == 1         # te 16384
    assert G.op_ntiles(_desc(G, "add", 1, (16384,))) == 1         # te 16384
    assert G.op_ntiles(_desc(G, "gelu", 1, (16384,))) == 1        # te 16384
    assert G.op_ntiles(_desc(G, "gelu", 0, (16385,))) == 2        # te 16384
    assert G.op_ntiles(_desc(G, "relu", 0, (8193,))) == 1         # te 16384
    assert G.op_ntiles(_desc(G, "relu", 0, (16385,))) == 2        # te 16384
    assert G.op_ntiles(_desc(G, "mul", 0, (1000,))) == 1
    assert G.op_ntiles(_desc(G, "add", 0, (65536,))) == 4         # te 16384
    assert G.op_ntiles(_desc(G, "add", 1, (65536,))) == 4         # te 16384
    assert G.op_ntiles(_desc(G, "add", 0, (1 << 20,))) == 64      # te 16384 (fp32 cap)
    assert G.op_ntiles(_desc(G, "add", 1, (1 << 20,))) == 32      # te 32768 (bf16 cap)
    assert G.op_ntiles(_desc(G, "gelu", 1, (1 << 20,))) == 32     # te 32768 (bf16 cap)
    assert G.op_ntiles(_desc(G, "gelu", 1, (40000,))) == 3        # te 16384 >= 40000/16
    assert G.op_ntiles(_desc(G, "gelu", 1, (600000,))) == 19      # n/16 wants 65536: te 32768 (bf16 cap)
    # a GELU with a dependency keeps the finer split: te from 1024
    assert G.op_ntiles(_desc(G, "gelu", 1, (4096,), dep=(5, 0))) == 4      # te 1024
    assert G.op_ntiles(_desc(G, "gelu", 1, (4096,), dep=(0, 5))) == 4
    assert G.op_ntiles(_desc(G, "gelu", 1, (1000,), dep=(5, 0))) == 1
    assert G.op_ntiles(_desc(G, "add", 1, (4096,), dep=(5, 0))) == 1       # add/mul/ReLU: no change
    assert G.op_ntiles(_desc(G, "gelu", 0, (0,))) == 1            # empty op: one tile
    assert G.op_ntiles(_desc(G, "softmax", 1, (37, 1024))) == 37  # one row per tile
    assert G.op_ntiles(_desc(G, "rope", 1, (5, 32, 128))) == 5 * 8  # four heads per tile
    assert G.op_ntiles(_desc(G, "rope", 1, (2, 6, 64))) == 2 * 2
    kv = _desc(G, "kv_write", 1, (3, 30, 128, 4096), out=0x2000, aux1=0x3000)
    assert G.op_ntiles(kv) == 3 * 8
    # attention: at most floor(1536 / pairs) chunks per (request, head) pair,
    # of equal length rounded up to 32 rows. 96 pairs x 1025 rows: 16 wanted,
    # 65 -> 96-row chunks, 11 per pair
    assert G.op_ntiles(_desc(G, "sdpa", 1, (3, 32, 128, 4096, 1025, 96))) == 96 * 11
    assert G.op_ntiles(_desc(G, "sdpa", 1, (8, 32, 128, 4096, 4096, 256))) == 256 * 6   # 704-row chunks
    assert G.op_ntiles(_desc(G, "sdpa", 1, (1, 32, 128, 4096, 2000, 32))) == 32 * 32   # 64-row chunks
    assert G.op_ntiles(_desc(G, "sdpa", 1, (2, 1, 128, 4096, 4096, 2))) == 2 * 128     # 32 rows at least
    assert G.op_ntiles(_desc(G, "vecmat", 1, (1024, 1024))) == 128
    assert G.op_ntiles(_desc(G, "vecmat", 1, (1024, 1000))) == 125
    assert G.op_ntiles(_desc(G, "nop")) == 1


def test_device_tile_ranges_cover_each_op(G):
    """The device recovers the element-wise tile size and the attention chunk
    length from the host's ntiles (the rule stated in gpuos.h); for every
    size the ranges must cover the op, stay 16-byte aligned, fit the largest
    tile, and (attention) use no more partials than the workspace holds."""
    for (dt, cap), op in [(dc, o) for dc in ((0, 16384), (1, 32768)) for o in ("add", "gelu")]:
        for n in [1, 255, 256, 257, 1023, 1024, 1025, 4095, 4096, 4097, 16383, 16385, 65535, 65536,
                  65537, 100003, 1 << 20, (1 << 20) + 7, 3 * 8192 + 1]:
            nt = G.op_ntiles(_desc(G, op, dt, (n,)))
            te = -(-(-(-n // nt)) // 256) * 256
            assert te * nt >= n and te <= cap and te % 256 == 0, (dt, n, nt, te)
            assert (nt - 1) * te < n  # no tile starts past the end
    for B, H, L in ((1, 32, 1), (1, 32, 33), (1, 32, 2000), (3, 32, 1025), (8, 32, 4096), (2, 1, 4096),
                    (1, 1, 100), (4, 8, 777)):
        nt = G.op_ntiles(_desc(G, "sdpa", 1, (B, H, 128, 4096, L, B * H)))
        assert nt % (B * H) == 0
        nch = nt // (B * H)
        ch = -(-(-(-L // nch)) // 32) * 32
        assert ch * nch >= L and (nch - 1) * ch < L  # covered, no empty chunk
        assert nch <= -(-L // 32)  # within the workspace's partials
        assert nt <= max(1536, B * H)  # one wave on the default executor


def _sdpa_device_chunks(B, H, Lmax, nt, lens):
    """The decode-attention op body's chunk rule, restated: with one request
    or one chunk per pair, the host's chunks; otherwise the host's chunk
    length, shortened to round_up(ceil(H sum(lens) / (nt - B H)), 32) (at
    least 32) when that is shorter; chunks numbered request by request, then
    head, then chunk; a tile's partial goes to workspace slot `tile`.
    Returns {tile: (b, h, first_row, end_row, slot of the pair's first chunk)}."""
    nch = nt // (B * H)
    ch = -(-(-(-Lmax // nch)) // 32) * 32
    out = {}
    if nch == 1 or B == 1:  # the host's chunks
        for t in range(nt):
            b, rem = divmod(t, H * nch)
            h, c = divmod(rem, nch)
            if c * ch < lens[b]:
                out[t] = (b, h, c * ch, min(lens[b], (c + 1) * ch), t - c)
        return out
    spare = B * H * (nch - 1)
    cn = max(32, -(-(-(-(H * sum(lens)) // spare)) // 32) * 32)
    ch = min(ch, cn)
    t = 0
    for b in range(B):
        nb = -(-lens[b] // ch)
        for h in range(H):
            first = t
            for c in range(nb):
                out[t] = (b, h, c * ch, min(lens[b], (c + 1) * ch), first)
                t += 1
    assert t <= nt, (B, H, Lmax, nt, t)
    return out


def test_sdpa_device_chunks_cover_every_request(G):
    """For request lengths of every spread, the chunks the op body derives
    cover each (request, head) pair's rows [0, L_b) once, stay within the op's
    tiles (so within the workspace's partials), and a pair's chunks sit in
    consecutive workspace slots, where its last chunk merges them."""
    rng = np.random.default_rng(9)
    cases = [(1, 32, [2000]), (8, 32, [4096] * 8), (8, 32, [128, 4096, 33, 1, 700, 4095, 2048, 64]),
             (3, 32, [1025, 1, 1]), (2, 1, [4096, 32]), (4, 8, [777, 776, 1, 500]), (47, 32, list(range(1, 48)))]
    for _ in range(40):
        B = int(rng.integers(1, 12))
        cases.append((B, int(rng.choice([1, 4, 32])), rng.integers(1, 4097, size=B).tolist()))
    for B, H, lens in cases:
        Lmax = max(lens)
        nts = [G.op_ntiles(_desc(G, "sdpa", 1, (B, H, 128, 4096, Lmax, B * H)))]
        if B * H <= 256:
            # the allocation-free entry point's split: chunks of 256 rows
            nts.append(B * H * -(-Lmax // 256))
        for nt in nts:
            _check_sdpa_chunks(B, H, Lmax, nt, lens)


def _check_sdpa_chunks(B, H, Lmax, nt, lens):
    m = _sdpa_device_chunks(B, H, Lmax, nt, lens)
    assert max(m) < nt
    for b in range(B):
        for h in range(H):
            rows = sorted((v[2], v[3], t, v[4]) for t, v in m.items() if v[0] == b and v[1] == h)
            assert rows[0][0] == 0 and rows[-1][1] == lens[b]
            assert all(x[1] == y[0] for x, y in zip(rows, rows[1:]))
            assert all(r[0] % 32 == 0 and r[1] > r[0] for r in rows)
            assert [r[2] for r in rows] == list(range(rows[0][3], rows[0][3] + len(rows)))


@pytest.mark.parametrize("bad", [
    dict(op=20, dims=(4,)),                                      # reserved id
    dict(op="add", dtype=7, dims=(4,)),                          # bad dtype
    dict(op="add", dims=(4,), a=0),                              # null input
    dict(op="softmax", dtype=0, dims=(2, 8)),                    # row ops are bf16
    dict(op="sdpa", dims=(1, 32, 64, 4096, 100, 32)),            # D must be 128
    dict(op="sdpa", dims=(1, 32, 128, 4096, 5000, 32)),          # Lmax > Lcap
    dict(op="sdpa", dims=(2, 32, 128, 4096, 100, 32)),           # counters < B*H
    dict(op="sdpa", dims=(1, 32, 128, 4096, 100, 32), aux2=0x1008),  # unaligned workspace
    dict(op="rope", dims=(1, 32, 127)),                          # odd D
])
def test_host_bounds_checks_reject(G, bad):
    kw = dict(bad)
    op = kw.pop("op")
    dtype = kw.pop("dtype", 1)
    dims = kw.pop("dims")
    d = _desc(G, op, dtype, dims, **kw)
    n = C.c_uint32()
    assert G.lib().gpuos_op_ntiles(d.ctypes.data, C.byref(n)) == G.EINVAL


def test_elementwise_validation_cases(G):
    """The element-wise checks (taken without data-dependent branches on the
    host): each bad field alone is rejected, and what the op does not read
    may be null."""
    n = C.c_uint32()

    def rc(op, dt=1, dims=(4096,), **kw):
        return G.lib().gpuos_op_ntiles(_desc(G, op, dt, dims, **kw).ctypes.data, C.byref(n))

    for op in ("add", "mul", "relu", "gelu"):
        for dt in (0, 1):
            assert rc(op, dt) == G.OK
            assert rc(op, dt, a=0) == G.EINVAL
            assert rc(op, dt, out=0) == G.EINVAL
            assert rc(op, 5) == G.EINVAL                          # dtype
            assert rc(op, dt, dims=(0,), a=0, b=0, out=0) == G.OK  # empty: nothing is read
            assert n.value == 1
    assert rc("add", b=0) == G.EINVAL and rc("mul", b=0) == G.EINVAL
    assert rc("relu", b=0) == G.OK and rc("gelu", b=0) == G.OK      # unary: b unused
    d = _desc(G, "add", 1, (4096,))
    d["flags"] = 4                                                 # unknown flag bit
    assert G.lib().gpuos_op_ntiles(d.ctypes.data, C.byref(n)) == G.EINVAL
    d["flags"] = 1 | 2                                             # FENCE | DEP_REL
    assert G.lib().gpuos_op_ntiles(d.ctypes.data, C.byref(n)) == G.OK


def test_sdpa_workspace_formula_matches_stream_layout(G):
    from workloads.streams import sdpa_workspace_bytes
    for B, H, L in ((1, 32, 4096), (8, 32, 4096), (3, 4, 513), (2, 1, 1)):
        assert G.sdpa_workspace_bytes(B, H, 128, L) == sdpa_workspace_bytes(B, H, 128, L)


def test_strerror_and_clock(G):
    assert "ring full" in G.strerror(G.EAGAIN)
    assert "dependency" in G.strerror(G.ST_DEP_TIMEOUT, True)
    t0 = G.host_now_ns()
    t1 = G.host_now_ns()
    assert t1 >= t0 > 0


def test_init_without_gpu_fails_cleanly(G):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    ctx = C.c_void_p()
    cfg = G.default_config()
    rc = G.lib().gpuos_init(C.byref(cfg), C.byref(ctx))
    assert rc in (G.ECUDA, G.ENOMEM) and not ctx.value


def test_init_rejects_bad_config(G):
    ctx = C.c_void_p()
    for kw in (dict(ring_entries=100), dict(ring_entries=32), dict(warps_per_block=1),
               dict(tq_entries=1000), dict(tq_entries=1 << 18), dict(backoff_min_ns=0),
               dict(stage_bytes=1000), dict(stage_bytes=32768),
               dict(warps_per_block=13),                             # > 12 warps (168 registers each)
               dict(warps_per_block=12, stage_bytes=24576)):  # 12 x 24 KB staging > 227 KB
        cfg = G.default_config(**kw)
        assert G.lib().gpuos_init(C.byref(cfg), C.byref(ctx)) == G.EINVAL, kw
