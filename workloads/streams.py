"""Seeded synthetic descriptor streams for the persistent micro-op dispatcher.

This module is the only code shared by the CPU oracle and the CUDA path. It
holds input generation and the data layout of each stream, and none of the
arithmetic of the micro-ops: it draws buffers (NumPy PCG64, fixed seeds),
lays out operands, records which earlier descriptors each descriptor depends
on, and checks that those dependencies order every conflicting pair of
accesses (the hazard checker). Both sides materialise the same buffers from
the arrays built here and then apply the same list of ``Op`` records.

Streams follow the five workloads of the GPUOS evaluation ("GPUOS: A GPU
Operating System Primitive for Transparent Operation Fusion", §3 Q3, Table 2:
element-wise, attention decoding and mixed pipeline) at the sizes fixed for
this build:

* ``c1``  smallest stream: fp32 add/mul/ReLU on 4,096-element tensors.
* ``c2``  variable-shape element-wise stream, 30 % chained.
* ``c2l`` the same ops on large tensors (64 K .. 1 M elements), unchained.
* ``c3``  row softmax / LayerNorm / row sum, max, min.
* ``c4``  decode attention: RoPE -> KV-cache slot write -> decode SDPA.
* ``c5``  a synthetic 32-layer decoder, 7 chained micro-ops per layer.

Values written "N(m, s)" below use the second number as the standard
deviation (``torch.normal(mean, std)`` convention).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

# ----------------------------------------------------------------------------
# Element types. bf16 values are stored as their raw uint16 bit patterns.
# ----------------------------------------------------------------------------
ESIZE = {"f32": 4, "bf16": 2, "i32": 4, "u8": 1}
NPTYPE = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32, "u8": np.uint8}

# Op names. Each side maps these to its own representation.
ELEMENTWISE = ("add", "mul", "relu", "gelu")
ROWOPS = ("softmax", "layernorm", "rowsum", "rowmax", "rowmin")
ALL_OPS = ELEMENTWISE + ROWOPS + ("rope", "kv_write", "sdpa", "vecmat", "nop")

# Decode attention splits each (request, head) into chunks of at least this
# many key positions; the CUDA path keeps one partial (m, l, 2 pad, acc[D])
# per chunk in a caller-provided fp32 workspace after one uint32 counter per
# (request, head). The layout is part of the descriptor contract.
SDPA_CHUNK_MIN = 32

# Canary byte written into every output arena before a run; bytes that no op
# writes must still hold it afterwards.
CANARY_BYTE = 0x5A


def sdpa_workspace_bytes(B: int, H: int, D: int, Lmax: int) -> int:
    """Bytes of the split-K workspace of decode-SDPA descriptors with at most
    B requests: B*H uint32 counters (rounded up to 4), then one fp32 partial
    (m, l, 2 pad, acc[D]) per (request, head, chunk) at the finest split."""
    nch = max(1, -(-Lmax // SDPA_CHUNK_MIN))
    return 4 * ((B * H + 3) // 4 * 4) + 4 * (B * H * nch * (D + 4))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even), returned as uint16.

    Used only to build bf16 *inputs* from float32 normal draws. Inputs are
    finite, so NaN handling is not needed here.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    # in 32-bit arithmetic: for a finite binary32 pattern (at most 0xFF7FFFFF)
    # adding at most 0x8000 cannot wrap
    r = u >> np.uint32(16)
    r &= np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# Stream records
# ----------------------------------------------------------------------------
@dataclass
class Buf:
    """A buffer: host initial contents (``data``) or a fill byte (outputs)."""

    name: str
    dtype: str
    nelem: int
    data: Optional[np.ndarray] = None  # storage dtype NPTYPE[dtype]
    fill: int = CANARY_BYTE  # used when data is None

    @property
    def nbytes(self) -> int:
        return self.nelem * ESIZE[self.dtype]

    def materialize(self) -> np.ndarray:
        """Host array with the buffer's initial contents (a fresh copy)."""
        if self.data is not None:
            return np.array(self.data, dtype=NPTYPE[self.dtype], copy=True)
        raw = np.full(self.nbytes, self.fill, dtype=np.uint8)
        return raw.view(NPTYPE[self.dtype])


@dataclass(frozen=True)
class Ref:
    buf: int  # index into Stream.buffers
    off: int = 0  # element offset


@dataclass
class Op:
    """One descriptor. Field meanings per op are listed in ``OP_FIELDS``."""

    op: str
    dtype: str = "bf16"
    a: Optional[Ref] = None
    b: Optional[Ref] = None
    out: Optional[Ref] = None
    aux0: Optional[Ref] = None
    aux1: Optional[Ref] = None
    aux2: Optional[Ref] = None
    dims: Tuple[int, ...] = ()
    fparam: Tuple[float, ...] = ()
    deps: Tuple[int, ...] = ()  # indices of earlier ops in the stream
    fence: bool = False  # wait for every earlier op


# Operand roles per op (the descriptor layout shared by both sides):
#   add/mul   a[n], b[n] -> out[n]                 dims=(n,)        dtype f32|bf16
#   relu/gelu a[n] -> out[n]                       dims=(n,)        dtype f32|bf16
#   softmax   a=x[R,H] -> out[R,H]                 dims=(R,H)       bf16
#   layernorm a=x[R,H], b=gamma[H], aux0=beta[H] -> out[R,H]; dims=(R,H), fparam=(eps,)
#   rowsum    a=x[R,H] -> out f32[R]; rowmax/rowmin -> out bf16[R]
#   rope      a=q[B,H,D], b=k[B,H,D] rotated in place, aux0=lens i32[B]
#             (position = lens[b]-1); dims=(B,H,D), fparam=(theta,)
#   kv_write  a=k[B,H,D], b=v[B,H,D], aux0=lens i32[B], out=Kc, aux1=Vc with
#             caches laid out [B][H][Lcap][D]; row lens[b]-1 is written.
#             dims=(B,H,D,Lcap)
#   sdpa      a=q[B,H,D], b=Kc, aux1=Vc, aux0=lens i32[B], out=o[B,H,D],
#             aux2=workspace (sdpa_workspace_bytes of the largest B);
#             dims=(B,H,D,Lcap,Lmax,Ccap) with every lens[b] <= Lmax <= Lcap and
#             Ccap = counters reserved at the workspace start (>= B*H, the same
#             for every descriptor sharing the workspace); fparam=(scale,)
#   vecmat    a=x[K], b=W[K,N] row-major -> out=y[N]; dims=(K,N)
#   nop       no operands
OP_FIELDS = ("a", "b", "out", "aux0", "aux1", "aux2")


@dataclass
class Stream:
    name: str
    buffers: List[Buf] = field(default_factory=list)
    ops: List[Op] = field(default_factory=list)
    meta: Dict[str, object] = field(default_factory=dict)

    def add_buf(self, name: str, dtype: str, nelem: int, data=None, fill=CANARY_BYTE) -> int:
        if data is not None:
            data = np.ascontiguousarray(data, dtype=NPTYPE[dtype]).reshape(-1)
            assert data.size == nelem, (name, data.size, nelem)
        self.buffers.append(Buf(name, dtype, int(nelem), data, fill))
        return len(self.buffers) - 1

    def buf_index(self, name: str) -> int:
        for i, b in enumerate(self.buffers):
            if b.name == name:
                return i
        raise KeyError(name)


# ----------------------------------------------------------------------------
# Access extents (element ranges per buffer) for the hazard checker and the
# canary check. Layout only: no arithmetic of the ops.
# ----------------------------------------------------------------------------
def op_accesses(s: Stream, o: Op) -> List[Tuple[int, int, int, bool]]:
    """List of (buf, lo, hi, is_write) element ranges touched by ``o``."""
    acc: List[Tuple[int, int, int, bool]] = []

    def R(ref: Optional[Ref], n: int, w: bool = False):
        if ref is not None and n > 0:
            acc.append((ref.buf, ref.off, ref.off + n, w))

    d = o.dims
    if o.op in ("add", "mul"):
        R(o.a, d[0]); R(o.b, d[0]); R(o.out, d[0], True)
    elif o.op in ("relu", "gelu"):
        R(o.a, d[0]); R(o.out, d[0], True)
    elif o.op in ("softmax",):
        R(o.a, d[0] * d[1]); R(o.out, d[0] * d[1], True)
    elif o.op == "layernorm":
        R(o.a, d[0] * d[1]); R(o.b, d[1]); R(o.aux0, d[1]); R(o.out, d[0] * d[1], True)
    elif o.op in ("rowsum", "rowmax", "rowmin"):
        R(o.a, d[0] * d[1]); R(o.out, d[0], True)
    elif o.op == "rope":
        B, H, D = d[:3]
        R(o.aux0, B); R(o.a, B * H * D); R(o.b, B * H * D)
        R(o.a, B * H * D, True); R(o.b, B * H * D, True)
    elif o.op == "kv_write":
        B, H, D, Lc = d[:4]
        R(o.a, B * H * D); R(o.b, B * H * D); R(o.aux0, B)
        R(o.out, B * H * Lc * D, True); R(o.aux1, B * H * Lc * D, True)
    elif o.op == "sdpa":
        B, H, D, Lc, Lm, Cc = d[:6]
        R(o.a, B * H * D); R(o.aux0, B)
        R(o.b, B * H * Lc * D); R(o.aux1, B * H * Lc * D)
        R(o.out, B * H * D, True)
        if o.aux2 is not None:
            ws = sdpa_workspace_bytes(max(B, Cc // H), H, D, Lm)
            R(o.aux2, ws); R(o.aux2, ws, True)
    elif o.op == "vecmat":
        K, N = d[:2]
        R(o.a, K); R(o.b, K * N); R(o.out, N, True)
    elif o.op == "nop":
        pass
    else:
        raise ValueError(o.op)
    return acc


def check_hazards(s: Stream) -> None:
    """Assert that declared deps/fences order every conflicting access pair.

    Two accesses conflict when their element ranges overlap in the same
    buffer and at least one writes. Each new access is compared with the live
    earlier accesses it overlaps (a write that fully covers an earlier record
    retires it, since ordering against the newer write implies ordering
    against the older one). The earlier op must be an ancestor of the later
    one through ``deps`` (transitively) or a fence.
    """
    BUCKET = 1 << 16

    def is_ancestor(i: int, j: int) -> bool:
        stack = [j]
        seen = set()
        while stack:
            k = stack.pop()
            if k == i:
                return True
            if k in seen or k < i:
                continue
            seen.add(k)
            if s.ops[k].fence and k > i:
                return True
            stack.extend(s.ops[k].deps)
        return False

    # buckets[(buf, bucket)] -> list of records [lo, hi, op, is_write, alive]
    buckets: Dict[Tuple[int, int], List[list]] = {}
    for j, o in enumerate(s.ops):
        for (b, lo, hi, w) in op_accesses(s, o):
            seen_rec = set()
            for k in range(lo // BUCKET, (hi - 1) // BUCKET + 1):
                lst = buckets.get((b, k))
                if not lst:
                    continue
                alive = []
                for r in lst:
                    if not r[4]:
                        continue
                    rlo, rhi, i, rw, _ = r
                    if id(r) not in seen_rec and rlo < hi and lo < rhi and i != j and (w or rw):
                        seen_rec.add(id(r))
                        if not is_ancestor(i, j):
                            raise AssertionError(
                                f"{s.name}: op {j} ({o.op}) conflicts with op {i} "
                                f"({s.ops[i].op}) on buffer {s.buffers[b].name} "
                                f"without an ordering dependency")
                    if w and i != j and lo <= rlo and rhi <= hi:
                        r[4] = False
                        continue
                    alive.append(r)
                buckets[(b, k)] = alive
            rec = [lo, hi, j, w, True]
            for k in range(lo // BUCKET, (hi - 1) // BUCKET + 1):
                buckets.setdefault((b, k), []).append(rec)


# ----------------------------------------------------------------------------
# Generators
# ----------------------------------------------------------------------------
def _pool(rng: np.random.Generator, nelem: int, dtype: str, std: float = 1.0, mean: float = 0.0):
    x = rng.standard_normal(nelem, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return x if dtype == "f32" else f32_to_bf16_bits(x)


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


class _Arena:
    """Bump allocator over one output buffer with a guard band per output."""

    def __init__(self, align: int = 256, guard: int = 64):
        self.top = 0
        self.align = align
        self.guard = guard

    def take(self, n: int) -> int:
        off = self.top
        self.top = _round_up(off + n + self.guard, self.align)
        return off


def stream_c1(n_desc: int = 1000, n: int = 4096, seed: int = 1) -> Stream:
    """Smallest stream: fp32 add/mul/ReLU on contiguous n-element tensors."""
    rng = np.random.default_rng(seed)
    s = Stream("c1", meta=dict(seed=seed, n_desc=n_desc, n=n))
    kinds = rng.integers(0, 3, size=n_desc)
    stride = _round_up(n, 256)
    ia = s.add_buf("a", "f32", n_desc * stride, _pool(rng, n_desc * stride, "f32"))
    ib = s.add_buf("b", "f32", n_desc * stride, _pool(rng, n_desc * stride, "f32"))
    arena = _Arena()
    offs = [arena.take(n) for _ in range(n_desc)]
    io = s.add_buf("out", "f32", arena.top)
    for i in range(n_desc):
        op = ("add", "mul", "relu")[int(kinds[i])]
        s.ops.append(Op(op, "f32", a=Ref(ia, i * stride),
                        b=Ref(ib, i * stride) if op != "relu" else None,
                        out=Ref(io, offs[i]), dims=(n,)))
    return s


def stream_elementwise(name: str, n_desc: int, n_lo: int, n_hi: int, chain_frac: float,
                       pool_elems: int, seed: int) -> Stream:
    """Element-wise stream over {add, mul, ReLU, GELU} x {fp32, bf16}.

    Sizes are log-uniform in [n_lo, n_hi]. With probability ``chain_frac`` a
    descriptor consumes the previous descriptor's output: it inherits that
    dtype and reads a prefix of length min(n_draw, n_prev). Other inputs are
    slices at random 256-element-aligned offsets of an N(0,1) pool (one per
    dtype) much larger than L2; every output goes to a fresh region of an
    output arena with a canary guard band after it.
    """
    rng = np.random.default_rng(seed)
    s = Stream(name, meta=dict(seed=seed, n_desc=n_desc, n_lo=n_lo, n_hi=n_hi,
                               chain_frac=chain_frac, pool_elems=pool_elems))
    pf = s.add_buf("pool_f32", "f32", pool_elems, _pool(rng, pool_elems, "f32"))
    pb = s.add_buf("pool_bf16", "bf16", pool_elems, _pool(rng, pool_elems, "bf16"))
    kinds = rng.integers(0, 4, size=n_desc)
    dts = rng.integers(0, 2, size=n_desc)
    ns = np.exp(rng.uniform(math.log(n_lo), math.log(n_hi), size=n_desc)).astype(np.int64)
    ns = np.clip(ns, n_lo, n_hi)
    chained = rng.random(n_desc) < chain_frac
    chained[0] = False
    arena = {"f32": _Arena(), "bf16": _Arena()}
    recs = []  # (op, dtype, a_ref_kind, a_off, b_off, out_off, n, dep)
    prev = None  # (dtype, out_off, n, index)
    for i in range(n_desc):
        op = ELEMENTWISE[int(kinds[i])]
        n = int(ns[i])
        if chained[i] and prev is not None:
            dt, a_off, pn, pidx = prev
            n = min(n, pn)
            a_src = ("out", a_off)
            dep = (pidx,)
        else:
            dt = ("f32", "bf16")[int(dts[i])]
            a_src = ("pool", int(rng.integers(0, (pool_elems - n) // 256 + 1)) * 256)
            dep = ()
        b_off = int(rng.integers(0, (pool_elems - n) // 256 + 1)) * 256 if op in ("add", "mul") else None
        out_off = arena[dt].take(n)
        recs.append((op, dt, a_src, b_off, out_off, n, dep))
        prev = (dt, out_off, n, i)
    of = s.add_buf("out_f32", "f32", max(arena["f32"].top, 256))
    ob = s.add_buf("out_bf16", "bf16", max(arena["bf16"].top, 256))
    pool_of = {"f32": pf, "bf16": pb}
    out_of = {"f32": of, "bf16": ob}
    for (op, dt, a_src, b_off, out_off, n, dep) in recs:
        a = Ref(out_of[dt], a_src[1]) if a_src[0] == "out" else Ref(pool_of[dt], a_src[1])
        b = Ref(pool_of[dt], b_off) if b_off is not None else None
        s.ops.append(Op(op, dt, a=a, b=b, out=Ref(out_of[dt], out_off), dims=(n,), deps=dep))
    return s


def stream_c2(n_desc: int = 100_000, pool_elems: int = 1 << 27, seed: int = 2) -> Stream:
    return stream_elementwise("c2", n_desc, 256, 65536, 0.30, pool_elems, seed)


def stream_c2l(n_desc: int = 4000, pool_elems: int = 1 << 27, seed: int = 6) -> Stream:
    return stream_elementwise("c2l", n_desc, 65536, 1 << 20, 0.0, pool_elems, seed)


def stream_c3(n_desc: int = 50_000, pool_elems: int = 1 << 27, seed: int = 3,
              hiddens: Sequence[int] = (1024, 2048, 4096), max_rows: int = 64) -> Stream:
    """Row-op stream: softmax, LayerNorm, row sum/max/min over bf16 [R, H].

    R ~ U{1..max_rows}, H uniform over ``hiddens``, x ~ N(0, 2) (std 2),
    gamma ~ N(1, 0.1), beta ~ N(0, 0.1) sliced per descriptor, eps = 1e-5.
    Ops are uniform over the five kinds.
    """
    rng = np.random.default_rng(seed)
    s = Stream("c3", meta=dict(seed=seed, n_desc=n_desc, pool_elems=pool_elems))
    px = s.add_buf("pool_x", "bf16", pool_elems, _pool(rng, pool_elems, "bf16", std=2.0))
    gpool = 1 << 20
    pg = s.add_buf("pool_gamma", "bf16", gpool, _pool(rng, gpool, "bf16", std=0.1, mean=1.0))
    pbeta = s.add_buf("pool_beta", "bf16", gpool, _pool(rng, gpool, "bf16", std=0.1))
    kinds = rng.integers(0, 5, size=n_desc)
    rows = rng.integers(1, max_rows + 1, size=n_desc)
    hs = np.asarray(hiddens)[rng.integers(0, len(hiddens), size=n_desc)]
    ab, af = _Arena(), _Arena()
    recs = []
    for i in range(n_desc):
        op = ROWOPS[int(kinds[i])]
        R, H = int(rows[i]), int(hs[i])
        x_off = int(rng.integers(0, (pool_elems - R * H) // 256 + 1)) * 256
        if op in ("softmax", "layernorm"):
            out = ("bf16", ab.take(R * H))
        elif op == "rowsum":
            out = ("f32", af.take(R))
        else:
            out = ("bf16", ab.take(R))
        g_off = int(rng.integers(0, (gpool - H) // 256 + 1)) * 256 if op == "layernorm" else None
        b_off = int(rng.integers(0, (gpool - H) // 256 + 1)) * 256 if op == "layernorm" else None
        recs.append((op, R, H, x_off, out, g_off, b_off))
    ob = s.add_buf("out_bf16", "bf16", max(ab.top, 256))
    of = s.add_buf("out_f32", "f32", max(af.top, 256))
    for (op, R, H, x_off, out, g_off, b_off) in recs:
        o = Op(op, "bf16", a=Ref(px, x_off),
               out=Ref(ob if out[0] == "bf16" else of, out[1]), dims=(R, H))
        if op == "layernorm":
            o.b = Ref(pg, g_off)
            o.aux0 = Ref(pbeta, b_off)
            o.fparam = (1e-5,)
        s.ops.append(o)
    return s


def stream_c4(n_steps: int = 2000, B_max: int = 8, H: int = 32, D: int = 128, Lcap: int = 4096,
              L_lo: int = 128, seed: int = 4, theta: float = 10000.0) -> Stream:
    """Decode-attention micro-batch: per step RoPE -> KV write -> SDPA.

    Each step draws B ~ U{1..B_max}; fresh q, k, v [B, H, D] ~ N(0,1) bf16;
    per-request lengths L ~ U[L_lo, Lcap]. The new token is written at row
    L-1 of the caches (prefilled once with N(0,1) bf16, laid out
    [B_max][H][Lcap][D]) and attention covers rows 0..L-1.

    Dependencies: KV write waits for the step's RoPE (reads the rotated k)
    and for the previous step's SDPA (it may overwrite a row that SDPA read);
    SDPA waits for the step's KV write.
    """
    rng = np.random.default_rng(seed)
    s = Stream("c4", meta=dict(seed=seed, n_steps=n_steps, B_max=B_max, H=H, D=D, Lcap=Lcap))
    cache_n = B_max * H * Lcap * D
    ik = s.add_buf("Kc", "bf16", cache_n, _pool(rng, cache_n, "bf16"))
    iv = s.add_buf("Vc", "bf16", cache_n, _pool(rng, cache_n, "bf16"))
    Bs = rng.integers(1, B_max + 1, size=n_steps)
    row = H * D
    qkv_total = int(Bs.sum()) * row
    iq = s.add_buf("q", "bf16", qkv_total, _pool(rng, qkv_total, "bf16"))
    ikn = s.add_buf("k_new", "bf16", qkv_total, _pool(rng, qkv_total, "bf16"))
    ivn = s.add_buf("v_new", "bf16", qkv_total, _pool(rng, qkv_total, "bf16"))
    lens = np.concatenate([rng.integers(L_lo, Lcap + 1, size=int(b)) for b in Bs]).astype(np.int32)
    il = s.add_buf("lens", "i32", lens.size, lens)
    io = s.add_buf("o", "bf16", qkv_total)
    ws = s.add_buf("sdpa_ws", "u8", sdpa_workspace_bytes(B_max, H, D, Lcap), fill=0)
    scale = 1.0 / math.sqrt(D)
    qoff = 0
    loff = 0
    prev_sdpa = None
    for t in range(n_steps):
        B = int(Bs[t])
        Lm = int(lens[loff:loff + B].max())
        r = len(s.ops)
        s.ops.append(Op("rope", "bf16", a=Ref(iq, qoff), b=Ref(ikn, qoff), aux0=Ref(il, loff),
                        dims=(B, H, D), fparam=(theta,)))
        deps = (r,) if prev_sdpa is None else (r, prev_sdpa)
        s.ops.append(Op("kv_write", "bf16", a=Ref(ikn, qoff), b=Ref(ivn, qoff), aux0=Ref(il, loff),
                        out=Ref(ik, 0), aux1=Ref(iv, 0), dims=(B, H, D, Lcap), deps=deps))
        s.ops.append(Op("sdpa", "bf16", a=Ref(iq, qoff), b=Ref(ik, 0), aux1=Ref(iv, 0),
                        aux0=Ref(il, loff), out=Ref(io, qoff), aux2=Ref(ws, 0),
                        dims=(B, H, D, Lcap, Lm, B_max * H), fparam=(scale,), deps=(r + 1,)))
        prev_sdpa = r + 2
        qoff += B * row
        loff += B
    return s


def stream_c5(n_tokens: int = 500, n_layers: int = 32, hidden: int = 4096, H: int = 32, D: int = 128,
              Lcap: int = 4096, vm: int = 1024, seed: int = 5, theta: float = 10000.0,
              L_lo: int = 256, walk: int = 32) -> Stream:
    """Mixed pipeline: a synthetic decoder, one strict chain of 7 ops per layer.

    Per token and layer: LayerNorm(x) -> h; vecmat(h[:vm], W_l) -> y;
    RoPE(q_t, k_t) at position L-1; KV write of (k_t, v_t) into the layer's
    caches at row L-1; SDPA(q_t, caches, L) -> o; GELU(o) -> g; residual add
    x' = x + g. Every op depends on the op before it. The 1 x vm vecmat cannot
    produce the H*D-wide projections, so q_t, k_t, v_t are fresh N(0,1) inputs
    per token and layer (synthetic glue), and y is an output of its own. L
    follows a random walk L_{t+1} = clamp(L_t + U{-walk..walk}, L_lo, Lcap)
    shared by all layers of a token. Weights W ~ N(0, 0.02), gamma ~ N(1, 0.1),
    beta ~ N(0, 0.1); caches prefilled with N(0,1).
    """
    assert H * D == hidden
    rng = np.random.default_rng(seed)
    s = Stream("c5", meta=dict(seed=seed, n_tokens=n_tokens, n_layers=n_layers, hidden=hidden))
    nl = n_layers
    iW = s.add_buf("W", "bf16", nl * vm * vm, _pool(rng, nl * vm * vm, "bf16", std=0.02))
    ig = s.add_buf("gamma", "bf16", nl * hidden, _pool(rng, nl * hidden, "bf16", std=0.1, mean=1.0))
    ib = s.add_buf("beta", "bf16", nl * hidden, _pool(rng, nl * hidden, "bf16", std=0.1))
    cache_n = H * Lcap * D
    iK = s.add_buf("Kc", "bf16", nl * cache_n, _pool(rng, nl * cache_n, "bf16"))
    iV = s.add_buf("Vc", "bf16", nl * cache_n, _pool(rng, nl * cache_n, "bf16"))
    kv_n = n_tokens * nl * hidden
    iqn = s.add_buf("q_new", "bf16", kv_n, _pool(rng, kv_n, "bf16"))
    ik = s.add_buf("k_new", "bf16", kv_n, _pool(rng, kv_n, "bf16"))
    iv = s.add_buf("v_new", "bf16", kv_n, _pool(rng, kv_n, "bf16"))
    ix = s.add_buf("x", "bf16", (n_tokens * nl + 1) * hidden, fill=0)
    x0 = _pool(rng, hidden, "bf16")
    s.buffers[ix].data = np.zeros((n_tokens * nl + 1) * hidden, dtype=np.uint16)
    s.buffers[ix].data[:hidden] = x0
    Ls = np.empty(n_tokens, dtype=np.int32)
    L = int(rng.integers(L_lo, Lcap + 1))
    for t in range(n_tokens):
        Ls[t] = L
        L = int(np.clip(L + int(rng.integers(-walk, walk + 1)), L_lo, Lcap))
    il = s.add_buf("lens", "i32", n_tokens, Ls)
    ih = s.add_buf("h", "bf16", n_tokens * nl * hidden)
    iy = s.add_buf("y", "bf16", n_tokens * nl * vm)
    io = s.add_buf("o", "bf16", n_tokens * nl * hidden)
    igl = s.add_buf("g", "bf16", n_tokens * nl * hidden)
    ws = s.add_buf("sdpa_ws", "u8", sdpa_workspace_bytes(1, H, D, Lcap), fill=0)
    scale = 1.0 / math.sqrt(D)
    for t in range(n_tokens):
        Lt = int(Ls[t])
        for l in range(nl):
            u = t * nl + l
            hx = u * hidden
            base = len(s.ops)
            dep0 = (base - 1,) if base > 0 else ()
            s.ops.append(Op("layernorm", "bf16", a=Ref(ix, hx), b=Ref(ig, l * hidden),
                            aux0=Ref(ib, l * hidden), out=Ref(ih, hx), dims=(1, hidden),
                            fparam=(1e-5,), deps=dep0))
            s.ops.append(Op("vecmat", "bf16", a=Ref(ih, hx), b=Ref(iW, l * vm * vm),
                            out=Ref(iy, u * vm), dims=(vm, vm), deps=(base,)))
            s.ops.append(Op("rope", "bf16", a=Ref(iqn, hx), b=Ref(ik, hx), aux0=Ref(il, t),
                            dims=(1, H, D), fparam=(theta,), deps=(base + 1,)))
            s.ops.append(Op("kv_write", "bf16", a=Ref(ik, hx), b=Ref(iv, hx), aux0=Ref(il, t),
                            out=Ref(iK, l * cache_n), aux1=Ref(iV, l * cache_n),
                            dims=(1, H, D, Lcap), deps=(base + 2,)))
            s.ops.append(Op("sdpa", "bf16", a=Ref(iqn, hx), b=Ref(iK, l * cache_n),
                            aux1=Ref(iV, l * cache_n), aux0=Ref(il, t), out=Ref(io, hx),
                            aux2=Ref(ws, 0), dims=(1, H, D, Lcap, Lt, H), fparam=(scale,),
                            deps=(base + 3,)))
            s.ops.append(Op("gelu", "bf16", a=Ref(io, hx), out=Ref(igl, hx), dims=(hidden,),
                            deps=(base + 4,)))
            s.ops.append(Op("add", "bf16", a=Ref(ix, hx), b=Ref(igl, hx), out=Ref(ix, hx + hidden),
                            dims=(hidden,), deps=(base + 5,)))
    return s


STREAMS = {
    "c1": stream_c1,
    "c2": stream_c2,
    "c2l": stream_c2l,
    "c3": stream_c3,
    "c4": stream_c4,
    "c5": stream_c5,
}


def op_bytes(o: Op) -> int:
    """Algorithmic HBM bytes of one op: unique reads and writes counted once."""
    d = o.dims
    e = ESIZE[o.dtype]
    if o.op in ("add", "mul"):
        return 3 * d[0] * e
    if o.op in ("relu", "gelu"):
        return 2 * d[0] * e
    if o.op == "softmax":
        return 2 * d[0] * d[1] * 2
    if o.op == "layernorm":
        return 2 * d[0] * d[1] * 2 + 2 * d[1] * 2
    if o.op == "rowsum":
        return d[0] * d[1] * 2 + 4 * d[0]
    if o.op in ("rowmax", "rowmin"):
        return d[0] * d[1] * 2 + 2 * d[0]
    if o.op == "rope":
        B, H, D = d[:3]
        return 2 * (2 * B * H * D * 2) + 4 * B
    if o.op == "kv_write":
        B, H, D = d[:3]
        return 2 * (2 * B * H * D * 2) + 4 * B
    if o.op == "vecmat":
        K, N = d[:2]
        return K * N * 2 + K * 2 + N * 2
    if o.op == "nop":
        return 0
    raise ValueError(o.op)


def sdpa_bytes(o: Op, lens: np.ndarray) -> int:
    """Algorithmic bytes of a decode-SDPA op given its per-request lengths."""
    B, H, D = o.dims[:3]
    kv = int(np.asarray(lens[:B], dtype=np.int64).sum()) * H * D * 2 * 2
    return kv + 2 * B * H * D * 2 + 4 * B


def stream_bytes(s: Stream) -> int:
    """Total algorithmic bytes of a stream (SDPA uses the drawn lengths)."""
    tot = 0
    for o in s.ops:
        if o.op == "sdpa":
            lens = s.buffers[o.aux0.buf].data[o.aux0.off:o.aux0.off + o.dims[0]]
            tot += sdpa_bytes(o, lens)
        else:
            tot += op_bytes(o)
    return tot


def stream_mixed_small(seed: int = 7) -> Stream:
    """Every op kind once or twice at small sizes, with ragged tails and a
    multi-chunk attention head (a quick end-to-end check)."""
    rng = np.random.default_rng(seed)
    s = Stream("mixed_small", meta=dict(seed=seed))
    pf = s.add_buf("pool_f32", "f32", 1 << 16, _pool(rng, 1 << 16, "f32"))
    pb = s.add_buf("pool_bf16", "bf16", 1 << 16, _pool(rng, 1 << 16, "bf16"))
    px = s.add_buf("pool_x", "bf16", 1 << 16, _pool(rng, 1 << 16, "bf16", std=2.0))
    pg = s.add_buf("gamma", "bf16", 4096, _pool(rng, 4096, "bf16", std=0.1, mean=1.0))
    pbt = s.add_buf("beta", "bf16", 4096, _pool(rng, 4096, "bf16", std=0.1))
    B, H, D, Lc = 2, 4, 128, 1100
    iK = s.add_buf("Kc", "bf16", B * H * Lc * D, _pool(rng, B * H * Lc * D, "bf16"))
    iV = s.add_buf("Vc", "bf16", B * H * Lc * D, _pool(rng, B * H * Lc * D, "bf16"))
    iq = s.add_buf("q", "bf16", B * H * D, _pool(rng, B * H * D, "bf16"))
    ik = s.add_buf("k_new", "bf16", B * H * D, _pool(rng, B * H * D, "bf16"))
    iv = s.add_buf("v_new", "bf16", B * H * D, _pool(rng, B * H * D, "bf16"))
    il = s.add_buf("lens", "i32", B, np.array([1037, 3], np.int32))
    iW = s.add_buf("W", "bf16", 300 * 72, _pool(rng, 300 * 72, "bf16", std=0.05))
    of = s.add_buf("out_f32", "f32", 1 << 15)
    ob = s.add_buf("out_bf16", "bf16", 1 << 16)
    io = s.add_buf("o", "bf16", B * H * D)
    ws = s.add_buf("sdpa_ws", "u8", sdpa_workspace_bytes(B, H, D, Lc), fill=0)
    ea, eb = _Arena(), _Arena()
    for op, dt, n in (("add", "f32", 4097), ("mul", "bf16", 9001), ("relu", "f32", 7), ("gelu", "bf16", 255),
                      ("gelu", "f32", 2049), ("add", "bf16", 0)):
        pool = pf if dt == "f32" else pb
        out = (of, ea.take(n)) if dt == "f32" else (ob, eb.take(n))
        s.ops.append(Op(op, dt, a=Ref(pool, 256), b=Ref(pool, 8192) if op in ("add", "mul") else None,
                        out=Ref(*out), dims=(n,)))
    s.ops.append(Op("relu", "f32", a=Ref(of, 0), out=Ref(of, ea.take(4097)), dims=(4097,), deps=(0,)))
    for op, R, Hh in (("softmax", 3, 1000), ("layernorm", 2, 4096), ("rowsum", 5, 2048), ("rowmax", 4, 33),
                      ("rowmin", 1, 5000), ("softmax", 2, 6000)):
        o = Op(op, "bf16", a=Ref(px, 512), dims=(R, Hh))
        if op in ("softmax", "layernorm"):
            o.out = Ref(ob, eb.take(R * Hh))
        elif op == "rowsum":
            o.out = Ref(of, ea.take(R))
        else:
            o.out = Ref(ob, eb.take(R))
        if op == "layernorm":
            o.b, o.aux0, o.fparam = Ref(pg, 0), Ref(pbt, 0), (1e-5,)
        s.ops.append(o)
    s.ops.append(Op("vecmat", "bf16", a=Ref(pb, 64), b=Ref(iW, 0), out=Ref(ob, eb.take(72)), dims=(300, 72)))
    s.ops.append(Op("vecmat", "bf16", a=Ref(pb, 64), b=Ref(iW, 0), out=Ref(ob, eb.take(36)), dims=(600, 36)))
    r = len(s.ops)
    s.ops.append(Op("rope", "bf16", a=Ref(iq, 0), b=Ref(ik, 0), aux0=Ref(il, 0), dims=(B, H, D), fparam=(10000.0,)))
    s.ops.append(Op("kv_write", "bf16", a=Ref(ik, 0), b=Ref(iv, 0), aux0=Ref(il, 0), out=Ref(iK, 0),
                    aux1=Ref(iV, 0), dims=(B, H, D, Lc), deps=(r,)))
    s.ops.append(Op("sdpa", "bf16", a=Ref(iq, 0), b=Ref(iK, 0), aux1=Ref(iV, 0), aux0=Ref(il, 0), out=Ref(io, 0),
                    aux2=Ref(ws, 0), dims=(B, H, D, Lc, 1037, B * H), fparam=(1.0 / math.sqrt(D),),
                    deps=(r + 1,)))
    # ragged head groups (6 = 4 + 2 and 5 = 4 + 1 heads), the element-pair
    # RoPE and element KV paths (D = 66), and a vecmat whose last tile holds
    # 8 of 16 columns, on the staged path (K % 8 == 0, aligned operands)
    for tag, (Bx, Hx, Dx, Lcx, lens) in (("2", (2, 6, 66, 40, [40, 17])), ("3", (1, 5, 64, 16, [9]))):
        nq = Bx * Hx * Dx
        jq = s.add_buf("q" + tag, "bf16", nq, _pool(rng, nq, "bf16"))
        jk = s.add_buf("k_new" + tag, "bf16", nq, _pool(rng, nq, "bf16"))
        jv = s.add_buf("v_new" + tag, "bf16", nq, _pool(rng, nq, "bf16"))
        nc = Bx * Hx * Lcx * Dx
        jK = s.add_buf("Kc" + tag, "bf16", nc, _pool(rng, nc, "bf16"))
        jV = s.add_buf("Vc" + tag, "bf16", nc, _pool(rng, nc, "bf16"))
        jl = s.add_buf("lens" + tag, "i32", Bx, np.array(lens, np.int32))
        r = len(s.ops)
        s.ops.append(Op("rope", "bf16", a=Ref(jq, 0), b=Ref(jk, 0), aux0=Ref(jl, 0), dims=(Bx, Hx, Dx),
                        fparam=(10000.0,)))
        s.ops.append(Op("kv_write", "bf16", a=Ref(jk, 0), b=Ref(jv, 0), aux0=Ref(jl, 0), out=Ref(jK, 0),
                        aux1=Ref(jV, 0), dims=(Bx, Hx, Dx, Lcx), deps=(r,)))
    iW2 = s.add_buf("W2", "bf16", 1024 * 40, _pool(rng, 1024 * 40, "bf16", std=0.05))
    s.ops.append(Op("vecmat", "bf16", a=Ref(pb, 1024), b=Ref(iW2, 0), out=Ref(ob, eb.take(40)), dims=(1024, 40)))
    s.ops.append(Op("nop", fence=True))
    return s
