"""Comparison rules between the CUDA path and the CPU oracle.

Tolerances (stated for the build; the pages give none):
  * integer, copy and order ops (KV write, row max/min, ReLU, fp32 and bf16
    add/mul on identical inputs): bit-exact;
  * fp32 results: |g - r| <= 1e-5 * max(|r|, 1e-3 * rms(r over the op));
  * bf16 results: |g - r_exact| <= max(2e-2, ulp_bf16(r_exact)), where
    r_exact is the oracle's unrounded (double) value; fp32-accumulated
    reductions that return fp32 (row sum) use 2e-2 + 1e-5 |r|.
An op whose inputs (produced by earlier ops) differ from the oracle's by a
rounding step is judged with the tolerance rule even if it is exact itself;
a first-order bound of that input difference carried through the op
(|d(a+b)| <= |da|+|db|, |d(ab)| <= |da||b|+|db||a|, |dGELU| <= 1.13|dx|,
the LayerNorm, softmax, vecmat and attention bounds in propagated_bound) is
added to its tolerance. The expected value is always the oracle's.

Widening is allowed only from producers that were themselves compared, and
passed, in the same report, and only for inputs read as they stood when the
consumer ran: if a differing input range has a writer that was not compared
(or failed), or a writer after the consumer that the reader cannot undo, the
consumer fails ("widening from an unchecked producer"). A reader (the
``gpu_read`` callable) may expose ``timed(buf) -> bool`` to say that it
returns a buffer as it stood right after the op being compared.
"""
from __future__ import annotations

import numpy as np

from workloads.streams import Op, Ref, Stream, bf16_bits_to_f32, op_accesses

EXACT_OPS = {"add", "mul", "relu", "rowmax", "rowmin", "kv_write", "nop"}


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(np.asarray(x, dtype=np.float64))
    ax = np.maximum(ax, 2.0 ** -126)
    e = np.floor(np.log2(ax))
    return 2.0 ** (e - 7)


def as_f64(vals: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_to_f32(vals).astype(np.float64)
    return np.asarray(vals).astype(np.float64)


class Report:
    def __init__(self):
        self.checked = 0
        self.exact = 0
        self.tol = 0
        self.ulp_branch = 0
        self.failures = []
        self.max_abs = 0.0
        self.max_rel = 0.0
        self.passed = set()  # ops compared in this report without a failure

    def fail(self, j, o, msg):
        if len(self.failures) < 20:
            self.failures.append(f"op {j} {o.op}/{o.dtype} dims={o.dims}: {msg}")
        else:
            self.failures.append("...")

    def ok(self):
        return not self.failures

    def summary(self):
        return (f"checked={self.checked} exact={self.exact} tol={self.tol} ulp_branch={self.ulp_branch} "
                f"max_abs={self.max_abs:.3g} max_rel={self.max_rel:.3g} failures={len(self.failures)}")


def written_buffers(s: Stream) -> set:
    w = getattr(s, "_written", None)
    if w is None:
        w = {b for o in s.ops for (b, lo, hi, wr) in op_accesses(s, o) if wr}
        s._written = w
    return w


_BUCKET = 1 << 16
_BIG = 8  # writes spanning more buckets than this are listed per buffer


def _write_index(s: Stream):
    """(buckets, big): small writes by (buffer, 64 K-element bucket), and
    writes spanning more than _BIG buckets by buffer; entries (lo, hi, op)."""
    idx = getattr(s, "_wr_index", None)
    if idx is None:
        buckets, big = {}, {}
        for i, o in enumerate(s.ops):
            for (bb, l2, h2, w) in op_accesses(s, o):
                if not w:
                    continue
                k0, k1 = l2 // _BUCKET, (h2 - 1) // _BUCKET
                if k1 - k0 > _BIG:
                    big.setdefault(bb, []).append((l2, h2, i))
                else:
                    for k in range(k0, k1 + 1):
                        buckets.setdefault((bb, k), []).append((l2, h2, i))
        idx = s._wr_index = (buckets, big)
    return idx


def _overlapping_writes(s: Stream, b: int, lo: int, hi: int):
    buckets, big = _write_index(s)
    for (l2, h2, i) in big.get(b, ()):
        if l2 < hi and lo < h2:
            yield i
    for k in range(lo // _BUCKET, (hi - 1) // _BUCKET + 1):
        for (l2, h2, i) in buckets.get((b, k), ()):
            if l2 < hi and lo < h2:
                yield i


def written_before(s: Stream, b: int, lo: int, hi: int, j: int) -> bool:
    """Does some op i < j write an element of [lo, hi) of buffer b?"""
    return any(i < j for i in _overlapping_writes(s, b, lo, hi))


def writers_of(s: Stream, b: int, lo: int, hi: int) -> list:
    """Every op that writes an element of [lo, hi) of buffer b, in order."""
    return sorted(set(_overlapping_writes(s, b, lo, hi)))


def _scratch(o: Op):
    """The op's scratch operand (decode attention's split-K workspace): the
    CUDA path's own working memory, whose contents are neither an input nor
    an output of the op's result (the oracle never touches it)."""
    return o.aux2 if o.op == "sdpa" else None


def operand_accesses(s: Stream, o: Op) -> list:
    """op_accesses without the op's scratch: the ranges its result reads and
    writes."""
    sc = _scratch(o)
    return [(b, lo, hi, w) for (b, lo, hi, w) in op_accesses(s, o)
            if not (sc is not None and b == sc.buf and lo == sc.off)]


def _differing_inputs(s: Stream, o: Op, gpu_read, mach) -> list:
    """Input ranges (buf, lo, hi) whose bytes differ between the GPU and the
    oracle. Inputs no earlier op wrote are identical by construction (the
    seeded inputs); others are compared as the reader returns them."""
    j = mach._op_index[id(o)]
    diff = []
    for (b, lo, hi, w) in operand_accesses(s, o):
        if w or not written_before(s, b, lo, hi, j):
            continue
        g = gpu_read(Ref(b, lo), hi - lo)
        r = mach.buf[b][lo:hi]
        if not np.array_equal(g.view(np.uint8), r.view(np.uint8)):
            diff.append((b, lo, hi))
    return diff


def _widening_sources_ok(rep: Report, s: Stream, j: int, o: Op, diff: list, gpu_read) -> bool:
    """Every differing input of op j must come from producers compared (and
    passed) in this report, read as it stood when op j ran."""
    timed = getattr(gpu_read, "timed", None)
    for (b, lo, hi) in diff:
        for i in writers_of(s, b, lo, hi):
            if i < j and i not in rep.passed:
                rep.fail(j, o, f"widening from an unchecked producer: op {i} ({s.ops[i].op}) "
                               f"writes buffer {s.buffers[b].name}")
                return False
            if i > j and not (timed is not None and timed(b)):
                rep.fail(j, o, f"widening from an unchecked producer: input buffer {s.buffers[b].name} "
                               f"is rewritten after the op by op {i} ({s.ops[i].op})")
                return False
    return True


def check_bf16(rep, j, o, g_bits, r_exact, extra_abs=0.0):
    g = as_f64(g_bits, "bf16")
    err = np.abs(g - r_exact)
    bound = np.maximum(2e-2, ulp_bf16(r_exact)) + extra_abs
    rep.ulp_branch += int(np.count_nonzero((err > 2e-2 + extra_abs) & (err <= bound)))
    bad = ~(err <= bound)
    rep.max_abs = max(rep.max_abs, float(err.max(initial=0.0)))
    if bad.any():
        k = int(np.argmax(bad))
        rep.fail(j, o, f"bf16 mismatch at {k}: gpu={g[k]!r} exact={r_exact[k]!r} err={err[k]:.3g} "
                       f"bound={bound[k] if np.ndim(bound) else bound:.3g} ({int(bad.sum())} bad)")
        return False
    return True


def check_f32(rep, j, o, g, r_exact, abs_floor=None, extra_rel=0.0):
    g = np.asarray(g, dtype=np.float64)
    err = np.abs(g - r_exact)
    rms = float(np.sqrt(np.mean(r_exact ** 2))) if r_exact.size else 0.0
    floor = 1e-3 * rms if abs_floor is None else abs_floor
    bound = (1e-5 + extra_rel) * np.maximum(np.abs(r_exact), floor)
    bad = ~(err <= bound)
    rel = err / np.maximum(np.abs(r_exact), 1e-30)
    rep.max_rel = max(rep.max_rel, float(rel.max(initial=0.0)))
    rep.max_abs = max(rep.max_abs, float(err.max(initial=0.0)))
    if bad.any():
        k = int(np.argmax(bad))
        rep.fail(j, o, f"fp32 mismatch at {k}: gpu={g[k]!r} exact={r_exact[k]!r} ({int(bad.sum())} bad)")
        return False
    return True


def _delta(s: Stream, ref, n: int, dtype: str, gpu_read, mach, j: int = None) -> np.ndarray:
    """|GPU input - oracle input| over n elements at ref (0 if no earlier op
    wrote them)."""
    if ref is None or n == 0:
        return np.zeros(n)
    if ref.buf not in written_buffers(s) or (j is not None and not written_before(s, ref.buf, ref.off, ref.off + n, j)):
        return np.zeros(n)
    g = as_f64(gpu_read(ref, n), dtype)
    r = as_f64(mach.view(ref, n), dtype)
    return np.abs(g - r)


def propagated_bound(s: Stream, o: Op, gpu_read, mach):
    """First-order bound on how much the op's exact result moves because its
    inputs (outputs of earlier ops) differ between the two sides by their own
    rounding. Returns an array shaped like the op's output (or 0)."""
    d = o.dims
    j = mach._op_index[id(o)]
    D = lambda ref, n, dt="bf16": _delta(s, ref, n, dt, gpu_read, mach, j)  # noqa: E731
    if o.op in ("add", "mul", "relu", "gelu"):
        n = d[0]
        da = D(o.a, n, o.dtype)
        if o.op == "add":
            return da + D(o.b, n, o.dtype)
        if o.op == "mul":
            db = D(o.b, n, o.dtype)
            a = np.abs(as_f64(mach.view(o.a, n), o.dtype))
            b = np.abs(as_f64(mach.view(o.b, n), o.dtype))
            return da * b + db * (a + da)
        return da * (1.0 if o.op == "relu" else 1.13)  # max |GELU'| < 1.13
    if o.op in ("softmax", "layernorm", "rowsum", "rowmax", "rowmin"):
        R, H = d[:2]
        dx = D(o.a, R * H).reshape(R, H)
        if o.op == "rowsum":
            return dx.sum(1)
        if o.op in ("rowmax", "rowmin"):
            return dx.max(1)
        if o.op == "softmax":
            y = np.abs(mach.exact[mach_index(mach, o)]["out"]).reshape(R, H)
            return (2.0 * dx.max(1, keepdims=True) * y).reshape(-1)
        x = as_f64(mach.view(o.a, R * H), "bf16").reshape(R, H)
        g = np.abs(as_f64(mach.view(o.b, H), "bf16"))
        mu = x.mean(1, keepdims=True)
        sd = np.sqrt(x.var(1, keepdims=True) + float(o.fparam[0]))
        m1 = dx.mean(1, keepdims=True)
        rms = np.sqrt((dx ** 2).mean(1, keepdims=True))
        return (g / sd * (dx + m1 + np.abs(x - mu) / sd * (rms + m1)) * 1.01).reshape(-1)
    if o.op == "vecmat":
        K, N = d[:2]
        dx = D(o.a, K)
        W = np.abs(as_f64(mach.view(o.b, K * N), "bf16").reshape(K, N))
        return dx @ W
    if o.op == "sdpa":
        B, H, Dh, Lc = d[:4]
        lens = mach.view(o.aux0, B)
        dq = D(o.a, B * H * Dh).reshape(B, H, Dh)
        q = np.abs(as_f64(mach.view(o.a, B * H * Dh), "bf16")).reshape(B, H, Dh)
        out = np.zeros((B, H, Dh))
        Kr, Vr = o.b, o.aux1
        for b in range(B):
            L = int(lens[b])
            for h in range(H):
                base = (b * H + h) * Lc * Dh
                from workloads.streams import Ref as _R
                K = np.abs(as_f64(mach.view(_R(Kr.buf, Kr.off + base), L * Dh), "bf16")).reshape(L, Dh)
                V = np.abs(as_f64(mach.view(_R(Vr.buf, Vr.off + base), L * Dh), "bf16")).reshape(L, Dh)
                dK = D(_R(Kr.buf, Kr.off + base), L * Dh).reshape(L, Dh)
                dV = D(_R(Vr.buf, Vr.off + base), L * Dh).reshape(L, Dh)
                ds = float(o.fparam[0]) * (K @ dq[b, h] + dK @ (q[b, h] + dq[b, h]))
                out[b, h] = 2.0 * ds.max() * V.max(0) + dV.max(0)
        return out.reshape(-1) * 1.01
    return 0.0


def mach_index(mach, o):
    return mach._op_index[id(o)]


def compare_op(rep: Report, s: Stream, j: int, gpu_read, mach) -> None:
    """Compare op j (see _compare_op_body); record it as passed when it added
    no failure."""
    before = len(rep.failures)
    _compare_op_body(rep, s, j, gpu_read, mach)
    if len(rep.failures) == before:
        rep.passed.add(j)


def _compare_op_body(rep: Report, s: Stream, j: int, gpu_read, mach) -> None:
    """Compare op j's outputs on the GPU (read via gpu_read(ref, n)) with the
    oracle machine state after it applied op j (exact results in mach.exact[j]).

    Must be called when both sides hold op j's outputs and inputs (none of
    them rewritten later in the stream). Inputs written by earlier ops may
    differ from the oracle's by those ops' rounding; the bound then grows by
    that difference propagated through the op (``propagated_bound``)."""
    o = s.ops[j]
    if not hasattr(mach, "_op_index"):
        mach._op_index = {id(op): k for k, op in enumerate(s.ops)}
    ex = mach.exact.get(j, {})
    rep.checked += 1
    d = o.dims
    if o.op == "nop":
        rep.exact += 1
        return
    diff = _differing_inputs(s, o, gpu_read, mach)
    same_in = not diff
    if not same_in and not _widening_sources_ok(rep, s, j, o, diff, gpu_read):
        return
    extra = 0.0 if same_in else propagated_bound(s, o, gpu_read, mach)
    if o.op in ("add", "mul", "relu", "gelu"):
        n = d[0]
        g = gpu_read(o.out, n)
        r = mach.view(o.out, n)
        if o.op != "gelu" and same_in:
            if np.array_equal(g.view(np.uint8), r.view(np.uint8)):
                rep.exact += 1
            else:
                diff = np.nonzero(g != r)[0]
                rep.fail(j, o, f"not bit-exact: {diff.size} elements differ, first {diff[:3]}")
            return
        rep.tol += 1
        if o.dtype == "f32":
            _check_f32_abs(rep, j, o, g, ex["out"], extra)
        else:
            check_bf16(rep, j, o, g, ex["out"], extra_abs=extra)
        return
    if o.op in ("softmax", "layernorm"):
        rep.tol += 1
        check_bf16(rep, j, o, gpu_read(o.out, d[0] * d[1]), ex["out"], extra_abs=extra)
        return
    if o.op == "rowsum":
        rep.tol += 1
        g = np.asarray(gpu_read(o.out, d[0]), dtype=np.float64)
        err = np.abs(g - ex["out"])
        bad = ~(err <= 2e-2 + 1e-5 * np.abs(ex["out"]) + extra)
        rep.max_abs = max(rep.max_abs, float(err.max(initial=0.0)))
        if bad.any():
            k = int(np.argmax(bad))
            rep.fail(j, o, f"rowsum mismatch at {k}: gpu={g[k]} exact={ex['out'][k]}")
        return
    if o.op in ("rowmax", "rowmin"):
        g = gpu_read(o.out, d[0])
        r = mach.view(o.out, d[0])
        if same_in:
            if np.array_equal(g, r):
                rep.exact += 1
            else:
                rep.fail(j, o, f"row extreme not exact: {np.nonzero(g != r)[0][:5]}")
        else:
            rep.tol += 1
            check_bf16(rep, j, o, g, ex["out"], extra_abs=extra)
        return
    if o.op == "rope":
        rep.tol += 1
        if not same_in:
            rep.fail(j, o, "in-place op on inputs produced by earlier ops: not comparable")
            return
        n = d[0] * d[1] * d[2]
        check_bf16(rep, j, o, gpu_read(o.a, n), ex["a"])
        check_bf16(rep, j, o, gpu_read(o.b, n), ex["b"])
        return
    if o.op == "sdpa":
        rep.tol += 1
        check_bf16(rep, j, o, gpu_read(o.out, d[0] * d[1] * d[2]), ex["out"], extra_abs=extra)
        return
    if o.op == "vecmat":
        rep.tol += 1
        check_bf16(rep, j, o, gpu_read(o.out, d[1]), ex["out"], extra_abs=extra)
        return
    if o.op == "kv_write":
        # the rows this op wrote (valid when no later op rewrote them)
        B, H, D, Lc = d[:4]
        lens = mach.view(o.aux0, B)
        for b in range(B):
            p = int(lens[b]) - 1
            for (ref, src) in ((o.out, o.a), (o.aux1, o.b)):
                for h in range(H):
                    off = ((b * H + h) * Lc + p) * D
                    g = gpu_read(Ref(ref.buf, ref.off + off), D)
                    r = mach.buf[ref.buf][ref.off + off:ref.off + off + D]
                    if same_in and not np.array_equal(g, r):
                        rep.fail(j, o, f"cache row (b={b}, h={h}, pos={p}) not bit-exact")
                        return
                    if not same_in and not check_bf16(rep, j, o, g, as_f64(r, "bf16")):
                        return
        if same_in:
            rep.exact += 1
        else:
            rep.tol += 1
        return
    raise ValueError(o.op)


def _check_f32_abs(rep, j, o, g, r_exact, extra_abs):
    g = np.asarray(g, dtype=np.float64)
    err = np.abs(g - r_exact)
    rms = float(np.sqrt(np.mean(r_exact ** 2))) if r_exact.size else 0.0
    bound = 1e-5 * np.maximum(np.abs(r_exact), 1e-3 * rms) + extra_abs * (1 + 1e-6)
    bad = ~(err <= bound)
    rep.max_abs = max(rep.max_abs, float(err.max(initial=0.0)))
    if bad.any():
        k = int(np.argmax(bad))
        rep.fail(j, o, f"fp32 (propagated) mismatch at {k}: gpu={g[k]!r} exact={r_exact[k]!r}")
