"""ctypes binding of ``libgpuos.so`` (the C ABI in include/gpuos.h).

Argument marshalling only: every step of the dispatch path runs in the
library and its CUDA kernels. If the library is missing this module raises;
there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgpuos.so")
EXT_CUBIN = os.path.join(HERE, "gpuos_ext_ops.cubin")

# ---- constants (mirror include/gpuos.h) --------------------------------------------
OK, EINVAL, EAGAIN, ETIMEDOUT, EDEVICE, ECUDA, ESTOPPED, ENOMEM, EBUSY, ETOOBIG, ECOMPILE = \
    0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -10
ST_OK, ST_BAD_OP, ST_BAD_ARGS, ST_DEP_TIMEOUT, ST_ABORTED, ST_BAD_DESC, ST_COPY_TIMEOUT = 0, 1, 2, 3, 4, 5, 6
OP = dict(nop=0, add=1, mul=2, relu=3, gelu=4, softmax=5, layernorm=6, rowsum=7, rowmax=8, rowmin=9,
          rope=10, kv_write=11, sdpa=12, vecmat=13)
OP_USER_FIRST = 64
F32, BF16 = 0, 1
DTYPE = {"f32": F32, "bf16": BF16}
FLAG_FENCE, FLAG_DEP_REL = 1, 2
U64_MAX = (1 << 64) - 1

# numpy view of gpuos_desc (128 bytes)
DESC_DTYPE = np.dtype([
    ("op_id", "<u2"), ("dtype", "u1"), ("flags", "u1"), ("ntiles", "<u4"),
    ("dep", "<u8", (2,)),
    ("a", "<u8"), ("b", "<u8"), ("out", "<u8"),
    ("aux0", "<u8"), ("aux1", "<u8"), ("aux2", "<u8"),
    ("dims", "<u4", (6,)), ("fparam", "<f4", (2,)),
    ("user", "<u8"), ("ticket", "<u8"), ("seq", "<u8"),
])
assert DESC_DTYPE.itemsize == 128

RECORD_DTYPE = np.dtype([
    ("ticket", "<u8"), ("status", "<i4"), ("version", "<u4"),
    ("t_commit_host_ns", "<u8"), ("t_dispatch_dev_ns", "<u8"), ("t_publish_dev_ns", "<u8"),
    ("t_start_dev_ns", "<u8"), ("t_done_dev_ns", "<u8"),
])
assert RECORD_DTYPE.itemsize == 56


class Config(C.Structure):
    _fields_ = [("ring_entries", C.c_uint32), ("warps_per_block", C.c_uint32), ("blocks", C.c_uint32),
                ("backoff_min_ns", C.c_uint32), ("backoff_max_ns", C.c_uint32), ("spin_polls", C.c_uint32),
                ("idle_exit_ms", C.c_uint32), ("dep_timeout_ms", C.c_uint32),
                ("ring_in_device_mem", C.c_uint32), ("device", C.c_int32), ("exit_after", C.c_uint64),
                ("tq_entries", C.c_uint32), ("deferred_start", C.c_uint32), ("stage_bytes", C.c_uint32),
                ("multi_producer", C.c_uint32), ("sequencers", C.c_uint32), ("reserved", C.c_uint32)]


class Record(C.Structure):
    _fields_ = [("ticket", C.c_uint64), ("status", C.c_int32), ("version", C.c_uint32),
                ("t_commit_host_ns", C.c_uint64), ("t_dispatch_dev_ns", C.c_uint64),
                ("t_publish_dev_ns", C.c_uint64), ("t_start_dev_ns", C.c_uint64),
                ("t_done_dev_ns", C.c_uint64)]


class Stats(C.Structure):
    _fields_ = [("submitted", C.c_uint64), ("completed", C.c_uint64), ("errors", C.c_uint64),
                ("sequenced", C.c_uint64), ("tiles", C.c_uint64), ("idle_polls", C.c_uint64),
                ("sleeps", C.c_uint64), ("dep_waits", C.c_uint64), ("version", C.c_uint32),
                ("running", C.c_uint32), ("exit_reason", C.c_uint32), ("blocks", C.c_uint32),
                ("warps_per_block", C.c_uint32), ("regs_per_thread", C.c_uint32),
                ("static_smem_bytes", C.c_uint32), ("reserved", C.c_uint32),
                ("seq_body_ns", C.c_uint64), ("seq_mirror_ns", C.c_uint64), ("seq_publish_ns", C.c_uint64),
                ("seq_batches", C.c_uint64), ("host_wait_ns", C.c_uint64), ("handoffs", C.c_uint64),
                ("handoff_link_ns", C.c_uint64), ("handoff_down_ns", C.c_uint64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "reserved"}


PROF_BUCKETS = 16


class TileProfile(C.Structure):
    _fields_ = [("tiles", C.c_uint64 * PROF_BUCKETS), ("body_ns", C.c_uint64 * PROF_BUCKETS),
                ("finish_ns", C.c_uint64 * PROF_BUCKETS), ("dep_ns", C.c_uint64 * PROF_BUCKETS)]


# every symbol include/gpuos.h declares
API = {
    "gpuos_default_config": (None, [C.POINTER(Config)]),
    "gpuos_init": (C.c_int, [C.POINTER(Config), C.POINTER(C.c_void_p)]),
    "gpuos_submit": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(C.c_uint64), C.c_uint32]),
    "gpuos_submit_batch": (C.c_int, [C.c_void_p, C.c_void_p, C.c_uint32, C.POINTER(C.c_uint64),
                                     C.POINTER(C.c_uint32), C.c_uint32]),
    "gpuos_sync": (C.c_int, [C.c_void_p, C.c_uint64, C.c_uint32]),
    "gpuos_query": (C.c_int, [C.c_void_p, C.c_uint64, C.POINTER(Record)]),
    "gpuos_set_history": (C.c_int, [C.c_void_p, C.c_void_p, C.c_uint64, C.c_uint64]),
    "gpuos_register_op": (C.c_int, [C.c_void_p, C.c_uint16, C.c_void_p, C.c_size_t, C.c_char_p]),
    "gpuos_load_module": (C.c_int, [C.c_void_p, C.c_void_p, C.c_size_t]),
    "gpuos_alias_op": (C.c_int, [C.c_void_p, C.c_uint16, C.c_uint16]),
    "gpuos_stats": (C.c_int, [C.c_void_p, C.POINTER(Stats)]),
    "gpuos_tile_profile_get": (C.c_int, [C.c_void_p, C.POINTER(TileProfile)]),
    "gpuos_compile_op": (C.c_int, [C.c_char_p, C.c_char_p, C.POINTER(C.c_void_p), C.POINTER(C.c_size_t),
                                   C.c_char_p, C.c_size_t]),
    "gpuos_free_image": (None, [C.c_void_p]),
    "gpuos_op_header": (C.c_char_p, []),
    "gpuos_calibrate": (C.c_int, [C.c_void_p, C.c_uint32, C.POINTER(C.c_int64), C.POINTER(C.c_int64),
                                  C.POINTER(C.c_uint64), C.c_void_p]),
    "gpuos_shutdown": (C.c_int, [C.c_void_p, C.c_uint32]),
    "gpuos_stop": (C.c_int, [C.c_void_p, C.c_uint32]),
    "gpuos_start": (C.c_int, [C.c_void_p]),
    "gpuos_executor_stream": (C.c_int, [C.c_void_p, C.POINTER(C.c_void_p)]),
    "gpuos_op_ntiles": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint32)]),
    "gpuos_sdpa_workspace_bytes": (C.c_size_t, [C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint32]),
    "gpuos_eager_run": (C.c_int, [C.c_void_p, C.c_uint32, C.c_uint32, C.c_void_p]),
    "gpuos_host_now_ns": (C.c_uint64, []),
    "gpuos_sdpa_noalloc": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_uint32,
                                     C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint32, C.c_float, C.c_void_p]),
    "gpuos_strerror": (C.c_char_p, [C.c_int, C.c_int]),
}

_lib = None


def lib():
    """Load the C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libgpuos.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in API.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class GpuosError(RuntimeError):
    def __init__(self, what: str, code: int):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


def strerror(code: int, is_status: bool = False) -> str:
    return lib().gpuos_strerror(code, 1 if is_status else 0).decode()


def check(code: int, what: str) -> int:
    if code != OK:
        raise GpuosError(what, code)
    return code


def default_config(**kw) -> Config:
    c = Config()
    lib().gpuos_default_config(C.byref(c))
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def sdpa_workspace_bytes(B: int, H: int, D: int, Lmax: int) -> int:
    return int(lib().gpuos_sdpa_workspace_bytes(B, H, D, Lmax))


def op_ntiles(desc: np.ndarray) -> int:
    n = C.c_uint32()
    check(lib().gpuos_op_ntiles(desc.ctypes.data, C.byref(n)), "gpuos_op_ntiles")
    return n.value


def host_now_ns() -> int:
    return int(lib().gpuos_host_now_ns())


def eager_run(descs: np.ndarray, stream_ptr: int = 0, stage_bytes: int = 16384) -> None:
    """Launch each descriptor as its own kernel on ``stream_ptr`` (cudaStream_t)."""
    descs = np.ascontiguousarray(descs, dtype=DESC_DTYPE)
    check(lib().gpuos_eager_run(descs.ctypes.data, len(descs), stage_bytes, C.c_void_p(stream_ptr)),
          "gpuos_eager_run")


def sdpa_noalloc(q: int, Kc: int, Vc: int, lens: int, out: int, B: int, H: int, D: int, Lcap: int, Lmax: int,
                 scale: float, stream_ptr: int = 0) -> int:
    """Decode attention with the library's fixed scratch (device pointers in);
    returns the raw return code."""
    return lib().gpuos_sdpa_noalloc(C.c_void_p(q), C.c_void_p(Kc), C.c_void_p(Vc), C.c_void_p(lens), C.c_void_p(out),
                                    B, H, D, Lcap, Lmax, scale, C.c_void_p(stream_ptr))


def compile_op(source: str, name: str = "gpuos_op.cu") -> bytes:
    """Compile operator source at run time (NVRTC) to a relocatable sm_103a
    cubin for Executor.load_module / register_op. Raises GpuosError with the
    compiler log on failure."""
    img = C.c_void_p()
    size = C.c_size_t()
    log = C.create_string_buffer(16384)
    rc = lib().gpuos_compile_op(source.encode(), name.encode(), C.byref(img), C.byref(size), log, len(log))
    if rc != OK:
        raise GpuosError("gpuos_compile_op: " + log.value.decode(errors="replace"), rc)
    try:
        return C.string_at(img.value, size.value)
    finally:
        lib().gpuos_free_image(img)


def op_header() -> str:
    """The operator ABI header compile_op puts before every source."""
    return lib().gpuos_op_header().decode()


def make_descs(n: int) -> np.ndarray:
    return np.zeros(n, dtype=DESC_DTYPE)


class Executor:
    """One persistent executor (one context): ring, table, kernel."""

    def __init__(self, config: Optional[Config] = None, **kw):
        cfg = config if config is not None else default_config(**kw)
        self._ctx = C.c_void_p()
        check(lib().gpuos_init(C.byref(cfg), C.byref(self._ctx)), "gpuos_init")
        self.config = cfg
        self._hist = None

    # -- submission ------------------------------------------------------------
    def submit(self, desc: np.ndarray, timeout_us: int = 5_000_000) -> int:
        d = np.ascontiguousarray(desc, dtype=DESC_DTYPE).reshape(-1)[:1]
        t = C.c_uint64()
        check(lib().gpuos_submit(self._ctx, d.ctypes.data, C.byref(t), timeout_us), "gpuos_submit")
        return t.value

    def submit_batch(self, descs: np.ndarray, timeout_us: int = 5_000_000) -> int:
        d = np.ascontiguousarray(descs, dtype=DESC_DTYPE)
        first = C.c_uint64()
        done = C.c_uint32()
        rc = lib().gpuos_submit_batch(self._ctx, d.ctypes.data, len(d), C.byref(first), C.byref(done), timeout_us)
        if rc != OK:
            raise GpuosError(f"gpuos_submit_batch (submitted {done.value} of {len(d)})", rc)
        return first.value

    def try_submit(self, desc: np.ndarray, timeout_us: int = 0) -> int:
        """Submit and return the raw return code (no exception)."""
        d = np.ascontiguousarray(desc, dtype=DESC_DTYPE).reshape(-1)[:1]
        t = C.c_uint64()
        return lib().gpuos_submit(self._ctx, d.ctypes.data, C.byref(t), timeout_us)

    def sync(self, ticket: Optional[int] = None, timeout_ms: int = 60_000, raise_on_error: bool = True) -> int:
        rc = lib().gpuos_sync(self._ctx, U64_MAX if ticket is None else ticket, timeout_ms)
        if raise_on_error:
            check(rc, "gpuos_sync")
        return rc

    def query(self, ticket: int) -> Record:
        r = Record()
        check(lib().gpuos_query(self._ctx, ticket, C.byref(r)), "gpuos_query")
        return r

    def set_history(self, base: int, capacity: int) -> np.ndarray:
        # written once per completion while descriptors stream in: touch every
        # page now (a lazily mapped zero page faults on its first write)
        self._hist = np.empty(capacity, dtype=RECORD_DTYPE)
        self._hist.view(np.uint8)[:] = 0
        check(lib().gpuos_set_history(self._ctx, self._hist.ctypes.data, base, capacity), "gpuos_set_history")
        return self._hist

    # -- operator table --------------------------------------------------------
    def register_op(self, op_id: int, image: bytes, symbol: str) -> None:
        buf = C.create_string_buffer(image, len(image))
        check(lib().gpuos_register_op(self._ctx, op_id, buf, len(image), symbol.encode()), "gpuos_register_op")

    def load_module(self, image: bytes) -> None:
        """Load a cubin while the executor is not resident (before start())."""
        buf = C.create_string_buffer(image, len(image))
        check(lib().gpuos_load_module(self._ctx, buf, len(image)), "gpuos_load_module")

    def alias_op(self, op_id: int, source_op: int) -> None:
        check(lib().gpuos_alias_op(self._ctx, op_id, source_op), "gpuos_alias_op")

    # -- measurement -----------------------------------------------------------
    def tile_profile(self) -> dict:
        """Per op name: tiles run and the mean device time per tile (µs)
        inside the op, finishing (counting, completing) and waiting for
        dependencies; user ops share the bucket "user"."""
        t = TileProfile()
        check(lib().gpuos_tile_profile_get(self._ctx, C.byref(t)), "gpuos_tile_profile_get")
        names = {v: k for k, v in OP.items()}
        out = {}
        for b in range(PROF_BUCKETS):
            n = int(t.tiles[b])
            if n == 0:
                continue
            out[names.get(b, "user")] = {"tiles": n, "body_us": t.body_ns[b] / n / 1e3,
                                         "finish_us": t.finish_ns[b] / n / 1e3, "dep_us": t.dep_ns[b] / n / 1e3}
        return out

    def stats(self) -> dict:
        s = Stats()
        check(lib().gpuos_stats(self._ctx, C.byref(s)), "gpuos_stats")
        return s.as_dict()

    def calibrate(self, pings: int = 200):
        """NOP ping-pong; returns (offset_lo, offset_hi, min_rtt_ns, rtts) where
        device clock - host clock lies in [offset_lo, offset_hi]."""
        lo = C.c_int64()
        hi = C.c_int64()
        rtt = C.c_uint64()
        rtts = np.zeros(pings, dtype=np.uint64)
        check(lib().gpuos_calibrate(self._ctx, pings, C.byref(lo), C.byref(hi), C.byref(rtt), rtts.ctypes.data),
              "gpuos_calibrate")
        return lo.value, hi.value, rtt.value, rtts

    def start(self) -> None:
        """Launch a context created with deferred_start=1."""
        check(lib().gpuos_start(self._ctx), "gpuos_start")

    def stop(self, timeout_ms: int = 30_000) -> int:
        """Drain, stop the executor kernel and wait for it to end."""
        return lib().gpuos_stop(self._ctx, timeout_ms)

    @property
    def stream(self) -> int:
        """cudaStream_t of the executor (for CUDA events around its launch)."""
        s = C.c_void_p()
        check(lib().gpuos_executor_stream(self._ctx, C.byref(s)), "gpuos_executor_stream")
        return s.value or 0

    def shutdown(self, timeout_ms: int = 30_000) -> int:
        if self._ctx:
            rc = lib().gpuos_shutdown(self._ctx, timeout_ms)
            self._ctx = C.c_void_p()
            return rc
        return OK

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.shutdown()

    def __del__(self):
        try:
            if self._ctx:
                self.shutdown()
        except Exception:
            pass


def exported_symbols() -> Sequence[str]:
    return list(API)
