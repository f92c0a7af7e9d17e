/*
 * gpuos.h -- C ABI of the GB300 persistent micro-op dispatcher.
 *
 * The method is the one described in "GPUOS: A GPU Operating System Primitive
 * for Transparent Operation Fusion" (Yang et al., 2026), §2 and §3 Q2:
 *   - a persistent executor kernel is launched once, one block per SM, and
 *     never exits while the context lives (§3 Q2 "2. Persistent Kernel
 *     Executor");
 *   - the host writes 64-128 B task descriptors {op_id, input_a, input_b,
 *     output, size, flags} into a lock-free single-producer ring in memory
 *     the device can see, committing each with a store-release; the device
 *     polls with load-acquire, claims work atomically, dispatches and
 *     releases the slot (§3 Q2 "1. Ring Buffer Communication Channel");
 *   - dispatch goes through a device-resident table of device-function
 *     pointers indexed by op_id, kept in two slots (active / inactive) that a
 *     version counter flips with a store-release (§3 Q2 "3. Dynamic Operator
 *     Table");
 *   - the ops are the page's operator library: element-wise add, mul, ReLU,
 *     GELU, softmax, LayerNorm; vector-matrix products; SDPA and rotary
 *     embeddings; KV-cache update; small sum/max/min reductions (§3 Q2,
 *     "Operator library").
 *
 * Conventions for every call:
 *   - Returns GPUOS_OK (0) or a negative GPUOS_E* code; nothing throws, aborts
 *     or falls back to the CPU.
 *   - Tensors named in descriptors are caller-owned device memory and must stay
 *     alive until their descriptor has completed. The library owns the ring,
 *     the completion records, the operator table, loaded modules and the
 *     executor's stream.
 *   - One producer thread per context (the ring is single-producer).
 *   - While the executor is resident, do not call cudaDeviceSynchronize() (it
 *     would wait for a kernel that does not end), and launch only kernels that
 *     were loaded before gpuos_init (under lazy module loading, loading a new
 *     kernel may wait for the device to go idle). The executor leaves by
 *     itself after `idle_exit_ms` without host activity, so no such mistake
 *     can hang the GPU for good.
 */
#ifndef GPUOS_H
#define GPUOS_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GPUOS_API __attribute__((visibility("default")))
#else
#define GPUOS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define GPUOS_OK 0
#define GPUOS_EINVAL (-1)    /* bad argument, op id, pointer or dims */
#define GPUOS_EAGAIN (-2)    /* ring full until the timeout ran out */
#define GPUOS_ETIMEDOUT (-3) /* a wait ran out */
#define GPUOS_EDEVICE (-4)   /* a descriptor completed with a device status != 0 */
#define GPUOS_ECUDA (-5)     /* a CUDA runtime/driver call failed */
#define GPUOS_ESTOPPED (-6)  /* the executor is no longer running */
#define GPUOS_ENOMEM (-7)
#define GPUOS_EBUSY (-8)     /* needs the executor not resident (see gpuos_load_module) */
#define GPUOS_ETOOBIG (-9)   /* sizes beyond a fixed limit (see gpuos_sdpa_noalloc) */
#define GPUOS_ECOMPILE (-10) /* operator source did not compile (see gpuos_compile_op's log) */

/* ---- device status codes (gpuos_record.status) -------------------------- */
#define GPUOS_ST_OK 0
#define GPUOS_ST_BAD_OP 1        /* op_id out of range or empty table entry */
#define GPUOS_ST_BAD_ARGS 2      /* dims / positions / lengths out of range */
#define GPUOS_ST_DEP_TIMEOUT 3   /* a dependency or fence wait ran out */
#define GPUOS_ST_ABORTED 4       /* the executor was leaving */
#define GPUOS_ST_BAD_DESC 5      /* ring slot did not hold the expected ticket */
#define GPUOS_ST_COPY_TIMEOUT 6  /* a shared-memory staging copy did not land within its bound */

/* ---- op ids (built-in operator library) --------------------------------- */
enum {
    GPUOS_OP_NOP = 0,       /* no effect; latency probe */
    GPUOS_OP_ADD = 1,       /* out[i] = a[i] + b[i]            dims = {n}          f32|bf16 */
    GPUOS_OP_MUL = 2,       /* out[i] = a[i] * b[i]            dims = {n}          f32|bf16 */
    GPUOS_OP_RELU = 3,      /* out[i] = max(a[i], +0)          dims = {n}          f32|bf16 */
    GPUOS_OP_GELU = 4,      /* out[i] = a Phi(a), erf form     dims = {n}          f32|bf16 */
    GPUOS_OP_SOFTMAX = 5,   /* row softmax of a[R][H] -> out   dims = {R, H}       bf16 */
    GPUOS_OP_LAYERNORM = 6, /* a[R][H], b=gamma[H], aux0=beta[H] -> out; fparam[0] = eps; bf16 */
    GPUOS_OP_ROWSUM = 7,    /* out f32[R] = sum_j a[r][j]      dims = {R, H}       bf16 in */
    GPUOS_OP_ROWMAX = 8,    /* out bf16[R] = max_j a[r][j]     dims = {R, H} */
    GPUOS_OP_ROWMIN = 9,    /* out bf16[R] = min_j a[r][j]     dims = {R, H} */
    GPUOS_OP_ROPE = 10,     /* in place on a=q[B][H][D], b=k[B][H][D]; aux0 = lens i32[B],
                               position lens[b]-1; half-split pairs (i, i+D/2);
                               fparam[0] = theta; dims = {B, H, D}, D even, D <= 256 */
    GPUOS_OP_KV_WRITE = 11, /* Kc[b][h][lens[b]-1][:] = a[b][h][:], same for Vc; out = Kc,
                               aux1 = Vc laid out [B][H][Lcap][D]; aux0 = lens i32[B];
                               dims = {B, H, D, Lcap}; bit-exact copy */
    GPUOS_OP_SDPA = 12,     /* o = softmax(scale q.K^T) V over rows 0..lens[b]-1; a = q[B][H][D],
                               b = Kc, aux1 = Vc [B][H][Lcap][D], aux0 = lens, out = o[B][H][D],
                               aux2 = 16-byte aligned fp32 workspace: first round_up(Ccap, 4)
                               uint32 counters, then B*H*ceil(Lmax/32) partials of 132 floats
                               {m, l, 2 pad, acc[128]}
                               (gpuos_sdpa_workspace_bytes(Bcap, H, D, Lmax) with Ccap = Bcap*H);
                               the counters must be zero before first use and every descriptor
                               leaves them zero; descriptors sharing a workspace use one Ccap;
                               dims = {B, H, D=128, Lcap, Lmax >= every lens[b], Ccap >= B*H};
                               fparam[0] = scale */
    GPUOS_OP_VECMAT = 13,   /* out[n] = sum_k a[k] b[k][n]; b row-major [K][N]; dims = {K, N}; bf16 */
    GPUOS_OP_BUILTIN_COUNT = 14,
    GPUOS_OP_USER_FIRST = 64, /* ids >= this are free for gpuos_register_op */
    GPUOS_MAX_OPS = 256
};

#define GPUOS_F32 0
#define GPUOS_BF16 1

/* descriptor flags */
#define GPUOS_FLAG_FENCE 1u   /* start only after every earlier descriptor completed */
#define GPUOS_FLAG_DEP_REL 2u /* dep[i] holds a backward distance (1 = the previous
                                 descriptor) instead of an absolute ticket + 1 */

/*
 * Task descriptor: 128 bytes, one ring slot (the page gives 64-128 B holding
 * {op_id, input_a, input_b, output, size, flags}, §3 Q2 "1. Ring Buffer
 * Communication Channel"). Fields marked [lib] are written by the library.
 *
 * dep[i]: 0 = none; otherwise ticket + 1 of an earlier descriptor this one
 * must wait for (or a distance with GPUOS_FLAG_DEP_REL). ntiles is computed by
 * the library for built-in ops; for user ops (id >= GPUOS_OP_USER_FIRST) the
 * caller sets it (>= 0; each tile is handed to one warp).
 */
typedef struct gpuos_desc {
    uint16_t op_id;
    uint8_t dtype;  /* GPUOS_F32 | GPUOS_BF16 */
    uint8_t flags;  /* GPUOS_FLAG_* */
    uint32_t ntiles;
    uint64_t dep[2];
    uint64_t a, b, out;       /* device pointers */
    uint64_t aux0, aux1, aux2; /* device pointers, per op */
    uint32_t dims[6];
    float fparam[2];
    uint64_t user;   /* caller tag, not read by the device */
    uint64_t ticket; /* [lib] */
    uint64_t seq;    /* [lib] commit word: ticket + 1 once the slot is published */
} gpuos_desc;

/* Executor / ring configuration. gpuos_default_config() fills defaults. */
typedef struct gpuos_config {
    uint32_t ring_entries;    /* power of two in [64, 65536]; default 8192 (the page's default is
                                 4096: with 8192 the submitting thread waits less often for the
                                 one slot a slow descriptor still holds, and the ring's 1 MB
                                 stays in a Grace core's L2) */
    uint32_t warps_per_block; /* 2..12; default 12 */
    uint32_t blocks;          /* 0 = one block per SM; block 0 holds only the sequencer warp
                                 (when blocks > 1) */
    uint32_t backoff_min_ns;  /* first idle sleep; default 32 */
    uint32_t backoff_max_ns;  /* idle sleep cap of worker warps waiting for work; default 8000
                                 (the sequencers' ring poll and dependency waits sleep at
                                 most 256 ns, or this if smaller) */
    uint32_t spin_polls;      /* polls of pure spinning before backing off; default 4096 */
    uint32_t idle_exit_ms;    /* leave after this long with no host activity; 0 = never; default 10000 */
    uint32_t dep_timeout_ms;  /* bound of every device-side wait; default 5000 */
    uint32_t ring_in_device_mem; /* 0: ring in pinned host memory (default);
                                    1: managed memory preferred on the device */
    int32_t device;           /* CUDA device ordinal; default 0 */
    uint64_t exit_after;      /* 0 = run until shutdown; n = leave once n descriptors completed */
    uint32_t tq_entries;      /* work-queue entries: 0 (default) = 4096 x ring_entries; else a
                                 power of two above 2048 x ring_entries, at most 2^30 */
    uint32_t deferred_start;  /* 1: gpuos_init does not launch; gpuos_start does (descriptors
                                 may be submitted before, up to ring_entries of them) */
    uint32_t stage_bytes;     /* shared-memory staging per warp for bulk (TMA) copies: 0 = none
                                 (register path; leaves shared memory to co-running kernels),
                                 else a multiple of 1024 up to 24576; default 16384 */
    uint32_t multi_producer;  /* 0 (default): one submitting thread (SPSC ring, no locks);
                                 1: any number of host threads may call gpuos_submit /
                                 gpuos_submit_batch concurrently (see gpuos_submit) */
    uint32_t sequencers;      /* warps that take descriptors off the ring, 1..4, one per block
                                 (blocks 0 .. sequencers-1 run no workers; fewer than blocks;
                                 1 when blocks == 1); 0 = default: 4 on 32 blocks or more, 2
                                 on 16 or more, else 1. Tickets are cut into windows of 128
                                 (or ring_entries, if smaller), taken in turn; work-queue
                                 space is still given out in ticket order */
    uint32_t reserved;
} gpuos_config;

/* Completion record of one ticket (device clock = %globaltimer, host clock =
 * CLOCK_REALTIME in ns; gpuos_calibrate bounds their offset). */
typedef struct gpuos_record {
    uint64_t ticket;
    int32_t status;             /* GPUOS_ST_* */
    uint32_t version;           /* operator-table version the descriptor ran with */
    uint64_t t_commit_host_ns;  /* host clock just before the commit store-release */
    uint64_t t_dispatch_dev_ns; /* when the executor saw the commit (picked it off the ring) */
    uint64_t t_publish_dev_ns;  /* when its batch was handed to the work queue (just before
                                   its entries were written) */
    uint64_t t_start_dev_ns;    /* when a warp began its tile 0 (dependencies met) */
    uint64_t t_done_dev_ns;     /* when its last tile finished */
} gpuos_record;

typedef struct gpuos_stats_t {
    uint64_t submitted;     /* host: descriptors committed */
    uint64_t completed;     /* host: completions harvested */
    uint64_t errors;        /* host: completions with status != 0 */
    uint64_t sequenced;     /* device: descriptors taken off the ring */
    uint64_t tiles;         /* device: tiles executed */
    uint64_t idle_polls;    /* device: empty polls of workers and sequencer */
    uint64_t sleeps;        /* device: __nanosleep backoffs */
    uint64_t dep_waits;     /* device: tiles that waited on a dependency */
    uint32_t version;       /* current operator-table version */
    uint32_t running;       /* 1 while the executor kernel is resident */
    uint32_t exit_reason;   /* 0 running, 1 stop, 2 idle watchdog, 3 exit_after, 4 internal */
    uint32_t blocks;
    uint32_t warps_per_block;
    uint32_t regs_per_thread; /* of the executor kernel */
    uint32_t static_smem_bytes;
    uint32_t reserved;
    uint64_t seq_body_ns;    /* device: sequencer time reading, validating and mirroring descriptors */
    uint64_t seq_mirror_ns;  /* device: sequencer time in the fence after mirroring */
    uint64_t seq_publish_ns; /* device: sequencer time publishing work-queue entries */
    uint64_t seq_batches;    /* device: batches the sequencer took off the ring (lone descriptors
                                it ran itself not counted) */
    uint64_t host_wait_ns;   /* host: time submitting threads waited for a free ring slot */
    uint64_t handoffs;        /* host: executor relaunches that took in a new operator module */
    uint64_t handoff_link_ns; /* host, last hand-off: linking the module set (the old executor
                                 still runs meanwhile) */
    uint64_t handoff_down_ns; /* host, last hand-off: from the stop request to the new
                                 executor running (nothing is dispatched meanwhile) */
} gpuos_stats_t;

/* Where the executor's worker warps spent their time, per op id (device
 * clock, summed over warps). Bucket b < GPUOS_OP_BUILTIN_COUNT is op id b;
 * bucket GPUOS_OP_BUILTIN_COUNT gathers every user op id. */
#define GPUOS_PROF_BUCKETS 16
#define GPUOS_PROF_FIELDS 4
typedef struct gpuos_tile_profile {
    uint64_t tiles[GPUOS_PROF_BUCKETS];     /* tiles run */
    uint64_t body_ns[GPUOS_PROF_BUCKETS];   /* inside the op's entry point */
    uint64_t finish_ns[GPUOS_PROF_BUCKETS]; /* counting the helper's tiles and completing */
    uint64_t dep_ns[GPUOS_PROF_BUCKETS];    /* from finding the work-queue entry to its
                                               dependencies being met (mirror read included) */
} gpuos_tile_profile;

typedef struct gpuos_ctx gpuos_ctx;

/* Fill *cfg with defaults. Source: GPUOS page, §3 Q2 "1. Ring Buffer
 * Communication Channel" (4096 ring entries by default there; 8192 here,
 * as ring_entries says) and "2. Persistent
 * Kernel Executor" (one block per SM; spin under load, exponential backoff
 * when idle). */
GPUOS_API void gpuos_default_config(gpuos_config *cfg);

/* Allocate the ring, completion records and operator table, fill both table
 * slots with the built-in ops (version 0) and launch the executor once on a
 * non-blocking stream (grid = blocks, block = 32 * warps_per_block). *out
 * receives the context. Errors: EINVAL (bad config), ECUDA, ENOMEM.
 * Source: GPUOS page, §1 and §3 Q2 "2. Persistent Kernel Executor" (the
 * persistent kernel is launched once when the process starts, one block per
 * SM) with the ring of "1. Ring Buffer Communication Channel" and the table
 * of "3. Dynamic Operator Table"; the name gpuos_init is this library's. */
GPUOS_API int gpuos_init(const gpuos_config *cfg, gpuos_ctx **out);

/* Launch the executor of a context made with deferred_start (once). Lets a
 * caller fill the ring first (a bounded, replayable run for profilers) or put
 * the single launch inside a timed region. Errors: EINVAL (already started),
 * ECUDA. Source: the single launch of GPUOS page §3 Q2 "2. Persistent Kernel
 * Executor", split from gpuos_init; the page has no separate start step. */
GPUOS_API int gpuos_start(gpuos_ctx *ctx);

/* The non-blocking stream the executor runs on (a cudaStream_t), so callers
 * can bracket the kernel with CUDA events. Measurement only; the page has no
 * counterpart. */
GPUOS_API int gpuos_executor_stream(gpuos_ctx *ctx, void **stream);

/* Submit one descriptor (§3 Q2 ring protocol: acquire slot, write, commit
 * with store-release). Validates op_id, pointers, dims and deps on the host,
 * computes ntiles for built-in ops, waits up to timeout_us for a free slot
 * (EAGAIN after that, nothing submitted). *ticket (may be NULL) receives the
 * ticket. Errors: EINVAL, EAGAIN, ESTOPPED.
 *
 * With multi_producer = 1 several threads may submit at once (§3 Q3, ring
 * contention with concurrent host threads): a submission first validates all
 * its descriptors, waits up to timeout_us for room in the ring (EAGAIN,
 * nothing submitted), then reserves consecutive tickets with one atomic add
 * and commits them. A reserved ticket is always committed (the executor
 * takes tickets in order, so an abandoned one would stall every later one):
 * after the reservation the call waits for its slots without a timeout,
 * returning ESTOPPED only if the executor has left. Tickets of different
 * threads interleave; a GPUOS_FLAG_DEP_REL distance counts in that global
 * order. The context must have been started (EINVAL otherwise). */
GPUOS_API int gpuos_submit(gpuos_ctx *ctx, const gpuos_desc *d, uint64_t *ticket, uint32_t timeout_us);

/* Submit count descriptors in order (same as count gpuos_submit calls);
 * *first_ticket receives the first ticket. Stops at the first failure and
 * returns its code; *n_done (may be NULL) receives how many were submitted.
 * Source: the host half of GPUOS page §3 Q2 "1. Ring Buffer Communication
 * Channel" (acquire slot, write, commit with a store-release), once per
 * descriptor. With one producer the call writes the bodies of a run of
 * consecutive descriptors, then one release fence, then their commit words:
 * every commit still follows its own body, as the protocol requires. */
GPUOS_API int gpuos_submit_batch(gpuos_ctx *ctx, const gpuos_desc *d, uint32_t count, uint64_t *first_ticket,
                       uint32_t *n_done, uint32_t timeout_us);

/* Wait until `ticket` (or, with ticket == UINT64_MAX, everything submitted so
 * far) has completed, up to timeout_ms. Source: the device's "release slot"
 * step of GPUOS page §3 Q2 "1. Ring Buffer Communication Channel" is a
 * store-release of the ticket's completion record, which this call reads
 * with load-acquire; the name gpuos_sync is this library's. Returns EDEVICE if any descriptor
 * harvested by this call completed with a nonzero status, ETIMEDOUT on
 * timeout, ESTOPPED if the executor left with work outstanding. */
GPUOS_API int gpuos_sync(gpuos_ctx *ctx, uint64_t ticket, uint32_t timeout_ms);

/* Completion record of a finished ticket still in the history window (the
 * last `ring_entries` tickets, or the whole run with gpuos_set_history).
 * Errors: EAGAIN (not finished yet), EINVAL (outside the window). Source:
 * the completion ("release slot") of GPUOS page §3 Q2 "1. Ring Buffer
 * Communication Channel", with the timestamps the latency breakdown of §3 Q3
 * needs. */
GPUOS_API int gpuos_query(gpuos_ctx *ctx, uint64_t ticket, gpuos_record *rec);

/* Keep every harvested completion record of tickets [base, base + capacity)
 * in caller memory (host), for latency statistics (GPUOS page §3 Q3, latency
 * breakdown). buf may be NULL to stop. */
GPUOS_API int gpuos_set_history(gpuos_ctx *ctx, gpuos_record *buf, uint64_t base, uint64_t capacity);

/* Source: GPUOS page §3 Q2 "3. Dynamic Operator Table", step (2): load the
 * operator's module through the CUDA Driver API.
 * Add an operator module: a relocatable sm_103a cubin (nvcc -cubin
 * -rdc=true; the bytes are copied) that defines device functions with the op
 * signature and `__device__` variables holding their addresses. A
 * device-function pointer is only callable inside the module that holds its
 * code, so the library links every added module with its relocatable
 * executor build (driver JIT linker) and launches the executor from the
 * linked module. Before gpuos_start (deferred_start) the module is linked at
 * the launch. With the executor running, the call hands off (a module load
 * waits for the device to go idle, which a resident executor never does):
 * every submitted descriptor completes, the executor leaves, the module set
 * is linked again and the executor is launched from it, continuing at the
 * next ticket with the ring, the completion records and every operator
 * binding carried over (the table is rebuilt with the new module's
 * addresses). The hand-off takes milliseconds; descriptors submitted after
 * it run on the new kernel, none is lost or run twice. It needs a
 * single-producer context (EBUSY with multi_producer = 1), and per-warp
 * counters of gpuos_stats restart with the new kernel. Adding an image
 * already added is a no-op. Errors: EINVAL (does not link), EBUSY, ESTOPPED,
 * ETIMEDOUT, ECUDA (the context accepts no more work after a failed
 * hand-off). */
GPUOS_API int gpuos_load_module(gpuos_ctx *ctx, const void *image, size_t len);

/* Run-time compilation of an operator (§3 Q2 "3. Dynamic Operator Table",
 * step 1). source: CUDA C++ that defines a device operator
 *     __device__ int my_op(const gpuos_devdesc *d, uint32_t tile) { ... }
 * and exports it as  __device__ gpuos_op_fn my_op_ptr = my_op;
 * The library prepends the operator ABI header (gpuos_op_header(): the
 * 128-byte gpuos_devdesc seen by operators, gpuos_op_fn, status codes) and
 * compiles with NVRTC (opened at run time) for sm_103a, relocatable, with
 * the executor's per-thread register cap. On success *image (malloc'd; free
 * with gpuos_free_image) and *size hold a cubin for gpuos_load_module /
 * gpuos_register_op. log (may be NULL) receives NVRTC's log, truncated to
 * log_cap bytes. name (may be NULL) names the source in that log. Runs on
 * the CPU only; no context is needed. Errors: EINVAL, ECOMPILE (see log),
 * ECUDA (NVRTC missing or failed), ENOMEM. */
GPUOS_API int gpuos_compile_op(const char *source, const char *name, void **image, size_t *size, char *log,
                               size_t log_cap);
GPUOS_API void gpuos_free_image(void *image);
/* The header text gpuos_compile_op puts before every operator source (the
 * operator ABI of §3 Q2 "3. Dynamic Operator Table": the descriptor an
 * operator receives, its signature and status codes). A static string owned
 * by the library; never fails. */
GPUOS_API const char *gpuos_op_header(void);

/* Runtime operator injection (§3 Q2 "3. Dynamic Operator Table", steps 3-5):
 * for a module added with gpuos_load_module (and so linked into the running
 * executor), read its `__device__` variable `fnptr_symbol` holding the
 * address of a device function with the op signature, write it into the
 * inactive table slot (a copy of the active one with entry op_id replaced),
 * then flip the version with a store-release. Nothing stops: descriptors
 * sequenced before the flip finish with the old entry; later ones use the new
 * one. Before a later flip reuses that slot the call waits until every
 * descriptor sequenced under the older version has completed. The function
 * must use at most the executor's registers per thread (compile it with the
 * same -maxrregcount). An image not yet added is added first with
 * gpuos_load_module (a hand-off if the executor runs). Errors: EINVAL (bad id
 * or symbol, image does not link), EBUSY (executor not yet launched, or a
 * hand-off with several producers), ECUDA, ETIMEDOUT. */
GPUOS_API int gpuos_register_op(gpuos_ctx *ctx, uint16_t op_id, const void *image, size_t len,
                      const char *fnptr_symbol);

/* Source: GPUOS page §3 Q2 "3. Dynamic Operator Table", steps (4) and (5)
 * (write the inactive slot, flip the version counter), with an entry that is
 * already in the table.
 * Point op_id back at a built-in op or an earlier registered function:
 * `source_op` names the entry to copy from the active table. Same flip and
 * grace-period protocol as gpuos_register_op. */
GPUOS_API int gpuos_alias_op(gpuos_ctx *ctx, uint16_t op_id, uint16_t source_op);

/* Live counters (host and device): polls, sleeps, tiles, sequencer phase
 * times. Measurement only (the poll loop and backoff of GPUOS page §3 Q2
 * "2. Persistent Kernel Executor"); the page has no counterpart. */
GPUOS_API int gpuos_stats(gpuos_ctx *ctx, gpuos_stats_t *st);

/* Source: measurement of the dispatch latency of GPUOS page §3 Q3 (latency
 * breakdown: ~100 ns dispatch); the page has no calibration step.
 * NOP ping-pong: `pings` round trips. Each commits a NOP (host clock t0)
 * and spins until the executor's echo of the time it saw the commit appears
 * in the ticket's record (host clock t1; the echo is written the moment the
 * commit is seen, before the descriptor is read). Since the device sees the
 * commit between t0 and t1, every ping bounds off = device clock - host clock
 * to [t_dispatch - t1, t_dispatch - t0]; *off_lo / *off_hi receive the
 * intersection over all pings and *min_rtt_ns the smallest t1 - t0. rtts
 * (may be NULL) receives every echo round trip. It first waits for every
 * submitted ticket; no other thread may submit while it runs. */
GPUOS_API int gpuos_calibrate(gpuos_ctx *ctx, uint32_t pings, int64_t *off_lo, int64_t *off_hi,
                              uint64_t *min_rtt_ns, uint64_t *rtts);

/* Drain (wait for everything submitted, up to timeout_ms), set the stop flag
 * and wait (up to timeout_ms) for the executor kernel to end; the context
 * stays valid (stats, queries) but accepts no more work. Source: none; the
 * executor of GPUOS page §3 Q2 "2. Persistent Kernel Executor" never exits
 * while the process lives, and this call is how a process ends it. */
GPUOS_API int gpuos_stop(gpuos_ctx *ctx, uint32_t timeout_ms);

/* gpuos_stop, then free everything. The context is freed even on error.
 * Source: none on the page (see gpuos_stop); the name gpuos_shutdown is this
 * library's. */
GPUOS_API int gpuos_shutdown(gpuos_ctx *ctx, uint32_t timeout_ms);

/* Sum the worker warps' tile profiles (a snapshot; exact once the executor
 * has left). Errors: EINVAL, ECUDA. Measurement only (where per-op time goes,
 * GPUOS page §3 Q3 latency breakdown); the page has no counterpart. */
GPUOS_API int gpuos_tile_profile_get(gpuos_ctx *ctx, gpuos_tile_profile *out);

/* Source: the page's executor runs one descriptor per warp (GPUOS page §3 Q2
 * "2. Persistent Kernel Executor"); its §4 critique notes the missing
 * multi-block cooperation, which this split into warp tiles supplies.
 * Host tiling rule of a built-in op (what ntiles the library will write);
 * one tile is one warp's unit of work:
 *   add/mul/relu/gelu  ceil(n / te), te the smallest power of two >= n / 16
 *                      within [16384 (a GELU with a dependency: 1024),
 *                      16384 (f32) or 32768 (bf16)]
 *                      elements;
 *                      the device splits n into ntiles ranges of
 *                      round_up(ceil(n / ntiles), 256) elements
 *   row ops            R (one row per tile)
 *   rope, kv_write     B * ceil(H / 4) (one request, four heads per tile)
 *   sdpa               B * H * ceil(Lmax / c), c = round_up(ceil(Lmax / w), 32)
 *                      key rows (at least 32), w = floor(1536 / (B * H)) or 1
 *                      if B * H >= 1536: at most 1536 tiles (or B * H), one
 *                      wave on the default executor; a tile attends at most
 *                      round_up(ceil(Lmax / chunks), 32) rows (the device
 *                      shortens the chunks when the requests' lengths lens[b]
 *                      leave tiles idle: see the sdpa op body)
 *   vecmat             ceil(N / 8) (eight output columns per tile)
 *   nop / empty op     1
 * Returns GPUOS_EINVAL for a descriptor the library would reject. */
GPUOS_API int gpuos_op_ntiles(const gpuos_desc *d, uint32_t *ntiles);

/* Source: the SDPA op of GPUOS page §3 Q2, operator library (attention);
 * the page gives no workspace, which the split-K form here needs.
 * Workspace bytes a decode-SDPA descriptor needs: one uint32 counter per
 * (b, h), rounded up to 4, then fp32 partials for the finest split (32-row
 * chunks). */
GPUOS_API size_t gpuos_sdpa_workspace_bytes(uint32_t B, uint32_t H, uint32_t D, uint32_t Lmax);

/* Source: the eager baseline of GPUOS page §3 Q3 (Table 2, latency
 * breakdown: one kernel launch per operation).
 * Eager baseline: launch the same op bodies as ordinary kernels, one
 * cudaLaunchKernel per descriptor (one warp per tile, one warp per block), in
 * order, on `stream` (a cudaStream_t; 0 = legacy default). Element-wise ops
 * take smaller tiles than in the executor (te within [4096 (GELU: 1024),
 * 4096 (f32) or 8192 (bf16)], the rule above otherwise): a launch runs one
 * op, so its tiles are all its parallelism. With stage_bytes
 * of shared-memory staging per warp as in gpuos_config. Deps are implied by
 * stream order. Does not synchronize. Errors: EINVAL (as gpuos_submit),
 * ECUDA. */
GPUOS_API int gpuos_eager_run(const gpuos_desc *d, uint32_t count, uint32_t stage_bytes, void *stream);

/* Decode attention that allocates nothing. The method has no counterpart of
 * this call; it exists for callers that cannot allocate device memory at the
 * time they attend: code running beside a resident executor (cudaFree, and a
 * cudaMalloc that must grow the heap, wait for an idle device, which a
 * resident executor never gives) and code held to a memory budget fixed up
 * front. It computes what GPUOS_OP_SDPA computes (same op body, one launch on
 * `stream`, a cudaStream_t, 0 = legacy default) with inputs and output given
 * as for that op: q[B][H][D], caches Kc/Vc [B][H][Lcap][D] bf16, lens i32[B]
 * in device memory, out[B][H][D] bf16; all 16-byte aligned; D = 128. Every
 * lens[b] must lie in [1, Lmax]: the lengths stay in device memory, which the
 * call does not read on the host, so a request whose length is outside that
 * range is not detected; its heads' outputs are left unwritten and the call
 * still returns GPUOS_OK. The
 * split-K scratch is a fixed device array inside the library (about 2 MiB per
 * device, held until the process exits) instead of a caller workspace; it
 * bounds B * H <= 256 and Lmax <= 4096, and larger sizes return
 * GPUOS_ETOOBIG. The first call on a device looks up the array's device
 * address (make that call before any stream capture). Every call on a device
 * shares the array and the call clears its counters first, so calls that
 * overlap on the GPU (different streams, no ordering) race: order them.
 * No allocation happens (no cudaMalloc, cudaFree or allocating library
 * routine). Errors: EINVAL, ETOOBIG, ECUDA. Asynchronous: the caller
 * synchronizes `stream`. */
GPUOS_API int gpuos_sdpa_noalloc(const void *q, const void *Kc, const void *Vc, const int32_t *lens, void *out,
                                 uint32_t B, uint32_t H, uint32_t D, uint32_t Lcap, uint32_t Lmax, float scale,
                                 void *stream);

/* CLOCK_REALTIME in ns (the host clock of gpuos_record). Measurement only;
 * the page has no counterpart. */
GPUOS_API uint64_t gpuos_host_now_ns(void);

/* Text for a return code or, with is_status != 0, a device status. The page
 * has no counterpart. */
GPUOS_API const char *gpuos_strerror(int code, int is_status);

#ifdef __cplusplus
}
#endif

#endif /* GPUOS_H */
