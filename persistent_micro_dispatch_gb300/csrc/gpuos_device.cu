/*
 * Device side of the GB300 persistent micro-op dispatcher (sm_103a).
 *
 * Method: "GPUOS: A GPU Operating System Primitive for Transparent Operation
 * Fusion", §2 and §3 Q2. A persistent executor, launched once with one block
 * per SM, polls a single-producer ring of task descriptors with load-acquire,
 * claims work atomically, dispatches it through a device-resident operator
 * table indexed by op_id, releases the slot and backs off exponentially when
 * idle; new operators enter through a dual-slot table flipped by a version
 * counter.
 *
 * GB300 design (what differs from the page's per-warp poll/claim):
 *   - Warp 0 of blocks 0..S-1 (S = 4 by default; those blocks run nothing
 *     else) are the *sequencers*. They take the host ring in windows of 128
 *     tickets in turn: a sequencer polls its window's commit words with
 *     relaxed system-scope loads across NVLink-C2C, takes the committed ones
 *     under one acquire fence, copies them into a device-memory mirror with
 *     the entry point of the table version they run with, and publishes one
 *     work-queue entry per helper warp. Work-queue space is reserved in
 *     ticket order by a turn passed from batch to batch as one word. Only
 *     the sequencers read host memory on the hot path.
 *   - Every other warp is a *worker*. It claims work-queue entries with one
 *     64-bit atomicAdd each (the page's atomic claim); a helper starts with
 *     its own tile and takes further ones from the descriptor's tile counter,
 *     so a large op is split across many warps on many SMs (the page lists
 *     in-kernel multi-block cooperation as missing, §4 "design binding
 *     critique"), while a tiny op is one tile on one warp.
 *   - The last tile of a descriptor completes it: a device-memory done stamp
 *     for dependency waits (released first), then status and timestamps into
 *     the host-visible record and the store-release of the slot's
 *     host-visible completion word, which releases the ring slot to the host.
 *   - Every wait is bounded (dependency and fence waits by dep_timeout_ns,
 *     copies into shared memory by an iteration limit, idle polling by the
 *     host-heartbeat watchdog) and ends in a status, never a trap.
 *   - Ops are memory-bound and use no tensor cores: operands arrive in each
 *     warp's shared-memory staging buffer by TMA bulk copies (or by 16-byte
 *     vector loads that bypass L1: data produced by other SMs inside this
 *     same kernel must not be read from a stale L1 line), fp32 arithmetic,
 *     warp shuffles for reductions.
 */
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "gpuos_internal.h"

#define DEV __device__ __forceinline__

/* ---------------------------------------------------------------------------
 * Memory-order primitives (PTX memory model).
 * ------------------------------------------------------------------------- */
DEV uint64_t ld_acquire_sys(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.acquire.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
DEV uint64_t ld_acquire_gpu(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
DEV uint32_t ld_acquire_gpu32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
/* Spin loops poll with relaxed loads (they read L2 and leave L1 alone) and
 * take the acquire once, with a fence after the poll that succeeded: an
 * acquire load also invalidates the SM's L1, and a spinning warp issuing one
 * per poll would keep evicting the stack of the warp running an op on the
 * same SM; a re-read would cost another L2 round trip. */
DEV uint64_t ld_relaxed_gpu(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
DEV uint64_t ld_relaxed_sys(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.relaxed.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
DEV uint32_t ld_relaxed_sys32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
DEV uint32_t ld_relaxed_gpu32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
DEV void st_release_sys(uint64_t *p, uint64_t v)
{
    asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
DEV void st_release_gpu(uint64_t *p, uint64_t v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
DEV void st_relaxed_sys(uint64_t *p, uint64_t v)
{
    asm volatile("st.relaxed.sys.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
DEV void st_relaxed_sys32(uint32_t *p, uint32_t v)
{
    asm volatile("st.relaxed.sys.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
DEV void st_relaxed_gpu(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
/* Add with release (this thread's earlier writes) and acquire (the writes
 * of every earlier adder) semantics at GPU scope; returns the old value. */
DEV unsigned long long atom_add_acq_rel_gpu(unsigned long long *p, unsigned long long v)
{
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}
DEV uint32_t atom_add_acq_rel_gpu32(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
DEV void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
DEV void st_relaxed_gpu32(uint32_t *p, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
DEV uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
DEV uint32_t lane_id() { return threadIdx.x & 31u; }

/* Elapsed-time accumulator for bounded waits. %globaltimer can read stale
 * right after a launch and can jump when the driver resynchronises it, so a
 * deadline adds up the deltas between consecutive checks, each clamped to
 * 1 ms: one bad reading moves it by at most 1 ms. */
struct Elapsed {
    uint64_t last, acc;
    __device__ __forceinline__ void start() { last = 0; acc = 0; }
    __device__ __forceinline__ uint64_t tick(uint64_t now)
    {
        if (last != 0) {
            uint64_t d = now - last;
            acc += d > 1000000ull ? 1000000ull : d;
        }
        last = now;
        return acc;
    }
};

/* Idle backoff: spin for `spin` polls, then sleep min_ns << k up to max_ns.
 * Workers waiting for work sleep up to the configured cap (power when the
 * ring stays empty); the sequencers' ring poll and the waits on a dependency
 * or a fence, which sit on the dispatch path, sleep at most
 * GPUOS_SHORT_SLEEP_NS. */
DEV uint32_t short_cap(const gpuos_exec_params &p)
{
    return p.backoff_max_ns < GPUOS_SHORT_SLEEP_NS ? p.backoff_max_ns : GPUOS_SHORT_SLEEP_NS;
}
DEV void backoff(uint32_t &polls, uint32_t spin, uint32_t min_ns, uint32_t max_ns, uint64_t *sleeps)
{
    if (polls < spin) {
        polls++;
        return;
    }
    uint32_t k = polls - spin;
    k = k > 16 ? 16 : k;
    uint32_t ns = min_ns << k;
    ns = ns > max_ns ? max_ns : ns;
    __nanosleep(ns);
    polls++;
    (*sleeps)++;
}

/* ---------------------------------------------------------------------------
 * bf16 helpers. Widening is exact; narrowing rounds to nearest-even.
 * ------------------------------------------------------------------------- */
DEV float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
DEV float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
DEV float bf1(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
DEV uint32_t pack_bf2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
DEV uint16_t to_bf(float x)
{
    __nv_bfloat16 v = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&v);
}
DEV void unpack8(const uint4 &v, float *f)
{
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}
DEV uint4 pack8(const float *f)
{
    return make_uint4(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]), pack_bf2(f[4], f[5]), pack_bf2(f[6], f[7]));
}
DEV float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
DEV float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
DEV float warp_min(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

/* ---------------------------------------------------------------------------
 * Per-warp shared-memory staging. Dynamic shared memory of the executor (and
 * of the eager kernel) starts with a 16-byte header {stride, stage_bytes},
 * followed by one region per warp: a 32-byte {mbarrier[2], phase[2]} block
 * and a staging buffer of stage_bytes (16-byte aligned). Single-buffered ops
 * use barrier 0 over the whole buffer; double-buffered ops use barrier i for
 * half i. stage_bytes == 0 means "no staging": ops use their register path.
 * ------------------------------------------------------------------------- */
struct StageHdr {
    uint32_t stride;      /* bytes between warp regions */
    uint32_t stage_bytes; /* staging buffer per warp */
    uint32_t pad[2];
};
struct WarpStage {
    unsigned long long mbar[2]; /* completion barriers of the warp's bulk copies */
    uint32_t phase[2];          /* parity of the next phase to wait for, per barrier */
    uint32_t pad[2];
    /* A row op may take its helper's further rows itself (row_pipe), so
     * that it can copy the next row while it works on the current one. The
     * worker sets claim_ctr (the descriptor's tile counter; null: one tile
     * per call) and claim_base (its helper count) before the call; an op
     * that took rows itself sets claim_done and reports the tiles it ran or
     * skipped (claim_count) and the next claimed tile (claim_next, >= the
     * tile count once none is left). */
    uint32_t *claim_ctr;
    uint32_t claim_base, claim_count, claim_next, claim_done;
    uint32_t pad2[2];
};
#define GPUOS_WARP_STAGE_HDR 64u
static_assert(sizeof(WarpStage) == GPUOS_WARP_STAGE_HDR, "warp staging header");
extern __shared__ __align__(16) unsigned char g_dyn_smem[];

DEV StageHdr *stage_hdr() { return reinterpret_cast<StageHdr *>(g_dyn_smem); }
DEV WarpStage *warp_stage()
{
    return reinterpret_cast<WarpStage *>(g_dyn_smem + 16 + (threadIdx.x >> 5) * stage_hdr()->stride);
}
DEV unsigned char *warp_stage_buf() { return reinterpret_cast<unsigned char *>(warp_stage()) + GPUOS_WARP_STAGE_HDR; }
DEV uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

/* Lay out the header and every warp's barriers (all threads of the block). */
DEV void stage_init(uint32_t stage_bytes)
{
    if (threadIdx.x == 0) {
        stage_hdr()->stride = GPUOS_WARP_STAGE_HDR + stage_bytes;
        stage_hdr()->stage_bytes = stage_bytes;
    }
    __syncthreads();
    if ((threadIdx.x & 31u) == 0) {
        WarpStage *w = warp_stage();
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&w->mbar[0])) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&w->mbar[1])) : "memory");
        w->phase[0] = 0;
        w->phase[1] = 0;
        w->claim_ctr = nullptr;
        w->claim_done = 0;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
}

/* Bulk-copy `bytes` (multiple of 16, 16-byte aligned ends) from global to the
 * warp's shared buffer; completes on the warp's mbarrier (lane 0 only). */
DEV void bulk_g2s(void *sdst, const void *gsrc, uint32_t bytes, unsigned long long *mbar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(sdst)), "l"(gsrc), "r"(bytes), "r"(smem_addr(mbar)) : "memory");
}
DEV void mbar_expect(unsigned long long *mbar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(mbar)), "r"(bytes) : "memory");
}
/* Wait (bounded) for the phase of the given parity; false if the bound ran
 * out. Every lane calls it. */
DEV bool mbar_wait(unsigned long long *mbar, uint32_t parity)
{
    const uint32_t a = smem_addr(mbar);
    for (uint32_t i = 0; i < (1u << 24); i++) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done) : "r"(a), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}

/* ===========================================================================
 * Operator library. Every op is a warp-cooperative device function
 *     int op(const gpuos_devdesc *d, uint32_t tile)
 * called by all 32 lanes of one warp with the same arguments; it returns a
 * GPUOS_ST_* status, identical on every lane. Tiles past the end of an op
 * are no-ops.
 * ======================================================================== */

enum { EW_ADD = 0, EW_MUL = 1, EW_RELU = 2, EW_GELU = 3 };

/* erfc(x) by the Chebyshev fit of Numerical Recipes (Press, Teukolsky,
 * Vetterling, Flannery, 2nd ed., section 6.2, function erfcc): for z = |x|,
 * t = 1 / (1 + z/2), erfc(z) = t exp(-z^2 + P(t)) with a degree-9 polynomial
 * P, fractional error below 1.2e-7 for every z >= 0; erfc(-z) = 2 - erfc(z).
 * No branch: one hardware reciprocal, one hardware exp2 and about fifteen
 * multiply-adds per element, a fraction of a library erfc's code (the op
 * bodies run from a cold instruction cache more often than not). */
DEV float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
/* e^y as 2^(y log2 e): the product's rounding error is carried as a residual
 * (one fma) and applied to first order, so the result keeps the accuracy of
 * the hardware's ex2 (a few ulps) for |y| up to ~87. */
DEV float exp_ex2(float y)
{
    const float t = y * 1.44269504f;
    const float e = fmaf(y, 1.44269504f, -t) + y * 1.92596299e-8f;
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return fmaf(r, e * 0.693147181f, r);
}
DEV float erfc_nr(float x)
{
    const float z = fabsf(x);
    const float t = rcp_approx(fmaf(0.5f, z, 1.0f));
    float p = 0.17087277f;
    p = fmaf(t, p, -0.82215223f);
    p = fmaf(t, p, 1.48851587f);
    p = fmaf(t, p, -1.13520398f);
    p = fmaf(t, p, 0.27886807f);
    p = fmaf(t, p, -0.18628806f);
    p = fmaf(t, p, 0.09678418f);
    p = fmaf(t, p, 0.37409196f);
    p = fmaf(t, p, 1.00002368f);
    p = fmaf(t, p, -1.26551223f);
    const float r = t * exp_ex2(fmaf(-z, z, p));
    return x >= 0.0f ? r : 2.0f - r;
}

template <int OP>
DEV float ew1(float a, float b)
{
    if (OP == EW_ADD) return __fadd_rn(a, b);
    if (OP == EW_MUL) return __fmul_rn(a, b);
    if (OP == EW_RELU) return a > 0.0f ? a : 0.0f;
    /* GELU, exact form x * Phi(x) with Phi(x) = erfc(-x / sqrt 2) / 2: the
     * complementary error function keeps full relative accuracy for x < 0,
     * where 1 + erf(x / sqrt 2) would cancel */
    return 0.5f * a * erfc_nr(-a * 0.70710678118654752f);
}

template <int OP, bool BF>
DEV uint4 ew_vec(const uint4 &va, const uint4 &vb)
{
    if (BF) {
        float fa[8], fb[8], r[8];
        unpack8(va, fa);
        unpack8(vb, fb);
#pragma unroll
        for (int i = 0; i < 8; i++) r[i] = ew1<OP>(fa[i], fb[i]);
        return pack8(r);
    } else {
        uint4 r;
        r.x = __float_as_uint(ew1<OP>(__uint_as_float(va.x), __uint_as_float(vb.x)));
        r.y = __float_as_uint(ew1<OP>(__uint_as_float(va.y), __uint_as_float(vb.y)));
        r.z = __float_as_uint(ew1<OP>(__uint_as_float(va.z), __uint_as_float(vb.z)));
        r.w = __float_as_uint(ew1<OP>(__uint_as_float(va.w), __uint_as_float(vb.w)));
        return r;
    }
}

/* Elements per tile of an element-wise op. The host chose ntiles as
 * ceil(n / te) for a te that is a multiple of GPUOS_EW_ALIGN; rounding
 * ceil(n / ntiles) up to that multiple gives back a size no larger than te
 * whose ntiles tiles cover n, so tile starts stay 16-byte aligned. */
DEV uint32_t ew_tile_elems(uint64_t n, uint32_t ntiles)
{
    const uint64_t nt = ntiles ? ntiles : 1u;
    const uint64_t per = (n + nt - 1) / nt;
    return (uint32_t)((per + GPUOS_EW_ALIGN - 1) / GPUOS_EW_ALIGN * GPUOS_EW_ALIGN);
}

/* Element-wise tile in registers: rounds of 8 (GELU: 2) independent 16-byte
 * vector loads per operand per lane. Unaligned operands take a scalar path
 * with the same arithmetic. */
template <int OP, bool BF>
DEV int ew_tile(const gpuos_devdesc *d, uint32_t tile)
{
    constexpr uint32_t VEC = BF ? 8 : 4;
    constexpr uint32_t ES = BF ? 2 : 4;
    constexpr bool BIN = (OP == EW_ADD || OP == EW_MUL);
    constexpr int U = (OP == EW_GELU) ? 2 : 8; /* GELU: short code, it is long per element */
    const uint32_t lane = lane_id();
    const uint64_t n = d->dims[0];
    const uint32_t TILE = ew_tile_elems(n, d->ntiles);
    const uint64_t start = (uint64_t)tile * TILE;
    if (start >= n) return GPUOS_ST_OK;
    const uint32_t cnt = (uint32_t)((n - start) < TILE ? (n - start) : TILE);
    const char *pa = reinterpret_cast<const char *>(d->a) + start * ES;
    const char *pb = BIN ? reinterpret_cast<const char *>(d->b) + start * ES : pa;
    char *po = reinterpret_cast<char *>(d->out) + start * ES;
    const bool aligned = (((uintptr_t)pa | (uintptr_t)pb | (uintptr_t)po) & 15u) == 0;
    const uint32_t nvec = aligned ? cnt / VEC : 0;
    const uint4 *va = reinterpret_cast<const uint4 *>(pa);
    const uint4 *vb = reinterpret_cast<const uint4 *>(pb);
    uint4 *vo = reinterpret_cast<uint4 *>(po);
    for (uint32_t v0 = 0; v0 < nvec; v0 += 32 * U) {
        uint4 ra[U], rb[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const uint32_t v = v0 + u * 32 + lane;
            if (v < nvec) {
                ra[u] = __ldcg(va + v);
                rb[u] = BIN ? __ldcg(vb + v) : ra[u];
            }
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const uint32_t v = v0 + u * 32 + lane;
            if (v < nvec) __stcg(vo + v, ew_vec<OP, BF>(ra[u], rb[u]));
        }
    }
    for (uint32_t i = nvec * VEC + lane; i < cnt; i += 32) {
        if (BF) {
            const uint16_t *a16 = reinterpret_cast<const uint16_t *>(pa);
            const uint16_t *b16 = reinterpret_cast<const uint16_t *>(pb);
            reinterpret_cast<uint16_t *>(po)[i] = to_bf(ew1<OP>(bf1(a16[i]), bf1(b16[i])));
        } else {
            const float *a32 = reinterpret_cast<const float *>(pa);
            const float *b32 = reinterpret_cast<const float *>(pb);
            reinterpret_cast<float *>(po)[i] = ew1<OP>(a32[i], b32[i]);
        }
    }
    return GPUOS_ST_OK;
}

/* Element-wise tile through the warp's shared staging buffer: lane 0 issues
 * one TMA bulk copy per operand and chunk (up to stage_bytes in flight per
 * warp, no registers held), every lane waits on the warp's mbarrier, then
 * computes from shared memory and stores 16-byte vectors. Used when every
 * operand is 16-byte aligned; the ragged tail takes the scalar path. */
template <int OP, bool BF>
DEV int ew_tile_staged(const gpuos_devdesc *d, uint32_t tile, uint32_t stage_bytes)
{
    constexpr uint32_t VEC = BF ? 8 : 4;
    constexpr uint32_t ES = BF ? 2 : 4;
    constexpr bool BIN = (OP == EW_ADD || OP == EW_MUL);
    constexpr uint32_t NOPS = BIN ? 2 : 1;
    const uint32_t lane = lane_id();
    const uint64_t n = d->dims[0];
    const uint32_t TILE = ew_tile_elems(n, d->ntiles);
    const uint64_t start = (uint64_t)tile * TILE;
    if (start >= n) return GPUOS_ST_OK;
    const uint32_t cnt = (uint32_t)((n - start) < TILE ? (n - start) : TILE);
    const char *pa = reinterpret_cast<const char *>(d->a) + start * ES;
    const char *pb = BIN ? reinterpret_cast<const char *>(d->b) + start * ES : pa;
    char *po = reinterpret_cast<char *>(d->out) + start * ES;
    const uint32_t nel = cnt / VEC * VEC;                      /* whole 16-byte vectors */
    const uint32_t chunk = (stage_bytes / NOPS) / 16u * 16u / ES; /* elements per operand */
    WarpStage *w = warp_stage();
    unsigned char *sa = warp_stage_buf();
    unsigned char *sb = sa + chunk * ES;
    uint32_t phase = w->phase[0];
    int32_t st = GPUOS_ST_OK;
    for (uint32_t c0 = 0; c0 < nel; c0 += chunk) {
        const uint32_t ce = (nel - c0) < chunk ? (nel - c0) : chunk;
        const uint32_t bytes = ce * ES;
        if (lane == 0) {
            /* earlier generic reads of the buffer before the async writes */
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_expect(&w->mbar[0], bytes * NOPS);
            bulk_g2s(sa, pa + (uint64_t)c0 * ES, bytes, &w->mbar[0]);
            if (BIN) bulk_g2s(sb, pb + (uint64_t)c0 * ES, bytes, &w->mbar[0]);
        }
        if (!mbar_wait(&w->mbar[0], phase)) {
            /* the copy did not land within the bound: wait once more (also
             * bounded) so that no copy is left writing the buffer, then fail */
            mbar_wait(&w->mbar[0], phase);
            st = GPUOS_ST_COPY_TIMEOUT;
            phase ^= 1u;
            break;
        }
        phase ^= 1u;
        const uint4 *va = reinterpret_cast<const uint4 *>(sa);
        const uint4 *vb = reinterpret_cast<const uint4 *>(sb);
        uint4 *vo = reinterpret_cast<uint4 *>(po + (uint64_t)c0 * ES);
        const uint32_t nv = bytes / 16u;
        if (OP == EW_GELU) {
#pragma unroll 1
            for (uint32_t v = lane; v < nv; v += 32) {
                const uint4 x = va[v];
                __stcg(vo + v, ew_vec<OP, BF>(x, x));
            }
        } else {
#pragma unroll 4
            for (uint32_t v = lane; v < nv; v += 32) {
                const uint4 x = va[v];
                __stcg(vo + v, ew_vec<OP, BF>(x, BIN ? vb[v] : x));
            }
        }
        __syncwarp();
    }
    if (lane == 0) w->phase[0] = phase;
    __syncwarp();
    for (uint32_t i = nel + lane; i < cnt; i += 32) {
        if (BF) {
            const uint16_t *a16 = reinterpret_cast<const uint16_t *>(pa);
            const uint16_t *b16 = reinterpret_cast<const uint16_t *>(pb);
            reinterpret_cast<uint16_t *>(po)[i] = to_bf(ew1<OP>(bf1(a16[i]), bf1(b16[i])));
        } else {
            const float *a32 = reinterpret_cast<const float *>(pa);
            const float *b32 = reinterpret_cast<const float *>(pb);
            reinterpret_cast<float *>(po)[i] = ew1<OP>(a32[i], b32[i]);
        }
    }
    return st;
}

template <int OP, bool BF>
DEV int ew_pick(const gpuos_devdesc *d, uint32_t tile)
{
    const uint32_t sbytes = stage_hdr()->stage_bytes;
    const bool bin = (OP == EW_ADD || OP == EW_MUL);
    const uint64_t al = d->a | (bin ? d->b : 0) | d->out;
    if (sbytes >= 2048 && (al & 15u) == 0) return ew_tile_staged<OP, BF>(d, tile, sbytes);
    return ew_tile<OP, BF>(d, tile);
}

template <int OP>
DEV int ew_dispatch(const gpuos_devdesc *d, uint32_t tile)
{
    if (d->dtype == GPUOS_BF16) return ew_pick<OP, true>(d, tile);
    if (d->dtype == GPUOS_F32) return ew_pick<OP, false>(d, tile);
    return GPUOS_ST_BAD_ARGS;
}

/* ---- row ops: one row per tile -------------------------------------------- */
enum { ROW_SOFTMAX = 0, ROW_LN = 1, ROW_SUM = 2, ROW_MAX = 3, ROW_MIN = 4 };

/* Rows of H <= GPUOS_ROW_REG_MAX bf16 with H % 8 == 0 and 16-byte aligned
 * operands: the row is read once into registers (16 vectors per lane). */
template <int K>
DEV int row_reg(const gpuos_devdesc *d, uint32_t row, uint32_t H)
{
    constexpr int J = GPUOS_ROW_REG_MAX / 256;
    const uint32_t lane = lane_id();
    const uint32_t nv = H / 8;
    const uint4 *x = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(d->a) + (uint64_t)row * H);
    /* LayerNorm: gamma and beta come into the warp's staging buffer by TMA
     * bulk copies issued before the row is read, so their latency hides
     * behind the row load and the two reductions */
    const bool stg = (K == ROW_LN) && stage_hdr()->stage_bytes >= 4u * H;
    WarpStage *w = warp_stage();
    const uint4 *sgam = reinterpret_cast<const uint4 *>(warp_stage_buf());
    const uint4 *sbet = sgam + nv;
    if (stg && lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect(&w->mbar[0], 4u * H);
        bulk_g2s(warp_stage_buf(), reinterpret_cast<const void *>(d->b), 2u * H, &w->mbar[0]);
        bulk_g2s(warp_stage_buf() + 2u * H, reinterpret_cast<const void *>(d->aux0), 2u * H, &w->mbar[0]);
    }
    uint4 r[J];
#pragma unroll
    for (int j = 0; j < J; j++) {
        const uint32_t v = lane + 32u * j;
        if (v < nv) r[j] = __ldcg(x + v);
    }
    /* reductions keep one accumulator per element of a vector: eight
     * independent chains of J steps instead of one chain of 8 J */
    if (K == ROW_SUM || K == ROW_MAX || K == ROW_MIN) {
        const float init = (K == ROW_SUM) ? 0.0f : (K == ROW_MAX ? -INFINITY : INFINITY);
        float a8[8];
#pragma unroll
        for (int i = 0; i < 8; i++) a8[i] = init;
#pragma unroll
        for (int j = 0; j < J; j++) {
            const uint32_t v = lane + 32u * j;
            if (v < nv) {
                float f[8];
                unpack8(r[j], f);
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    if (K == ROW_SUM) a8[i] += f[i];
                    else if (K == ROW_MAX) a8[i] = fmaxf(a8[i], f[i]);
                    else a8[i] = fminf(a8[i], f[i]);
                }
            }
        }
        float acc = a8[0];
#pragma unroll
        for (int i = 1; i < 8; i++) {
            if (K == ROW_SUM) acc += a8[i];
            else if (K == ROW_MAX) acc = fmaxf(acc, a8[i]);
            else acc = fminf(acc, a8[i]);
        }
        if (K == ROW_SUM) acc = warp_sum(acc);
        else if (K == ROW_MAX) acc = warp_max(acc);
        else acc = warp_min(acc);
        if (lane == 0) {
            if (K == ROW_SUM) reinterpret_cast<float *>(d->out)[row] = acc;
            else reinterpret_cast<uint16_t *>(d->out)[row] = to_bf(acc);
        }
        return GPUOS_ST_OK;
    }
    uint4 *y = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(d->out) + (uint64_t)row * H);
    if (K == ROW_SOFTMAX) {
        float m8[8], s8[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            m8[i] = -INFINITY;
            s8[i] = 0.0f;
        }
#pragma unroll
        for (int j = 0; j < J; j++) {
            if (lane + 32u * j < nv) {
                float f[8];
                unpack8(r[j], f);
#pragma unroll
                for (int i = 0; i < 8; i++) m8[i] = fmaxf(m8[i], f[i]);
            }
        }
        float m = m8[0];
#pragma unroll
        for (int i = 1; i < 8; i++) m = fmaxf(m, m8[i]);
        m = warp_max(m);
#pragma unroll
        for (int j = 0; j < J; j++) {
            if (lane + 32u * j < nv) {
                float f[8];
                unpack8(r[j], f);
#pragma unroll
                for (int i = 0; i < 8; i++) s8[i] += __expf(f[i] - m);
            }
        }
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; i++) s += s8[i];
        const float inv = 1.0f / warp_sum(s);
#pragma unroll
        for (int j = 0; j < J; j++) {
            const uint32_t v = lane + 32u * j;
            if (v < nv) {
                float f[8];
                unpack8(r[j], f);
#pragma unroll
                for (int i = 0; i < 8; i++) f[i] = __expf(f[i] - m) * inv;
                __stcg(y + v, pack8(f));
            }
        }
        return GPUOS_ST_OK;
    }
    /* LayerNorm: biased variance, two passes over the registers. */
    float s8[8], q8[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        s8[i] = 0.0f;
        q8[i] = 0.0f;
    }
#pragma unroll
    for (int j = 0; j < J; j++) {
        if (lane + 32u * j < nv) {
            float f[8];
            unpack8(r[j], f);
#pragma unroll
            for (int i = 0; i < 8; i++) s8[i] += f[i];
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) s += s8[i];
    const float mean = warp_sum(s) / (float)H;
#pragma unroll
    for (int j = 0; j < J; j++) {
        if (lane + 32u * j < nv) {
            float f[8];
            unpack8(r[j], f);
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const float t = f[i] - mean;
                q8[i] = fmaf(t, t, q8[i]);
            }
        }
    }
    float q = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) q += q8[i];
    const float rstd = rsqrtf(warp_sum(q) / (float)H + d->fparam[0]);
    const uint4 *g = reinterpret_cast<const uint4 *>(d->b);
    const uint4 *bt = reinterpret_cast<const uint4 *>(d->aux0);
    if (stg) {
        const uint32_t ph = w->phase[0];
        const bool ok = mbar_wait(&w->mbar[0], ph);
        if (!ok) mbar_wait(&w->mbar[0], ph); /* leave no copy writing the buffer */
        __syncwarp();
        if (lane == 0) w->phase[0] = ph ^ 1u;
        __syncwarp();
        if (!ok) return GPUOS_ST_COPY_TIMEOUT;
    }
#pragma unroll
    for (int j = 0; j < J; j++) {
        const uint32_t v = lane + 32u * j;
        if (v < nv) {
            float f[8], gf[8], bf[8];
            unpack8(r[j], f);
            unpack8(stg ? sgam[v] : __ldcg(g + v), gf);
            unpack8(stg ? sbet[v] : __ldcg(bt + v), bf);
#pragma unroll
            for (int i = 0; i < 8; i++) f[i] = (f[i] - mean) * rstd * gf[i] + bf[i];
            __stcg(y + v, pack8(f));
        }
    }
    __syncwarp(); /* every lane's reads of the buffer before it is reused */
    return GPUOS_ST_OK;
}

/* Rows staged in the warp's shared buffer: the row (and LayerNorm's gamma
 * and beta) arrive by TMA bulk copies and every pass is a rolled loop over
 * shared memory, so the code a tile runs stays a few hundred instructions
 * (the op bodies mostly run from a cold instruction cache). LayerNorm rows
 * whose x, gamma and beta do not fit together keep x resident and stream
 * gamma and beta through the rest of the buffer in column chunks. */
DEV bool stage_wait0(WarpStage *w)
{
    const uint32_t ph = w->phase[0];
    const bool ok = mbar_wait(&w->mbar[0], ph);
    if (!ok) mbar_wait(&w->mbar[0], ph); /* leave no copy writing the buffer */
    __syncwarp();
    if (lane_id() == 0) w->phase[0] = ph ^ 1u;
    __syncwarp();
    return ok;
}

template <int K>
DEV int row_staged(const gpuos_devdesc *d, uint32_t row, uint32_t H, uint32_t C)
{
    const uint32_t lane = lane_id(), nv = H / 8;
    WarpStage *w = warp_stage();
    unsigned char *buf = warp_stage_buf();
    const uint4 *sx = reinterpret_cast<const uint4 *>(buf);
    const uint16_t *x = reinterpret_cast<const uint16_t *>(d->a) + (uint64_t)row * H;
    if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect(&w->mbar[0], 2u * H + (K == ROW_LN ? 4u * C : 0u));
        bulk_g2s(buf, x, 2u * H, &w->mbar[0]);
        if (K == ROW_LN) {
            bulk_g2s(buf + 2u * H, reinterpret_cast<const void *>(d->b), 2u * C, &w->mbar[0]);
            bulk_g2s(buf + 2u * H + 2u * C, reinterpret_cast<const void *>(d->aux0), 2u * C, &w->mbar[0]);
        }
    }
    if (!stage_wait0(w)) return GPUOS_ST_COPY_TIMEOUT;
    if (K == ROW_SUM || K == ROW_MAX || K == ROW_MIN) {
        const float init = (K == ROW_SUM) ? 0.0f : (K == ROW_MAX ? -INFINITY : INFINITY);
        float a8[8];
#pragma unroll
        for (int i = 0; i < 8; i++) a8[i] = init;
#pragma unroll 1
        for (uint32_t v = lane; v < nv; v += 32) {
            float f[8];
            unpack8(sx[v], f);
#pragma unroll
            for (int i = 0; i < 8; i++) {
                if (K == ROW_SUM) a8[i] += f[i];
                else if (K == ROW_MAX) a8[i] = fmaxf(a8[i], f[i]);
                else a8[i] = fminf(a8[i], f[i]);
            }
        }
        float acc = a8[0];
#pragma unroll
        for (int i = 1; i < 8; i++) {
            if (K == ROW_SUM) acc += a8[i];
            else if (K == ROW_MAX) acc = fmaxf(acc, a8[i]);
            else acc = fminf(acc, a8[i]);
        }
        if (K == ROW_SUM) acc = warp_sum(acc);
        else if (K == ROW_MAX) acc = warp_max(acc);
        else acc = warp_min(acc);
        if (lane == 0) {
            if (K == ROW_SUM) reinterpret_cast<float *>(d->out)[row] = acc;
            else reinterpret_cast<uint16_t *>(d->out)[row] = to_bf(acc);
        }
        __syncwarp();
        return GPUOS_ST_OK;
    }
    uint4 *y = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(d->out) + (uint64_t)row * H);
    if (K == ROW_SOFTMAX) {
        float m = -INFINITY;
#pragma unroll 1
        for (uint32_t v = lane; v < nv; v += 32) {
            float f[8];
            unpack8(sx[v], f);
#pragma unroll
            for (int i = 0; i < 8; i++) m = fmaxf(m, f[i]);
        }
        m = warp_max(m);
        float s8[8];
#pragma unroll
        for (int i = 0; i < 8; i++) s8[i] = 0.0f;
#pragma unroll 1
        for (uint32_t v = lane; v < nv; v += 32) {
            float f[8];
            unpack8(sx[v], f);
#pragma unroll
            for (int i = 0; i < 8; i++) s8[i] += __expf(f[i] - m);
        }
        float sum = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; i++) sum += s8[i];
        const float inv = 1.0f / warp_sum(sum);
#pragma unroll 1
        for (uint32_t v = lane; v < nv; v += 32) {
            float f[8];
            unpack8(sx[v], f);
#pragma unroll
            for (int i = 0; i < 8; i++) f[i] = __expf(f[i] - m) * inv;
            __stcg(y + v, pack8(f));
        }
        __syncwarp();
        return GPUOS_ST_OK;
    }
    /* LayerNorm: biased variance, mean and variance in two passes */
    float s8[8];
#pragma unroll
    for (int i = 0; i < 8; i++) s8[i] = 0.0f;
#pragma unroll 1
    for (uint32_t v = lane; v < nv; v += 32) {
        float f[8];
        unpack8(sx[v], f);
#pragma unroll
        for (int i = 0; i < 8; i++) s8[i] += f[i];
    }
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) sum += s8[i];
    const float mean = warp_sum(sum) / (float)H;
#pragma unroll
    for (int i = 0; i < 8; i++) s8[i] = 0.0f;
#pragma unroll 1
    for (uint32_t v = lane; v < nv; v += 32) {
        float f[8];
        unpack8(sx[v], f);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float t = f[i] - mean;
            s8[i] = fmaf(t, t, s8[i]);
        }
    }
    float q = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) q += s8[i];
    const float rstd = rsqrtf(warp_sum(q) / (float)H + d->fparam[0]);
    const uint4 *sg = sx + nv;
    const uint32_t cv = C / 8; /* vectors per gamma/beta chunk */
    for (uint32_t c0 = 0; c0 < nv; c0 += cv) {
        if (c0 > 0) {
            /* next chunk of gamma and beta, once every lane is done with this one */
            __syncwarp();
            const uint32_t cb = min(cv, nv - c0) * 16u;
            if (lane == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_expect(&w->mbar[0], 2u * cb);
                bulk_g2s(buf + 2u * H, reinterpret_cast<const unsigned char *>(d->b) + c0 * 16u, cb, &w->mbar[0]);
                bulk_g2s(buf + 2u * H + 2u * C, reinterpret_cast<const unsigned char *>(d->aux0) + c0 * 16u, cb,
                         &w->mbar[0]);
            }
            if (!stage_wait0(w)) return GPUOS_ST_COPY_TIMEOUT;
        }
        const uint32_t ce = min(nv, c0 + cv);
#pragma unroll 1
        for (uint32_t v = c0 + lane; v < ce; v += 32) {
            float f[8], gf[8], bf[8];
            unpack8(sx[v], f);
            unpack8(sg[v - c0], gf);
            unpack8(sg[cv + v - c0], bf);
#pragma unroll
            for (int i = 0; i < 8; i++) f[i] = (f[i] - mean) * rstd * gf[i] + bf[i];
            __stcg(y + v, pack8(f));
        }
    }
    __syncwarp(); /* every lane's reads of the buffer before it is reused */
    return GPUOS_ST_OK;
}

/* Any width or alignment: scalar passes re-reading the row. */
template <int K>
DEV int row_generic(const gpuos_devdesc *d, uint32_t row, uint32_t H)
{
    const uint32_t lane = lane_id();
    const uint16_t *x = reinterpret_cast<const uint16_t *>(d->a) + (uint64_t)row * H;
    if (K == ROW_SUM || K == ROW_MAX || K == ROW_MIN) {
        float acc = (K == ROW_SUM) ? 0.0f : (K == ROW_MAX ? -INFINITY : INFINITY);
        for (uint32_t j = lane; j < H; j += 32) {
            const float f = bf1(__ldcg(x + j));
            if (K == ROW_SUM) acc += f;
            else if (K == ROW_MAX) acc = fmaxf(acc, f);
            else acc = fminf(acc, f);
        }
        if (K == ROW_SUM) acc = warp_sum(acc);
        else if (K == ROW_MAX) acc = warp_max(acc);
        else acc = warp_min(acc);
        if (lane == 0) {
            if (K == ROW_SUM) reinterpret_cast<float *>(d->out)[row] = acc;
            else reinterpret_cast<uint16_t *>(d->out)[row] = to_bf(acc);
        }
        return GPUOS_ST_OK;
    }
    uint16_t *y = reinterpret_cast<uint16_t *>(d->out) + (uint64_t)row * H;
    if (K == ROW_SOFTMAX) {
        float m = -INFINITY;
        for (uint32_t j = lane; j < H; j += 32) m = fmaxf(m, bf1(__ldcg(x + j)));
        m = warp_max(m);
        float s = 0.0f;
        for (uint32_t j = lane; j < H; j += 32) s += __expf(bf1(__ldcg(x + j)) - m);
        const float inv = 1.0f / warp_sum(s);
        for (uint32_t j = lane; j < H; j += 32) y[j] = to_bf(__expf(bf1(__ldcg(x + j)) - m) * inv);
        return GPUOS_ST_OK;
    }
    float s = 0.0f;
    for (uint32_t j = lane; j < H; j += 32) s += bf1(__ldcg(x + j));
    const float mean = warp_sum(s) / (float)H;
    float q = 0.0f;
    for (uint32_t j = lane; j < H; j += 32) {
        const float t = bf1(__ldcg(x + j)) - mean;
        q += t * t;
    }
    const float rstd = rsqrtf(warp_sum(q) / (float)H + d->fparam[0]);
    const uint16_t *g = reinterpret_cast<const uint16_t *>(d->b);
    const uint16_t *bt = reinterpret_cast<const uint16_t *>(d->aux0);
    for (uint32_t j = lane; j < H; j += 32)
        y[j] = to_bf((bf1(__ldcg(x + j)) - mean) * rstd * bf1(__ldcg(g + j)) + bf1(__ldcg(bt + j)));
    return GPUOS_ST_OK;
}

/* Lane 0: bulk-copy row `row` (2H bytes) into half hb of the warp's buffer. */
DEV void row_issue(WarpStage *w, unsigned char *half, const uint16_t *X, uint32_t row, uint32_t H, uint32_t hb)
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_expect(&w->mbar[hb], 2u * H);
    bulk_g2s(half, X + (uint64_t)row * H, 2u * H, &w->mbar[hb]);
}

/* Rows that fit half the staging buffer (softmax, row sum/max/min:
 * 4H <= stage_bytes; LayerNorm, whose gamma and beta stay in the buffer for
 * all of the helper's rows: 8H <= stage_bytes; H % 8 == 0, 16-byte aligned):
 * the op takes its helper's rows itself. While one row is worked on in one
 * half of the row space, the next row (claimed from the descriptor's tile
 * counter) is already on its way into the other, so a helper's rows after
 * the first cost their passes, not a copy round trip each; and the helper's
 * rows run in one call of the op. Without a claim context (the eager
 * kernel) it runs the one row. Buffer: [gamma | beta] (LayerNorm only),
 * then two row halves. The passes are rolled loops: unrolled twice, the
 * row stream ran 17 % slower (more code to fetch per op, five row ops in
 * turn on every SM). */
template <int K>
DEV int row_pipe(const gpuos_devdesc *d, uint32_t row, uint32_t R, uint32_t H)
{
    const uint32_t lane = lane_id(), nv = H / 8;
    WarpStage *w = warp_stage();
    unsigned char *buf = warp_stage_buf();
    const uint32_t roff = (K == ROW_LN) ? 4u * H : 0u;
    const uint32_t hbytes = (K == ROW_LN) ? 2u * H : stage_hdr()->stage_bytes / 2u;
    uint32_t *ctr = w->claim_ctr;
    const uint32_t base = w->claim_base;
    const bool claim = ctr != nullptr && base < R;
    const uint16_t *X = reinterpret_cast<const uint16_t *>(d->a);
    uint32_t ph = w->phase[0] | (w->phase[1] << 1); /* bit hb: parity to wait for on half hb */
    uint32_t hb = 0, count = 0, next = R;
    int32_t st = GPUOS_ST_OK;
    if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect(&w->mbar[0], 2u * H + (K == ROW_LN ? 4u * H : 0u));
        bulk_g2s(buf + roff, X + (uint64_t)row * H, 2u * H, &w->mbar[0]);
        if (K == ROW_LN) {
            bulk_g2s(buf, reinterpret_cast<const void *>(d->b), 2u * H, &w->mbar[0]);
            bulk_g2s(buf + 2u * H, reinterpret_cast<const void *>(d->aux0), 2u * H, &w->mbar[0]);
        }
    }
    while (true) {
        /* the next row: claimed, and its copy started into the other half */
        uint32_t nx = R;
        if (claim && lane == 0) {
            nx = base + atomicAdd(ctr, 1u);
            if (nx < R) row_issue(w, buf + roff + (hb ^ 1u) * hbytes, X, nx, H, hb ^ 1u);
        }
        nx = __shfl_sync(0xFFFFFFFFu, nx, 0);
        count++;
        if (!mbar_wait(&w->mbar[hb], (ph >> hb) & 1u)) {
            /* leave no copy writing the buffer: wait once more (bounded) on
             * this half and on the other if a copy went out to it; the
             * claimed next row goes back to the worker, which counts it */
            mbar_wait(&w->mbar[hb], (ph >> hb) & 1u);
            ph ^= 1u << hb;
            if (nx < R) {
                mbar_wait(&w->mbar[hb ^ 1u], (ph >> (hb ^ 1u)) & 1u);
                ph ^= 1u << (hb ^ 1u);
            }
            st = GPUOS_ST_COPY_TIMEOUT;
            next = nx;
            break;
        }
        ph ^= 1u << hb;
        const uint4 *sx = reinterpret_cast<const uint4 *>(buf + roff + hb * hbytes);
        if (K == ROW_LN) {
            /* biased variance, mean and variance in two passes */
            uint4 *y = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(d->out) + (uint64_t)row * H);
            const uint4 *sg = reinterpret_cast<const uint4 *>(buf);
            const uint4 *sbt = sg + nv;
            float s8[8];
#pragma unroll
            for (int i = 0; i < 8; i++) s8[i] = 0.0f;
#pragma unroll 1
            for (uint32_t v = lane; v < nv; v += 32) {
                float f[8];
                unpack8(sx[v], f);
#pragma unroll
                for (int i = 0; i < 8; i++) s8[i] += f[i];
            }
            float sum = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; i++) sum += s8[i];
            const float mean = warp_sum(sum) / (float)H;
#pragma unroll
            for (int i = 0; i < 8; i++) s8[i] = 0.0f;
#pragma unroll 1
            for (uint32_t v = lane; v < nv; v += 32) {
                float f[8];
                unpack8(sx[v], f);
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const float t = f[i] - mean;
                    s8[i] = fmaf(t, t, s8[i]);
                }
            }
            float q = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; i++) q += s8[i];
            const float rstd = rsqrtf(warp_sum(q) / (float)H + d->fparam[0]);
#pragma unroll 1
            for (uint32_t v = lane; v < nv; v += 32) {
                float f[8], gf[8], bf[8];
                unpack8(sx[v], f);
                unpack8(sg[v], gf);
                unpack8(sbt[v], bf);
#pragma unroll
                for (int i = 0; i < 8; i++) f[i] = (f[i] - mean) * rstd * gf[i] + bf[i];
                __stcg(y + v, pack8(f));
            }
        } else if (K == ROW_SUM || K == ROW_MAX || K == ROW_MIN) {
            const float init = (K == ROW_SUM) ? 0.0f : (K == ROW_MAX ? -INFINITY : INFINITY);
            float a8[8];
#pragma unroll
            for (int i = 0; i < 8; i++) a8[i] = init;
#pragma unroll 1
            for (uint32_t v = lane; v < nv; v += 32) {
                float f[8];
                unpack8(sx[v], f);
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    if (K == ROW_SUM) a8[i] += f[i];
                    else if (K == ROW_MAX) a8[i] = fmaxf(a8[i], f[i]);
                    else a8[i] = fminf(a8[i], f[i]);
                }
            }
            float acc = a8[0];
#pragma unroll
            for (int i = 1; i < 8; i++) {
                if (K == ROW_SUM) acc += a8[i];
                else if (K == ROW_MAX) acc = fmaxf(acc, a8[i]);
                else acc = fminf(acc, a8[i]);
            }
            if (K == ROW_SUM) acc = warp_sum(acc);
            else if (K == ROW_MAX) acc = warp_max(acc);
            else acc = warp_min(acc);
            if (lane == 0) {
                if (K == ROW_SUM) reinterpret_cast<float *>(d->out)[row] = acc;
                else reinterpret_cast<uint16_t *>(d->out)[row] = to_bf(acc);
            }
        } else {
            uint4 *y = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(d->out) + (uint64_t)row * H);
            float m = -INFINITY;
#pragma unroll 1
            for (uint32_t v = lane; v < nv; v += 32) {
                float f[8];
                unpack8(sx[v], f);
#pragma unroll
                for (int i = 0; i < 8; i++) m = fmaxf(m, f[i]);
            }
            m = warp_max(m);
            float s8[8];
#pragma unroll
            for (int i = 0; i < 8; i++) s8[i] = 0.0f;
#pragma unroll 1
            for (uint32_t v = lane; v < nv; v += 32) {
                float f[8];
                unpack8(sx[v], f);
#pragma unroll
                for (int i = 0; i < 8; i++) s8[i] += __expf(f[i] - m);
            }
            float sum = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; i++) sum += s8[i];
            const float inv = 1.0f / warp_sum(sum);
#pragma unroll 1
            for (uint32_t v = lane; v < nv; v += 32) {
                float f[8];
                unpack8(sx[v], f);
#pragma unroll
                for (int i = 0; i < 8; i++) f[i] = __expf(f[i] - m) * inv;
                __stcg(y + v, pack8(f));
            }
        }
        /* every lane is done with half hb before the next claim refills it */
        __syncwarp();
        if (nx >= R) {
            next = nx;
            break;
        }
        row = nx;
        hb ^= 1u;
    }
    if (lane == 0) {
        w->phase[0] = ph & 1u;
        w->phase[1] = (ph >> 1) & 1u;
        w->claim_count = count;
        w->claim_next = next;
        w->claim_done = ctr != nullptr ? 1u : 0u;
    }
    __syncwarp();
    return st;
}

template <int K>
DEV int row_tile(const gpuos_devdesc *d, uint32_t row)
{
    const uint32_t R = d->dims[0], H = d->dims[1];
    if (row >= R) return GPUOS_ST_OK;
    if (H == 0) return GPUOS_ST_BAD_ARGS;
    bool ok = (H & 7u) == 0 && (d->a & 15u) == 0;
    if (K == ROW_SOFTMAX || K == ROW_LN) ok = ok && (d->out & 15u) == 0;
    if (K == ROW_LN) ok = ok && ((d->b | d->aux0) & 15u) == 0;
    if (!ok) return row_generic<K>(d, row, H);
    /* staged: two rows at a time (with LayerNorm's gamma and beta, if they
     * fit beside them); else the row, plus
     * (LayerNorm) gamma and beta in chunks of C columns, a multiple of 8 of
     * at least 256 (or all H) */
    const uint32_t sb = stage_hdr()->stage_bytes;
    if ((K == ROW_LN ? 8u : 4u) * H <= sb) return row_pipe<K>(d, row, R, H);
    if (2u * H <= sb) {
        uint32_t C = 0;
        if (K == ROW_LN) {
            C = ((sb - 2u * H) / 4u) & ~7u;
            if (C > H) C = H;
        }
        if (K != ROW_LN || C == H || C >= 256u) return row_staged<K>(d, row, H, C);
    }
    return H <= GPUOS_ROW_REG_MAX ? row_reg<K>(d, row, H) : row_generic<K>(d, row, H);
}

/* ---- RoPE: one (request, group of GPUOS_HEAD_GROUP heads) per tile --------
 * Pairs (i, i + D/2) of every q and k row of the group rotate by the angle
 * pos * theta^(-2i/D). With D % 4 == 0 and 4-byte aligned rows, lane l owns
 * the pairs of elements 2w and 2w + 1 for words w = l, l + 32 of a half-row:
 * every load of the tile is issued before the first rotation. */
/* sin and cos of x: Cody-Waite reduction by 2 pi (2 pi split in three parts,
 * the first exact in 8 bits, so k * part is exact for |k| < 2^15) to
 * r in [-pi, pi], then the hardware sin/cos, whose absolute error there is
 * below 4e-7. */
DEV void sincos_cw(float x, float *sn, float *cs)
{
    const float k = rintf(x * 0.159154943f);
    float r = fmaf(-k, 6.28125f, x);
    r = fmaf(-k, 1.935307169e-3f, r);
    r = fmaf(-k, 1.025313168e-11f, r);
    __sincosf(r, sn, cs);
}

DEV int rope_tile(const gpuos_devdesc *d, uint32_t tile)
{
    const uint32_t B = d->dims[0], H = d->dims[1], D = d->dims[2];
    if (H == 0 || D == 0 || (D & 1u) || D > 256) return GPUOS_ST_BAD_ARGS;
    const uint32_t ng = (H + GPUOS_HEAD_GROUP - 1) / GPUOS_HEAD_GROUP;
    const uint32_t b = tile / ng, h0 = (tile - b * ng) * GPUOS_HEAD_GROUP;
    if (b >= B) return GPUOS_ST_OK;
    const uint32_t nh = (H - h0) < GPUOS_HEAD_GROUP ? (H - h0) : GPUOS_HEAD_GROUP;
    const int32_t pos = __ldcg(reinterpret_cast<const int32_t *>(d->aux0) + b) - 1;
    if (pos < 0) return GPUOS_ST_BAD_ARGS;
    const uint32_t lane = lane_id(), half = D / 2;
    /* theta^(-2i/D) = 2^(-(2i/D) log2 theta) */
    const float l2t = log2f(d->fparam[0]) * (-2.0f / (float)D);
    const uint64_t row0 = ((uint64_t)b * H + h0) * D; /* first element of the group */
    if ((D & 3u) == 0 && ((d->a | d->b) & 3u) == 0) {
        const uint32_t hw = half / 2; /* words per half-row, <= 64 */
        float c[2][2], sn[2][2];
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const uint32_t wd = lane + 32u * j;
#pragma unroll
            for (int e = 0; e < 2; e++) {
                c[j][e] = 1.0f;
                sn[j][e] = 0.0f;
                if (wd < hw) {
                    float inv;
                    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(l2t * (float)(2u * wd + e)));
                    sincos_cw((float)pos * inv, &sn[j][e], &c[j][e]);
                }
            }
        }
        uint32_t x0[2][GPUOS_HEAD_GROUP][2], x1[2][GPUOS_HEAD_GROUP][2];
#pragma unroll
        for (int which = 0; which < 2; which++) {
            const uint32_t *base = reinterpret_cast<const uint32_t *>(reinterpret_cast<const uint16_t *>(
                which ? d->b : d->a) + row0);
#pragma unroll
            for (int hh = 0; hh < GPUOS_HEAD_GROUP; hh++) {
#pragma unroll
                for (int j = 0; j < 2; j++) {
                    const uint32_t wd = lane + 32u * j;
                    if ((uint32_t)hh < nh && wd < hw) {
                        x0[which][hh][j] = __ldcg(base + (uint64_t)hh * (D / 2) + wd);
                        x1[which][hh][j] = __ldcg(base + (uint64_t)hh * (D / 2) + hw + wd);
                    }
                }
            }
        }
#pragma unroll
        for (int which = 0; which < 2; which++) {
            uint32_t *base = reinterpret_cast<uint32_t *>(reinterpret_cast<uint16_t *>(which ? d->b : d->a) + row0);
#pragma unroll
            for (int hh = 0; hh < GPUOS_HEAD_GROUP; hh++) {
#pragma unroll
                for (int j = 0; j < 2; j++) {
                    const uint32_t wd = lane + 32u * j;
                    if ((uint32_t)hh < nh && wd < hw) {
                        const uint32_t u0 = x0[which][hh][j], u1 = x1[which][hh][j];
                        const float a0 = bf_lo(u0), a1 = bf_hi(u0), b0 = bf_lo(u1), b1 = bf_hi(u1);
                        base[(uint64_t)hh * (D / 2) + wd] =
                            pack_bf2(a0 * c[j][0] - b0 * sn[j][0], a1 * c[j][1] - b1 * sn[j][1]);
                        base[(uint64_t)hh * (D / 2) + hw + wd] =
                            pack_bf2(b0 * c[j][0] + a0 * sn[j][0], b1 * c[j][1] + a1 * sn[j][1]);
                    }
                }
            }
        }
        return GPUOS_ST_OK;
    }
    /* any even D or 2-byte alignment: one element pair per lane and step */
    for (int which = 0; which < 2; which++) {
        uint16_t *base = reinterpret_cast<uint16_t *>(which ? d->b : d->a) + row0;
        for (uint32_t k = lane; k < nh * half; k += 32) {
            const uint32_t hh = k / half, i = k - hh * half;
            float sv, cv, inv;
            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(l2t * (float)i));
            sincos_cw((float)pos * inv, &sv, &cv);
            uint16_t *row = base + (uint64_t)hh * D;
            const float a0 = bf1(__ldcg(row + i)), b0 = bf1(__ldcg(row + i + half));
            row[i] = to_bf(a0 * cv - b0 * sv);
            row[i + half] = to_bf(b0 * cv + a0 * sv);
        }
    }
    return GPUOS_ST_OK;
}

/* ---- KV-cache slot write: one (request, group of GPUOS_HEAD_GROUP heads) per
 * tile, k and v rows of the group copied bit for bit into row lens[b] - 1 of
 * each head's cache; up to 8 16-byte loads per lane in flight per round ---- */
DEV int kv_tile(const gpuos_devdesc *d, uint32_t tile)
{
    const uint32_t B = d->dims[0], H = d->dims[1], D = d->dims[2], Lcap = d->dims[3];
    if (H == 0) return GPUOS_ST_BAD_ARGS;
    const uint32_t ng = (H + GPUOS_HEAD_GROUP - 1) / GPUOS_HEAD_GROUP;
    const uint32_t b = tile / ng, h0 = (tile - b * ng) * GPUOS_HEAD_GROUP;
    if (b >= B) return GPUOS_ST_OK;
    const uint32_t nh = (H - h0) < GPUOS_HEAD_GROUP ? (H - h0) : GPUOS_HEAD_GROUP;
    const int32_t pos = __ldcg(reinterpret_cast<const int32_t *>(d->aux0) + b) - 1;
    if (pos < 0 || (uint32_t)pos >= Lcap) return GPUOS_ST_BAD_ARGS;
    const uint32_t lane = lane_id();
    const uint64_t bh0 = (uint64_t)b * H + h0;
    const uint16_t *src[2] = {reinterpret_cast<const uint16_t *>(d->a) + bh0 * D,
                              reinterpret_cast<const uint16_t *>(d->b) + bh0 * D};
    uint16_t *dst[2] = {reinterpret_cast<uint16_t *>(d->out) + (bh0 * Lcap + (uint64_t)pos) * D,
                        reinterpret_cast<uint16_t *>(d->aux1) + (bh0 * Lcap + (uint64_t)pos) * D};
    const uint64_t hstride = (uint64_t)Lcap * D; /* elements between heads in the cache */
    if ((D & 7u) == 0 && ((d->a | d->b | d->out | d->aux1) & 15u) == 0) {
        const uint32_t nvr = D / 8, per = nh * nvr, total = 2u * per;
        constexpr int U = 8;
        for (uint32_t i0 = 0; i0 < total; i0 += 32u * U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const uint32_t i = i0 + 32u * u + lane;
                if (i < total) {
                    const uint32_t which = i >= per, r = i - which * per, h = r / nvr, e = r - h * nvr;
                    v[u] = __ldcg(reinterpret_cast<const uint4 *>(src[which] + (uint64_t)h * D) + e);
                }
            }
#pragma unroll
            for (int u = 0; u < U; u++) {
                const uint32_t i = i0 + 32u * u + lane;
                if (i < total) {
                    const uint32_t which = i >= per, r = i - which * per, h = r / nvr, e = r - h * nvr;
                    __stcg(reinterpret_cast<uint4 *>(dst[which] + h * hstride) + e, v[u]);
                }
            }
        }
        return GPUOS_ST_OK;
    }
    for (int which = 0; which < 2; which++) {
        for (uint32_t i = lane; i < nh * D; i += 32) {
            const uint32_t h = i / D, e = i - h * D;
            dst[which][h * hstride + e] = src[which][(uint64_t)h * D + e];
        }
    }
    return GPUOS_ST_OK;
}

/* ---- decode SDPA: one (request, head, chunk of key rows) per tile ---------
 * The host picks the number of chunks per head (at most 1,536 tiles in all,
 * chunks of at least 32 rows); the tile recovers the chunk length from Lmax
 * and ntiles, and shortens it when the requests' lengths would leave tiles
 * idle (see sdpa_tile). Four 8-lane groups walk interleaved key rows; in a
 * group lane li owns dims [8 li, 8 li + 8) and [64 + 8 li, 64 + 8 li + 8) of
 * q, K and V (two 16-byte pieces 128 bytes apart, so a quarter-warp reads 128
 * contiguous bytes of a row: no shared-memory bank conflicts). Scores use
 * exp2 with log2(e) folded into the query scale; each group keeps an
 * online-softmax state (m, l, acc), the four states merge by shuffles, and
 * multi-chunk heads merge through the workspace in the last chunk to finish.
 * With shared-memory staging the K and V rows arrive by TMA bulk copies into
 * the two halves of the warp's buffer in turn (stage_bytes / 1024 rows of
 * each per half), so the next rows load while the current ones are scored. */
#define GPUOS_SDPA_PART 132 /* floats per partial: m, l, 2 pad, acc[128] (16-byte multiple) */
DEV void sdpa_merge(float &m, float &l, float *acc, float mo, float lo, const float *acco)
{
    const float mn = fmaxf(m, mo);
    const float mu = (mn == -INFINITY) ? 0.0f : mn;
    const float a = exp2f(m - mu), b = exp2f(mo - mu);
    l = l * a + lo * b;
#pragma unroll
    for (int i = 0; i < 16; i++) acc[i] = acc[i] * a + acco[i] * b;
    m = mn;
}

/* One online-softmax step over UK keys held as (k0,k1,v0,v1) pieces. */
template <int UK>
DEV void sdpa_step(const float *q, const uint4 (&kv)[UK][2], const uint4 (&vv)[UK][2], const bool *valid, float &m,
                   float &l, float *acc)
{
    float sc[UK];
#pragma unroll
    for (int u = 0; u < UK; u++) {
        float kf[16];
        unpack8(kv[u][0], kf);
        unpack8(kv[u][1], kf + 8);
        float p = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; i++) p = fmaf(q[i], kf[i], p);
        p += __shfl_xor_sync(0xFFFFFFFFu, p, 1);
        p += __shfl_xor_sync(0xFFFFFFFFu, p, 2);
        p += __shfl_xor_sync(0xFFFFFFFFu, p, 4);
        sc[u] = valid[u] ? p : -INFINITY;
    }
    float mn = m;
#pragma unroll
    for (int u = 0; u < UK; u++) mn = fmaxf(mn, sc[u]);
    const float mu = (mn == -INFINITY) ? 0.0f : mn;
    const float corr = exp2f(m - mu);
    l *= corr;
#pragma unroll
    for (int i = 0; i < 16; i++) acc[i] *= corr;
#pragma unroll
    for (int u = 0; u < UK; u++) {
        const float p = exp2f(sc[u] - mu);
        l += p;
        float vf[16];
        unpack8(vv[u][0], vf);
        unpack8(vv[u][1], vf + 8);
#pragma unroll
        for (int i = 0; i < 16; i++) acc[i] = fmaf(p, vf[i], acc[i]);
    }
    m = mn;
}

/* Lane 0: bulk-copy key rows [tb, tb + nk) of K and V into half hb. */
DEV void sdpa_issue(WarpStage *w, unsigned char *buf, uint32_t SUB, uint32_t hb, const uint16_t *Kb,
                    const uint16_t *Vb, uint32_t tb, uint32_t nk)
{
    unsigned char *sK = buf + hb * SUB * 512u;
    unsigned char *sV = sK + SUB * 256u;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_expect(&w->mbar[hb], 2u * nk * 256u);
    bulk_g2s(sK, Kb + (uint64_t)tb * 128, nk * 256u, &w->mbar[hb]);
    bulk_g2s(sV, Vb + (uint64_t)tb * 128, nk * 256u, &w->mbar[hb]);
}

DEV int sdpa_tile(const gpuos_devdesc *d, uint32_t tile)
{
    const uint32_t B = d->dims[0], H = d->dims[1], D = d->dims[2], Lcap = d->dims[3], Lmax = d->dims[4];
    const uint32_t BH = B * H;
    if (D != 128 || BH == 0 || Lmax == 0 || Lmax > Lcap || d->dims[5] < BH) return GPUOS_ST_BAD_ARGS;
    const uint32_t nch = d->ntiles / BH;
    if (nch == 0) return GPUOS_ST_BAD_ARGS;
    if (tile >= BH * nch) return GPUOS_ST_OK;
    const uint32_t lane = lane_id(), g = lane >> 3, li = lane & 7u;
    const int32_t *lens = reinterpret_cast<const int32_t *>(d->aux0);
    /* Chunks. The host's rule cuts every (request, head) pair's keys into
     * at most nch chunks of CH = round_up(ceil(Lmax / nch), 32) rows; a
     * request shorter than Lmax then leaves some of its nch tiles idle, and
     * the op takes as long as one CH-row chunk whatever the other requests'
     * lengths. With the lengths known here the chunk shrinks to what lets
     * the requests' chunks fill the op's tiles:
     *   CH' = round_up(ceil(H sum_b L_b / (ntiles - B H)), 32), at least 32,
     * which gives at most H sum_b ceil(L_b / CH') <= H sum_b L_b / CH' + B H
     * <= ntiles chunks. Chunks are numbered request by request (b, then h,
     * then c), so a tile finds its request by a prefix sum over the
     * requests' chunk counts H ceil(L_b / CH); its partial (split-K) is
     * slot `tile` of the workspace, below ntiles like before. */
    uint32_t CH = ((Lmax + nch - 1) / nch + 31u) & ~31u; /* key rows per chunk */
    uint32_t b, h, c, nchb, L;
    uint64_t pfirst; /* workspace slot of the (b, h) pair's first chunk */
    uint4 q0, q1;
    if (nch == 1 || B == 1) {
        /* one chunk per pair, or one request (whose length is Lmax): the
         * host's chunks; the length and the query in one round trip */
        b = tile / (H * nch);
        const uint32_t rem = tile - b * H * nch;
        h = rem / nch;
        c = rem - h * nch;
        const int32_t Lb = __ldcg(lens + b);
        const uint16_t *qp = reinterpret_cast<const uint16_t *>(d->a) + ((uint64_t)b * H + h) * 128;
        q0 = __ldcg(reinterpret_cast<const uint4 *>(qp + 8 * li));
        q1 = __ldcg(reinterpret_cast<const uint4 *>(qp + 64 + 8 * li));
        if (Lb < 1 || (uint32_t)Lb > Lmax) return GPUOS_ST_BAD_ARGS;
        L = (uint32_t)Lb;
        nchb = (L + CH - 1u) / CH;
        if (c >= nchb) return GPUOS_ST_OK;
        pfirst = (uint64_t)tile - c;
    } else {
        /* every length, checked and summed (one round trip for B <= 32) */
        const int32_t l0 = lane < B ? __ldcg(lens + lane) : 1;
        bool bad = l0 < 1 || (uint32_t)l0 > Lmax;
        unsigned long long sum = lane < B ? (unsigned long long)l0 : 0ull;
        for (uint32_t i = lane + 32u; i < B; i += 32) {
            const int32_t v = __ldcg(lens + i);
            bad |= v < 1 || (uint32_t)v > Lmax;
            sum += (unsigned long long)(v > 0 ? v : 0);
        }
        if (__any_sync(0xFFFFFFFFu, bad)) return GPUOS_ST_BAD_ARGS;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        const unsigned long long spare = (unsigned long long)BH * (nch - 1u);
        unsigned long long cn = ((unsigned long long)H * sum + spare - 1ull) / spare;
        cn = (cn + 31ull) & ~31ull;
        if (cn < GPUOS_SDPA_CHUNK_MIN) cn = GPUOS_SDPA_CHUNK_MIN;
        if (cn < CH) CH = (uint32_t)cn;
        /* the tile's request: prefix sums of H ceil(L_i / CH), 32 requests at a time */
        uint32_t base = 0, off = 0, found = 0;
        L = 0;
        b = 0;
        for (uint32_t i0 = 0; i0 < B; i0 += 32) {
            const uint32_t i = i0 + lane;
            const uint32_t Li = i >= B ? 0u : (i0 == 0 ? (uint32_t)l0 : (uint32_t)__ldcg(lens + i));
            const uint32_t cnt = H * ((Li + CH - 1u) / CH);
            uint32_t incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= (uint32_t)o) incl += v;
            }
            const uint32_t lo = base + incl - cnt;
            const uint32_t bal = __ballot_sync(0xFFFFFFFFu, cnt && tile >= lo && tile < lo + cnt);
            if (bal) {
                const int src = __ffs(bal) - 1;
                b = i0 + (uint32_t)src;
                L = __shfl_sync(0xFFFFFFFFu, Li, src);
                off = tile - __shfl_sync(0xFFFFFFFFu, lo, src);
                found = 1;
                break;
            }
            base += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (!found) return GPUOS_ST_OK; /* past the last chunk */
        nchb = (L + CH - 1u) / CH;
        h = off / nchb;
        c = off - h * nchb;
        pfirst = (uint64_t)tile - c;
        const uint16_t *qp = reinterpret_cast<const uint16_t *>(d->a) + ((uint64_t)b * H + h) * 128;
        q0 = __ldcg(reinterpret_cast<const uint4 *>(qp + 8 * li));
        q1 = __ldcg(reinterpret_cast<const uint4 *>(qp + 64 + 8 * li));
    }
    const uint64_t bh = (uint64_t)b * H + h;
    const uint32_t t0 = c * CH;
    const uint32_t t1 = min(L, t0 + CH);
    const uint16_t *Kb = reinterpret_cast<const uint16_t *>(d->b) + bh * Lcap * 128;
    const uint16_t *Vb = reinterpret_cast<const uint16_t *>(d->aux1) + bh * Lcap * 128;
    const uint32_t SUB = stage_hdr()->stage_bytes / 1024u; /* key rows per half: K and V, 256 bytes each */
    const uint32_t nsub = SUB >= 8 ? (t1 - t0 + SUB - 1) / SUB : 0;
    WarpStage *w = warp_stage();
    unsigned char *buf = warp_stage_buf();
    if (SUB >= 8 && lane == 0) {
        sdpa_issue(w, buf, SUB, 0, Kb, Vb, t0, min(SUB, t1 - t0));
        if (nsub > 1) sdpa_issue(w, buf, SUB, 1, Kb, Vb, t0 + SUB, min(SUB, t1 - t0 - SUB));
    }
    const float qs = d->fparam[0] * 1.4426950408889634f;
    float q[16];
    unpack8(q0, q);
    unpack8(q1, q + 8);
#pragma unroll
    for (int i = 0; i < 16; i++) q[i] *= qs;
    float m = -INFINITY, l = 0.0f, acc[16];
#pragma unroll
    for (int i = 0; i < 16; i++) acc[i] = 0.0f;
    constexpr int UK = 2; /* keys per group per step */
    int32_t status = GPUOS_ST_OK;
    if (SUB >= 8) {
        uint32_t phs = w->phase[0] | (w->phase[1] << 1); /* bit hb: parity to wait for on half hb */
        for (uint32_t sI = 0; sI < nsub; sI++) {
            const uint32_t hb = sI & 1u;
            const uint32_t tb = t0 + sI * SUB;
            const uint32_t nk = min(SUB, t1 - tb);
            if (!mbar_wait(&w->mbar[hb], (phs >> hb) & 1u)) {
                /* leave no copy writing the buffer: wait once more (bounded)
                 * on this half and on the other one if it has a copy out */
                mbar_wait(&w->mbar[hb], (phs >> hb) & 1u);
                phs ^= 1u << hb;
                if (sI + 1 < nsub) {
                    mbar_wait(&w->mbar[hb ^ 1u], (phs >> (hb ^ 1u)) & 1u);
                    phs ^= 1u << (hb ^ 1u);
                }
                status = GPUOS_ST_COPY_TIMEOUT;
                break;
            }
            phs ^= 1u << hb;
            const unsigned char *sK = buf + hb * SUB * 512u;
            const unsigned char *sV = sK + SUB * 256u;
            for (uint32_t kk = 0; kk < nk; kk += 4 * UK) {
                uint4 kv[UK][2], vv[UK][2];
                bool valid[UK];
#pragma unroll
                for (int u = 0; u < UK; u++) {
                    const uint32_t t = kk + g + 4 * u;
                    valid[u] = t < nk;
                    const uint32_t tt = valid[u] ? t : 0u;
                    const uint4 *kr = reinterpret_cast<const uint4 *>(sK + tt * 256u) + li;
                    const uint4 *vr = reinterpret_cast<const uint4 *>(sV + tt * 256u) + li;
                    kv[u][0] = kr[0];
                    kv[u][1] = kr[8];
                    vv[u][0] = vr[0];
                    vv[u][1] = vr[8];
                }
                sdpa_step<UK>(q, kv, vv, valid, m, l, acc);
            }
            __syncwarp(); /* every lane is done with half hb before it is refilled */
            if (lane == 0 && sI + 2 < nsub) sdpa_issue(w, buf, SUB, hb, Kb, Vb, tb + 2 * SUB, min(SUB, t1 - tb - 2 * SUB));
        }
        if (lane == 0) {
            w->phase[0] = phs & 1u;
            w->phase[1] = (phs >> 1) & 1u;
        }
        __syncwarp();
    } else {
        for (uint32_t tb = t0; tb < t1; tb += 4 * UK) {
            uint4 kv[UK][2], vv[UK][2];
            bool valid[UK];
#pragma unroll
            for (int u = 0; u < UK; u++) {
                const uint32_t t = tb + g + 4 * u;
                valid[u] = t < t1;
                if (valid[u]) {
                    const uint4 *kr = reinterpret_cast<const uint4 *>(Kb + (uint64_t)t * 128) + li;
                    const uint4 *vr = reinterpret_cast<const uint4 *>(Vb + (uint64_t)t * 128) + li;
                    kv[u][0] = __ldcg(kr);
                    kv[u][1] = __ldcg(kr + 8);
                    vv[u][0] = __ldcg(vr);
                    vv[u][1] = __ldcg(vr + 8);
                } else {
                    kv[u][0] = kv[u][1] = vv[u][0] = vv[u][1] = make_uint4(0, 0, 0, 0);
                }
            }
            sdpa_step<UK>(q, kv, vv, valid, m, l, acc);
        }
    }
    if (status != GPUOS_ST_OK) return status;
    /* merge the four groups (lanes li, li+8, li+16, li+24) */
#pragma unroll
    for (int o = 8; o <= 16; o <<= 1) {
        float acco[16];
        const float mo = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        const float lo = __shfl_xor_sync(0xFFFFFFFFu, l, o);
#pragma unroll
        for (int i = 0; i < 16; i++) acco[i] = __shfl_xor_sync(0xFFFFFFFFu, acc[i], o);
        sdpa_merge(m, l, acc, mo, lo, acco);
    }
    uint16_t *o16 = reinterpret_cast<uint16_t *>(d->out) + bh * 128;
    if (nchb == 1) {
        if (g == 0) {
            const float inv = 1.0f / l;
            float r[16];
#pragma unroll
            for (int i = 0; i < 16; i++) r[i] = acc[i] * inv;
            reinterpret_cast<uint4 *>(o16 + 8 * li)[0] = pack8(r);
            reinterpret_cast<uint4 *>(o16 + 64 + 8 * li)[0] = pack8(r + 8);
        }
        return GPUOS_ST_OK;
    }
    /* split-K: publish this chunk's (m, l, acc[128]) and let the last chunk
     * merge. Workspace: round_up(Ccap, 4) uint32 counters, then partials of
     * GPUOS_SDPA_PART floats {m, l, -, -, acc[128]} */
    uint32_t *cnt = reinterpret_cast<uint32_t *>(d->aux2);
    float *ws = reinterpret_cast<float *>(d->aux2) + ((d->dims[5] + 3u) & ~3u);
    float *part = ws + (uint64_t)tile * GPUOS_SDPA_PART;
    if (g == 0) {
        float4 *pa = reinterpret_cast<float4 *>(part + 4);
        __stcg(pa + 2 * li, make_float4(acc[0], acc[1], acc[2], acc[3]));
        __stcg(pa + 2 * li + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
        __stcg(pa + 16 + 2 * li, make_float4(acc[8], acc[9], acc[10], acc[11]));
        __stcg(pa + 16 + 2 * li + 1, make_float4(acc[12], acc[13], acc[14], acc[15]));
        if (li == 0) {
            __stcg(part, m);
            __stcg(part + 1, l);
        }
    }
    __syncwarp();
    /* one acq_rel add: releases this chunk's partial (the warp barrier above
     * orders the other lanes' stores before lane 0's), and the last chunk
     * acquires every other chunk's */
    uint32_t last = 0;
    if (lane == 0) last = (atom_add_acq_rel_gpu32(cnt + bh, 1u) == nchb - 1) ? 1u : 0u;
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (!last) return GPUOS_ST_OK;
    /* the merge, in batches of 16 chunks whose (m, l, acc slice) loads are
     * all in flight together; a running maximum rescales earlier batches */
    float M = -INFINITY, den = 0.0f;
    float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
    for (uint32_t k0 = 0; k0 < nchb; k0 += 16) {
        float mk[16], lk[16];
        float4 vk[16];
#pragma unroll
        for (int k = 0; k < 16; k++) {
            const uint32_t kc = min(k0 + (uint32_t)k, nchb - 1); /* duplicates past the end weigh 0 below */
            const float *pk = ws + (pfirst + kc) * GPUOS_SDPA_PART;
            mk[k] = __ldcg(pk);
            lk[k] = __ldcg(pk + 1);
            vk[k] = __ldcg(reinterpret_cast<const float4 *>(pk + 4) + lane);
        }
        float mb = M;
#pragma unroll
        for (int k = 0; k < 16; k++)
            if (k0 + k < nchb) mb = fmaxf(mb, mk[k]);
        const float sc = exp2f(M - mb); /* 0 on the first batch (M = -inf) */
        den *= sc;
        o4.x *= sc;
        o4.y *= sc;
        o4.z *= sc;
        o4.w *= sc;
#pragma unroll
        for (int k = 0; k < 16; k++) {
            const float wk = (k0 + k < nchb) ? exp2f(mk[k] - mb) : 0.0f;
            den = fmaf(lk[k], wk, den);
            o4.x = fmaf(vk[k].x, wk, o4.x);
            o4.y = fmaf(vk[k].y, wk, o4.y);
            o4.z = fmaf(vk[k].z, wk, o4.z);
            o4.w = fmaf(vk[k].w, wk, o4.w);
        }
        M = mb;
    }
    const float inv = 1.0f / den;
    uint2 st;
    st.x = pack_bf2(o4.x * inv, o4.y * inv);
    st.y = pack_bf2(o4.z * inv, o4.w * inv);
    reinterpret_cast<uint2 *>(o16)[lane] = st;
    if (lane == 0) atomicExch(cnt + bh, 0u); /* leave the workspace zeroed */
    return GPUOS_ST_OK;
}

/* ---- vector-matrix product: GPUOS_VM_COLS (8) output columns per tile ----
 * y[n] = sum_k x[k] W[k][n], W row-major [K][N]. A tile owns 8 columns, one
 * 16-byte piece of every row of W (the neighbouring tile reads the other
 * half of each 32-byte sector at about the same time). Lane l sums rows
 * k = l, l + 32, ...; the 32 partial sums then reduce by shuffles. With
 * staging, blocks of R rows (their W pieces and x values) arrive by 16-byte
 * cp.async copies into the two halves of the warp's buffer in turn, so the
 * next block loads while the current one is summed and no registers are
 * held by loads in flight. */
DEV void cp_async16(void *sdst, const void *gsrc)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(sdst)), "l"(gsrc) : "memory");
}
DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
DEV void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
DEV void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

/* Every lane: copy rows [k0, k0 + nk) into a half: W pieces first (16 bytes
 * per row), then the rows' x values (nk is a multiple of 8 here). */
DEV void vm_issue(unsigned char *half, const uint16_t *x, const uint16_t *W, uint32_t N, uint32_t c0, uint32_t R,
                  uint32_t k0, uint32_t nk, uint32_t lane)
{
    for (uint32_t r = lane; r < nk; r += 32) cp_async16(half + r * 16u, W + (uint64_t)(k0 + r) * N + c0);
    for (uint32_t i = lane; i < nk / 8u; i += 32) cp_async16(half + R * 16u + i * 16u, x + k0 + 8u * i);
}

DEV int vecmat_tile(const gpuos_devdesc *d, uint32_t tile)
{
    const uint32_t K = d->dims[0], N = d->dims[1];
    const uint32_t c0 = tile * GPUOS_VM_COLS;
    if (c0 >= N) return GPUOS_ST_OK;
    const uint32_t lane = lane_id();
    const uint16_t *x = reinterpret_cast<const uint16_t *>(d->a);
    const uint16_t *W = reinterpret_cast<const uint16_t *>(d->b);
    uint16_t *y = reinterpret_cast<uint16_t *>(d->out);
    if ((N & 7u) == 0 && ((d->b | d->out) & 15u) == 0) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; i++) acc[i] = 0.0f;
        const uint32_t sbytes = stage_hdr()->stage_bytes;
        /* rows per half: W pieces (16 B) and x values (2 B), a multiple of 32 */
        const uint32_t R = (sbytes / 2u / 18u) & ~31u;
        /* x is copied in 16-byte pieces of 8 values: it must be 16-byte
         * aligned, and with K % 8 == 0 (R being a multiple of 32) every
         * block holds a whole number of pieces, so no copy reads past x[K-1] */
        if (R >= 32 && (d->a & 15u) == 0 && (K & 7u) == 0) {
            unsigned char *buf = warp_stage_buf();
            const uint32_t nblk = (K + R - 1) / R;
            const uint32_t hbytes = sbytes / 2u;
            vm_issue(buf, x, W, N, c0, R, 0, min(R, K), lane);
            cp_async_commit();
            if (nblk > 1) vm_issue(buf + hbytes, x, W, N, c0, R, R, min(R, K - R), lane);
            cp_async_commit();
            for (uint32_t s = 0; s < nblk; s++) {
                cp_async_wait1(); /* this lane's copies of block s have landed */
                __syncwarp();     /* ... and every other lane's */
                const unsigned char *hf = buf + (s & 1u) * hbytes;
                const uint32_t nk = min(R, K - s * R);
                const uint16_t *xs = reinterpret_cast<const uint16_t *>(hf + R * 16u);
#pragma unroll 7
                for (uint32_t r = lane; r < nk; r += 32) {
                    float wf[8];
                    unpack8(*reinterpret_cast<const uint4 *>(hf + r * 16u), wf);
                    const float xv = bf1(xs[r]);
#pragma unroll
                    for (int i = 0; i < 8; i++) acc[i] = fmaf(xv, wf[i], acc[i]);
                }
                __syncwarp(); /* every lane is done with this half before it is refilled */
                if (s + 2 < nblk) vm_issue(buf + (s & 1u) * hbytes, x, W, N, c0, R, (s + 2) * R,
                                           min(R, K - (s + 2) * R), lane);
                cp_async_commit();
            }
            cp_async_wait0();
            __syncwarp();
        } else {
            constexpr int UR = 8;
            for (uint32_t k0 = 0; k0 < K; k0 += 32 * UR) {
                uint4 w[UR];
                float xv[UR];
#pragma unroll
                for (int u = 0; u < UR; u++) {
                    const uint32_t k = k0 + lane + 32 * u;
                    if (k < K) {
                        w[u] = __ldcg(reinterpret_cast<const uint4 *>(W + (uint64_t)k * N + c0));
                        xv[u] = bf1(__ldcg(x + k));
                    } else {
                        w[u] = make_uint4(0, 0, 0, 0);
                        xv[u] = 0.0f;
                    }
                }
#pragma unroll
                for (int u = 0; u < UR; u++) {
                    float wf[8];
                    unpack8(w[u], wf);
#pragma unroll
                    for (int i = 0; i < 8; i++) acc[i] = fmaf(xv[u], wf[i], acc[i]);
                }
            }
        }
#pragma unroll
        for (int o = 1; o <= 16; o <<= 1) {
#pragma unroll
            for (int i = 0; i < 8; i++) acc[i] += __shfl_xor_sync(0xFFFFFFFFu, acc[i], o);
        }
        if (lane == 0) __stcg(reinterpret_cast<uint4 *>(y + c0), pack8(acc));
        return GPUOS_ST_OK;
    }
    /* any N or alignment: lane (g, j) sums column c0 + j over rows g, g + 4, ... */
    const uint32_t j = lane & 7u, g = lane >> 3, col = c0 + j;
    float acc = 0.0f;
    if (col < N)
        for (uint32_t k = g; k < K; k += 4) acc = fmaf(bf1(__ldcg(x + k)), bf1(__ldcg(W + (uint64_t)k * N + col)), acc);
    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 8);
    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 16);
    if (g == 0 && col < N) y[col] = to_bf(acc);
    return GPUOS_ST_OK;
}

/* ---- table entries ----------------------------------------------------------- */
__device__ __noinline__ int op_nop(const gpuos_devdesc *, uint32_t) { return GPUOS_ST_OK; }
__device__ __noinline__ int op_add(const gpuos_devdesc *d, uint32_t t) { return ew_dispatch<EW_ADD>(d, t); }
__device__ __noinline__ int op_mul(const gpuos_devdesc *d, uint32_t t) { return ew_dispatch<EW_MUL>(d, t); }
__device__ __noinline__ int op_relu(const gpuos_devdesc *d, uint32_t t) { return ew_dispatch<EW_RELU>(d, t); }
__device__ __noinline__ int op_gelu(const gpuos_devdesc *d, uint32_t t) { return ew_dispatch<EW_GELU>(d, t); }
__device__ __noinline__ int op_softmax(const gpuos_devdesc *d, uint32_t t) { return row_tile<ROW_SOFTMAX>(d, t); }
__device__ __noinline__ int op_layernorm(const gpuos_devdesc *d, uint32_t t) { return row_tile<ROW_LN>(d, t); }
__device__ __noinline__ int op_rowsum(const gpuos_devdesc *d, uint32_t t) { return row_tile<ROW_SUM>(d, t); }
__device__ __noinline__ int op_rowmax(const gpuos_devdesc *d, uint32_t t) { return row_tile<ROW_MAX>(d, t); }
__device__ __noinline__ int op_rowmin(const gpuos_devdesc *d, uint32_t t) { return row_tile<ROW_MIN>(d, t); }
__device__ __noinline__ int op_rope(const gpuos_devdesc *d, uint32_t t) { return rope_tile(d, t); }
__device__ __noinline__ int op_kv_write(const gpuos_devdesc *d, uint32_t t) { return kv_tile(d, t); }
__device__ __noinline__ int op_sdpa(const gpuos_devdesc *d, uint32_t t) { return sdpa_tile(d, t); }
__device__ __noinline__ int op_vecmat(const gpuos_devdesc *d, uint32_t t) { return vecmat_tile(d, t); }

__device__ gpuos_op_fn g_builtin_ops[GPUOS_OP_BUILTIN_COUNT] = {
    op_nop, op_add, op_mul, op_relu, op_gelu, op_softmax, op_layernorm,
    op_rowsum, op_rowmax, op_rowmin, op_rope, op_kv_write, op_sdpa, op_vecmat,
};

/* The body of built-in op `kind`, inlined (the eager kernel). */
DEV int builtin_call(uint32_t kind, const gpuos_devdesc *d, uint32_t t)
{
    switch (kind) {
    case GPUOS_OP_NOP: return GPUOS_ST_OK;
    case GPUOS_OP_ADD: return ew_dispatch<EW_ADD>(d, t);
    case GPUOS_OP_MUL: return ew_dispatch<EW_MUL>(d, t);
    case GPUOS_OP_RELU: return ew_dispatch<EW_RELU>(d, t);
    case GPUOS_OP_GELU: return ew_dispatch<EW_GELU>(d, t);
    case GPUOS_OP_SOFTMAX: return row_tile<ROW_SOFTMAX>(d, t);
    case GPUOS_OP_LAYERNORM: return row_tile<ROW_LN>(d, t);
    case GPUOS_OP_ROWSUM: return row_tile<ROW_SUM>(d, t);
    case GPUOS_OP_ROWMAX: return row_tile<ROW_MAX>(d, t);
    case GPUOS_OP_ROWMIN: return row_tile<ROW_MIN>(d, t);
    case GPUOS_OP_ROPE: return rope_tile(d, t);
    case GPUOS_OP_KV_WRITE: return kv_tile(d, t);
    case GPUOS_OP_SDPA: return sdpa_tile(d, t);
    case GPUOS_OP_VECMAT: return vecmat_tile(d, t);
    default: return GPUOS_ST_BAD_OP;
    }
}

/* ===========================================================================
 * Persistent executor
 * ======================================================================== */

/* Work-queue entry word: [63:28] stamp = (index + 1) mod 2^36, [27:12] ring
 * slot, [11:0] helper index (the helper's first tile). One 64-bit word, so
 * the claimer learns everything with the acquire load that finds it
 * published. The queue holds more than GPUOS_HELPERS x ring_entries entries,
 * so the entry a publication overwrites belongs to a ticket at least
 * ring_entries older, which has completed; completion implies every helper
 * entry of it was read. No producer-side check is needed. */
DEV uint64_t tq_word(uint64_t idx, uint32_t slot, uint32_t helper)
{
    return (((idx + 1) & GPUOS_TQ_STAMP_MASK) << 28) | ((uint64_t)(slot & 0xFFFFu) << 12) | (helper & 0xFFFu);
}
DEV bool tq_is(uint64_t w, uint64_t idx) { return (w >> 28) == ((idx + 1) & GPUOS_TQ_STAMP_MASK); }

DEV void fence_acq_rel_sys() { asm volatile("fence.acq_rel.sys;" ::: "memory"); }

/* Complete one descriptor (single thread). The device-memory done stamp
 * that dependent tiles wait on is released first; the host-visible record
 * (stores across NVLink-C2C, whose acknowledgements a release would have to
 * wait for) is written after it. */
DEV void complete_desc(const gpuos_exec_params &p, uint64_t ticket, uint32_t slot, int32_t status, uint32_t version)
{
    gpuos_rec_dev *r = p.rec + slot;
    const uint64_t t_done = globaltimer();
    /* release the stamp first (the tiles' outputs: a sole tile's through the
     * warp barrier before this call, other tiles' through their acq_rel
     * counter adds, which this thread acquired); the slot's counters are
     * reset after it: only a ticket ring_entries later reuses them, and the
     * host frees the slot only after the record's release below */
    st_release_gpu(p.done_dev + slot, ticket + 1);
    st_relaxed_gpu32(p.err + slot, 0u);
    st_relaxed_gpu(p.tiles_done + slot, 0ull);
    st_relaxed_gpu32(p.tile_ctr + slot, 0u);
    const uint64_t t_pub = *reinterpret_cast<volatile uint64_t *>(p.t_pub + slot);
    const uint64_t t_start = *reinterpret_cast<volatile uint64_t *>(p.t_start + slot);
    const uint64_t t_disp = *reinterpret_cast<volatile uint64_t *>(p.t_disp + slot);
    st_relaxed_sys32(reinterpret_cast<uint32_t *>(&r->status), (uint32_t)status);
    st_relaxed_sys32(&r->version, version);
    st_relaxed_sys(&r->t_dispatch, t_disp);
    st_relaxed_sys(&r->t_publish, t_pub);
    st_relaxed_sys(&r->t_start, t_start);
    st_relaxed_sys(&r->t_done, t_done);
    /* release: the record's fields before the slot's completion word (which
     * also frees the ring slot for the host); the words of eight slots
     * share a line, so the host's check of a run of slots reads few lines */
    st_release_sys(p.done_host + slot, (ticket + 1) | (status != GPUOS_ST_OK ? GPUOS_DONE_FAILED : 0ull));
    atomicAdd(&p.dctl->completed, 1ull);
}

DEV void set_exit(const gpuos_exec_params &p, uint32_t reason)
{
    st_relaxed_gpu32(&p.dctl->exit_flag, reason);
    st_relaxed_sys32(&p.hctl->exit_reason, reason);
    st_relaxed_sys32(&p.hctl->state, 2u);
}

/* Helper warps per descriptor: one per tile, except row ops, whose tiles
 * (one row) are small: one helper per four rows; at most GPUOS_HELPERS and
 * at most the executor's worker warps (more would only queue). */
DEV uint32_t helper_count(uint32_t op_id, uint32_t ntiles, uint32_t workers)
{
    uint32_t hlp = ntiles;
    if (op_id >= GPUOS_OP_SOFTMAX && op_id <= GPUOS_OP_ROWMIN) hlp = (ntiles + 3u) / 4u;
    const uint32_t cap = workers < GPUOS_HELPERS ? (workers ? workers : 1u) : GPUOS_HELPERS;
    return hlp < cap ? hlp : cap;
}

/* Work-queue reservation shared by the sequencer warps (each on an SM of its
 * own; the turn lives in device memory, dctl->turn). Work-queue space is
 * given out in ticket order: the warp whose batch starts at the turn's
 * ticket takes the turn's queue index, advances it by the batch's entries
 * and passes the turn on. Workers claim entries in queue order, so an entry
 * of a descriptor is never queued behind the entries of a later descriptor
 * that may wait for it (with several sequencers, a later window may be
 * ready first).
 *
 * Ticket and queue index travel in one 64-bit word (32 bits each), so a
 * hand-over is one relaxed store and one relaxed load that finds it: the
 * next holder needs nothing else from the previous one (its work-queue
 * stores are found by the workers through their stamps), so neither side
 * takes a fence. A fence here would also wait for the holder's next ring
 * poll, in flight across NVLink-C2C, and the turn passes once per batch.
 * Both fields are taken modulo 2^32 and widened against what the waiter
 * already knows: its ticket (the turn it waits for), and a work-queue
 * index at or below the current one and less than 2^32 below it (its own
 * last reservation: between two reservations of one sequencer the other
 * sequencers reserve at most S windows of 128 descriptors of at most
 * GPUOS_HELPERS entries each). */
DEV uint64_t turn_word(uint64_t ticket, uint64_t tq)
{
    return (tq << 32) | (ticket & 0xFFFFFFFFull);
}

/* Lane 0: wait (bounded) for the turn of the batch starting at ticket s;
 * on success *tq is the next free work-queue index, widened from `known`. */
DEV bool baton_wait(const gpuos_exec_params &p, uint64_t s, uint64_t known, uint64_t bound_ns, unsigned long long *tq)
{
    Elapsed w;
    w.start();
    uint32_t n = 0;
    uint64_t v;
    while ((uint32_t)(v = ld_relaxed_gpu(&p.dctl->turn)) != (uint32_t)s) {
        if ((++n & 63u) == 0 && w.tick(globaltimer()) > bound_ns) return false;
    }
    *tq = known + (uint32_t)((uint32_t)(v >> 32) - (uint32_t)known);
    return true;
}

/* Lane 0: pass the turn on to the batch starting at ticket `next`, with the
 * next free work-queue index. */
DEV void baton_pass(const gpuos_exec_params &p, uint64_t tq_head, uint64_t next)
{
    st_relaxed_gpu(reinterpret_cast<unsigned long long *>(&p.dctl->turn), turn_word(next, tq_head));
}

/* A sequencer warp: ring -> mirror + work queue, up to 128 descriptors per
 * batch (four ring slots per lane: slot s + lane + 32 h). With S sequencer
 * warps (warp 0 of blocks 0 .. S-1), tickets are cut into windows of 128
 * (or the ring size, if smaller) and sequencer sq takes windows sq,
 * sq + S, sq + 2S, ...: reading, checking and mirroring descriptors run in
 * parallel on S SMs; only the reservation of work-queue space follows
 * ticket order (baton_wait / baton_pass). */
#define SEQ_SPL 2    /* ring slots per lane in one half of a batch (64 descriptors) */
#define SEQ_HALVES 2 /* halves per batch */
#define SEQ_POLL (SEQ_SPL * SEQ_HALVES)
DEV void sequencer(const gpuos_exec_params &p, gpuos_devdesc *sd, uint32_t gw, unsigned long long *s_table,
                   uint32_t sq, uint32_t S)
{
    const uint32_t lane = lane_id();
    uint32_t cached_version = 0xFFFFFFFFu; /* version whose table slot s_table holds */
    uint64_t *ws = p.warp_stats + (uint64_t)gw * GPUOS_WS_N;
    uint64_t s = 0, e = 0;
    uint64_t n_seq = 0, n_idle = 0, n_sleep = 0, t_body = 0, t_mirror = 0, t_pubs = 0, n_inline = 0;
    uint32_t n_batches = 0;
    uint32_t polls = 0;
    uint64_t hb = ld_relaxed_sys(&p.hctl->heartbeat);
    uint64_t t_active = 0;
    Elapsed idle;
    idle.start();
    const uint32_t N = p.ring_mask + 1;
    const uint32_t WIN = N < 32u * SEQ_POLL ? N : 32u * SEQ_POLL; /* window of tickets, and batch limit */
    const uint64_t WSKIP = (uint64_t)WIN * (S - 1);               /* other sequencers' windows */
    s = p.ticket_base + (uint64_t)WIN * sq;
    e = p.tq_base;
    uint64_t wend = s + WIN;
    if (lane == 0 && sq == 0) st_relaxed_sys32(&p.hctl->state, 1u);

    /* commit words of slots s + lane + 32 h (h < SEQ_POLL), polled ahead
     * (relaxed; the batch's fence comes after they are seen): the poll for
     * the next batch is issued before the current one is published, so its
     * NVLink-C2C round trip overlaps the publication. A batch of up to 128
     * descriptors is read and mirrored in halves of 64 (two per lane) under
     * one acquire fence, one mirror fence and one publication. */
    uint64_t seqv[SEQ_POLL];
    uint32_t cheap = 0; /* the last poll read slot s only */
#pragma unroll
    for (int h = 0; h < SEQ_POLL; h++)
        seqv[h] = ld_relaxed_sys(&p.ring[(uint32_t)((s + lane + 32u * h) & p.ring_mask)].seq);
    while (true) {
        uint64_t rm[SEQ_HALVES];
#pragma unroll
        for (int q = 0; q < SEQ_HALVES; q++) {
            rm[q] = 0;
#pragma unroll
            for (int h = 0; h < SEQ_SPL; h++) {
                const uint32_t pos = lane + 32u * (SEQ_SPL * q + h);
                rm[q] |= (uint64_t)__ballot_sync(0xFFFFFFFFu, seqv[SEQ_SPL * q + h] == s + pos + 1) << (32 * h);
            }
        }
        uint32_t k = (rm[0] != ~0ull) ? (uint32_t)(__ffsll((long long)~rm[0]) - 1)
                                      : 64u + ((rm[1] == ~0ull) ? 64u : (uint32_t)(__ffsll((long long)~rm[1]) - 1));
        if (k > wend - s) k = (uint32_t)(wend - s);
        if (cheap) {
            /* the last poll read slot s alone: it only tells whether the
             * window has started; count the batch with a full poll */
            cheap = 0;
            if (k) {
#pragma unroll
                for (int h = 0; h < SEQ_POLL; h++)
                    seqv[h] = ld_relaxed_sys(&p.ring[(uint32_t)((s + lane + 32u * h) & p.ring_mask)].seq);
                continue;
            }
        }
        if (k == 0) {
            /* idle: stop flag, exit_after, watchdog */
            if (n_idle++ == 0 || polls == 0) {
                if (lane == 0 && sq == 0) st_relaxed_sys(&p.hctl->sequenced, s);
            }
            if ((polls & 31u) == 0) {
                uint32_t reason = 0;
                /* another sequencer decided to leave: follow it */
                const uint32_t follow = S > 1 ? ld_relaxed_gpu32(&p.dctl->exit_flag) : 0u;
                if (__shfl_sync(0xFFFFFFFFu, follow, 0)) break;
                if (ld_relaxed_sys32(&p.hctl->stop)) reason = 1;
                if (p.exit_after && *reinterpret_cast<volatile unsigned long long *>(&p.dctl->completed) >= p.exit_after)
                    reason = 3;
                const uint64_t now = globaltimer();
                const uint64_t h2 = ld_relaxed_sys(&p.hctl->heartbeat);
                if (h2 != hb) {
                    hb = h2;
                    idle.start();
                }
                if (idle.tick(now) > p.idle_exit_ns && p.idle_exit_ns) reason = 2;
                t_active = now - idle.acc;
                reason = __shfl_sync(0xFFFFFFFFu, reason, 0);
                if (reason) {
                    if (lane == 0) {
                        /* what the decision saw, for the host's diagnostics */
                        st_relaxed_sys(&p.hctl->exit_now, now);
                        st_relaxed_sys(&p.hctl->exit_active, t_active);
                        set_exit(p, reason);
                    }
                    break;
                }
            }
            backoff(polls, p.spin_polls, p.backoff_min_ns, short_cap(p), &n_sleep);
            /* Idle. The warp whose window holds the next ticket to be given
             * work-queue space polls all of its slots; the others read only
             * their window's first slot (one line across NVLink-C2C instead
             * of 128), so that idle sequencers do not crowd the SM's
             * outstanding loads and slow the poll that matters. */
            if (S > 1 && (uint32_t)ld_relaxed_gpu(&p.dctl->turn) != (uint32_t)s) {
                cheap = 1;
#pragma unroll
                for (int h = 0; h < SEQ_POLL; h++) seqv[h] = 0;
                if (lane == 0) seqv[0] = ld_relaxed_sys(&p.ring[(uint32_t)(s & p.ring_mask)].seq);
            } else {
#pragma unroll
                for (int h = 0; h < SEQ_POLL; h++)
                    seqv[h] = ld_relaxed_sys(&p.ring[(uint32_t)((s + lane + 32u * h) & p.ring_mask)].seq);
            }
            continue;
        }
        const uint64_t t_obs = globaltimer();
        polls = 0;
        /* a lone descriptor's observation time goes to its record at once
         * (a posted write): the host times commit -> observe and calibrates
         * the clocks with it. Every record gets it again at completion,
         * from t_disp (the mirror fence orders that store before the
         * publication); a batch's early echo would make this batch's fence
         * wait for its stores across NVLink-C2C. */
        if (k == 1 && lane == 0) st_relaxed_sys(&p.rec[(uint32_t)(s & p.ring_mask)].t_dispatch, t_obs);
        /* the commits seen above happen-before everything below */
        fence_acq_rel_sys();
        uint32_t version = 0;
        int32_t status[SEQ_POLL];
        uint32_t nt[SEQ_POLL];
#pragma unroll
        for (int h = 0; h < SEQ_POLL; h++) {
            status[h] = GPUOS_ST_OK;
            nt[h] = 0;
        }
        /* the second half's bodies start towards L2 now (coherent with the
         * host's writes): their NVLink-C2C round trip overlaps the first
         * half's */
#pragma unroll
        for (int h = 0; h < SEQ_SPL; h++) {
            const uint32_t pos = 64u + lane + 32u * h;
            if (pos < k) {
                const char *src = reinterpret_cast<const char *>(p.ring + (uint32_t)((s + pos) & p.ring_mask));
#pragma unroll
                for (int i = 0; i < 4; i++) asm volatile("prefetch.global.L2 [%0];" ::"l"(src + 32 * i));
            }
        }
        gpuos_desc dsc[SEQ_SPL];
#pragma unroll
        for (int q = 0; q < SEQ_HALVES; q++) {
            const uint32_t base = 64u * q;
            if (base >= k) break; /* k is warp-uniform */
#pragma unroll
            for (int h = 0; h < SEQ_SPL; h++) {
                const uint32_t pos = base + lane + 32u * h;
                if (pos < k) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(p.ring + (uint32_t)((s + pos) & p.ring_mask));
                    uint4 *dv = reinterpret_cast<uint4 *>(&dsc[h]);
#pragma unroll
                    for (int i = 0; i < 8; i++) dv[i] = src[i];
                }
            }
            if (q == 0) {
                /* the table version: a relaxed load after the fence above,
                 * so at least the version stored before these commits */
                if (lane == 0) version = ld_relaxed_sys32(&p.hctl->version);
                version = __shfl_sync(0xFFFFFFFFu, version, 0);
                if (version != cached_version) {
                    /* a new version: the fence makes the host's slot writes,
                     * which preceded its store of this version, visible;
                     * then the slot is copied into shared memory */
                    fence_acq_rel_sys();
                    __syncwarp();
                    for (uint32_t i = lane; i < GPUOS_MAX_OPS; i += 32)
                        s_table[i] = ld_relaxed_sys(p.table + (version & 1u) * GPUOS_MAX_OPS + i);
                    __syncwarp();
                    cached_version = version;
                }
            }
            /* a FENCE descriptor must start a batch; cut the batch before it */
            uint64_t fmask = 0;
#pragma unroll
            for (int h = 0; h < SEQ_SPL; h++) {
                const uint32_t pos = base + lane + 32u * h;
                fmask |= (uint64_t)__ballot_sync(0xFFFFFFFFu, pos < k && (dsc[h].flags & GPUOS_FLAG_FENCE))
                         << (32 * h);
            }
            const uint64_t later = (q == 0) ? (fmask & ~1ull) : fmask;
            if (later) {
                const uint32_t cut = base + (uint32_t)(__ffsll((long long)later) - 1);
                if (cut < k) k = cut;
            }
            uint32_t fence_status = GPUOS_ST_OK;
            if (q == 0 && (fmask & 1ull)) {
                if (lane == 0) {
                    Elapsed w;
                    w.start();
                    uint32_t fp = 0;
                    while (*reinterpret_cast<volatile unsigned long long *>(&p.dctl->completed) < s) {
                        if (w.tick(globaltimer()) > p.dep_timeout_ns) {
                            fence_status = GPUOS_ST_DEP_TIMEOUT;
                            break;
                        }
                        backoff(fp, p.spin_polls, p.backoff_min_ns, short_cap(p), &n_sleep);
                    }
                    __threadfence();
                }
                fence_status = __shfl_sync(0xFFFFFFFFu, fence_status, 0);
            }
            /* validate and mirror */
#pragma unroll
            for (int h = 0; h < SEQ_SPL; h++) {
                const uint32_t pos = base + lane + 32u * h;
                const uint64_t my_t = s + pos;
                if (pos < k) {
                    int32_t st = GPUOS_ST_OK;
                    *reinterpret_cast<volatile uint64_t *>(p.t_disp + (uint32_t)(my_t & p.ring_mask)) = t_obs;
                    if (dsc[h].ticket != my_t) st = GPUOS_ST_BAD_DESC;
                    else if (dsc[h].op_id >= GPUOS_MAX_OPS) st = GPUOS_ST_BAD_OP;
                    else if (dsc[h].ntiles == 0 || dsc[h].ntiles > GPUOS_TILE_MAX) st = GPUOS_ST_BAD_ARGS;
                    if (pos == 0 && fence_status) st = (int32_t)fence_status;
                    status[SEQ_SPL * q + h] = st;
                    if (st == GPUOS_ST_OK) {
                        /* one work-queue entry per helper warp (at most
                         * GPUOS_HELPERS); helper i starts with tile i and takes
                         * later tiles from the descriptor's tile counter */
                        const uint32_t hc = helper_count(dsc[h].op_id, dsc[h].ntiles, p.workers);
                        nt[SEQ_SPL * q + h] = hc;
                        dsc[h].user = s_table[dsc[h].op_id];                 /* -> fn */
                        dsc[h].seq = (uint64_t)version | ((uint64_t)hc << 32); /* -> version, helpers */
                        uint4 *mv = reinterpret_cast<uint4 *>(p.mirror + (uint32_t)(my_t & p.ring_mask));
                        const uint4 *dv = reinterpret_cast<const uint4 *>(&dsc[h]);
#pragma unroll
                        for (int i = 0; i < 8; i++) __stcg(mv + i, dv[i]);
                    }
                }
            }
        }
        const uint64_t t_b = globaltimer();
        /* An idle ring (a batch of one) and a dependency-free single-tile
         * descriptor: the sequencer runs the tile itself, sparing the
         * mirror -> work queue -> worker hop. (k == 1: dsc[0] holds it.) */
        uint32_t inl = 0;
        if (lane == 0)
            inl = (k == 1 && status[0] == GPUOS_ST_OK && dsc[0].ntiles == 1 && dsc[0].dep[0] == 0 &&
                   dsc[0].dep[1] == 0) ? 1u : 0u;
        inl = __shfl_sync(0xFFFFFFFFu, inl, 0);
        if (inl) {
            const uint32_t slot = (uint32_t)(s & p.ring_mask);
            if (S > 1) {
                /* no work-queue space, but the turn passes through it */
                uint32_t ok = 1;
                unsigned long long e0 = 0;
                if (lane == 0) {
                    ok = baton_wait(p, s, e, p.dep_timeout_ns, &e0) ? 1u : 0u;
                    if (ok) baton_pass(p, e0, s + 1);
                    else set_exit(p, 4u);
                }
                if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
                e = __shfl_sync(0xFFFFFFFFu, e0, 0);
            }
            if (lane == 0) {
                uint4 *sv = reinterpret_cast<uint4 *>(sd);
                const uint4 *dv = reinterpret_cast<const uint4 *>(&dsc[0]);
#pragma unroll
                for (int i = 0; i < 8; i++) sv[i] = dv[i];
                const uint64_t ts = globaltimer();
                *reinterpret_cast<volatile uint64_t *>(p.t_pub + slot) = ts;
                *reinterpret_cast<volatile uint64_t *>(p.t_start + slot) = ts;
            }
            __syncwarp();
            const gpuos_op_fn fn = reinterpret_cast<gpuos_op_fn>(sd->fn);
            const int32_t st = fn ? fn(sd, 0) : GPUOS_ST_BAD_OP;
            __syncwarp();
            if (lane == 0) complete_desc(p, s, slot, st, version);
            s += 1;
            if (S == 1) {
                wend = s + WIN; /* one sequencer: batches start anywhere */
            } else if (s == wend) {
                s += WSKIP;
                wend = s + WIN;
            }
            n_seq += 1;
            n_inline += 1;
            if (lane == 0) {
                if (sq == 0) st_relaxed_sys(&p.hctl->sequenced, s);
                ws[GPUOS_WS_SEQ] = n_seq;
                ws[GPUOS_WS_TILES] = n_inline;
            }
            idle.start();
#pragma unroll
            for (int h = 0; h < SEQ_POLL; h++)
                seqv[h] = ld_relaxed_sys(&p.ring[(uint32_t)((s + lane + 32u * h) & p.ring_mask)].seq);
            continue;
        }
        /* the batch's publication time, stored before the fence below like
         * the mirror writes: a worker that finds an entry of the batch (and
         * so may complete its descriptor) sees it */
#pragma unroll
        for (int h = 0; h < SEQ_POLL; h++) {
            const uint32_t pos = lane + 32u * h;
            if (pos < k) *reinterpret_cast<volatile uint64_t *>(p.t_pub + (uint32_t)((s + pos) & p.ring_mask)) = t_b;
        }
        /* every lane's mirror writes happen-before every lane's fence */
        __syncwarp();
        __threadfence();
        const uint64_t t_m = globaltimer();
        /* where the next batch starts (this window, or this warp's next one) */
        uint64_t s_next = s + k, wend_next = wend;
        if (S == 1) {
            wend_next = s_next + WIN; /* one sequencer: batches start anywhere */
        } else if (s_next == wend) {
            s_next += WSKIP;
            wend_next = s_next + WIN;
        }
        /* the next batch's poll, in flight during the publication below */
#pragma unroll
        for (int h = 0; h < SEQ_POLL; h++)
            seqv[h] = ld_relaxed_sys(&p.ring[(uint32_t)((s_next + lane + 32u * h) & p.ring_mask)].seq);
        /* exclusive prefix of entry counts in ticket order -> queue ranges
         * (position lane + 32 h for h < SEQ_POLL) */
        uint32_t excl[SEQ_POLL];
        uint32_t base = 0;
#pragma unroll
        for (int h = 0; h < SEQ_POLL; h++) {
            uint32_t incl = nt[h];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= (uint32_t)o) incl += v;
            }
            excl[h] = base + incl - nt[h];
            base += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        const uint32_t total = base;
        if (S > 1) {
            /* this batch's turn to reserve work-queue space */
            uint32_t ok = 1;
            unsigned long long e0 = 0;
            if (lane == 0) {
                ok = baton_wait(p, s, e, p.dep_timeout_ns, &e0) ? 1u : 0u;
                if (ok) {
                    baton_pass(p, e0 + total, s + k);
                } else {
                    set_exit(p, 4u);
                }
            }
            if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
            e = __shfl_sync(0xFFFFFFFFu, e0, 0);
        }
        /* Publication. Each lane writes the first (up to 16) entries of its own
         * descriptors; descriptors with more entries are finished by the
         * whole warp, one after another. Entry j of a descriptor whose first
         * entry has index i0 is tq_word(i0 + j, slot, j) = W0 + j * TQ_STEP
         * with W0 = tq_word(i0, slot, 0): the stamp field takes the carry-free
         * (mod 2^64) sum and the helper field j < 4096 never carries. The
         * queue index is taken modulo 2^32 (the queue is smaller). */
        {
            constexpr uint64_t TQ_STEP = (1ull << 28) + 1ull;
            uint32_t most = 0;
#pragma unroll
            for (int h = 0; h < SEQ_POLL; h++) most = nt[h] > most ? nt[h] : most;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) most = max(most, __shfl_xor_sync(0xFFFFFFFFu, most, o));
            const uint32_t jmax = most < 16u ? most : 16u;
#pragma unroll
            for (int h = 0; h < SEQ_POLL; h++) {
                const uint32_t slot = (uint32_t)((s + lane + 32u * h) & p.ring_mask);
                const uint64_t i0 = e + excl[h];
                const uint32_t q0 = (uint32_t)i0;
                uint64_t wd = tq_word(i0, slot, 0);
                const uint32_t nj = nt[h] < jmax ? nt[h] : jmax;
#pragma unroll 4
                for (uint32_t j = 0; j < jmax; j++) {
                    if (j < nj)
                        *reinterpret_cast<volatile unsigned long long *>(p.tq + ((q0 + j) & p.tq_mask)) = wd;
                    wd += TQ_STEP;
                }
            }
            if (most > 16u) {
#pragma unroll
                for (int h = 0; h < SEQ_POLL; h++) {
                    uint32_t big = __ballot_sync(0xFFFFFFFFu, nt[h] > 16u);
                    while (big) {
                        const uint32_t i = (uint32_t)(__ffs(big) - 1);
                        big &= big - 1;
                        const uint32_t nti = __shfl_sync(0xFFFFFFFFu, nt[h], i);
                        const uint32_t bi = __shfl_sync(0xFFFFFFFFu, excl[h], i);
                        const uint32_t slot = (uint32_t)((s + i + 32u * h) & p.ring_mask);
                        const uint64_t i0 = e + bi;
                        const uint32_t q0 = (uint32_t)i0;
                        uint64_t wd = tq_word(i0, slot, 0) + (uint64_t)(16u + lane) * TQ_STEP;
                        for (uint32_t j = 16u + lane; j < nti; j += 32) {
                            *reinterpret_cast<volatile unsigned long long *>(p.tq + ((q0 + j) & p.tq_mask)) = wd;
                            wd += 32ull * TQ_STEP;
                        }
                    }
                }
            }
        }
        const uint64_t t_pub = globaltimer();
#pragma unroll
        for (int h = 0; h < SEQ_POLL; h++) {
            const uint32_t pos = lane + 32u * h;
            const uint64_t my_t = s + pos;
            const uint32_t slot = (uint32_t)(my_t & p.ring_mask);
            /* descriptors that failed validation complete at once */
            if (pos < k && status[h] != GPUOS_ST_OK) complete_desc(p, my_t, slot, status[h], version);
        }
        e += total;
        s = s_next;
        wend = wend_next;
        n_seq += k;
        t_body += t_b - t_obs;
        t_mirror += t_m - t_b;
        t_pubs += t_pub - t_m;
        if (lane == 0) {
            /* the host-visible count (statistics and diagnostics only) goes
             * out every 16th batch and when the ring runs dry: a store
             * across NVLink-C2C per batch would make the next batch's
             * system-scope fence wait for its acknowledgement */
            if ((++n_batches & 15u) == 0 && sq == 0) st_relaxed_sys(&p.hctl->sequenced, s);
            ws[GPUOS_WS_SEQ] = n_seq;
            ws[GPUOS_WS_IDLE] = n_idle;
            ws[GPUOS_WS_SLEEPS] = n_sleep;
            ws[GPUOS_WS_T_BODY] = t_body;
            ws[GPUOS_WS_T_MIRROR] = t_mirror;
            ws[GPUOS_WS_T_PUB] = t_pubs;
            ws[GPUOS_WS_BATCHES] = n_batches;
        }
        idle.start();
    }
    if (lane == 0) {
        ws[GPUOS_WS_SEQ] = n_seq;
        ws[GPUOS_WS_IDLE] = n_idle;
        ws[GPUOS_WS_SLEEPS] = n_sleep;
    }
}

/* A worker warp: claim a tile, wait for its dependencies, dispatch, count. */
DEV void worker(const gpuos_exec_params &p, gpuos_devdesc *sd, uint32_t gw, uint64_t *sprof)
{
    const uint32_t lane = lane_id();
    uint64_t *ws = p.warp_stats + (uint64_t)gw * GPUOS_WS_N;
    uint64_t t_found = 0, t_deps = 0; /* lane 0: entry found, dependencies met */
    uint64_t n_tiles = 0, n_idle = 0, n_sleep = 0, n_depw = 0;
    const uint32_t N = p.ring_mask + 1;
    unsigned long long e = 0;
    if (lane == 0) e = atomicAdd(&p.dctl->tq_claim, 1ull);
    e = __shfl_sync(0xFFFFFFFFu, e, 0);
    while (true) {
        unsigned long long *ent = p.tq + (e & p.tq_mask);
        uint32_t polls = 0;
        uint32_t leave = 0;
        uint64_t w = 0;
        if (lane == 0) {
            while (true) {
                w = ld_relaxed_gpu(reinterpret_cast<const uint64_t *>(ent));
                if (tq_is(w, e)) {
                    fence_acq_rel_gpu(); /* the acquire, once */
                    t_found = globaltimer();
                    break;
                }
                n_idle++;
                if ((polls & 15u) == 0 && ld_relaxed_gpu32(&p.dctl->exit_flag)) {
                    leave = 1;
                    break;
                }
                backoff(polls, p.spin_polls, p.backoff_min_ns, p.backoff_max_ns, &n_sleep);
            }
        }
        leave = __shfl_sync(0xFFFFFFFFu, leave, 0);
        if (leave) break;
        w = __shfl_sync(0xFFFFFFFFu, w, 0);
        __syncwarp(); /* lane 0's acquire before every lane's mirror read */
        const uint32_t slot = (uint32_t)((w >> 12) & 0xFFFFu);
        uint32_t tile = (uint32_t)(w & 0xFFFu); /* helper index = its first tile */
        /* descriptor -> shared memory */
        reinterpret_cast<uint32_t *>(sd)[lane] = __ldcg(reinterpret_cast<const uint32_t *>(p.mirror + slot) + lane);
        __syncwarp();
        const uint64_t ticket = sd->ticket;
        const uint32_t ntiles = sd->ntiles;
        const uint32_t helpers = sd->pad; /* helper count fixed by the sequencer */
        const gpuos_op_fn fn = reinterpret_cast<gpuos_op_fn>(sd->fn);
        int32_t dstatus = GPUOS_ST_OK;
        if (lane == 0) {
            for (int i = 0; i < 2; i++) {
                const uint64_t dep = sd->dep[i];
                if (dep == 0) continue;
                if (dep > ticket) {
                    dstatus = GPUOS_ST_BAD_DESC;
                    break;
                }
                if (ticket + 1 - dep >= N) continue; /* older than the ring window: done */
                const uint32_t dslot = (uint32_t)((dep - 1) & p.ring_mask);
                const uint64_t *stamp = p.done_dev + dslot;
                if (ld_acquire_gpu(stamp) >= dep) continue;
                n_depw++;
                /* A split dependency is complete as soon as its tile counter
                 * reaches its tile count: every helper's acq_rel add is in the
                 * counter's release sequence, so acquiring the final value
                 * acquires every tile's writes; the last helper's own round
                 * trip and the stamp's release come later. The counter is
                 * zero before the dependency's helpers count (the previous
                 * user of the slot reset it before its record freed the ring
                 * slot, which happens-before this descriptor was published)
                 * and is reset only after the dependency completed, so a
                 * match never comes early. Sole-tile dependencies never count
                 * (ntiles 1): they are seen through the stamp. */
                const uint32_t dnt = __ldcg(&p.mirror[dslot].ntiles);
                const unsigned long long *dcnt = p.tiles_done + dslot;
                Elapsed w;
                w.start();
                uint32_t dp = 0;
                while (ld_relaxed_gpu(stamp) < dep &&
                       (dnt < 2 || (uint32_t)ld_relaxed_gpu(reinterpret_cast<const uint64_t *>(dcnt)) != dnt)) {
                    if (w.tick(globaltimer()) > p.dep_timeout_ns) {
                        dstatus = GPUOS_ST_DEP_TIMEOUT;
                        break;
                    }
                    if ((dp & 15u) == 0 && ld_relaxed_gpu32(&p.dctl->exit_flag)) {
                        dstatus = GPUOS_ST_ABORTED;
                        break;
                    }
                    backoff(dp, p.spin_polls, p.backoff_min_ns, short_cap(p), &n_sleep);
                }
                if (dstatus) break;
                fence_acq_rel_gpu(); /* the acquire, once */
            }
        }
        dstatus = __shfl_sync(0xFFFFFFFFu, dstatus, 0);
        /* tile 0 starts once its dependencies are met */
        if (lane == 0) {
            t_deps = globaltimer();
            if (tile == 0) *reinterpret_cast<volatile uint64_t *>(p.t_start + slot) = t_deps;
        }
        __syncwarp();
        /* the helper's tiles: its first tile, then tiles from the descriptor's
         * counter. Each next tile is claimed before the current one runs
         * (the claim's latency overlaps the work), and the helper counts its
         * tiles done only after its last claim: the descriptor cannot
         * complete (and its counters be recycled) while a helper may still
         * claim. */
        int32_t status = dstatus;
        uint32_t count = 0;
        /* row ops may take the helper's further rows themselves (the claim
         * context in the warp's staging header); anything else, or a row op
         * that did not, gets one tile per call */
        const bool rowop = sd->op_id >= GPUOS_OP_SOFTMAX && sd->op_id <= GPUOS_OP_ROWMIN;
        WarpStage *wst = warp_stage();
        while (true) {
            uint32_t next = ntiles;
            if (rowop) {
                if (lane == 0) {
                    wst->claim_ctr = ntiles > helpers ? p.tile_ctr + slot : nullptr;
                    wst->claim_base = helpers;
                    wst->claim_done = 0;
                }
                __syncwarp();
            } else if (ntiles > helpers && lane == 0) {
                next = helpers + atomicAdd(p.tile_ctr + slot, 1u);
            }
            if (status == GPUOS_ST_OK) {
                if (fn == nullptr) status = GPUOS_ST_BAD_OP;
                else status = fn(sd, tile);
            }
            if (rowop) {
                __syncwarp();
                if (wst->claim_done) {
                    count += wst->claim_count;
                    next = wst->claim_next;
                } else {
                    count++;
                    if (ntiles > helpers && lane == 0) next = helpers + atomicAdd(p.tile_ctr + slot, 1u);
                }
                if (lane == 0) {
                    wst->claim_ctr = nullptr;
                    wst->claim_done = 0;
                }
            } else {
                count++;
            }
            next = __shfl_sync(0xFFFFFFFFu, next, 0);
            if (next >= ntiles) break;
            tile = next;
        }
        __syncwarp();
        if (lane == 0) {
            const uint64_t t_body = globaltimer();
            if (ntiles == 1) {
                /* sole tile: no counter round trip; the warp barrier above
                 * orders every lane's writes before the completion releases */
                complete_desc(p, ticket, slot, status, sd->version);
            } else {
                /* one acq_rel add per helper: its tiles' writes are released
                 * to the last helper, which acquires every helper's; a failed
                 * helper records its status first and counts itself in the
                 * high word */
                if (status) atomicCAS(p.err + slot, 0u, (uint32_t)status);
                const unsigned long long add = (unsigned long long)count | (status ? (1ull << 32) : 0ull);
                const unsigned long long old = atom_add_acq_rel_gpu(p.tiles_done + slot, add);
                if ((uint32_t)old + count == ntiles) {
                    const bool failed = (old >> 32) != 0 || status != GPUOS_ST_OK;
                    const int32_t st = failed ? (int32_t)ld_relaxed_gpu32(p.err + slot) : GPUOS_ST_OK;
                    complete_desc(p, ticket, slot, st, sd->version);
                }
            }
            /* tile profile: accumulated in shared memory, written through
             * to the warp's row (stores only, no read round trip) */
            const uint32_t bk = sd->op_id < GPUOS_OP_BUILTIN_COUNT ? sd->op_id : GPUOS_OP_BUILTIN_COUNT;
            const uint64_t t_fin = globaltimer();
            const uint64_t add[GPUOS_PROF_FIELDS] = {count, t_body - t_deps, t_fin - t_body, t_deps - t_found};
#pragma unroll
            for (int f = 0; f < GPUOS_PROF_FIELDS; f++) {
                const uint64_t v = sprof[f * GPUOS_PROF_BUCKETS + bk] + add[f];
                sprof[f * GPUOS_PROF_BUCKETS + bk] = v;
                ws[GPUOS_WS_PROF + f * GPUOS_PROF_BUCKETS + bk] = v;
            }
            n_tiles += count;
            ws[GPUOS_WS_TILES] = n_tiles;
            ws[GPUOS_WS_IDLE] = n_idle;
            ws[GPUOS_WS_SLEEPS] = n_sleep;
            ws[GPUOS_WS_DEPWAIT] = n_depw;
        }
        /* claim the next entry only now: a claim held while this warp was
         * busy would keep a published tile waiting behind this one */
        unsigned long long e_next = 0;
        if (lane == 0) e_next = atomicAdd(&p.dctl->tq_claim, 1ull);
        e = __shfl_sync(0xFFFFFFFFu, e_next, 0);
        __syncwarp();
    }
    if (lane == 0) {
        ws[GPUOS_WS_TILES] = n_tiles;
        ws[GPUOS_WS_IDLE] = n_idle;
        ws[GPUOS_WS_SLEEPS] = n_sleep;
        ws[GPUOS_WS_DEPWAIT] = n_depw;
    }
}

extern "C" __global__ void __launch_bounds__(GPUOS_MAX_WPB * 32, 1) gpuos_executor_kernel(gpuos_exec_params p)
{
    __shared__ __align__(16) gpuos_devdesc sdesc[GPUOS_MAX_WPB];
    __shared__ unsigned long long s_table[GPUOS_MAX_OPS]; /* the sequencer's copy of one table slot */
    __shared__ uint64_t s_prof[GPUOS_MAX_WPB][GPUOS_PROF_FIELDS * GPUOS_PROF_BUCKETS]; /* tile profiles */
    const uint32_t warp = threadIdx.x >> 5;
    for (uint32_t i = threadIdx.x & 31u; i < GPUOS_PROF_FIELDS * GPUOS_PROF_BUCKETS; i += 32) s_prof[warp][i] = 0;
    stage_init(p.stage_bytes); /* (its block barriers also order the clearing above) */
    const uint32_t gw = blockIdx.x * (blockDim.x >> 5) + warp;
    /* Blocks 0 .. S-1 each hold one sequencer warp and nothing else (unless
     * there is only one block): worker warps beside a sequencer would share
     * its issue slots and load/store pipe, and sequencers on one SM slowed
     * each other (one SM's outstanding loads across NVLink-C2C). */
    const uint32_t S = p.sequencers;
    if (gridDim.x == 1) {
        if (warp == 0) sequencer(p, &sdesc[0], gw, s_table, 0u, 1u);
        else worker(p, &sdesc[warp], gw, s_prof[warp]);
    } else if (blockIdx.x < S) {
        if (warp == 0) sequencer(p, &sdesc[0], gw, s_table, blockIdx.x, S);
    } else {
        worker(p, &sdesc[warp], gw, s_prof[warp]);
    }
}

/* ===========================================================================
 * Eager baseline: the same op bodies, one launch per descriptor, one warp
 * per tile, one warp per block (spreads a descriptor over many SMs).
 * ======================================================================== */
#define EAGER_WPB 1
extern "C" __global__ void __launch_bounds__(EAGER_WPB * 32) gpuos_eager_kernel(gpuos_devdesc d, uint32_t stage_bytes)
{
    __shared__ __align__(16) gpuos_devdesc sd[EAGER_WPB];
    stage_init(stage_bytes);
    const uint32_t warp = threadIdx.x >> 5;
    reinterpret_cast<uint32_t *>(&sd[warp])[lane_id()] = reinterpret_cast<const uint32_t *>(&d)[lane_id()];
    __syncwarp();
    const uint32_t tile = blockIdx.x * EAGER_WPB + warp;
    if (tile < sd[warp].ntiles) (void)builtin_call(sd[warp].op_id, &sd[warp], tile);
}

/* ===========================================================================
 * Host-side launch helpers
 * ======================================================================== */
extern "C" uint32_t gpuos_dev_dyn_smem(uint32_t wpb, uint32_t stage_bytes)
{
    return 16u + wpb * (GPUOS_WARP_STAGE_HDR + stage_bytes);
}

extern "C" int gpuos_dev_launch_executor(const gpuos_exec_params *p, uint32_t blocks, uint32_t wpb, void *stream)
{
    const uint32_t dyn = gpuos_dev_dyn_smem(wpb, p->stage_bytes);
    if (cudaFuncSetAttribute(gpuos_executor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn) !=
        cudaSuccess)
        return -1;
    gpuos_executor_kernel<<<blocks, wpb * 32, dyn, (cudaStream_t)stream>>>(*p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

extern "C" int gpuos_dev_builtin_table(gpuos_op_fn *host_out, uint32_t n)
{
    if (n > GPUOS_OP_BUILTIN_COUNT) n = GPUOS_OP_BUILTIN_COUNT;
    return cudaMemcpyFromSymbol(host_out, g_builtin_ops, n * sizeof(gpuos_op_fn)) == cudaSuccess ? 0 : -1;
}

extern "C" int gpuos_dev_executor_attrs(uint32_t *regs, uint32_t *smem)
{
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, gpuos_executor_kernel) != cudaSuccess) return -1;
    *regs = (uint32_t)a.numRegs;
    *smem = (uint32_t)a.sharedSizeBytes;
    return 0;
}

extern "C" int gpuos_dev_preload(void)
{
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, gpuos_executor_kernel) != cudaSuccess) return -1;
    if (cudaFuncGetAttributes(&a, gpuos_eager_kernel) != cudaSuccess) return -1;
    return 0;
}

extern "C" int gpuos_dev_eager_launch(const gpuos_desc *d, uint32_t ntiles, uint32_t stage_bytes, void *stream)
{
    gpuos_devdesc dd;
    static_assert(sizeof(dd) == sizeof(*d), "layout");
    memcpy(&dd, d, sizeof(dd));
    dd.ntiles = ntiles;
    const uint32_t grid = (ntiles + EAGER_WPB - 1) / EAGER_WPB;
    const uint32_t dyn = gpuos_dev_dyn_smem(EAGER_WPB, stage_bytes);
    static uint32_t attr_set = 0;
    if (dyn > attr_set) {
        if (cudaFuncSetAttribute(gpuos_eager_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn) !=
            cudaSuccess)
            return -1;
        attr_set = dyn;
    }
    gpuos_eager_kernel<<<grid, EAGER_WPB * 32, dyn, (cudaStream_t)stream>>>(dd, stage_bytes);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

/* ===========================================================================
 * Decode attention that allocates nothing.
 *
 * Some callers cannot allocate device memory when they attend: a serving
 * loop that runs beside a resident persistent executor (cudaFree, and a
 * cudaMalloc that has to grow the heap, wait for the device to go idle, which
 * a resident executor never does), and code that runs under a fixed memory
 * budget reserved up front. gpuos_sdpa_noalloc gives them the split-K decode
 * attention with its scratch in a file-scope device array of fixed size
 * instead of a caller workspace. The caller still passes every input and the
 * output.
 * ======================================================================== */
#define GPUOS_NOALLOC_MAX_BH 256u  /* requests x heads */
#define GPUOS_NOALLOC_MAX_L 4096u  /* rows attended per request (16 chunks of 256) */
#define GPUOS_NOALLOC_CTR_BYTES (4u * GPUOS_NOALLOC_MAX_BH)
#define GPUOS_NOALLOC_BYTES \
    (GPUOS_NOALLOC_CTR_BYTES + 4u * GPUOS_NOALLOC_MAX_BH * (GPUOS_NOALLOC_MAX_L / GPUOS_SDPA_CHUNK) * GPUOS_SDPA_PART)

/* Shared by every call on a device and kept until the process exits. In host
 * code this name is only a stand-in for the device array: never pass it to a
 * kernel; use the address cudaGetSymbolAddress returns for the device. */
static __device__ __align__(256) unsigned char g_sdpa_scratch[GPUOS_NOALLOC_BYTES];

extern "C" __global__ void __launch_bounds__(32) gpuos_sdpa_noalloc_kernel(gpuos_devdesc d)
{
    __shared__ __align__(16) gpuos_devdesc sd;
    stage_init(0); /* the op body reads the staging header: none here (register path) */
    reinterpret_cast<uint32_t *>(&sd)[lane_id()] = reinterpret_cast<const uint32_t *>(&d)[lane_id()];
    __syncwarp();
    if (blockIdx.x < sd.ntiles) (void)sdpa_tile(&sd, blockIdx.x);
}

extern "C" GPUOS_API int gpuos_sdpa_noalloc(const void *q, const void *Kc, const void *Vc, const int32_t *lens,
                                            void *out, uint32_t B, uint32_t H, uint32_t D, uint32_t Lcap,
                                            uint32_t Lmax, float scale, void *stream)
{
    if (!q || !Kc || !Vc || !lens || !out || B == 0 || H == 0 || D != 128 || Lcap == 0 || Lmax == 0 || Lmax > Lcap)
        return GPUOS_EINVAL;
    if (((uintptr_t)q | (uintptr_t)Kc | (uintptr_t)Vc | (uintptr_t)out) & 15u) return GPUOS_EINVAL;
    if ((uint64_t)B * H > GPUOS_NOALLOC_MAX_BH || Lmax > GPUOS_NOALLOC_MAX_L) return GPUOS_ETOOBIG;
    /* set-up, once per device with that device current: the device address of
     * the scratch array (the first call on a device does this) */
    static void *scratch[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GPUOS_ECUDA;
    if (!scratch[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_sdpa_scratch) != cudaSuccess || !ptr) return GPUOS_ECUDA;
        scratch[dev] = ptr;
    }
    /* the split-K counters must start at zero; the partials need no clearing */
    if (cudaMemsetAsync(scratch[dev], 0, GPUOS_NOALLOC_CTR_BYTES, (cudaStream_t)stream) != cudaSuccess)
        return GPUOS_ECUDA;
    gpuos_devdesc d;
    memset(&d, 0, sizeof(d));
    d.op_id = GPUOS_OP_SDPA;
    d.dtype = GPUOS_BF16;
    d.a = (uint64_t)(uintptr_t)q;
    d.b = (uint64_t)(uintptr_t)Kc;
    d.aux1 = (uint64_t)(uintptr_t)Vc;
    d.aux0 = (uint64_t)(uintptr_t)lens;
    d.out = (uint64_t)(uintptr_t)out;
    d.aux2 = (uint64_t)(uintptr_t)scratch[dev];
    d.dims[0] = B;
    d.dims[1] = H;
    d.dims[2] = D;
    d.dims[3] = Lcap;
    d.dims[4] = Lmax;
    d.dims[5] = GPUOS_NOALLOC_MAX_BH; /* counters reserved at the start of the array */
    d.fparam[0] = scale;
    d.ntiles = B * H * ((Lmax + GPUOS_SDPA_CHUNK - 1) / GPUOS_SDPA_CHUNK);
    gpuos_sdpa_noalloc_kernel<<<d.ntiles, 32, gpuos_dev_dyn_smem(1, 0), (cudaStream_t)stream>>>(d);
    return cudaGetLastError() == cudaSuccess ? GPUOS_OK : GPUOS_ECUDA;
}
