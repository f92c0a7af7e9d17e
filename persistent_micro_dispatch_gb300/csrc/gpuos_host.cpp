/*
 * Host side of the GB300 persistent micro-op dispatcher: the C ABI declared
 * in include/gpuos.h.
 *
 * Protocol ("GPUOS: A GPU Operating System Primitive for Transparent
 * Operation Fusion", §3 Q2 "1. Ring Buffer Communication Channel"): the host
 * takes the next ticket, acquires its slot (free once the descriptor that
 * last used it has completed), writes the 128-byte descriptor and commits it
 * with a store-release of the slot's commit word. The device's completion
 * record of each ticket is written with a store-release at system scope; the
 * host harvests records with load-acquire, in ticket order, and that is also
 * what frees slots.
 *
 * Operator injection (§3 Q2 "3. Dynamic Operator Table"): a precompiled
 * sm_103a cubin is loaded through the driver API, the address of its device
 * function is read from a __device__ variable, the inactive half of the
 * dual-slot table is written and the version counter flips. The sequencer
 * warp reads the version once per descriptor, so a descriptor runs entirely
 * with the old or entirely with the new entry.
 */
#include <cuda.h>
#include <cuda_runtime.h>

#include <dlfcn.h>
#include <sched.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <ctime>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "gpuos_internal.h"

namespace {

/* ---- driver API, resolved through the runtime (no link-time libcuda) ---- */
typedef CUresult (*pfn_cuModuleLoadData)(CUmodule *, const void *);
typedef CUresult (*pfn_cuModuleGetGlobal)(CUdeviceptr *, size_t *, CUmodule, const char *);
typedef CUresult (*pfn_cuModuleUnload)(CUmodule);
typedef CUresult (*pfn_cuModuleGetFunction)(CUfunction *, CUmodule, const char *);
typedef CUresult (*pfn_cuLinkCreate)(unsigned int, CUjit_option *, void **, CUlinkState *);
typedef CUresult (*pfn_cuLinkAddData)(CUlinkState, CUjitInputType, void *, size_t, const char *, unsigned int,
                                      CUjit_option *, void **);
typedef CUresult (*pfn_cuLinkComplete)(CUlinkState, void **, size_t *);
typedef CUresult (*pfn_cuLinkDestroy)(CUlinkState);
typedef CUresult (*pfn_cuFuncSetAttribute)(CUfunction, CUfunction_attribute, int);
typedef CUresult (*pfn_cuFuncGetAttribute)(int *, CUfunction_attribute, CUfunction);
typedef CUresult (*pfn_cuLaunchKernel)(CUfunction, unsigned int, unsigned int, unsigned int, unsigned int,
                                       unsigned int, unsigned int, unsigned int, CUstream, void **, void **);

struct Driver {
    pfn_cuModuleLoadData load = nullptr;
    pfn_cuModuleGetGlobal get_global = nullptr;
    pfn_cuModuleUnload unload = nullptr;
    pfn_cuModuleGetFunction get_function = nullptr;
    pfn_cuLinkCreate link_create = nullptr;
    pfn_cuLinkAddData link_add = nullptr;
    pfn_cuLinkComplete link_complete = nullptr;
    pfn_cuLinkDestroy link_destroy = nullptr;
    pfn_cuFuncSetAttribute func_set_attr = nullptr;
    pfn_cuFuncGetAttribute func_get_attr = nullptr;
    pfn_cuLaunchKernel launch = nullptr;
    bool ok = false;
};

bool resolve(const char *name, void **fn)
{
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q) != cudaSuccess) return false;
    return q == cudaDriverEntryPointSuccess && *fn != nullptr;
}

Driver &driver()
{
    static Driver d;
    if (!d.ok) {
        d.ok = resolve("cuModuleLoadData", (void **)&d.load) &&
               resolve("cuModuleGetGlobal", (void **)&d.get_global) &&
               resolve("cuModuleUnload", (void **)&d.unload) &&
               resolve("cuModuleGetFunction", (void **)&d.get_function) &&
               resolve("cuLinkCreate", (void **)&d.link_create) &&
               resolve("cuLinkAddData", (void **)&d.link_add) &&
               resolve("cuLinkComplete", (void **)&d.link_complete) &&
               resolve("cuLinkDestroy", (void **)&d.link_destroy) &&
               resolve("cuFuncSetAttribute", (void **)&d.func_set_attr) &&
               resolve("cuFuncGetAttribute", (void **)&d.func_get_attr) &&
               resolve("cuLaunchKernel", (void **)&d.launch);
    }
    return d;
}

/* The relocatable build of the executor (gpuos_exec_rdc.cubin), read from
 * the directory this library was loaded from. */
const std::vector<unsigned char> &exec_rdc_image()
{
    static std::vector<unsigned char> img;
    static bool tried = false;
    if (!tried) {
        tried = true;
        Dl_info info;
        if (dladdr((void *)&exec_rdc_image, &info) && info.dli_fname) {
            std::string path(info.dli_fname);
            const size_t cut = path.find_last_of('/');
            path = (cut == std::string::npos ? std::string(".") : path.substr(0, cut)) + "/gpuos_exec_rdc.cubin";
            FILE *f = fopen(path.c_str(), "rb");
            if (f) {
                fseek(f, 0, SEEK_END);
                const long n = ftell(f);
                fseek(f, 0, SEEK_SET);
                if (n > 0) {
                    img.resize((size_t)n);
                    if (fread(img.data(), 1, (size_t)n, f) != (size_t)n) img.clear();
                }
                fclose(f);
            }
        }
    }
    return img;
}

/* Link the relocatable executor with the given relocatable op objects into
 * one loadable image (driver JIT linker). Returns GPUOS_OK and the image. */
int link_images(const std::vector<std::vector<unsigned char>> &objs, std::vector<unsigned char> *out)
{
    Driver &drv = driver();
    if (!drv.ok) return GPUOS_ECUDA;
    const std::vector<unsigned char> &exe = exec_rdc_image();
    if (exe.empty()) return GPUOS_ECUDA;
    CUlinkState st = nullptr;
    if (drv.link_create(0, nullptr, nullptr, &st) != CUDA_SUCCESS) return GPUOS_ECUDA;
    int rc = GPUOS_OK;
    if (drv.link_add(st, CU_JIT_INPUT_CUBIN, (void *)exe.data(), exe.size(), "gpuos_exec", 0, nullptr, nullptr) !=
        CUDA_SUCCESS)
        rc = GPUOS_ECUDA;
    for (size_t i = 0; rc == GPUOS_OK && i < objs.size(); i++) {
        if (drv.link_add(st, CU_JIT_INPUT_CUBIN, (void *)objs[i].data(), objs[i].size(), "gpuos_op_module", 0,
                         nullptr, nullptr) != CUDA_SUCCESS)
            rc = GPUOS_EINVAL;
    }
    void *cubin = nullptr;
    size_t n = 0;
    if (rc == GPUOS_OK && drv.link_complete(st, &cubin, &n) != CUDA_SUCCESS) rc = GPUOS_EINVAL;
    if (rc == GPUOS_OK) out->assign((unsigned char *)cubin, (unsigned char *)cubin + n);
    drv.link_destroy(st);
    return rc;
}

uint64_t now_ns()
{
    timespec ts;
    clock_gettime(CLOCK_REALTIME, &ts);
    return (uint64_t)ts.tv_sec * 1000000000ull + (uint64_t)ts.tv_nsec;
}

/* A spin-wait step: a compiler barrier, so every poll reloads memory (no
 * architecture-specific hint, the same code on every host). */
inline void cpu_relax() { std::atomic_signal_fence(std::memory_order_seq_cst); }

template <typename T>
T load_acq(const T *p)
{
    return __atomic_load_n(p, __ATOMIC_ACQUIRE);
}
template <typename T>
void store_rel(T *p, T v)
{
    __atomic_store_n(p, v, __ATOMIC_RELEASE);
}

bool is_pow2(uint32_t x) { return x && !(x & (x - 1)); }

}  // namespace

struct gpuos_ctx {
    gpuos_config cfg;
    int device = 0;
    uint32_t N = 0, mask = 0, Q = 0;
    uint32_t blocks = 0, wpb = 0;
    /* host-visible (pinned or managed) */
    gpuos_desc *ring = nullptr;      /* host pointer */
    gpuos_desc *ring_dev = nullptr;  /* device view */
    gpuos_rec_dev *rec = nullptr;
    gpuos_rec_dev *rec_dev = nullptr;
    uint64_t *cw = nullptr; /* completion words, one per slot (host-visible) */
    uint64_t *cw_dev = nullptr;
    gpuos_hostctl *hctl = nullptr;
    gpuos_hostctl *hctl_dev = nullptr;
    bool ring_managed = false;
    /* device memory */
    gpuos_devdesc *mirror = nullptr;
    unsigned long long *tiles_done = nullptr;
    uint32_t *err = nullptr, *tile_ctr = nullptr;
    uint64_t *done_dev = nullptr;
    uint64_t *t_start = nullptr;
    unsigned long long *tq = nullptr;
    uint64_t *t_pub = nullptr;
    uint64_t *t_disp = nullptr;
    gpuos_devctl *dctl = nullptr;
    uint64_t *table = nullptr;     /* [2][GPUOS_MAX_OPS], pinned host memory */
    uint64_t *table_dev = nullptr; /* its device address */
    uint64_t *warp_stats = nullptr;
    uint32_t *version_stage = nullptr; /* pinned staging words (hand-off) */
    cudaStream_t exec_stream = nullptr, ctl_stream = nullptr;
    /* host state */
    bool mp = false;       /* multi-producer submission */
    std::mutex hmu;        /* (multi-producer) harvest state: low, hv, history, counts */
    uint64_t head = 0;     /* next ticket (reserved, with multiple producers) */
    uint64_t low = 0;      /* every ticket < low harvested */
    std::vector<uint64_t> commit_ns;
    std::vector<uint64_t> hv; /* per slot: ticket + 1 last harvested */
    gpuos_record *history = nullptr;
    uint64_t hist_base = 0, hist_cap = 0;
    uint64_t n_completed = 0, n_errors = 0;
    uint64_t host_wait_ns = 0; /* submitters' time waiting for a free slot */
    uint64_t pending_errors = 0; /* errors harvested since the last sync report */
    /* operator table shadow, and what each entry is bound to (a built-in op,
     * or a `__device__` variable of a loaded module holding the function's
     * address): function addresses are valid only inside one loaded module,
     * so a relaunch from a newly linked module rebuilds the table from these */
    uint64_t table_host[2][GPUOS_MAX_OPS];
    struct Binding {
        int builtin = -1; /* built-in op id, or -1 */
        std::string sym;  /* module symbol, when builtin < 0 */
    };
    Binding binding[2][GPUOS_MAX_OPS];
    bool user_registered[GPUOS_MAX_OPS];
    uint32_t version = 0;
    uint64_t flip_head = 0; /* head when the current version was published */
    struct Module {
        uint64_t hash;
        std::vector<unsigned char> bytes;
    };
    std::vector<Module> modules;  /* op objects linked into the executor */
    CUmodule linked = nullptr;    /* executor + op objects, when modules exist */
    CUfunction linked_exec = nullptr;
    uint32_t regs = 0, smem = 0;
    gpuos_exec_params params;
    uint32_t n_handoffs = 0; /* executor relaunches that took in a new module */
    uint64_t handoff_link_ns = 0, handoff_down_ns = 0; /* of the last one */
    bool accepting = false; /* submissions allowed (until stop) */
    bool launched = false;  /* executor kernel launched */
    bool running = false;   /* executor believed resident */
};

/* Host activity for the executor's idle watchdog: the host clock in units
 * of 2^20 ns (about a millisecond), stored only when it has moved on. The
 * device polls this line, so every store is an invalidation across
 * NVLink-C2C, and several producer threads would contend for it; one store
 * a millisecond is plenty for a watchdog counted in seconds. */
static inline void heartbeat(gpuos_ctx *c)
{
    const uint64_t ms = now_ns() >> 20;
    if (__atomic_load_n(&c->hctl->heartbeat, __ATOMIC_RELAXED) != ms)
        __atomic_store_n(&c->hctl->heartbeat, ms, __ATOMIC_RELAXED);
}

static inline uint64_t head_of(gpuos_ctx *c) { return __atomic_load_n(&c->head, __ATOMIC_ACQUIRE); }

/* The harvest state's lock, taken only with multiple producers. */
struct HarvestLock {
    std::mutex *m;
    explicit HarvestLock(gpuos_ctx *c) : m(c->mp ? &c->hmu : nullptr)
    {
        if (m) m->lock();
    }
    ~HarvestLock()
    {
        if (m) m->unlock();
    }
};

extern "C" {

uint64_t gpuos_host_now_ns(void) { return now_ns(); }

const char *gpuos_strerror(int code, int is_status)
{
    if (is_status) {
        switch (code) {
        case GPUOS_ST_OK: return "ok";
        case GPUOS_ST_BAD_OP: return "bad op id or empty table entry";
        case GPUOS_ST_BAD_ARGS: return "dims, position or length out of range";
        case GPUOS_ST_DEP_TIMEOUT: return "dependency or fence wait timed out";
        case GPUOS_ST_ABORTED: return "executor was leaving";
        case GPUOS_ST_BAD_DESC: return "ring slot did not hold the expected ticket";
        case GPUOS_ST_COPY_TIMEOUT: return "a staging copy did not complete within its bound";
        default: return "unknown device status";
        }
    }
    switch (code) {
    case GPUOS_OK: return "ok";
    case GPUOS_EINVAL: return "invalid argument";
    case GPUOS_EAGAIN: return "ring full (timed out waiting for a slot)";
    case GPUOS_ETIMEDOUT: return "timed out";
    case GPUOS_EDEVICE: return "a descriptor completed with a device error status";
    case GPUOS_ECUDA: return "CUDA call failed";
    case GPUOS_ESTOPPED: return "executor is not running";
    case GPUOS_ENOMEM: return "out of memory";
    case GPUOS_EBUSY: return "not allowed while the executor is resident (load modules before gpuos_start)";
    case GPUOS_ETOOBIG: return "sizes exceed the fixed scratch of gpuos_sdpa_noalloc (B*H <= 256, Lmax <= 4096)";
    case GPUOS_ECOMPILE: return "operator source did not compile (see the compile log)";
    default: return "unknown error";
    }
}

void gpuos_default_config(gpuos_config *c)
{
    memset(c, 0, sizeof(*c));
    c->ring_entries = 8192;
    c->warps_per_block = 12;
    c->blocks = 0;
    c->backoff_min_ns = 32;
    c->backoff_max_ns = 8000;
    c->spin_polls = 4096;
    c->idle_exit_ms = 10000;
    c->dep_timeout_ms = 5000;
    c->ring_in_device_mem = 0;
    c->device = 0;
    c->exit_after = 0;
    c->tq_entries = 0; /* sized from ring_entries */
    c->stage_bytes = 16384;
}

size_t gpuos_sdpa_workspace_bytes(uint32_t B, uint32_t H, uint32_t D, uint32_t Lmax)
{
    /* the host splits keys into chunks of GPUOS_SDPA_CHUNK_MIN rows at the finest */
    uint64_t nch = (Lmax + GPUOS_SDPA_CHUNK_MIN - 1) / GPUOS_SDPA_CHUNK_MIN;
    if (nch == 0) nch = 1;
    (void)D; /* partials hold 132 floats {m, l, 2 pad, acc[128]}; D is fixed at 128 */
    const uint64_t ctr = ((uint64_t)B * H + 3u) & ~3ull;
    return (size_t)(4ull * ctr + 4ull * B * H * nch * 132ull);
}

static uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
static bool al16(uint64_t p) { return (p & 15u) == 0; }

/* Element-wise tiles: the smallest power of two >= n / GPUOS_EW_SPLIT, kept
 * within [the op's smallest tile, the largest tile]. add/mul/ReLU ops up to
 * 16,384 elements stay one tile and larger ones take tiles of 16,384 (fp32)
 * or up to 32,768 (bf16): a tile carries about 6 us of fixed warp time
 * (claim, descriptor read, completion counter, dependency wait) against
 * 5-7 us of copying, so fewer, larger tiles raise what the worker warps
 * sustain (measured on the variable-shape stream from a pre-filled ring:
 * 40.5 -> 49.4 M descriptors/s with 4,096-element tiles -> 16,384; large
 * ops 0.89 -> 0.95 of the copy peak). A free GELU takes the same tiles; a
 * GELU with a dependency splits down to 1,024 elements (gelu_tile_min).
 * The device recovers the tile size from n and ntiles alone
 * (round_up(ceil(n / ntiles), 256)). */
static_assert((GPUOS_EW_TILE_MIN & (GPUOS_EW_TILE_MIN - 1)) == 0 && (GPUOS_GELU_TILE_MIN & (GPUOS_GELU_TILE_MIN - 1)) == 0 &&
                  (GPUOS_GELU_DEP_TILE_MIN & (GPUOS_GELU_DEP_TILE_MIN - 1)) == 0 &&
                  (GPUOS_EW_TILE_F32 & (GPUOS_EW_TILE_F32 - 1)) == 0 &&
                  (GPUOS_EW_TILE_BF16 & (GPUOS_EW_TILE_BF16 - 1)) == 0,
              "element-wise tile sizes are powers of two");
/* The tile: the smallest of tile_min, 2 tile_min, 4 tile_min, ... that cuts
 * n into at most GPUOS_EW_SPLIT tiles, capped at tile_max. With powers of
 * two that is the power of two at or above ceil(n / SPLIT), clamped to
 * [tile_min, tile_max]: computed without a loop (the descriptor mix makes a
 * data-dependent loop a branch the host mispredicts). */
static uint64_t ew_tiles(uint64_t n, uint64_t tile_min, uint64_t tile_max)
{
    const uint64_t lo = tile_min < tile_max ? tile_min : tile_max;
    const uint64_t need = (n + GPUOS_EW_SPLIT - 1) / GPUOS_EW_SPLIT;
    const uint64_t p2 = need <= 1 ? 1 : 2ull << (63 - __builtin_clzll(need - 1));
    uint64_t te = p2 > lo ? p2 : lo;
    te = te < tile_max ? te : tile_max;
    return (n + te - 1) >> __builtin_ctzll(te);
}

/* A GELU that waits on another descriptor sits on a dependency chain, where
 * its latency adds up: it keeps the finer split (measured on the mixed
 * pipeline, whose every op has a dependency: 1,024-element tiles 129.4 K
 * ops/s, 2,048 127.5 K); a free GELU only needs throughput, which fewer,
 * larger tiles serve better (variable-shape stream, free GELUs from 2,048 /
 * 4,096 / 8,192 / 16,384 elements: 49.2-50.8 / 51.6-53.0 / 55.1 / 55.8 M
 * descriptors/s, each step measured against the one before on one box;
 * the mixed pipeline unchanged). */
static uint64_t gelu_tile_min(const gpuos_desc *d)
{
    return (d->dep[0] | d->dep[1]) ? GPUOS_GELU_DEP_TILE_MIN : GPUOS_GELU_TILE_MIN;
}

/* Decode-attention chunks: every (b, h) pair's keys are cut into at most
 * floor(GPUOS_SDPA_SPLIT / (B * H)) chunks (at least one) of equal length,
 * a multiple of 32 rows: the op has at most GPUOS_SDPA_SPLIT tiles (or B * H),
 * all of which the default executor runs at once. A second, partial wave of
 * tiles would leave most warps idle while it runs. The device recovers the
 * chunk length from Lmax and ntiles: round_up(ceil(Lmax / nchunks), 32),
 * which is at most the length chosen here, with no chunk starting past
 * Lmax. */
static uint64_t sdpa_chunks(uint64_t BH, uint64_t Lmax)
{
    const uint64_t want = BH < GPUOS_SDPA_SPLIT ? GPUOS_SDPA_SPLIT / BH : 1;
    uint64_t ch = (ceil_div(Lmax, want) + 31) & ~31ull;
    if (ch < GPUOS_SDPA_CHUNK_MIN) ch = GPUOS_SDPA_CHUNK_MIN;
    return ceil_div(Lmax, ch);
}

/* Host-side validation (the page's "bounds checking") and tiling rule. */
static int validate_and_tile(const gpuos_desc *d, uint32_t *ntiles_out, bool user_op_known)
{
    const uint32_t *m = d->dims;
    uint64_t nt = 1;
    /* element-wise ops, the bulk of a throughput stream: the same checks and
     * tiling as the general path below, with the conditions combined into
     * one branch (the op mix would make each its own mispredicted branch) */
    if ((uint32_t)d->op_id - GPUOS_OP_ADD < 4u) {
        const uint32_t op = d->op_id;
        const bool f32 = d->dtype == GPUOS_F32;
        const bool bin = op <= GPUOS_OP_MUL;
        const bool bad = (!f32 && d->dtype != GPUOS_BF16) |
                         (m[0] != 0 && ((d->a == 0) | (d->out == 0) | (bin & (d->b == 0)))) |
                         ((d->flags & ~(GPUOS_FLAG_FENCE | GPUOS_FLAG_DEP_REL)) != 0);
        nt = ew_tiles(m[0], op == GPUOS_OP_GELU ? gelu_tile_min(d) : GPUOS_EW_TILE_MIN,
                      f32 ? GPUOS_EW_TILE_F32 : GPUOS_EW_TILE_BF16);
        nt += (nt == 0);
        if (bad | (nt > GPUOS_TILE_MAX)) return GPUOS_EINVAL;
        *ntiles_out = (uint32_t)nt;
        return GPUOS_OK;
    }
    if (d->op_id >= GPUOS_MAX_OPS) return GPUOS_EINVAL;
    switch (d->op_id) {
    case GPUOS_OP_NOP: nt = 1; break;
    case GPUOS_OP_ADD:
    case GPUOS_OP_MUL:
    case GPUOS_OP_RELU:
    case GPUOS_OP_GELU: {
        if (d->dtype != GPUOS_F32 && d->dtype != GPUOS_BF16) return GPUOS_EINVAL;
        const bool bin = d->op_id == GPUOS_OP_ADD || d->op_id == GPUOS_OP_MUL;
        if (m[0] && (!d->a || !d->out || (bin && !d->b))) return GPUOS_EINVAL;
        nt = ew_tiles(m[0], d->op_id == GPUOS_OP_GELU ? gelu_tile_min(d) : GPUOS_EW_TILE_MIN,
                      d->dtype == GPUOS_F32 ? GPUOS_EW_TILE_F32 : GPUOS_EW_TILE_BF16);
        break;
    }
    case GPUOS_OP_SOFTMAX:
    case GPUOS_OP_LAYERNORM:
    case GPUOS_OP_ROWSUM:
    case GPUOS_OP_ROWMAX:
    case GPUOS_OP_ROWMIN:
        if (d->dtype != GPUOS_BF16) return GPUOS_EINVAL;
        if (m[0] && (m[1] == 0 || !d->a || !d->out)) return GPUOS_EINVAL;
        if (m[0] && d->op_id == GPUOS_OP_LAYERNORM && (!d->b || !d->aux0)) return GPUOS_EINVAL;
        nt = m[0];
        break;
    case GPUOS_OP_ROPE:
        if (m[0] && (!d->a || !d->b || !d->aux0 || m[1] == 0 || m[2] == 0 || (m[2] & 1) || m[2] > 256))
            return GPUOS_EINVAL;
        nt = (uint64_t)m[0] * ceil_div(m[1], GPUOS_HEAD_GROUP);
        break;
    case GPUOS_OP_KV_WRITE:
        if (m[0] && (!d->a || !d->b || !d->aux0 || !d->out || !d->aux1 || m[1] == 0 || m[2] == 0 || m[3] == 0))
            return GPUOS_EINVAL;
        nt = (uint64_t)m[0] * ceil_div(m[1], GPUOS_HEAD_GROUP);
        break;
    case GPUOS_OP_SDPA:
        if (m[0]) {
            if (!d->a || !d->b || !d->aux0 || !d->aux1 || !d->out || !d->aux2) return GPUOS_EINVAL;
            if (m[1] == 0 || m[2] != 128 || m[3] == 0 || m[4] == 0 || m[4] > m[3]) return GPUOS_EINVAL;
            if ((uint64_t)m[5] < (uint64_t)m[0] * m[1]) return GPUOS_EINVAL;
            if (!al16(d->a) || !al16(d->b) || !al16(d->aux1) || !al16(d->out) || !al16(d->aux2)) return GPUOS_EINVAL;
        }
        nt = (uint64_t)m[0] * m[1] * sdpa_chunks((uint64_t)m[0] * m[1], m[4]);
        break;
    case GPUOS_OP_VECMAT:
        if (m[1] && (!d->a || !d->b || !d->out || m[0] == 0)) return GPUOS_EINVAL;
        nt = ceil_div(m[1], GPUOS_VM_COLS);
        break;
    default:
        if (d->op_id < GPUOS_OP_USER_FIRST && d->op_id >= GPUOS_OP_BUILTIN_COUNT) return GPUOS_EINVAL;
        if (!user_op_known) return GPUOS_EINVAL;
        nt = d->ntiles;
        break;
    }
    if (d->flags & ~(GPUOS_FLAG_FENCE | GPUOS_FLAG_DEP_REL)) return GPUOS_EINVAL;
    if (nt == 0) nt = 1; /* an empty op still waits for its dependencies */
    if (nt > GPUOS_TILE_MAX) return GPUOS_EINVAL;
    *ntiles_out = (uint32_t)nt;
    return GPUOS_OK;
}

int gpuos_op_ntiles(const gpuos_desc *d, uint32_t *ntiles)
{
    if (!d || !ntiles) return GPUOS_EINVAL;
    return validate_and_tile(d, ntiles, true);
}

static void free_all(gpuos_ctx *c)
{
    if (c->linked && driver().ok) driver().unload(c->linked);
    c->linked = nullptr;
    c->modules.clear();
    if (c->ring) {
        if (c->ring_managed) cudaFree(c->ring);
        else cudaFreeHost(c->ring);
    }
    if (c->rec) cudaFreeHost(c->rec);
    if (c->cw) cudaFreeHost(c->cw);
    if (c->hctl) cudaFreeHost(c->hctl);
    if (c->version_stage) cudaFreeHost(c->version_stage);
    cudaFree(c->mirror);
    cudaFree(c->tiles_done);
    cudaFree(c->err);
    cudaFree(c->tile_ctr);
    cudaFree(c->done_dev);
    cudaFree(c->t_start);
    cudaFree(c->t_pub);
    cudaFree(c->t_disp);
    cudaFree(c->tq);
    cudaFree(c->dctl);
    if (c->table) cudaFreeHost(c->table);
    cudaFree(c->warp_stats);
    if (c->exec_stream) cudaStreamDestroy(c->exec_stream);
    if (c->ctl_stream) cudaStreamDestroy(c->ctl_stream);
    delete c;
}

/* The executor kernel has ended (normally or with an error). */
static bool executor_gone(gpuos_ctx *c)
{
    const cudaError_t q = cudaStreamQuery(c->exec_stream);
    if (q == cudaErrorNotReady) return false;
    if (q != cudaSuccess || getenv("GPUOS_DEBUG"))
        fprintf(stderr, "gpuos: executor ended (%s), state=%u exit_reason=%u sequenced=%llu\n",
                cudaGetErrorString(q), c->hctl->state, c->hctl->exit_reason,
                (unsigned long long)c->hctl->sequenced);
    return true;
}

int gpuos_init(const gpuos_config *cfg_in, gpuos_ctx **out)
{
    if (!out) return GPUOS_EINVAL;
    *out = nullptr;
    gpuos_config cfg;
    if (cfg_in) cfg = *cfg_in;
    else gpuos_default_config(&cfg);
    if (!is_pow2(cfg.ring_entries) || cfg.ring_entries < 64 || cfg.ring_entries > 65536) return GPUOS_EINVAL;
    if (cfg.warps_per_block < 2 || cfg.warps_per_block > GPUOS_MAX_WPB) return GPUOS_EINVAL;
    /* the work queue must hold more than GPUOS_HELPERS entries per ring slot
     * (0 = the smallest such power of two) */
    if (cfg.tq_entries == 0 && cfg.ring_entries <= 65536) cfg.tq_entries = 2u * GPUOS_HELPERS * cfg.ring_entries;
    if (!is_pow2(cfg.tq_entries) || cfg.tq_entries > GPUOS_TQ_MAX ||
        (uint64_t)cfg.tq_entries <= (uint64_t)GPUOS_HELPERS * cfg.ring_entries)
        return GPUOS_EINVAL;
    if (cfg.backoff_min_ns == 0 || cfg.backoff_max_ns < cfg.backoff_min_ns) return GPUOS_EINVAL;
    if ((cfg.stage_bytes & 1023u) || cfg.stage_bytes > 24576u) return GPUOS_EINVAL;
    if (cfg.multi_producer > 1u) return GPUOS_EINVAL;
    if (cfg.sequencers > GPUOS_MAX_SEQ) return GPUOS_EINVAL;
    /* every warp's staging region and the executor's static shared memory
     * (descriptor copies, the sequencer's table copy, tile profiles) must fit
     * the 227 KB a block can hold */
    if (gpuos_dev_dyn_smem(cfg.warps_per_block, cfg.stage_bytes) + GPUOS_EXEC_STATIC_SMEM > 232448u) return GPUOS_EINVAL;

    gpuos_ctx *c = new (std::nothrow) gpuos_ctx();
    if (!c) return GPUOS_ENOMEM;
    c->cfg = cfg;
    c->mp = cfg.multi_producer != 0;
    c->device = cfg.device;
    c->N = cfg.ring_entries;
    c->mask = c->N - 1;
    c->Q = cfg.tq_entries;
    memset(c->table_host, 0, sizeof(c->table_host));
    memset(c->user_registered, 0, sizeof(c->user_registered));
#define CK(x)                                                                                       \
    do {                                                                                            \
        cudaError_t e_ = (x);                                                                       \
        if (e_ != cudaSuccess) {                                                                    \
            fprintf(stderr, "gpuos: %s failed: %s\n", #x, cudaGetErrorString(e_));                  \
            free_all(c);                                                                            \
            return e_ == cudaErrorMemoryAllocation ? GPUOS_ENOMEM : GPUOS_ECUDA;                    \
        }                                                                                           \
    } while (0)
    CK(cudaSetDevice(c->device));
    int sms = 0;
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, c->device));
    c->blocks = cfg.blocks ? cfg.blocks : (uint32_t)sms;
    c->wpb = cfg.warps_per_block;
    /* sequencers (warp 0 of blocks 0 .. S-1, SMs without workers): four on a
     * large grid, fewer on a small one, one with a single block */
    if (cfg.sequencers == 0) cfg.sequencers = c->blocks >= 32 ? 4u : (c->blocks >= 16 ? 2u : 1u);
    if ((c->blocks == 1 && cfg.sequencers != 1) || (c->blocks > 1 && cfg.sequencers >= c->blocks)) {
        free_all(c);
        return GPUOS_EINVAL;
    }
    c->cfg.sequencers = cfg.sequencers;
    if (gpuos_dev_preload() != 0) {
        free_all(c);
        return GPUOS_ECUDA;
    }
    gpuos_dev_executor_attrs(&c->regs, &c->smem);
    CK(cudaStreamCreateWithFlags(&c->exec_stream, cudaStreamNonBlocking));
    CK(cudaStreamCreateWithFlags(&c->ctl_stream, cudaStreamNonBlocking));

    const size_t ring_bytes = (size_t)c->N * sizeof(gpuos_desc);
    if (cfg.ring_in_device_mem) {
        int direct = 0;
        CK(cudaDeviceGetAttribute(&direct, cudaDevAttrDirectManagedMemAccessFromHost, c->device));
        if (!direct) {
            free_all(c);
            return GPUOS_EINVAL;
        }
        CK(cudaMallocManaged((void **)&c->ring, ring_bytes, cudaMemAttachGlobal));
        c->ring_managed = true;
        cudaMemLocation loc;
        loc.type = cudaMemLocationTypeDevice;
        loc.id = c->device;
        CK(cudaMemAdvise(c->ring, ring_bytes, cudaMemAdviseSetPreferredLocation, loc));
        cudaMemLocation hl;
        hl.type = cudaMemLocationTypeHost;
        hl.id = 0;
        CK(cudaMemAdvise(c->ring, ring_bytes, cudaMemAdviseSetAccessedBy, hl));
        CK(cudaMemPrefetchAsync(c->ring, ring_bytes, loc, 0, c->ctl_stream));
        CK(cudaMemsetAsync(c->ring, 0, ring_bytes, c->ctl_stream));
        CK(cudaStreamSynchronize(c->ctl_stream));
        c->ring_dev = c->ring;
    } else {
        CK(cudaHostAlloc((void **)&c->ring, ring_bytes, cudaHostAllocMapped | cudaHostAllocPortable));
        memset(c->ring, 0, ring_bytes);
        CK(cudaHostGetDevicePointer((void **)&c->ring_dev, c->ring, 0));
    }
    CK(cudaHostAlloc((void **)&c->rec, (size_t)c->N * sizeof(gpuos_rec_dev), cudaHostAllocMapped | cudaHostAllocPortable));
    memset(c->rec, 0, (size_t)c->N * sizeof(gpuos_rec_dev));
    CK(cudaHostGetDevicePointer((void **)&c->rec_dev, c->rec, 0));
    CK(cudaHostAlloc((void **)&c->cw, (size_t)c->N * sizeof(uint64_t), cudaHostAllocMapped | cudaHostAllocPortable));
    memset(c->cw, 0, (size_t)c->N * sizeof(uint64_t));
    CK(cudaHostGetDevicePointer((void **)&c->cw_dev, c->cw, 0));
    CK(cudaHostAlloc((void **)&c->hctl, sizeof(gpuos_hostctl), cudaHostAllocMapped | cudaHostAllocPortable));
    memset(c->hctl, 0, sizeof(gpuos_hostctl));
    CK(cudaHostGetDevicePointer((void **)&c->hctl_dev, c->hctl, 0));
    CK(cudaHostAlloc((void **)&c->version_stage, 64, cudaHostAllocPortable));
    /* the operator table: both slots in pinned host memory, written by the
     * host with plain stores and published by the version's store-release */
    CK(cudaHostAlloc((void **)&c->table, sizeof(c->table_host), cudaHostAllocMapped | cudaHostAllocPortable));
    CK(cudaHostGetDevicePointer((void **)&c->table_dev, c->table, 0));

    const uint32_t total_warps = c->blocks * c->wpb;
    CK(cudaMalloc((void **)&c->mirror, (size_t)c->N * sizeof(gpuos_devdesc)));
    CK(cudaMalloc((void **)&c->tiles_done, (size_t)c->N * 8));
    CK(cudaMalloc((void **)&c->err, (size_t)c->N * 4));
    CK(cudaMalloc((void **)&c->tile_ctr, (size_t)c->N * 4));
    CK(cudaMalloc((void **)&c->done_dev, (size_t)c->N * 8));
    CK(cudaMalloc((void **)&c->t_start, (size_t)c->N * 8));
    CK(cudaMalloc((void **)&c->tq, (size_t)c->Q * 8));
    CK(cudaMalloc((void **)&c->t_pub, (size_t)c->N * 8));
    CK(cudaMalloc((void **)&c->t_disp, (size_t)c->N * 8));
    CK(cudaMalloc((void **)&c->dctl, sizeof(gpuos_devctl)));
    CK(cudaMalloc((void **)&c->warp_stats, (size_t)total_warps * GPUOS_WS_N * 8));
    CK(cudaMemsetAsync(c->mirror, 0, (size_t)c->N * sizeof(gpuos_devdesc), c->ctl_stream));
    CK(cudaMemsetAsync(c->tiles_done, 0, (size_t)c->N * 8, c->ctl_stream));
    CK(cudaMemsetAsync(c->err, 0, (size_t)c->N * 4, c->ctl_stream));
    CK(cudaMemsetAsync(c->tile_ctr, 0, (size_t)c->N * 4, c->ctl_stream));
    CK(cudaMemsetAsync(c->done_dev, 0, (size_t)c->N * 8, c->ctl_stream));
    CK(cudaMemsetAsync(c->t_start, 0, (size_t)c->N * 8, c->ctl_stream));
    CK(cudaMemsetAsync(c->tq, 0, (size_t)c->Q * 8, c->ctl_stream));
    CK(cudaMemsetAsync(c->t_pub, 0, (size_t)c->N * 8, c->ctl_stream));
    CK(cudaMemsetAsync(c->t_disp, 0, (size_t)c->N * 8, c->ctl_stream));
    CK(cudaMemsetAsync(c->dctl, 0, sizeof(gpuos_devctl), c->ctl_stream));
    CK(cudaMemsetAsync(c->warp_stats, 0, (size_t)total_warps * GPUOS_WS_N * 8, c->ctl_stream));

    gpuos_op_fn builtin[GPUOS_OP_BUILTIN_COUNT];
    if (gpuos_dev_builtin_table(builtin, GPUOS_OP_BUILTIN_COUNT) != 0) {
        free_all(c);
        return GPUOS_ECUDA;
    }
    for (int s = 0; s < 2; s++)
        for (int i = 0; i < GPUOS_OP_BUILTIN_COUNT; i++) {
            c->table_host[s][i] = (uint64_t)(uintptr_t)builtin[i];
            c->binding[s][i].builtin = i;
        }
    memcpy(c->table, c->table_host, sizeof(c->table_host));
    CK(cudaStreamSynchronize(c->ctl_stream));

    c->commit_ns.assign(c->N, 0);
    c->hv.assign(c->N, 0);

    gpuos_exec_params &p = c->params;
    memset(&p, 0, sizeof(p));
    p.ring = c->ring_dev;
    p.rec = c->rec_dev;
    p.done_host = c->cw_dev;
    p.hctl = c->hctl_dev;
    p.mirror = c->mirror;
    p.tiles_done = c->tiles_done;
    p.err = c->err;
    p.tile_ctr = c->tile_ctr;
    p.done_dev = c->done_dev;
    p.t_start = c->t_start;
    p.t_pub = c->t_pub;
    p.t_disp = c->t_disp;
    p.tq = c->tq;
    p.dctl = c->dctl;
    p.table = c->table_dev;
    p.warp_stats = c->warp_stats;
    p.ring_mask = c->mask;
    p.tq_mask = c->Q - 1;
    p.backoff_min_ns = cfg.backoff_min_ns;
    p.backoff_max_ns = cfg.backoff_max_ns;
    p.spin_polls = cfg.spin_polls;
    p.stage_bytes = cfg.stage_bytes;
    /* worker warps: block 0 holds only the sequencers (when there are others) */
    p.sequencers = cfg.sequencers;
    p.workers = c->blocks > 1 ? (c->blocks - cfg.sequencers) * c->wpb : c->wpb - 1;
    p.idle_exit_ns = (uint64_t)cfg.idle_exit_ms * 1000000ull;
    p.dep_timeout_ns = (uint64_t)(cfg.dep_timeout_ms ? cfg.dep_timeout_ms : 5000) * 1000000ull;
    p.exit_after = cfg.exit_after;
    c->accepting = true;
    if (!cfg.deferred_start) {
        const int rc = gpuos_start(c);
        if (rc != GPUOS_OK) {
            free_all(c);
            return rc;
        }
    }
    *out = c;
    return GPUOS_OK;
#undef CK
}

/* With op modules loaded: link them with the relocatable executor, load the
 * result, take the built-in table from it (function pointers are valid only
 * inside the module that holds the code) and launch its executor. */
static int launch_linked(gpuos_ctx *c, const std::vector<unsigned char> *prelinked)
{
    Driver &drv = driver();
    std::vector<unsigned char> img;
    if (prelinked) {
        img = *prelinked;
    } else {
        std::vector<std::vector<unsigned char>> objs;
        for (auto &m : c->modules) objs.push_back(m.bytes);
        const int rc = link_images(objs, &img);
        if (rc) return rc;
    }
    if (drv.load(&c->linked, img.data()) != CUDA_SUCCESS) return GPUOS_ECUDA;
    CUdeviceptr tab = 0;
    size_t tsz = 0;
    if (drv.get_global(&tab, &tsz, c->linked, "g_builtin_ops") != CUDA_SUCCESS ||
        tsz != GPUOS_OP_BUILTIN_COUNT * sizeof(gpuos_op_fn))
        return GPUOS_ECUDA;
    uint64_t builtin[GPUOS_OP_BUILTIN_COUNT];
    if (cudaMemcpy(builtin, (const void *)tab, sizeof(builtin), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GPUOS_ECUDA;
    /* both table slots from the bindings, with this module's addresses */
    for (int sl = 0; sl < 2; sl++)
        for (int i = 0; i < GPUOS_MAX_OPS; i++) {
            const gpuos_ctx::Binding &b = c->binding[sl][i];
            uint64_t v = 0;
            if (b.builtin >= 0) {
                v = builtin[b.builtin];
            } else if (!b.sym.empty()) {
                CUdeviceptr gp = 0;
                size_t gsz = 0;
                if (drv.get_global(&gp, &gsz, c->linked, b.sym.c_str()) != CUDA_SUCCESS || gsz != sizeof(uint64_t) ||
                    cudaMemcpy(&v, (const void *)gp, 8, cudaMemcpyDeviceToHost) != cudaSuccess)
                    return GPUOS_ECUDA;
            }
            c->table_host[sl][i] = v;
        }
    /* no executor runs here (not yet launched, or the old one has left) */
    memcpy(c->table, c->table_host, sizeof(c->table_host));
    if (drv.get_function(&c->linked_exec, c->linked, "gpuos_executor_kernel") != CUDA_SUCCESS) return GPUOS_ECUDA;
    /* every function of the executor and of the op modules was compiled with
     * at most GPUOS_MAX_REGS registers; the linked kernel must hold that many
     * per thread, or an indirect call could use registers it does not own */
    int regs = 0;
    if (drv.func_get_attr(&regs, CU_FUNC_ATTRIBUTE_NUM_REGS, c->linked_exec) != CUDA_SUCCESS) return GPUOS_ECUDA;
    if (regs < GPUOS_MAX_REGS) {
        fprintf(stderr, "gpuos: linked executor holds %d registers per thread, below %d\n", regs, GPUOS_MAX_REGS);
        return GPUOS_EINVAL;
    }
    c->regs = (uint32_t)regs;
    const uint32_t dyn = gpuos_dev_dyn_smem(c->wpb, c->params.stage_bytes);
    if (drv.func_set_attr(c->linked_exec, CU_FUNC_ATTRIBUTE_MAX_DYNAMIC_SHARED_SIZE_BYTES, (int)dyn) != CUDA_SUCCESS)
        return GPUOS_ECUDA;
    void *args[] = {&c->params};
    if (drv.launch(c->linked_exec, c->blocks, 1, 1, c->wpb * 32, 1, 1, dyn, (CUstream)c->exec_stream, args,
                   nullptr) != CUDA_SUCCESS)
        return GPUOS_ECUDA;
    return GPUOS_OK;
}

int gpuos_start(gpuos_ctx *c)
{
    if (!c || c->launched) return GPUOS_EINVAL;
    if (cudaSetDevice(c->device) != cudaSuccess) return GPUOS_ECUDA;
    heartbeat(c);
    if (!c->modules.empty()) {
        const int rc = launch_linked(c, nullptr);
        if (rc) {
            fprintf(stderr, "gpuos: linked executor launch failed (%d)\n", rc);
            return rc;
        }
    } else if (gpuos_dev_launch_executor(&c->params, c->blocks, c->wpb, c->exec_stream) != 0) {
        fprintf(stderr, "gpuos: executor launch failed: %s\n", cudaGetErrorString(cudaGetLastError()));
        return GPUOS_ECUDA;
    }
    c->launched = true;
    /* wait (bounded) for the sequencer to report that it runs */
    const uint64_t t0 = now_ns();
    while (load_acq(&c->hctl->state) == 0u) {
        if (cudaStreamQuery(c->exec_stream) != cudaErrorNotReady || now_ns() - t0 > 10000000000ull) {
            fprintf(stderr, "gpuos: executor did not start\n");
            store_rel(&c->hctl->stop, 1u);
            return GPUOS_ECUDA;
        }
        cpu_relax();
    }
    c->running = true;
    return GPUOS_OK;
}

int gpuos_executor_stream(gpuos_ctx *c, void **stream)
{
    if (!c || !stream) return GPUOS_EINVAL;
    *stream = (void *)c->exec_stream;
    return GPUOS_OK;
}

/* ---- harvesting completion records ------------------------------------------ */
/* Ticket t's completion: the slot's completion word (ticket + 1, and a flag
 * for a nonzero status) frees the slot; the record (status, version,
 * timestamps) stays in its slot until ticket t + ring_entries completes, and
 * is read only when asked for (gpuos_query, the history). The word is a
 * quarter of the bytes and eight slots share a line, so the submitting
 * thread's check of a slot rarely misses on a line the device wrote. */
static bool is_done(gpuos_ctx *c, uint64_t t)
{
    return (load_acq(&c->cw[t & c->mask]) & GPUOS_DONE_TICKET_MASK) >= t + 1;
}

/* The record of a completed ticket whose slot has not been reused (the
 * caller's is_done(t) acquired it). */
static gpuos_record read_record(gpuos_ctx *c, uint64_t t)
{
    const uint32_t slot = (uint32_t)(t & c->mask);
    const gpuos_rec_dev *r = c->rec + slot;
    gpuos_record R;
    R.ticket = t;
    R.status = __atomic_load_n(&r->status, __ATOMIC_RELAXED);
    R.version = __atomic_load_n(&r->version, __ATOMIC_RELAXED);
    R.t_commit_host_ns = c->commit_ns[slot];
    R.t_dispatch_dev_ns = __atomic_load_n(&r->t_dispatch, __ATOMIC_RELAXED);
    R.t_publish_dev_ns = __atomic_load_n(&r->t_publish, __ATOMIC_RELAXED);
    R.t_start_dev_ns = __atomic_load_n(&r->t_start, __ATOMIC_RELAXED);
    R.t_done_dev_ns = __atomic_load_n(&r->t_done, __ATOMIC_RELAXED);
    return R;
}

/* Harvest completed ticket t (once; the caller's is_done(t) acquired it):
 * count it, note a failure, keep its record if the history covers it.
 * Counts it in n_completed, unless `tally` is given: then the caller adds
 * *tally later (several producers would otherwise contend for the counter
 * once per ticket). */
static void harvest_one(gpuos_ctx *c, uint64_t t, uint64_t *tally = nullptr)
{
    const uint32_t slot = (uint32_t)(t & c->mask);
    uint64_t seen = __atomic_load_n(&c->hv[slot], __ATOMIC_ACQUIRE);
    if (seen >= t + 1) return;
    /* read before the ticket is marked harvested: a producer reuses the
     * slot (and the device then rewrites word and record) only after that */
    const uint64_t w = __atomic_load_n(&c->cw[slot], __ATOMIC_RELAXED);
    const bool keep = c->history && t >= c->hist_base && t - c->hist_base < c->hist_cap;
    gpuos_record R;
    if (keep) R = read_record(c, t);
    /* one harvester per ticket: with several producers, a producer reusing
     * the slot and a sweeping thread may reach the same ticket together; a
     * single-producer context harvests from one thread */
    if (c->mp) {
        if (!__atomic_compare_exchange_n(&c->hv[slot], &seen, t + 1, false, __ATOMIC_ACQ_REL, __ATOMIC_ACQUIRE))
            return;
    } else {
        __atomic_store_n(&c->hv[slot], t + 1, __ATOMIC_RELAXED);
    }
    if (keep) c->history[t - c->hist_base] = R;
    if (tally)
        (*tally)++;
    else if (c->mp)
        __atomic_fetch_add(&c->n_completed, (uint64_t)1, __ATOMIC_RELAXED);
    else
        __atomic_store_n(&c->n_completed, __atomic_load_n(&c->n_completed, __ATOMIC_RELAXED) + 1, __ATOMIC_RELAXED);
    if (w & GPUOS_DONE_FAILED) {
        __atomic_fetch_add(&c->n_errors, (uint64_t)1, __ATOMIC_RELAXED);
        __atomic_fetch_add(&c->pending_errors, (uint64_t)1, __ATOMIC_RELAXED);
    }
}

static void sweep(gpuos_ctx *c)
{
    /* one producer: tickets older than head - N were harvested when their
     * slot was reused (it is reused only after they completed). Several
     * producers reserve tickets before their slots are free, so there every
     * ticket is checked */
    const uint64_t head = head_of(c);
    if (!c->mp && head > c->N && c->low < head - c->N) __atomic_store_n(&c->low, head - c->N, __ATOMIC_RELEASE);
    uint64_t low = c->low;
    while (low < head) {
        const uint32_t slot = (uint32_t)(low & c->mask);
        if (__atomic_load_n(&c->hv[slot], __ATOMIC_ACQUIRE) < low + 1) {
            if (!is_done(c, low)) break;
            harvest_one(c, low);
        }
        low++;
    }
    __atomic_store_n(&c->low, low, __ATOMIC_RELEASE);
}

/* Write a descriptor's body (everything before the commit word) into its
 * ring slot: the caller's words, with the library's fields (tile count,
 * resolved dependencies, flags the device reads, ticket) put in on the way,
 * in registers: patching a stack copy with narrow stores and reading it back
 * in wide pieces would stall on store forwarding. */
static inline void write_body(gpuos_desc *slot, const gpuos_desc *d, uint32_t nt, uint64_t dep0, uint64_t dep1,
                              uint64_t t)
{
    struct Head {
        uint16_t op_id;
        uint8_t dtype;
        uint8_t flags;
        uint32_t ntiles;
    } h = {d->op_id, d->dtype, (uint8_t)(d->flags & GPUOS_FLAG_FENCE), nt};
    static_assert(sizeof(Head) == 8 && offsetof(gpuos_desc, dep) == 8, "descriptor head is 8 bytes");
    static_assert(offsetof(gpuos_desc, ticket) == 14 * 8 && offsetof(gpuos_desc, seq) == 15 * 8,
                  "ticket and commit word are the last two words");
    uint64_t w0;
    memcpy(&w0, &h, 8);
    const uint64_t *src = reinterpret_cast<const uint64_t *>(d);
    uint64_t *dst = reinterpret_cast<uint64_t *>(slot);
    dst[0] = w0;
    dst[1] = dep0;
    dst[2] = dep1;
    for (int i = 3; i < 14; i++) dst[i] = src[i];
    dst[14] = t;
}

static int submit_one(gpuos_ctx *c, const gpuos_desc *d, uint64_t *ticket, uint32_t timeout_us)
{
    if (!c || !d) return GPUOS_EINVAL;
    if (!c->accepting || (c->launched && !c->running)) return GPUOS_ESTOPPED;
    if (!c->launched && c->head >= c->N) return GPUOS_EAGAIN; /* deferred: ring capacity */
    if (c->launched && __atomic_load_n(&c->hctl->state, __ATOMIC_RELAXED) == 2u) {
        c->running = false; /* the executor is leaving (stop or watchdog) */
        if (getenv("GPUOS_DEBUG"))
            fprintf(stderr,
                    "gpuos: submit refused, executor leaving: exit_reason=%u sequenced=%llu now=%llu active=%llu "
                    "idle_exit_ns=%llu\n",
                    c->hctl->exit_reason, (unsigned long long)c->hctl->sequenced,
                    (unsigned long long)c->hctl->exit_now, (unsigned long long)c->hctl->exit_active,
                    (unsigned long long)c->params.idle_exit_ns);
        return GPUOS_ESTOPPED;
    }
    uint32_t nt = 0;
    const bool user_known = d->op_id >= GPUOS_OP_USER_FIRST && c->user_registered[d->op_id];
    int rc = validate_and_tile(d, &nt, user_known);
    if (rc) return rc;
    const uint64_t t = c->head;
    uint64_t deps[2];
    for (int i = 0; i < 2; i++) {
        uint64_t v = d->dep[i];
        if (v && (d->flags & GPUOS_FLAG_DEP_REL)) {
            if (v > t) return GPUOS_EINVAL;
            v = t - v + 1; /* ticket + 1 of the descriptor v back */
        }
        if (v > t) return GPUOS_EINVAL; /* depends on itself or the future */
        deps[i] = v;
    }
    const uint32_t slot = (uint32_t)(t & c->mask);
    if (t >= c->N) {
        const uint64_t prev = t - c->N;
        if (!is_done(c, prev)) {
            const uint64_t t0 = now_ns();
            uint32_t spins = 0;
            while (!is_done(c, prev)) {
                if ((++spins & 1023u) == 0) {
                    heartbeat(c);
                    if (now_ns() - t0 > (uint64_t)timeout_us * 1000ull) return GPUOS_EAGAIN;
                    if (executor_gone(c)) {
                        c->running = false;
                        return GPUOS_ESTOPPED;
                    }
                }
                cpu_relax();
            }
            __atomic_fetch_add(&c->host_wait_ns, now_ns() - t0, __ATOMIC_RELAXED);
        }
        harvest_one(c, prev);
    }
    gpuos_desc *s = c->ring + slot;
    /* body (first 120 bytes), then the commit word with a store-release */
    write_body(s, d, nt, deps[0], deps[1], t);
    c->commit_ns[slot] = now_ns();
    store_rel(&s->seq, t + 1);
    c->head = t + 1;
    if ((t & 63u) == 0) heartbeat(c);
    if (ticket) *ticket = t;
    return GPUOS_OK;
}

/* Single producer, a run of descriptors. Up to GPUOS_COMMIT_RUN at a time:
 * each is validated and tiled, takes its slot (once the slot's previous
 * ticket has completed) and has its body written; then one release fence
 * and the commit words of the whole run. Every commit word still follows
 * its own body (the fence orders all of the run's bodies before any of its
 * commits), which is all the device's acquire relies on; the run shares one
 * host commit timestamp, taken before the fence (so at or before every
 * commit of the run). Stops at the first failure, after committing what was
 * written before it. */
#define GPUOS_COMMIT_RUN 64u
static int submit_run_spsc(gpuos_ctx *c, const gpuos_desc *d, uint32_t count, uint32_t *n_done, uint32_t timeout_us)
{
    if (!c->accepting || (c->launched && !c->running)) return GPUOS_ESTOPPED;
    if (c->launched && __atomic_load_n(&c->hctl->state, __ATOMIC_RELAXED) == 2u) {
        c->running = false;
        return GPUOS_ESTOPPED;
    }
    uint32_t done = 0;
    int rc = GPUOS_OK;
    while (done < count && rc == GPUOS_OK) {
        const uint32_t m = count - done < GPUOS_COMMIT_RUN ? count - done : GPUOS_COMMIT_RUN;
        const uint64_t t0 = c->head;
        uint32_t k = 0;
        for (; k < m; k++) {
            const gpuos_desc *di = d + done + k;
            const uint64_t t = t0 + k;
            if (!c->launched && t >= c->N) {
                rc = GPUOS_EAGAIN; /* deferred start: ring capacity */
                break;
            }
            uint32_t nt = 0;
            const bool user_known = di->op_id >= GPUOS_OP_USER_FIRST && c->user_registered[di->op_id];
            rc = validate_and_tile(di, &nt, user_known);
            if (rc) break;
            /* dependencies: an absolute ticket + 1 must be at most t, a
             * distance (DEP_REL) at most t as well (then t - v + 1 <= t) */
            uint64_t deps[2];
            bool dbad = false;
            const bool rel = (di->flags & GPUOS_FLAG_DEP_REL) != 0;
            for (int q = 0; q < 2; q++) {
                const uint64_t v = di->dep[q];
                dbad |= v > t;
                deps[q] = (rel && v) ? t - v + 1 : v;
            }
            if (dbad) {
                rc = GPUOS_EINVAL;
                break;
            }
            const uint32_t slot = (uint32_t)(t & c->mask);
            if (t >= c->N) {
                const uint64_t prev = t - c->N;
                if (!is_done(c, prev)) {
                    const uint64_t w0 = now_ns();
                    uint32_t spins = 0;
                    while (!is_done(c, prev)) {
                        if ((++spins & 1023u) == 0) {
                            heartbeat(c);
                            if (now_ns() - w0 > (uint64_t)timeout_us * 1000ull) {
                                rc = GPUOS_EAGAIN;
                                break;
                            }
                            if (executor_gone(c)) {
                                c->running = false;
                                rc = GPUOS_ESTOPPED;
                                break;
                            }
                        }
                        cpu_relax();
                    }
                    __atomic_fetch_add(&c->host_wait_ns, now_ns() - w0, __ATOMIC_RELAXED);
                    if (rc) break;
                }
                harvest_one(c, prev);
            }
            /* the body: the slot's previous descriptor completed, so the
             * device no longer reads it; nothing reads the new body before
             * its commit word */
            write_body(c->ring + slot, di, nt, deps[0], deps[1], t);
        }
        if (k) {
            const uint64_t stamp = now_ns();
            __atomic_thread_fence(__ATOMIC_RELEASE);
            for (uint32_t q = 0; q < k; q++) {
                const uint64_t t = t0 + q;
                const uint32_t slot = (uint32_t)(t & c->mask);
                c->commit_ns[slot] = stamp;
                __atomic_store_n(&c->ring[slot].seq, t + 1, __ATOMIC_RELAXED);
            }
            __atomic_store_n(&c->head, t0 + k, __ATOMIC_RELEASE);
            done += k;
        }
        heartbeat(c);
    }
    if (n_done) *n_done = done;
    return rc;
}

/* A waiting producer's spin step. Every 256 polls: the deadline (when one
 * is given), the heartbeat and, when the device has flagged that it is
 * leaving or 10 ms have passed, whether the executor kernel has ended (a
 * CUDA runtime query, which takes a lock the other producers would fight
 * over if it ran on every poll). After a few thousand polls the thread
 * yields its core: there may be more producer threads than cores. */
struct ProducerWait {
    uint64_t t0 = 0, last = 0;
    uint32_t spins = 0;
    int step(gpuos_ctx *c, uint64_t timeout_ns)
    {
        if ((++spins & 255u) != 0) {
            cpu_relax();
            return GPUOS_OK;
        }
        const uint64_t now = now_ns();
        if (t0 == 0) t0 = last = now;
        heartbeat(c);
        if (timeout_ns && now - t0 > timeout_ns) return GPUOS_EAGAIN;
        if (__atomic_load_n(&c->hctl->state, __ATOMIC_RELAXED) == 2u || now - last > 10000000ull) {
            last = now;
            if (executor_gone(c)) {
                c->running = false;
                return GPUOS_ESTOPPED;
            }
        }
        if (spins > 4096u) sched_yield();
        return GPUOS_OK;
    }
};

/* Multiple producers: validate every descriptor, wait (up to the timeout)
 * until the slot the batch's last ticket would take is free, reserve count
 * consecutive tickets with one atomic add, then write every body (each once
 * its slot is free: another producer may have taken the tickets counted on),
 * one release fence and the commit words. Each producer harvests the
 * records of the slots it reuses, so no lock is taken on this path. The
 * work queue hands out space in ticket order, which with these per-slot
 * waits keeps its wrap-around safe. */
static int submit_mp(gpuos_ctx *c, const gpuos_desc *d, uint32_t count, uint64_t *first_ticket,
                     uint32_t *n_done, uint32_t timeout_us)
{
    if (n_done) *n_done = 0;
    if (!c->launched) return GPUOS_EINVAL;
    if (!c->accepting || !c->running) return GPUOS_ESTOPPED;
    if (__atomic_load_n(&c->hctl->state, __ATOMIC_RELAXED) == 2u) {
        c->running = false;
        return GPUOS_ESTOPPED;
    }
    if (count == 0) return GPUOS_OK;
    if (count > c->N) return GPUOS_EINVAL;
    uint32_t nts_small[64];
    std::vector<uint32_t> nts_big;
    uint32_t *nts = nts_small;
    if (count > 64) {
        nts_big.resize(count);
        nts = nts_big.data();
    }
    const uint64_t h0 = head_of(c);
    for (uint32_t i = 0; i < count; i++) {
        const bool user_known = d[i].op_id >= GPUOS_OP_USER_FIRST && c->user_registered[d[i].op_id];
        int rc = validate_and_tile(d + i, &nts[i], user_known);
        if (rc) return rc;
        /* the ticket will be >= h0 + i, so these bounds hold for it */
        for (int k = 0; k < 2; k++)
            if (d[i].dep[k] > h0 + i) return GPUOS_EINVAL;
    }
    /* room: the slot of the last ticket the batch would take from the
     * current head is free */
    ProducerWait wt;
    while (true) {
        const uint64_t h = head_of(c);
        if (h + count <= c->N || is_done(c, h + count - 1 - c->N)) break;
        const int rc = wt.step(c, (uint64_t)timeout_us * 1000ull);
        if (rc) return rc;
    }
    if (wt.t0) __atomic_fetch_add(&c->host_wait_ns, now_ns() - wt.t0, __ATOMIC_RELAXED);
    const uint64_t t0 = __atomic_fetch_add(&c->head, (uint64_t)count, __ATOMIC_ACQ_REL);
    if (first_ticket) *first_ticket = t0;
    /* A reserved ticket is always committed (the executor takes tickets in
     * order): from here the waits have no deadline, only the executor's end. */
    uint64_t harvested = 0;
    ProducerWait ws;
    for (uint32_t i = 0; i < count; i++) {
        const uint64_t t = t0 + i;
        const uint32_t slot = (uint32_t)(t & c->mask);
        if (t >= c->N) {
            const uint64_t prev = t - c->N;
            while (!is_done(c, prev)) {
                const int rc = ws.step(c, 0);
                if (rc) return rc;
            }
            harvest_one(c, prev, &harvested); /* lock-free: one harvester per ticket */
        }
        uint64_t dv[2];
        for (int k = 0; k < 2; k++) {
            dv[k] = d[i].dep[k];
            if (dv[k] && (d[i].flags & GPUOS_FLAG_DEP_REL)) dv[k] = t - dv[k] + 1;
        }
        write_body(c->ring + slot, d + i, nts[i], dv[0], dv[1], t);
    }
    const uint64_t stamp = now_ns();
    __atomic_thread_fence(__ATOMIC_RELEASE);
    for (uint32_t i = 0; i < count; i++) {
        const uint64_t t = t0 + i;
        const uint32_t slot = (uint32_t)(t & c->mask);
        c->commit_ns[slot] = stamp;
        __atomic_store_n(&c->ring[slot].seq, t + 1, __ATOMIC_RELAXED);
    }
    if (n_done) *n_done = count;
    if (harvested) __atomic_fetch_add(&c->n_completed, harvested, __ATOMIC_RELAXED);
    if (ws.t0) __atomic_fetch_add(&c->host_wait_ns, now_ns() - ws.t0, __ATOMIC_RELAXED);
    heartbeat(c);
    return GPUOS_OK;
}

int gpuos_submit(gpuos_ctx *c, const gpuos_desc *d, uint64_t *ticket, uint32_t timeout_us)
{
    if (c && c->mp) {
        if (!d) return GPUOS_EINVAL;
        return submit_mp(c, d, 1, ticket, nullptr, timeout_us);
    }
    return submit_one(c, d, ticket, timeout_us);
}

int gpuos_submit_batch(gpuos_ctx *c, const gpuos_desc *d, uint32_t count, uint64_t *first_ticket,
                       uint32_t *n_done, uint32_t timeout_us)
{
    if (!c || (!d && count)) return GPUOS_EINVAL;
    if (c->mp) return submit_mp(c, d, count, first_ticket, n_done, timeout_us);
    if (first_ticket) *first_ticket = c->head;
    if (count == 0) {
        if (n_done) *n_done = 0;
        return GPUOS_OK;
    }
    if (count == 1) {
        const int rc = submit_one(c, d, nullptr, timeout_us);
        if (n_done) *n_done = rc == GPUOS_OK ? 1u : 0u;
        return rc;
    }
    return submit_run_spsc(c, d, count, n_done, timeout_us);
}

int gpuos_sync(gpuos_ctx *c, uint64_t ticket, uint32_t timeout_ms)
{
    if (!c) return GPUOS_EINVAL;
    const uint64_t head = head_of(c);
    const uint64_t target = (ticket == UINT64_MAX) ? head : ticket + 1;
    if (target > head) return GPUOS_EINVAL;
    if (!c->launched && target > c->low) return GPUOS_ESTOPPED;
    const uint64_t t0 = now_ns();
    uint32_t spins = 0;
    heartbeat(c);
    while (true) {
        bool done;
        {
            HarvestLock lk(c);
            sweep(c);
            done = c->low >= target;
            if (!done && ticket != UINT64_MAX && (head_of(c) - ticket <= c->N) && is_done(c, ticket)) {
                harvest_one(c, ticket);
                done = true;
            }
        }
        if (done) break;
        if ((++spins & 1023u) == 0) {
            heartbeat(c);
            if (now_ns() - t0 > (uint64_t)timeout_ms * 1000000ull) return GPUOS_ETIMEDOUT;
            if (executor_gone(c)) {
                HarvestLock lk(c);
                sweep(c);
                if (c->low >= target) break;
                c->running = false;
                return GPUOS_ESTOPPED;
            }
        }
        cpu_relax();
    }
    HarvestLock lk(c);
    if (__atomic_exchange_n(&c->pending_errors, (uint64_t)0, __ATOMIC_ACQ_REL)) return GPUOS_EDEVICE;
    return GPUOS_OK;
}

int gpuos_query(gpuos_ctx *c, uint64_t ticket, gpuos_record *rec)
{
    if (!c || !rec) return GPUOS_EINVAL;
    HarvestLock lk(c);
    if (ticket >= head_of(c)) return GPUOS_EINVAL;
    if (c->history && ticket >= c->hist_base && ticket - c->hist_base < c->hist_cap &&
        c->history[ticket - c->hist_base].ticket == ticket && ticket < c->low) {
        *rec = c->history[ticket - c->hist_base];
        return GPUOS_OK;
    }
    if (head_of(c) - ticket > c->N) return GPUOS_EINVAL;
    /* inside the window the slot still holds this ticket's record: the
     * ticket ring_entries later has not been taken */
    if (!is_done(c, ticket)) return GPUOS_EAGAIN;
    *rec = read_record(c, ticket);
    harvest_one(c, ticket);
    return GPUOS_OK;
}

int gpuos_set_history(gpuos_ctx *c, gpuos_record *buf, uint64_t base, uint64_t capacity)
{
    if (!c || (buf == nullptr && capacity)) return GPUOS_EINVAL;
    c->history = buf;
    c->hist_base = base;
    c->hist_cap = buf ? capacity : 0;
    if (buf)
        for (uint64_t i = 0; i < capacity; i++) buf[i].ticket = UINT64_MAX;
    return GPUOS_OK;
}

/* ---- dual-slot table flip ------------------------------------------------------- */
static int flip_entry(gpuos_ctx *c, uint16_t op_id, uint64_t fnval, const gpuos_ctx::Binding &bind)
{
    /* grace period: descriptors sequenced under version-1 (all tickets below
     * the head recorded at the last flip) must have completed before the
     * slot they read is rewritten */
    const uint64_t t0 = now_ns();
    while (true) {
        {
            HarvestLock lk(c);
            sweep(c);
            if (c->low >= c->flip_head) break;
        }
        if (now_ns() - t0 > (uint64_t)c->cfg.dep_timeout_ms * 2000000ull) return GPUOS_ETIMEDOUT;
        if (executor_gone(c)) return GPUOS_ESTOPPED;
        heartbeat(c);
        cpu_relax();
    }
    const uint32_t nv = c->version + 1;
    const uint32_t ns = nv & 1u;
    memcpy(c->table_host[ns], c->table_host[c->version & 1u], sizeof(c->table_host[0]));
    c->table_host[ns][op_id] = fnval;
    for (int i = 0; i < GPUOS_MAX_OPS; i++) c->binding[ns][i] = c->binding[c->version & 1u][i];
    c->binding[ns][op_id] = bind;
    /* the inactive slot with plain stores (no sequencer reads it: each copies
     * a slot only when it first sees that slot's version), then the version
     * with a store-release: a sequencer that sees the new version sees the
     * slot written, and every descriptor committed after this store runs
     * with it (the run's release fence orders the two) */
    memcpy(c->table + (size_t)ns * GPUOS_MAX_OPS, c->table_host[ns], sizeof(c->table_host[0]));
    store_rel(&c->hctl->version, nv);
    c->version = nv;
    c->flip_head = head_of(c);
    heartbeat(c);
    return GPUOS_OK;
}

static uint64_t fnv1a(const void *p, size_t n)
{
    const unsigned char *b = static_cast<const unsigned char *>(p);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < n; i++) h = (h ^ b[i]) * 1099511628211ull;
    return h;
}

static bool executor_resident(gpuos_ctx *c)
{
    return c->launched && cudaStreamQuery(c->exec_stream) == cudaErrorNotReady;
}

/* index of the loaded module holding `image`, or -1 */
static int find_module(gpuos_ctx *c, const void *image, size_t len, uint64_t h)
{
    for (size_t i = 0; i < c->modules.size(); i++) {
        const auto &m = c->modules[i];
        if (m.hash == h && m.bytes.size() == len && memcmp(m.bytes.data(), image, len) == 0) return (int)i;
    }
    return -1;
}

/* Take a new operator module into a running executor (an executor hand-off).
 * A module load waits for the device to go idle, and a function address is
 * callable only inside the module that holds its code, so the module cannot
 * join the resident kernel: every submitted descriptor completes, the
 * executor leaves, the module set is linked again with the new module and
 * the executor is launched from it. The ring, the completion records, the
 * tickets and the operator bindings carry over: the new kernel starts at the
 * next ticket and after the last work-queue index the old one handed out,
 * and its table is rebuilt from the bindings with the new module's
 * addresses. Single-producer contexts only (the caller's thread is the only
 * submitter, so nothing is committed meanwhile). */
static int handoff(gpuos_ctx *c, const void *image, size_t len, uint64_t h)
{
    if (c->mp) return GPUOS_EBUSY;
    if (!c->running) return GPUOS_ESTOPPED;
    Driver &drv = driver();
    if (!drv.ok) return GPUOS_ECUDA;
    const uint64_t ts0 = now_ns();
    /* the new set must link before anything stops */
    std::vector<std::vector<unsigned char>> objs;
    for (auto &m : c->modules) objs.push_back(m.bytes);
    objs.emplace_back((const unsigned char *)image, (const unsigned char *)image + len);
    std::vector<unsigned char> img;
    int rc = link_images(objs, &img);
    if (rc) return rc;
    const uint64_t ts1 = now_ns();
    /* drain under the old executor (an error status harvested here stays
     * pending for the caller's next gpuos_sync) */
    rc = gpuos_sync(c, UINT64_MAX, 2 * c->cfg.dep_timeout_ms + 1000);
    if (rc == GPUOS_EDEVICE) __atomic_fetch_add(&c->pending_errors, (uint64_t)1, __ATOMIC_RELAXED);
    else if (rc != GPUOS_OK) return rc;
    /* the executor is idle: let it leave (from here until the new kernel
     * runs, nothing is dispatched) */
    const uint64_t t_down = now_ns();
    store_rel(&c->hctl->stop, 1u);
    const uint64_t t0 = now_ns();
    while (cudaStreamQuery(c->exec_stream) == cudaErrorNotReady) {
        if (now_ns() - t0 > 10000000000ull) {
            c->running = false;
            return GPUOS_ETIMEDOUT;
        }
        cpu_relax();
    }
    c->running = false;
    c->launched = false;
    if (cudaStreamQuery(c->exec_stream) != cudaSuccess) return GPUOS_ECUDA;
    const uint64_t ts2 = now_ns();
    gpuos_ctx::Module m;
    m.hash = h;
    m.bytes = std::move(objs.back());
    c->modules.push_back(std::move(m));
    if (c->linked) drv.unload(c->linked);
    c->linked = nullptr;
    c->linked_exec = nullptr;
    /* where the new kernel starts: the next ticket, and the work-queue index
     * after every one the old kernel's workers claimed (none past it was
     * ever written in this lap, so no stale entry matches) */
    uint64_t *claim = reinterpret_cast<uint64_t *>(c->version_stage + 4);
    if (cudaMemcpyAsync(claim, &c->dctl->tq_claim, 8, cudaMemcpyDeviceToHost, c->ctl_stream) != cudaSuccess ||
        cudaMemsetAsync(&c->dctl->exit_flag, 0, 4, c->ctl_stream) != cudaSuccess ||
        cudaStreamSynchronize(c->ctl_stream) != cudaSuccess)
        return GPUOS_ECUDA;
    c->params.ticket_base = c->head;
    c->params.tq_base = *claim;
    /* the sequencers' turn starts there too (both fields modulo 2^32) */
    uint64_t *turn = reinterpret_cast<uint64_t *>(c->version_stage + 8);
    turn[0] = ((c->params.tq_base & 0xFFFFFFFFull) << 32) | (c->params.ticket_base & 0xFFFFFFFFull);
    if (cudaMemcpyAsync(&c->dctl->turn, turn, 8, cudaMemcpyHostToDevice, c->ctl_stream) != cudaSuccess ||
        cudaStreamSynchronize(c->ctl_stream) != cudaSuccess)
        return GPUOS_ECUDA;
    store_rel(&c->hctl->stop, 0u);
    __atomic_store_n(&c->hctl->exit_reason, 0u, __ATOMIC_RELAXED);
    store_rel(&c->hctl->state, 0u);
    c->flip_head = c->head; /* nothing sequenced under an older version is in flight */
    heartbeat(c);
    rc = launch_linked(c, &img);
    if (rc) return rc;
    c->launched = true;
    const uint64_t t1 = now_ns();
    while (load_acq(&c->hctl->state) == 0u) {
        if (cudaStreamQuery(c->exec_stream) != cudaErrorNotReady || now_ns() - t1 > 10000000000ull) {
            store_rel(&c->hctl->stop, 1u);
            return GPUOS_ECUDA;
        }
        cpu_relax();
    }
    c->running = true;
    c->n_handoffs++;
    c->handoff_link_ns = ts1 - ts0;
    c->handoff_down_ns = now_ns() - t_down;
    if (getenv("GPUOS_DEBUG"))
        fprintf(stderr, "gpuos: hand-off %u: link %.2f ms, drain and leave %.2f ms, load and relaunch %.2f ms\n",
                c->n_handoffs, (ts1 - ts0) / 1e6, (ts2 - ts1) / 1e6, (now_ns() - ts2) / 1e6);
    return GPUOS_OK;
}

int gpuos_load_module(gpuos_ctx *c, const void *image, size_t len)
{
    if (!c || !image || !len) return GPUOS_EINVAL;
    const uint64_t h = fnv1a(image, len);
    if (find_module(c, image, len, h) >= 0) return GPUOS_OK;
    if (c->launched) return handoff(c, image, len, h); /* a running executor: hand off */
    /* check now that the object links with the executor */
    std::vector<std::vector<unsigned char>> objs(1);
    objs[0].assign((const unsigned char *)image, (const unsigned char *)image + len);
    std::vector<unsigned char> img;
    const int rc = link_images(objs, &img);
    if (rc) return rc;
    gpuos_ctx::Module m;
    m.hash = h;
    m.bytes = std::move(objs[0]);
    c->modules.push_back(std::move(m));
    return GPUOS_OK;
}

int gpuos_register_op(gpuos_ctx *c, uint16_t op_id, const void *image, size_t len, const char *sym)
{
    if (!c || !image || !len || !sym || op_id >= GPUOS_MAX_OPS || op_id == GPUOS_OP_NOP) return GPUOS_EINVAL;
    if (op_id >= GPUOS_OP_BUILTIN_COUNT && op_id < GPUOS_OP_USER_FIRST) return GPUOS_EINVAL;
    if (!c->accepting) return GPUOS_ESTOPPED;
    if (find_module(c, image, len, fnv1a(image, len)) < 0) {
        /* not linked into the executor: linked at the launch, or, with the
         * executor running, taken in by a hand-off */
        const int rc = gpuos_load_module(c, image, len);
        if (rc) return rc;
    }
    if (!c->launched || !c->linked) return GPUOS_EBUSY; /* the swap needs the linked, running executor */
    heartbeat(c);
    CUdeviceptr gp = 0;
    size_t gsz = 0;
    if (driver().get_global(&gp, &gsz, c->linked, sym) != CUDA_SUCCESS || gsz != sizeof(uint64_t))
        return GPUOS_EINVAL;
    uint64_t fnval = 0;
    if (cudaMemcpyAsync(c->version_stage + 2, (const void *)gp, 8, cudaMemcpyDeviceToHost, c->ctl_stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(c->ctl_stream) != cudaSuccess)
        return GPUOS_ECUDA;
    memcpy(&fnval, c->version_stage + 2, 8);
    if (fnval == 0) return GPUOS_EINVAL;
    gpuos_ctx::Binding bind;
    bind.sym = sym;
    const int rc = flip_entry(c, op_id, fnval, bind);
    if (rc == GPUOS_OK && op_id >= GPUOS_OP_USER_FIRST) c->user_registered[op_id] = true;
    return rc;
}

int gpuos_alias_op(gpuos_ctx *c, uint16_t op_id, uint16_t source_op)
{
    if (!c || op_id >= GPUOS_MAX_OPS || source_op >= GPUOS_MAX_OPS || op_id == GPUOS_OP_NOP) return GPUOS_EINVAL;
    if (op_id >= GPUOS_OP_BUILTIN_COUNT && op_id < GPUOS_OP_USER_FIRST) return GPUOS_EINVAL;
    if (!c->accepting) return GPUOS_ESTOPPED;
    const uint64_t v = c->table_host[c->version & 1u][source_op];
    if (v == 0) return GPUOS_EINVAL;
    const int rc = flip_entry(c, op_id, v, c->binding[c->version & 1u][source_op]);
    if (rc == GPUOS_OK && op_id >= GPUOS_OP_USER_FIRST) c->user_registered[op_id] = true;
    return rc;
}

int gpuos_stats(gpuos_ctx *c, gpuos_stats_t *st)
{
    if (!c || !st) return GPUOS_EINVAL;
    memset(st, 0, sizeof(*st));
    const uint32_t tw = c->blocks * c->wpb;
    std::vector<uint64_t> ws((size_t)tw * GPUOS_WS_N);
    if (cudaMemcpyAsync(ws.data(), c->warp_stats, ws.size() * 8, cudaMemcpyDeviceToHost, c->ctl_stream) != cudaSuccess ||
        cudaStreamSynchronize(c->ctl_stream) != cudaSuccess)
        return GPUOS_ECUDA;
    for (uint32_t w = 0; w < tw; w++) {
        const uint64_t *x = &ws[(size_t)w * GPUOS_WS_N];
        st->tiles += x[GPUOS_WS_TILES];
        st->idle_polls += x[GPUOS_WS_IDLE];
        st->sleeps += x[GPUOS_WS_SLEEPS];
        st->dep_waits += x[GPUOS_WS_DEPWAIT];
    }
    /* warp 0 of blocks 0 .. sequencers-1 are the sequencers: their phase
     * timers (summed) and the descriptors they took off the ring */
    uint64_t seq_taken = 0;
    for (uint32_t b = 0; b < c->cfg.sequencers && b < c->blocks; b++) {
        const uint64_t *x = &ws[(size_t)b * c->wpb * GPUOS_WS_N];
        st->seq_body_ns += x[GPUOS_WS_T_BODY];
        st->seq_mirror_ns += x[GPUOS_WS_T_MIRROR];
        st->seq_publish_ns += x[GPUOS_WS_T_PUB];
        st->seq_batches += x[GPUOS_WS_BATCHES];
        seq_taken += x[GPUOS_WS_SEQ];
    }
    st->host_wait_ns = __atomic_load_n(&c->host_wait_ns, __ATOMIC_RELAXED);
    st->handoffs = c->n_handoffs;
    st->handoff_link_ns = c->handoff_link_ns;
    st->handoff_down_ns = c->handoff_down_ns;
    {
        HarvestLock lk(c);
        sweep(c);
        st->completed = __atomic_load_n(&c->n_completed, __ATOMIC_RELAXED);
        st->errors = __atomic_load_n(&c->n_errors, __ATOMIC_RELAXED);
    }
    st->submitted = head_of(c);
    st->sequenced = seq_taken;
    st->version = c->version;
    st->running = (c->running && !executor_gone(c)) ? 1u : 0u;
    st->exit_reason = __atomic_load_n(&c->hctl->exit_reason, __ATOMIC_RELAXED);
    st->blocks = c->blocks;
    st->warps_per_block = c->wpb;
    st->regs_per_thread = c->regs;
    st->static_smem_bytes = c->smem;
    heartbeat(c);
    return GPUOS_OK;
}

int gpuos_tile_profile_get(gpuos_ctx *c, gpuos_tile_profile *out)
{
    if (!c || !out) return GPUOS_EINVAL;
    memset(out, 0, sizeof(*out));
    const uint32_t tw = c->blocks * c->wpb;
    std::vector<uint64_t> ws((size_t)tw * GPUOS_WS_N);
    if (cudaMemcpyAsync(ws.data(), c->warp_stats, ws.size() * 8, cudaMemcpyDeviceToHost, c->ctl_stream) != cudaSuccess ||
        cudaStreamSynchronize(c->ctl_stream) != cudaSuccess)
        return GPUOS_ECUDA;
    uint64_t *rows[GPUOS_PROF_FIELDS] = {out->tiles, out->body_ns, out->finish_ns, out->dep_ns};
    for (uint32_t w = 0; w < tw; w++) {
        const uint64_t *x = &ws[(size_t)w * GPUOS_WS_N + GPUOS_WS_PROF];
        for (uint32_t f = 0; f < GPUOS_PROF_FIELDS; f++)
            for (uint32_t b = 0; b < GPUOS_PROF_BUCKETS; b++) rows[f][b] += x[f * GPUOS_PROF_BUCKETS + b];
    }
    return GPUOS_OK;
}

int gpuos_calibrate(gpuos_ctx *c, uint32_t pings, int64_t *off_lo, int64_t *off_hi, uint64_t *min_rtt_ns,
                    uint64_t *rtts)
{
    if (!c || pings == 0) return GPUOS_EINVAL;
    int rc = gpuos_sync(c, UINT64_MAX, 10000);
    if (rc != GPUOS_OK && rc != GPUOS_EDEVICE) return rc;
    gpuos_desc nop;
    memset(&nop, 0, sizeof(nop));
    nop.op_id = GPUOS_OP_NOP;
    uint64_t best = UINT64_MAX;
    int64_t lo = INT64_MIN, hi = INT64_MAX;
    for (uint32_t i = 0; i < pings; i++) {
        uint64_t t = 0;
        /* every earlier ticket has completed and been harvested (the sync
         * above, and each ping below waits for its own completion), so no
         * completion rewrites this record any more: clear the field the
         * sequencer echoes its observation time into (it still holds the
         * previous ticket's) */
        __atomic_store_n(&c->rec[head_of(c) & c->mask].t_dispatch, (uint64_t)0, __ATOMIC_RELAXED);
        const uint64_t t0 = now_ns();
        rc = gpuos_submit(c, &nop, &t, 1000000);
        if (rc) return rc;
        const gpuos_rec_dev *r = c->rec + (t & c->mask);
        uint32_t spins = 0;
        /* the sequencer echoes its observation time into the record as soon
         * as it sees the commit: t0 <= observation <= t1 */
        uint64_t td = 0;
        while ((td = __atomic_load_n(&r->t_dispatch, __ATOMIC_ACQUIRE)) == 0) {
            if ((++spins & 0xFFFFFu) == 0 && executor_gone(c)) return GPUOS_ESTOPPED;
        }
        const uint64_t t1 = now_ns();
        while (!is_done(c, t)) {
            if ((++spins & 0xFFFFFu) == 0 && executor_gone(c)) return GPUOS_ESTOPPED;
        }
        const uint64_t rtt = t1 - t0;
        if (rtts) rtts[i] = rtt;
        if (rtt < best) best = rtt;
        const int64_t a = (int64_t)(td - t1), b = (int64_t)(td - t0);
        if (a > lo) lo = a;
        if (b < hi) hi = b;
        HarvestLock lk(c);
        harvest_one(c, t);
        sweep(c);
    }
    if (off_lo) *off_lo = lo;
    if (off_hi) *off_hi = hi;
    if (min_rtt_ns) *min_rtt_ns = best;
    return GPUOS_OK;
}

int gpuos_stop(gpuos_ctx *c, uint32_t timeout_ms)
{
    if (!c) return GPUOS_EINVAL;
    int rc = GPUOS_OK;
    if (c->running) {
        const int s = gpuos_sync(c, UINT64_MAX, timeout_ms);
        if (s == GPUOS_ETIMEDOUT) rc = s;
    }
    c->accepting = false;
    store_rel(&c->hctl->stop, 1u);
    if (!c->launched) return rc;
    const uint64_t t0 = now_ns();
    while (true) {
        const cudaError_t q = cudaStreamQuery(c->exec_stream);
        if (q != cudaErrorNotReady) {
            if (q != cudaSuccess && rc == GPUOS_OK) rc = GPUOS_ECUDA;
            c->running = false;
            HarvestLock lk(c);
            sweep(c);
            return rc;
        }
        if (now_ns() - t0 > (uint64_t)(timeout_ms ? timeout_ms : 1) * 1000000ull) break;
        cpu_relax();
    }
    return rc == GPUOS_OK ? GPUOS_ETIMEDOUT : rc;
}

int gpuos_shutdown(gpuos_ctx *c, uint32_t timeout_ms)
{
    if (!c) return GPUOS_EINVAL;
    const int rc = gpuos_stop(c, timeout_ms);
    if (c->launched && cudaStreamQuery(c->exec_stream) == cudaErrorNotReady) {
        /* the kernel still runs (it will leave through its watchdog); device
         * memory cannot be released under it, so only the host side goes */
        delete c;
        return rc;
    }
    free_all(c);
    return rc;
}

int gpuos_eager_run(const gpuos_desc *d, uint32_t count, uint32_t stage_bytes, void *stream)
{
    if (!d && count) return GPUOS_EINVAL;
    if ((stage_bytes & 1023u) || stage_bytes > 24576u) return GPUOS_EINVAL;
    for (uint32_t i = 0; i < count; i++) {
        uint32_t nt = 0;
        if (d[i].op_id >= GPUOS_OP_BUILTIN_COUNT) return GPUOS_EINVAL;
        const int rc = validate_and_tile(d + i, &nt, false);
        if (rc) return rc;
        /* element-wise ops: smaller tiles than the executor's. A launch runs
         * one op, so its warps are all the parallelism it has; the
         * executor's larger tiles pay off only because many ops run at
         * once */
        const uint16_t op = d[i].op_id;
        if (op == GPUOS_OP_ADD || op == GPUOS_OP_MUL || op == GPUOS_OP_RELU || op == GPUOS_OP_GELU) {
            const uint64_t e = ew_tiles(d[i].dims[0], op == GPUOS_OP_GELU ? GPUOS_EAGER_GELU_TILE_MIN : GPUOS_EAGER_TILE_MIN,
                                        d[i].dtype == GPUOS_F32 ? GPUOS_EAGER_TILE_F32 : GPUOS_EAGER_TILE_BF16);
            if (e > GPUOS_TILE_MAX) return GPUOS_EINVAL;
            nt = e ? (uint32_t)e : 1u;
        }
        if (gpuos_dev_eager_launch(d + i, nt, stage_bytes, stream) != 0) return GPUOS_ECUDA;
    }
    return GPUOS_OK;
}

}  // extern "C"
