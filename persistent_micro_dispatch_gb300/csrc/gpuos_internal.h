/*
 * Internal layouts shared by the host library (gpuos_host.cpp) and the device
 * code (gpuos_device.cu). Not part of the public ABI.
 */
#ifndef GPUOS_INTERNAL_H
#define GPUOS_INTERNAL_H

#include <stdint.h>

#include "gpuos.h"

/* Tiling constants of the built-in ops (one tile = one warp's unit of work). */
#define GPUOS_EW_TILE_F32 16384           /* largest fp32 element-wise tile the host picks (64 KB an operand) */
#define GPUOS_EW_TILE_BF16 32768          /* ... and bf16 tile */
#define GPUOS_EW_TILE_MIN 16384           /* smallest add/mul/ReLU tile the host picks */
#define GPUOS_GELU_TILE_MIN 16384         /* ... and GELU tile (as add/mul/ReLU) */
#define GPUOS_GELU_DEP_TILE_MIN 1024      /* ... and GELU tile of a descriptor with a dependency */
#define GPUOS_EAGER_TILE_F32 4096         /* element-wise tiles of the eager baseline: largest fp32 */
#define GPUOS_EAGER_TILE_BF16 8192        /* ... largest bf16 */
#define GPUOS_EAGER_TILE_MIN 4096         /* ... smallest add/mul/ReLU */
#define GPUOS_EAGER_GELU_TILE_MIN 1024    /* ... smallest GELU */
#define GPUOS_EW_SPLIT 16                 /* element-wise ops aim at this many tiles */
#define GPUOS_EW_ALIGN 256                /* element-wise tile sizes are multiples of this */
#define GPUOS_SDPA_CHUNK 256              /* key rows per tile of the allocation-free attention */
#define GPUOS_SDPA_CHUNK_MIN 32           /* key rows per decode-attention tile at least (workspace sizing) */
#define GPUOS_SDPA_SPLIT 1536             /* decode-attention tiles at most (unless B * H is more) */
#define GPUOS_HEAD_GROUP 4                /* heads per RoPE / KV-write tile */
#define GPUOS_VM_COLS 8                   /* output columns per vecmat tile (16 bytes of a row) */
#define GPUOS_ROW_REG_MAX 4096            /* rows up to this width stay in registers */
#define GPUOS_MAX_WPB 12
#define GPUOS_MAX_SEQ 4 /* sequencer warps at most */
#define GPUOS_SHORT_SLEEP_NS 256u /* longest idle sleep on the dispatch path (ring poll, dependency waits) */
/* static shared memory of the executor kernel: descriptor copies, the
 * sequencer's table copy, per-warp tile profiles */
#define GPUOS_EXEC_STATIC_SMEM (GPUOS_MAX_WPB * 128 + 256 * 8 + GPUOS_MAX_WPB * GPUOS_PROF_FIELDS * GPUOS_PROF_BUCKETS * 8)
#define GPUOS_MAX_REGS 168 /* registers per thread: 65536 / (12 warps x 32), in steps of 8 */
#define GPUOS_TILE_MAX (1u << 30)          /* tiles per descriptor */
#define GPUOS_HELPERS 2048                 /* work-queue entries (helper warps) per descriptor at most */
#define GPUOS_TQ_MAX (1u << 30)            /* work-queue entries */
#define GPUOS_TQ_STAMP_MASK 0xFFFFFFFFFull /* 36-bit stamps */

/* Mirror of a descriptor in device memory, written by a sequencer warp.
 * Same layout as gpuos_desc except the last fields. */
typedef struct gpuos_devdesc {
    uint16_t op_id;
    uint8_t dtype;
    uint8_t flags;
    uint32_t ntiles;
    uint64_t dep[2];
    uint64_t a, b, out;
    uint64_t aux0, aux1, aux2;
    uint32_t dims[6];
    float fparam[2];
    uint64_t fn;         /* op entry point, fixed with the version at sequencing (replaces `user`) */
    uint64_t ticket;
    uint32_t version;    /* table version fixed at sequencing (replaces `seq`) */
    uint32_t pad;        /* the helper warps (work-queue entries) published for it */
} gpuos_devdesc;

/* Work-queue entries are single 64-bit words (see tq_word in the device
 * code): 36-bit stamp, 16-bit ring slot, 12-bit helper index. */

/* Completion record in host-visible memory, written by the device. */
/* Completion word of a ring slot (host-visible, one 8-byte word per slot,
 * eight slots to a cache line): ticket + 1 in bits 0..55 once the ticket is
 * complete, bit 63 set if it completed with a nonzero status (the record
 * holds the status itself). Stored with release at system scope after the
 * record's fields; the host's load-acquire of it frees the slot. */
#define GPUOS_DONE_TICKET_MASK ((1ull << 56) - 1ull)
#define GPUOS_DONE_FAILED (1ull << 63)

typedef struct gpuos_rec_dev {
    uint64_t reserved; /* (the completion word lives in the compact done array) */
    int32_t status;
    uint32_t version;
    uint64_t t_dispatch;
    uint64_t t_publish; /* tiles published to the work queue */
    uint64_t t_start;   /* tile 0 began */
    uint64_t t_done;
    uint64_t pad[2];
} gpuos_rec_dev;

/* Host-visible control block (pinned host memory). */
typedef struct gpuos_hostctl {
    uint64_t heartbeat; /* host: bumped by API calls */
    uint32_t stop;      /* host: 1 = leave when idle */
    uint32_t pad0[29];
    uint32_t version;   /* host: operator-table version, flipped with a store-release
                         * after the inactive slot of the table is written */
    uint32_t padv[31];
    uint32_t state;       /* device: 1 running, 2 leaving */
    uint32_t exit_reason; /* device: see gpuos_stats_t */
    uint64_t sequenced;   /* device: tickets taken off the ring */
    uint64_t exit_now;    /* device: clock when the sequencer decided to leave */
    uint64_t exit_active; /* device: last activity it had seen then */
    uint32_t pad1[24];
} gpuos_hostctl;

/* Device-memory control block; hot words on their own 128-byte lines. */
typedef struct gpuos_devctl {
    unsigned long long tq_claim; /* next work-queue index to claim */
    uint64_t pad0[15];
    unsigned long long completed; /* descriptors completed */
    uint64_t pad1[15];
    uint32_t exit_flag; /* nonzero: workers leave when they find no work */
    uint32_t pad_x;
    uint64_t pad2[15];
    uint64_t turn;      /* sequencers' turn, one word: [31:0] the first ticket whose work-queue
                           space is not reserved (mod 2^32), [63:32] the next free work-queue
                           index (mod 2^32) */
    uint64_t pad3[15];
} gpuos_devctl;

/* Per-warp counters (owned by one warp each, plain stores). */
enum { GPUOS_WS_TILES = 0, GPUOS_WS_IDLE = 1, GPUOS_WS_SLEEPS = 2, GPUOS_WS_DEPWAIT = 3,
       GPUOS_WS_SEQ = 4, GPUOS_WS_T_BODY = 5, GPUOS_WS_T_MIRROR = 6, GPUOS_WS_T_PUB = 7,
       GPUOS_WS_BATCHES = 8,
       /* tile profile: GPUOS_PROF_FIELDS rows of GPUOS_PROF_BUCKETS (op id, or the last
        * bucket for user ops): tiles, body ns, finish ns, dependency ns */
       GPUOS_WS_PROF = 9, GPUOS_WS_N = 9 + GPUOS_PROF_FIELDS * GPUOS_PROF_BUCKETS };

typedef int (*gpuos_op_fn)(const gpuos_devdesc *d, uint32_t tile);

typedef struct gpuos_exec_params {
    const gpuos_desc *ring;  /* host-visible ring */
    gpuos_rec_dev *rec;      /* host-visible completion records */
    uint64_t *done_host;     /* host-visible completion words, [ring_entries] */
    gpuos_hostctl *hctl;
    gpuos_devdesc *mirror;   /* [ring_entries] */
    unsigned long long *tiles_done; /* [ring_entries]: tiles done (low 32 bits), failed helpers (high 32) */
    uint32_t *err;           /* [ring_entries] */
    uint32_t *tile_ctr;      /* [ring_entries], next extra tile (past the helpers' first tiles) */
    uint64_t *done_dev;      /* [ring_entries], ticket + 1 stamps for dependency waits */
    uint64_t *t_start;       /* [ring_entries], device clock when tile 0 began */
    uint64_t *t_pub;         /* [ring_entries], device clock when tiles were published */
    uint64_t *t_disp;        /* [ring_entries], device clock when the commit was seen */
    unsigned long long *tq;  /* [tq_entries] work-queue words */
    gpuos_devctl *dctl;
    const uint64_t *table;   /* [2][GPUOS_MAX_OPS] op entry points, host-visible (pinned) */
    uint64_t *warp_stats;    /* [total warps][GPUOS_WS_N] */
    uint32_t ring_mask, tq_mask;
    uint32_t backoff_min_ns, backoff_max_ns, spin_polls, stage_bytes;
    uint32_t workers;        /* worker warps (all warps but the sequencers) */
    uint32_t sequencers;     /* sequencer warps (warps 0.. of block 0) */
    uint64_t idle_exit_ns, dep_timeout_ns, exit_after;
    uint64_t ticket_base;    /* first ticket this launch takes (0, or where a hand-off resumes) */
    uint64_t tq_base;        /* first work-queue index this launch reserves */
} gpuos_exec_params;

#ifdef __cplusplus
static_assert(sizeof(gpuos_desc) == 128, "descriptor must be 128 bytes");
static_assert(sizeof(gpuos_devdesc) == 128, "mirror must be 128 bytes");
static_assert(sizeof(gpuos_rec_dev) == 64, "record must be 64 bytes");
#endif

/* Launch helpers implemented in gpuos_device.cu (host side). */
#ifdef __cplusplus
extern "C" {
#endif
int gpuos_dev_launch_executor(const gpuos_exec_params *p, uint32_t blocks, uint32_t wpb, void *stream);
int gpuos_dev_builtin_table(gpuos_op_fn *host_out, uint32_t n);
int gpuos_dev_executor_attrs(uint32_t *regs, uint32_t *smem);
int gpuos_dev_eager_launch(const gpuos_desc *d, uint32_t ntiles, uint32_t stage_bytes, void *stream);
uint32_t gpuos_dev_dyn_smem(uint32_t wpb, uint32_t stage_bytes);
int gpuos_dev_preload(void);
#ifdef __cplusplus
}
#endif

#endif /* GPUOS_INTERNAL_H */
