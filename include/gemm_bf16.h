/*
 * gemm_bf16.h -- C ABI of a persistent, warp-specialised, TMA-fed bf16 GEMM for
 * NVIDIA GB300 (sm_103a):
 *
 *     D[m][n] = bf16( sum_k A[m][k] * B[n][k] ),  0 <= m < M, 0 <= n < N
 *
 * A is M x K and B is N x K, both row-major with the contraction index
 * contiguous ("K-major"), bf16; products are accumulated in fp32 in tensor
 * memory and rounded once to bf16 (nearest, ties to even) when stored.
 *
 * Where the operation and its pipeline come from:
 *  - Fuser issue #3941, "Allow separate sub-DAG for load and compute warp groups
 *    with warp-specialized circular buffering": the persistent matmul (a
 *    grid-stride loop over output tiles with a cta-k loop inside), the load warp
 *    group's merged tile x cta-k loop, the compute side's separate tile and k
 *    loops, the fp32 -> bf16 epilogue with a TMA store, and the register
 *    rebalancing between load and compute warps (Scheduling Proposal,
 *    Lowering Proposal, Pseudo-code).
 *  - Fuser PR #3446, "Use mbarrier for WAR for circular buffering": the stage
 *    ring with one "full" barrier (data landed, read-after-write) and one
 *    "empty" barrier (data fully read, write-after-read) per stage, and the
 *    __syncthreads-WAR loop it replaces (both kept as ablations).
 *  - cutlass PR #3316, "[Tutorial] Fix race condition in 2SM TMEM alloc for Cute
 *    Blackwell Tutorial 04/05": in the 2-CTA (paired-SM) mode a cluster barrier
 *    precedes the paired tensor-memory allocation.
 *
 * Conventions for every entry point:
 *  - Return value: GEMM_BF16_OK (0) or a negative gemm_bf16_status.  No entry
 *    point aborts, throws or prints; gemm_bf16_strerror() names a status.
 *  - Device pointers are plain CUDA device addresses of the device the handle
 *    was created on; the caller owns them.  "stream" is a cudaStream_t passed as
 *    void* (NULL = the legacy default stream); the caller owns it.
 *  - A handle is not thread-safe: use one handle per host thread.
 */
#ifndef GEMM_BF16_H
#define GEMM_BF16_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define GEMM_BF16_API __declspec(dllexport)
#else
#define GEMM_BF16_API __attribute__((visibility("default")))
#endif

typedef struct gemm_bf16 *gemm_bf16_t;

typedef enum gemm_bf16_status {
    GEMM_BF16_OK = 0,
    GEMM_BF16_ERR_INVALID_ARG = -1,    /* null handle/pointer, size <= 0, ld < extent, bad option */
    GEMM_BF16_ERR_ALIGNMENT = -2,      /* a TMA rule broken: A/B base not 16-byte aligned, lda*2 or ldb*2 not a multiple of 16 */
    GEMM_BF16_ERR_NOT_PLANNED = -3,    /* run before a successful plan */
    GEMM_BF16_ERR_CUDA = -4,           /* a CUDA runtime call failed (launch, copy, allocation) */
    GEMM_BF16_ERR_TENSORMAP = -5,      /* the driver refused a TMA tensor-map encoding */
    GEMM_BF16_ERR_DEVICE_TIMEOUT = -6, /* a kernel's bounded barrier wait ran out; the kernel returned early */
    GEMM_BF16_ERR_UNSUPPORTED = -7     /* device is not sm_103, or the option combination cannot run on it */
} gemm_bf16_status;

/* Pipeline variants (GEMM_BF16_OPT_PIPELINE). */
typedef enum gemm_bf16_pipeline {
    /* Warp-specialised: one TMA producer warp, one tcgen05 MMA warp, two epilogue
     * warpgroups; full/empty mbarrier ring; persistent tile loop. (default) */
    GEMM_BF16_PIPE_WS = 0,
    /* Not specialised, write-after-read guarded by __syncthreads(): one elected
     * thread loads and issues the MMAs; every thread waits for the data and for
     * the MMAs to finish, then the block synchronises (the loop Fuser PR #3446
     * starts from).  One tile per CTA, 1-CTA mode only. */
    GEMM_BF16_PIPE_SYNC_WAR = 1,
    /* Not specialised, write-after-read guarded by an "empty" mbarrier per stage
     * that the MMA completion arrives on (the loop Fuser PR #3446 adds).  One
     * tile per CTA, 1-CTA mode only. */
    GEMM_BF16_PIPE_MBAR_WAR = 2
} gemm_bf16_pipeline;

/* Options, set before gemm_bf16_plan (a later plan picks them up). */
typedef enum gemm_bf16_option {
    GEMM_BF16_OPT_PIPELINE = 1,      /* gemm_bf16_pipeline; default GEMM_BF16_PIPE_WS */
    GEMM_BF16_OPT_CTA_GROUP = 2,     /* 0 = automatic (default: an SM pair, except one SM for
                                        problems of at most 512 x 512 outputs and 512^3
                                        multiply-adds, which are bound by fixed latency),
                                        1 = one SM per tile (128x256),
                                        2 = SM pair per tile (256x256, cta_group::2, WS only) */
    GEMM_BF16_OPT_PERSISTENT = 3,    /* 1 (default): grid = resident CTAs, grid-stride tile loop;
                                        0: one tile per CTA (grid = tiles) */
    GEMM_BF16_OPT_ACC_BUFFERS = 4,   /* tensor-memory accumulators per CTA: 2 (default) lets the
                                        epilogue of a tile overlap the next tile's main loop; 1 */
    GEMM_BF16_OPT_SETMAXNREG = 5,    /* 1: the producer/MMA warpgroup drops to 56 registers per
                                        thread and the epilogue warpgroups rise to 224;
                                        0 (default): no rebalancing (the accumulator lives in
                                        tensor memory, so no role needs more than the launch's
                                        168 registers, and the 56-register limit spills) */
    GEMM_BF16_OPT_STAGES = 6,        /* stage-ring depth; 0 (default) = as deep as shared memory allows */
    GEMM_BF16_OPT_RASTER_GROUP = 7,  /* tile order: groups of this many tile rows walked column by
                                        column (default 8); 0 = plain row-major */
    GEMM_BF16_OPT_EPILOGUE = 8,      /* 0 = automatic (default): TMA store when D's base is 16-byte
                                        aligned and ldd*2 is a multiple of 16, else masked stores;
                                        1 = TMA store (run fails with ALIGNMENT if not allowed);
                                        2 = masked coalesced st.global */
    GEMM_BF16_OPT_MAX_CTAS = 9,      /* upper bound on the persistent grid (0 = no bound) */
    GEMM_BF16_OPT_WATCHDOG_NS = 10,  /* limit of every in-kernel barrier wait, ns (default 1e9).
                                        plan raises it to 2 us per 64-wide k-block of K when that
                                        is longer: no wait outlasts one tile's k-range of MMAs
                                        (~0.3 us per k-block), so long-k problems never trip it */
    GEMM_BF16_OPT_FAULT_SKIP_LOAD = 11, /* test hook: each CTA's producer skips its load at this
                                          ring iteration, so the MMA warp's wait runs out and
                                          the kernel reports GEMM_BF16_ERR_DEVICE_TIMEOUT;
                                          -1 (default) = off */
    GEMM_BF16_OPT_STAGE_GROUP = 12,  /* ring stages released per MMA commit (WS only): 1 = every
                                        k-block; 2 = stages pair up behind one "empty" barrier
                                        (the ring depth must then be even); 0 (default) = 1 */
    GEMM_BF16_OPT_STREAM_K = 13,     /* Splitting tiles along k in the persistent WS kernel.  A
                                        non-owner part of a split tile leaves an fp32 partial in a
                                        handle-owned workspace (128 KiB per CTA and part, allocated
                                        by plan) that the owner of the tile's first k-block adds
                                        before storing.
                                        1 (default): with at least one whole wave of tiles, the
                                        tiles that would form a partial last wave are split over
                                        all resident SM (pairs); with fewer tiles T than resident
                                        SM (pairs) C, every tile may be split at one k-block H:
                                        SM (pair) t computes [0, H) of tile t and n <= C - T others
                                        share the tails [H, KB), with n and H picked by a cost
                                        model measured on GB300 (the split is taken only when it
                                        beats whole tiles by a margin; plan_info.sk_head reports it);
                                        2: the partial-last-wave split only;
                                        3: as 1, but every problem with fewer tiles than SM (pairs)
                                        is split over all of them, whatever the cost (for tests
                                        and measurements);
                                        0: every tile runs whole */
    GEMM_BF16_OPT_PDL = 14,           /* 1 (default): launch with programmatic stream serialization,
                                        so the kernel's prologue (barrier set-up, tensor-memory
                                        allocation) overlaps the previous kernel on the stream; every
                                        global access waits for that kernel (griddepcontrol.wait).
                                        0: plain stream order */
    GEMM_BF16_OPT_EPI_SCHEDULE = 15,  /* WS kernel's epilogue warpgroups.  0 (default) = cooperative:
                                        both warpgroups drain every tile (a warp: 32 rows x 128
                                        columns).  1 = ping-pong: warpgroup g drains the tiles of
                                        tensor-memory accumulator g, i.e. every other tile (a warp:
                                        32 rows x 256 columns); needs ACC_BUFFERS = 2, else plan
                                        fails with INVALID_ARG */
    GEMM_BF16_OPT_SCHEDULER = 16,     /* WS kernel's tile order.  0 (default) = static: each SM
                                        (pair) walks the grid-stride sequence.  1 = dynamic: after
                                        its stream-K share, each SM (pair) takes the next whole tile
                                        from a device counter owned by the handle, so faster SMs
                                        take more tiles; the last SM (pair) to finish resets the
                                        counter, so launches of one handle must not overlap */
    GEMM_BF16_OPT_REPACK = 17,        /* operands whose row pitch (lda or ldb, in bytes) is not a
                                        multiple of 128: TMA then reads each 128-byte box row as two
                                        L2 lines and the GEMM slows by ~28%.  Such an operand can be
                                        copied first (one HBM read + write, same stream) into a
                                        handle-owned buffer with a 128-byte-multiple pitch.
                                        0 (default) = automatic: A when N >= 4096, B when M >= 4096
                                        (where the GEMM's saving exceeds the copy);
                                        1 = always when misaligned; 2 = never */
    GEMM_BF16_OPT_K_ORDER = 18,       /* WS kernel's k direction per whole tile.  0 = ascending;
                                        1 (default) = alternating: each SM (pair)'s odd-numbered whole tiles load
                                        their k-blocks last to first, so a wave starts on the operand
                                        slices the previous wave loaded last (still in L2).  Changes
                                        only the fp32 summation order (within the rounding bound;
                                        results stay deterministic).  Measured on 8192^3: DRAM reads
                                        -15%, and under the power cap +1% throughput */
    GEMM_BF16_OPT_SERPENTINE = 19,    /* tile order: 1 (default) = odd bands of RASTER_GROUP tile rows
                                        walk their columns right to left, so a band's first tiles
                                        reuse the B panels the previous band read last (8192^3: DRAM
                                        reads -8.6%, +1% under the power cap); 0 = every band left
                                        to right */
    GEMM_BF16_OPT_FAULT_TENSORMAP = 20, /* test hook: 1 = every run of the handle fails its tensor-map
                                        encode as a driver error would, and returns
                                        GEMM_BF16_ERR_TENSORMAP before launching anything;
                                        0 (default) = off */
    GEMM_BF16_OPT_THIN = 21,          /* Problems with min(M, N) <= 64 (decode-like, bound by
                                        streaming the other operand from HBM) can run on the thin
                                        kernel: the large operand in 128-row tiles is the MMA's M
                                        side, the small one its N side (rounded up to 16, 32, 48 or
                                        64), at most one CTA per SM with a ring of up to 12 stages;
                                        each tile's k-blocks split over a thread-block cluster, or
                                        the (tile, k-block) units split evenly over the SMs
                                        (GEMM_BF16_OPT_THIN_CLUSTER); split tiles summed in a fixed
                                        order, across the SMs from fp32 partials in a handle-owned
                                        workspace (2 slots of 128 x 64 fp32 per SM, 4 flags per
                                        slot, and two words).  Of the other options only
                                        WATCHDOG_NS, FAULT_SKIP_LOAD, PDL, REPACK and
                                        FAULT_TENSORMAP apply to it.
                                        1 (default) = automatic: the thin kernel where it measured
                                        faster on GB300, min(M, N) <= 64 with max(M, N) >= 4096 and
                                        K >= 2048, and only while every option that shapes the
                                        square kernel (PIPELINE, CTA_GROUP, PERSISTENT, ACC_BUFFERS,
                                        SETMAXNREG, STAGES, EPILOGUE, MAX_CTAS, STAGE_GROUP,
                                        EPI_SCHEDULE, SCHEDULER) is at its default;
                                        2 = the thin kernel whenever min(M, N) <= 64;
                                        0 = never */
    GEMM_BF16_OPT_THIN_CLUSTER = 22   /* How the thin kernel splits its work.  Across the SMs: the
                                        (tile, k-block) units in one contiguous range per SM, split
                                        tiles summed through the workspace.  Or one tile per
                                        thread-block cluster of C CTAs: the CTAs split the tile's
                                        k-blocks, and rank 0 adds the others' fp32 partials, read
                                        from their shared memory, in rank order (C = 1: one CTA per
                                        whole tile, nothing to add).  Both orders are fixed, so
                                        results do not depend on timing.
                                        1 (default) = automatic: clusters of the largest C <= 8 with
                                        tiles * C <= SMs whose clusters are all resident at once,
                                        when tiles * C reaches 60 % of the SMs and each CTA streams
                                        at most 160 k-blocks (short decode-like problems, where the
                                        split tiles' traffic through global memory cost more than
                                        the idle SMs); else across the SMs;
                                        2..8 = clusters of this size (at most the k-blocks),
                                        UNSUPPORTED if none can be resident;
                                        0 = always across the SMs */
} gemm_bf16_option;

/* What a plan resolved to (filled by gemm_bf16_plan_info). */
typedef struct gemm_bf16_plan_info_s {
    int64_t tiles;                /* output tiles (one per CTA pair in 2-CTA mode) */
    int64_t k_blocks;             /* 64-wide k-blocks per tile */
    int32_t grid_ctas;            /* CTAs per launch */
    int32_t threads_per_cta;
    int32_t cta_group;            /* 1 or 2 */
    int32_t pipeline;             /* gemm_bf16_pipeline */
    int32_t persistent;
    int32_t stages;               /* stage-ring depth */
    int32_t acc_buffers;
    int32_t setmaxnreg;
    int32_t tile_m;               /* rows of D per tile */
    int32_t tile_n;               /* columns of D per tile */
    int32_t tile_k;               /* k per stage */
    int32_t smem_bytes;           /* dynamic shared memory per CTA */
    int32_t num_sms;
    int32_t epilogue_tma_allowed; /* 1 if ldd permits the TMA-store epilogue */
    int32_t raster_group;
    int32_t regs_per_thread;      /* registers per thread the kernel is launched with */
    int32_t stage_group;          /* ring stages released per commit */
    int32_t sk_tiles;             /* tiles split along k (stream-K); 0 = none */
    int32_t epi_schedule;         /* 0 = cooperative, 1 = ping-pong */
    int32_t scheduler;            /* 0 = static, 1 = dynamic */
    int32_t repack;               /* operands copied to an aligned pitch: bit 0 = A, bit 1 = B */
    int32_t packed_ld;            /* their pitch in elements (K rounded up to 64); 0 = none */
    int32_t k_order;              /* 0 = ascending, 1 = alternating */
    int32_t serpentine;           /* 1 = odd tile bands walk right to left */
    int32_t sk_head;              /* > 0: every tile split at this k-block (head/tail stream-K) */
    int32_t sk_slots;             /* fp32 partial slots (128 x 256 each) the workspace holds */
    int32_t thin;                 /* the thin kernel's small-operand width (16, 32, 48 or 64); 0 = the
                                     square kernel.  Then tile_m = 128 rows of the large operand,
                                     tile_n = thin, and tiles counts the large operand's tiles */
    int32_t thin_cluster;         /* thin kernel: 0 = units split across the SMs; else CTAs per tile
                                     (1 = whole tiles, >= 2 = a cluster; GEMM_BF16_OPT_THIN_CLUSTER) */
} gemm_bf16_plan_info_t;

/* Creates a handle bound to CUDA device `device` (-1 = the calling thread's
 * current device).  Allocates the handle (host) and 16 bytes of device memory:
 * the status word that the kernels' watchdog writes and the dynamic
 * scheduler's tile counter.  Fails with UNSUPPORTED unless the device
 * is compute capability 10.3 (sm_103), with CUDA if no device is usable.
 * On success *out owns both allocations until gemm_bf16_destroy. */
GEMM_BF16_API int gemm_bf16_create(int device, gemm_bf16_t *out);

/* Frees the handle.  Waits for nothing: the caller must not destroy a handle
 * whose launches are still running.  NULL is accepted (no-op). */
GEMM_BF16_API int gemm_bf16_destroy(gemm_bf16_t h);

/* Sets one option (gemm_bf16_option) for the next gemm_bf16_plan.
 * INVALID_ARG for an unknown key or a value outside the documented range. */
GEMM_BF16_API int gemm_bf16_set_option(gemm_bf16_t h, int key, int64_t value);
GEMM_BF16_API int gemm_bf16_get_option(gemm_bf16_t h, int key, int64_t *value);

/* Host-only validation of a problem shape, shared by gemm_bf16_plan and usable
 * without a GPU.  INVALID_ARG: M, N or K < 1 or > 2^31-1, lda < K, ldb < K or
 * ldd < N.  ALIGNMENT: lda*2 or ldb*2 not a multiple of 16 bytes (every row of
 * a TMA-loaded operand must start 16-byte aligned).  ldd may be any value >= N. */
GEMM_BF16_API int gemm_bf16_check_problem(int64_t M, int64_t N, int64_t K,
                                          int64_t lda, int64_t ldb, int64_t ldd);

/* Validates the problem (as gemm_bf16_check_problem), resolves the options,
 * and picks the kernel (the square SM-pair kernel, or the thin kernel of
 * GEMM_BF16_OPT_THIN), stage count, tile order and grid.  Allocates (or grows)
 * the handle's device scratch the plan needs: the stream-K workspace, the thin
 * kernel's partials and tile counters, the packed operand copies.  Re-planning
 * a handle is allowed and replaces the previous plan.  Launches nothing. */
GEMM_BF16_API int gemm_bf16_plan(gemm_bf16_t h, int64_t M, int64_t N, int64_t K,
                                 int64_t lda, int64_t ldb, int64_t ldd);

/* Fills *info from the current plan (NOT_PLANNED before one). */
GEMM_BF16_API int gemm_bf16_plan_info(gemm_bf16_t h, gemm_bf16_plan_info_t *info);

/* Enqueues D = A * B^T on `stream` and returns without synchronising.
 * Launches of one handle share its device scratch (stream-K workspace, tile
 * counter, thin-kernel partials, flags and epoch, packed operand copies): do
 * not let two launches of the same handle run at the same time (e.g. on two
 * streams without an ordering between them); use one handle per stream
 * instead.  When the plan repacks an operand
 * (plan_info.repack) a copy kernel runs on `stream` before the GEMM.
 *   A: device, M rows of lda bf16 (first K read);  B: device, N rows of ldb;
 *   D: device, M rows of ldd bf16 -- only the M x N sub-matrix is written.
 * A and B must be 16-byte aligned (ALIGNMENT otherwise), D 2-byte aligned.
 * The TMA tensor maps are rebuilt only when a pointer differs from the last run.
 * Argument errors are returned before anything is enqueued; a launch failure
 * returns CUDA.  A watchdog timeout inside the kernel is reported later by
 * gemm_bf16_device_status.  The call may be captured into a CUDA graph (plan
 * outside the capture: planning may allocate).  While `stream` is capturing,
 * a plan that splits tiles also enqueues a clear of its split-tile flags
 * before the launch, so that every replay of the graph waits for its own
 * partial sums. */
GEMM_BF16_API int gemm_bf16_run(gemm_bf16_t h, const void *A, const void *B, void *D,
                                void *stream);

/* Fused-epilogue variant:
 *     D[m][n] = bf16( alpha * sum_k A[m][k] * B[n][k] + beta * C[m][n] + bias[n] )
 * computed in fp32 in the epilogue and rounded once to bf16 (Fuser issue #3941,
 * Pseudo-code: the epilogue is where the fp32 sums are converted and stored, the
 * one place a GEMM fuses element-wise work).
 *   C    : device, M rows of ldc bf16 (ldc >= N), or NULL (then beta is ignored);
 *          C may be D itself (ldc == ldd) for an in-place D = alpha*AB^T + beta*D;
 *          16-byte-aligned rows (C base and ldc*2) load as vectors, other layouts
 *          element by element.
 *   bias : device, N bf16 values broadcast over rows, or NULL.
 * Same planning, layouts and error rules as gemm_bf16_run; additionally
 * INVALID_ARG if ldc < N, ALIGNMENT if C or bias is not 2-byte aligned. */
GEMM_BF16_API int gemm_bf16_run_fused(gemm_bf16_t h, const void *A, const void *B, void *D,
                                      const void *C, int64_t ldc, const void *bias,
                                      float alpha, float beta, void *stream);

/* End-to-end variant with HOST operands: enqueues on `stream` the copies
 * hA -> dA and hB -> dB (the M x K and N x K sub-matrices, row pitches lda and
 * ldb), the GEMM on dA, dB, dD, and the copy of the M x N result dD -> hD (row
 * pitch ldd).  Returns without synchronising; page-locked host buffers make the
 * copies asynchronous.  The caller owns all six buffers. */
GEMM_BF16_API int gemm_bf16_run_host(gemm_bf16_t h, const void *hA, const void *hB, void *hD,
                                     void *dA, void *dB, void *dD, void *stream);

/* Synchronises the stream of the last run, reads and clears the device status
 * word.  Returns OK, or DEVICE_TIMEOUT if a kernel's bounded wait ran out since
 * the last call (then *detail, if not NULL, receives the recorded word: bit 31
 * set, bits 24..27 the waiting role, bits 12..23 the CTA, bits 0..11 the ring
 * stage or buffer). */
GEMM_BF16_API int gemm_bf16_device_status(gemm_bf16_t h, uint32_t *detail);

/* GEMM for callers that cannot allocate device memory (no counterpart in the
 * pages: this is a property of the library's interface, not of the method).
 * Runtimes whose pool owns all device memory, and loops that cannot afford an
 * allocation's synchronisation, cannot call gemm_bf16_create (it allocates);
 * they call this instead.  It keeps no handle: it computes D = A * B^T with
 * the same arguments, alignment rules and kernel (SM-pair tiles, deepest ring,
 * persistent grid, grouped serpentine raster, alternating k direction) as
 * gemm_bf16_run with the default options, with A, B, D and the stream
 * supplied by the caller, and allocates nothing -- no cudaMalloc, cudaFree or
 * allocating library call.  Parts of the default plan it leaves out: stream-K
 * (it needs a partials workspace; every tile runs whole), operand repacking (it
 * needs a packed copy; a row pitch that is not a multiple of 128 bytes is read
 * in place, at the slower rate), the thin kernel (it needs a partials
 * workspace; decode-like shapes run on the square kernel), and the
 * programmatic-dependent-launch attribute (the launch waits for the previous
 * work on the stream to finish before its prologue starts).  Its results
 * differ from gemm_bf16_run's only in the fp32 summation order of the tiles
 * that gemm_bf16_run splits (exact whenever every partial sum is).
 *
 * Its scratch (the kernel watchdog's status word, 4 bytes) lives in a fixed
 * 256-byte device array inside the library that every GPU loading the library
 * holds until the process exits.  A call needing more scratch than that array
 * is refused with INVALID_ARG before anything is enqueued.  Every call shares
 * the array: each call clears the status word on `stream` before its launch,
 * so calls that overlap on the GPU (different streams, or threads) race on it.
 *
 * `status` may be NULL.  Otherwise it must point to page-locked host memory
 * (cudaHostAlloc / cudaHostRegister) or to device memory: the status word
 * after the kernel (0 = fine, else the watchdog word described at
 * gemm_bf16_device_status) is copied there on `stream`, asynchronously, and is
 * valid once the stream has synchronised.  Pageable host memory would turn
 * that copy into one that blocks the calling thread until the GEMM is done,
 * so it is refused with INVALID_ARG before anything is enqueued.
 *
 * The first call on each device (with that device current) does a one-time
 * set-up: it looks up the array's device address, sets the kernel's shared-
 * memory limit and sizes the persistent grid.  Make that first call before any
 * stream capture.  Uses the calling thread's current device. */
GEMM_BF16_API int gemm_bf16_run_noalloc(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                        int64_t ldd, const void *A, const void *B, void *D,
                                        void *stream, uint32_t *status);

/* Static, never-NULL description of a status code. */
GEMM_BF16_API const char *gemm_bf16_strerror(int status);

/* Library version string, e.g. "gemm_bf16 1.0 sm_103a". */
GEMM_BF16_API const char *gemm_bf16_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_BF16_H */
