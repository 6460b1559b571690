// Host side of the C ABI declared in include/gemm_bf16.h: handle and options,
// problem validation, plan (kernel variant, ring depth, grid), TMA tensor-map
// encoding, launch, the host-operand end-to-end call and the watchdog status.
#include "gemm_bf16.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "gemm_kernels.h"
#include "thin_split.h"

using namespace wstma;

namespace {

constexpr int kNumOptions = 23;
constexpr int64_t kMaxDim = 0x7FFFFFFFLL;
constexpr uint64_t kWatchdogNsPerKBlock = 2000;  // lower bound of the watchdog limit per k-block of K

struct Plan {
    bool valid = false;
    int64_t M = 0, N = 0, K = 0, lda = 0, ldb = 0, ldd = 0;
    int pipeline = GEMM_BF16_PIPE_WS;
    int cta_group = 1;
    int persistent = 1;
    int acc_buffers = 2;
    int stage_group = 1;
    int sk_tiles = 0;
    int sk_head = 0;        // > 0: head/tail stream-K (fewer tiles than clusters)
    int sk_pieces = 0;      // workspace slots per contributing cluster
    int64_t sk_units = 0;   // units divided among the clusters' ranges
    size_t sk_slots = 0;    // partial slots (per CTA) the workspace must hold
    int setmaxnreg = 0;
    int stages = 0;
    int raster_group = 8;
    int epilogue_opt = 0;
    int epi_pingpong = 0;
    int sched_dynamic = 0;
    int k_order = 0;
    int serpentine = 0;
    bool repack_a = false, repack_b = false;  // operands copied to a 128-byte-multiple pitch first
    int64_t ldp = 0;                          // that pitch in elements
    int thin_nt = 0;                          // > 0: the thin kernel, small-operand width 16..64
    bool thin_transposed = false;             // thin kernel: the large operand is B
    int64_t thin_units = 0;                   // thin kernel: tiles * k-blocks
    int thin_push = 0;                        // thin cluster form: partials stored into rank 0
    int thin_cluster = 0;                     // thin kernel: 0 = units split across the SMs, else
                                              // CTAs per tile (1 = whole tiles, > 1 = a cluster)
    int64_t tiles = 0;
    int num_m_blocks = 0, num_n_blocks = 0, num_k_blocks = 0;
    int grid_ctas = 0;
    int threads = 0;
    size_t smem = 0;
    int regs = 0;
    const void *fn = nullptr;
    bool epi_tma_allowed = false;
    int fault_skip = -1;
    uint64_t watchdog_ns = 1000000000ull;
};

}  // namespace

struct gemm_bf16 {
    int device = 0;
    int num_sms = 0;
    size_t max_smem_optin = 0;
    // device words: [0] watchdog status, [1] unused, [2] dynamic scheduler's next
    // whole tile, [3] clusters finished (both 0 between launches)
    uint32_t *d_err = nullptr;
    int64_t opt[kNumOptions];
    Plan plan;
    // tensor-map cache
    bool maps_valid = false;
    const void *mA = nullptr;
    const void *mB = nullptr;
    void *mD = nullptr;
    CUtensorMap tmA, tmB, tmD;
    cudaStream_t last_stream = nullptr;
    // stream-K workspace (partials + flags), grown on demand by plan
    float *ws = nullptr;
    uint32_t *ws_flags = nullptr;
    size_t ws_slots = 0;
    uint32_t epoch = 0;
    // packed operand copies (A then B), grown on demand by plan
    void *pack = nullptr;
    size_t pack_bytes = 0;
    // thin kernel's partials and their flags (grown on demand by plan) and
    // its device-side epoch and arrival count (allocated once)
    float *thin_ws = nullptr;
    size_t thin_ws_floats = 0;
    uint32_t *thin_flags = nullptr;
    size_t thin_flags_n = 0;
    uint32_t *thin_sync = nullptr;
};

namespace {

int64_t default_option(int key)
{
    switch (key) {
    case GEMM_BF16_OPT_PIPELINE: return GEMM_BF16_PIPE_WS;
    case GEMM_BF16_OPT_CTA_GROUP: return 0;
    case GEMM_BF16_OPT_PERSISTENT: return 1;
    case GEMM_BF16_OPT_ACC_BUFFERS: return 2;
    case GEMM_BF16_OPT_SETMAXNREG: return 0;
    case GEMM_BF16_OPT_STAGES: return 0;
    case GEMM_BF16_OPT_RASTER_GROUP: return 8;
    case GEMM_BF16_OPT_EPILOGUE: return 0;
    case GEMM_BF16_OPT_MAX_CTAS: return 0;
    case GEMM_BF16_OPT_WATCHDOG_NS: return 1000000000LL;
    case GEMM_BF16_OPT_FAULT_SKIP_LOAD: return -1;
    case GEMM_BF16_OPT_STAGE_GROUP: return 0;
    case GEMM_BF16_OPT_STREAM_K: return 1;
    case GEMM_BF16_OPT_PDL: return 1;
    case GEMM_BF16_OPT_EPI_SCHEDULE: return 0;
    case GEMM_BF16_OPT_SCHEDULER: return 0;
    case GEMM_BF16_OPT_REPACK: return 0;
    case GEMM_BF16_OPT_K_ORDER: return 1;
    case GEMM_BF16_OPT_SERPENTINE: return 1;
    case GEMM_BF16_OPT_FAULT_TENSORMAP: return 0;
    case GEMM_BF16_OPT_THIN: return 1;
    case GEMM_BF16_OPT_THIN_CLUSTER: return 1;
    default: return 0;
    }
}

bool option_in_range(int key, int64_t v)
{
    switch (key) {
    case GEMM_BF16_OPT_PIPELINE: return v >= 0 && v <= 2;
    case GEMM_BF16_OPT_CTA_GROUP: return v >= 0 && v <= 2;
    case GEMM_BF16_OPT_PERSISTENT: return v == 0 || v == 1;
    case GEMM_BF16_OPT_ACC_BUFFERS: return v == 1 || v == 2;
    case GEMM_BF16_OPT_SETMAXNREG: return v == 0 || v == 1;
    case GEMM_BF16_OPT_STAGES: return v >= 0 && v <= kMaxStages;
    case GEMM_BF16_OPT_RASTER_GROUP: return v >= 0 && v <= 4096;
    case GEMM_BF16_OPT_EPILOGUE: return v >= 0 && v <= 2;
    case GEMM_BF16_OPT_MAX_CTAS: return v >= 0 && v <= (1 << 20);
    case GEMM_BF16_OPT_WATCHDOG_NS: return v >= 1000 && v <= 600LL * 1000000000LL;
    case GEMM_BF16_OPT_FAULT_SKIP_LOAD: return v >= -1 && v <= kMaxDim;
    case GEMM_BF16_OPT_STAGE_GROUP: return v >= 0 && v <= 2;
    case GEMM_BF16_OPT_STREAM_K: return v >= 0 && v <= 3;
    case GEMM_BF16_OPT_PDL: return v == 0 || v == 1;
    case GEMM_BF16_OPT_EPI_SCHEDULE: return v == 0 || v == 1;
    case GEMM_BF16_OPT_SCHEDULER: return v == 0 || v == 1;
    case GEMM_BF16_OPT_REPACK: return v >= 0 && v <= 2;
    case GEMM_BF16_OPT_K_ORDER: return v == 0 || v == 1;
    case GEMM_BF16_OPT_SERPENTINE: return v == 0 || v == 1;
    case GEMM_BF16_OPT_FAULT_TENSORMAP: return v == 0 || v == 1;
    case GEMM_BF16_OPT_THIN: return v >= 0 && v <= 2;
    case GEMM_BF16_OPT_THIN_CLUSTER: return v >= 0 && v <= kThinMaxCluster;
    default: return false;
    }
}

// Head/tail stream-K for T tiles of KB k-blocks on up to C clusters (T < C):
// cluster t < T computes k-blocks [0, H) of tile t (the head) and owns the
// tile, and n more clusters share the T * (KB - H) tail k-blocks in
// contiguous ranges of `share` k-blocks.  Times are in k-blocks of one SM
// pair's MMA time (~0.3 us); the constants were measured on GB300 with
// clock-stamped timelines of the kernel:
//  - a tail k-block takes kTailWeight % of a head k-block (tail slices have
//    fewer concurrent readers, so more of them come from DRAM);
//  - after its last MMA a tail range needs kTailEnd to store its fp32
//    partial (128 KiB per CTA) and raise its flag;
//  - an owner folds each partial into a spare tensor-memory accumulator as it
//    arrives; one that arrives at the end costs it kFold;
// so the owner's epilogue can start at H when
//   H >= w * share + kTailEnd + kFold * (most ranges reaching into one tile),
// which fixes H for each n.  A range that covers more than two tiles stores a
// partial per tile while it computes the next; with tails shorter than
// kMinPiece k-blocks those stores hold its MMAs back (2048 x 2048 x 8192,
// 14-k-block tails: 18% slower than whole tiles), so such layouts are not
// used.  The n with the least H is chosen, and the split is taken when H beats
// a whole tile by >= kMinSaving.
struct HeadTail {
    int64_t head = 0, n = 0, units = 0, pieces = 0;
};

// For tails of L k-blocks cut into n ranges: the most ranges that reach into
// one tile, and the most tiles one range reaches into.
void tail_layout(int64_t T, int64_t L, int64_t n, std::vector<int32_t> &cnt, int64_t *most, int64_t *pieces)
{
    const int64_t U = T * L;
    std::fill(cnt.begin(), cnt.end(), 0);
    *most = 0;
    *pieces = 1;
    for (int64_t j = 0; j < n; ++j) {
        const int64_t b = j * U / n, e = (j + 1) * U / n;
        if (e <= b)
            continue;
        *pieces = std::max<int64_t>(*pieces, (e - 1) / L - b / L + 1);
        for (int64_t t = b / L; t <= (e - 1) / L; ++t)
            *most = std::max<int64_t>(*most, ++cnt[(size_t)t]);
    }
}

bool choose_head_tail(int64_t T, int64_t KB, int64_t C, bool forced, HeadTail *out)
{
    constexpr int64_t kTailWeight = 125;
    constexpr int64_t kTailEnd = 15;
    constexpr int64_t kFold = 6;
    constexpr int64_t kMinPiece = 24;
    constexpr int64_t kMinSaving = 8;
    // forced: every cluster takes part, whatever the gain
    int64_t best = forced ? INT64_MAX : KB - kMinSaving + 1;
    bool found = false;
    std::vector<int32_t> cnt((size_t)T);
    for (int64_t n = forced ? C - T : 1; n <= C - T; ++n) {
        const int64_t den = 100 * n + kTailWeight * T;
        // balance without the end costs first, to count the ranges per tile
        const int64_t h0 = (kTailWeight * T * KB + den - 1) / den;
        if (h0 >= KB)
            continue;
        int64_t most, pieces;
        tail_layout(T, KB - h0, n, cnt, &most, &pieces);
        int64_t head = (kTailWeight * T * KB + 100 * n * (kTailEnd + kFold * most) + den - 1) / den;
        head = std::min<int64_t>(head, KB - 1);
        tail_layout(T, KB - head, n, cnt, &most, &pieces);
        if (!forced && pieces > 2 && KB - head < kMinPiece)
            continue;
        if (head < best) {
            best = head;
            out->head = head;
            out->n = n;
            out->units = T * (KB - head);
            out->pieces = pieces;
            found = true;
        }
    }
    return found;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 tensor map: `cols` contiguous elements per row, `rows` rows,
// `row_bytes` between rows; box = box_cols x box_rows, with 128-byte swizzling
// unless `swizzle` is false (then the box is plain row-major in shared memory);
// out-of-bounds elements of a load read as zero, those of a store are dropped.
int encode_2d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint64_t row_bytes, uint32_t box_cols,
              uint32_t box_rows, bool swizzle = true)
{
    auto fn = encode_fn();
    if (!fn)
        return GEMM_BF16_ERR_TENSORMAP;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_BF16_OK : GEMM_BF16_ERR_TENSORMAP;
}

int set_device(gemm_bf16_t h)
{
    return cudaSetDevice(h->device) == cudaSuccess ? GEMM_BF16_OK : GEMM_BF16_ERR_CUDA;
}

// The dynamic shared-memory limit is an attribute of the kernel function, shared
// by every handle: it is raised to the device's opt-in maximum (not to this
// plan's size), so plans of other handles with deeper rings still launch.
int prepare_kernel(const void *fn, size_t max_smem, int *regs)
{
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, fn) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    *regs = a.numRegs;
    return GEMM_BF16_OK;
}

// The square kernel's plan: CTA mode, ring depth, kernel variant, persistent
// grid and stream-K split (with its workspace).
int plan_square(gemm_bf16_t h, Plan &pl)
{
    const int64_t M = pl.M, N = pl.N, K = pl.K;
    int rc;
    int cg = (int)h->opt[GEMM_BF16_OPT_CTA_GROUP];
    const bool ws = pl.pipeline == GEMM_BF16_PIPE_WS;
    if (!ws) {
        if (cg == 2)
            return GEMM_BF16_ERR_UNSUPPORTED;  // the ablation loops are single-CTA
        cg = 1;
        pl.persistent = 0;
        pl.acc_buffers = 1;
        pl.setmaxnreg = 0;
        pl.epi_pingpong = 0;
        pl.sched_dynamic = 0;
        pl.k_order = 0;
    } else if (cg == 0) {
        // An SM pair per 256x256 tile halves each SM's operand traffic.  Problems
        // of at most 512^3 multiply-adds are bound by fixed latency instead, and
        // the single-CTA kernel (no cluster barriers, half the epilogue per CTA)
        // measured faster there: 256^3 10.8 against 12.1 us, 512^3 12.3 against
        // 12.7 us, with L2 flushed (1024^3: 16.4 against 16.0).
        cg = (M * N <= (int64_t)512 * 512 && M * N * K <= (int64_t)512 * 512 * 512) ? 1 : 2;
    }
    pl.cta_group = cg;
    if (pl.epi_pingpong && pl.acc_buffers != 2)
        return GEMM_BF16_ERR_INVALID_ARG;  // each epilogue warpgroup owns one accumulator

    pl.num_m_blocks = (int)((M + (int64_t)kBlockM * cg - 1) / ((int64_t)kBlockM * cg));
    pl.num_n_blocks = (int)((N + kBlockN - 1) / kBlockN);
    pl.num_k_blocks = (int)((K + kBlockK - 1) / kBlockK);
    // No in-kernel wait lasts longer than about one tile's k-range of MMAs (the
    // epilogue waiting for an accumulator, an owner for a partial), ~0.3 us per
    // k-block on GB300: a limit of 2 us per k-block keeps a long-k problem from
    // tripping the watchdog, whatever the limit asked for.
    pl.watchdog_ns = std::max<uint64_t>(pl.watchdog_ns, (uint64_t)pl.num_k_blocks * kWatchdogNsPerKBlock);
    pl.tiles = (int64_t)pl.num_m_blocks * pl.num_n_blocks;
    if (pl.tiles > kMaxDim / 2)
        return GEMM_BF16_ERR_INVALID_ARG;

    // ring depth: as deep as shared memory allows, or the requested depth
    int max_stages = 0;
    for (int s = kMaxStages; s >= 2; --s) {
        const size_t need = ws ? ws_smem_bytes(cg, s) : nows_smem_bytes(s);
        if (need <= h->max_smem_optin) {
            max_stages = s;
            break;
        }
    }
    if (max_stages < 2)
        return GEMM_BF16_ERR_UNSUPPORTED;
    const int req = (int)h->opt[GEMM_BF16_OPT_STAGES];
    if (req > max_stages || req == 1)
        return GEMM_BF16_ERR_INVALID_ARG;
    pl.stages = req ? req : max_stages;
    // k-blocks released per commit (WS only): 0 = automatic = 1 (measured
    // fastest once the MMA issuer's probe is a try_wait; pairing stages costs
    // ring slack)
    const int g = (int)h->opt[GEMM_BF16_OPT_STAGE_GROUP];
    if (!ws || g == 0) {
        pl.stage_group = 1;
    } else {
        if (pl.stages % g != 0)
            return GEMM_BF16_ERR_INVALID_ARG;
        pl.stage_group = g;
    }
    pl.smem = ws ? ws_smem_bytes(cg, pl.stages) : nows_smem_bytes(pl.stages);

    if (ws) {
        pl.fn = cg == 2 ? ws_kernel_c2(pl.setmaxnreg != 0) : ws_kernel_c1(pl.setmaxnreg != 0);
        pl.threads = kWsThreads;
    } else {
        pl.fn = nows_kernel(pl.pipeline == GEMM_BF16_PIPE_MBAR_WAR);
        pl.threads = kNowsThreads;
    }
    if ((rc = prepare_kernel(pl.fn, h->max_smem_optin, &pl.regs)) != GEMM_BF16_OK)
        return rc;
    // setmaxnreg.inc can only hand out registers the CTA was launched with.
    if (ws && pl.setmaxnreg &&
        pl.regs * kWsThreads < kProducerRegs * 128 + kConsumerRegs * (kWsThreads - 128))
        return GEMM_BF16_ERR_UNSUPPORTED;

    // grid
    const int64_t max_ctas = h->opt[GEMM_BF16_OPT_MAX_CTAS];
    pl.sk_tiles = 0;
    pl.sk_head = 0;
    pl.sk_pieces = 0;
    pl.sk_units = 0;
    pl.sk_slots = 0;
    if (!ws || !pl.persistent) {
        pl.grid_ctas = (int)(pl.tiles * cg);
    } else {
        int64_t slots;
        if (cg == 1) {
            slots = h->num_sms;
        } else {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3((unsigned)(2 * std::max<int64_t>(1, h->num_sms / 2)), 1, 1);
            cfg.blockDim = dim3(kWsThreads, 1, 1);
            cfg.dynamicSmemBytes = pl.smem;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, pl.fn, &cfg) != cudaSuccess || clusters < 1) {
                cudaGetLastError();
                clusters = h->num_sms / 2;
            }
            slots = (int64_t)clusters * 2;
        }
        if (max_ctas > 0)
            slots = std::min<int64_t>(slots, std::max<int64_t>(cg, (max_ctas / cg) * cg));
        pl.grid_ctas = (int)std::min<int64_t>(pl.tiles * cg, slots);
        // Stream-K for the tiles that would run as a partial last wave: their
        // k-blocks are split evenly over every resident cluster, and the other
        // tiles run whole.  Only when there is at least one whole wave (with
        // fewer tiles than clusters every tile would be split, the clusters that
        // share A/B panels would sit at different k offsets, and the L2 reuse
        // is lost: measured 19% slower on 2048x2048x32768) and each cluster
        // gets >= 4 k-blocks of the split work.
        const int64_t clusters = slots / cg;
        const int64_t rem = pl.tiles % clusters;
        const int64_t sk_opt = h->opt[GEMM_BF16_OPT_STREAM_K];
        const int64_t KB = pl.num_k_blocks;
        if (sk_opt && pl.tiles >= clusters && rem != 0 && rem * KB >= 4 * clusters) {
            pl.sk_tiles = (int)rem;
            pl.sk_units = rem * KB;
            pl.sk_pieces = 1;
            pl.sk_slots = (size_t)(clusters * cg);
            pl.grid_ctas = (int)(clusters * cg);
        } else if ((sk_opt == 1 || sk_opt == 3) && pl.tiles < clusters) {
            // Head/tail form: every tile is split at the same k-block H, so the
            // tiles' owners all start at k-block 0 and walk k in step (the A and
            // B panels they share are read from DRAM once, as with whole tiles),
            // while n of the clusters that would idle share the tails.
            HeadTail ht;
            if (choose_head_tail(pl.tiles, KB, clusters, sk_opt == 3, &ht)) {
                pl.sk_tiles = (int)pl.tiles;
                pl.sk_head = (int)ht.head;
                pl.sk_units = ht.units;
                pl.sk_pieces = (int)ht.pieces;
                pl.sk_slots = (size_t)(ht.n * ht.pieces * cg);
                pl.grid_ctas = (int)((pl.tiles + ht.n) * cg);
            }
        }
    }
    if (!ws && max_ctas > 0)
        return GEMM_BF16_ERR_UNSUPPORTED;  // one tile per CTA: the grid is fixed by the problem
    if (pl.sk_tiles > 0 && pl.sk_slots > h->ws_slots) {
        // one partial slot (128 x 256 fp32) and one flag per contributor CTA and
        // piece; flags start at 0 and every launch waits for its own epoch, so
        // they are never reset
        float *nws = nullptr;
        uint32_t *nflags = nullptr;
        if (cudaMalloc(&nws, pl.sk_slots * kPartialFloats * sizeof(float)) != cudaSuccess ||
            cudaMalloc(&nflags, pl.sk_slots * sizeof(uint32_t)) != cudaSuccess ||
            cudaMemset(nflags, 0, pl.sk_slots * sizeof(uint32_t)) != cudaSuccess) {
            cudaGetLastError();
            if (nws)
                cudaFree(nws);
            if (nflags)
                cudaFree(nflags);
            return GEMM_BF16_ERR_CUDA;
        }
        if (h->ws)
            cudaFree(h->ws);
        if (h->ws_flags)
            cudaFree(h->ws_flags);
        h->ws = nws;
        h->ws_flags = nflags;
        h->ws_slots = pl.sk_slots;
    }
    return GEMM_BF16_OK;
}

// How many clusters of c thin-kernel CTAs can be resident at once (0 if none).
int thin_max_active_clusters(const void *fn, int c, size_t smem, int threads)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)c, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// The thin kernel's plan (gemm_thin.cuh): the large operand in 128-row tiles,
// the small one as the MMA's N side, one CTA per SM, the (tile, k-block) units
// split evenly, and the workspace for the split tiles' partials.
int plan_thin(gemm_bf16_t h, Plan &pl)
{
    int rc;
    // the small operand is B when N is small enough (D's rows are then the
    // accumulator's rows), else A (D is the accumulator transposed)
    const bool transposed = pl.N > kThinMaxRows;
    const int64_t small = transposed ? pl.M : pl.N;
    const int64_t large = transposed ? pl.N : pl.M;
    pl.thin_nt = thin_nt(small);
    pl.thin_transposed = transposed;
    pl.pipeline = GEMM_BF16_PIPE_WS;
    pl.cta_group = 1;
    pl.persistent = 1;
    pl.acc_buffers = 2;
    pl.setmaxnreg = 0;
    pl.stage_group = 1;
    pl.epi_pingpong = 0;
    pl.sched_dynamic = 0;
    pl.k_order = 0;
    pl.serpentine = 0;
    pl.raster_group = 0;
    pl.num_k_blocks = (int)((pl.K + kBlockK - 1) / kBlockK);
    pl.tiles = (large + kBlockM - 1) / kBlockM;
    pl.num_m_blocks = (int)pl.tiles;
    pl.num_n_blocks = 1;
    pl.thin_units = pl.tiles * pl.num_k_blocks;
    pl.watchdog_ns = std::max<uint64_t>(pl.watchdog_ns, (uint64_t)pl.num_k_blocks * kWatchdogNsPerKBlock);
    pl.stages = 0;
    for (int s = kThinMaxStages; s >= 2; --s)
        if (thin_smem_bytes(pl.thin_nt, s) <= h->max_smem_optin) {
            pl.stages = s;
            break;
        }
    if (pl.stages < 2)
        return GEMM_BF16_ERR_UNSUPPORTED;
    pl.smem = thin_smem_bytes(pl.thin_nt, pl.stages);
    pl.fn = thin_kernel(pl.thin_nt);
    pl.threads = kThinThreads;
    if ((rc = prepare_kernel(pl.fn, h->max_smem_optin, &pl.regs)) != GEMM_BF16_OK)
        return rc;
    // Across the SMs, or one tile per cluster of C CTAs (gemm_thin.cuh).  The
    // cluster form leaves SMs idle when tiles * C < SMs but has no split-tile
    // traffic through global memory; on GB300 it was faster where tiles * C
    // reaches ~60 % of the SMs and each CTA streams at most ~160 k-blocks
    // (16x8192x8192: 28.9 -> ~26 us; 16x4096x8192: 14.7 -> ~11 us), slower on
    // long runs (16x16384x16384, one CTA per tile: 91 -> 95 us).
    const int64_t copt = h->opt[GEMM_BF16_OPT_THIN_CLUSTER];
    const int64_t T = pl.tiles, KB = pl.num_k_blocks;
    pl.thin_cluster = 0;
    if (copt >= 2) {
        pl.thin_cluster = (int)std::min<int64_t>(copt, KB);
        if (pl.thin_cluster > 1 && thin_max_active_clusters(pl.fn, pl.thin_cluster, pl.smem, pl.threads) < 1)
            return GEMM_BF16_ERR_UNSUPPORTED;
    } else if (copt == 1 && T <= h->num_sms) {
        int32_t resident[kThinMaxCluster + 1] = {0};
        resident[1] = h->num_sms;  // one CTA per SM
        for (int c = 2; c <= kThinMaxCluster && c <= KB && c * T <= h->num_sms; ++c)
            resident[c] = thin_max_active_clusters(pl.fn, c, pl.smem, pl.threads);
        pl.thin_cluster = thin_auto_cluster(T, KB, h->num_sms, resident);
    }
    pl.grid_ctas = pl.thin_cluster > 0
                       ? (int)(T * pl.thin_cluster)
                       : (int)std::min<int64_t>(std::min<int64_t>(h->num_sms, kThinMaxGrid), pl.thin_units);
    // In the cluster form the other ranks store their partials into rank 0's
    // shared memory (no remote reads at the end of the launch), in a receive
    // area beside the ring; the ring gives up stages for it, down to 4.  The
    // short per-CTA runs of this form lose less to a shallower ring than to
    // the remote reads: 16x4096x8192 13.36 -> 12.85 us with 11 stages instead
    // of 12, 64x4096x8192 16.17 -> 15.38 us with 5 instead of 9.  Where not
    // even 4 stages fit, rank 0 reads the others' rings.
    pl.thin_push = 0;
    if (pl.thin_cluster > 1) {
        const size_t recv = (size_t)(pl.thin_cluster - 1) * kBlockM * (size_t)pl.thin_nt * sizeof(float);
        int s = pl.stages;
        while (s >= 4 && thin_smem_bytes(pl.thin_nt, s) + recv > h->max_smem_optin)
            --s;
        if (s >= 4) {
            pl.stages = s;
            pl.smem = thin_smem_bytes(pl.thin_nt, s) + recv;
            pl.thin_push = 1;
        }
    }
    pl.sk_tiles = pl.sk_head = pl.sk_pieces = 0;
    pl.sk_units = 0;
    pl.sk_slots = 0;
    // two partial slots per CTA (thin_split.h) of 128 x thin_nt fp32, and a
    // flag per slot and epilogue warp; a flag holds the epoch of the launch
    // that last stored that warp's rows, and the epoch starts at 1 and only
    // grows, so a fresh flag allocation is zeroed and never cleared afterwards
    const size_t floats = (size_t)2 * (size_t)pl.grid_ctas * kBlockM * (size_t)pl.thin_nt;
    if (floats > h->thin_ws_floats) {
        float *nws = nullptr;
        if (cudaMalloc(&nws, floats * sizeof(float)) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_BF16_ERR_CUDA;
        }
        if (h->thin_ws)
            cudaFree(h->thin_ws);
        h->thin_ws = nws;
        h->thin_ws_floats = floats;
    }
    const size_t nflags = (size_t)2 * 4 * (size_t)pl.grid_ctas;
    if (nflags > h->thin_flags_n) {
        uint32_t *nf = nullptr;
        if (cudaMalloc(&nf, nflags * sizeof(uint32_t)) != cudaSuccess ||
            cudaMemset(nf, 0, nflags * sizeof(uint32_t)) != cudaSuccess) {
            cudaGetLastError();
            if (nf)
                cudaFree(nf);
            return GEMM_BF16_ERR_CUDA;
        }
        if (h->thin_flags)
            cudaFree(h->thin_flags);
        h->thin_flags = nf;
        h->thin_flags_n = nflags;
    }
    if (!h->thin_sync) {
        const uint32_t init[2] = {1u, 0u};  // epoch 1, no CTA arrived
        uint32_t *ns = nullptr;
        if (cudaMalloc(&ns, sizeof(init)) != cudaSuccess ||
            cudaMemcpy(ns, init, sizeof(init), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            if (ns)
                cudaFree(ns);
            return GEMM_BF16_ERR_CUDA;
        }
        h->thin_sync = ns;
    }
    return GEMM_BF16_OK;
}

}  // namespace

extern "C" {

GEMM_BF16_API const char *gemm_bf16_strerror(int status)
{
    switch (status) {
    case GEMM_BF16_OK: return "ok";
    case GEMM_BF16_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_BF16_ERR_ALIGNMENT: return "alignment: TMA needs 16-byte aligned bases and row strides";
    case GEMM_BF16_ERR_NOT_PLANNED: return "not planned: call gemm_bf16_plan first";
    case GEMM_BF16_ERR_CUDA: return "a CUDA runtime call failed";
    case GEMM_BF16_ERR_TENSORMAP: return "TMA tensor-map encoding failed";
    case GEMM_BF16_ERR_DEVICE_TIMEOUT: return "device watchdog: a barrier wait ran out and the kernel returned early";
    case GEMM_BF16_ERR_UNSUPPORTED: return "unsupported device or option combination";
    default: return "unknown status";
    }
}

GEMM_BF16_API const char *gemm_bf16_version(void) { return "gemm_bf16 1.0 sm_103a"; }

GEMM_BF16_API int gemm_bf16_check_problem(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldd)
{
    if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return GEMM_BF16_ERR_INVALID_ARG;
    if (lda < K || ldb < K || ldd < N)
        return GEMM_BF16_ERR_INVALID_ARG;
    if (lda > (int64_t(1) << 38) || ldb > (int64_t(1) << 38) || ldd > (int64_t(1) << 38))
        return GEMM_BF16_ERR_INVALID_ARG;
    if ((lda * 2) % 16 != 0 || (ldb * 2) % 16 != 0)
        return GEMM_BF16_ERR_ALIGNMENT;
    return GEMM_BF16_OK;
}

GEMM_BF16_API int gemm_bf16_create(int device, gemm_bf16_t *out)
{
    if (!out)
        return GEMM_BF16_ERR_INVALID_ARG;
    *out = nullptr;
    int dev = device;
    if (dev < 0 && cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || dev >= count) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    if (cudaSetDevice(dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    int major = 0, minor = 0, sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    if (major != 10 || minor != 3)
        return GEMM_BF16_ERR_UNSUPPORTED;
    gemm_bf16_t h = new (std::nothrow) gemm_bf16();
    if (!h)
        return GEMM_BF16_ERR_CUDA;
    h->device = dev;
    h->num_sms = sms;
    h->max_smem_optin = (size_t)optin;
    for (int k = 0; k < kNumOptions; ++k)
        h->opt[k] = default_option(k);
    if (cudaMalloc(&h->d_err, 4 * sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(h->d_err, 0, 4 * sizeof(uint32_t)) != cudaSuccess) {
        cudaGetLastError();
        if (h->d_err)
            cudaFree(h->d_err);
        delete h;
        return GEMM_BF16_ERR_CUDA;
    }
    *out = h;
    return GEMM_BF16_OK;
}

GEMM_BF16_API int gemm_bf16_destroy(gemm_bf16_t h)
{
    if (!h)
        return GEMM_BF16_OK;
    cudaSetDevice(h->device);
    if (h->d_err)
        cudaFree(h->d_err);
    if (h->ws)
        cudaFree(h->ws);
    if (h->ws_flags)
        cudaFree(h->ws_flags);
    if (h->pack)
        cudaFree(h->pack);
    if (h->thin_ws)
        cudaFree(h->thin_ws);
    if (h->thin_flags)
        cudaFree(h->thin_flags);
    if (h->thin_sync)
        cudaFree(h->thin_sync);
    delete h;
    return GEMM_BF16_OK;
}

GEMM_BF16_API int gemm_bf16_set_option(gemm_bf16_t h, int key, int64_t value)
{
    if (!h || key < 1 || key >= kNumOptions || !option_in_range(key, value))
        return GEMM_BF16_ERR_INVALID_ARG;
    h->opt[key] = value;
    return GEMM_BF16_OK;
}

GEMM_BF16_API int gemm_bf16_get_option(gemm_bf16_t h, int key, int64_t *value)
{
    if (!h || !value || key < 1 || key >= kNumOptions)
        return GEMM_BF16_ERR_INVALID_ARG;
    *value = h->opt[key];
    return GEMM_BF16_OK;
}

GEMM_BF16_API int gemm_bf16_plan(gemm_bf16_t h, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                 int64_t ldd)
{
    if (!h)
        return GEMM_BF16_ERR_INVALID_ARG;
    h->plan.valid = false;
    h->maps_valid = false;
    int rc = gemm_bf16_check_problem(M, N, K, lda, ldb, ldd);
    if (rc != GEMM_BF16_OK)
        return rc;
    if ((rc = set_device(h)) != GEMM_BF16_OK)
        return rc;

    Plan pl;
    pl.M = M, pl.N = N, pl.K = K, pl.lda = lda, pl.ldb = ldb, pl.ldd = ldd;
    pl.pipeline = (int)h->opt[GEMM_BF16_OPT_PIPELINE];
    pl.persistent = (int)h->opt[GEMM_BF16_OPT_PERSISTENT];
    pl.acc_buffers = (int)h->opt[GEMM_BF16_OPT_ACC_BUFFERS];
    pl.setmaxnreg = (int)h->opt[GEMM_BF16_OPT_SETMAXNREG];
    pl.raster_group = (int)h->opt[GEMM_BF16_OPT_RASTER_GROUP];
    pl.epilogue_opt = (int)h->opt[GEMM_BF16_OPT_EPILOGUE];
    pl.epi_pingpong = (int)h->opt[GEMM_BF16_OPT_EPI_SCHEDULE];
    pl.sched_dynamic = (int)h->opt[GEMM_BF16_OPT_SCHEDULER];
    pl.k_order = (int)h->opt[GEMM_BF16_OPT_K_ORDER];
    pl.serpentine = (int)h->opt[GEMM_BF16_OPT_SERPENTINE];
    pl.fault_skip = (int)h->opt[GEMM_BF16_OPT_FAULT_SKIP_LOAD];
    pl.watchdog_ns = (uint64_t)h->opt[GEMM_BF16_OPT_WATCHDOG_NS];
    pl.epi_tma_allowed = ((ldd * 2) % 16) == 0;

    // the thin kernel for decode-like shapes, else the square kernel
    const int64_t thin_opt = h->opt[GEMM_BF16_OPT_THIN];
    const bool square_defaults =
        h->opt[GEMM_BF16_OPT_PIPELINE] == GEMM_BF16_PIPE_WS && h->opt[GEMM_BF16_OPT_CTA_GROUP] == 0 &&
        h->opt[GEMM_BF16_OPT_PERSISTENT] == 1 && h->opt[GEMM_BF16_OPT_ACC_BUFFERS] == 2 &&
        h->opt[GEMM_BF16_OPT_SETMAXNREG] == 0 && h->opt[GEMM_BF16_OPT_STAGES] == 0 &&
        h->opt[GEMM_BF16_OPT_EPILOGUE] == 0 && h->opt[GEMM_BF16_OPT_MAX_CTAS] == 0 &&
        h->opt[GEMM_BF16_OPT_STAGE_GROUP] == 0 && h->opt[GEMM_BF16_OPT_EPI_SCHEDULE] == 0 &&
        h->opt[GEMM_BF16_OPT_SCHEDULER] == 0;
    // automatic: where the thin kernel measured faster on GB300, one operand of
    // at most 64 rows against >= 4096 rows of the other with K >= 2048 (4-25 %
    // faster in either orientation; even at 64 x 4096 x 4096); at K = 1024 the
    // square kernel was 20 % faster
    const bool thin_auto_shape = std::max(M, N) >= 4096 && K >= 2048;
    const bool thin = std::min(M, N) <= kThinMaxRows &&
                      (thin_opt == 2 || (thin_opt == 1 && square_defaults && thin_auto_shape));
    if ((rc = thin ? plan_thin(h, pl) : plan_square(h, pl)) != GEMM_BF16_OK)
        return rc;
    // Operand repacking: a row pitch that is not a multiple of 128 bytes makes
    // every TMA box row straddle two L2 lines (~28% slower GEMM, measured).  A
    // copy costs one HBM read + write of the operand, i.e. time ~ rows * K,
    // while the GEMM's saving grows with rows * K * (other dimension): it pays
    // once the other dimension is >= 4096 (automatic mode).
    {
        const int64_t mode = h->opt[GEMM_BF16_OPT_REPACK];
        const bool mis_a = (lda * 2) % 128 != 0, mis_b = (ldb * 2) % 128 != 0;
        pl.repack_a = mis_a && (mode == 1 || (mode == 0 && N >= 4096));
        pl.repack_b = mis_b && (mode == 1 || (mode == 0 && M >= 4096));
        if (pl.repack_a || pl.repack_b) {
            pl.ldp = (K + 63) / 64 * 64;
            const size_t need = (size_t)((pl.repack_a ? M : 0) + (pl.repack_b ? N : 0)) * (size_t)pl.ldp * 2;
            if (need > h->pack_bytes) {
                void *np = nullptr;
                if (cudaMalloc(&np, need) != cudaSuccess) {
                    cudaGetLastError();
                    if (mode == 1)
                        return GEMM_BF16_ERR_CUDA;
                    pl.repack_a = pl.repack_b = false;  // automatic: run on the original pitch
                    pl.ldp = 0;
                } else {
                    if (h->pack)
                        cudaFree(h->pack);
                    h->pack = np;
                    h->pack_bytes = need;
                }
            }
        }
    }
    pl.valid = true;
    h->plan = pl;
    return GEMM_BF16_OK;
}

GEMM_BF16_API int gemm_bf16_plan_info(gemm_bf16_t h, gemm_bf16_plan_info_t *info)
{
    if (!h || !info)
        return GEMM_BF16_ERR_INVALID_ARG;
    if (!h->plan.valid)
        return GEMM_BF16_ERR_NOT_PLANNED;
    const Plan &p = h->plan;
    std::memset(info, 0, sizeof(*info));
    info->tiles = p.tiles;
    info->k_blocks = p.num_k_blocks;
    info->grid_ctas = p.grid_ctas;
    info->threads_per_cta = p.threads;
    info->cta_group = p.cta_group;
    info->pipeline = p.pipeline;
    info->persistent = p.persistent;
    info->stages = p.stages;
    info->acc_buffers = p.acc_buffers;
    info->setmaxnreg = p.setmaxnreg;
    info->stage_group = p.stage_group;
    info->sk_tiles = p.sk_tiles;
    info->sk_head = p.sk_head;
    info->sk_slots = (int32_t)p.sk_slots;
    info->tile_m = kBlockM * p.cta_group;
    info->tile_n = p.thin_nt ? p.thin_nt : kBlockN;
    info->tile_k = kBlockK;
    info->smem_bytes = (int32_t)p.smem;
    info->num_sms = h->num_sms;
    info->epilogue_tma_allowed = p.epi_tma_allowed ? 1 : 0;
    info->raster_group = p.raster_group;
    info->regs_per_thread = p.regs;
    info->epi_schedule = p.epi_pingpong;
    info->scheduler = p.sched_dynamic;
    info->repack = (p.repack_a ? 1 : 0) | (p.repack_b ? 2 : 0);
    info->packed_ld = (int32_t)p.ldp;
    info->k_order = p.k_order;
    info->serpentine = p.serpentine;
    info->thin = p.thin_nt;
    info->thin_cluster = p.thin_cluster;
    return GEMM_BF16_OK;
}

}  // extern "C"

namespace {

struct FusedArgs {
    const void *C;
    int64_t ldc;
    const void *bias;
    float alpha, beta;
};

// A launch's epoch for the square kernel's stream-K flags: never 0 (flags start at 0).
void next_epoch(gemm_bf16_t h)
{
    do
        ++h->epoch;
    while (h->epoch == 0u);
}

// The operands as run_impl resolved them: the caller's pointers, and the ones
// the kernel reads (the packed copies where the plan repacks).
struct OperandView {
    const void *A, *B;    // caller's
    const void *Ae, *Be;  // read by the GEMM
    int64_t lda_e, ldb_e;
    void *pack_a, *pack_b;
};

// The square kernel's stream-K flags mean "written in this launch" when they
// equal the launch's epoch, a kernel parameter (the thin kernel keeps its
// epoch in device memory and needs none of this).  A launch captured into a CUDA graph keeps the
// epoch it was captured with on every replay, so while `st` is capturing, a
// clear of the flags is enqueued before the launch: each replay then starts
// from flags no replay has raised yet.  Launches outside a capture need none.
int clear_flags_if_capturing(uint32_t *flags, size_t n, cudaStream_t st)
{
    if (!flags || n == 0)
        return GEMM_BF16_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    if (cs == cudaStreamCaptureStatusActive && cudaMemsetAsync(flags, 0, n * sizeof(uint32_t), st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    return GEMM_BF16_OK;
}

int launch_repacks(gemm_bf16_t h, const OperandView &ops, cudaStream_t st)
{
    const Plan &pl = h->plan;
    if (!ops.pack_a && !ops.pack_b)
        return GEMM_BF16_OK;
    RepackJob jobs[2];
    int nj = 0;
    if (ops.pack_a)
        jobs[nj++] = {ops.A, ops.pack_a, pl.lda, pl.ldp, pl.M, pl.K};
    if (ops.pack_b)
        jobs[nj++] = {ops.B, ops.pack_b, pl.ldb, pl.ldp, pl.N, pl.K};
    return launch_repack(jobs, nj, h->num_sms, st) != 0 ? GEMM_BF16_ERR_CUDA : GEMM_BF16_OK;
}

// One launch of the thin kernel (plan_thin): tensor maps of the large operand
// (box 64 x 128) and the small one (box 64 x thin_nt), then the launch.
int run_thin(gemm_bf16_t h, const OperandView &ops, void *D, const FusedArgs *fz, cudaStream_t st, bool fault_maps)
{
    const Plan &pl = h->plan;
    int rc;
    const void *large = pl.thin_transposed ? ops.Be : ops.Ae;
    const void *small = pl.thin_transposed ? ops.Ae : ops.Be;
    const int64_t large_rows = pl.thin_transposed ? pl.N : pl.M;
    const int64_t small_rows = pl.thin_transposed ? pl.M : pl.N;
    const int64_t ld_large = pl.thin_transposed ? ops.ldb_e : ops.lda_e;
    const int64_t ld_small = pl.thin_transposed ? ops.lda_e : ops.ldb_e;
    // Each CTA's last tile goes out by one TMA store when D allows it (16-byte
    // aligned base and rows, and N a multiple of 8: a store clips D's columns
    // only at 16-byte boundaries, so a box reaching past column N of a row
    // with padding would write into the padding) and the epilogue is the
    // plain one: a box of 128 columns by thin_nt rows of D (transposed) or
    // thin_nt columns by 128 rows.
    bool d_tma = !fz && (reinterpret_cast<uintptr_t>(D) & 15u) == 0 && (pl.ldd * 2) % 16 == 0 && pl.N % 8 == 0;
    if (fault_maps || !h->maps_valid || h->mA != ops.Ae || h->mB != ops.Be || (d_tma && h->mD != D)) {
        if (fault_maps) {
            h->maps_valid = false;
            return GEMM_BF16_ERR_TENSORMAP;
        }
        if ((rc = encode_2d(&h->tmA, large, (uint64_t)pl.K, (uint64_t)large_rows, (uint64_t)ld_large * 2, kBlockK,
                            kBlockM)) ||
            (rc = encode_2d(&h->tmB, small, (uint64_t)pl.K, (uint64_t)small_rows, (uint64_t)ld_small * 2, kBlockK,
                            (uint32_t)pl.thin_nt))) {
            h->maps_valid = false;
            return rc;
        }
        // a D the driver will not describe is stored by the threads instead
        if (d_tma && encode_2d(&h->tmD, D, (uint64_t)pl.N, (uint64_t)pl.M, (uint64_t)pl.ldd * 2,
                               pl.thin_transposed ? (uint32_t)kBlockM : (uint32_t)pl.thin_nt,
                               pl.thin_transposed ? (uint32_t)pl.thin_nt : (uint32_t)kBlockM, false) != GEMM_BF16_OK)
            d_tma = false;
        if (!d_tma)
            std::memset(&h->tmD, 0, sizeof(h->tmD));  // passed, never used
        h->mA = ops.Ae, h->mB = ops.Be, h->mD = d_tma ? D : nullptr;
        h->maps_valid = true;
    }
    if ((rc = launch_repacks(h, ops, st)) != GEMM_BF16_OK)
        return rc;

    ThinParams tp;
    tp.rows = (int32_t)large_rows;
    tp.thin = (int32_t)small_rows;
    tp.num_k_blocks = pl.num_k_blocks;
    tp.num_tiles = (int32_t)pl.tiles;
    tp.units = pl.thin_units;
    tp.stages = pl.stages;
    tp.transposed = pl.thin_transposed ? 1 : 0;
    tp.d_vec = ((reinterpret_cast<uintptr_t>(D) & 15u) == 0 && pl.ldd % 8 == 0) ? 1 : 0;
    tp.d_pair = ((reinterpret_cast<uintptr_t>(D) & 3u) == 0 && pl.ldd % 2 == 0) ? 1 : 0;
    tp.d_tma = d_tma ? 1 : 0;
    tp.fault_skip_it = pl.fault_skip;
    tp.ldd = pl.ldd;
    tp.D = D;
    tp.err = h->d_err;
    tp.watchdog_ns = pl.watchdog_ns;
    tp.partials = h->thin_ws;
    tp.flags = h->thin_flags;
    tp.sync = h->thin_sync;
    tp.cluster = pl.thin_cluster > 1 ? pl.thin_cluster : 1;
    tp.push = pl.thin_push;
    tp.C = nullptr;
    tp.bias = nullptr;
    tp.ldc = 0;
    tp.alpha = 1.f;
    tp.beta = 0.f;
    tp.fused = 0;
    if (fz) {
        tp.fused = kFusedOn;
        tp.alpha = fz->alpha;
        tp.beta = fz->beta;
        if (fz->C) {
            tp.C = fz->C;
            tp.ldc = fz->ldc;
            tp.fused |= kFusedC;
        }
        if (fz->bias) {
            tp.bias = fz->bias;
            tp.fused |= kFusedBias;
        }
    }

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    unsigned nattr = 0;
    cfg.gridDim = dim3((unsigned)pl.grid_ctas, 1, 1);
    cfg.blockDim = dim3((unsigned)pl.threads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    if (h->opt[GEMM_BF16_OPT_PDL]) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    if (tp.cluster > 1) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = (unsigned)tp.cluster;
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    cfg.attrs = nattr ? attr : nullptr;
    cfg.numAttrs = nattr;
    void *args[4] = {&h->tmA, &h->tmB, &h->tmD, &tp};
    if (cudaLaunchKernelExC(&cfg, pl.fn, args) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    h->last_stream = st;
    return GEMM_BF16_OK;
}

int run_impl(gemm_bf16_t h, const void *A, const void *B, void *D, const FusedArgs *fz, void *stream)
{
    if (!h || !A || !B || !D)
        return GEMM_BF16_ERR_INVALID_ARG;
    if (!h->plan.valid)
        return GEMM_BF16_ERR_NOT_PLANNED;
    const Plan &pl = h->plan;
    if ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u) ||
        (reinterpret_cast<uintptr_t>(D) & 1u))
        return GEMM_BF16_ERR_ALIGNMENT;
    const bool d_aligned = (reinterpret_cast<uintptr_t>(D) & 15u) == 0;
    bool epi_tma;
    if (pl.epilogue_opt == 1) {
        if (!pl.epi_tma_allowed || !d_aligned)
            return GEMM_BF16_ERR_ALIGNMENT;
        epi_tma = true;
    } else if (pl.epilogue_opt == 2) {
        epi_tma = false;
    } else {
        epi_tma = pl.epi_tma_allowed && d_aligned;
    }
    int rc = set_device(h);
    if (rc != GEMM_BF16_OK)
        return rc;

    // Operands routed through the packed buffer are copied first, on the same
    // stream; the GEMM's tensor maps then describe the packed copies.
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void *pack_a = pl.repack_a ? h->pack : nullptr;
    void *pack_b = pl.repack_b ? static_cast<uint16_t *>(h->pack) + (pl.repack_a ? pl.M * pl.ldp : 0) : nullptr;
    const void *Ae = pack_a ? pack_a : A;
    const void *Be = pack_b ? pack_b : B;
    const int64_t lda_e = pack_a ? pl.ldp : pl.lda;
    const int64_t ldb_e = pack_b ? pl.ldp : pl.ldb;

    // test hook: the encode fails as a driver error would, before any launch
    const bool fault_maps = h->opt[GEMM_BF16_OPT_FAULT_TENSORMAP] != 0;
    if (pl.thin_nt) {
        const OperandView ops = {A, B, Ae, Be, lda_e, ldb_e, pack_a, pack_b};
        return run_thin(h, ops, D, fz, st, fault_maps);
    }
    if (fault_maps || !h->maps_valid || h->mA != Ae || h->mB != Be || h->mD != D) {
        if (fault_maps) {
            h->maps_valid = false;
            return GEMM_BF16_ERR_TENSORMAP;
        }
        const uint32_t b_rows = (uint32_t)(kBlockN / pl.cta_group);
        if ((rc = encode_2d(&h->tmA, Ae, (uint64_t)pl.K, (uint64_t)pl.M, (uint64_t)lda_e * 2, kBlockK, kBlockM)) ||
            (rc = encode_2d(&h->tmB, Be, (uint64_t)pl.K, (uint64_t)pl.N, (uint64_t)ldb_e * 2, kBlockK, b_rows))) {
            h->maps_valid = false;
            return rc;
        }
        if (pl.epi_tma_allowed && d_aligned) {
            if ((rc = encode_2d(&h->tmD, D, (uint64_t)pl.N, (uint64_t)pl.M, (uint64_t)pl.ldd * 2, 64, 32))) {
                h->maps_valid = false;
                return rc;
            }
        } else {
            std::memset(&h->tmD, 0, sizeof(h->tmD));  // never dereferenced on the masked path
        }
        h->mA = Ae, h->mB = Be, h->mD = D;
        h->maps_valid = true;
    }
    {
        const OperandView ops = {A, B, Ae, Be, lda_e, ldb_e, pack_a, pack_b};
        if ((rc = launch_repacks(h, ops, st)) != GEMM_BF16_OK)
            return rc;
    }
    if (pl.sk_tiles > 0 && (rc = clear_flags_if_capturing(h->ws_flags, pl.sk_slots, st)) != GEMM_BF16_OK)
        return rc;

    GemmParams prm;
    prm.M = (int32_t)pl.M;
    prm.N = (int32_t)pl.N;
    prm.K = (int32_t)pl.K;
    prm.num_m_blocks = pl.num_m_blocks;
    prm.num_n_blocks = pl.num_n_blocks;
    prm.num_k_blocks = pl.num_k_blocks;
    prm.num_tiles = (int32_t)pl.tiles;
    prm.raster_group = pl.raster_group;
    prm.stages = pl.stages;
    prm.acc_buffers = pl.acc_buffers;
    prm.stage_group = pl.stage_group;
    prm.epi_tma = epi_tma ? 1 : 0;
    prm.fault_skip_it = pl.fault_skip;
    prm.ldd = pl.ldd;
    prm.D = D;
    prm.err = h->d_err;
    prm.watchdog_ns = pl.watchdog_ns;
    prm.sk_tiles = pl.sk_tiles;
    prm.sk_units = pl.sk_units;
    prm.sk_head = pl.sk_head;
    prm.sk_pieces = pl.sk_pieces;
    prm.workspace = pl.sk_tiles ? h->ws : nullptr;
    prm.flags = pl.sk_tiles ? h->ws_flags : nullptr;
    next_epoch(h);
    prm.epoch = h->epoch;
    prm.C = nullptr;
    prm.bias = nullptr;
    prm.ldc = 0;
    prm.alpha = 1.f;
    prm.beta = 0.f;
    prm.fused = 0;
    prm.epi_pingpong = pl.epi_pingpong;
    prm.sched_dynamic = pl.sched_dynamic;
    prm.sched = h->d_err + 2;
    prm.k_order = pl.k_order;
    prm.serpentine = pl.serpentine;
    if (fz) {
        prm.fused = kFusedOn;
        prm.alpha = fz->alpha;
        prm.beta = fz->beta;
        if (fz->C) {
            prm.C = fz->C;
            prm.ldc = fz->ldc;
            prm.fused |= kFusedC;
            if ((reinterpret_cast<uintptr_t>(fz->C) & 15u) == 0 && fz->ldc % 8 == 0)
                prm.fused |= kFusedCVec;
        }
        if (fz->bias) {
            prm.bias = fz->bias;
            prm.fused |= kFusedBias;
            if ((reinterpret_cast<uintptr_t>(fz->bias) & 15u) == 0)
                prm.fused |= kFusedBiasVec;
        }
    }

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    unsigned nattr = 0;
    cfg.gridDim = dim3((unsigned)pl.grid_ctas, 1, 1);
    cfg.blockDim = dim3((unsigned)pl.threads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    if (pl.cta_group == 2) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = 2;
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    if (h->opt[GEMM_BF16_OPT_PDL]) {
        // the kernel's prologue may overlap the previous kernel on the stream;
        // griddepcontrol.wait orders every global access after it
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    cfg.attrs = nattr ? attr : nullptr;
    cfg.numAttrs = nattr;
    void *args[4] = {&h->tmA, &h->tmB, &h->tmD, &prm};
    if (cudaLaunchKernelExC(&cfg, pl.fn, args) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    h->last_stream = static_cast<cudaStream_t>(stream);
    return GEMM_BF16_OK;
}

}  // namespace

extern "C" {

GEMM_BF16_API int gemm_bf16_run(gemm_bf16_t h, const void *A, const void *B, void *D, void *stream)
{
    return run_impl(h, A, B, D, nullptr, stream);
}

GEMM_BF16_API int gemm_bf16_run_fused(gemm_bf16_t h, const void *A, const void *B, void *D, const void *C,
                                      int64_t ldc, const void *bias, float alpha, float beta, void *stream)
{
    if (!h)
        return GEMM_BF16_ERR_INVALID_ARG;
    if (!h->plan.valid)
        return GEMM_BF16_ERR_NOT_PLANNED;
    if (C && (ldc < h->plan.N || ldc > (int64_t(1) << 38)))
        return GEMM_BF16_ERR_INVALID_ARG;
    if ((C && (reinterpret_cast<uintptr_t>(C) & 1u)) || (bias && (reinterpret_cast<uintptr_t>(bias) & 1u)))
        return GEMM_BF16_ERR_ALIGNMENT;
    const FusedArgs fz = {C, C ? ldc : 0, bias, alpha, beta};
    return run_impl(h, A, B, D, &fz, stream);
}

}  // extern "C"

namespace {

// `rows` rows of `cols` bf16 between two buffers of row pitch `ld` (elements):
// one linear copy when the rows are contiguous, else a pitched copy of the
// sub-matrix (the padding between rows is not copied).
cudaError_t copy_rows(void *dst, const void *src, int64_t ld, int64_t cols, int64_t rows, cudaMemcpyKind kind,
                      cudaStream_t st)
{
    if (ld == cols)
        return cudaMemcpyAsync(dst, src, (size_t)(rows * cols * 2), kind, st);
    return cudaMemcpy2DAsync(dst, (size_t)(ld * 2), src, (size_t)(ld * 2), (size_t)(cols * 2), (size_t)rows, kind, st);
}

}  // namespace

extern "C" {

GEMM_BF16_API int gemm_bf16_run_host(gemm_bf16_t h, const void *hA, const void *hB, void *hD, void *dA, void *dB,
                                     void *dD, void *stream)
{
    if (!h || !hA || !hB || !hD || !dA || !dB || !dD)
        return GEMM_BF16_ERR_INVALID_ARG;
    if (!h->plan.valid)
        return GEMM_BF16_ERR_NOT_PLANNED;
    const Plan &pl = h->plan;
    int rc = set_device(h);
    if (rc != GEMM_BF16_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (copy_rows(dA, hA, pl.lda, pl.K, pl.M, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        copy_rows(dB, hB, pl.ldb, pl.K, pl.N, cudaMemcpyHostToDevice, st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    if ((rc = gemm_bf16_run(h, dA, dB, dD, stream)) != GEMM_BF16_OK)
        return rc;
    if (copy_rows(hD, dD, pl.ldd, pl.N, pl.M, cudaMemcpyDeviceToHost, st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    return GEMM_BF16_OK;
}

GEMM_BF16_API int gemm_bf16_device_status(gemm_bf16_t h, uint32_t *detail)
{
    if (!h)
        return GEMM_BF16_ERR_INVALID_ARG;
    int rc = set_device(h);
    if (rc != GEMM_BF16_OK)
        return rc;
    if (cudaStreamSynchronize(h->last_stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    uint32_t w = 0;
    // Clearing the whole block also puts the tile counter back to 0: after a
    // watchdog give-up it is the only thing that does (normally the last SM
    // pair of each launch resets it).
    if (cudaMemcpy(&w, h->d_err, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess ||
        (w != 0 && cudaMemset(h->d_err, 0, 4 * sizeof(uint32_t)) != cudaSuccess) ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    if (detail)
        *detail = w;
    return w ? GEMM_BF16_ERR_DEVICE_TIMEOUT : GEMM_BF16_OK;
}

}  // extern "C"
