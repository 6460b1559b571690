// Internal interface between the host library (gemm_bf16_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace wstma {

// Tile geometry shared by every kernel: a CTA owns a 128-row slab of the output
// tile, a stage holds one 64-wide k-block (one 128-byte swizzle row per operand
// row), and the accumulator is 256 fp32 columns of tensor memory.
constexpr int kBlockM = 128;      // rows of D per CTA
constexpr int kBlockN = 256;      // columns of D per tile (both modes)
constexpr int kBlockK = 64;       // k per stage (64 bf16 = 128 bytes)
constexpr int kEpiWarps = 8;      // two epilogue warpgroups in the WS kernel
constexpr int kWsThreads = 384;   // WG0: producer / MMA / TMEM-alloc / spare warp; WG1-2: epilogue
constexpr int kNowsThreads = 128; // the non-specialised ablation kernels
constexpr int kStagingBytes = 32 * 64 * 2;  // per-warp epilogue staging: 32 rows x 64 bf16
constexpr int kMaxStages = 8;
constexpr int kRingSlots = 8;     // schedule ring depth (power of two)

// Producer / consumer register budgets for setmaxnreg (whole warpgroups).
constexpr int kProducerRegs = 56;
constexpr int kConsumerRegs = 224;

struct GemmParams {
    int32_t M, N, K;
    int32_t num_m_blocks;   // tiles along M (tile height 128 * cta_group)
    int32_t num_n_blocks;   // tiles along N (tile width 256)
    int32_t num_k_blocks;   // ceil(K / 64)
    int32_t num_tiles;
    int32_t raster_group;   // 0 = row-major tile order
    int32_t stages;
    int32_t acc_buffers;    // 1 or 2 (WS only)
    int32_t stage_group;    // k-blocks released per commit: 1, or 2 (stages pair up; S even) (WS only)
    int32_t epi_tma;        // 1 = TMA-store epilogue, 0 = masked st.global
    int32_t fault_skip_it;  // test hook, -1 = off
    int64_t ldd;
    void *D;
    uint32_t *err;          // device status word (0 = fine)
    uint64_t watchdog_ns;
    // stream-K (WS only): tiles [0, sk_tiles) are split along k, the other
    // tiles are walked whole.  0 = off.  Two forms:
    //   sk_head == 0 (partial last wave): the split tiles' (tile, k-block)
    //     units are divided among all clusters;
    //   sk_head  > 0 (fewer tiles than clusters, sk_tiles = num_tiles): cluster
    //     t computes k-blocks [0, sk_head) of tile t, and the tails [sk_head, KB)
    //     of every tile are divided among the remaining clusters.
    int32_t sk_tiles;
    uint32_t epoch;         // this launch's flag value (never 0)
    int64_t sk_units;       // units divided among clusters: sk_tiles * (num_k_blocks - sk_head)
    int32_t sk_head;
    int32_t sk_pieces;      // workspace slots per contributing cluster (1 when sk_head == 0)
    float *workspace;       // partials: per (slot, rank) 128 x 256 fp32 = kPartialFloats
    uint32_t *flags;        // per (slot, rank): == epoch once that partial is complete
    // fused epilogue D = alpha * acc + beta * C + bias (when fused != 0)
    const void *C;          // bf16, row pitch ldc (may alias D with ldc == ldd)
    const void *bias;       // bf16 [N]
    int64_t ldc;
    float alpha, beta;
    uint32_t fused;         // kFused* bits; 0 = plain store of the accumulator
    // schedules (WS only)
    int32_t epi_pingpong;   // 1 = epilogue warpgroup g drains the tiles of accumulator g
    int32_t sched_dynamic;  // 1 = whole tiles are taken from the counter sched[0]
    uint32_t *sched;        // [0] next whole tile, [1] clusters finished; both 0 between launches
    int32_t k_order;        // 1 = a CTA's odd-numbered whole tiles load their k-blocks last to first
    int32_t serpentine;     // 1 = odd tile bands walk their columns right to left
};

enum : uint32_t {
    kFusedOn = 1u,          // apply alpha (and beta*C, bias when present)
    kFusedC = 2u,           // C present
    kFusedBias = 4u,        // bias present
    kFusedCVec = 8u,        // C rows 16-byte aligned: vector loads
    kFusedBiasVec = 16u     // bias 16-byte aligned: vector loads
};

constexpr int kPartialFloats = kBlockM * kBlockN;  // one CTA's accumulator slice

// Dynamic shared memory a kernel needs for `stages` ring stages.
inline size_t ws_smem_bytes(int cta_group, int stages)
{
    const size_t stage = (size_t)kBlockM * kBlockK * 2 + (size_t)(kBlockN / cta_group) * kBlockK * 2;
    return 1024 /* alignment slack */ + (size_t)stages * stage + (size_t)kEpiWarps * kStagingBytes +
           512 /* schedule ring, barriers, tmem slot, abort flag, epilogue go words */;
}

inline size_t nows_smem_bytes(int stages)
{
    const size_t stage = (size_t)kBlockM * kBlockK * 2 + (size_t)kBlockN * kBlockK * 2;
    return 1024 + (size_t)stages * stage + 4 * (size_t)kStagingBytes + 256;
}

// The thin kernel (gemm_thin.cuh): one operand has at most 64 rows.  The
// other ("large") operand is cut into 128-row tiles, each a tcgen05.mma M side,
// and the small one is the MMA's N side, rounded up to kThinN (16, 32, 48 or 64).
constexpr int kThinThreads = 256;  // warp 0 producer, 1 MMA, 2 TMEM allocation, 4-7 epilogue
constexpr int kThinMaxStages = 12;
constexpr int kThinMaxRows = 64;

struct ThinParams {
    int32_t rows;           // rows of the large operand
    int32_t thin;           // rows of the small operand (1..64)
    int32_t num_k_blocks;   // ceil(K / 64)
    int32_t num_tiles;      // ceil(rows / 128)
    int64_t units;          // num_tiles * num_k_blocks, split among the CTAs (thin_split.h)
    int32_t stages;
    int32_t transposed;     // 1: the large operand is B, so D[m][n] is accumulator row n, column m
    int32_t d_vec;          // 1: rows of D are 16-byte aligned (vector stores, not transposed only)
    int32_t d_pair;         // 1: rows of D are 4-byte aligned (paired stores, transposed only)
    int32_t d_tma;          // 1: each CTA's last tile is stored by TMA (tensor map of D; not fused)
    int32_t fault_skip_it;  // test hook, -1 = off
    int64_t ldd;
    void *D;
    uint32_t *err;
    uint64_t watchdog_ns;
    float *partials;        // 2 slots per CTA, 128 x NT fp32 each
    uint32_t *flags;        // 4 per slot (one per epilogue warp): == epoch once that warp's rows are stored
    uint32_t *sync;         // {epoch (never 0), CTAs that have read it}, advanced on the device
    int32_t cluster;        // > 1: clusters of this many CTAs split each tile's k-blocks (one tile per
                            // cluster, partials summed through distributed shared memory); 1: the
                            // units are split across the CTAs (thin_split.h)
    int32_t push;           // cluster form: 1 = ranks 1..C-1 store their partials into rank 0's
                            // receive area after its barriers ((C - 1) x 128 x NT fp32), 0 = rank 0 reads them
    // fused epilogue, as in GemmParams
    const void *C;
    const void *bias;
    int64_t ldc;
    float alpha, beta;
    uint32_t fused;
};

inline int thin_nt(int64_t thin_rows) { return (int)((thin_rows + 15) / 16 * 16); }

inline size_t thin_stage_bytes(int nt) { return (size_t)kBlockM * kBlockK * 2 + (size_t)nt * kBlockK * 2; }

inline size_t thin_smem_bytes(int nt, int stages)
{
    return 1024 /* alignment slack */ + (size_t)stages * thin_stage_bytes(nt) + 512 /* barriers, tmem slot, flags */;
}

// Kernel entry points, one per compiled variant.  All take
// (CUtensorMap A, CUtensorMap B, CUtensorMap D, GemmParams).
const void *ws_kernel_c1(bool setmaxnreg);
const void *ws_kernel_c2(bool setmaxnreg);
const void *nows_kernel(bool mbar_war);
// (CUtensorMap large, CUtensorMap small, CUtensorMap D, ThinParams); nt = 16, 32, 48 or 64.
const void *thin_kernel(int nt);

// One operand copy: `rows` rows of `cols` bf16 from pitch ld_src to pitch
// ld_dst (elements; both multiples of 8, both bases 16-byte aligned).
struct RepackJob {
    const void *src;
    void *dst;
    int64_t ld_src, ld_dst, rows, cols;
};
// Runs one or two copies in one launch on `stream`; returns a cudaError_t value.
int launch_repack(const RepackJob *jobs, int njobs, int num_sms, cudaStream_t stream);

}  // namespace wstma
