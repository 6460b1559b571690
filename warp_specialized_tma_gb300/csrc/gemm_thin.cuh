// The thin kernel: D = A * B^T when one of M, N is at most 64 (decode-like
// problems).  Such problems are bound by streaming the large operand from
// HBM, not by the tensor pipe.  In the square kernel a 64-row operand would
// still fill a 128-row MMA side, and 7/8 or more of its shared-memory stage
// would hold TMA's zero fill.  Here the large operand takes the 128-row M
// side of each tcgen05.mma.  The small operand is the N side, rounded up to
// NT = 16..64, so a stage is 16 KiB of the large operand plus NT x 128 bytes.
// The ring is then up to 12 stages deep and keeps ~2x the bytes in flight per
// SM.
//
// At most one CTA per SM (shared memory), in clusters or not (below).  Roles:
//   warp 0, lane 0   TMA producer: for each of the CTA's items, per k-block:
//                    wait "empty", expect_tx, load the large tile (64 x 128)
//                    and the small one (64 x NT)
//   warp 1, lane 0   MMA issuer: four tcgen05.mma (K = 16) per k-block into one
//                    of two NT-column tensor-memory accumulators, commit ->
//                    "empty"; after an item, commit -> accumulator full
//   warp 2           allocates (and frees) tensor memory
//   warps 4-7        epilogue: tensor memory -> registers; a split tile's
//                    pieces meet as described below; the CTA's last tile is
//                    staged in the drained ring and written by one TMA store
//                    when D allows it, other tiles by the threads
// Every wait is bounded by the watchdog (WaitCtl in ptx.cuh).
//
// Two ways to split the work.  Across the SMs (the default for large or long
// problems): the (tile, k-block) units are cut into one contiguous range per
// CTA, and a split tile's pieces meet through global memory, as follows.  In
// clusters (problems whose tiles times a cluster size of 2..8 nearly fill the
// GPU): the C CTAs of cluster c split tile c's k-blocks evenly, rank r > 0
// leaves its fp32 partial in its own shared memory (the drained ring) and
// arrives, per epilogue warp, on a barrier of rank 0 with release at cluster
// scope; rank 0's warp waits on it (bounded), reads the rows of ranks 1..C-1
// through distributed shared memory in rank order, adds, and stores.  Where
// rank 0's shared memory has room for the others' partials beside a ring of
// at least 4 stages, they store them there instead (remote stores, which do
// not wait) and rank 0 reads its own shared memory.  A cluster barrier at exit
// keeps every rank's shared memory alive until rank 0 has read it.  One CTA
// per whole tile is the cluster form with C = 1.
//
// Across the SMs, the piece of a split tile that holds k-block 0 (the last
// item of its range) owns the tile (thin_split.h), and the pieces meet through
// fp32 partials in a workspace and one flag per partial slot and epilogue
// warp.  A contributor warp stores its 32 rows, meets at a warp barrier, and
// its lane 0 writes the launch's epoch to the flag with a release store; the
// owner warp's lane 0 polls the flag with acquire loads, the warp meets at a
// warp barrier, and the 32 lanes read the rows.  The four warps of a CTA do
// not wait for one another on this path.  The epoch lives in device memory:
// every CTA reads it after the grid-dependency wait, and the last CTA to have
// read it advances it for the next launch, so launches replayed from a CUDA
// graph get a new epoch each time as well, and flags never need clearing.
#pragma once

#include "gemm_kernels.h"
#include "ptx.cuh"
#include "ring_index.h"
#include "thin_split.h"

namespace wstma {

// Lane 0 of an owner warp waits (bounded) until a contributor warp's flag
// carries this launch's epoch; false if the wait gave up.
__device__ __forceinline__ bool thin_poll_flag(const WaitCtl &ctl, const uint32_t *flag, uint32_t epoch)
{
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 0; ld_acquire_gpu_u32(flag) != epoch; ++n) {
        if (ctl.aborted())
            return false;
        if (globaltimer_ns() - t0 > ctl.limit_ns || n > (1u << 30)) {
            ctl.fail(kRoleFixup, 0);
            return false;
        }
        __nanosleep(32);
    }
    return true;
}

__device__ __forceinline__ uint32_t thin_ld_relaxed_u32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// fp32 accumulator element -> the stored value (fused: alpha * acc + beta * C + bias).
__device__ __forceinline__ float thin_epilogue_value(float acc, int64_t m, int64_t n, const ThinParams &p)
{
    if (!p.fused)
        return acc;
    float c = 0.f, b = 0.f;
    if (p.fused & kFusedC)
        c = __uint_as_float((uint32_t)(static_cast<const uint16_t *>(p.C)[m * p.ldc + n]) << 16);
    if (p.fused & kFusedBias)
        b = __uint_as_float((uint32_t)(static_cast<const uint16_t *>(p.bias)[n]) << 16);
    return fmaf(p.alpha, acc, fmaf(p.beta, c, b));
}

__device__ __forceinline__ uint16_t thin_bf16(float f)
{
    return (uint16_t)(pack_bf16x2(__float_as_uint(f), 0u) & 0xFFFFu);
}

// Stores one accumulator row (this thread's row r of the large operand's tile)
// to D.  Not transposed: D[r][0 .. thin).  Transposed: D[0 .. thin)[r], so the
// 32 lanes of a warp store 32 consecutive elements of one row of D; when the
// warp's 32 columns all lie inside D and its rows are 4-byte aligned, lane
// pairs trade one value per two rows (the even lane stores row i of columns
// r, r + 1, the odd lane row i + 1) and store 4-byte words, half as many
// stores.  Called by all 32 lanes of a warp.
template <int NT>
__device__ __forceinline__ void thin_store_row(const float (&v)[NT], int64_t r, const ThinParams &p)
{
    uint16_t *const D = static_cast<uint16_t *>(p.D);
    if (p.transposed) {
        const int lane = (int)(threadIdx.x & 31u);
        if (p.d_pair && !p.fused && r - lane + 32 <= p.rows) {
            const bool odd = (lane & 1) != 0;
#pragma unroll
            for (int i = 0; i < NT; i += 2) {
                const float got = __shfl_xor_sync(0xFFFFFFFFu, odd ? v[i] : v[i + 1], 1);
                if (!odd) {
                    if (i < p.thin)
                        *reinterpret_cast<uint32_t *>(D + (int64_t)i * p.ldd + r) =
                            pack_bf16x2(__float_as_uint(v[i]), __float_as_uint(got));
                } else if (i + 1 < p.thin) {
                    *reinterpret_cast<uint32_t *>(D + (int64_t)(i + 1) * p.ldd + r - 1) =
                        pack_bf16x2(__float_as_uint(got), __float_as_uint(v[i + 1]));
                }
            }
            return;
        }
        if (r >= p.rows)
            return;
#pragma unroll
        for (int i = 0; i < NT; ++i)
            if (i < p.thin)
                D[(int64_t)i * p.ldd + r] = thin_bf16(thin_epilogue_value(v[i], i, r, p));
        return;
    }
    if (r >= p.rows)
        return;
    uint16_t *const row = D + r * p.ldd;
    if (p.d_vec && !p.fused && p.thin == NT) {
#pragma unroll
        for (int i = 0; i < NT; i += 8) {
            uint4 q;
            q.x = pack_bf16x2(__float_as_uint(v[i]), __float_as_uint(v[i + 1]));
            q.y = pack_bf16x2(__float_as_uint(v[i + 2]), __float_as_uint(v[i + 3]));
            q.z = pack_bf16x2(__float_as_uint(v[i + 4]), __float_as_uint(v[i + 5]));
            q.w = pack_bf16x2(__float_as_uint(v[i + 6]), __float_as_uint(v[i + 7]));
            *reinterpret_cast<uint4 *>(row + i) = q;
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < NT; ++i)
        if (i < p.thin)
            row[i] = thin_bf16(thin_epilogue_value(v[i], r, i, p));
}

// Writes one accumulator row (row_in_tile of the tile) as bf16 into the staging
// buffer of the tile's TMA store.  Transposed: the box is 128 columns of D by
// NT rows, so D row i holds this row's value i at column row_in_tile; else the
// box is NT columns by 128 rows, this row's NT values contiguous.
template <int NT>
__device__ __forceinline__ void thin_stage_row(const float (&v)[NT], int row_in_tile, uint32_t stage, bool transposed)
{
    if (transposed) {
#pragma unroll
        for (int i = 0; i < NT; ++i)
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(stage + (uint32_t)(i * kBlockM + row_in_tile) * 2u),
                         "h"(thin_bf16(v[i]))
                         : "memory");
        return;
    }
    const uint32_t row = stage + (uint32_t)(row_in_tile * NT) * 2u;
#pragma unroll
    for (int i = 0; i < NT; i += 8)
        st_shared_v4(row + (uint32_t)i * 2u, pack_bf16x2(__float_as_uint(v[i]), __float_as_uint(v[i + 1])),
                     pack_bf16x2(__float_as_uint(v[i + 2]), __float_as_uint(v[i + 3])),
                     pack_bf16x2(__float_as_uint(v[i + 4]), __float_as_uint(v[i + 5])),
                     pack_bf16x2(__float_as_uint(v[i + 6]), __float_as_uint(v[i + 7])));
}

// Stores a CTA's last tile: every epilogue thread stages its row in the ring
// (drained: the CTA has no loads or MMAs left), the four warps meet, and one
// thread issues the tile's TMA store and waits until it has read the staging.
// The TMA engine writes whole lines of D, where per-thread stores of a
// transposed tile write 64-byte pieces of NT rows at once in every CTA.
template <int NT>
__device__ __forceinline__ void thin_store_tile_tma(const float (&v)[NT], int row_in_tile, int64_t t, uint32_t stage,
                                                    const CUtensorMap *tmD, const ThinParams &p)
{
    thin_stage_row<NT>(v, row_in_tile, stage, p.transposed != 0);
    fence_proxy_async_shared();  // the staging writes come before the async-proxy read
    named_barrier_sync(1u, 128u);
    if (threadIdx.x == 128) {
        const int32_t at = (int32_t)(t * kBlockM);
        tma_store_2d(tmD, stage, p.transposed ? at : 0, p.transposed ? 0 : at);
        bulk_commit_group();
        bulk_wait_read_all();
    }
}

template <int NT>
__global__ void __launch_bounds__(kThinThreads, 1)
    gemm_thin_kernel(const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmS,
                     const __grid_constant__ CUtensorMap tmD, const ThinParams p)
{
    static_assert(NT % 16 == 0 && NT >= 16 && NT <= kThinMaxRows, "NT: 16, 32, 48 or 64");
    constexpr uint32_t kLBytes = (uint32_t)kBlockM * kBlockK * 2;  // 128 rows of the large operand
    constexpr uint32_t kSBytes = (uint32_t)NT * kBlockK * 2;       // NT rows of the small one
    constexpr uint32_t kStageBytes = kLBytes + kSBytes;             // a multiple of 1024
    constexpr uint32_t kIdesc = idesc_bf16_f32(kBlockM, NT);
    constexpr uint32_t kAllocCols = 2 * NT <= 32 ? 32u : (2 * NT <= 64 ? 64u : 128u);
    static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int S = p.stages;
    const uint32_t stage0 = base;
    const uint32_t full_bar = base + (uint32_t)S * kStageBytes;
    const uint32_t empty_bar = full_bar + 8u * S;
    const uint32_t accf_bar = empty_bar + 8u * S;
    const uint32_t acce_bar = accf_bar + 16u;
    const uint32_t done_bar = acce_bar + 16u;
    const uint32_t ready_bar = done_bar + 8u;  // 4, one per epilogue warp (rank 0 of a cluster)
    const uint32_t tmem_slot = ready_bar + 32u;
    const uint32_t abort_flag = tmem_slot + 4u;
    const uint32_t epoch_word = abort_flag + 4u;
    const uint32_t go_words = epoch_word + 4u;  // 2 words, alternating by item
    // cluster form with push: ranks 1..C-1's partials, one 128 x NT fp32 slot each
    const uint32_t recv = stage0 + (uint32_t)S * kStageBytes + 512u;
    constexpr uint32_t kPartBytes = (uint32_t)kBlockM * NT * 4u;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar + 8u * s, 1);
            mbar_init(empty_bar + 8u * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar + 8u * a, 1);
            mbar_init(acce_bar + 8u * a, 4);  // one arrival per epilogue warp
        }
        mbar_init(done_bar, 1);
        if (p.cluster > 1)
            for (int q = 0; q < 4; ++q)
                mbar_init(ready_bar + 8u * q, (uint32_t)p.cluster - 1u);  // one arrival per other rank
        st_shared_u32(abort_flag, 0u);
        fence_mbarrier_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmL);
        prefetch_tensormap(&tmS);
    }
    if (p.cluster > 1) {
        __syncwarp();
        cluster_arrive_wait();  // every rank's barriers are initialised before any remote arrive
    } else {
        __syncthreads();
    }
    if (warp == 2) {
        tmem_alloc<1>(tmem_slot, kAllocCols);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = ld_shared_u32(tmem_slot);
    // Everything above touched only this CTA's shared and tensor memory, and so
    // does the work split below (kernel parameters only): both may overlap the
    // previous kernel on the stream.  The producer and the epilogue wait for
    // that kernel before their first global access; the MMA issuer touches
    // only shared and tensor memory.

    WaitCtl ctl;
    ctl.abort_flag = abort_flag;
    ctl.peer_abort_flag = 0u;
    ctl.err = p.err;
    ctl.set_limit(p.watchdog_ns);

    const int32_t KB = p.num_k_blocks;
    const int32_t G = (int32_t)gridDim.x;
    const int32_t j = (int32_t)blockIdx.x;
    const int64_t ub = thin_begin(p.units, G, j);
    const int64_t ue = thin_begin(p.units, G, j + 1);
    const int64_t t_first = ub / KB;
    const int64_t t_last = (ue - 1) / KB;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        grid_dependency_wait();
        int s = 0;
        uint32_t ph = 0;
        int32_t it = 0;
        bool ok = true;
        for (int64_t t = t_first; ok && t <= t_last; ++t) {
            const int32_t kb0 = (int32_t)(ub > t * KB ? ub - t * KB : 0);
            const int32_t kb1 = (int32_t)(ue < (t + 1) * KB ? ue - t * KB : KB);
            const int32_t y = (int32_t)(t * kBlockM);
            for (int32_t kb = kb0; kb < kb1; ++kb) {
                if (!ctl.wait<false>(empty_bar + 8u * s, ring_empty_parity(ph), kRoleProducer, (uint32_t)s)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = full_bar + 8u * s;
                const uint32_t sa = stage0 + (uint32_t)s * kStageBytes;
                if (it != p.fault_skip_it) {
                    mbar_arrive_expect_tx(fb, kStageBytes);
                    tma_load_2d(sa, &tmL, kb * kBlockK, y, fb);
                    tma_load_2d(sa + kLBytes, &tmS, kb * kBlockK, 0, fb);
                }
                ++it;
                ring_advance(s, ph, S);
            }
        }
        grid_launch_dependents();
        // Teardown: the last S loads may still be in flight if a role gave up.
        const int32_t n = it < S ? it : S;
        for (int32_t d = 1; d <= n; ++d) {
            const int32_t i = it - d;
            if (i == p.fault_skip_it)
                continue;
            ctl.wait_drain<false>(full_bar + 8u * (uint32_t)ring_stage_of(i, S), ring_parity_of(i, S),
                                  (uint32_t)ring_stage_of(i, S));
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        const uint64_t ldesc0 = smem_desc_sw128(stage0);
        const uint64_t sdesc0 = smem_desc_sw128(stage0 + kLBytes);
        int s = 0;
        uint32_t ph = 0;
        int acc = 0;
        uint32_t acc_ph = 0;
        bool ok = true;
        for (int64_t t = t_first; ok && t <= t_last; ++t) {
            const int32_t kb0 = (int32_t)(ub > t * KB ? ub - t * KB : 0);
            const int32_t kb1 = (int32_t)(ue < (t + 1) * KB ? ue - t * KB : KB);
            if (!ctl.wait<false>(acce_bar + 8u * acc, acc_ph ^ 1u, kRoleMmaAcc, (uint32_t)acc)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * NT);
            for (int32_t kb = kb0; kb < kb1; ++kb) {
                if (!ctl.wait<false>(full_bar + 8u * s, ring_full_parity(ph), kRoleMmaFull, (uint32_t)s)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t step = (uint64_t)(((uint32_t)s * kStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kBlockK / 16; ++kk)
                    mma_bf16<1>(d_tmem, ldesc0 + step + 2u * kk, sdesc0 + step + 2u * kk, kIdesc,
                                (kb != kb0 || kk != 0) ? 1u : 0u);
                mma_commit(empty_bar + 8u * s);
                ring_advance(s, ph, S);
            }
            if (!ok)
                break;
            mma_commit(accf_bar + 8u * acc);
            acc ^= 1;
            if (acc == 0)
                acc_ph ^= 1u;
        }
        // no MMA may still be writing tensor memory when it is freed
        mma_commit(done_bar);
        ctl.wait_drain<false>(done_bar, 0u, 0xFFFu);
    } else if (warp >= 4) {
        // ---------------- epilogue ----------------
        grid_dependency_wait();
        if (threadIdx.x == 128) {
            // this launch's epoch; the last CTA to read it advances it (the
            // acquire-release add orders every CTA's read before that store)
            const uint32_t ep = thin_ld_relaxed_u32(p.sync);
            st_volatile_shared_u32(epoch_word, ep);
            uint32_t before;
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(before) : "l"(p.sync + 1) : "memory");
            if (before == (uint32_t)G - 1u) {
                const uint32_t next = ep + 1u == 0u ? 1u : ep + 1u;
                asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" ::"l"(p.sync + 1) : "memory");
                asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p.sync), "r"(next) : "memory");
            }
        }
        named_barrier_sync(1u, 128u);
        const uint32_t epoch = ld_volatile_shared_u32(epoch_word);
        const int q = warp & 3;  // tensor-memory lane quadrant
        const int32_t row_in_tile = q * 32 + lane;
        int acc = 0;
        uint32_t acc_ph = 0;
        uint32_t item_parity = 0;
        for (int64_t t = t_first; t <= t_last; ++t) {
            const int32_t kb0 = (int32_t)(ub > t * KB ? ub - t * KB : 0);
            const int32_t kb1 = (int32_t)(ue < (t + 1) * KB ? ue - t * KB : KB);
            // One thread waits for the accumulator and posts the outcome to all
            // four warps, so that they all take the same branch; the posted word
            // alternates with the item, so a warp one item behind reads its own.
            const uint32_t go = go_words + 4u * item_parity;
            item_parity ^= 1u;
            if (threadIdx.x == 128)
                st_volatile_shared_u32(
                    go, ctl.wait<false>(accf_bar + 8u * acc, acc_ph, kRoleEpilogue, (uint32_t)acc) ? 1u : 0u);
            named_barrier_sync(1u, 128u);
            if (ld_volatile_shared_u32(go) == 0u)
                break;
            tc_fence_after_sync();
            float v[NT];
            {
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * NT);
                uint32_t r[16];
#pragma unroll
                for (int c = 0; c < NT / 16; ++c) {
                    tmem_load_32x16(taddr + (uint32_t)(c * 16), r);
                    tmem_load_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        asm volatile("" : "+r"(r[i])::"memory");
                        v[c * 16 + i] = __uint_as_float(r[i]);
                    }
                }
            }
            // every read of this accumulator is done: hand it back to the MMA warp
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acce_bar + 8u * acc);
            acc ^= 1;
            if (acc == 0)
                acc_ph ^= 1u;

            const int64_t r = t * kBlockM + row_in_tile;
            // the CTA's last item is stored by TMA from the drained ring
            const bool tma_store = p.d_tma && t == t_last;
            if (kb0 == 0 && kb1 == KB) {  // this range holds the whole tile
                if (tma_store)
                    thin_store_tile_tma<NT>(v, row_in_tile, t, stage0, &tmD, p);
                else
                    thin_store_row<NT>(v, r, p);
                continue;
            }
            if (p.cluster > 1) {
                // Cluster form: this CTA's only item is rank r's share of tile c.
                // The ring is drained (every load landed, and the MMAs that read
                // it completed before the accumulator was handed over), so its
                // first bytes hold the partial, as float4 columns of 128 rows.
                const uint32_t part = stage0 + (uint32_t)row_in_tile * 16u;
                if (kb0 > 0) {
                    if (p.push) {
                        const uint32_t dst = mapa_shared(
                            recv + (cluster_ctarank() - 1u) * kPartBytes + (uint32_t)row_in_tile * 16u, 0u);
#pragma unroll
                        for (int i = 0; i < NT; i += 4)
                            st_shared_cluster_v4(dst + (uint32_t)((i >> 2) * kBlockM) * 16u, __float_as_uint(v[i]),
                                                 __float_as_uint(v[i + 1]), __float_as_uint(v[i + 2]),
                                                 __float_as_uint(v[i + 3]));
                    } else {
#pragma unroll
                        for (int i = 0; i < NT; i += 4)
                            st_shared_v4(part + (uint32_t)((i >> 2) * kBlockM) * 16u, __float_as_uint(v[i]),
                                         __float_as_uint(v[i + 1]), __float_as_uint(v[i + 2]),
                                         __float_as_uint(v[i + 3]));
                    }
                    __syncwarp();  // the warp's stores come before lane 0's release
                    if (lane == 0)
                        mbar_arrive_cluster(mapa_shared(ready_bar + 8u * (uint32_t)q, 0u));
                    continue;
                }
                uint32_t ok = 1u;
                if (lane == 0)
                    ok = ctl.wait<true>(ready_bar + 8u * (uint32_t)q, 0u, kRoleFixup, (uint32_t)q) ? 1u : 0u;
                __syncwarp();  // lane 0's acquire comes before the lanes' loads
                // if the watchdog gave up, the rows are stored unsummed (the
                // status says so): every warp still reaches the store
                const bool have_parts = __shfl_sync(0xFFFFFFFFu, ok, 0) != 0u;
                for (int rk = 1; have_parts && rk < p.cluster; ++rk) {
                    // all of a rank's loads first, then the adds: a remote
                    // round trip each, overlapped rather than one after another
                    uint32_t w[NT];
                    if (p.push) {
                        const uint32_t lp = recv + (uint32_t)(rk - 1) * kPartBytes + (uint32_t)row_in_tile * 16u;
#pragma unroll
                        for (int i = 0; i < NT; i += 4)
                            ld_shared_v4(lp + (uint32_t)((i >> 2) * kBlockM) * 16u, w[i], w[i + 1], w[i + 2], w[i + 3]);
                    } else {
                        const uint32_t rp = mapa_shared(part, (uint32_t)rk);
#pragma unroll
                        for (int i = 0; i < NT; i += 4)
                            ld_shared_cluster_v4(rp + (uint32_t)((i >> 2) * kBlockM) * 16u, w[i], w[i + 1], w[i + 2],
                                                 w[i + 3]);
                    }
#pragma unroll
                    for (int i = 0; i < NT; ++i)
                        v[i] += __uint_as_float(w[i]);
                }
                if (tma_store)
                    thin_store_tile_tma<NT>(v, row_in_tile, t, stage0, &tmD, p);
                else
                    thin_store_row<NT>(v, r, p);
                continue;
            }
            // A piece of a split tile.  The piece that holds k-block 0 owns the
            // tile: it is always the last item of its range, while the other
            // pieces (the start of a later range, or a whole later range) leave
            // their fp32 partials in workspace slots and raise one flag per
            // warp to this launch's epoch.  Each owner warp waits for the flag
            // of the same warp of every later piece, adds those partials to its
            // own sums in range order (a fixed order, so the result does not
            // depend on which piece finishes first) and stores its 32 rows.  A
            // slot holds the 128 x NT partial as NT / 4 columns of float4, each
            // column the 128 rows in order, so that a warp's 32 rows of one
            // column are 512 contiguous bytes.
            if (kb0 > 0) {
                const int32_t slot = thin_slot(p.units, G, KB, j, t);
                float4 *const mine =
                    reinterpret_cast<float4 *>(p.partials) + (size_t)slot * (kBlockM * NT / 4) + row_in_tile;
#pragma unroll
                for (int i = 0; i < NT; i += 4)
                    __stcg(mine + (i >> 2) * kBlockM, make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
                __syncwarp();  // the warp's stores come before lane 0's release
                if (lane == 0)
                    st_release_gpu_u32(p.flags + (size_t)slot * 4 + q, epoch);
                continue;
            }
            const int32_t jl = thin_range_of(p.units, G, (t + 1) * KB - 1);
            for (int32_t jj = j + 1; jj <= jl; ++jj) {
                const int32_t sj = thin_slot(p.units, G, KB, jj, t);
                uint32_t ok = 1u;
                if (lane == 0)
                    ok = thin_poll_flag(ctl, p.flags + (size_t)sj * 4 + q, epoch) ? 1u : 0u;
                __syncwarp();  // lane 0's acquire comes before the lanes' loads
                if (__shfl_sync(0xFFFFFFFFu, ok, 0) == 0u)
                    break;  // the watchdog gave up: the rows are stored unsummed, the status says so
                const float4 *part =
                    reinterpret_cast<const float4 *>(p.partials) + (size_t)sj * (kBlockM * NT / 4) + row_in_tile;
#pragma unroll
                for (int i = 0; i < NT; i += 4) {
                    const float4 f = __ldcg(part + (i >> 2) * kBlockM);
                    v[i] += f.x;
                    v[i + 1] += f.y;
                    v[i + 2] += f.z;
                    v[i + 3] += f.w;
                }
            }
            if (tma_store)
                thin_store_tile_tma<NT>(v, row_in_tile, t, stage0, &tmD, p);
            else
                thin_store_row<NT>(v, r, p);
        }
    }

    // ---------------- teardown ----------------
    tc_fence_before_sync();
    if (p.cluster > 1) {
        __syncwarp();
        cluster_arrive_wait();  // rank 0 may still read the others' shared memory
    } else {
        __syncthreads();
    }
    if (warp == 2) {
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, kAllocCols);
    }
}

}  // namespace wstma
