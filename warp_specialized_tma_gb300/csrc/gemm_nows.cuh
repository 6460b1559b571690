// The two non-specialised circular-buffer loops that Fuser PR #3446 ("Use
// mbarrier for WAR for circular buffering") compares, on tcgen05: one CTA of
// 128 threads per 128x256 output tile, S-stage ring, prefetch distance S-1.
//
//   kMbarWar = false  (the loop the PR starts from): an elected thread issues
//     the TMA for k-block i+S-1, every thread waits for k-block i to land,
//     the elected thread issues the MMAs, every thread waits for them to
//     retire, and __syncthreads() guards the stage against the next load
//     (write-after-read).
//   kMbarWar = true   (the loop the PR adds): before loading k-block i+S-1 the
//     elected thread waits on that stage's "empty" barrier, which the MMAs of
//     the previous lap arrive on when they retire (tcgen05.commit); nothing
//     else synchronises the block.  Load and compute still share one thread,
//     so issuing MMA i waits behind the retirement of MMA i-1: the false
//     dependency the PR names as the reason to specialise warps.
//
// Both are ablations of the warp-specialised kernel (gemm_ws.cuh), not the
// production path.
#pragma once

#include "gemm_common.cuh"

namespace wstma {

template <bool kMbarWar>
__global__ void __launch_bounds__(kNowsThreads, 1)
    gemm_nows_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmD, const GemmParams p)
{
    constexpr uint32_t kABytes = kBlockM * kBlockK * 2;
    constexpr uint32_t kBBytes = kBlockN * kBlockK * 2;
    constexpr uint32_t kStageBytes = kABytes + kBBytes;
    constexpr uint32_t kIdesc = idesc_bf16_f32(kBlockM, kBlockN);
    constexpr uint32_t kAccCols = kBlockN;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int S = p.stages;
    const uint32_t stage0 = base;
    const uint32_t staging0 = base + (uint32_t)S * kStageBytes;
    const uint32_t full_bar = staging0 + 4u * kStagingBytes;
    const uint32_t empty_bar = full_bar + 8u * S;
    const uint32_t mmadone_bar = empty_bar + 8u * S;
    const uint32_t accf_bar = mmadone_bar + 8u;
    const uint32_t done_bar = accf_bar + 8u;
    const uint32_t tmem_slot = done_bar + 8u;
    const uint32_t abort_flag = tmem_slot + 4u;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool elected = threadIdx.x == 0;

    if (elected) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar + 8u * s, 1);
            mbar_init(empty_bar + 8u * s, 1);
        }
        mbar_init(mmadone_bar, 1);
        mbar_init(accf_bar, 1);
        mbar_init(done_bar, 1);
        st_shared_u32(abort_flag, 0u);
        fence_mbarrier_init();
    }
    __syncthreads();
    if (warp == 0) {
        tmem_alloc<1>(tmem_slot, kAccCols);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = ld_shared_u32(tmem_slot);
    grid_dependency_wait();  // A, B and D are touched only after this point

    WaitCtl ctl;
    ctl.abort_flag = abort_flag;
    ctl.peer_abort_flag = 0u;
    ctl.err = p.err;
    ctl.set_limit(p.watchdog_ns);

    const TileCoord tc = tile_coord((int32_t)blockIdx.x, p);  // one whole tile per CTA (no stream-K)
    const int32_t ya = tc.mb * kBlockM;
    const int32_t yb = tc.nb * kBlockN;
    const int32_t KB = p.num_k_blocks;

    auto issue = [&](int32_t j) {
        if (j == p.fault_skip_it)  // test hook: this stage never fills
            return;
        const uint32_t s = (uint32_t)(j % S);
        const uint32_t sa = stage0 + s * kStageBytes;
        mbar_arrive_expect_tx(full_bar + 8u * s, kStageBytes);
        tma_load_2d(sa, &tmA, j * kBlockK, ya, full_bar + 8u * s);
        tma_load_2d(sa + kABytes, &tmB, j * kBlockK, yb, full_bar + 8u * s);
    };

    int32_t issued = 0;
    bool ok = true;
    if (elected) {
        for (; issued < S - 1 && issued < KB; ++issued)
            issue(issued);
    }

    for (int32_t i = 0; i < KB; ++i) {
        const uint32_t s = (uint32_t)(i % S);
        const uint32_t ph = (uint32_t)((i / S) & 1);
        if (elected && ok) {
            const int32_t j = i + S - 1;
            if (j < KB) {
                if (kMbarWar && j >= S)  // wait-compute: the previous lap's MMAs left the stage
                    ok = ctl.wait<false>(empty_bar + 8u * (uint32_t)(j % S), (uint32_t)(((j / S) - 1) & 1),
                                         kRoleNoWs, (uint32_t)(j % S));
                if (ok) {
                    issue(j);
                    issued = j + 1;
                }
            }
        }
        // wait-load: every thread
        bool mine = ok && ctl.wait<false>(full_bar + 8u * s, ph, kRoleNoWs, s);
        const uint64_t step = (uint64_t)((s * kStageBytes) >> 4);
        const uint64_t ad = smem_desc_sw128(stage0) + step;
        const uint64_t bd = smem_desc_sw128(stage0 + kABytes) + step;
        if (elected && mine) {
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < kBlockK / 16; ++kk)
                mma_bf16<1>(tmem_base, ad + 2u * kk, bd + 2u * kk, kIdesc, (i | kk) != 0 ? 1u : 0u);
            mma_commit(kMbarWar ? (empty_bar + 8u * s) : mmadone_bar);  // arrive-compute
        }
        if constexpr (!kMbarWar) {
            // compute is complete only when the MMAs have read the stage ...
            mine = mine && ctl.wait<false>(mmadone_bar, (uint32_t)(i & 1), kRoleNoWs, 0x800u);
            // ... and the block-wide barrier keeps the next load off it
            if (__syncthreads_or(mine ? 0 : 1)) {
                ok = false;
                break;
            }
        } else if (!mine) {
            ok = false;
            break;
        }
    }

    const bool all_ok = __syncthreads_or(ok ? 0 : 1) == 0;
    if (all_ok) {
        if (elected)
            mma_commit(accf_bar);
        if (warp_wait<false>(ctl, accf_bar, 0u, kRoleNoWs, 0x801u, lane)) {
            tc_fence_after_sync();
            const uint32_t staging = staging0 + (uint32_t)warp * kStagingBytes;
            const uint32_t tbase = tmem_base + ((uint32_t)(warp * 32) << 16);
            const int32_t y = ya + warp * 32;
#pragma unroll 1
            for (int c = 0; c < kBlockN / 64; ++c) {
                uint32_t v0[32], v1[32];
                tmem_load_32x32(tbase + (uint32_t)(c * 64), v0);
                tmem_load_32x32(tbase + (uint32_t)(c * 64 + 32), v1);
                tmem_load_wait();
                reg_fence(v0);
                reg_fence(v1);
                if (p.fused)
                    epilogue_fused(v0, v1, yb + c * 64, y + lane, p);
                epilogue_store_chunk(v0, v1, staging, lane, p.epi_tma != 0, &tmD, yb + c * 64, y, p);
            }
            if (lane == 0)
                bulk_wait_all();
            __syncwarp();
        }
    }

    // teardown: no TMA load and no MMA may still be in flight
    if (elected) {
        const int32_t n = issued < S ? issued : S;
        for (int32_t d = 1; d <= n; ++d) {
            const int32_t j = issued - d;
            if (j == p.fault_skip_it)
                continue;
            ctl.wait_drain<false>(full_bar + 8u * (uint32_t)(j % S), (uint32_t)((j / S) & 1), (uint32_t)(j % S));
        }
        mma_commit(done_bar);
        ctl.wait_drain<false>(done_bar, 0u, 0xFFFu);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, kAccCols);
    }
}

}  // namespace wstma
