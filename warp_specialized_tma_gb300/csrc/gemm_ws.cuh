// The persistent, warp-specialised GEMM kernel: D = A * B^T, bf16 in, fp32
// accumulation in tensor memory, bf16 out.
//
// Roles (384 threads, one CTA per SM):
//   warpgroup 0: warp 0 lane 0  = TMA producer (and, with the dynamic scheduler,
//                                 the leader's publisher of the work sequence)
//                warp 1 lane 0  = tcgen05 MMA issuer (leader CTA only in 2-CTA mode)
//                warp 2         = tensor-memory allocator
//                warp 3         = spare
//   warpgroups 1, 2 (warps 4..11) = epilogue: TMEM -> registers -> bf16 -> smem -> TMA store
//
// Fuser issue #3941 ("Allow separate sub-DAG for load and compute warp groups
// with warp-specialized circular buffering") gives the loop structure: the
// producer runs ONE serial loop over the merged (output tile, cta-k) space and
// the stage ring is indexed by that merged counter, while the compute side
// keeps the tile loop and the k loop apart because the store has no k; the
// load warps give registers back and the compute warps take them
// (setmaxnreg).  Fuser PR #3446 ("Use mbarrier for WAR for circular
// buffering") gives the ring: per stage a "full" mbarrier (TMA bytes landed)
// and an "empty" mbarrier (the MMAs reading the stage completed).  On this
// hardware the MMA is asynchronous and retires through tcgen05.commit, so the
// "empty" arrive is the commit itself and the epilogue runs in its own warps
// against two tensor-memory accumulators (accumulator-full / -empty barriers).
// cutlass PR #3316 ("Fix race condition in 2SM TMEM alloc ...") gives the
// 2-CTA rule: both CTAs pass a cluster barrier before the paired
// tcgen05.alloc.
//
// Two schedule options (runtime switches in GemmParams):
//   epilogue  cooperative (default): both epilogue warpgroups drain every tile;
//             ping-pong: warpgroup g drains the tiles of accumulator g, so the
//             two groups alternate tiles (Fuser #3941's second consumer
//             schedule, with TMEM accumulators instead of register ones).
//   tiles     static (default): every role walks the same grid-stride sequence;
//             dynamic: the leader's producer takes whole tiles from a global
//             counter and publishes them through the schedule ring.
//
// Split tiles (stream-K, GemmParams::sk_*): before its whole tiles, each SM
// (pair) may take part of a tile's k-range.  Either the tiles of a partial last
// wave are cut into equal shares, or, with fewer tiles than SM (pairs), every
// tile is cut at one k-block into a head, computed by its owner, and a tail,
// shared by the other SM (pairs).  A contributor leaves its fp32 partial in a
// workspace slot and raises a flag; the owner adds the partials before its
// epilogue stores the tile (gemm_common.cuh: WorkIter, ContribIter).
#pragma once

#include "gemm_common.cuh"

namespace wstma {

template <int CG, bool kSetMaxNReg>
__global__ void __launch_bounds__(kWsThreads, 1)
    gemm_ws_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const GemmParams p)
{
    static_assert(CG == 1 || CG == 2, "one CTA or an SM pair per tile");
    constexpr bool kCluster = (CG == 2);
    constexpr uint32_t kABytes = kBlockM * kBlockK * 2;          // 16 KiB: this CTA's 128 rows of A
    constexpr uint32_t kBRows = kBlockN / CG;                    // rows of B this CTA loads
    constexpr uint32_t kBBytes = kBRows * kBlockK * 2;
    constexpr uint32_t kStageBytes = kABytes + kBBytes;
    constexpr uint32_t kTxBytes = kStageBytes * CG;              // bytes landing on the leader's full barrier
    constexpr uint32_t kIdesc = idesc_bf16_f32(kBlockM * CG, kBlockN);
    constexpr int32_t kTileM = kBlockM * CG;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int S = p.stages;
    // stages released per commit, 1 or 2: as a shift and a mask, since a
    // division would sit on the single MMA thread's critical path
    const uint32_t g_shift = p.stage_group == 2 ? 1u : 0u;
    const uint32_t g_mask = p.stage_group == 2 ? 1u : 0u;
    const uint32_t stage0 = base;
    const uint32_t staging0 = base + (uint32_t)S * kStageBytes;
    const uint32_t ring = staging0 + kEpiWarps * kStagingBytes;  // kRingSlots x 16 B work items
    const uint32_t full_bar = ring + 16u * kRingSlots;
    const uint32_t empty_bar = full_bar + 8u * S;
    const uint32_t accf_bar = empty_bar + 8u * S;
    const uint32_t acce_bar = accf_bar + 16u;
    const uint32_t done_bar = acce_bar + 16u;
    const uint32_t ring_full = done_bar + 8u;
    const uint32_t ring_empty = ring_full + 8u * kRingSlots;
    const uint32_t tmem_slot = ring_empty + 8u * kRingSlots;
    const uint32_t abort_flag = tmem_slot + 4u;
    const uint32_t go_area = abort_flag + 4u;  // 2 groups x 2 parities x 4 words, see the epilogue

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = kCluster ? cluster_ctarank() : 0u;
    const uint32_t acc_cols = (uint32_t)kBlockN * (uint32_t)p.acc_buffers;  // 256 or 512
    const bool pingpong = p.epi_pingpong != 0;
    const bool dyn = p.sched_dynamic != 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar + 8u * s, 1);
            mbar_init(empty_bar + 8u * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar + 8u * a, 1);
            // every warp of the warpgroup(s) that drain accumulator a, in both CTAs
            mbar_init(acce_bar + 8u * a, (pingpong ? kEpiWarps / 2 : kEpiWarps) * CG);
        }
        mbar_init(done_bar, 1);
        for (int r = 0; r < kRingSlots; ++r) {
            mbar_init(ring_full + 8u * r, 1);
            mbar_init(ring_empty + 8u * r, 2 * CG);  // MMA issuer, CG epilogue pollers, CG-1 peer producers
        }
        st_shared_u32(abort_flag, 0u);
        fence_mbarrier_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmD);
    }
    // Both CTAs of a pair have initialised their barriers and are resident
    // before any cross-CTA arrive, TMA completion or the paired allocation.
    if constexpr (kCluster)
        cluster_arrive_wait();
    else
        __syncthreads();

    if (warp == 2) {
        tmem_alloc<CG>(tmem_slot, acc_cols);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = ld_shared_u32(tmem_slot);
    // Everything above touched only this CTA's shared and tensor memory, so it
    // may overlap the previous kernel on the stream.  The roles that read or
    // write global memory (A, B, D, the workspace, the tile counter) -- the
    // producer and the epilogue -- wait for that kernel before their first
    // access; the MMA issuer touches only shared and tensor memory.

    WaitCtl ctl;
    ctl.abort_flag = abort_flag;
    ctl.peer_abort_flag = kCluster ? mapa_shared(abort_flag, rank ^ 1u) : 0u;
    ctl.err = p.err;
    ctl.set_limit(p.watchdog_ns);

    const int32_t cluster_id = (int32_t)blockIdx.x / CG;
    const int32_t num_clusters = (int32_t)gridDim.x / CG;
    const int32_t KB = p.num_k_blocks;
    // readers release ring slots on the leader's empty barriers
    const uint32_t leader_ring_empty = kCluster ? mapa_shared(ring_empty, 0u) : ring_empty;

    if (warp < 4) {
        if constexpr (kSetMaxNReg)
            setmaxnreg_dec<kProducerRegs>();

        // The producer and MMA roles are single threads (lane 0 of their warp).
        // Measured on GB300: a whole-warp loop with one issuing lane reacts to its
        // barrier through a shuffle and starves the ring (producer) or adds
        // per-k-block latency (MMA issuer).
        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer: one loop over (tile, k-block) ----------------
            const uint32_t full_target = kCluster ? mapa_shared(full_bar, 0u) : full_bar;
            const bool publisher = dyn && rank == 0;
            const uint32_t peer_ring = kCluster ? mapa_shared(ring, 1u) : 0u;
            const uint32_t peer_ring_full = kCluster ? mapa_shared(ring_full, 1u) : 0u;
            int s = 0;
            uint32_t ph = 0;
            int32_t it = 0;
            int32_t seq = 0;
            int32_t whole = 0;  // whole-tile items so far: their parity picks the k direction
            bool ok = true;
            bool counter_done = false;
            WorkIter wi;
            wi.init(p, cluster_id, num_clusters);
            if (dyn)
                wi.dp = wi.T;  // whole tiles come from the counter, not from the grid stride
            WorkItem w;
            // The first item of the static schedule and its coordinates depend
            // only on kernel parameters: they are worked out before the wait for
            // the previous kernel, so that the first loads issue as soon as its
            // memory is visible.
            bool first = !dyn;
            bool have0 = false;
            TileCoord tc0 = {0, 0};
            if (first) {
                have0 = wi.next(w);
                if (have0)
                    tc0 = tile_coord(w.tile, p);
            }
            grid_dependency_wait();
            for (;;) {
                bool have;
                if (first) {
                    have = have0;
                } else if (!dyn) {
                    have = wi.next(w);
                } else if (publisher) {
                    // this cluster's stream-K share first, then whole tiles on demand
                    have = wi.next(w);
                    if (!have && !counter_done) {
                        const int32_t t = p.sk_tiles + (int32_t)atomicAdd(p.sched, 1u);
                        if (t < p.num_tiles) {
                            w.tile = t;
                            w.kb0 = 0;
                            w.kb1 = KB;
                            have = true;
                        } else {
                            counter_done = true;
                        }
                    }
                    WorkItem out = w;
                    if (!have)
                        out.tile = -1;
                    if (!ring_put<kCluster>(ctl, ring, ring_full, ring_empty, peer_ring, peer_ring_full, seq, out)) {
                        ok = false;
                        break;
                    }
                    ++seq;
                } else {
                    if (!ring_get<kCluster>(ctl, ring, ring_full, leader_ring_empty, seq, w)) {
                        ok = false;
                        break;
                    }
                    ++seq;
                    have = w.tile >= 0;
                }
                if (!have)
                    break;
                const TileCoord tc = first ? tc0 : tile_coord(w.tile, p);
                first = false;
                const int32_t ya = tc.mb * kTileM + (int32_t)rank * kBlockM;
                const int32_t yb = tc.nb * kBlockN + (int32_t)rank * (int32_t)kBRows;
                // Alternating k direction: all SM pairs are in the same wave of whole
                // tiles at about the same time, and consecutive waves of a band share
                // their A panels.  A wave that walks k in the opposite direction to
                // the previous one starts on the k-slices that wave loaded last, which
                // are still in L2.  The MMA side only counts k-blocks (accumulation
                // starts at the first one it is given), so only the loads change.
                const bool whole_tile = w.kb0 == 0 && w.kb1 == KB;
                const bool rev = p.k_order == 1 && whole_tile && (whole & 1);
                whole += whole_tile ? 1 : 0;
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                    // wait until the MMAs that read this stage (group) one lap ago
                    // have retired; a group of G stages is released by one commit
                    if (ring_group_first(s, g_mask) &&
                        !ctl.wait<kCluster>(empty_bar + 8u * ring_group(s, g_shift), ring_empty_parity(ph),
                                            kRoleProducer, (uint32_t)s)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_target + 8u * s;
                    const uint32_t sa = stage0 + (uint32_t)s * kStageBytes;
                    const int32_t x = (rev ? w.kb0 + w.kb1 - 1 - kb : kb) * kBlockK;
                    if (it != p.fault_skip_it) {
                        if (!kCluster || rank == 0)
                            mbar_arrive_expect_tx(full_bar + 8u * s, kTxBytes);
                        if constexpr (kCluster) {
                            tma_load_2d_pair(sa, &tmA, x, ya, fb);
                            tma_load_2d_pair(sa + kABytes, &tmB, x, yb, fb);
                        } else {
                            tma_load_2d(sa, &tmA, x, ya, fb);
                            tma_load_2d(sa + kABytes, &tmB, x, yb, fb);
                        }
                    }
                    ++it;
                    ring_advance(s, ph, S);
                }
                if (!ok)
                    break;
            }
            if (publisher) {
                // A second end marker: ping-pong epilogue groups read alternate slots.
                if (ok) {
                    WorkItem end = {-1, 0, 0};
                    ring_put<kCluster>(ctl, ring, ring_full, ring_empty, peer_ring, peer_ring_full, seq, end);
                }
                // This cluster takes no more tiles.  The last cluster to get here
                // (every other one has made its last counter access) puts the
                // counter back to 0 for the next launch.
                __threadfence();
                if (atomicAdd(p.sched + 1, 1u) == (uint32_t)num_clusters - 1u) {
                    atomicExch(p.sched, 0u);
                    atomicExch(p.sched + 1, 0u);
                    __threadfence();
                }
            }
            // This CTA issues no more loads: the next kernel on the stream may begin
            // launching (its CTAs start as this grid's CTAs exit).
            grid_launch_dependents();
            // Teardown: the last S loads may still be in flight if a role gave up.
            if (!kCluster || rank == 0) {
                const int32_t n = it < S ? it : S;
                for (int32_t d = 1; d <= n; ++d) {
                    const int32_t j = it - d;
                    if (j == p.fault_skip_it)
                        continue;
                    ctl.wait_drain<kCluster>(full_bar + 8u * (uint32_t)ring_stage_of(j, S), ring_parity_of(j, S),
                                             (uint32_t)ring_stage_of(j, S));
                }
            } else if (ctl.aborted()) {
                // The peer's loads complete on the leader's barriers, which this CTA
                // cannot poll: give them a fixed grace period instead.
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 50000ull) {
                }
            }
        } else if (warp == 1 && lane == 0 && (!kCluster || rank == 0)) {
            // ---------------- MMA issuer: tile { k-block { 4 x tcgen05.mma } } ----------------
            const uint64_t adesc0 = smem_desc_sw128(stage0);
            const uint64_t bdesc0 = smem_desc_sw128(stage0 + kABytes);
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t acc_ph = 0;
            int32_t seq = 0;
            bool ok = true;
            bool ready = false;  // outcome of the look-ahead probe of ring slot (s, ph)
            WorkIter wi;
            wi.init(p, cluster_id, num_clusters);
            WorkItem w;
            for (;;) {
                if (dyn) {
                    if (!ring_get<kCluster>(ctl, ring, ring_full, leader_ring_empty, seq, w)) {
                        ok = false;
                        break;
                    }
                    ++seq;
                    if (w.tile < 0)
                        break;
                } else if (!wi.next(w)) {
                    break;
                }
                // the epilogue has drained this accumulator (one lap ago)
                if (!ctl.wait<kCluster>(acce_bar + 8u * acc, acc_ph ^ 1u, kRoleMmaAcc, (uint32_t)acc)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBlockN);
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!ready && !ctl.wait<kCluster>(full_bar + 8u * s, ring_full_parity(ph), kRoleMmaFull, (uint32_t)s)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t step = (uint64_t)(((uint32_t)s * kStageBytes) >> 4);
                    const uint64_t ad = adesc0 + step;
                    const uint64_t bd = bdesc0 + step;
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk)
                        mma_bf16<CG>(d_tmem, ad + 2u * kk, bd + 2u * kk, kIdesc, (kb != w.kb0 || kk != 0) ? 1u : 0u);
                    // the stage group is free once its MMAs have read it.  One commit
                    // per G k-blocks: measured on GB300, a commit every 4 MMAs keeps the
                    // tensor pipe ~93% busy, one every 8 MMAs keeps it ~100% busy.
                    if (ring_group_last(s, g_mask)) {
                        if constexpr (kCluster)
                            mma_commit_pair(empty_bar + 8u * ring_group(s, g_shift), (uint16_t)0x3);
                        else
                            mma_commit(empty_bar + 8u * ring_group(s, g_shift));
                    }
                    ring_advance(s, ph, S);
                    // Look at the next slot without blocking (try_wait with a zero
                    // suspend hint).  Measured on GB300: a test_wait probe here costs
                    // ~7% of the tensor pipe's throughput, a try_wait probe nothing.
                    ready = mbar_try_wait<kCluster>(full_bar + 8u * s, ring_full_parity(ph), 0u);
                }
                if (!ok)
                    break;
                // the accumulator is complete once every MMA of the tile has retired
                if constexpr (kCluster)
                    mma_commit_pair(accf_bar + 8u * acc, (uint16_t)0x3);
                else
                    mma_commit(accf_bar + 8u * acc);
                if (p.acc_buffers == 2) {
                    acc ^= 1;
                    if (acc == 0)
                        acc_ph ^= 1u;
                } else {
                    acc_ph ^= 1u;
                }
            }
            // no MMA may still be writing tensor memory when it is freed
            if constexpr (kCluster)
                mma_commit_pair(done_bar, (uint16_t)0x1);
            else
                mma_commit(done_bar);
            ctl.wait_drain<kCluster>(done_bar, 0u, 0xFFFu);
        }
    } else {
        if constexpr (kSetMaxNReg)
            setmaxnreg_inc<kConsumerRegs>();

        // ---------------- epilogue: tile { TMEM -> bf16 -> D } ----------------
        grid_dependency_wait();
        // Cooperative: both warpgroups drain every tile, a warp takes 32 rows x
        // 128 columns.  Ping-pong: warpgroup g drains the items that use
        // accumulator g (items g, g+2, ... of the sequence), a warp takes 32 rows
        // x 256 columns.
        const int ew = warp - 4;        // 0..7
        const int q = warp & 3;         // tensor-memory lane quadrant this warp may read
        const int grp = pingpong ? (ew >> 2) : 0;
        const uint32_t group_threads = pingpong ? 128u : (uint32_t)kEpiWarps * 32u;
        const bool poller = pingpong ? (q == 0) : (ew == 0);
        const int nchunks = pingpong ? 4 : 2;
        const int32_t col0 = pingpong ? 0 : (ew >> 2) * 128;
        const int32_t seq_step = pingpong ? 2 : 1;
        const uint32_t staging = staging0 + (uint32_t)ew * kStagingBytes;
        const uint32_t acce_target = kCluster ? mapa_shared(acce_bar, 0u) : acce_bar;
        const bool tma_store = p.epi_tma != 0;
        int acc = grp;
        uint32_t acc_ph = 0;
        uint32_t tile_parity = 0;
        int32_t seq = grp;
        WorkIter wi;
        wi.init(p, cluster_id, num_clusters);
        if (pingpong && grp == 1 && !dyn) {
            WorkItem skip;
            wi.next(skip);
        }
        // Head/tail stream-K owner (cooperative schedule): this cluster's only
        // item is the head of tile cluster_id, accumulating in buffer 0, and
        // buffer 1 stays free.  While the head's MMAs run, the epilogue warps
        // fold each tail's partial into buffer 1 as soon as that tail raises its
        // flag (the tails finish one after another), so after the last MMA the
        // tile's epilogue adds one sum from tensor memory and at most the last
        // tail's partial was read on the critical path.
        const bool parked = p.sk_head > 0 && cluster_id < p.sk_tiles && !pingpong && p.acc_buffers == 2;
        if (parked) {
            const uint32_t spare = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(kBlockN + col0);
            const TileCoord htc = tile_coord(cluster_id, p);  // the head's tile
            const bool row_live = htc.mb * kTileM + (int32_t)rank * kBlockM + q * 32 + lane < p.M;
            ContribIter ci;
            ci.init(p, cluster_id, cluster_id, num_clusters);
            int32_t s2;
            bool first = true;
            while (ci.next(p, s2)) {
                const int32_t slot2 = s2 * CG + (int32_t)rank;
                if (!warp_wait_flag(ctl, p.flags + slot2, p.epoch, lane))
                    break;
#pragma unroll 1
                for (int c = 0; c < nchunks; ++c) {
                    const int32_t col = col0 + c * 64;
                    const int pw = (col >> 7) * 4 + q;
                    const int pc = (col >> 6) & 1;
                    float *const part = p.workspace + (size_t)slot2 * kPartialFloats;
                    const bool live = row_live && htc.nb * kBlockN + col < p.N;
                    uint32_t v0[32], v1[32];
                    if (first) {
                        partial_load(part, pw, pc, lane, live, v0, v1);
                    } else {
                        tmem_load_32x32(spare + (uint32_t)(c * 64), v0);
                        tmem_load_32x32(spare + (uint32_t)(c * 64 + 32), v1);
                        tmem_load_wait();
                        reg_fence(v0);
                        reg_fence(v1);
                        partial_add(part, pw, pc, lane, live, v0, v1);
                    }
                    tmem_store_32x32(spare + (uint32_t)(c * 64), v0);
                    tmem_store_32x32(spare + (uint32_t)(c * 64 + 32), v1);
                }
                // the next tail's pass reads what this one stored
                tmem_store_wait();
                first = false;
            }
        }
        for (;;) {
            // One thread per group polls the accumulator barrier and posts the
            // outcome; the other warps sleep on a named barrier instead of polling
            // (every poll competes with the MMA issuer).  With the static schedule
            // every epilogue thread walks the work sequence itself and prepares
            // the item before the group meets, so that only the broadcast stands
            // between the accumulator becoming ready and the first tensor-memory
            // load; with the dynamic scheduler the poller also posts the item it
            // took from the schedule ring.  The posted words alternate with the
            // item parity, so a warp that is one item behind never reads the next
            // item's words.
            const uint32_t go = go_area + 16u * (2u * (uint32_t)grp + tile_parity);
            WorkItem w = {0, 0, 0};
            uint32_t st = 1;  // 1 = drain item w, 2 = no more items, 0 = gave up
            if (!dyn) {
                if (!wi.next(w)) {
                    st = 2;
                } else if (pingpong) {
                    WorkItem skip;  // the other group's item
                    wi.next(skip);
                }
            }
            TileCoord tc = {0, 0};
            if (!dyn && st == 1u)
                tc = tile_coord(w.tile, p);
            if (poller) {
                if (dyn && lane == 0) {
                    if (!ring_get<kCluster>(ctl, ring, ring_full, leader_ring_empty, seq, w))
                        st = 0;
                    else if (w.tile < 0)
                        st = 2;
                }
                st = __shfl_sync(0xFFFFFFFFu, st, 0);
                if (st == 1u &&
                    !warp_wait<kCluster>(ctl, accf_bar + 8u * acc, acc_ph, kRoleEpilogue, (uint32_t)acc, lane))
                    st = 0;
                if (lane == 0) {
                    if (dyn) {
                        st_volatile_shared_u32(go + 4u, (uint32_t)w.tile);
                        st_volatile_shared_u32(go + 8u, (uint32_t)w.kb0);
                        st_volatile_shared_u32(go + 12u, (uint32_t)w.kb1);
                    }
                    st_volatile_shared_u32(go, st);
                }
            }
            named_barrier_sync(1u + (uint32_t)grp, group_threads);
            if (ld_volatile_shared_u32(go) != 1u)
                break;
            if (dyn) {
                w.tile = (int32_t)ld_volatile_shared_u32(go + 4u);
                w.kb0 = (int32_t)ld_volatile_shared_u32(go + 8u);
                w.kb1 = (int32_t)ld_volatile_shared_u32(go + 12u);
                tc = tile_coord(w.tile, p);
            }
            seq += seq_step;
            tc_fence_after_sync();
            const int32_t y = tc.mb * kTileM + (int32_t)rank * kBlockM + q * 32;
            // A stream-K item that does not start at k-block 0 is a contributor: it
            // leaves its fp32 partial for the tile's owner.  The item holding
            // k-block 0 of a split tile is the owner: it adds every contributor's
            // partial before storing.
            const bool contributor = w.kb0 > 0;
            const bool owner = w.kb0 == 0 && w.kb1 < KB;
            int32_t slot_id = 0;
            if (contributor) {
                const int32_t j = p.sk_head > 0 ? cluster_id - p.sk_tiles : cluster_id;
                slot_id = sk_slot(p, j, sk_begin(p, j, sk_ranges(p, num_clusters)), w.tile) * CG + (int32_t)rank;
            }
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBlockN + col0);
#pragma unroll 1
            for (int c = 0; c < nchunks; ++c) {
                const int32_t col = col0 + c * 64;  // column of the chunk inside the tile
                // the partials keep one layout whatever the schedule: the chunk of
                // column `col` and quadrant q belongs to (virtual) warp pw, chunk pc
                const int pw = (col >> 7) * 4 + q;
                const int pc = (col >> 6) & 1;
                uint32_t v0[32], v1[32];
                tmem_load_32x32(tbase + (uint32_t)(c * 64), v0);
                tmem_load_32x32(tbase + (uint32_t)(c * 64 + 32), v1);
                tmem_load_wait();
                reg_fence(v0);
                reg_fence(v1);
                if (owner && parked) {
                    // the tails' summed partials, parked in the other accumulator
                    const uint32_t spare = tbase + (uint32_t)kBlockN + (uint32_t)(c * 64);
                    tmem_add_32x32(spare, v0);
                    tmem_add_32x32(spare + 32u, v1);
                }
                if (c == nchunks - 1) {
                    // every read of this accumulator is done: hand it back to the MMA warp
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (kCluster)
                            mbar_arrive_cluster_handoff(acce_target + 8u * acc);
                        else
                            mbar_arrive(acce_bar + 8u * acc);
                    }
                }
                const int32_t x = tc.nb * kBlockN + col;
                // parts of a split tile outside D are neither stored nor read
                const bool live = y + lane < p.M && x < p.N;
                if (contributor) {
                    partial_store(p.workspace + (size_t)slot_id * kPartialFloats, pw, pc, lane, live, v0, v1);
                    continue;
                }
                if (owner && !parked) {
                    ContribIter ci;
                    ci.init(p, w.tile, cluster_id, num_clusters);
                    int32_t s2;
                    while (ci.next(p, s2)) {
                        const int32_t slot2 = s2 * CG + (int32_t)rank;
                        if (c == 0 && !warp_wait_flag(ctl, p.flags + slot2, p.epoch, lane))
                            break;
                        partial_add(p.workspace + (size_t)slot2 * kPartialFloats, pw, pc, lane, live, v0, v1);
                    }
                }
                if (p.fused)
                    epilogue_fused(v0, v1, x, y + lane, p);
                epilogue_store_chunk(v0, v1, staging, lane, tma_store, &tmD, x, y, p);
            }
            if (contributor) {
                // publish the partial: every writer fences, then one thread raises the flag
                __threadfence();
                named_barrier_sync(3u + (uint32_t)grp, group_threads);
                if (poller && lane == 0)
                    st_release_gpu_u32(p.flags + slot_id, p.epoch);
            }
            if (pingpong) {
                acc_ph ^= 1u;
            } else if (p.acc_buffers == 2) {
                acc ^= 1;
                if (acc == 0)
                    acc_ph ^= 1u;
            } else {
                acc_ph ^= 1u;
            }
            tile_parity ^= 1u;
        }
        // The staging buffers must have been read before the CTA exits; the
        // stores' writes to D complete before the grid is reported complete.
        if (lane == 0)
            bulk_wait_read_all();
        __syncwarp();
    }

    // ---------------- teardown ----------------
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (kCluster)
        cluster_arrive_wait();  // the peer is done with its reads and the leader's MMAs into it
    if (warp == 2) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem_base, acc_cols);
    }
}

}  // namespace wstma
