// Pieces shared by the warp-specialised kernel and the non-specialised
// ablation kernels: the output-tile order and the epilogue store of one chunk.
// The tile order and the stream-K work split are also host functions, so
// that tests can check them on the CPU.
#pragma once

#include "gemm_kernels.h"
#include "ptx.cuh"
#include "ring_index.h"

namespace wstma {

struct TileCoord {
    int32_t mb;  // tile row
    int32_t nb;  // tile column
};

// Linear output-tile index -> tile coordinates.  With raster_group G > 0 the
// tiles are walked in bands of G tile rows, column by column inside a band, so
// the tiles that run at the same time share A and B rows in L2; G = 0 is plain
// row-major order.  With p.serpentine, odd bands walk their columns right to
// left: the first wave of a band then needs the B panels the last wave of the
// previous band has just read.
__host__ __device__ __forceinline__ TileCoord tile_coord(int32_t t, const GemmParams &p)
{
    if (p.raster_group <= 0)
        return {t / p.num_n_blocks, t % p.num_n_blocks};
    const int32_t span = p.raster_group * p.num_n_blocks;
    const int32_t band = t / span;
    const int32_t first = band * p.raster_group;
    const int32_t rows = p.num_m_blocks - first < p.raster_group ? p.num_m_blocks - first : p.raster_group;
    const int32_t r = t - band * span;
    const int32_t col = r / rows;
    return {first + r % rows, (p.serpentine && (band & 1)) ? p.num_n_blocks - 1 - col : col};
}

// ----------------------------------------------------------------- work items
// One item of a cluster's work: k-blocks [kb0, kb1) of output tile `tile`.
struct WorkItem {
    int32_t tile;
    int32_t kb0;
    int32_t kb1;
};

// Stream-K units.  The split tiles' k-blocks that are shared out form a line of
// sk_units units: unit u is k-block sk_head + u % L of tile u / L, with
// L = num_k_blocks - sk_head units per tile.  The line is cut into n
// contiguous, near-equal ranges, range j = [sk_begin(j), sk_begin(j + 1)):
//   sk_head == 0: L = KB, n = C, cluster c takes range c;
//   sk_head  > 0: n = C - sk_tiles, cluster sk_tiles + j takes range j, and
//                 cluster t < sk_tiles computes the head [0, sk_head) of tile t.
// A contributor (an item that does not start at k-block 0) leaves its fp32
// partial in workspace slot sk_slot(); the item that holds k-block 0 (the
// owner) adds every contributor's partial before it stores the tile.
__host__ __device__ __forceinline__ int64_t sk_begin(const GemmParams &p, int32_t j, int32_t n)
{
    return (int64_t)j * p.sk_units / n;
}

__host__ __device__ __forceinline__ int32_t sk_ranges(const GemmParams &p, int32_t C)
{
    return p.sk_head > 0 ? C - p.sk_tiles : C;
}

// Slot of range j's partial of `tile` (its range starts at unit b).  With
// sk_head == 0 a range contributes at most once, its first item; with
// sk_head > 0 every item of a range is a contributor, one per tile.
__host__ __device__ __forceinline__ int32_t sk_slot(const GemmParams &p, int32_t j, int64_t b, int32_t tile)
{
    if (p.sk_head == 0)
        return j;
    const int64_t L = p.num_k_blocks - p.sk_head;
    return j * p.sk_pieces + (tile - (int32_t)(b / L));
}

// A cluster's work, in order: its stream-K items (its range of units, or the
// head of its tile), then the whole tiles sk_tiles + c, sk_tiles + c + C, ...
// Every role of the CTA walks the same sequence.
struct WorkIter {
    int64_t u, u_end, L;
    int32_t koff, dp, C, T, KB;

    __host__ __device__ __forceinline__ void init(const GemmParams &p, int32_t cluster, int32_t nclusters)
    {
        KB = p.num_k_blocks;
        C = nclusters;
        T = p.num_tiles;
        dp = p.sk_tiles + cluster;
        if (p.sk_head > 0 && cluster < p.sk_tiles) {
            L = p.num_k_blocks;
            koff = 0;
            u = (int64_t)cluster * L;
            u_end = u + p.sk_head;
        } else {
            const int32_t j = p.sk_head > 0 ? cluster - p.sk_tiles : cluster;
            const int32_t n = sk_ranges(p, nclusters);
            L = p.num_k_blocks - p.sk_head;
            koff = p.sk_head;
            u = sk_begin(p, j, n);
            u_end = sk_begin(p, j + 1, n);
        }
    }

    __host__ __device__ __forceinline__ bool next(WorkItem &w)
    {
        if (u < u_end) {
            const int64_t t = u / L;
            const int64_t k0 = u - t * L;
            const int64_t k1 = (k0 + (u_end - u) < L) ? k0 + (u_end - u) : L;
            w.tile = (int32_t)t;
            w.kb0 = koff + (int32_t)k0;
            w.kb1 = koff + (int32_t)k1;
            u += k1 - k0;
            return true;
        }
        if (dp < T) {
            w.tile = dp;
            w.kb0 = 0;
            w.kb1 = KB;
            dp += C;
            return true;
        }
        return false;
    }
};

// The contributors to split tile `tile`, whose owner is cluster `owner`: the
// non-empty ranges that reach into the tile's units, in range order.  next()
// gives each one's workspace slot.
struct ContribIter {
    int64_t lo, hi;
    int32_t j, n, tile;

    __host__ __device__ __forceinline__ void init(const GemmParams &p, int32_t tile_, int32_t owner, int32_t C)
    {
        tile = tile_;
        n = sk_ranges(p, C);
        const int64_t L = p.num_k_blocks - p.sk_head;
        lo = (int64_t)tile * L;
        hi = lo + L;
        // sk_head == 0: the owner's own range holds unit lo, the later ones the
        // rest.  sk_head > 0: no range before floor(tile * n / sk_tiles) ends
        // after lo, since that range begins at or before lo.
        j = p.sk_head > 0 ? (int32_t)((int64_t)tile * n / p.sk_tiles) : owner + 1;
    }

    __host__ __device__ __forceinline__ bool next(const GemmParams &p, int32_t &slot)
    {
        for (; j < n; ++j) {
            const int64_t b = sk_begin(p, j, n);
            if (b >= hi)
                return false;
            const int64_t e = sk_begin(p, j + 1, n);
            if (e > b && e > lo) {
                slot = sk_slot(p, j, b, tile);
                ++j;
                return true;
            }
        }
        return false;
    }
};

// Epilogue of one chunk: the warp holds 32 rows x 64 fp32 columns of the
// accumulator (thread = row; v0 = columns 0..31, v1 = columns 32..63).  They
// are rounded to bf16 (nearest even), written to the warp's staging buffer in
// the 128-byte-swizzled layout (16-byte unit u of row r at u ^ (r & 7)), and
// stored to D[y .. y+31][x .. x+63] either by one TMA tensor store (which drops
// rows >= M and whole 16-byte column groups beyond N) or by coalesced, masked
// st.global row by row.  The masked path is taken when D's layout does not
// allow TMA, and for the chunk holding a partial 16-byte group at column N
// (N not a multiple of 8): a TMA store writes that group whole, which would
// touch the padding columns n >= N.
__device__ __forceinline__ void epilogue_store_chunk(const uint32_t (&v0)[32], const uint32_t (&v1)[32],
                                                     uint32_t staging, int lane, bool tma_store,
                                                     const CUtensorMap *tmD, int32_t x, int32_t y,
                                                     const GemmParams &p)
{
    uint32_t pk[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        pk[j] = pack_bf16x2(v0[2 * j], v0[2 * j + 1]);
        pk[16 + j] = pack_bf16x2(v1[2 * j], v1[2 * j + 1]);
    }

    // The staging buffer is free once the previous TMA store finished reading it
    // (or, on the masked path, once every lane finished its loads).
    if (tma_store && lane == 0)
        bulk_wait_read_all();
    __syncwarp();

    const uint32_t row = staging + (uint32_t)lane * 128u;
    const uint32_t sw = (uint32_t)lane & 7u;
#pragma unroll
    for (uint32_t u = 0; u < 8; ++u)
        st_shared_v4(row + ((u ^ sw) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);

    if (tma_store && (x + 64 <= p.N || (p.N & 7) == 0)) {
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0 && x < p.N && y < p.M) {
            tma_store_2d(tmD, staging, x, y);
            bulk_commit_group();
        }
        return;
    }

    __syncwarp();
    const int32_t col = x + 2 * lane;
    const uint32_t unit = (uint32_t)lane >> 2;
    const uint32_t word = ((uint32_t)lane & 3u) << 2;
    uint16_t *const D = static_cast<uint16_t *>(p.D);
    for (int r = 0; r < 32; ++r) {
        const int32_t row_g = y + r;
        if (row_g >= p.M)
            break;
        const uint32_t w = ld_shared_u32(staging + (uint32_t)r * 128u + ((unit ^ ((uint32_t)r & 7u)) << 4) + word);
        if (col < p.N) {
            uint16_t *dst = D + (int64_t)row_g * p.ldd + col;
            if (col + 1 < p.N && (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
                *reinterpret_cast<uint32_t *>(dst) = w;
            } else {
                dst[0] = (uint16_t)(w & 0xFFFFu);
                if (col + 1 < p.N)
                    dst[1] = (uint16_t)(w >> 16);
            }
        }
    }
}

// ----------------------------------------------------------------- fused epilogue
__device__ __forceinline__ void unpack_bf16x8(const uint4 q, float (&f)[8])
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// v <- alpha * v + (beta * C[row][col] + bias[col]) in fp32 for this thread's
// row and the chunk's 64 columns x .. x+63 (v0: x .. x+31, v1: x+32 .. x+63).
// Columns >= N and rows >= M load nothing (their values are never stored).
// Each element of C is read by the thread that later writes the same element
// of D, so C may alias D.
__device__ __forceinline__ void epilogue_fused(uint32_t (&v0)[32], uint32_t (&v1)[32], int32_t x, int32_t row,
                                               const GemmParams &p)
{
    const bool has_c = (p.fused & kFusedC) && row < p.M;
    const bool has_b = (p.fused & kFusedBias) != 0;
    const uint16_t *crow = has_c ? static_cast<const uint16_t *>(p.C) + (int64_t)row * p.ldc : nullptr;
    const uint16_t *bias = static_cast<const uint16_t *>(p.bias);
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const int32_t col = x + 8 * g;
        uint32_t *v = g < 4 ? &v0[8 * g] : &v1[8 * (g - 4)];
        float cv[8], bv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            cv[i] = bv[i] = 0.f;
        if (has_c) {
            if ((p.fused & kFusedCVec) && col + 8 <= p.N) {
                unpack_bf16x8(*reinterpret_cast<const uint4 *>(crow + col), cv);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (col + i < p.N)
                        cv[i] = __uint_as_float((uint32_t)crow[col + i] << 16);
            }
        }
        if (has_b) {
            if ((p.fused & kFusedBiasVec) && col + 8 <= p.N) {
                unpack_bf16x8(__ldg(reinterpret_cast<const uint4 *>(bias + col)), bv);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (col + i < p.N)
                        bv[i] = __uint_as_float((uint32_t)bias[col + i] << 16);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = __float_as_uint(fmaf(p.alpha, __uint_as_float(v[i]), fmaf(p.beta, cv[i], bv[i])));
    }
}

// ----------------------------------------------------------------- stream-K partials
// A CTA's fp32 partial accumulator (128 rows x 256 columns) in its workspace
// slot, laid out as the epilogue holds it: for warp ew, chunk c, the 64 values
// of each lane's row go as 16 float4 groups j, and group j of all 32 lanes is
// 512 contiguous bytes (coalesced stores and loads).  A lane whose row or chunk
// lies outside D (`live` false) neither stores nor reads its part: contributor
// and owner skip the same parts, which matters for thin problems, where most
// of a tile is padding.
__device__ __forceinline__ float4 *partial_addr(float *slot, int ew, int c, int j, int lane)
{
    return reinterpret_cast<float4 *>(slot) + (((ew * 2 + c) * 16 + j) * 32 + lane);
}

__device__ __forceinline__ void partial_store(float *slot, int ew, int c, int lane, bool live,
                                              const uint32_t (&v0)[32], const uint32_t (&v1)[32])
{
    if (!live)
        return;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint32_t *v = j < 8 ? &v0[4 * j] : &v1[4 * (j - 8)];
        __stcg(partial_addr(slot, ew, c, j, lane),
               make_float4(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]),
                           __uint_as_float(v[3])));
    }
}

__device__ __forceinline__ void partial_load(float *slot, int ew, int c, int lane, bool live, uint32_t (&v0)[32],
                                             uint32_t (&v1)[32])
{
    if (!live) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            v0[i] = v1[i] = 0u;
        return;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float4 f = __ldcg(partial_addr(slot, ew, c, j, lane));
        uint32_t *v = j < 8 ? &v0[4 * j] : &v1[4 * (j - 8)];
        v[0] = __float_as_uint(f.x);
        v[1] = __float_as_uint(f.y);
        v[2] = __float_as_uint(f.z);
        v[3] = __float_as_uint(f.w);
    }
}

__device__ __forceinline__ void partial_add(float *slot, int ew, int c, int lane, bool live, uint32_t (&v0)[32],
                                            uint32_t (&v1)[32])
{
    if (!live)
        return;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float4 f = __ldcg(partial_addr(slot, ew, c, j, lane));
        uint32_t *v = j < 8 ? &v0[4 * j] : &v1[4 * (j - 8)];
        v[0] = __float_as_uint(__uint_as_float(v[0]) + f.x);
        v[1] = __float_as_uint(__uint_as_float(v[1]) + f.y);
        v[2] = __float_as_uint(__uint_as_float(v[2]) + f.z);
        v[3] = __float_as_uint(__uint_as_float(v[3]) + f.w);
    }
}

// v += the 32 fp32 columns of tensor memory at taddr (this warp's 32 lanes).
__device__ __forceinline__ void tmem_add_32x32(uint32_t taddr, uint32_t (&v)[32])
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t t[16];
        tmem_load_32x16(taddr + 16u * (uint32_t)h, t);
        tmem_load_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            asm volatile("" : "+r"(t[i])::"memory");
            v[16 * h + i] = __float_as_uint(__uint_as_float(v[16 * h + i]) + __uint_as_float(t[i]));
        }
    }
}

// Lane 0 waits (bounded) until a contributor's flag carries this launch's
// epoch, then the whole warp proceeds; false if the wait gave up.
__device__ __forceinline__ bool warp_wait_flag(const WaitCtl &ctl, const uint32_t *flag, uint32_t epoch, int lane)
{
    uint32_t ok = 1;
    if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t n = 0; ld_acquire_gpu_u32(flag) != epoch; ++n) {
            if (ctl.aborted()) {
                ok = 0;
                break;
            }
            if ((n & 63u) == 63u && (globaltimer_ns() - t0 > ctl.limit_ns || n > (1u << 30))) {
                ctl.fail(kRoleFixup, 0);
                ok = 0;
                break;
            }
            __nanosleep(100);
        }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    return ok != 0;
}

// Lane 0 waits on a barrier for the whole warp and broadcasts the outcome, so
// that a watchdog give-up is warp-uniform before any .sync.aligned tcgen05 op.
template <bool kClusterScope>
__device__ __forceinline__ bool warp_wait(const WaitCtl &ctl, uint32_t bar, uint32_t parity, uint32_t role,
                                          uint32_t where, int lane)
{
    uint32_t ok = 0;
    if (lane == 0)
        ok = ctl.wait<kClusterScope>(bar, parity, role, where) ? 1u : 0u;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    return ok != 0;
}

// ----------------------------------------------------------------- schedule ring
// With the dynamic scheduler the leader CTA's producer decides the work
// sequence (its stream-K share, then whole tiles taken from a global counter)
// and publishes item `seq` in slot seq % kRingSlots of every CTA of the
// cluster.  Each slot has a "full" barrier (count 1, in every CTA) and an
// "empty" barrier on the leader that collects one arrival from each reader:
// the MMA issuer, one epilogue thread per CTA and the peer's producer.  A tile
// of -1 ends the sequence.

// Publisher: wait until the slot's previous item has been read by every
// reader, write the item into this CTA's slot and the peer's, arrive on both
// full barriers.
template <bool kCluster>
__device__ __forceinline__ bool ring_put(const WaitCtl &ctl, uint32_t ring, uint32_t ring_full, uint32_t ring_empty,
                                         uint32_t peer_ring, uint32_t peer_full, int32_t seq, const WorkItem &w)
{
    const uint32_t r = (uint32_t)seq & (uint32_t)(kRingSlots - 1);
    const uint32_t ph = ((uint32_t)seq / (uint32_t)kRingSlots) & 1u;
    if (!ctl.wait<kCluster>(ring_empty + 8u * r, ph ^ 1u, kRoleSched, 0x800u | r))
        return false;
    st_shared_v4(ring + 16u * r, (uint32_t)w.tile, (uint32_t)w.kb0, (uint32_t)w.kb1, 0u);
    mbar_arrive(ring_full + 8u * r);
    if constexpr (kCluster) {
        st_shared_cluster_v4(peer_ring + 16u * r, (uint32_t)w.tile, (uint32_t)w.kb0, (uint32_t)w.kb1, 0u);
        mbar_arrive_cluster(peer_full + 8u * r);  // release.cluster: the item is visible first
    }
    return true;
}

// Reader: wait for item `seq`, copy it, release the slot on the leader's empty
// barrier (`leader_empty` is a shared::cluster address in 2-CTA mode).
template <bool kCluster>
__device__ __forceinline__ bool ring_get(const WaitCtl &ctl, uint32_t ring, uint32_t ring_full, uint32_t leader_empty,
                                         int32_t seq, WorkItem &w)
{
    const uint32_t r = (uint32_t)seq & (uint32_t)(kRingSlots - 1);
    const uint32_t ph = ((uint32_t)seq / (uint32_t)kRingSlots) & 1u;
    if (!ctl.wait<kCluster>(ring_full + 8u * r, ph, kRoleSched, r))
        return false;
    uint32_t a, b, c, d;
    ld_shared_v4(ring + 16u * r, a, b, c, d);
    w.tile = (int32_t)a;
    w.kb0 = (int32_t)b;
    w.kb1 = (int32_t)c;
    if constexpr (kCluster)
        mbar_arrive_cluster(leader_empty + 8u * r);
    else
        mbar_arrive(leader_empty + 8u * r);
    return true;
}

}  // namespace wstma
