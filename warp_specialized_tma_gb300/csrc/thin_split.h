// Work split of the thin kernel (gemm_thin.cuh), shared with the CPU check of
// it (tests/thin_split_check.cpp).  Plain C++: no CUDA types.
//
// The large operand is cut into tiles of 128 rows, each of KB k-blocks, which
// gives U = tiles * KB units.  CTA j of a grid of G (G <= U) takes the
// contiguous units [begin(j), begin(j + 1)), begin(j) = j U / G, and every range
// holds at least one unit.  A range covers whole tiles in its middle; its first
// and its last tile may be partial, and so a range leaves at most two fp32
// partials: slot 2j for its first tile and slot 2j + 1 for its last.  The
// pieces of tile t are the ranges from range_of(t KB) to range_of((t + 1) KB - 1).
// The piece holding the tile's k-block 0 (the owner, see below) adds the
// other pieces' partials, in range order, and stores the tile.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define WSTMA_THIN_FN __host__ __device__ __forceinline__
#else
#define WSTMA_THIN_FN inline
#endif

namespace wstma {

WSTMA_THIN_FN int64_t thin_begin(int64_t U, int32_t G, int32_t j) { return (int64_t)j * U / G; }

// The range that holds unit u (0 <= u < U).
WSTMA_THIN_FN int32_t thin_range_of(int64_t U, int32_t G, int64_t u)
{
    int32_t j = (int32_t)(u * G / U);
    while (j + 1 < G && thin_begin(U, G, j + 1) <= u)
        ++j;
    while (j > 0 && thin_begin(U, G, j) > u)
        --j;
    return j;
}

// Workspace slot of range j's partial of tile t (t is its first or its last tile).
WSTMA_THIN_FN int32_t thin_slot(int64_t U, int32_t G, int32_t KB, int32_t j, int64_t t)
{
    return 2 * j + (t == thin_begin(U, G, j) / KB ? 0 : 1);
}

// The owner of a split tile is the piece that holds its k-block 0, i.e. the
// range thin_range_of(t * KB).  That piece is always the last item of its
// range: a range that starts inside the tile ends in a later tile, and one
// that starts at the tile's first unit without ending at its last one ends
// inside it.  The other pieces leave partials and raise their slots' flags;
// the owner adds them in range order.

// The grid is one CTA per SM; this bounds the partial slots (2 per CTA).
constexpr int32_t kThinMaxGrid = 1024;

// The cluster form (gemm_thin.cuh) is the split above with G = T * C: every
// C-th range starts at a tile boundary (begin(c C) = c KB exactly), so cluster
// c's C ranges lie in tile c, rank r holding k-blocks [floor(r KB / C),
// floor((r + 1) KB / C)), rank 0 holding k-block 0.  C <= KB keeps every range
// non-empty.
constexpr int32_t kThinMaxCluster = 8;            // portable cluster size limit
constexpr int64_t kThinClusterMaxKBlocks = 160;  // automatic cluster form: k-blocks per CTA at most

// The automatic choice: the largest C <= kThinMaxCluster with T * C <= sms,
// C <= KB and all T clusters of C resident at once (resident[C] >= T, where
// resident[c] is how many clusters of c CTAs fit on the device, c = 1..8);
// taken when T * C reaches 60 % of the SMs and each CTA streams at most
// kThinClusterMaxKBlocks k-blocks.  Returns C (1 = one CTA per whole tile), or
// 0 for the split across the SMs.
WSTMA_THIN_FN int32_t thin_auto_cluster(int64_t T, int64_t KB, int32_t sms, const int32_t *resident)
{
    if (T < 1 || KB < 1 || T > sms)
        return 0;
    int64_t c = sms / T;
    if (c > kThinMaxCluster)
        c = kThinMaxCluster;
    if (c > KB)
        c = KB;
    while (c > 1 && resident[c] < T)
        --c;
    if (T * c * 10 >= (int64_t)sms * 6 && (KB + c - 1) / c <= kThinClusterMaxKBlocks)
        return (int32_t)c;
    return 0;
}

}  // namespace wstma
