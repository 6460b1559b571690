// Host-side check of the GEMM kernel's work split and tile order, compiled
// from the kernel's own header (gemm_common.cuh) and run on the CPU.
//
// For every layout the planner can produce -- the partial-last-wave stream-K
// split (T >= C) and the head/tail split (T < C, every head H and every
// number n of tail ranges) -- it walks each cluster's WorkIter sequence and
// checks that:
//   - every (tile, k-block) is computed by exactly one item;
//   - each split tile has exactly one owner (the item holding k-block 0);
//   - the contributors the owner's ContribIter lists are exactly the items
//     that computed the tile's other k-blocks, and their workspace slots are
//     distinct and inside the workspace the planner allocates;
//   - no cluster waits behind its own contributions: in the partial-wave form
//     a contributor is its cluster's first item, and in the head/tail form a
//     head is its cluster's only item and tail clusters own nothing;
// and that tile_coord maps [0, T) one to one onto the tile grid.
// Prints "ok" and exits 0, or prints the first failure and exits 1.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <set>
#include <vector>

#include "gemm_common.cuh"

using namespace wstma;

namespace {

int failures = 0;

#define CHECK(cond, ...)                                                            \
    do {                                                                            \
        if (!(cond)) {                                                              \
            if (failures++ == 0) {                                                  \
                std::printf("FAIL %s:%d: %s: ", __FILE__, __LINE__, #cond);         \
                std::printf(__VA_ARGS__);                                           \
                std::printf("\n");                                                  \
            }                                                                       \
            return;                                                                 \
        }                                                                           \
    } while (0)

GemmParams base(int T, int KB)
{
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    p.num_tiles = T;
    p.num_k_blocks = KB;
    return p;
}

// Items of the first tile that range j touches; the planner's workspace has
// room for the largest such count per range (sk_pieces).
int max_tiles_per_range(int64_t U, int64_t L, int n)
{
    int most = 1;
    for (int j = 0; j < n; ++j) {
        const int64_t b = (int64_t)j * U / n, e = (int64_t)(j + 1) * U / n;
        if (e > b)
            most = std::max<int>(most, (int)((e - 1) / L - b / L + 1));
    }
    return most;
}

// Walks the layout described by p on C clusters; slots = workspace size.
void check_layout(const GemmParams &p, int C, int slots)
{
    const int T = p.num_tiles, KB = p.num_k_blocks;
    std::vector<int> cover((size_t)T * KB, -1);
    std::map<int, int> owner_of;                   // tile -> owner cluster
    std::map<int, std::multiset<int>> contrib_of;  // tile -> contributor slots
    std::set<int> used;
    for (int c = 0; c < C; ++c) {
        WorkIter wi;
        wi.init(p, c, C);
        WorkItem w;
        int idx = 0, owners = 0, contribs = 0;
        while (wi.next(w)) {
            CHECK(w.tile >= 0 && w.tile < T && w.kb0 >= 0 && w.kb0 < w.kb1 && w.kb1 <= KB,
                  "cluster %d item %d: tile %d k [%d,%d)", c, idx, w.tile, w.kb0, w.kb1);
            for (int k = w.kb0; k < w.kb1; ++k) {
                int &cv = cover[(size_t)w.tile * KB + k];
                CHECK(cv < 0, "tile %d k-block %d computed by clusters %d and %d", w.tile, k, cv, c);
                cv = c;
            }
            if (w.kb0 == 0 && w.kb1 < KB) {
                CHECK(owner_of.count(w.tile) == 0, "tile %d has two owners", w.tile);
                owner_of[w.tile] = c;
                ++owners;
                if (p.sk_head > 0)
                    CHECK(idx == 0, "head/tail owner item is not cluster %d's first", c);
            }
            if (w.kb0 > 0) {
                const int j = p.sk_head > 0 ? c - p.sk_tiles : c;
                CHECK(j >= 0, "cluster %d contributes but has no range", c);
                const int s = sk_slot(p, j, sk_begin(p, j, sk_ranges(p, C)), w.tile);
                CHECK(s >= 0 && s < slots, "slot %d outside [0,%d)", s, slots);
                CHECK(used.insert(s).second, "slot %d used twice", s);
                contrib_of[w.tile].insert(s);
                ++contribs;
                if (p.sk_head == 0)
                    CHECK(idx == 0, "partial-wave contributor is not cluster %d's first item", c);
            }
            ++idx;
        }
        if (p.sk_head > 0) {
            if (c < p.sk_tiles)
                CHECK(idx == 1 && owners == 1, "head cluster %d has %d items", c, idx);
            else
                CHECK(owners == 0, "tail cluster %d owns a tile", c);
        } else {
            CHECK(contribs <= 1, "cluster %d contributes %d times", c, contribs);
        }
    }
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < KB; ++k)
            CHECK(cover[(size_t)t * KB + k] >= 0, "tile %d k-block %d not computed", t, k);
    for (auto &kv : contrib_of)
        CHECK(owner_of.count(kv.first), "tile %d has contributors but no owner", kv.first);
    for (auto &kv : owner_of) {
        ContribIter ci;
        ci.init(p, kv.first, kv.second, C);
        std::multiset<int> listed;
        int s;
        while (ci.next(p, s))
            listed.insert(s);
        CHECK(listed == contrib_of[kv.first], "tile %d: owner lists %zu contributors, %zu exist", kv.first,
              listed.size(), contrib_of[kv.first].size());
        CHECK(!listed.empty(), "split tile %d has no contributor", kv.first);
    }
}

void check_partial_wave(int T, int KB, int C)
{
    GemmParams p = base(T, KB);
    const int rem = T % C;
    if (rem) {
        p.sk_tiles = rem;
        p.sk_units = (int64_t)rem * KB;
        p.sk_pieces = 1;
    }
    check_layout(p, C, C);
}

void check_head_tail(int T, int KB, int n, int H)
{
    GemmParams p = base(T, KB);
    const int64_t L = KB - H;
    p.sk_tiles = T;
    p.sk_head = H;
    p.sk_units = T * L;
    p.sk_pieces = max_tiles_per_range(p.sk_units, L, n);
    check_layout(p, T + n, n * p.sk_pieces);
}

void check_tile_order(int mb, int nb, int group, int serp)
{
    GemmParams p = base(mb * nb, 1);
    p.num_m_blocks = mb;
    p.num_n_blocks = nb;
    p.raster_group = group;
    p.serpentine = serp;
    std::vector<int> seen((size_t)mb * nb, 0);
    for (int t = 0; t < mb * nb; ++t) {
        const TileCoord tc = tile_coord(t, p);
        CHECK(tc.mb >= 0 && tc.mb < mb && tc.nb >= 0 && tc.nb < nb, "tile %d -> (%d,%d)", t, tc.mb, tc.nb);
        CHECK(seen[(size_t)tc.mb * nb + tc.nb]++ == 0, "(%d,%d) reached twice", tc.mb, tc.nb);
    }
}

}  // namespace

int main()
{
    const int kbs[] = {1, 2, 3, 5, 8, 13, 64, 65, 129};
    long layouts = 0;
    for (int C = 1; C <= 24; ++C)
        for (int T = 1; T <= 60; ++T)
            for (int KB : kbs) {
                if (T >= C) {
                    check_partial_wave(T, KB, C);
                    ++layouts;
                    continue;
                }
                for (int n = 1; n <= C - T; ++n)
                    for (int H = 1; H < KB; ++H) {
                        if (KB > 16 && H > 3 && H < KB - 3 && H % 7 != 0)
                            continue;
                        check_head_tail(T, KB, n, H);
                        ++layouts;
                    }
            }
    // the full GPU's cluster count, with the long-k and square workloads' shapes
    for (int T : {1, 4, 16, 36, 48, 64, 70, 75})
        for (int KB : {64, 128, 256, 512})
            for (int n : {1, 2, 7, 12, 76 - T})
                for (int H : {1, KB / 4, KB / 2, (int)(0.87 * KB), KB - 1}) {
                    if (n > 76 - T || H < 1 || H >= KB)
                        continue;
                    check_head_tail(T, KB, n, H);
                    ++layouts;
                }
    for (int T : {76, 100, 256, 576, 1024, 4096})
        for (int KB : {64, 65, 128}) {
            check_partial_wave(T, KB, 76);
            ++layouts;
        }
    for (int mb = 1; mb <= 33; mb += 4)
        for (int nb = 1; nb <= 33; nb += 3)
            for (int g : {0, 1, 3, 8, 64})
                for (int serp : {0, 1})
                    check_tile_order(mb, nb, g, serp);
    if (failures) {
        std::printf("%d failure(s)\n", failures);
        return 1;
    }
    std::printf("ok %ld layouts\n", layouts);
    return 0;
}
