// CPU check of the thin kernel's work split (warp_specialized_tma_gb300/csrc/
// thin_split.h), compiled from the kernel's own header.  For grids of G CTAs
// over T tiles of KB k-blocks (G <= T * KB) it checks that every unit belongs
// to exactly one range and every range is non-empty; that range_of inverts
// the split; that a tile covered by one range is whole and every other tile's
// pieces are the ranges from range_of(first unit) to range_of(last unit); that
// each piece's workspace slot is its range's first- or last-tile slot, and
// that no two pieces share a slot; and that the owner of each split tile (the
// piece holding its k-block 0, range_of(t * KB)) is the last tile of its range,
// so that an owner never waits for anything before its own last item, and the
// other pieces are not.  For the cluster form (G = T * C, C <= KB) it checks
// that cluster c's C ranges lie in tile c with rank r holding k-blocks
// [floor(r KB / C), floor((r + 1) KB / C)); and it checks the automatic cluster
// size against a device model of 8 clusters-capable groups of 19 SMs: fixed
// cases, and on a sweep that the choice meets every condition and no larger
// size would.
// Prints "ok" and exits 0, or prints the first failure and exits 1.
#include <cstdio>
#include <set>
#include <vector>

#include "thin_split.h"

using namespace wstma;

namespace {

int failures = 0;

#define CHECK(cond, ...)                                                    \
    do {                                                                    \
        if (!(cond)) {                                                      \
            if (failures++ == 0) {                                          \
                std::printf("FAIL %s:%d: %s: ", __FILE__, __LINE__, #cond); \
                std::printf(__VA_ARGS__);                                   \
                std::printf("\n");                                          \
            }                                                               \
            return;                                                         \
        }                                                                   \
    } while (0)

void check_split(int64_t T, int32_t KB, int32_t G)
{
    const int64_t U = T * KB;
    std::vector<int> owner((size_t)U, -1);
    for (int32_t j = 0; j < G; ++j) {
        const int64_t b = thin_begin(U, G, j), e = thin_begin(U, G, j + 1);
        CHECK(e > b, "T=%lld KB=%d G=%d: range %d empty", (long long)T, KB, G, j);
        for (int64_t u = b; u < e; ++u) {
            CHECK(owner[(size_t)u] < 0, "unit %lld in two ranges", (long long)u);
            owner[(size_t)u] = j;
        }
    }
    CHECK(thin_begin(U, G, 0) == 0 && thin_begin(U, G, G) == U, "ranges do not cover [0, U)");
    for (int64_t u = 0; u < U; ++u)
        CHECK(thin_range_of(U, G, u) == owner[(size_t)u], "range_of(%lld) = %d, not %d", (long long)u,
              thin_range_of(U, G, u), owner[(size_t)u]);
    std::set<int32_t> slots;
    for (int64_t t = 0; t < T; ++t) {
        const int32_t jf = thin_range_of(U, G, t * KB), jl = thin_range_of(U, G, (t + 1) * KB - 1);
        for (int32_t j = jf; j <= jl; ++j) {
            const int64_t b = thin_begin(U, G, j), e = thin_begin(U, G, j + 1);
            const int64_t kb0 = b > t * KB ? b - t * KB : 0;
            const int64_t kb1 = e < (t + 1) * KB ? e - t * KB : KB;
            CHECK(kb0 < kb1, "tile %lld piece %d empty", (long long)t, j);
            // the kernel treats an item as whole exactly when it covers the tile
            const bool whole = kb0 == 0 && kb1 == KB;
            CHECK(whole == (jf == jl), "tile %lld: whole=%d but %d pieces", (long long)t, (int)whole, jl - jf + 1);
            if (whole)
                continue;
            CHECK(t == b / KB || t == (e - 1) / KB, "tile %lld is inside range %d", (long long)t, j);
            // the owner holds k-block 0 and is its range's last tile; no other piece holds k-block 0
            CHECK((kb0 == 0) == (j == jf), "tile %lld piece %d: kb0=%lld but owner %d", (long long)t, j,
                  (long long)kb0, jf);
            if (j == jf)
                CHECK((e - 1) / KB == t, "tile %lld: owner range %d ends in tile %lld", (long long)t, j,
                      (long long)((e - 1) / KB));
            const int32_t s = thin_slot(U, G, KB, j, t);
            CHECK(s >= 0 && s < 2 * G, "slot %d outside [0, %d)", s, 2 * G);
            CHECK(slots.insert(s).second, "slot %d used twice", s);
        }
    }
}

void check_cluster_split(int64_t T, int32_t KB, int32_t C)
{
    const int64_t U = T * KB;
    const int32_t G = (int32_t)(T * C);
    for (int64_t c = 0; c < T; ++c)
        for (int32_t r = 0; r < C; ++r) {
            const int32_t j = (int32_t)(c * C + r);
            const int64_t b = thin_begin(U, G, j), e = thin_begin(U, G, j + 1);
            CHECK(b == c * KB + (int64_t)r * KB / C && e == c * KB + (int64_t)(r + 1) * KB / C,
                  "T=%lld KB=%d C=%d: rank %d of cluster %lld holds [%lld, %lld)", (long long)T, KB, C, r,
                  (long long)c, (long long)b, (long long)e);
            CHECK(e > b, "T=%lld KB=%d C=%d: rank %d of cluster %lld is empty", (long long)T, KB, C, r, (long long)c);
        }
}

// resident[c]: clusters of c CTAs (one CTA per SM) that fit at once on 8 groups
// of 19 SMs, a cluster never spanning two groups
void gb300_model(int32_t (&resident)[kThinMaxCluster + 1])
{
    resident[0] = 0;
    resident[1] = 152;
    for (int c = 2; c <= kThinMaxCluster; ++c)
        resident[c] = 8 * (19 / c);
}

void check_auto_cluster_case(int64_t T, int64_t KB, int32_t want)
{
    int32_t resident[kThinMaxCluster + 1];
    gb300_model(resident);
    const int32_t got = thin_auto_cluster(T, KB, 152, resident);
    CHECK(got == want, "T=%lld KB=%lld: cluster %d, expected %d", (long long)T, (long long)KB, got, want);
}

void check_auto_cluster_sweep()
{
    int32_t resident[kThinMaxCluster + 1];
    gb300_model(resident);
    const int32_t sms = 152;
    for (int64_t T = 1; T <= 300; ++T)
        for (int64_t KB : {1, 2, 3, 5, 8, 16, 33, 64, 128, 160, 161, 256, 320, 512}) {
            const int32_t c = thin_auto_cluster(T, KB, sms, resident);
            if (c == 0)
                continue;
            CHECK(c >= 1 && c <= kThinMaxCluster && c <= KB && T * c <= sms, "T=%lld KB=%lld: cluster %d out of range",
                  (long long)T, (long long)KB, c);
            CHECK(c == 1 || resident[c] >= T, "T=%lld: %d clusters of %d do not fit at once", (long long)T, (int)T, c);
            CHECK(T * c * 10 >= (int64_t)sms * 6, "T=%lld C=%d fills less than 60 %% of the SMs", (long long)T, c);
            CHECK((KB + c - 1) / c <= kThinClusterMaxKBlocks, "T=%lld KB=%lld C=%d: runs too long", (long long)T,
                  (long long)KB, c);
            for (int32_t d = c + 1; d <= kThinMaxCluster && d <= KB && T * d <= sms; ++d)
                CHECK(resident[d] < T, "T=%lld KB=%lld: cluster %d chosen but %d also fits", (long long)T,
                      (long long)KB, c, d);
        }
}

}  // namespace

int main()
{
    long n = 0;
    for (int64_t T = 1; T <= 40; ++T)
        for (int32_t KB : {1, 2, 3, 7, 16, 65, 128})
            for (int32_t C = 1; C <= kThinMaxCluster && C <= KB; ++C) {
                check_cluster_split(T, KB, C);
                ++n;
            }
    // the decode-like shapes of the bench and the tests (tiles of 128 rows, k-blocks of 64)
    check_auto_cluster_case(64, 128, 2);    // 16 x 8192 x 8192
    check_auto_cluster_case(32, 128, 4);    // 16 x 4096 x 8192
    check_auto_cluster_case(32, 32, 4);     // 16 x 4096 x 2048
    check_auto_cluster_case(96, 128, 1);    // 16 x 12288 x 8192: whole tiles
    check_auto_cluster_case(128, 256, 0);   // 16 x 16384 x 16384: 256 k-blocks per CTA
    check_auto_cluster_case(224, 128, 0);   // 16 x 28672 x 8192: more tiles than SMs
    check_auto_cluster_case(8, 8, 0);       // 16 x 1024 x 512: too few CTAs
    check_auto_cluster_case(20, 128, 6);    // 7 per cluster would leave clusters waiting
    check_auto_cluster_case(64, 1, 0);      // one k-block: whole tiles on 64 SMs only
    check_auto_cluster_sweep();
    n += 10;
    for (int64_t T = 1; T <= 24; ++T)
        for (int32_t KB : {1, 2, 3, 7, 16, 65, 128})
            for (int32_t G : {1, 2, 3, 5, 8, 13, 33, 76, 152})
                if ((int64_t)G <= T * KB) {
                    check_split(T, KB, G);
                    ++n;
                }
    for (int64_t T : {32, 64, 256})
        for (int32_t KB : {64, 128, 512})
            for (int32_t G : {148, 152}) {
                check_split(T, KB, G);
                ++n;
            }
    if (failures) {
        std::printf("%d failure(s)\n", failures);
        return 1;
    }
    std::printf("ok %ld splits\n", n);
    return 0;
}
