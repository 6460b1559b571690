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
// other pieces are not.
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

}  // namespace

int main()
{
    long n = 0;
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
