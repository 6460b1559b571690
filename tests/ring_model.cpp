// CPU model of the GEMM kernel's shared-memory stage ring, run with threads.
//
// The kernel's index arithmetic (warp_specialized_tma_gb300/csrc/ring_index.h)
// drives four threads that stand in for the kernel's agents:
//   producer     waits on a release group's "empty" barrier before the group's
//                first stage, arrives with the stage's byte count on its
//                "full" barrier and hands the copy to the copy engine;
//   copy engine  completes the copies in any order after random delays,
//                writing the stage and completing its bytes on "full";
//   MMA issuer   waits on "full", queues the stage's MMAs and, after a group's
//                last stage, a commit that arrives on the group's "empty";
//   tensor pipe  retires MMAs and commits in issue order after random delays.
// The barrier model keeps the phase count, pending arrivals and transaction
// bytes of an mbarrier; a wait names the parity of the phase it waits for, and
// a fresh barrier's previous phase counts as complete.
//
// Checks: the MMA issuer only reads a stage holding this iteration's data
// (read after write); the copy engine only overwrites a stage whose previous
// lap has been read by the tensor pipe, and no MMA sees its stage change under
// it (write after read).  Every wait is bounded: faults (a dropped copy, a
// dropped commit, an "empty" barrier expecting two arrivals) must end in a
// reported timeout, not a hang, and deliberately broken protocols (the
// producer not waiting, the issuer waiting for the wrong parity) must be
// caught.  Prints one line per scenario; exits 0 when every expectation holds.
#include <atomic>
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <mutex>
#include <random>
#include <string>
#include <thread>
#include <vector>

#include "ring_index.h"

using namespace wstma;
using Clock = std::chrono::steady_clock;

namespace {

constexpr int64_t kStageBytes = 65536;
constexpr auto kLimit = std::chrono::milliseconds(300);

struct Outcome {
    std::atomic<bool> abort{false};
    std::atomic<int> violations{0};
    std::atomic<int> timeouts{0};
    std::mutex m;
    std::string first;

    void note(const char *kind, const char *fmt, ...)
    {
        char buf[256];
        va_list ap;
        va_start(ap, fmt);
        std::vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        std::lock_guard<std::mutex> g(m);
        if (first.empty())
            first = std::string(kind) + ": " + buf;
    }
    void violation(const char *fmt, int a, int b)
    {
        violations++;
        note("violation", fmt, a, b);
        abort = true;
    }
    void timeout(const char *who, int it)
    {
        timeouts++;
        note("timeout", "%s at iteration %d", who, it);
        abort = true;
    }
};

// An mbarrier: `count` arrivals and zero outstanding transaction bytes
// complete the current phase.
struct MBar {
    std::mutex m;
    int count = 1, pending = 1;
    int64_t tx = 0;
    uint64_t phase = 0;  // completed phases

    void init(int c)
    {
        count = pending = c;
        tx = 0;
        phase = 0;
    }
    void complete_if()
    {
        if (pending == 0 && tx == 0) {
            ++phase;
            pending = count;
        }
    }
    void arrive()
    {
        std::lock_guard<std::mutex> g(m);
        --pending;
        complete_if();
    }
    void arrive_expect_tx(int64_t bytes)
    {
        std::lock_guard<std::mutex> g(m);
        tx += bytes;
        --pending;
        complete_if();
    }
    void complete_tx(int64_t bytes)
    {
        std::lock_guard<std::mutex> g(m);
        tx -= bytes;
        complete_if();
    }
    bool try_wait(uint32_t parity)
    {
        std::lock_guard<std::mutex> g(m);
        return (phase & 1u) != parity;
    }
};

bool wait(MBar &b, uint32_t parity, Outcome &out, const char *who, int it)
{
    const auto t0 = Clock::now();
    while (!b.try_wait(parity)) {
        if (out.abort)
            return false;
        if (Clock::now() - t0 > kLimit) {
            out.timeout(who, it);
            return false;
        }
        std::this_thread::yield();
    }
    return true;
}

void jitter(std::mt19937 &rng)
{
    const unsigned r = rng() % 64;
    if (r < 8)
        std::this_thread::yield();
    for (volatile unsigned i = 0; i < r * 20; ++i) {
    }
}

struct Scenario {
    const char *name;
    int S, g_shift, iters;
    int drop_load = -1;       // iteration whose copy never happens
    int drop_commit = -1;     // iteration whose group commit is never issued
    int empty_count = 1;      // arrivals an "empty" barrier expects per phase
    bool producer_waits = true;
    bool issuer_parity_flipped = false;
    enum Expect { kClean, kTimeout, kCaught } expect;
};

struct Job {
    int kind;  // 0 = MMA of (stage, iteration), 1 = commit to group
    int a, b;
};

bool run(const Scenario &sc, unsigned seed)
{
    const int S = sc.S;
    const uint32_t g_shift = (uint32_t)sc.g_shift;
    const uint32_t g_mask = (1u << g_shift) - 1u;
    std::vector<MBar> full(S), empty(S);
    for (auto &b : full)
        b.init(1);
    for (auto &b : empty)
        b.init(sc.empty_count);
    std::vector<std::atomic<int>> data(S), consumed(S);
    for (int s = 0; s < S; ++s) {
        data[s] = -1;
        consumed[s] = s - S;  // "lap -1" has been read
    }
    Outcome out;
    std::mutex qm;
    std::vector<std::pair<int, int>> copies;  // (stage, iteration), completed in any order
    std::deque<Job> pipe;                     // retired in order
    std::atomic<bool> producer_done{false}, issuer_done{false};

    std::thread producer([&] {
        int s = 0;
        uint32_t ph = 0;
        for (int it = 0; it < sc.iters && !out.abort; ++it) {
            if (sc.producer_waits && ring_group_first(s, g_mask) &&
                !wait(empty[ring_group(s, g_shift)], ring_empty_parity(ph), out, "producer", it))
                break;
            full[s].arrive_expect_tx(kStageBytes);
            if (it != sc.drop_load) {
                std::lock_guard<std::mutex> g(qm);
                copies.push_back({s, it});
            }
            ring_advance(s, ph, S);
        }
        producer_done = true;
    });
    std::thread copier([&] {
        std::mt19937 rng(seed * 7 + 1);
        for (;;) {
            std::pair<int, int> c;
            {
                std::lock_guard<std::mutex> g(qm);
                if (copies.empty()) {
                    if (producer_done || out.abort)
                        break;
                    continue;
                }
                const size_t k = rng() % copies.size();
                c = copies[k];
                copies.erase(copies.begin() + (long)k);
            }
            jitter(rng);
            const int s = c.first, it = c.second;
            if (consumed[s] != it - S)
                out.violation("copy of iteration %d overwrote stage %d before its previous lap was read", it, s);
            data[s] = it;
            full[s].complete_tx(kStageBytes);
        }
    });
    std::thread issuer([&] {
        int s = 0;
        uint32_t ph = 0;
        const uint32_t flip = sc.issuer_parity_flipped ? 1u : 0u;
        for (int it = 0; it < sc.iters && !out.abort; ++it) {
            if (!wait(full[s], ring_full_parity(ph) ^ flip, out, "MMA issuer", it))
                break;
            if (data[s] != it)
                out.violation("MMA of iteration %d read stage %d before its data landed", it, s);
            {
                std::lock_guard<std::mutex> g(qm);
                pipe.push_back({0, s, it});
                if (ring_group_last(s, g_mask) && it != sc.drop_commit)
                    pipe.push_back({1, (int)ring_group(s, g_shift), it});
            }
            ring_advance(s, ph, S);
        }
        issuer_done = true;
    });
    std::thread tensor([&] {
        std::mt19937 rng(seed * 13 + 5);
        for (;;) {
            Job j;
            {
                std::lock_guard<std::mutex> g(qm);
                if (pipe.empty()) {
                    if (issuer_done || out.abort)
                        break;
                    continue;
                }
                j = pipe.front();
                pipe.pop_front();
            }
            if (j.kind == 0) {
                jitter(rng);
                if (data[j.a] != j.b)
                    out.violation("stage %d changed while MMA of iteration %d read it", j.a, j.b);
                consumed[j.a] = j.b;
            } else {
                empty[j.a].arrive();
            }
        }
    });
    producer.join();
    copier.join();
    issuer.join();
    tensor.join();

    bool ok;
    switch (sc.expect) {
    case Scenario::kClean: ok = out.violations == 0 && out.timeouts == 0; break;
    case Scenario::kTimeout: ok = out.violations == 0 && out.timeouts > 0; break;
    default: ok = out.violations > 0 || out.timeouts > 0; break;
    }
    std::printf("%-44s S=%d G=%d seed=%u: %s (%d violations, %d timeouts)%s%s\n", sc.name, S, 1 << sc.g_shift, seed,
                ok ? "as expected" : "UNEXPECTED", out.violations.load(), out.timeouts.load(),
                out.first.empty() ? "" : "; first ", out.first.c_str());
    return ok;
}

}  // namespace

int main()
{
    std::vector<Scenario> scs;
    for (int S : {1, 2, 3, 4, 6, 8})
        scs.push_back({"ring, one stage per release", S, 0, 600, -1, -1, 1, true, false, Scenario::kClean});
    for (int S : {2, 4, 6, 8})
        scs.push_back({"ring, stage pairs released together", S, 1, 600, -1, -1, 1, true, false, Scenario::kClean});
    scs.push_back({"fault: a copy never lands", 6, 0, 600, 137, -1, 1, true, false, Scenario::kTimeout});
    scs.push_back({"fault: a commit never issued", 6, 0, 600, -1, 203, 1, true, false, Scenario::kTimeout});
    scs.push_back({"fault: paired commit never issued", 6, 1, 600, -1, 203, 1, true, false, Scenario::kTimeout});
    scs.push_back({"fault: empty barrier expects two arrivals", 4, 0, 600, -1, -1, 2, true, false,
                   Scenario::kTimeout});
    scs.push_back({"broken: producer never waits for release", 3, 0, 600, -1, -1, 1, false, false,
                   Scenario::kCaught});
    scs.push_back({"broken: issuer waits for the wrong parity", 4, 0, 600, -1, -1, 1, true, true,
                   Scenario::kCaught});
    int bad = 0;
    for (const Scenario &sc : scs) {
        const int seeds = sc.expect == Scenario::kClean ? 3 : 1;
        for (int k = 0; k < seeds; ++k)
            bad += run(sc, 11u + 97u * (unsigned)k) ? 0 : 1;
    }
    if (bad) {
        std::printf("%d unexpected outcome(s)\n", bad);
        return 1;
    }
    std::printf("ok\n");
    return 0;
}
