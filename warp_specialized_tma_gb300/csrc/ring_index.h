// Index arithmetic of the shared-memory stage ring, shared by the GEMM kernel
// and by the CPU model of the ring's protocol (tests/ring_model.cpp).  Plain
// C++: no CUDA types, so a host compiler can build the model from it.
//
// Ring iteration i uses stage s = i % S in lap i / S.  Each stage has a "full"
// barrier (its data landed: RAW) and each release group of G = 2^g_shift
// stages an "empty" barrier (the MMAs that read the group retired: WAR).  An
// mbarrier wait names the parity of the phase it waits for; a freshly
// initialised barrier counts the phase before its first as complete.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define WSTMA_RING_FN __host__ __device__ __forceinline__
#else
#define WSTMA_RING_FN inline
#endif

namespace wstma {

// Next stage; the lap parity flips when the ring wraps.
WSTMA_RING_FN void ring_advance(int &s, uint32_t &ph, int S)
{
    if (++s == S) {
        s = 0;
        ph ^= 1u;
    }
}

// The producer of lap parity ph waits for the release of the previous lap (on
// the first lap: the phase before the barrier's first, already complete).
WSTMA_RING_FN uint32_t ring_empty_parity(uint32_t ph) { return ph ^ 1u; }

// The consumer of lap parity ph waits for this lap's data.
WSTMA_RING_FN uint32_t ring_full_parity(uint32_t ph) { return ph; }

// Release groups: the producer waits on a group's "empty" barrier before the
// group's first stage; the consumer commits to it after the group's last.
WSTMA_RING_FN bool ring_group_first(int s, uint32_t g_mask) { return ((uint32_t)s & g_mask) == 0u; }
WSTMA_RING_FN bool ring_group_last(int s, uint32_t g_mask) { return ((uint32_t)s & g_mask) == g_mask; }
WSTMA_RING_FN uint32_t ring_group(int s, uint32_t g_shift) { return (uint32_t)s >> g_shift; }

// Stage and full-barrier parity of ring iteration i.
WSTMA_RING_FN int ring_stage_of(int32_t i, int S) { return i % S; }
WSTMA_RING_FN uint32_t ring_parity_of(int32_t i, int S) { return (uint32_t)((i / S) & 1); }

}  // namespace wstma
