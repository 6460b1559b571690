// Operand repacking: a copy of a K-major bf16 operand into rows whose pitch is
// a multiple of 128 bytes.
//
// The GEMM's TMA loads read a 64-element (128-byte) box row per operand row
// and k-block.  When the row pitch is a multiple of 128 bytes every box row is
// one whole 128-byte L2 line; with any other pitch (e.g. 4104 bf16 = 8208 bytes)
// each box row straddles two lines, the loads touch a fifth more sectors, and
// the GEMM runs ~28% slower (measured on GB300).  When the other dimension of
// the problem is large the GEMM's saving exceeds the cost of this copy, so the
// plan can route an operand through a packed copy first.
//
// The copy is HBM-bound: one read and one write of the operand.  Both operands
// go in one launch (blockIdx.y = operand).  Each CTA owns a block of rows and
// sweeps it as one flat range of 16-byte vectors -- both pitches are multiples
// of 16 bytes, the condition the GEMM already places on lda and ldb -- with
// several loads in flight per thread; a row length that is not a multiple of
// 8 elements leaves a 2-byte tail per row.  Source reads are marked streaming
// (read once, evict first); the packed rows are stored normally so that the
// GEMM launched next finds much of them in L2.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_kernels.h"

namespace wstma {

namespace {

constexpr int kRepackThreads = 256;
constexpr int kRepackUnroll = 4;

struct JobArgs {
    const uint16_t *src;
    uint16_t *dst;
    int64_t ld_src, ld_dst, rows, cols;
    int32_t rows_per_cta;
};

__global__ void __launch_bounds__(kRepackThreads) repack_rows_kernel(const JobArgs j0, const JobArgs j1)
{
    const JobArgs &j = blockIdx.y == 0 ? j0 : j1;
    const int64_t r0 = (int64_t)blockIdx.x * j.rows_per_cta;
    if (r0 >= j.rows)
        return;
    const int64_t nrows64 = j.rows - r0 < j.rows_per_cta ? j.rows - r0 : j.rows_per_cta;
    const int32_t nrows = (int32_t)nrows64;
    const int32_t nvec = (int32_t)(j.cols >> 3);  // whole 16-byte vectors per row
    const int32_t total = nrows * nvec;           // < 2^31 by the choice of rows_per_cta
    const uint16_t *src = j.src + r0 * j.ld_src;
    uint16_t *dst = j.dst + r0 * j.ld_dst;
    for (int32_t f = threadIdx.x; f < total; f += kRepackThreads * kRepackUnroll) {
        uint4 x[kRepackUnroll];
        int32_t r[kRepackUnroll], v[kRepackUnroll];
#pragma unroll
        for (int u = 0; u < kRepackUnroll; ++u) {
            const int32_t g = f + kRepackThreads * u;
            r[u] = g / nvec;
            v[u] = g - r[u] * nvec;
            if (g < total)
                x[u] = __ldcs(reinterpret_cast<const uint4 *>(src + (int64_t)r[u] * j.ld_src) + v[u]);
        }
#pragma unroll
        for (int u = 0; u < kRepackUnroll; ++u)
            if (f + kRepackThreads * u < total)
                reinterpret_cast<uint4 *>(dst + (int64_t)r[u] * j.ld_dst)[v[u]] = x[u];
    }
    const int32_t tail = (int32_t)(j.cols & 7);
    if (tail) {
        for (int32_t f = threadIdx.x; f < nrows * tail; f += kRepackThreads) {
            const int32_t rr = f / tail;
            const int64_t c = (int64_t)nvec * 8 + (f - rr * tail);
            dst[(int64_t)rr * j.ld_dst + c] = src[(int64_t)rr * j.ld_src + c];
        }
    }
    // This CTA's rows are copied: the GEMM launched next on the stream (with
    // programmatic dependent launch) may start its prologue once every CTA of
    // this grid got here; its loads still wait for this grid's memory.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

JobArgs make_job(const RepackJob &in, int num_sms, int njobs)
{
    JobArgs a;
    a.src = static_cast<const uint16_t *>(in.src);
    a.dst = static_cast<uint16_t *>(in.dst);
    a.ld_src = in.ld_src;
    a.ld_dst = in.ld_dst;
    a.rows = in.rows;
    a.cols = in.cols;
    // about 8 CTAs per SM over all jobs; a CTA's flat range stays below 2^30 vectors
    const int64_t target = (int64_t)(num_sms > 0 ? num_sms : 1) * 8 / njobs;
    int64_t rpc = (in.rows + target - 1) / target;
    const int64_t nvec = in.cols >> 3;
    const int64_t cap = nvec > 0 ? ((int64_t)1 << 30) / nvec : rpc;
    if (rpc > cap)
        rpc = cap;
    if (rpc < 1)
        rpc = 1;
    a.rows_per_cta = (int32_t)rpc;
    return a;
}

}  // namespace

int launch_repack(const RepackJob *jobs, int njobs, int num_sms, cudaStream_t stream)
{
    if (njobs <= 0)
        return 0;
    if (njobs > 2)
        return (int)cudaErrorInvalidValue;
    const JobArgs a = make_job(jobs[0], num_sms, njobs);
    const JobArgs b = njobs == 2 ? make_job(jobs[1], num_sms, njobs) : a;
    const int64_t ga = (a.rows + a.rows_per_cta - 1) / a.rows_per_cta;
    const int64_t gb = (b.rows + b.rows_per_cta - 1) / b.rows_per_cta;
    const int64_t gx = ga > gb ? ga : gb;
    if (gx > 0x7FFFFFFF)
        return (int)cudaErrorInvalidValue;
    repack_rows_kernel<<<dim3((unsigned)gx, (unsigned)njobs, 1), kRepackThreads, 0, stream>>>(a, b);
    return (int)cudaGetLastError();
}

}  // namespace wstma
