// gemm_bf16_run_noalloc: the GEMM for callers that must not allocate.
//
// Some callers cannot call cudaMalloc at the point where they multiply:
// runtimes that own every byte of device memory through their own pool and
// forbid raw allocations, and latency-critical loops where an allocation's
// implicit synchronisation is not acceptable.  gemm_bf16_create() allocates (a
// host handle and a device status word), so those callers use this entry
// point instead: it takes the problem, the operands and the stream, keeps no
// handle, and finds its scratch -- the kernel watchdog's status word -- in a
// file-scope device array that every GPU loading this library holds until the
// process exits.
//
// It runs the same kernel as gemm_bf16_run with the default plan (SM-pair
// 256x256 tiles, deepest ring, persistent grid, 1 s watchdog) except that every
// tile runs whole (splitting tiles along k, stream-K, needs a partials
// workspace of several MiB), operands are read in place (repacking needs a
// copy) and the launch carries no programmatic-dependent-launch attribute.  It
// calls no cudaMalloc, cudaFree or allocating library routine.
#include "gemm_bf16.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gemm_kernels.h"

using namespace wstma;

namespace {

// Scratch words this entry point needs per call (the status word), and the
// array's fixed capacity: 64 words = 256 bytes per device.
constexpr int kScratchWordsNeeded = 1;
constexpr int kScratchWordsMax = 64;
static_assert(kScratchWordsNeeded <= kScratchWordsMax, "a call's scratch must fit the fixed array");
constexpr int kMaxDevices = 64;
constexpr uint64_t kWatchdogNs = 1000000000ull;
constexpr uint64_t kWatchdogNsPerKBlock = 2000;  // no wait outlasts one tile's k-range of MMAs

static __device__ __align__(256) uint32_t g_noalloc_scratch[kScratchWordsMax];

struct DeviceSetup {
    bool ready = false;
    uint32_t *scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
    int clusters = 0;             // resident SM pairs for the persistent grid
    int stages = 0;
    size_t smem = 0;
};

std::mutex g_mu;
DeviceSetup g_setup[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint64_t row_bytes, uint32_t box_cols,
            uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Once per device, with that device current: the scratch array's device
// address (the array's name is only a host-side stand-in in host code), the
// kernel's shared-memory limit and the persistent grid size.
int setup_device(int dev, DeviceSetup **out)
{
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceSetup &d = g_setup[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0, optin = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_BF16_ERR_CUDA;
        }
        if (major != 10 || minor != 3)
            return GEMM_BF16_ERR_UNSUPPORTED;
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return GEMM_BF16_ERR_CUDA;
        }
        int stages = 0;
        for (int s = kMaxStages; s >= 2; --s)
            if (ws_smem_bytes(2, s) <= (size_t)optin) {
                stages = s;
                break;
            }
        if (stages < 2)
            return GEMM_BF16_ERR_UNSUPPORTED;
        const void *fn = ws_kernel_c2(false);
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_BF16_ERR_CUDA;
        }
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)(2 * std::max(1, sms / 2)), 1, 1);
        cfg.blockDim = dim3(kWsThreads, 1, 1);
        cfg.dynamicSmemBytes = ws_smem_bytes(2, stages);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            clusters = std::max(1, sms / 2);
        }
        d.scratch = static_cast<uint32_t *>(ptr);
        d.num_sms = sms;
        d.clusters = clusters;
        d.stages = stages;
        d.smem = ws_smem_bytes(2, stages);
        d.ready = true;
    }
    *out = &d;
    return GEMM_BF16_OK;
}

}  // namespace

extern "C" GEMM_BF16_API int gemm_bf16_run_noalloc(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                                   int64_t ldd, const void *A, const void *B, void *D,
                                                   void *stream, uint32_t *status)
{
    if (!A || !B || !D)
        return GEMM_BF16_ERR_INVALID_ARG;
    int rc = gemm_bf16_check_problem(M, N, K, lda, ldb, ldd);
    if (rc != GEMM_BF16_OK)
        return rc;
    if ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u) ||
        (reinterpret_cast<uintptr_t>(D) & 1u))
        return GEMM_BF16_ERR_ALIGNMENT;
    // A pageable `status` would make the status copy block this thread until
    // the GEMM is done (and cannot be captured): only page-locked host memory
    // or device memory is taken.
    if (status) {
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, status) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_BF16_ERR_INVALID_ARG;
        }
        if (pa.type != cudaMemoryTypeHost && pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeManaged)
            return GEMM_BF16_ERR_INVALID_ARG;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    DeviceSetup *ds = nullptr;
    if ((rc = setup_device(dev, &ds)) != GEMM_BF16_OK)
        return rc;

    const int num_m_blocks = (int)((M + 2 * kBlockM - 1) / (2 * kBlockM));
    const int num_n_blocks = (int)((N + kBlockN - 1) / kBlockN);
    const int64_t tiles = (int64_t)num_m_blocks * num_n_blocks;
    if (tiles > 0x3FFFFFFFLL)
        return GEMM_BF16_ERR_INVALID_ARG;
    const bool epi_tma = ((ldd * 2) % 16) == 0 && (reinterpret_cast<uintptr_t>(D) & 15u) == 0;

    CUtensorMap tmA, tmB, tmD;
    std::memset(&tmD, 0, sizeof tmD);
    if (!encode(&tmA, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda * 2, kBlockK, kBlockM) ||
        !encode(&tmB, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb * 2, kBlockK, kBlockN / 2) ||
        (epi_tma && !encode(&tmD, D, (uint64_t)N, (uint64_t)M, (uint64_t)ldd * 2, 64, 32)))
        return GEMM_BF16_ERR_TENSORMAP;

    GemmParams prm;
    prm.M = (int32_t)M;
    prm.N = (int32_t)N;
    prm.K = (int32_t)K;
    prm.num_m_blocks = num_m_blocks;
    prm.num_n_blocks = num_n_blocks;
    prm.num_k_blocks = (int32_t)((K + kBlockK - 1) / kBlockK);
    prm.num_tiles = (int32_t)tiles;
    prm.raster_group = 8;
    prm.stages = ds->stages;
    prm.acc_buffers = 2;
    prm.stage_group = 1;
    prm.epi_tma = epi_tma ? 1 : 0;
    prm.fault_skip_it = -1;
    prm.ldd = ldd;
    prm.D = D;
    prm.err = ds->scratch;  // word 0 of the shared scratch array
    prm.watchdog_ns = kWatchdogNs > (uint64_t)prm.num_k_blocks * kWatchdogNsPerKBlock
                          ? kWatchdogNs
                          : (uint64_t)prm.num_k_blocks * kWatchdogNsPerKBlock;
    prm.sk_tiles = 0;  // stream-K needs a partials workspace, which this entry point does not have
    prm.epoch = 1;
    prm.sk_units = 0;
    prm.sk_head = 0;
    prm.sk_pieces = 0;
    prm.workspace = nullptr;
    prm.flags = nullptr;
    prm.C = nullptr;
    prm.bias = nullptr;
    prm.ldc = 0;
    prm.alpha = 1.f;
    prm.beta = 0.f;
    prm.fused = 0;
    prm.epi_pingpong = 0;
    prm.sched_dynamic = 0;  // the counter lives in a handle
    prm.sched = nullptr;
    prm.k_order = 1;  // alternating k direction per whole tile, as in the default plan
    prm.serpentine = 1;  // as in the default plan

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the status word must start at zero for this call (the array keeps the
    // previous call's contents)
    if (cudaMemsetAsync(ds->scratch, 0, kScratchWordsNeeded * sizeof(uint32_t), st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(2 * std::min<int64_t>(tiles, ds->clusters)), 1, 1);
    cfg.blockDim = dim3(kWsThreads, 1, 1);
    cfg.dynamicSmemBytes = ds->smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[4] = {&tmA, &tmB, &tmD, &prm};
    if (cudaLaunchKernelExC(&cfg, ws_kernel_c2(false), args) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    if (status &&
        cudaMemcpyAsync(status, ds->scratch, sizeof(uint32_t), cudaMemcpyDefault, st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_BF16_ERR_CUDA;
    }
    return GEMM_BF16_OK;
}
