// Thin kernel (gemm_thin.cuh): one variant per small-operand width.
#include "gemm_thin.cuh"

namespace wstma {

const void *thin_kernel(int nt)
{
    switch (nt) {
    case 16: return reinterpret_cast<const void *>(&gemm_thin_kernel<16>);
    case 32: return reinterpret_cast<const void *>(&gemm_thin_kernel<32>);
    case 48: return reinterpret_cast<const void *>(&gemm_thin_kernel<48>);
    case 64: return reinterpret_cast<const void *>(&gemm_thin_kernel<64>);
    default: return nullptr;
    }
}

}  // namespace wstma
