// Non-specialised ablation kernels (__syncthreads WAR and mbarrier WAR).
#include "gemm_nows.cuh"

namespace wstma {

const void *nows_kernel(bool mbar_war)
{
    return mbar_war ? reinterpret_cast<const void *>(&gemm_nows_kernel<true>)
                    : reinterpret_cast<const void *>(&gemm_nows_kernel<false>);
}

}  // namespace wstma
