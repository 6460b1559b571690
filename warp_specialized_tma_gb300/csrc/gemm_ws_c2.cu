// Warp-specialised kernel, an SM pair (2-CTA cluster) per 256x256 output tile
// (cta_group::2).
#include "gemm_ws.cuh"

namespace wstma {

const void *ws_kernel_c2(bool setmaxnreg)
{
    return setmaxnreg ? reinterpret_cast<const void *>(&gemm_ws_kernel<2, true>)
                      : reinterpret_cast<const void *>(&gemm_ws_kernel<2, false>);
}

}  // namespace wstma
