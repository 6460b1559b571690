// Warp-specialised kernel, one CTA per 128x256 output tile (cta_group::1).
#include "gemm_ws.cuh"

namespace wstma {

const void *ws_kernel_c1(bool setmaxnreg)
{
    return setmaxnreg ? reinterpret_cast<const void *>(&gemm_ws_kernel<1, true>)
                      : reinterpret_cast<const void *>(&gemm_ws_kernel<1, false>);
}

}  // namespace wstma
