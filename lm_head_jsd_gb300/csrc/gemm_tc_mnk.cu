// Instantiations of the tensor-core GEMM kernel for MN-major A and K-major B (the remaining layout of the GEMM entry point).
#include "gemm_tc_kernel.cuh"

namespace fljsd {
namespace tcgemm {

FLJSD_TC_LAUNCHER(launch_mnk) {
  if (mc)
    return p.epi_groups == 2 ? launch_g<true, false, true, 2>(ma, mb, mcm, msm, d, p, st)
                             : launch_g<true, false, true, 1>(ma, mb, mcm, msm, d, p, st);
  return p.epi_groups == 2 ? launch_g<true, false, false, 2>(ma, mb, mcm, msm, d, p, st)
                           : launch_g<true, false, false, 1>(ma, mb, mcm, msm, d, p, st);
}

}  // namespace tcgemm
}  // namespace fljsd
