// Instantiations of the tensor-core GEMM kernel for MN-major A and B (grad_weight: dZ^T . X).
#include "gemm_tc_kernel.cuh"

namespace fljsd {
namespace tcgemm {

FLJSD_TC_LAUNCHER(launch_mnmn) {
  if (mc)
    return p.epi_groups == 2 ? launch_g<true, true, true, 2>(ma, mb, mcm, msm, d, p, st)
                             : launch_g<true, true, true, 1>(ma, mb, mcm, msm, d, p, st);
  return p.epi_groups == 2 ? launch_g<true, true, false, 2>(ma, mb, mcm, msm, d, p, st)
                           : launch_g<true, true, false, 1>(ma, mb, mcm, msm, d, p, st);
}

}  // namespace tcgemm
}  // namespace fljsd
