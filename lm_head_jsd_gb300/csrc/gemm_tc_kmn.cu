// Instantiations of the tensor-core GEMM kernel for K-major A and MN-major B (grad_input: dZ . W).
#include "gemm_tc_kernel.cuh"

namespace fljsd {
namespace tcgemm {

FLJSD_TC_LAUNCHER(launch_kmn) {
  if (mc)
    return p.epi_groups == 2 ? launch_g<false, true, true, 2>(ma, mb, mcm, msm, d, p, st)
                             : launch_g<false, true, true, 1>(ma, mb, mcm, msm, d, p, st);
  return p.epi_groups == 2 ? launch_g<false, true, false, 2>(ma, mb, mcm, msm, d, p, st)
                           : launch_g<false, true, false, 1>(ma, mb, mcm, msm, d, p, st);
}

}  // namespace tcgemm
}  // namespace fljsd
