// Instantiations of the tensor-core GEMM kernel for K-major A and B (the logits: X . W^T).
#include "gemm_tc_kernel.cuh"

namespace fljsd {
namespace tcgemm {

FLJSD_TC_LAUNCHER(launch_kk) {
  if (mc)
    return p.epi_groups == 2 ? launch_g<false, false, true, 2>(ma, mb, mcm, msm, d, p, st)
                             : launch_g<false, false, true, 1>(ma, mb, mcm, msm, d, p, st);
  return p.epi_groups == 2 ? launch_g<false, false, false, 2>(ma, mb, mcm, msm, d, p, st)
                           : launch_g<false, false, false, 1>(ma, mb, mcm, msm, d, p, st);
}

}  // namespace tcgemm
}  // namespace fljsd
