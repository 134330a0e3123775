// Instantiations of the tensor-core GEMM kernel for MN-major A and B (grad_weight: dZ^T . X).
#include "gemm_tc_kernel.cuh"

namespace fljsd {
namespace tcgemm {

FLJSD_TC_LAUNCHER(launch_mnmn) {
  return pair ? launch_modes<true, true, true>(ma, mb, mcm, msm, d, p, st)
              : launch_modes<true, true, false>(ma, mb, mcm, msm, d, p, st);
}

}  // namespace tcgemm
}  // namespace fljsd
