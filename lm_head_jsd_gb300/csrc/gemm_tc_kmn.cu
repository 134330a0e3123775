// Instantiations of the tensor-core GEMM kernel for K-major A and MN-major B (grad_input: dZ . W).
#include "gemm_tc_kernel.cuh"

namespace fljsd {
namespace tcgemm {

FLJSD_TC_LAUNCHER(launch_kmn) {
  return pair ? launch_modes<false, true, true>(ma, mb, mcm, msm, d, p, st)
              : launch_modes<false, true, false>(ma, mb, mcm, msm, d, p, st);
}

}  // namespace tcgemm
}  // namespace fljsd
