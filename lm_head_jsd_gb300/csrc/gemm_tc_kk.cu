// Instantiations of the tensor-core GEMM kernel for K-major A and B (the logits: X . W^T).
#include "gemm_tc_kernel.cuh"

namespace fljsd {
namespace tcgemm {

FLJSD_TC_LAUNCHER(launch_kk) {
  return pair ? launch_modes<false, false, true>(ma, mb, mcm, msm, d, p, st)
              : launch_modes<false, false, false>(ma, mb, mcm, msm, d, p, st);
}

}  // namespace tcgemm
}  // namespace fljsd
