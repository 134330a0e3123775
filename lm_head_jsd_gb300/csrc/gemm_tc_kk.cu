// Instantiations of the tensor-core GEMM kernel for K-major A and B (the logits: X . W^T).
#include "gemm_tc_kernel.cuh"

namespace fljsd {
namespace tcgemm {

FLJSD_TC_LAUNCHER(launch_kk) {
  return launch_modes<false, false>(ma, mb, mcm, msm, d, p, st);
}

}  // namespace tcgemm
}  // namespace fljsd
