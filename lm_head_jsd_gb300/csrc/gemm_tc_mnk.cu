// Instantiations of the tensor-core GEMM kernel for MN-major A and K-major B (the remaining layout of the GEMM entry point).
#include "gemm_tc_kernel.cuh"

namespace fljsd {
namespace tcgemm {

FLJSD_TC_LAUNCHER(launch_mnk) {
  return pair ? launch_modes<true, false, true>(ma, mb, mcm, msm, d, p, st)
              : launch_modes<true, false, false>(ma, mb, mcm, msm, d, p, st);
}

}  // namespace tcgemm
}  // namespace fljsd
