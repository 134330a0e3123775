// Tensor-core GEMM interface (internal). See gemm_tc.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fljsd {

// D[m x n] (+)= A . B^T, bf16 operands and output, fp32 accumulation.
//   a_mn == 0: A is stored [m x k] row-major (k contiguous), row stride lda
//   a_mn == 1: A is stored [k x m] row-major (m contiguous), row stride lda
//   b_mn == 0: B is stored [n x k] row-major, row stride ldb
//   b_mn == 1: B is stored [k x n] row-major, row stride ldb
//   D is stored [m x ldd] row-major.
// Requirements: 16-byte aligned pointers, lda / ldb / ldd multiples of 8.
struct TcGemmArgs {
  const void* a; int64_t lda; int a_mn;
  const void* b; int64_t ldb; int b_mn;
  void* d; int64_t ldd;
  int64_t m, n, k;
  int accumulate;        // 1: D = D + A.B^T (fp32 add, one rounding)
  // tile order: 0 = bands of m-blocks sweeping all n-blocks (the band of A
  // stays in L2 while B streams); 1 = n-blocks fastest
  int raster_n_fastest;
  int* status;           // device word that receives FLJSD_ERR_TIMEOUT, or null
  // Optional row statistics of the stored output (requires accumulate == 0):
  // for row r and column block j (TC_STATS_COLS columns),
  // stats[r * ceil(n / TC_STATS_COLS) + j]
  // = (m, sum 2^(x - m)) over x = bf16(D[r, col]) * stats_scale, where m is the
  // largest rounded product and each x - m is formed from the exact product.
  float2* stats;
  float stats_scale;
  // Optional fp32 accumulator [m x ldd] (16-byte aligned). With d32 set the
  // product goes to d32 (added to it when accumulate == 1) and D is not
  // touched, unless finalize == 1: then D = round(d32 + product).
  float* d32;
  int finalize;
  // Test of the bounded waits: with stall_producer no copy is issued, so the
  // MMA's first wait expires after timeout_ns (0 = the 10 s default) and the
  // kernel reports FLJSD_ERR_TIMEOUT in *status and exits cleanly.
  unsigned long long timeout_ns;
  int stall_producer;
  // Optional fp32 scratch for split-K (used when the output has too few tiles
  // to fill the GPU, accumulate == 0 and no d32 / stats): up to
  // tc_splitk_bytes(m, n, k, ...) bytes, 16-byte aligned.
  float* splitk_ws;
  size_t splitk_ws_bytes;
  // 1: one CTA per 128 x 256 tile even where a CTA pair could take a
  // 256 x 256 tile (the results are identical either way)
  int single_cta = 0;
};

constexpr int TC_STATS_COLS = 128;  // columns per pass-1 partial
// CTAs a plan assumes when it sizes the split-K scratch (the launch uses the
// device's own count, capped by the scratch it is given).
constexpr int TC_PLAN_CTAS = 152;
// Scratch bytes the split-K schedule of this contraction would use.
size_t tc_splitk_bytes(int64_t m, int64_t n, int64_t k, int ctas);

bool tc_gemm_supported(const TcGemmArgs& g);
cudaError_t launch_gemm_tc(const TcGemmArgs& g, cudaStream_t st);

}  // namespace fljsd
