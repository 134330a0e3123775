// Internal declarations shared by the translation units of libfljsd.so.
// Nothing here is part of the C ABI (that is include/fljsd.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "fljsd.h"

namespace fljsd {

// ---------------------------------------------------------------------------
// launch accounting / tracing (fljsd_api.cu)
// ---------------------------------------------------------------------------
void trace_begin(int kind, cudaStream_t st);
void trace_end(int kind, cudaStream_t st);
// counts a kernel launched inside a traced call beyond the call's first
void count_extra_launch();

// Number of SMs of the current device (cached per device).
int num_sms();

// ---------------------------------------------------------------------------
// row kernels (rows.cu)
// ---------------------------------------------------------------------------
struct JsdRowArgs {
  void* zs;              // [rows x ld] student logits in, dlogits out (dtype)
  const void* zt;        // [rows x ld] teacher logits (dtype)
  int64_t ld;            // row stride in elements (multiple of 8)
  int64_t v;             // vocabulary size
  int64_t rows;          // rows of this chunk
  int64_t row0;          // global index of the first row of this chunk
  const int64_t* labels; // [bt] or null
  int64_t ignore_index;
  const float* row_grad; // [bt] or null (reduction NONE only)
  const int* n_valid;    // device scalar
  float* loss_rows;      // [bt], indexed by global row
  // Pass-1 partials from the logits GEMM epilogue, or null (then pass 1 runs
  // here): [rows x ntiles] (max, sum 2^(x - max)) of x = z * log2(e) / T.
  const float2* stats_s;
  const float2* stats_t;
  int64_t ntiles;
  int reduction;
  float beta;
  float inv_temperature;
  float scale_log2;  // log2(e) / T, the same constant the GEMM epilogue used
  float loss_scale;  // 1, or T^2 with FLJSD_FLAG_T2 (loss and gradients)
  int64_t cache_vec; // set by the launcher: vectors of X - log M kept in shared memory
  int rows_prefetch; // set by the launcher: L2 prefetch ahead of pass 2 (lean path)
};

cudaError_t launch_count_valid(const int64_t* labels, int64_t bt, int64_t ignore_index,
                               int* n_valid, cudaStream_t st);
cudaError_t launch_jsd_rows(int dtype, const JsdRowArgs& a, cudaStream_t st);

cudaError_t launch_reduce_loss(const float* loss_rows, int64_t bt, int64_t v, int reduction,
                               const int* n_valid, float* loss, cudaStream_t st);
cudaError_t launch_scale(int dtype, void* p, int64_t n, const float* g, cudaStream_t st);

// Distances over given distributions (dist_rows.cu): log-space JSD and TVD.
struct DistArgs {
  const void* x;          // log-space JSD: input log Q; TVD: p   [rows x v]
  const void* y;          // log-space JSD: target log P; TVD: q  [rows x v]
  void* grad;             // d loss / d x, same dtype            [rows x v]
  int64_t rows, v;
  const int64_t* labels;  // [rows] or null
  int64_t ignore_index;
  const int* n_valid;
  float* loss_rows;       // [rows]
  float* loss_elem;       // TVD with reduction none: [rows x v] fp32, else null
  int reduction;
  float beta;
};
cudaError_t launch_jsd_logspace(int dtype, const DistArgs& a, cudaStream_t st);
cudaError_t launch_tvd(int dtype, const DistArgs& a, cudaStream_t st);

// ---------------------------------------------------------------------------
// GEMMs. C[m, n] (+)= sum_k A(m, k) * B(n, k), fp32 accumulation, one rounding
// to the output dtype. A(m, k) = A[m * sam + k * sak], B(n, k) = B[n * sbn + k * sbk].
// ---------------------------------------------------------------------------
struct GemmArgs {
  const void* a; int64_t sam, sak;
  const void* b; int64_t sbn, sbk;
  void* c; int64_t ldc;
  int64_t m, n, k;
  int accumulate;  // 0: C = A.B^T ; 1: C = C + A.B^T (fp32 add, one rounding)
  float* c32;      // optional fp32 accumulator [m x ldc]: as TcGemmArgs::d32
  int finalize;
};

// CUDA-core FFMA GEMM for any layout (fp32 path, and shapes the tensor-core
// path does not take).
cudaError_t launch_gemm_simt(int dtype, const GemmArgs& g, cudaStream_t st);

}  // namespace fljsd
