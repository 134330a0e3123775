// CUDA-core FFMA GEMM, C (+)= A . B^T with arbitrary operand strides.
//
// It carries the fp32 path (the 5th-generation tensor cores take no fp32
// operands, and kind::tf32 would lose about three decimal digits), and it is
// the plain reference the tensor-core GEMMs are unit-tested against. fp32
// accumulation; with `accumulate` the stored value is read, the fp32 product
// added, and the sum rounded once ("perf(flce): write the weight-gradient
// product directly into grad_weight", Liger-Kernel PR 1429, "Summary").
#include "internal.cuh"

namespace fljsd {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, THREADS = 256;

template <typename T> __device__ __forceinline__ float ld_f(const T* p);
template <> __device__ __forceinline__ float ld_f<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ T to_t(float x);
template <> __device__ __forceinline__ float to_t<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 to_t<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Load a [rows x BK] tile of a strided operand into s[BK][rows + 4] (k-major
// in shared memory). The thread-to-element map walks the contiguous
// dimension fastest.
template <typename T, int ROWS>
__device__ __forceinline__ void load_tile(float (*s)[ROWS + 4], const T* p, int64_t srow,
                                          int64_t sk, int64_t row0, int64_t k0, int64_t nrow,
                                          int64_t nk) {
  const bool k_contig = (sk == 1);
  for (int i = threadIdx.x; i < ROWS * BK; i += THREADS) {
    int kk, rr;
    if (k_contig) { kk = i % BK; rr = i / BK; }
    else { rr = i % ROWS; kk = i / ROWS; }
    const int64_t r = row0 + rr, k = k0 + kk;
    s[kk][rr] = (r < nrow && k < nk) ? ld_f<T>(p + r * srow + k * sk) : 0.f;
  }
}

template <typename T>
__global__ void __launch_bounds__(THREADS) k_gemm_simt(GemmArgs g) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const T* A = reinterpret_cast<const T*>(g.a);
  const T* B = reinterpret_cast<const T*>(g.b);
  T* C = reinterpret_cast<T*>(g.c);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int64_t k0 = 0; k0 < g.k; k0 += BK) {
    load_tile<T, BM>(As, A, g.sam, g.sak, m0, k0, g.m, g.k);
    load_tile<T, BN>(Bs, B, g.sbn, g.sbk, n0, k0, g.n, g.k);
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= g.m) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx * 4 + j;
      if (n >= g.n) continue;
      T* out = C + m * g.ldc + n;
      float v = acc[i][j];
      if (g.c32 != nullptr) {
        float* o32 = g.c32 + m * g.ldc + n;
        if (g.accumulate || g.finalize) v += *o32;
        if (g.finalize) *out = to_t<T>(v);
        else *o32 = v;
      } else {
        if (g.accumulate) v += ld_f<T>(out);
        *out = to_t<T>(v);
      }
    }
  }
}

}  // namespace

cudaError_t launch_gemm_simt(int dtype, const GemmArgs& g, cudaStream_t st) {
  if (g.m <= 0 || g.n <= 0) return cudaSuccess;
  const int64_t gx = (g.n + BN - 1) / BN, gy = (g.m + BM - 1) / BM;
  if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)gx, (unsigned)gy);
  if (dtype == FLJSD_BF16)
    k_gemm_simt<__nv_bfloat16><<<grid, THREADS, 0, st>>>(g);
  else
    k_gemm_simt<float><<<grid, THREADS, 0, st>>>(g);
  return cudaGetLastError();
}

}  // namespace fljsd
