// Distances over given distributions (no GEMM): the log-space JSD and the
// total variation distance, one pass over each row.
//
// Log-space JSD: the public contract of Liger's _jsd_kernel ("[Perf] Fuse
// log-softmax into fused_linear_jsd kernel", PR 1352, Open questions 3): the
// inputs are already log-probabilities -- `input` X = log Q (student) and
// `target` Y = log P (teacher) -- so there is no softmax and no cross-column
// term: the gradient is d loss / d X element by element.
//
// TVD: 0.5 * |p - q| per element with the gradient in p taken as
// 0.5 * sign(p - q) with the three-way sign, exactly 0 at p == q ("Fix TVD
// gradient at p == q", PR 1374, Summary).
//
// Both are HBM-bound: read two [rows x V] tensors, write one.
#include "internal.cuh"
#include "jsd_math.cuh"

namespace fljsd {
namespace {

using namespace rowmath;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float block_sum(float v, float* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  float r = sh[0];
  for (int w = 1; w < kWarps; ++w) r += sh[w];
  __syncthreads();
  return r;
}

__device__ __forceinline__ float row_weight(int reduction, int n_valid, int64_t v) {
  switch (reduction) {
    case FLJSD_RED_NONE:
    case FLJSD_RED_SUM: return 1.f;
    case FLJSD_RED_BATCHMEAN: return n_valid > 0 ? (float)(1.0 / (double)n_valid) : 0.f;
    default: return n_valid > 0 ? (float)(1.0 / ((double)n_valid * (double)v)) : 0.f;
  }
}

// Log-space JSD of one element (natural-log inputs): loss and d loss / d X.
template <int BRANCH, bool PREC>
__device__ __forceinline__ void logspace_elem(float x, float y, float beta, float omb,
                                              float& ell, float& dx) {
  const float L2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;
  const float Y2 = __fmul_rn(y, L2E);
  const float d = __fsub_rn(__fmul_rn(x, L2E), Y2);
  float ell2, g2;
  elem_loss<BRANCH, PREC>(Y2, d, beta, omb, ell2, g2);
  ell = LN2 * ell2;
  if (BRANCH == 0) {
    dx = -pexp2<PREC>(Y2);  // d/dX of P (Y - X)
  } else if (BRANCH == 1) {
    dx = pexp2<PREC>(Y2 + d) * fmaf(LN2, d, 1.f);  // d/dX of Q (X - Y) = Q (X - Y + 1)
  } else {
    dx = LN2 * g2;  // (1 - beta) Q (X - log M); exactly 0 at a tie
  }
}

template <typename T, int BRANCH>
__global__ void __launch_bounds__(kThreads) k_jsd_logspace(DistArgs a) {
  using V = Vec<T>;
  constexpr int N = V::N;
  constexpr bool PREC = sizeof(T) == 4;
  __shared__ float sh[kWarps];
  const float beta = a.beta, omb = 1.f - a.beta;
  const int n_valid = *a.n_valid;
  const float w = row_weight(a.reduction, n_valid, a.v);
  for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
    const T* xr = reinterpret_cast<const T*>(a.x) + r * a.v;
    const T* yr = reinterpret_cast<const T*>(a.y) + r * a.v;
    T* gr = reinterpret_cast<T*>(a.grad) + r * a.v;
    const bool valid = (a.labels == nullptr) || (a.labels[r] != a.ignore_index);
    const bool vec = ((((uintptr_t)xr) | ((uintptr_t)yr) | ((uintptr_t)gr)) & 15u) == 0;
    const int64_t nvec = vec ? a.v / N : 0;
    float acc = 0.f;
    for (int64_t i = threadIdx.x; i < nvec; i += blockDim.x) {
      float xs[N], ys[N], g[N];
      if (valid) {
        V::load(xr + i * N, xs);
        V::load(yr + i * N, ys);
#pragma unroll
        for (int k = 0; k < N; ++k) {
          float ell, dx;
          logspace_elem<BRANCH, PREC>(xs[k], ys[k], beta, omb, ell, dx);
          acc += ell;
          g[k] = dx * w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < N; ++k) g[k] = 0.f;
      }
      V::store(gr + i * N, g);
    }
    for (int64_t j = nvec * N + threadIdx.x; j < a.v; j += blockDim.x) {
      float g = 0.f;
      if (valid) {
        float ell, dx;
        logspace_elem<BRANCH, PREC>(V::one(xr + j), V::one(yr + j), beta, omb, ell, dx);
        acc += ell;
        g = dx * w;
      }
      V::put(gr + j, g);
    }
    const float tot = block_sum(acc, sh);
    if (threadIdx.x == 0) a.loss_rows[r] = valid ? tot : 0.f;
  }
}

// TVD: loss 0.5 |p - q|, gradient 0.5 sign3(p - q) * w. With reduction none
// the loss is written per element into loss_elem.
template <typename T>
__global__ void __launch_bounds__(kThreads) k_tvd(DistArgs a) {
  using V = Vec<T>;
  constexpr int N = V::N;
  __shared__ float sh[kWarps];
  const int n_valid = *a.n_valid;
  const float hw = 0.5f * row_weight(a.reduction, n_valid, a.v);
  for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
    const T* pr = reinterpret_cast<const T*>(a.x) + r * a.v;
    const T* qr = reinterpret_cast<const T*>(a.y) + r * a.v;
    T* gr = reinterpret_cast<T*>(a.grad) + r * a.v;
    float* le = a.loss_elem ? a.loss_elem + r * a.v : nullptr;
    const bool valid = (a.labels == nullptr) || (a.labels[r] != a.ignore_index);
    const bool vec = ((((uintptr_t)pr) | ((uintptr_t)qr) | ((uintptr_t)gr) |
                       ((uintptr_t)le)) & 15u) == 0;
    const int64_t nvec = vec ? a.v / N : 0;
    float acc = 0.f;
    for (int64_t i = threadIdx.x; i < nvec; i += blockDim.x) {
      float p[N], q[N], g[N], l[N];
      V::load(pr + i * N, p);
      V::load(qr + i * N, q);
#pragma unroll
      for (int k = 0; k < N; ++k) {
        const float diff = p[k] - q[k];
        const float sgn = (diff > 0.f) ? 1.f : ((diff < 0.f) ? -1.f : 0.f);
        l[k] = valid ? 0.5f * fabsf(diff) : 0.f;
        g[k] = valid ? hw * sgn : 0.f;
        acc += l[k];
      }
      V::store(gr + i * N, g);
      if (le) {
#pragma unroll
        for (int k = 0; k < N; ++k) le[i * N + k] = l[k];
      }
    }
    for (int64_t j = nvec * N + threadIdx.x; j < a.v; j += blockDim.x) {
      const float diff = V::one(pr + j) - V::one(qr + j);
      const float sgn = (diff > 0.f) ? 1.f : ((diff < 0.f) ? -1.f : 0.f);
      const float l = valid ? 0.5f * fabsf(diff) : 0.f;
      V::put(gr + j, valid ? hw * sgn : 0.f);
      if (le) le[j] = l;
      acc += l;
    }
    const float tot = block_sum(acc, sh);
    if (threadIdx.x == 0) a.loss_rows[r] = tot;
  }
}

template <typename T>
cudaError_t launch_logspace_t(const DistArgs& a, cudaStream_t st) {
  const int64_t cap = (int64_t)num_sms() * 4;
  const unsigned grid = (unsigned)(a.rows < cap ? a.rows : cap);
  if (a.beta == 0.f)
    k_jsd_logspace<T, 0><<<grid, kThreads, 0, st>>>(a);
  else if (a.beta == 1.f)
    k_jsd_logspace<T, 1><<<grid, kThreads, 0, st>>>(a);
  else
    k_jsd_logspace<T, 2><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_jsd_logspace(int dtype, const DistArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  trace_begin(FLJSD_KERNEL_JSD_ROWS, st);
  cudaError_t e = dtype == FLJSD_BF16 ? launch_logspace_t<__nv_bfloat16>(a, st)
                                      : launch_logspace_t<float>(a, st);
  trace_end(FLJSD_KERNEL_JSD_ROWS, st);
  return e;
}

cudaError_t launch_tvd(int dtype, const DistArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  trace_begin(FLJSD_KERNEL_JSD_ROWS, st);
  const int64_t cap = (int64_t)num_sms() * 4;
  const unsigned grid = (unsigned)(a.rows < cap ? a.rows : cap);
  if (dtype == FLJSD_BF16)
    k_tvd<__nv_bfloat16><<<grid, kThreads, 0, st>>>(a);
  else
    k_tvd<float><<<grid, kThreads, 0, st>>>(a);
  trace_end(FLJSD_KERNEL_JSD_ROWS, st);
  return cudaGetLastError();
}

}  // namespace fljsd
