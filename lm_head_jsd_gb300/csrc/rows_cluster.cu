// Passes 2 and 3 of the generalized JSD for bf16 logits, one 4-CTA cluster per
// row ("[Perf] Fuse log-softmax into fused_linear_jsd kernel", PR 1352,
// "Details": pass 2 accumulates the loss and dX_sum, pass 3 writes dX through
// the softmax Jacobian over the student logits buffer).
//
// Each CTA of the cluster owns a quarter of the row. Pass 2 keeps every
// element's X - log M (fp32, log2 units) in shared memory, so pass 3 needs
// only Q = 2^X and that cached value -- one ex2 per element instead of three,
// and no second read of the teacher logits. The row sums of the four quarters
// are exchanged through distributed shared memory and added in a fixed order,
// so every CTA (and every run) gets the same totals. Pass 1 comes from the
// logits GEMM's per-tile partials, which each CTA combines for the whole row.
#include "internal.cuh"
#include "jsd_math.cuh"

#include <math_constants.h>

namespace fljsd {
namespace {

using namespace rowmath;

constexpr int kCl = 4;          // CTAs per row
constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCacheBytes = 200 * 1024;

__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Read a float2 at the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float2 ld_peer_f2(const float2* local, uint32_t rank) {
  uint32_t addr = static_cast<uint32_t>(__cvta_generic_to_shared(local)), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(remote)
               : "memory");
  return v;
}

struct MD {
  float m, d;
};
__device__ __forceinline__ MD md_combine(MD a, MD b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -CUDART_INF_F) return MD{m, 0.f};
  return MD{m, (a.m == -CUDART_INF_F ? 0.f : a.d * ex2(a.m - m)) +
                   (b.m == -CUDART_INF_F ? 0.f : b.d * ex2(b.m - m))};
}
__device__ __forceinline__ MD block_md(MD v, MD* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = md_combine(v, MD{__shfl_xor_sync(0xffffffffu, v.m, o),
                         __shfl_xor_sync(0xffffffffu, v.d, o)});
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  MD r = sh[0];
  for (int w = 1; w < kWarps; ++w) r = md_combine(r, sh[w]);
  __syncthreads();
  return r;
}
__device__ __forceinline__ float2 block_sum2(float2 v, float2* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
  }
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  float2 r = sh[0];
  for (int w = 1; w < kWarps; ++w) {
    r.x += sh[w].x;
    r.y += sh[w].y;
  }
  __syncthreads();
  return r;
}

// X2 = log2 Q and Y2 = log2 P of one element, the exact product rounded once
// relative to the row maximum (as the row kernel does), then the generalized
// terms: Q, P, xm = X2 - log2 M, ym = Y2 - log2 M (0 at a tie).
__device__ __forceinline__ void terms(float zs, float zt, float c, float ma, float lda, float mb,
                                      float ldb, float beta, float omb, float& X2, float& Q,
                                      float& P, float& xm, float& ym) {
  X2 = __fsub_rn(__fmaf_rn(zs, c, -ma), lda);
  const float Y2 = __fsub_rn(__fmaf_rn(zt, c, -mb), ldb);
  Q = ex2(X2);
  P = ex2(Y2);
  const float lM = lg2(fmaxf(fmaf(omb, Q, beta * P), 1.17549435e-38f));
  const bool tie = X2 == Y2;
  xm = tie ? 0.f : X2 - lM;
  ym = tie ? 0.f : Y2 - lM;
}

__global__ void __launch_bounds__(kThreads, 1) k_jsd_rows_cluster(JsdRowArgs a) {
  extern __shared__ float xm_cache[];
  __shared__ MD sh_md[kWarps];
  __shared__ float2 sh_s[kWarps];
  __shared__ float2 part[2];  // this CTA's (sum Q xm, sum P ym), double-buffered by row
  const uint32_t rank = cl_rank();
  const int cid = blockIdx.x / kCl, ncl = gridDim.x / kCl;
  const float c = a.scale_log2;
  const float beta = a.beta, omb = 1.f - a.beta;
  const int n_valid = *a.n_valid;
  const int64_t nvec = a.v / 8;                  // 16-byte vectors of 8 bf16
  const int64_t q = (nvec + kCl - 1) / kCl;      // vectors per CTA
  const int64_t v0 = (int64_t)rank * q;
  const int64_t v1 = v0 + q < nvec ? v0 + q : nvec;
  const bool last = rank == kCl - 1;             // also owns the scalar tail
  const int64_t tail0 = nvec * 8;
  int it = 0;  // counts valid rows: the parity of `part` alternates between them

  for (int64_t r = cid; r < a.rows; r += ncl) {
    const int64_t grow = a.row0 + r;
    uint4* zs = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.zs) + r * a.ld);
    const uint4* zt =
        reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.zt) + r * a.ld);
    __nv_bfloat16* zse = reinterpret_cast<__nv_bfloat16*>(a.zs) + r * a.ld;
    const __nv_bfloat16* zte = reinterpret_cast<const __nv_bfloat16*>(a.zt) + r * a.ld;
    const bool valid = (a.labels == nullptr) || (a.labels[grow] != a.ignore_index);
    if (!valid) {
      // every CTA of the cluster sees the same row and skips it together
      for (int64_t i = v0 + threadIdx.x; i < v1; i += blockDim.x) zs[i] = make_uint4(0, 0, 0, 0);
      if (last)
        for (int64_t j = tail0 + threadIdx.x; j < a.v; j += blockDim.x)
          zse[j] = __float2bfloat16_rn(0.f);
      if (rank == 0 && threadIdx.x == 0) a.loss_rows[grow] = 0.f;
      continue;
    }
    float w = 1.f;
    switch (a.reduction) {
      case FLJSD_RED_NONE: w = a.row_grad ? a.row_grad[grow] : 1.f; break;
      case FLJSD_RED_SUM: w = 1.f; break;
      case FLJSD_RED_BATCHMEAN: w = n_valid > 0 ? (float)(1.0 / (double)n_valid) : 0.f; break;
      default: w = n_valid > 0 ? (float)(1.0 / ((double)n_valid * (double)a.v)) : 0.f; break;
    }

    // ---- pass 1: combine the GEMM epilogue's per-tile partials ----
    MD sa{-CUDART_INF_F, 0.f}, sb{-CUDART_INF_F, 0.f};
    const float2* ps = a.stats_s + r * a.ntiles;
    const float2* pt = a.stats_t + r * a.ntiles;
    for (int64_t i = threadIdx.x; i < a.ntiles; i += blockDim.x) {
      sa = md_combine(sa, MD{ps[i].x, ps[i].y});
      sb = md_combine(sb, MD{pt[i].x, pt[i].y});
    }
    sa = block_md(sa, sh_md);
    sb = block_md(sb, sh_md);
    const float ma = sa.m, mb = sb.m, lda = lg2(sa.d), ldb = lg2(sb.d);

    // ---- pass 2 over this CTA's quarter; cache X - log M ----
    float accq = 0.f, accp = 0.f;
    for (int64_t i = v0 + threadIdx.x; i < v1; i += blockDim.x) {
      const uint4 ws = zs[i], wt = zt[i];
      const uint32_t s4[4] = {ws.x, ws.y, ws.z, ws.w}, t4[4] = {wt.x, wt.y, wt.z, wt.w};
      float xm8[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float X2, Q, P, xm, ym;
        terms(__uint_as_float(s4[e] << 16), __uint_as_float(t4[e] << 16), c, ma, lda, mb, ldb,
              beta, omb, X2, Q, P, xm, ym);
        accq = fmaf(Q, xm, accq);
        accp = fmaf(P, ym, accp);
        xm8[2 * e] = xm;
        terms(__uint_as_float(s4[e] & 0xffff0000u), __uint_as_float(t4[e] & 0xffff0000u), c, ma,
              lda, mb, ldb, beta, omb, X2, Q, P, xm, ym);
        accq = fmaf(Q, xm, accq);
        accp = fmaf(P, ym, accp);
        xm8[2 * e + 1] = xm;
      }
      float4* dst = reinterpret_cast<float4*>(xm_cache + (i - v0) * 8);
      dst[0] = make_float4(xm8[0], xm8[1], xm8[2], xm8[3]);
      dst[1] = make_float4(xm8[4], xm8[5], xm8[6], xm8[7]);
    }
    if (last) {
      for (int64_t j = tail0 + threadIdx.x; j < a.v; j += blockDim.x) {
        float X2, Q, P, xm, ym;
        terms(__bfloat162float(zse[j]), __bfloat162float(zte[j]), c, ma, lda, mb, ldb, beta, omb,
              X2, Q, P, xm, ym);
        accq = fmaf(Q, xm, accq);
        accp = fmaf(P, ym, accp);
      }
    }
    const float2 mine = block_sum2(make_float2(accq, accp), sh_s);
    // part[it & 1] was last read by the peers before the previous valid row's
    // cluster barrier, which this CTA has passed
    if (threadIdx.x == 0) part[it & 1] = mine;
    cl_sync();  // every quarter's sums are visible cluster-wide
    float2 tot = make_float2(0.f, 0.f);
    for (uint32_t k = 0; k < kCl; ++k) {  // fixed order: identical totals in all CTAs
      const float2 u = ld_peer_f2(&part[it & 1], k);
      tot.x += u.x;
      tot.y += u.y;
    }
    const float S2 = omb * tot.x;
    const float L2 = fmaf(beta, tot.y, S2);
    if (rank == 0 && threadIdx.x == 0)
      a.loss_rows[grow] = 0.6931471805599453f * L2 * a.loss_scale;

    // ---- pass 3: dz = ln2 * scale * Q * ((1-beta) xm - S) ----
    const float k0 = 0.6931471805599453f * w * a.inv_temperature * a.loss_scale;
    const float k1 = k0 * omb, k2 = k0 * S2;
    for (int64_t i = v0 + threadIdx.x; i < v1; i += blockDim.x) {
      const uint4 ws = zs[i];
      const uint32_t s4[4] = {ws.x, ws.y, ws.z, ws.w};
      const float4* src = reinterpret_cast<const float4*>(xm_cache + (i - v0) * 8);
      const float4 c0 = src[0], c1 = src[1];
      const float xm8[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float X0 = __fsub_rn(__fmaf_rn(__uint_as_float(s4[e] << 16), c, -ma), lda);
        const float X1 = __fsub_rn(__fmaf_rn(__uint_as_float(s4[e] & 0xffff0000u), c, -ma), lda);
        const float g0 = ex2(X0) * fmaf(k1, xm8[2 * e], -k2);
        const float g1 = ex2(X1) * fmaf(k1, xm8[2 * e + 1], -k2);
        __nv_bfloat162 h = __floats2bfloat162_rn(g0, g1);
        o[e] = *reinterpret_cast<uint32_t*>(&h);
      }
      zs[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (last) {
      for (int64_t j = tail0 + threadIdx.x; j < a.v; j += blockDim.x) {
        float X2, Q, P, xm, ym;
        terms(__bfloat162float(zse[j]), __bfloat162float(zte[j]), c, ma, lda, mb, ldb, beta, omb,
              X2, Q, P, xm, ym);
        zse[j] = __float2bfloat16_rn(Q * fmaf(k1, xm, -k2));
      }
    }
    ++it;
    __syncthreads();
  }
  cl_sync();  // no CTA leaves while a peer may still read its partial sums
}

}  // namespace

bool jsd_rows_cluster_supported(const JsdRowArgs& a) {
  const int64_t nvec = a.v / 8;
  const int64_t q = (nvec + kCl - 1) / kCl;
  return a.stats_s != nullptr && a.stats_t != nullptr && a.beta > 0.f && a.beta < 1.f &&
         a.ld % 8 == 0 && q * 8 * (int64_t)sizeof(float) <= kMaxCacheBytes && nvec >= kCl;
}

cudaError_t launch_jsd_rows_cluster(const JsdRowArgs& a, cudaStream_t st) {
  const int64_t nvec = a.v / 8;
  const int64_t q = (nvec + kCl - 1) / kCl;
  const size_t smem = (size_t)q * 8 * sizeof(float);
  static int max_clusters[64] = {0};
  static size_t smem_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cache = dev >= 0 && dev < 64;
  if (!cache || smem_set[dev] < smem) {
    cudaError_t e = cudaFuncSetAttribute(k_jsd_rows_cluster,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMaxCacheBytes);
    if (e != cudaSuccess) return e;
    if (cache) smem_set[dev] = kMaxCacheBytes;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!cache || max_clusters[dev] == 0) {
    int n = 0;
    cfg.gridDim = dim3(kCl * (num_sms() / kCl));
    cfg.dynamicSmemBytes = kMaxCacheBytes;
    if (cudaOccupancyMaxActiveClusters(&n, k_jsd_rows_cluster, &cfg) != cudaSuccess || n <= 0)
      n = 1;
    cfg.dynamicSmemBytes = smem;
    if (cache) max_clusters[dev] = n;
    else max_clusters[0] = n;
  }
  const int mc = cache ? max_clusters[dev] : max_clusters[0];
  const int64_t clusters = a.rows < mc ? a.rows : mc;
  cfg.gridDim = dim3((unsigned)(kCl * clusters));
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_jsd_rows_cluster, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace fljsd
