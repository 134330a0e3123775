// Row kernels of the fused-linear JSD: the passes over the vocabulary, the
// valid-row count, the final loss reduction and the backward scaling.
//
// The three-pass structure follows "[Perf] Fuse log-softmax into
// fused_linear_jsd kernel" (Liger-Kernel PR 1352), "Details": pass 1 builds
// the running max m and denominator d of the student and teacher softmaxes
// together (online softmax, Milakov & Gimelshein, Algorithm 3); pass 2
// accumulates the per-row loss and the cross-column term dX_sum; pass 3
// recomputes dX and writes the logit gradient over the student logits
// buffer. On the tensor-core path pass 1 runs in the logits GEMM's epilogue
// and this kernel only combines its per-tile partials. Logits are read in the
// input dtype and widened at load; all math is fp32 in registers; e^x is
// evaluated as 2^(x*log2 e) (the ex2 unit for bf16, exp2f for fp32).
#include "internal.cuh"
#include "jsd_math.cuh"

#include <cuda_fp16.h>
#include <math_constants.h>

#include <cstdlib>

namespace fljsd {
namespace {

using namespace rowmath;

constexpr int kRowThreads = 1024;
constexpr int64_t kCacheVecMax = 14336;  // 224 KB of fp16 (8 elements per vector)
constexpr int kWarps = kRowThreads / 32;
constexpr int kRowsPrefetchChunks = 2;  // L2 prefetch distance of pass 2, in chunks

// ---- (max, sum of 2^(x - max)) pairs -----------------------------------------
struct MD {
  float m, d;
};
__device__ __forceinline__ MD md_combine(MD a, MD b) {
  float m = fmaxf(a.m, b.m);
  if (m == -CUDART_INF_F) return MD{m, 0.f};
  float d = (a.m == -CUDART_INF_F ? 0.f : a.d * ex2(a.m - m)) +
            (b.m == -CUDART_INF_F ? 0.f : b.d * ex2(b.m - m));
  return MD{m, d};
}

// Fold a group of logits z into a running (m, d) of x = z * c (log2 units):
// m is the largest rounded product, and each x - m comes from the exact
// product rounded once (the same rule as the GEMM epilogue's partials).
template <int N>
__device__ __forceinline__ void md_fold(MD& s, const float (&z)[N], float c) {
  float vm = __fmul_rn(z[0], c);
#pragma unroll
  for (int i = 1; i < N; ++i) vm = fmaxf(vm, __fmul_rn(z[i], c));
  if (vm > s.m) {
    s.d = (s.m == -CUDART_INF_F) ? 0.f : s.d * ex2(s.m - vm);
    s.m = vm;
  }
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) acc += ex2(__fmaf_rn(z[i], c, -s.m));
  s.d += acc;
}

// Block-wide reductions in a fixed order (deterministic): inside each warp,
// then over the per-warp results in warp 0, the total broadcast from the slot
// after theirs.
__device__ __forceinline__ float2 warp_sum2(float2 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = __fadd2_rn(v, make_float2(__shfl_xor_sync(0xffffffffu, v.x, o),
                                  __shfl_xor_sync(0xffffffffu, v.y, o)));
  return v;
}
// Largest value over the warp in one instruction (exact, so order-free).
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
// The student's and the teacher's (m, d) over a warp: the warp's largest m,
// every lane's d rescaled to it, and those summed in a fixed butterfly order
// (one ex2 a lane instead of one per butterfly level).
__device__ __forceinline__ void warp_md2(MD& a, MD& b) {
  const float ma = warp_max(a.m), mb = warp_max(b.m);
  float2 d = make_float2(ma == -CUDART_INF_F ? 0.f : a.d * ex2(a.m - ma),
                         mb == -CUDART_INF_F ? 0.f : b.d * ex2(b.m - mb));
  d = warp_sum2(d);
  a = MD{ma, d.x};
  b = MD{mb, d.y};
}
// The student's and the teacher's (m, d) together: one pair of barriers.
// sh holds 2 * (NW + 1).
template <int NW>
__device__ __forceinline__ void block_md2(MD& va, MD& vb, MD* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_md2(va, vb);
  if (lane == 0) {
    sh[2 * warp] = va;
    sh[2 * warp + 1] = vb;
  }
  __syncthreads();
  if (warp == 0) {
    MD ua = lane < NW ? sh[2 * lane] : MD{-CUDART_INF_F, 0.f};
    MD ub = lane < NW ? sh[2 * lane + 1] : MD{-CUDART_INF_F, 0.f};
    warp_md2(ua, ub);
    if (lane == 0) {
      sh[2 * NW] = ua;
      sh[2 * NW + 1] = ub;
    }
  }
  __syncthreads();
  va = sh[2 * NW];
  vb = sh[2 * NW + 1];
}

template <int NW>
__device__ __forceinline__ float2 block_sum2(float2 v, float2* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum2(v);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float2 u = lane < NW ? sh[lane] : make_float2(0.f, 0.f);
    u = warp_sum2(u);
    if (lane == 0) sh[NW] = u;
  }
  __syncthreads();
  return sh[NW];
}

// Bulk prefetch of [p, p + bytes) into L2 (16-byte aligned, a multiple of 16
// bytes); nothing waits for it.
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// The 16-byte units that lie wholly inside [p, p + bytes) into L2 (a
// prefetch; bytes outside the span are not touched).
__device__ __forceinline__ void l2_prefetch_span(const void* p, size_t bytes) {
  const uintptr_t b = ((uintptr_t)p + 15u) & ~(uintptr_t)15u;
  const uintptr_t e = ((uintptr_t)p + bytes) & ~(uintptr_t)15u;
  if (e > b) l2_prefetch(reinterpret_cast<const void*>(b), (uint32_t)(e - b));
}

// Two floats to fp16x2 (lo in the low half), saturated to the finite range.
__device__ __forceinline__ uint32_t pack_half2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Generalized-branch terms of one bf16 element for the lean path: X2, Y2 from
// one fma each, P, Q, and the log ratios X - log M, Y - log M (both exactly 0
// at a tie), in log2 units.
__device__ __forceinline__ void lean_terms(float zs, float zt, float c, float oa, float ob,
                                           float beta, float omb, float& Q, float& P,
                                           float& xm, float& ym) {
  const float X2 = __fmaf_rn(zs, c, -oa);
  const float Y2 = __fmaf_rn(zt, c, -ob);
  Q = ex2(X2);
  P = ex2(Y2);
  // M + 2^-126 instead of max(M, 2^-126): the same guard against log2(0)
  // where both terms flush to zero, one instruction less. At a tie log2 M is
  // taken as X2 (= Y2) itself, so that both log ratios are exactly 0.
  const float lM = (X2 == Y2) ? X2 : lg2(fmaf(omb, Q, fmaf(beta, P, 1.17549435e-38f)));
  xm = X2 - lM;
  ym = Y2 - lM;
}

// lean_terms for two elements at a time, on the packed fp32x2 FMA / ADD / MUL
// instructions (each lane rounds exactly like the scalar operation, so the
// terms are bitwise those of lean_terms). c2 = (c, c), noa = (-oa, -oa), ...
__device__ __forceinline__ void lean_terms2(float2 zs, float2 zt, float2 c2, float2 noa,
                                            float2 nob, float2 beta2, float2 omb2, float2& Q,
                                            float2& P, float2& xm, float2& ym) {
  const float2 X2 = __ffma2_rn(zs, c2, noa);
  const float2 Y2 = __ffma2_rn(zt, c2, nob);
  Q = make_float2(ex2(X2.x), ex2(X2.y));
  P = make_float2(ex2(Y2.x), ex2(Y2.y));
  const float2 M = __ffma2_rn(omb2, Q, __ffma2_rn(beta2, P, make_float2(1.17549435e-38f, 1.17549435e-38f)));
  const float2 lM = make_float2((X2.x == Y2.x) ? X2.x : lg2(M.x), (X2.y == Y2.y) ? X2.y : lg2(M.y));
  const float2 m1 = make_float2(-1.f, -1.f);
  xm = __ffma2_rn(lM, m1, X2);  // X2 - lM, exact product, one rounding
  ym = __ffma2_rn(lM, m1, Y2);
}

template <typename T, int BRANCH>
__global__ void __launch_bounds__(kRowThreads, 1) k_jsd_rows(JsdRowArgs a) {
  using V = Vec<T>;
  constexpr bool PREC = sizeof(T) == 4;
  constexpr int N = V::N;
  __shared__ MD sh_md[2 * (kWarps + 1)];
  __shared__ float2 sh_s[kWarps + 1];
  extern __shared__ uint4 xm_cache[];  // lean path: fp16 X - log M of cache_vec vectors

  const float c = a.scale_log2;  // log2(e) / T
  const float beta = a.beta, omb = 1.f - a.beta;
  const int64_t nvec = a.v / N;
  const int64_t tail0 = nvec * N;
  const int n_valid = *a.n_valid;

  for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
    const int64_t grow = a.row0 + r;
    T* zs = reinterpret_cast<T*>(a.zs) + r * a.ld;
    const T* zt = reinterpret_cast<const T*>(a.zt) + r * a.ld;
    if (threadIdx.x == 0 && a.rows_prefetch && r + gridDim.x < a.rows) {
      // the next row's label and pass-1 partials into L2, a row ahead: they
      // are the first loads of the row and nothing else would hide their latency
      const int64_t rn = r + gridDim.x;
      if (a.labels != nullptr)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.labels + a.row0 + rn) : "memory");
      if (a.stats_s != nullptr) {
        l2_prefetch_span(a.stats_s + rn * a.ntiles, (size_t)a.ntiles * sizeof(float2));
        l2_prefetch_span(a.stats_t + rn * a.ntiles, (size_t)a.ntiles * sizeof(float2));
      }
    }
    const bool valid = (a.labels == nullptr) || (a.labels[grow] != a.ignore_index);
    if (BRANCH == 2 && !PREC && valid && a.rows_prefetch && threadIdx.x == 0) {
      // the head of both rows, while pass 1's partials are combined (pass 2
      // keeps its prefetches ahead of the block from there on)
      const size_t head = (size_t)(nvec < 2 * kRowsPrefetchChunks * (int64_t)blockDim.x
                                       ? nvec
                                       : 2 * kRowsPrefetchChunks * (int64_t)blockDim.x) *
                          N * sizeof(T);
      l2_prefetch_span(zs, head);
      l2_prefetch_span(zt, head);
    }

    float w = 0.f;  // row weight w_r
    if (valid) {
      switch (a.reduction) {
        case FLJSD_RED_NONE: w = a.row_grad ? a.row_grad[grow] : 1.f; break;
        case FLJSD_RED_SUM: w = 1.f; break;
        case FLJSD_RED_BATCHMEAN: w = n_valid > 0 ? (float)(1.0 / (double)n_valid) : 0.f; break;
        default: w = n_valid > 0 ? (float)(1.0 / ((double)n_valid * (double)a.v)) : 0.f; break;
      }
    }
    if (!valid) {
      // ignored row: zero loss and zero gradient over [0, V)
      float zero[N];
#pragma unroll
      for (int i = 0; i < N; ++i) zero[i] = 0.f;
      for (int64_t i = threadIdx.x; i < nvec; i += blockDim.x) V::store(zs + i * N, zero);
      for (int64_t j = tail0 + threadIdx.x; j < a.v; j += blockDim.x) V::put(zs + j, 0.f);
      if (threadIdx.x == 0) a.loss_rows[grow] = 0.f;
      continue;
    }

    // ---- pass 1: m/d of student (a) and teacher (b) together ----
    MD ma{-CUDART_INF_F, 0.f}, mb{-CUDART_INF_F, 0.f};
    if (a.stats_s != nullptr) {
      // the logits GEMM already folded each 128 columns of this row
      const float2* ps = a.stats_s + r * a.ntiles;
      const float2* pt = a.stats_t + r * a.ntiles;
      if ((int64_t)threadIdx.x < a.ntiles) {  // a thread's first partial as it is
        const float2 u = ps[threadIdx.x], w2 = pt[threadIdx.x];
        ma = MD{u.x, u.y};
        mb = MD{w2.x, w2.y};
      }
      for (int64_t i = threadIdx.x + blockDim.x; i < a.ntiles; i += blockDim.x) {
        const float2 u = ps[i], w2 = pt[i];
        ma = md_combine(ma, MD{u.x, u.y});
        mb = md_combine(mb, MD{w2.x, w2.y});
      }
    } else {
      for (int64_t i = threadIdx.x; i < nvec; i += blockDim.x) {
        float xs[N], xt[N];
        V::load(zs + i * N, xs);
        V::load(zt + i * N, xt);
        md_fold<N>(ma, xs, c);
        md_fold<N>(mb, xt, c);
      }
      for (int64_t j = tail0 + threadIdx.x; j < a.v; j += blockDim.x) {
        float xs[1] = {V::one(zs + j)};
        float xt[1] = {V::one(zt + j)};
        md_fold<1>(ma, xs, c);
        md_fold<1>(mb, xt, c);
      }
    }
    block_md2<kWarps>(ma, mb, sh_md);
    const MD ra = ma, rb = mb;
    // log2 Q_j = z_j * c - m_a - log2 d_a, formed as fma(z, c, -m) - log2 d so
    // that the exact product is rounded once relative to the row maximum.
    // A one-element row has log-prob 0 whatever its logit.
    const bool single = (a.v == 1);
    const float ma_ = single ? 0.f : ra.m, mb_ = single ? 0.f : rb.m;
    const float lda = single ? 0.f : plog2<PREC>(ra.d);
    const float ldb = single ? 0.f : plog2<PREC>(rb.d);
    const float cz = single ? 0.f : c;

    // Lean path for the generalized branch on bf16 logits: the two row offsets
    // fold into one fma per element (exact to 2^-18 in log2 units while the
    // row maxima are below 64, a constant per-row shift that the loss does not
    // feel at first order), and the per-element products accumulate with fmas:
    // S = (1-beta) sum Q xm, L = beta sum P ym + S. Pass 2 also keeps
    // xm = X - log M (fp16) of the row's first `cache_vec` vectors in shared
    // memory, so pass 3 needs only Q = 2^X there: one ex2 instead of three and
    // no second read of the teacher logits.
    if (BRANCH == 2 && !PREC && fabsf(ma_) < 64.f && fabsf(mb_) < 64.f) {
      const float oa = ma_ + lda, ob = mb_ + ldb;
      float accq = 0.f, accp = 0.f;
      // pair forms of the constants, and pair accumulators (even and odd
      // elements, added at the end of the row)
      const float2 c2 = make_float2(cz, cz), noa = make_float2(-oa, -oa), nob = make_float2(-ob, -ob);
      const float2 beta2 = make_float2(beta, beta), omb2 = make_float2(omb, omb);
      float2 accq2 = make_float2(0.f, 0.f), accp2 = make_float2(0.f, 0.f);
      // 32-bit vector indices (nvec < 2^27): less index arithmetic per vector
      const int step = (int)blockDim.x;
      const int nv = (int)nvec;
      // Pass 2 streams both rows from DRAM. One thread keeps bulk L2
      // prefetches a few chunks (2 * step vectors of each row) ahead of the
      // block, so that the loads find their lines in L2 instead of waiting for
      // DRAM with only four 16-byte loads in flight per thread.
      const int chunk = 2 * step;
      auto prefetch_chunk = [&](int c0) {
        if (a.rows_prefetch && threadIdx.x == 0 && c0 < nv) {
          const uint32_t bytes = (uint32_t)((nv - c0 < chunk ? nv - c0 : chunk) * N * sizeof(T));
          l2_prefetch(zs + (int64_t)c0 * N, bytes);
          l2_prefetch(zt + (int64_t)c0 * N, bytes);
        }
      };
      // (the first kRowsPrefetchChunks chunks were prefetched at the row's start)
      const int ncache = (int)(nvec < a.cache_vec ? nvec : a.cache_vec);
      uint4* cache = reinterpret_cast<uint4*>(xm_cache);
      auto pass2_vec = [&](const float (&xs)[N], const float (&xt)[N], int v) {
        float xm8[N];
#pragma unroll
        for (int k = 0; k < N; k += 2) {
          float2 Q, P, xm, ym;
          lean_terms2(make_float2(xs[k], xs[k + 1]), make_float2(xt[k], xt[k + 1]), c2, noa, nob,
                      beta2, omb2, Q, P, xm, ym);
          accq2 = __ffma2_rn(Q, xm, accq2);
          accp2 = __ffma2_rn(P, ym, accp2);
          xm8[k] = xm.x;
          xm8[k + 1] = xm.y;
        }
        if (v < ncache) {
          // saturated to the fp16 range: where |xm| is that large Q is 0
          cache[v] = make_uint4(pack_half2_sat(xm8[0], xm8[1]), pack_half2_sat(xm8[2], xm8[3]),
                                pack_half2_sat(xm8[4], xm8[5]), pack_half2_sat(xm8[6], xm8[7]));
        }
      };
      int i = (int)threadIdx.x;
      // two vectors per iteration: four 16-byte loads in flight per thread
      for (; i + step < nv; i += 2 * step) {
        prefetch_chunk(i + kRowsPrefetchChunks * chunk);  // thread 0: i is the chunk start
        float xs[N], xt[N], xs2[N], xt2[N];
        V::load(zs + i * N, xs);
        V::load(zt + i * N, xt);
        V::load(zs + (i + step) * N, xs2);
        V::load(zt + (i + step) * N, xt2);
        pass2_vec(xs, xt, i);
        pass2_vec(xs2, xt2, i + step);
      }
      for (; i < nv; i += step) {
        float xs[N], xt[N];
        V::load(zs + i * N, xs);
        V::load(zt + i * N, xt);
        pass2_vec(xs, xt, i);
      }
      for (int64_t j = tail0 + threadIdx.x; j < a.v; j += blockDim.x) {
        float Q, P, xm, ym;
        lean_terms(V::one(zs + j), V::one(zt + j), cz, oa, ob, beta, omb, Q, P, xm, ym);
        accq = fmaf(Q, xm, accq);
        accp = fmaf(P, ym, accp);
      }
      accq += accq2.x + accq2.y;
      accp += accp2.x + accp2.y;
      const float2 tot = block_sum2<kWarps>(make_float2(accq, accp), sh_s);  // also orders the cache
      const float S2 = omb * tot.x;
      const float L2 = fmaf(beta, tot.y, S2);
      if (threadIdx.x == 0) a.loss_rows[grow] = 0.6931471805599453f * L2 * a.loss_scale;
      // dz = ln2 * scale * Q * ((1-beta) xm - S)
      const float k0 = 0.6931471805599453f * w * a.inv_temperature * a.loss_scale;
      const float k1 = k0 * omb, k2 = k0 * S2;
      const float2 k12 = make_float2(k1, k1), nk22 = make_float2(-k2, -k2);
      auto pass3_vec = [&](int v) {
        float xs[N];
        V::load(zs + v * N, xs);
        if (v < ncache) {
          const uint4 hv = cache[v];
          const uint32_t h[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 xm2 = __half22float2(*reinterpret_cast<const __half2*>(&h[e]));
            const float2 X = __ffma2_rn(make_float2(xs[2 * e], xs[2 * e + 1]), c2, noa);
            const float2 t = __ffma2_rn(k12, xm2, nk22);
            const float2 dz = __fmul2_rn(make_float2(ex2(X.x), ex2(X.y)), t);
            xs[2 * e] = dz.x;
            xs[2 * e + 1] = dz.y;
          }
        } else {
          float xt[N];
          V::load(zt + v * N, xt);
#pragma unroll
          for (int k = 0; k < N; k += 2) {
            float2 Q, P, xm, ym;
            lean_terms2(make_float2(xs[k], xs[k + 1]), make_float2(xt[k], xt[k + 1]), c2, noa, nob,
                        beta2, omb2, Q, P, xm, ym);
            const float2 dz = __fmul2_rn(Q, __ffma2_rn(k12, xm, nk22));
            xs[k] = dz.x;
            xs[k + 1] = dz.y;
          }
        }
        V::store(zs + v * N, xs);
      };
      // walk the row backwards: the lines pass 2 read last are the likeliest
      // to still be in L2
      int i3 = nv - 1 - (int)threadIdx.x;
      // four vectors per iteration; where all four are cached (the row's
      // first ncache vectors), their loads are all issued before any of them
      // is computed: more L2 reads in flight per thread (measured: 0.361 ->
      // 0.340 ms on 2048 full-length rows)
      for (; i3 - 3 * step >= 0; i3 -= 4 * step) {
        if (i3 >= ncache) {  // not all four cached: one at a time
          pass3_vec(i3);
          pass3_vec(i3 - step);
          pass3_vec(i3 - 2 * step);
          pass3_vec(i3 - 3 * step);
          continue;
        }
        // four cached vectors: all loads first
        float xs[4][N];
        uint4 hv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          V::load(zs + (i3 - u * step) * N, xs[u]);
          hv[u] = cache[i3 - u * step];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t h[4] = {hv[u].x, hv[u].y, hv[u].z, hv[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 xm2 = __half22float2(*reinterpret_cast<const __half2*>(&h[e]));
            const float2 X = __ffma2_rn(make_float2(xs[u][2 * e], xs[u][2 * e + 1]), c2, noa);
            const float2 t = __ffma2_rn(k12, xm2, nk22);
            const float2 dz = __fmul2_rn(make_float2(ex2(X.x), ex2(X.y)), t);
            xs[u][2 * e] = dz.x;
            xs[u][2 * e + 1] = dz.y;
          }
          V::store(zs + (i3 - u * step) * N, xs[u]);
        }
      }
      for (; i3 - step >= 0; i3 -= 2 * step) {
        pass3_vec(i3);
        pass3_vec(i3 - step);
      }
      for (; i3 >= 0; i3 -= step) pass3_vec(i3);
      for (int64_t j = tail0 + threadIdx.x; j < a.v; j += blockDim.x) {
        float Q, P, xm, ym;
        lean_terms(V::one(zs + j), V::one(zt + j), cz, oa, ob, beta, omb, Q, P, xm, ym);
        V::put(zs + j, Q * fmaf(k1, xm, -k2));
      }
      // no barrier here: the next row's pass-1 reduction (block_md2) holds
      // every thread before anyone writes the cache in its pass 2
      continue;
    }

    // ---- pass 2: loss and dX_sum ----
    float2 acc = make_float2(0.f, 0.f);
    for (int64_t i = threadIdx.x; i < nvec; i += blockDim.x) {
      float xs[N], xt[N];
      V::load(zs + i * N, xs);
      V::load(zt + i * N, xt);
#pragma unroll
      for (int k = 0; k < N; ++k) {
        const float Y2 = __fsub_rn(__fmaf_rn(xt[k], cz, -mb_), ldb);
        const float d = __fsub_rn(__fsub_rn(__fmaf_rn(xs[k], cz, -ma_), lda), Y2);
        float ell, g;
        elem_loss<BRANCH, PREC>(Y2, d, beta, omb, ell, g);
        acc.x += ell;
        acc.y += g;
      }
    }
    for (int64_t j = tail0 + threadIdx.x; j < a.v; j += blockDim.x) {
      const float Y2 = __fsub_rn(__fmaf_rn(V::one(zt + j), cz, -mb_), ldb);
      const float d = __fsub_rn(__fsub_rn(__fmaf_rn(V::one(zs + j), cz, -ma_), lda), Y2);
      float ell, g;
      elem_loss<BRANCH, PREC>(Y2, d, beta, omb, ell, g);
      acc.x += ell;
      acc.y += g;
    }
    const float2 tot = block_sum2<kWarps>(acc, sh_s);
    const float L2 = tot.x, S2 = tot.y;  // row loss and dX_sum, / ln 2
    if (threadIdx.x == 0) a.loss_rows[grow] = 0.6931471805599453f * L2 * a.loss_scale;

    // ---- pass 3: dlogits in place over the student logits ----
    const float scale = w * a.inv_temperature * a.loss_scale;
    // walk the row backwards: the lines pass 2 read last are the likeliest to
    // still be in L2
    for (int64_t i = nvec - 1 - threadIdx.x; i >= 0; i -= blockDim.x) {
      float xs[N], xt[N];
      V::load(zs + i * N, xs);
      V::load(zt + i * N, xt);
#pragma unroll
      for (int k = 0; k < N; ++k) {
        const float Y2 = __fsub_rn(__fmaf_rn(xt[k], cz, -mb_), ldb);
        const float d = __fsub_rn(__fsub_rn(__fmaf_rn(xs[k], cz, -ma_), lda), Y2);
        xs[k] = elem_grad<BRANCH, PREC>(Y2, d, beta, omb, L2, S2) * scale;
      }
      V::store(zs + i * N, xs);
    }
    for (int64_t j = tail0 + threadIdx.x; j < a.v; j += blockDim.x) {
      const float Y2 = __fsub_rn(__fmaf_rn(V::one(zt + j), cz, -mb_), ldb);
      const float d = __fsub_rn(__fsub_rn(__fmaf_rn(V::one(zs + j), cz, -ma_), lda), Y2);
      V::put(zs + j, elem_grad<BRANCH, PREC>(Y2, d, beta, omb, L2, S2) * scale);
    }
    __syncthreads();
  }
}

__global__ void k_count_valid(const int64_t* labels, int64_t bt, int64_t ignore_index,
                              int* n_valid) {
  __shared__ int sh[32];
  int c = 0;
  for (int64_t i = threadIdx.x; i < bt; i += blockDim.x)
    c += (labels == nullptr || labels[i] != ignore_index) ? 1 : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += sh[w];
    n_valid[0] = t;
    n_valid[1] = FLJSD_OK;  // the device status word that follows the count
  }
}

// Deterministic reduction of the per-row losses: each thread sums a fixed
// strided subset in double, then a fixed-order tree.
__global__ void k_reduce_loss(const float* loss_rows, int64_t bt, int64_t v, int reduction,
                              const int* n_valid, float* loss) {
  __shared__ double sh[1024];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < bt; i += blockDim.x) s += (double)loss_rows[i];
  sh[threadIdx.x] = s;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int n = *n_valid;
    double r = sh[0];
    if (n == 0) r = 0.0;
    else if (reduction == FLJSD_RED_BATCHMEAN) r /= (double)n;
    else if (reduction == FLJSD_RED_MEAN) r /= (double)n * (double)v;
    *loss = (float)r;
  }
}

template <typename T>
__global__ void k_scale(T* p, int64_t n, const float* gp) {
  const float g = *gp;
  if (g == 1.f) return;
  using V = Vec<T>;
  constexpr int N = V::N;
  const int64_t nvec = n / N;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec; i += stride) {
    float x[N];
    V::load(p + i * N, x);
#pragma unroll
    for (int k = 0; k < N; ++k) x[k] *= g;
    V::store(p + i * N, x);
  }
  for (int64_t j = nvec * N + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n; j += stride)
    V::put(p + j, V::one(p + j) * g);
}

template <typename T, int BRANCH>
cudaError_t launch_rows_t(JsdRowArgs a, cudaStream_t st) {
  // One row in flight per SM keeps the rows between pass 2 and pass 3 small
  // enough for L2 (152 rows of 2 x 256 KB at V = 128256 in bf16).
  const int64_t grid = a.rows < (int64_t)num_sms() ? a.rows : (int64_t)num_sms();
  size_t smem = 0;
  a.cache_vec = 0;
  if (BRANCH == 2 && sizeof(T) == 2) {
    // up to 224 KB of fp16 X - log M per row (14336 vectors of 8 elements; 200 KB
    // measured 3% slower at V = 128256, where it covers 80% of a row, not 89%)
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(k_jsd_rows<T, BRANCH>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kCacheVecMax * 16);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    const int64_t nvec = a.v / 8;
    a.cache_vec = nvec < kCacheVecMax ? nvec : kCacheVecMax;
    // FLJSD_ROWS_CACHE=0 recomputes every element in pass 3 instead
    if (const char* env = getenv("FLJSD_ROWS_CACHE"))
      if (env[0] == '0') a.cache_vec = 0;
    smem = (size_t)a.cache_vec * 16;
  }
  // FLJSD_ROWS_PREFETCH=0 turns pass 2's L2 prefetch off
  a.rows_prefetch = 1;
  if (const char* env = getenv("FLJSD_ROWS_PREFETCH"))
    if (env[0] == '0') a.rows_prefetch = 0;
  k_jsd_rows<T, BRANCH><<<(unsigned)grid, kRowThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_rows_dt(const JsdRowArgs& a, cudaStream_t st) {
  if (a.beta == 0.f) return launch_rows_t<T, 0>(a, st);
  if (a.beta == 1.f) return launch_rows_t<T, 1>(a, st);
  return launch_rows_t<T, 2>(a, st);
}

}  // namespace

cudaError_t launch_jsd_rows(int dtype, const JsdRowArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  trace_begin(FLJSD_KERNEL_JSD_ROWS, st);
  cudaError_t e = dtype == FLJSD_BF16 ? launch_rows_dt<__nv_bfloat16>(a, st)
                                      : launch_rows_dt<float>(a, st);
  trace_end(FLJSD_KERNEL_JSD_ROWS, st);
  return e;
}

cudaError_t launch_count_valid(const int64_t* labels, int64_t bt, int64_t ignore_index,
                               int* n_valid, cudaStream_t st) {
  trace_begin(FLJSD_KERNEL_SMALL, st);
  k_count_valid<<<1, 1024, 0, st>>>(labels, bt, ignore_index, n_valid);
  trace_end(FLJSD_KERNEL_SMALL, st);
  return cudaGetLastError();
}

cudaError_t launch_reduce_loss(const float* loss_rows, int64_t bt, int64_t v, int reduction,
                               const int* n_valid, float* loss, cudaStream_t st) {
  trace_begin(FLJSD_KERNEL_SMALL, st);
  k_reduce_loss<<<1, 1024, 0, st>>>(loss_rows, bt, v, reduction, n_valid, loss);
  trace_end(FLJSD_KERNEL_SMALL, st);
  return cudaGetLastError();
}

cudaError_t launch_scale(int dtype, void* p, int64_t n, const float* g, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  trace_begin(FLJSD_KERNEL_SMALL, st);
  const unsigned grid = (unsigned)num_sms() * 4;
  if (dtype == FLJSD_BF16)
    k_scale<__nv_bfloat16><<<grid, 256, 0, st>>>(reinterpret_cast<__nv_bfloat16*>(p), n, g);
  else
    k_scale<float><<<grid, 256, 0, st>>>(reinterpret_cast<float*>(p), n, g);
  trace_end(FLJSD_KERNEL_SMALL, st);
  return cudaGetLastError();
}

}  // namespace fljsd
