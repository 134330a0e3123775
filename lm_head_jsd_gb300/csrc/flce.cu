// Fused linear cross-entropy (FLCE): the lm_head GEMM, cross-entropy over the
// vocabulary, and both gradients, on the same tensor-core GEMMs, chunk planner
// and grad_weight epilogue as the fused-linear JSD.
//
// The grad_weight contract follows "perf(flce): write the weight-gradient
// product directly into grad_weight" (Liger-Kernel PR 1429), "Summary" and
// "Changes": the product goes straight into grad_weight, the first chunk
// overwrites, the outputs may be uninitialised. The per-row math is the
// standard softmax cross-entropy with the options that page's test list names
// (label smoothing, z-loss, softcap, reduction none):
//   c_j = softcap ? cap * tanh(z_j / cap) : z_j,  lse = log sum_j e^{c_j},
//   L = lse - (1 - eps) c_y - (eps / V) sum_j c_j + lambda lse^2,
//   dL/dc_j = softmax_j (1 + 2 lambda lse) - (1 - eps) [j == y] - eps / V,
//   dL/dz_j = dL/dc_j (1 - (c_j / cap)^2) with softcap.
// Rows whose label is ignore_index contribute 0; labels outside [0, V) are
// treated the same way and flagged in the workspace status word.
#include "internal.cuh"
#include "gemm_tc.cuh"
#include "jsd_math.cuh"

#include <cmath>

namespace fljsd {
namespace {

using namespace rowmath;

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
// vectors each thread loads before it stores in the lean pass 2 (bytes in flight)
constexpr int kCeUnroll = 2;
constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct CeRowArgs {
  void* z;  // [rows x ld] logits in, dlogits out
  int64_t ld, v, rows, row0;
  const int64_t* labels;
  int64_t ignore_index;
  const int* n_valid;
  int* status;
  float* loss_rows;
  const float2* stats;  // [rows x ntiles] partials of z * log2(e), or null
  int64_t ntiles;
  int reduction;
  float eps, lambda, cap, inv_cap;
};

struct MD {
  float m, d;
};
__device__ __forceinline__ MD md_combine(MD a, MD b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return MD{m, 0.f};
  return MD{m, (a.m == -INFINITY ? 0.f : a.d * ex2(a.m - m)) +
                   (b.m == -INFINITY ? 0.f : b.d * ex2(b.m - m))};
}

// Block-wide (m, d) and sum in a fixed order (deterministic): inside each
// warp, then over the per-warp results in warp 0, whose total every thread
// reads from the slot after theirs (shm, shs hold kWarps + 1). In a warp: the
// largest m in one instruction (exact, so order-free), every lane's d
// rescaled to it, and d and s summed in a fixed butterfly order.
__device__ __forceinline__ void warp_md_sum(MD& v, float& s) {
  float m;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(v.m));
  float2 ds = make_float2(m == -INFINITY ? 0.f : v.d * ex2(v.m - m), s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    ds = __fadd2_rn(ds, make_float2(__shfl_xor_sync(0xffffffffu, ds.x, o),
                                    __shfl_xor_sync(0xffffffffu, ds.y, o)));
  v = MD{m, ds.x};
  s = ds.y;
}
__device__ __forceinline__ void block_md2(MD& v, float& s, MD* shm, float* shs) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_md_sum(v, s);
  if (lane == 0) {
    shm[warp] = v;
    shs[warp] = s;
  }
  __syncthreads();
  if (warp == 0) {
    MD u = lane < kWarps ? shm[lane] : MD{-INFINITY, 0.f};
    float t = lane < kWarps ? shs[lane] : 0.f;
    warp_md_sum(u, t);
    if (lane == 0) {
      shm[kWarps] = u;
      shs[kWarps] = t;
    }
  }
  __syncthreads();
  v = shm[kWarps];
  s = shs[kWarps];
}

// Eight bf16 (one 16-byte load) to fp32: exact, a shift into the high half.
__device__ __forceinline__ void unpack_bf16x8(uint4 v, float (&o)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Bulk prefetch of the 16-byte units wholly inside [p, p + bytes) into L2.
__device__ __forceinline__ void l2_prefetch_span(const void* p, size_t bytes) {
  const uintptr_t b = ((uintptr_t)p + 15u) & ~(uintptr_t)15u;
  const uintptr_t e = ((uintptr_t)p + bytes) & ~(uintptr_t)15u;
  if (e > b)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(b), "r"((uint32_t)(e - b))
                 : "memory");
}

// capped logit c = cap * tanh(z / cap), with t = tanh(z / cap) returned for
// the derivative dc/dz = 1 - t^2 (inv_cap = 1 / cap, formed once on the host)
template <bool CAP>
__device__ __forceinline__ float capz(float z, float cap, float inv_cap, float* t = nullptr) {
  if (!CAP) return z;
  const float th = tanhf(z * inv_cap);
  if (t) *t = th;
  return cap * th;
}

template <typename T, bool CAP>
__global__ void __launch_bounds__(kThreads) k_ce_rows(CeRowArgs a) {
  using V = Vec<T>;
  constexpr int N = V::N;
  __shared__ MD shm[kWarps + 1];
  __shared__ float shs[kWarps + 1];
  const float L2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;
  const int n_valid = *a.n_valid;
  float w = 1.f;
  if (a.reduction == FLJSD_RED_MEAN || a.reduction == FLJSD_RED_BATCHMEAN)
    w = n_valid > 0 ? (float)(1.0 / (double)n_valid) : 0.f;
  const int64_t nvec = a.v / N, tail0 = nvec * N;
  const float eps_v = a.eps / (float)a.v;

  for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
    const int64_t grow = a.row0 + r;
    T* zr = reinterpret_cast<T*>(a.z) + r * a.ld;
    const int64_t y = a.labels[grow];
    bool valid = y != a.ignore_index;
    if (valid && (y < 0 || y >= a.v)) {
      valid = false;
      if (threadIdx.x == 0) atomicExch(a.status, (int)FLJSD_ERR_INVALID_ARG);
    }
    if (!valid) {
      float zero[N];
#pragma unroll
      for (int i = 0; i < N; ++i) zero[i] = 0.f;
      for (int64_t i = threadIdx.x; i < nvec; i += blockDim.x) V::store(zr + i * N, zero);
      for (int64_t j = tail0 + threadIdx.x; j < a.v; j += blockDim.x) V::put(zr + j, 0.f);
      if (threadIdx.x == 0) a.loss_rows[grow] = 0.f;
      continue;
    }
    const float cy = capz<CAP>(V::one(zr + y), a.cap, a.inv_cap);

    // ---- pass 1: (max, sum 2^(x - max)) of x = c * log2(e), and sum of c ----
    MD md{-INFINITY, 0.f};
    float csum = 0.f;
    const bool have_stats = (a.stats != nullptr) && !CAP;
    if (have_stats) {
      const float2* ps = a.stats + r * a.ntiles;
      if ((int64_t)threadIdx.x < a.ntiles) md = MD{ps[threadIdx.x].x, ps[threadIdx.x].y};
      for (int64_t i = threadIdx.x + blockDim.x; i < a.ntiles; i += blockDim.x)
        md = md_combine(md, MD{ps[i].x, ps[i].y});
    } else {
      for (int64_t i = threadIdx.x; i < nvec; i += blockDim.x) {
        float zs[N];
        V::load(zr + i * N, zs);
        float vm = -INFINITY;
#pragma unroll
        for (int k = 0; k < N; ++k) {
          zs[k] = capz<CAP>(zs[k], a.cap, a.inv_cap);
          csum += zs[k];
          vm = fmaxf(vm, __fmul_rn(zs[k], L2E));
        }
        if (vm > md.m) {
          md.d = (md.m == -INFINITY) ? 0.f : md.d * ex2(md.m - vm);
          md.m = vm;
        }
#pragma unroll
        for (int k = 0; k < N; ++k) md.d += ex2(__fmaf_rn(zs[k], L2E, -md.m));
      }
      for (int64_t j = tail0 + threadIdx.x; j < a.v; j += blockDim.x) {
        const float c = capz<CAP>(V::one(zr + j), a.cap, a.inv_cap);
        csum += c;
        const float x = __fmul_rn(c, L2E);
        if (x > md.m) {
          md.d = (md.m == -INFINITY) ? 0.f : md.d * ex2(md.m - x);
          md.m = x;
        }
        md.d += ex2(__fmaf_rn(c, L2E, -md.m));
      }
    }
    block_md2(md, csum, shm, shs);
    const float m = md.m, ld2 = lg2(md.d);
    const float lse = LN2 * (m + ld2);
    const float gsm = 1.f + 2.f * a.lambda * lse;  // softmax coefficient with the z-loss
    const float onehot = 1.f - a.eps;

    // ---- pass 2: dlogits in place (and the sum of c when pass 1 was folded) ----
    float csum2 = 0.f;
    if constexpr (!CAP && sizeof(T) == 2) {
      // bf16 without a cap: kCeUnroll vectors per iteration with bulk L2
      // prefetches three iterations ahead; the label's element is corrected once, by the
      // thread whose vector holds it; the sum of c only where label smoothing
      // needs it; packed fp32x2 arithmetic (each lane rounds as the scalar form)
      const int step = (int)blockDim.x, nv = (int)nvec, chunk = kCeUnroll * step;
      const bool need_sum = have_stats && a.eps != 0.f;
      const int yv = (int)(y / N), yk = (int)(y % N);
      const float2 l2e2 = make_float2(L2E, L2E), nm2 = make_float2(-m, -m);
      const float2 nld2 = make_float2(-ld2, -ld2), gsm2 = make_float2(gsm, gsm);
      const float2 neps2 = make_float2(-eps_v, -eps_v), w2 = make_float2(w, w);
      if (threadIdx.x == 0)
        l2_prefetch_span(zr, (size_t)(nv < 3 * chunk ? nv : 3 * chunk) * N * sizeof(T));
      auto vec = [&](float (&zs)[N]) {
#pragma unroll
        for (int k = 0; k < N; k += 2) {
          const float2 c = make_float2(zs[k], zs[k + 1]);
          if (need_sum) csum2 += c.x + c.y;
          const float2 x = __fadd2_rn(__ffma2_rn(c, l2e2, nm2), nld2);
          const float2 dc = __ffma2_rn(make_float2(ex2(x.x), ex2(x.y)), gsm2, neps2);
          const float2 g = __fmul2_rn(dc, w2);
          zs[k] = g.x;
          zs[k + 1] = g.y;
        }
      };
      // element yk of a vector, read and written with compile-time indices (a
      // runtime index would put the vector in local memory)
      auto pick = [&](const float (&zs)[N]) {
        float r = zs[0];
#pragma unroll
        for (int k = 1; k < N; ++k) r = k == yk ? zs[k] : r;
        return r;
      };
      auto put = [&](float (&zs)[N], float val) {
#pragma unroll
        for (int k = 0; k < N; ++k) zs[k] = k == yk ? val : zs[k];
      };
      // the label's element gets dc - (1 - eps), from its logit as loaded
      auto label_dz = [&](float z) {
        return (fmaf(ex2(__fmaf_rn(z, L2E, -m) - ld2), gsm, -eps_v) - onehot) * w;
      };
      int i = (int)threadIdx.x;
      for (; i + (kCeUnroll - 1) * step < nv; i += kCeUnroll * step) {
        if (threadIdx.x == 0 && i + 3 * chunk < nv)
          l2_prefetch_span(zr + (int64_t)(i + 3 * chunk) * N,
                           (size_t)(nv - (i + 3 * chunk) < chunk ? nv - (i + 3 * chunk) : chunk) *
                               N * sizeof(T));
        uint4 raw[kCeUnroll];  // packed bf16: 4 registers a vector in flight
#pragma unroll
        for (int u = 0; u < kCeUnroll; ++u)
          raw[u] = *reinterpret_cast<const uint4*>(zr + (int64_t)(i + u * step) * N);
#pragma unroll
        for (int u = 0; u < kCeUnroll; ++u) {
          float zs[N];
          unpack_bf16x8(raw[u], zs);
          const float yl = pick(zs);
          vec(zs);
          if (i + u * step == yv) put(zs, label_dz(yl));
          V::store(zr + (int64_t)(i + u * step) * N, zs);
        }
      }
      for (; i < nv; i += step) {
        float z0[N];
        V::load(zr + (int64_t)i * N, z0);
        const float y0 = pick(z0);
        vec(z0);
        if (i == yv) put(z0, label_dz(y0));
        V::store(zr + (int64_t)i * N, z0);
      }
    } else
    for (int64_t i = threadIdx.x; i < nvec; i += blockDim.x) {
      float zs[N];
      V::load(zr + i * N, zs);
#pragma unroll
      for (int k = 0; k < N; ++k) {
        float t = 0.f;
        const float c = capz<CAP>(zs[k], a.cap, a.inv_cap, &t);
        csum2 += c;
        const float p = ex2(__fmaf_rn(c, L2E, -m) - ld2);
        float dc = fmaf(p, gsm, -eps_v);
        if (i * N + k == y) dc -= onehot;
        if (CAP) dc *= fmaf(-t, t, 1.f);
        zs[k] = dc * w;
      }
      V::store(zr + i * N, zs);
    }
    for (int64_t j = tail0 + threadIdx.x; j < a.v; j += blockDim.x) {
      float t = 0.f;
      const float c = capz<CAP>(V::one(zr + j), a.cap, a.inv_cap, &t);
      csum2 += c;
      const float p = ex2(__fmaf_rn(c, L2E, -m) - ld2);
      float dc = fmaf(p, gsm, -eps_v);
      if (j == y) dc -= onehot;
      if (CAP) dc *= fmaf(-t, t, 1.f);
      V::put(zr + j, dc * w);
    }
    if (have_stats && a.eps != 0.f) {
      MD dummy{0.f, 0.f};
      block_md2(dummy, csum2, shm, shs);
      csum = csum2;
    }
    if (threadIdx.x == 0)
      a.loss_rows[grow] = lse - onehot * cy - eps_v * csum + a.lambda * lse * lse;
    // no barrier here: the reduction slots a row reads (shm / shs[kWarps]) are
    // written again only after the next row's first barrier
  }
}

template <typename T>
cudaError_t launch_ce_rows_t(const CeRowArgs& a, cudaStream_t st) {
  const int64_t grid = a.rows < (int64_t)num_sms() ? a.rows : (int64_t)num_sms();
  if (a.cap > 0.f)
    k_ce_rows<T, true><<<(unsigned)grid, kThreads, 0, st>>>(a);
  else
    k_ce_rows<T, false><<<(unsigned)grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

inline size_t dsize(int dt) { return dt == FLJSD_BF16 ? 2 : 4; }
inline bool aligned16(const void* q) { return ((uintptr_t)q & 15u) == 0; }

struct CeLayout {
  int64_t ld, ntiles;
  size_t z, stats, loss_rows, misc, acc32, splitk, splitk_bytes, total, logits_bytes, stats_bytes;
  bool use_acc32;
};

CeLayout ce_layout(const fljsd_ce_problem& p, int64_t c) {
  CeLayout L{};
  L.ld = (p.v + 7) / 8 * 8;
  L.ntiles = (p.v + TC_STATS_COLS - 1) / TC_STATS_COLS;
  const size_t zb = align_up((size_t)c * (size_t)L.ld * dsize(p.dtype));
  const size_t sb = align_up((size_t)c * (size_t)L.ntiles * sizeof(float2));
  L.z = 0;
  L.stats = zb;
  L.loss_rows = zb + sb;
  L.misc = L.loss_rows + align_up((size_t)p.bt * sizeof(float));
  L.use_acc32 = (p.flags & FLJSD_FLAG_ACCUM_FP32) && p.dtype == FLJSD_BF16 && c < p.bt;
  L.acc32 = L.misc + kAlign;
  L.splitk = L.acc32 + (L.use_acc32 ? align_up((size_t)p.v * (size_t)p.h * sizeof(float)) : 0);
  // fp32 partials of a split grad_input contraction (chunks with few tiles)
  L.splitk_bytes = p.dtype == FLJSD_BF16 && c > 0 ? align_up(tc_splitk_bytes(c, p.h, p.v, TC_PLAN_CTAS)) : 0;
  L.total = L.splitk + L.splitk_bytes;
  L.logits_bytes = (size_t)c * (size_t)L.ld * dsize(p.dtype);
  L.stats_bytes = sb + align_up((size_t)p.bt * sizeof(float)) + kAlign;
  return L;
}

fljsd_status ce_check(const fljsd_ce_problem* p) {
  if (!p) return FLJSD_ERR_INVALID_ARG;
  if (p->bt <= 0 || p->h <= 0 || p->v <= 0 || p->chunk_rows < 0) return FLJSD_ERR_INVALID_ARG;
  if (p->dtype != FLJSD_F32 && p->dtype != FLJSD_BF16) return FLJSD_ERR_INVALID_ARG;
  if (p->reduction < FLJSD_RED_NONE || p->reduction > FLJSD_RED_BATCHMEAN)
    return FLJSD_ERR_INVALID_ARG;
  if (!(p->label_smoothing >= 0.f && p->label_smoothing <= 1.f)) return FLJSD_ERR_INVALID_ARG;
  if (!(p->lse_square_scale >= 0.f) || !std::isfinite(p->lse_square_scale))
    return FLJSD_ERR_INVALID_ARG;
  if (!(p->softcap >= 0.f) || !std::isfinite(p->softcap)) return FLJSD_ERR_INVALID_ARG;
  if ((p->flags & ~FLJSD_FLAG_ACCUM_FP32) != 0) return FLJSD_ERR_INVALID_ARG;
  if (p->v > (int64_t)1 << 30 || p->bt > (int64_t)1 << 30 || p->h > (int64_t)1 << 20)
    return FLJSD_ERR_UNSUPPORTED;
  return FLJSD_OK;
}

// One contraction on the tensor cores when the strides allow TMA, else on the
// CUDA cores (same helper shape as the JSD path's).
cudaError_t ce_gemm(int dtype, int kind, const void* a, int64_t lda, int a_mn, const void* b,
                    int64_t ldb, int b_mn, void* d, int64_t ldd, int64_t m, int64_t n, int64_t k,
                    int accumulate, int raster_n_fastest, int* status, cudaStream_t st,
                    float2* stats, float stats_scale, bool* stats_done, float* d32,
                    int finalize, void* splitk_ws = nullptr,
                    size_t splitk_bytes = 0) {
  if (stats_done) *stats_done = false;
  if (m <= 0 || n <= 0) return cudaSuccess;
  cudaError_t e;
  trace_begin(kind, st);
  TcGemmArgs t{a,      lda,   a_mn,        b,   ldb,     b_mn, d, ldd, m, n, k, accumulate,
               raster_n_fastest, status, stats, stats_scale, d32, finalize};
  t.splitk_ws = static_cast<float*>(splitk_ws);
  t.splitk_ws_bytes = splitk_bytes;
  if (dtype == FLJSD_BF16 && tc_gemm_supported(t)) {
    e = launch_gemm_tc(t, st);
    if (stats_done) *stats_done = stats != nullptr;
  } else {
    GemmArgs g{};
    g.a = a; g.sam = a_mn ? 1 : lda; g.sak = a_mn ? lda : 1;
    g.b = b; g.sbn = b_mn ? 1 : ldb; g.sbk = b_mn ? ldb : 1;
    g.c = d; g.ldc = ldd; g.m = m; g.n = n; g.k = k; g.accumulate = accumulate;
    g.c32 = d32; g.finalize = finalize;
    e = launch_gemm_simt(dtype, g, st);
  }
  trace_end(kind, st);
  return e;
}

}  // namespace
}  // namespace fljsd

using namespace fljsd;

extern "C" {

fljsd_status fljsd_ce_plan(const fljsd_ce_problem* p, size_t free_hbm_bytes, fljsd_plan_t* out) {
  fljsd_status st = ce_check(p);
  if (st != FLJSD_OK) return st;
  if (!out) return FLJSD_ERR_INVALID_ARG;
  int64_t c;
  if (p->chunk_rows > 0) {
    c = p->chunk_rows < p->bt ? p->chunk_rows : p->bt;
  } else if (free_hbm_bytes == 0) {
    c = p->bt;
  } else {
    const size_t budget = free_hbm_bytes / 2;
    if (ce_layout(*p, p->bt).total <= budget) {
      c = p->bt;
    } else {
      // per-row growth without the split-K scratch (which shrinks as chunks grow)
      const CeLayout l0 = ce_layout(*p, 0), l1 = ce_layout(*p, 1);
      const size_t fixed = l0.total;
      const size_t per_row = (l1.total - l1.splitk_bytes) - (l0.total - l0.splitk_bytes);
      if (budget < fixed + per_row) return FLJSD_ERR_WORKSPACE;
      c = (int64_t)((budget - fixed) / (per_row ? per_row : 1));
      if (c >= 128) c = c / 128 * 128;
      while (c > 0 && ce_layout(*p, c).total > budget) c -= (c > 128 ? 128 : 1);
      if (c <= 0) return FLJSD_ERR_WORKSPACE;
    }
  }
  const CeLayout L = ce_layout(*p, c);
  out->chunk_rows = c;
  out->num_chunks = (p->bt + c - 1) / c;
  out->ld = L.ld;
  out->workspace_bytes = L.total;
  out->logits_bytes = L.logits_bytes;
  out->stats_bytes = L.stats_bytes;
  out->status_offset = L.misc + sizeof(int);
  return FLJSD_OK;
}

fljsd_status fljsd_ce_forward(const fljsd_ce_problem* p, const fljsd_plan_t* plan,
                              const void* x, const void* w, const int64_t* labels, float* loss,
                              void* grad_input, void* grad_weight, void* workspace,
                              size_t workspace_bytes, fljsd_stream_t stream_) {
  fljsd_status st = ce_check(p);
  if (st != FLJSD_OK) return st;
  if (!plan || !x || !w || !labels || !loss || !grad_input || !grad_weight || !workspace)
    return FLJSD_ERR_INVALID_ARG;
  const void* ptrs[] = {x, w, labels, grad_input, grad_weight, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return FLJSD_ERR_INVALID_ARG;
  if ((uintptr_t)loss & 3u) return FLJSD_ERR_INVALID_ARG;
  const int64_t c = plan->chunk_rows;
  if (c <= 0 || c > p->bt) return FLJSD_ERR_INVALID_ARG;
  const CeLayout L = ce_layout(*p, c);
  if (plan->ld != L.ld || plan->workspace_bytes != L.total ||
      plan->num_chunks != (p->bt + c - 1) / c)
    return FLJSD_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return FLJSD_ERR_WORKSPACE;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  char* ws = static_cast<char*>(workspace);
  void* z = ws + L.z;
  float2* stats = reinterpret_cast<float2*>(ws + L.stats);
  float* loss_rows = p->reduction == FLJSD_RED_NONE ? loss : reinterpret_cast<float*>(ws + L.loss_rows);
  int* n_valid = reinterpret_cast<int*>(ws + L.misc);
  int* status = n_valid + 1;
  float* acc32 = reinterpret_cast<float*>(ws + L.acc32);
  const size_t s = dsize(p->dtype);
  const float l2e = 1.4426950408889634f;

  if (launch_count_valid(labels, p->bt, p->ignore_index, n_valid, stream) != cudaSuccess)
    return FLJSD_ERR_CUDA;
  cudaError_t e;
  for (int64_t chunk = 0; chunk * c < p->bt; ++chunk) {
    const int64_t r0 = chunk * c;
    const int64_t rows = (p->bt - r0) < c ? (p->bt - r0) : c;
    const char* xc = static_cast<const char*>(x) + (size_t)r0 * p->h * s;
    bool st_done = false;
    // logits with the pass-1 partials of z * log2(e) (unused under softcap)
    e = ce_gemm(p->dtype, FLJSD_KERNEL_GEMM_LOGITS, xc, p->h, 0, w, p->h, 0, z, L.ld, rows, p->v,
                p->h, 0, 0, status, stream, p->softcap > 0.f ? nullptr : stats, l2e, &st_done,
                nullptr, 0);
    if (e != cudaSuccess) return FLJSD_ERR_CUDA;
    CeRowArgs ra{};
    ra.z = z; ra.ld = L.ld; ra.v = p->v; ra.rows = rows; ra.row0 = r0;
    ra.labels = labels; ra.ignore_index = p->ignore_index; ra.n_valid = n_valid;
    ra.status = status; ra.loss_rows = loss_rows; ra.stats = st_done ? stats : nullptr;
    ra.ntiles = L.ntiles; ra.reduction = p->reduction; ra.eps = p->label_smoothing;
    ra.lambda = p->lse_square_scale; ra.cap = p->softcap;
    ra.inv_cap = p->softcap > 0.f ? (float)(1.0 / (double)p->softcap) : 0.f;
    trace_begin(FLJSD_KERNEL_JSD_ROWS, stream);
    e = p->dtype == FLJSD_BF16 ? launch_ce_rows_t<__nv_bfloat16>(ra, stream)
                               : launch_ce_rows_t<float>(ra, stream);
    trace_end(FLJSD_KERNEL_JSD_ROWS, stream);
    if (e != cudaSuccess) return FLJSD_ERR_CUDA;
    e = ce_gemm(p->dtype, FLJSD_KERNEL_GEMM_GRAD_INPUT, z, L.ld, 0, w, p->h, 1,
                static_cast<char*>(grad_input) + (size_t)r0 * p->h * s, p->h, rows, p->h, p->v,
                0, 1, status, stream, nullptr, 0.f, nullptr, nullptr, 0, ws + L.splitk,
                L.splitk_bytes);
    if (e != cudaSuccess) return FLJSD_ERR_CUDA;
    const bool last = r0 + rows >= p->bt;
    e = ce_gemm(p->dtype, FLJSD_KERNEL_GEMM_GRAD_WEIGHT, z, L.ld, 1, xc, p->h, 1, grad_weight,
                p->h, p->v, p->h, rows, chunk > 0 ? 1 : 0, 1, status, stream, nullptr, 0.f,
                nullptr, L.use_acc32 ? acc32 : nullptr, (L.use_acc32 && last) ? 1 : 0);
    if (e != cudaSuccess) return FLJSD_ERR_CUDA;
  }
  if (p->reduction != FLJSD_RED_NONE) {
    // mean and batchmean divide by the valid-token count; sum does not
    const int red = p->reduction == FLJSD_RED_SUM ? FLJSD_RED_SUM : FLJSD_RED_BATCHMEAN;
    if (launch_reduce_loss(loss_rows, p->bt, p->v, red, n_valid, loss, stream) != cudaSuccess)
      return FLJSD_ERR_CUDA;
  }
  return FLJSD_OK;
}

}  // extern "C"
