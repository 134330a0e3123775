// Element arithmetic shared by the row kernels: the ex2/lg2 units, 16-byte
// vector loads, and the per-element terms of the JSD branches in log2 units.
// See rows.cu and dist_rows.cu for the passes that use them.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace fljsd {
namespace rowmath {

// ---- hardware transcendental units (hand-written PTX) ----------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- vector loads of 16 bytes ------------------------------------------------
template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void load(const float* p, float (&o)[4]) {
    float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  __device__ static void store(float* p, const float (&o)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
  __device__ static float one(const float* p) { return *p; }
  __device__ static void put(float* p, float x) { *p = x; }
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&o)[8]) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ static float one(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ static void put(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
};

// ---- per-element branch arithmetic (log2 units) -----------------------------
// The callers form X2 = fma(z_s, c, -m_a) - log2 d_a and Y2 likewise, and
// d = X2 - Y2: equal student and teacher rows give d == 0 exactly, which is
// what the tie rule tests.
// Inputs per element: Y2 = log2 P (teacher) and d = X2 - Y2 = log2(Q / P),
// X2 = log2 Q (student). The generalized branch works from the larger of the
// two probabilities, big = 2^max(X2, Y2), and the ratio e = 2^-|d| <= 1:
//   small = big * e,  M / big = w1 * e + w0  (w1, w0 = 1-beta, beta when
//   d <= 0, else beta, 1-beta),  lg = log2(M / big),
//   X2 - log2 M = min(d, 0) - lg,  Y2 - log2 M = -max(d, 0) - lg.
// Nothing overflows for any d, P and Q come out consistent, and when P and Q
// are close the log term is computed from their ratio, not from two rounded
// absolute values. BRANCH 0: forward KL(P||Q); 1: reverse KL(Q||P);
// 2: generalized JSD. PREC selects the accurate library exp2f/log2f (fp32
// inputs) instead of the ex2/lg2 units (bf16 inputs).
template <bool PREC>
__device__ __forceinline__ float pexp2(float x) {
  if (PREC) return exp2f(x);
  return ex2(x);
}
template <bool PREC>
__device__ __forceinline__ float plog2(float x) {
  if (PREC) return log2f(x);
  return lg2(x);
}

// Generalized-branch terms of one element: Q, P*beta, and the two log ratios.
template <bool PREC>
__device__ __forceinline__ void gen_terms(float Y2, float d, float beta, float omb, float& Q,
                                          float& bP, float& xm, float& ym) {
  const bool neg = d <= 0.f;
  const float e = pexp2<PREC>(-fabsf(d));
  const float big = pexp2<PREC>(Y2 + fmaxf(d, 0.f));
  const float small = big * e;
  const float lg = plog2<PREC>(fmaf(neg ? omb : beta, e, neg ? beta : omb));
  Q = neg ? small : big;
  bP = beta * (neg ? big : small);
  xm = fminf(d, 0.f) - lg;
  ym = -fmaxf(d, 0.f) - lg;
}

// Generalized-branch terms, direct form (bf16 inputs): P = 2^Y2, Q = 2^X2 and
// log2 M from their mixture. Both probabilities are <= 1, so nothing
// overflows; M is clamped to the smallest normal float so that rows whose P
// and Q both underflow give finite (zero-weighted) log terms. Cheaper than the
// ratio form, and accurate well inside the bf16 tolerances.
__device__ __forceinline__ void gen_terms_direct(float Y2, float d, float beta, float omb,
                                                 float& Q, float& bP, float& xm, float& ym) {
  const float X2 = Y2 + d;
  Q = ex2(X2);
  const float P = ex2(Y2);
  bP = beta * P;
  const float lM = lg2(fmaxf(fmaf(omb, Q, bP), 1.17549435e-38f));
  xm = X2 - lM;
  ym = Y2 - lM;
}

// Per-element loss (log2 units, loss / ln 2) and, for the generalized branch,
// the log-prob gradient dX (also / ln 2). A tie (d == 0) contributes exactly 0.
template <int BRANCH, bool PREC>
__device__ __forceinline__ void elem_loss(float Y2, float d, float beta, float omb,
                                          float& ell, float& g) {
  if (BRANCH == 0) {
    ell = -pexp2<PREC>(Y2) * d;  // P (Y - X)
    g = 0.f;
  } else if (BRANCH == 1) {
    ell = pexp2<PREC>(Y2 + d) * d;  // Q (X - Y)
    g = 0.f;
  } else {
    float Q, bP, xm, ym;
    if (PREC)
      gen_terms<PREC>(Y2, d, beta, omb, Q, bP, xm, ym);
    else
      gen_terms_direct(Y2, d, beta, omb, Q, bP, xm, ym);
    g = omb * Q * xm;
    ell = fmaf(bP, ym, g);
  }
  if (d == 0.f) {
    ell = 0.f;
    g = 0.f;
  }
}

// dlogit of one element before the row scale w_r / T (natural-log units).
// L2 and S2 are the row loss and dX_sum in log2 units.
template <int BRANCH, bool PREC>
__device__ __forceinline__ float elem_grad(float Y2, float d, float beta, float omb, float L2,
                                           float S2) {
  const float ln2 = 0.6931471805599453f;
  if (BRANCH == 0) {
    if (d == 0.f) return 0.f;
    return pexp2<PREC>(Y2 + d) - pexp2<PREC>(Y2);  // Q - P
  } else if (BRANCH == 1) {
    return pexp2<PREC>(Y2 + d) * (ln2 * (d - L2));  // Q (X - Y - L)
  } else {
    float Q, bP, xm, ym;
    if (PREC)
      gen_terms<PREC>(Y2, d, beta, omb, Q, bP, xm, ym);
    else
      gen_terms_direct(Y2, d, beta, omb, Q, bP, xm, ym);
    const float g = (d == 0.f) ? 0.f : omb * Q * xm;
    return ln2 * fmaf(-Q, S2, g);
  }
}

}  // namespace rowmath
}  // namespace fljsd
