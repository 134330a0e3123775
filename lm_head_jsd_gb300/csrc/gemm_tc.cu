// Tensor-core GEMM, host side: operand tensor maps, the schedule choice (CTA
// pairs, tile order, split-K, stored-output prefetch, staging, epilogue
// groups) and the split-K reduction. The kernel and its design notes are in
// gemm_tc_kernel.cuh.
#include "gemm_tc_kernel.cuh"

#include <cstdlib>
#include <mutex>

namespace fljsd {
namespace {

using namespace tcgemm;

// D[r, c] = round(sum over s of partial[s][r][c]), s in increasing order.
__global__ void k_splitk_reduce(const float* __restrict__ part, int splits, int64_t m, int64_t n,
                                int64_t ldd, __nv_bfloat16* __restrict__ D) {
  const int64_t n8 = n / 8;
  const int64_t total = m * n8;
  const int64_t plane = m * ldd;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / n8, c = (i - r * n8) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < splits; ++s) {
      const float4* src = reinterpret_cast<const float4*>(part + s * plane + r * ldd + c);
      const float4 a = src[0], b = src[1];
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    *reinterpret_cast<uint4*>(D + r * ldd + c) =
        make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]),
                   pack_bf16(acc[4], acc[5]), pack_bf16(acc[6], acc[7]));
  }
  // columns past the last multiple of 8
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < m * (n - n8 * 8);
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t w = n - n8 * 8;
    const int64_t r = i / w, c = n8 * 8 + (i - r * w);
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) acc += part[s * plane + r * ldd + c];
    D[r * ldd + c] = __float2bfloat16_rn(acc);
  }
}

// Split-K factor for a contraction with too few output tiles to fill the GPU
// (1 = no split); `ctas` is the number of CTAs to aim for.
int splitk_factor(int64_t m, int64_t n, int64_t k, int ctas) {
  const int64_t tiles = ((m + BM - 1) / BM) * ((n + BN - 1) / BN);
  const int64_t kblocks = (k + BK - 1) / BK;
  if (tiles * 2 > ctas || kblocks < 8) return 1;
  int64_t s = ctas / tiles;
  if (s > kblocks / 4) s = kblocks / 4;
  if (s > 16) s = 16;
  if (s < 2) return 1;
  const int64_t per = (kblocks + s - 1) / s;
  return (int)((kblocks + per - 1) / per);  // no empty split
}

// ---- host: tensor maps ------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D tensor map (bf16, or fp32 when f32) over a row-major [outer x inner]
// matrix with row stride ld elements; box = box_inner x box_outer; 128-byte
// swizzle; zero fill.
bool make_map(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int64_t ld,
              int box_inner, int box_outer, bool f32 = false) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * (f32 ? 4 : 2)};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// One launch in the layout of (a_mn, b_mn).
cudaError_t launch_layout(bool a_mn, bool b_mn, bool pair, const CUtensorMap& ma,
                          const CUtensorMap& mb, const CUtensorMap& mcm, const CUtensorMap& msm,
                          __nv_bfloat16* d, const KParams& p, cudaStream_t st) {
  if (!a_mn && !b_mn) return launch_kk(ma, mb, mcm, msm, d, p, pair, st);
  if (!a_mn && b_mn) return launch_kmn(ma, mb, mcm, msm, d, p, pair, st);
  if (a_mn && b_mn) return launch_mnmn(ma, mb, mcm, msm, d, p, pair, st);
  return launch_mnk(ma, mb, mcm, msm, d, p, pair, st);
}

}  // namespace

size_t tc_splitk_bytes(int64_t m, int64_t n, int64_t k, int ctas) {
  const int s = splitk_factor(m, n, k, ctas);
  if (s <= 1) return 0;
  const int64_t ldd = (n + 7) / 8 * 8;
  return (size_t)s * (size_t)m * (size_t)ldd * sizeof(float);
}

bool tc_gemm_supported(const TcGemmArgs& g) {
  auto al = [](const void* q) { return ((uintptr_t)q & 15u) == 0; };
  return g.m > 0 && g.n > 0 && g.k > 0 && al(g.a) && al(g.b) && al(g.d) && g.lda % 8 == 0 &&
         g.ldb % 8 == 0 && g.ldd % 8 == 0 && g.m < (1ll << 31) && g.n < (1ll << 31) &&
         g.k < (1ll << 31);
}

cudaError_t launch_gemm_tc(const TcGemmArgs& g, cudaStream_t st) {
  if (!tc_gemm_supported(g)) return cudaErrorInvalidValue;
  const int64_t mblocks = (g.m + BM - 1) / BM;
  // split-K (below) for outputs with too few tiles for the GPU; otherwise
  // pairs of m-blocks run as CTA pairs wherever there are two m-blocks to pair
  // and the contraction is at least 4 k-blocks deep (K >= 256): below that
  // the epilogue sets the pace and a pair's accumulator hand-offs cost more
  // than its halved B copies save (measured on the chunked grad_weight's
  // read-modify-write, grad_weight ms per headline step, pairs vs one CTA per
  // tile: K = 128 21.31 vs 20.66, K = 256 12.06 vs 13.75, K = 512 8.22 vs
  // 8.38). FLJSD_GEMM_PAIR=0 in the environment selects one CTA per tile for
  // every call, FLJSD_GEMM_PAIR=2 CTA pairs at any depth (both schedules
  // compute identical results).
  const char* senv = getenv("FLJSD_GEMM_SPLITK");
  const bool split_off = senv != nullptr && senv[0] == '0';
  int splits = 1;
  if (!split_off && g.splitk_ws != nullptr && !g.accumulate && g.d32 == nullptr &&
      g.stats == nullptr) {
    splits = splitk_factor(g.m, g.n, g.k, num_sms());
    while (splits > 1 &&
           (size_t)splits * (size_t)g.m * (size_t)g.ldd * sizeof(float) > g.splitk_ws_bytes)
      --splits;
  }
  const char* penv_pair = getenv("FLJSD_GEMM_PAIR");
  const bool pair_off = penv_pair != nullptr && penv_pair[0] == '0';
  const bool pair_any = penv_pair != nullptr && penv_pair[0] == '2';
  const bool deep = (g.k + BK - 1) / BK >= 4;
  // Waves of tiles over the GPU: pairs run ceil(mblocks / 2) 256-row tiles per
  // n-block on half as many clusters, so an odd m-block count leaves a pair
  // half empty and a small tile count can need one wave more. Pairs are kept
  // while their waves are at most 12% more than one CTA per tile needs (about
  // what a pair's halved B copies save per tile). Measured, ms per headline
  // step at 384 / 640 / 896 / 1152-row chunks, pairs vs one CTA: logits
  // 15.0 / 12.1 / 12.0 / 10.8 vs 13.1 / 11.7 / 11.5 / 11.6 (waves 14 / 20 / 27
  // / 33 vs 10 / 17 / 24 / 30); grad_input at 1152 rows 8.9 vs 5.4 (2 waves vs
  // 1), at 640 and 896 rows 7.9 and 6.1 vs 8.6 and 6.6 (1 wave each).
  const int64_t nblocks = (g.n + BN - 1) / BN;
  const int64_t sms = num_sms();
  const int64_t clusters = sms >= 2 ? sms / 2 : 1;
  const int64_t waves_one = (mblocks * nblocks + sms - 1) / sms;
  const int64_t waves_pair = ((mblocks + 1) / 2 * nblocks + clusters - 1) / clusters;
  const bool waves_ok = waves_pair * 100 <= waves_one * 112;
  const bool pair = mblocks >= 2 && splits <= 1 && !g.single_cta && !pair_off &&
                    ((deep && waves_ok) || pair_any);
  CUtensorMap ma, mb;
  bool ok;
  if (g.a_mn)  // A stored [k x m]
    ok = make_map(&ma, g.a, g.m, g.k, g.lda, 64, 64);
  else  // A stored [m x k]
    ok = make_map(&ma, g.a, g.k, g.m, g.lda, BK, BM);
  if (!ok) return cudaErrorInvalidValue;
  if (g.b_mn)  // B stored [k x n]
    ok = make_map(&mb, g.b, g.n, g.k, g.ldb, 64, 64);
  else  // B stored [n x k]; a CTA of a pair copies half the tile's rows
    ok = make_map(&mb, g.b, g.k, g.n, g.ldb, BK, pair ? BN / 2 : BN);
  if (!ok) return cudaErrorInvalidValue;
  KParams p{};
  p.m = g.m;
  p.n = g.n;
  p.k = g.k;
  p.ldd = g.ldd;
  p.num_m_blocks = (int)mblocks;
  p.num_n_blocks = (int)((g.n + BN - 1) / BN);
  p.num_k_blocks = (int)((g.k + BK - 1) / BK);
  const int64_t tiles = (int64_t)p.num_m_blocks * p.num_n_blocks;
  if (tiles > 0x7fffffff) return cudaErrorInvalidValue;
  p.num_tiles = (int)tiles;
  p.m_units = pair ? (p.num_m_blocks + 1) / 2 : p.num_m_blocks;
  p.num_units = p.m_units * p.num_n_blocks;
  p.raster = g.raster_n_fastest;
  {
    // band of A rows whose K extent stays around 32 MB (at least one unit);
    // FLJSD_GEMM_BAND_MB overrides the size. (Measured on the logits GEMM:
    // 16 MB bands read W four times, 32 MB bands twice and 3% faster.)
    int64_t band_bytes = 32ll << 20;
    if (const char* b = getenv("FLJSD_GEMM_BAND_MB")) {
      const long mbb = strtol(b, nullptr, 10);
      if (mbb > 0 && mbb <= 4096) band_bytes = (int64_t)mbb << 20;
    }
    const int64_t per_unit = (int64_t)BM * (pair ? 2 : 1) * g.k * 2;
    int64_t gm = per_unit > 0 ? band_bytes / per_unit : 1;
    if (gm < 1) gm = 1;
    if (gm > p.m_units) gm = p.m_units;
    p.group_m = (int)gm;
  }
  p.accumulate = g.accumulate;
  p.d32 = g.d32;
  p.finalize = g.finalize;
  p.timeout_ns = g.timeout_ns ? g.timeout_ns : kTimeoutNs;
  p.stall_producer = g.stall_producer;
  p.status = g.status;
  p.stats = g.stats;
  p.stats_scale = g.stats_scale;
  auto* d = reinterpret_cast<__nv_bfloat16*>(g.d);
  // split-K when the output has too few tiles for the GPU (plain stores
  // only); the partials go to the caller's scratch.
  // FLJSD_GEMM_SPLITK=0 in the environment turns it off.
  p.k_splits = 1;
  p.kb_per_split = p.num_k_blocks;
  p.partial = nullptr;
  if (splits > 1) {
    p.kb_per_split = (p.num_k_blocks + splits - 1) / splits;
    p.k_splits = (p.num_k_blocks + p.kb_per_split - 1) / p.kb_per_split;
    p.partial = g.splitk_ws;
    p.num_units = p.num_tiles * p.k_splits;
  }
  // stored-output prefetch for an accumulating epilogue (read-modify-write of
  // D, or of the fp32 side accumulator): fewer operand stages, a slab ring for
  // the old values. FLJSD_GEMM_PREFETCH=0 in the environment turns it off.
  // operand stages: 4 of 48 KB on one CTA, 6 of 32 KB in a pair (192 KB)
  p.nst = pair ? 6 : 4;
  p.nslab = 0;
  p.slab_cols = 64;
  p.cps = 2;
  p.slab_store = 0;
  p.slab_f32 = 0;
  p.stage_out = 0;
  p.nbuf = 0;
  CUtensorMap mcm = ma, msm = ma;  // unused unless nslab > 0
  const bool rmw = (g.accumulate && g.d32 == nullptr) ||
                   (g.d32 != nullptr && (g.accumulate || g.finalize));
  const char* penv = getenv("FLJSD_GEMM_PREFETCH");
  const bool pf_off = penv != nullptr && penv[0] == '0';
  bool two_groups = false;  // a second epilogue group chosen with the slab ring
  if (rmw && p.k_splits == 1 && !pf_off) {
    const bool f32 = g.d32 != nullptr;
    const void* src = f32 ? (const void*)g.d32 : g.d;
    if (((uintptr_t)src & 15u) == 0) {
      p.slab_cols = f32 ? 32 : 64;
      p.cps = p.slab_cols / 32;
      // the new values go back through the slab unless they change type
      // (fp32 accumulator in, bf16 result out) or the row length is not a
      // whole number of 16-byte units (measured: the store then also writes
      // the padding up to the next 16-byte boundary)
      const bool store = !(f32 && g.finalize) && (g.n * (f32 ? 4 : 2)) % 16 == 0;
      if (make_map(&mcm, src, g.n, g.m, g.ldd, p.slab_cols, BM, f32) &&
          (!store || make_map(&msm, src, g.n, g.m, g.ldd, p.slab_cols, 32, f32))) {
        p.slab_store = store ? 1 : 0;
        p.slab_f32 = f32 ? 1 : 0;
        // short contractions are bound by the read-modify-write: deeper ring
        // (measured on 128256 x 4096 outputs: up to K = 256 fastest with two
        // stages, eight slabs and two epilogue groups (K = 128: 320 us against
        // 431 us with 3 / 5 / one group), K = 512 and 1024 with 3 / 5 / one
        // (K = 512: 514 us against 673 us), beyond that 4 / 2 / one)
        // (a pair's stages are two thirds the size: one more of them fits)
        if (p.num_k_blocks <= 4) {
          p.nst = pair ? 3 : 2;
          p.nslab = 8;
        } else if (pair && !f32 && p.num_k_blocks <= 8) {
          // K = 320..512 on CTA pairs, bf16 D: four stages and a ring of six
          // slabs fit next to a second epilogue group (measured, grad_weight
          // ms per headline step against 4 / 5 / one group: K = 384 9.08 vs
          // 10.73, K = 512 7.58 vs 8.64; at K = 256, 640, 768 and 1024 the
          // rules around this one stay faster). Six entries are enough for
          // two groups here: a bf16 slab is 64 columns, two per group and
          // tile, so a warp's next slab is at most three ring positions past
          // the one it still holds back, and no wait can close a cycle.
          p.nst = 4;
          p.nslab = 6;
          two_groups = true;
        } else if (p.num_k_blocks <= 16) {
          p.nst = pair ? 4 : 3;
          p.nslab = 5;
        } else {
          p.nst = pair ? 6 : 4;
          p.nslab = 2;
        }
      }
    }
  }
  // plain bf16 output through staging buffers and TMA stores (rows a whole
  // number of 16-byte units: see the slab store above).
  // FLJSD_GEMM_STAGE_OUT=0 in the environment turns it off.
  const char* oenv = getenv("FLJSD_GEMM_STAGE_OUT");
  const bool so_off = oenv != nullptr && oenv[0] == '0';
  if (!rmw && !so_off && p.k_splits == 1 && g.d32 == nullptr && (g.n * 2) % 16 == 0 &&
      make_map(&msm, g.d, g.n, g.m, g.ldd, 64, 32, false)) {
    p.stage_out = 1;
    p.nbuf = 2;  // measured: 4 or 8 buffers (with fewer operand stages) do not help
  }
  p.stat_tiles = (int)((g.n + TC_STATS_COLS - 1) / TC_STATS_COLS);
  // Two epilogue groups where the epilogue bounds the tile (a short
  // contraction per unit: measured ~0.4 us per 32-column chunk and warp, a
  // latency chain that one warp per scheduler cannot hide). A slab ring then
  // needs more than the entries that two groups can hold back with one
  // release deferred per warp: 5 of the fp32 ring (8 entries), 3 of the bf16
  // one (6 or 8 entries, the rules above). Measured on
  // 128256 x 4096 outputs (same box, against one group): read-modify-write
  // 431 -> 320 us at K = 128; write-only 233 -> 190 us at K = 128, even at
  // K = 192, but 244 -> 301 us at K = 256, where the fourth operand stage
  // that the second group's staging buffers displace matters more.
  p.epi_groups = 1;
  if (two_groups || (p.nslab == 8 && p.kb_per_split <= 4) ||
      (p.nslab == 0 && p.kb_per_split <= 3)) {
    p.epi_groups = 2;
    if (p.stage_out) p.nst = pair ? 5 : 3;  // room for 8 warps x 2 staging buffers
  }
  p.epi_mode = p.stage_out ? EPI_STAGE
                           : (p.slab_store && !p.slab_f32 ? EPI_SLAB16 : EPI_GENERIC);
  if (smem_bytes(p.nst, p.nslab, p.stage_out ? 4 * p.epi_groups * p.nbuf : 0, pair) > SMEM_MAX)
    return cudaErrorInvalidConfiguration;  // a schedule above would not fit (never expected)
  if (p.k_splits > 1) {
    cudaError_t e = launch_layout(g.a_mn, g.b_mn, false, ma, mb, mcm, msm, d, p, st);
    if (e != cudaSuccess) return e;
    k_splitk_reduce<<<num_sms() * 4, 256, 0, st>>>(p.partial, p.k_splits, g.m, g.n, g.ldd, d);
    count_extra_launch();
    return cudaGetLastError();
  }
  return launch_layout(g.a_mn, g.b_mn, pair, ma, mb, mcm, msm, d, p, st);
}

}  // namespace fljsd
