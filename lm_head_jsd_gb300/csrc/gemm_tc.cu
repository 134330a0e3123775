// bf16 GEMM on the 5th-generation tensor cores (sm_103a): D (+)= A . B^T.
//
// Persistent, warp-specialised kernel, one CTA per SM:
//   warp 0      TMA producer: 128B-swizzled tiles of A and B into a 4-stage
//               shared-memory ring (mbarrier complete_tx).
//   warp 1      MMA issuer: tcgen05.mma kind::f16 (bf16 x bf16 -> fp32), tile
//               128 x 256 x 16, accumulating in tensor memory; two 256-column
//               accumulators so the epilogue of tile i overlaps the main loop
//               of tile i+1. Warp 1 also allocates / frees the 512 TMEM columns.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, rounding to bf16 with
//               16-byte stores, or a read-modify-write of the stored value (bf16
//               or an fp32 side accumulator) for accumulation, and optionally
//               the per-row (max, sum 2^(x - max)) partials of the stored tile
//               (pass 1 of the online softmax).
// Operands may be K-major (the contraction dimension contiguous) or MN-major;
// the three contractions of the fused-linear JSD need: logits = X . W^T
// (both K-major), grad_input = dZ . W (B MN-major), grad_weight = dZ^T . X
// (both MN-major).
//
// Pairs of m-blocks can run as a 2-CTA cluster that shares the B tile: each
// CTA fetches half of it with a TMA multicast into both CTAs, each MMA frees a
// stage in both CTAs with a multicast commit, and cluster barriers fence the
// start and the exit. Tile orders: bands of m-blocks sweeping all n-blocks
// (the band of A stays in L2 while B streams), or n-blocks fastest.
//
// Every wait on an mbarrier is bounded in time; on expiry the kernel records
// FLJSD_ERR_TIMEOUT in a device status word, stops issuing work, drains what
// it issued (again bounded) and frees its tensor memory.
#include "internal.cuh"
#include "gemm_tc.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

namespace fljsd {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int ACC_COLS = BN;                    // fp32 accumulator columns per tile
constexpr int TMEM_COLS = 2 * ACC_COLS;         // double-buffered accumulator
constexpr int THREADS = 192;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr unsigned long long kTimeoutNs = 10ull * 1000 * 1000 * 1000;  // 10 s by default

// ---- PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared-memory control block.
struct Ctrl {
  unsigned long long full[STAGES];
  unsigned long long empty[STAGES];
  unsigned long long tmem_full[2];
  unsigned long long tmem_empty[2];
  unsigned long long drain;
  unsigned long long timeout_ns;
  uint32_t tmem_base;
  volatile int abort;
};
static_assert(sizeof(Ctrl) <= 256, "control block");

// Bounded wait: true when the phase completed, false on timeout or abort
// (then the abort flag is set and the status word records the timeout).
__device__ __forceinline__ bool wait_bar(Ctrl* cb, uint32_t bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (cb->abort) return false;
      if (globaltimer() - t0 > cb->timeout_ns) {
        cb->abort = 1;
        if (status) atomicExch(status, (int)FLJSD_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// Same copy, delivered to the same shared-memory offset (and completing on the
// same mbarrier offset) in every CTA of the cluster named in cta_mask.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                               int32_t x, int32_t y, uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// tcgen05 shared-memory matrix descriptor (sm_100 family):
// [0,14) start >> 4, [16,30) leading-dimension byte offset >> 4,
// [32,46) stride-dimension byte offset >> 4, [46,48) version = 1,
// [49,52) base offset = 0, [52] LBO mode = 0, [61,64) layout: 2 = 128B swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32 ([4,6) = 1), A and B bf16
// ([7,10) = 1, [10,13) = 1), A / B major ([15], [16]: 1 = MN-major),
// N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t instr_desc(bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// Arrive on the mbarrier at this offset in every CTA of cta_mask once all
// previously issued MMAs of this thread have completed.
__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 columns of 32-bit accumulators: thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float ex2f_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

struct KParams {
  int64_t m, n, k;
  int64_t ldd;
  float2* stats;       // [m x num_n_blocks] (max, sum 2^(x - max)) per row and tile, or null
  float stats_scale;   // x = bf16(value) * stats_scale
  int num_m_blocks, num_n_blocks, num_k_blocks, num_tiles;
  // scheduling units: m-blocks (one CTA per tile) or pairs of m-blocks (a
  // 2-CTA cluster per pair, sharing the B tile through multicast)
  int m_units, num_units;
  int raster;   // 0: bands of group_m m-units sweeping all n-blocks; 1: n-blocks fastest
  int group_m;  // m-units per band
  int accumulate;
  float* d32;    // optional fp32 accumulator with row stride ldd (see TcGemmArgs)
  int finalize;
  unsigned long long timeout_ns;  // limit of every mbarrier wait
  int stall_producer;             // test of the bounded waits: issue no copies
  // split-K: unit t covers tile t / k_splits and k-blocks [s*kb_per, (s+1)*kb_per)
  // of split s = t % k_splits, written as fp32 to partial[s][m][ldd]
  int k_splits, kb_per_split;
  float* partial;
  int* status;
};

template <bool A_MN, bool B_MN, bool MC>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              __nv_bfloat16* __restrict__ D, KParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  Ctrl* cb = reinterpret_cast<Ctrl*>(gbase + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&cb->full[s]), 1);
      // with multicast both CTAs' MMAs must have read a stage before either
      // producer refills it (each producer writes into both CTAs)
      mbar_init(smem_u32(&cb->empty[s]), MC ? 2 : 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&cb->tmem_full[a]), 1);
      mbar_init(smem_u32(&cb->tmem_empty[a]), 4);
    }
    mbar_init(smem_u32(&cb->drain), 1);
    cb->abort = 0;
    cb->timeout_ns = p.timeout_ns;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&cb->tmem_base)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = cb->tmem_base;
  // the peer's multicast copies and commits target this CTA's barriers: they
  // must be initialised cluster-wide before anyone issues
  if (MC) cluster_sync_all();
  const uint32_t rank = MC ? cluster_ctarank() : 0u;
  const int unit0 = MC ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int unit_step = MC ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  // Tile order. n-fastest: all n-blocks of a few m-blocks run together (used
  // when B is small and A streams). Grouped: bands of group_m m-blocks; inside
  // a band the m-blocks vary fastest and the band walks every n-block, so the
  // band's slice of A stays in L2 while B streams through once per band.
  auto tile_coords = [&](int t, int& mb, int& nb) {
    int mu;
    if (p.raster == 1) {
      nb = t % p.num_n_blocks;
      mu = t / p.num_n_blocks;
    } else {
      const int band = t / (p.group_m * p.num_n_blocks);
      const int m0 = band * p.group_m;
      const int gm = min(p.group_m, p.m_units - m0);
      const int r = t - band * p.group_m * p.num_n_blocks;
      mu = m0 + r % gm;
      nb = r / gm;
    }
    mb = MC ? 2 * mu + (int)rank : mu;
  };
  auto unit_split = [&](int t, int& tile, int& split, int& kb0, int& kb1) {
    if (p.k_splits > 1) {
      tile = t / p.k_splits;
      split = t - tile * p.k_splits;
      kb0 = split * p.kb_per_split;
      kb1 = min(p.num_k_blocks, kb0 + p.kb_per_split);
    } else {
      tile = t;
      split = 0;
      kb0 = 0;
      kb1 = p.num_k_blocks;
    }
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_parity[STAGES];
      bool issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = false;
      bool ok = !p.stall_producer;
      for (int t = unit0; ok && t < p.num_units; t += unit_step) {
        int mb, nb, tile, split, kb0, kb1;
        unit_split(t, tile, split, kb0, kb1);
        tile_coords(tile, mb, nb);
        const int m0 = mb * BM, n0 = nb * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bar(cb, smem_u32(&cb->empty[stage]), phase ^ 1u, p.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&cb->full[stage]);
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const uint32_t sa = base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          const int k0 = kb * BK;
          if (A_MN) {
            tma_load_2d(sa, &tmA, fb, m0, k0);
            tma_load_2d(sa + 8192, &tmA, fb, m0 + 64, k0);
          } else {
            tma_load_2d(sa, &tmA, fb, k0, m0);
          }
          if (MC) {
            // this CTA fetches half of the B tile for both CTAs of the pair
            if (B_MN) {
#pragma unroll
              for (int j = 2 * (int)rank; j < 2 * (int)rank + 2; ++j)
                tma_load_2d_mc(sb + j * 8192, &tmB, fb, n0 + 64 * j, k0, (uint16_t)3);
            } else {
              tma_load_2d_mc(sb + rank * (B_BYTES / 2), &tmB, fb, k0, n0 + (int)rank * (BN / 2),
                             (uint16_t)3);
            }
          } else if (B_MN) {
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * 8192, &tmB, fb, n0 + 64 * j, k0);
          } else {
            tma_load_2d(sb, &tmB, fb, k0, n0);
          }
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: every issued copy has landed before the CTA may exit
      for (int s = 0; s < STAGES; ++s)
        if (issued[s]) wait_bar(cb, smem_u32(&cb->full[s]), issued_parity[s], p.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc(A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      bool any = false;
      for (int t = unit0; ok && t < p.num_units; t += unit_step, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!wait_bar(cb, smem_u32(&cb->tmem_empty[acc]), acc_phase ^ 1u, p.status)) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + acc * ACC_COLS;
        int tile_i, split_i, kb0, kb1;
        unit_split(t, tile_i, split_i, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bar(cb, smem_u32(&cb->full[stage]), phase, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            uint64_t ad, bd;
            if (A_MN)  // 16 k-rows of 128 B per step; MN atoms 8 KB apart
              ad = smem_desc(sa + kk * (UMMA_K * 128), 8192, 1024);
            else  // 32 bytes of k per step inside the 128-byte swizzled row
              ad = smem_desc(sa + kk * (UMMA_K * 2), 16, 1024);
            if (B_MN)
              bd = smem_desc(sb + kk * (UMMA_K * 128), 8192, 1024);
            else
              bd = smem_desc(sb + kk * (UMMA_K * 2), 16, 1024);
            mma_bf16(tmem_d, ad, bd, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          }
          // frees the stage once read (in both CTAs of a multicast pair)
          if (MC)
            mma_commit_mc(smem_u32(&cb->empty[stage]), (uint16_t)3);
          else
            mma_commit(smem_u32(&cb->empty[stage]));
          any = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&cb->tmem_full[acc]));
      }
      if (any) {
        // all issued MMAs have completed before tensor memory is released
        mma_commit(smem_u32(&cb->drain));
        wait_bar(cb, smem_u32(&cb->drain), 0, p.status);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int sub = warp & 3;  // TMEM lane quarter this warp may access
    int local = 0;
    for (int t = unit0; t < p.num_units; t += unit_step, ++local) {
      int mb, nb, tile, split, kb0, kb1;
      unit_split(t, tile, split, kb0, kb1);
      tile_coords(tile, mb, nb);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      bool ok = true;
      if (lane == 0) ok = wait_bar(cb, smem_u32(&cb->tmem_full[acc]), acc_phase, p.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const int64_t row = (int64_t)mb * BM + sub * 32 + lane;
      const bool row_ok = row < p.m;
      __nv_bfloat16* drow = D + row * p.ldd;
      // running (max, sum 2^(x - max)) of this row over the tile's columns, on
      // the values as stored (rounded to bf16) times stats_scale: pass 1 of the
      // online softmax, done here while the tile is in registers
      float st_m = -INFINITY, st_d = 0.f;
      for (int c = 0; c < ACC_COLS / 32; ++c) {
        float v[32];
        tmem_ld32(tmem_base + ((uint32_t)(sub * 32) << 16) + acc * ACC_COLS + c * 32, v);
        if (!row_ok) continue;
        const int64_t col0 = (int64_t)nb * BN + c * 32;
        if (p.k_splits > 1) {
          // split-K partial: plain fp32 store, summed later in a fixed order
          float* dst = p.partial + ((int64_t)split * p.m + row) * p.ldd + col0;
          if (col0 + 32 <= p.n) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              reinterpret_cast<float4*>(dst)[q] =
                  make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          } else {
            for (int e = 0; e < 32 && col0 + e < p.n; ++e) dst[e] = v[e];
          }
          continue;
        }
        if (p.stats) {
          float cm = -INFINITY;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float x = (col0 + e < p.n)
                ? __fmul_rn(__bfloat162float(__float2bfloat16_rn(v[e])), p.stats_scale)
                : -INFINITY;
            cm = fmaxf(cm, x);
          }
          if (cm > st_m) {
            st_d = (st_m == -INFINITY) ? 0.f : st_d * ex2f_approx(st_m - cm);
            st_m = cm;
          }
          // exponent = x * scale - max with the exact product rounded once, so
          // that large scaled logits (small T) keep their precision near the max
          float acc_d = 0.f;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if (col0 + e < p.n)
              acc_d += ex2f_approx(
                  __fmaf_rn(__bfloat162float(__float2bfloat16_rn(v[e])), p.stats_scale, -st_m));
          }
          st_d += acc_d;
        }
        // Read-modify-write of the stored value: issue the reads of the whole
        // 32-column chunk before using any of them (they are independent).
        const bool full_chunk = col0 + 32 <= p.n;
        const bool rmw16 = p.accumulate && p.d32 == nullptr;
        const bool rmw32 = p.d32 != nullptr && (p.accumulate || p.finalize);
        if (full_chunk && (rmw16 || rmw32)) {
          if (rmw16) {
            const uint4* src = reinterpret_cast<const uint4*>(drow + col0);
            uint4 o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) o[q] = src[q];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t ow[4] = {o[q].x, o[q].y, o[q].z, o[q].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                v[q * 8 + 2 * e] += bf16_lo(ow[e]);
                v[q * 8 + 2 * e + 1] += bf16_hi(ow[e]);
              }
            }
          } else {
            const float4* src = reinterpret_cast<const float4*>(p.d32 + row * p.ldd + col0);
            float4 o[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) o[q] = src[q];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              v[4 * q] += o[q].x;
              v[4 * q + 1] += o[q].y;
              v[4 * q + 2] += o[q].z;
              v[4 * q + 3] += o[q].w;
            }
          }
          if (p.d32 != nullptr && !p.finalize) {
            float4* dst = reinterpret_cast<float4*>(p.d32 + row * p.ldd + col0);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(drow + col0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pack_bf16(v[q * 8], v[q * 8 + 1]), pack_bf16(v[q * 8 + 2], v[q * 8 + 3]),
                                  pack_bf16(v[q * 8 + 4], v[q * 8 + 5]),
                                  pack_bf16(v[q * 8 + 6], v[q * 8 + 7]));
          }
          continue;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int64_t col = col0 + q * 8;
          if (col >= p.n) break;
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = v[q * 8 + e];
          __nv_bfloat16* dst = drow + col;
          if (p.d32 != nullptr) {
            // fp32 accumulator: D32 (+)= product, or on the last pass
            // D = round(D32 + product)
            float* s32 = p.d32 + row * p.ldd + col;
            const int ne = (col + 8 <= p.n) ? 8 : (int)(p.n - col);
            if (ne == 8) {
              if (p.accumulate || p.finalize) {
                const float4 a0 = reinterpret_cast<const float4*>(s32)[0];
                const float4 a1 = reinterpret_cast<const float4*>(s32)[1];
                x[0] += a0.x; x[1] += a0.y; x[2] += a0.z; x[3] += a0.w;
                x[4] += a1.x; x[5] += a1.y; x[6] += a1.z; x[7] += a1.w;
              }
              if (p.finalize) {
                *reinterpret_cast<uint4*>(dst) =
                    make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]),
                               pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
              } else {
                reinterpret_cast<float4*>(s32)[0] = make_float4(x[0], x[1], x[2], x[3]);
                reinterpret_cast<float4*>(s32)[1] = make_float4(x[4], x[5], x[6], x[7]);
              }
            } else {
              for (int e = 0; e < ne; ++e) {
                float y = x[e];
                if (p.accumulate || p.finalize) y += s32[e];
                if (p.finalize) dst[e] = __float2bfloat16_rn(y);
                else s32[e] = y;
              }
            }
          } else if (col + 8 <= p.n) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
            if (p.accumulate) {
              const uint4 o = *d4;
              const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                x[2 * e] += bf16_lo(ow[e]);
                x[2 * e + 1] += bf16_hi(ow[e]);
              }
            }
            *d4 = make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]),
                             pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
          } else {
            for (int e = 0; e < 8 && col + e < p.n; ++e) {
              float y = x[e];
              if (p.accumulate) y += __bfloat162float(dst[e]);
              dst[e] = __float2bfloat16_rn(y);
            }
          }
        }
      }
      if (p.stats && row_ok) p.stats[row * p.num_n_blocks + nb] = make_float2(st_m, st_d);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&cb->tmem_empty[acc]));
    }
  }

  tc_fence_before();
  __syncthreads();
  // no CTA of a pair leaves while its peer may still write into its shared
  // memory or arrive on its barriers
  if (MC) cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS));
  }
}

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

// 2-D bf16 tensor map over a row-major [outer x inner] matrix with row stride
// ld elements; box = box_inner x box_outer; 128-byte swizzle; zero fill.
bool make_map(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int64_t ld,
              int box_inner, int box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool A_MN, bool B_MN, bool MC>
cudaError_t launch_t(const CUtensorMap& ma, const CUtensorMap& mb, __nv_bfloat16* d, KParams p,
                     cudaStream_t st) {
  static int max_clusters[64] = {0};
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cache = dev >= 0 && dev < 64;
  auto kern = k_gemm_tc<A_MN, B_MN, MC>;
  if (!cache || !attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (cache) attr_set[dev] = true;
  }
  if (!MC) {
    const int grid = p.num_units < num_sms() ? p.num_units : num_sms();
    kern<<<grid, THREADS, SMEM_BYTES, st>>>(ma, mb, d, p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // a persistent grid must not exceed the clusters that can be resident at once
  if (!cache || max_clusters[dev] == 0) {
    int n = 0;
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) n = 1;
    if (cache) max_clusters[dev] = n;
    else max_clusters[0] = n;
  }
  const int mc = cache ? max_clusters[dev] : max_clusters[0];
  const int clusters = p.num_units < mc ? p.num_units : mc;
  cfg.gridDim = dim3(2 * clusters);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, d, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
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
  // pairs of m-blocks share B through a 2-CTA cluster whenever there are two
  // m-blocks to pair (and g.no_multicast is not set)
  const int64_t mblocks = (g.m + BM - 1) / BM;
  // FLJSD_GEMM_MULTICAST=0 in the environment selects one CTA per tile for
  // every call (both schedules compute identical results)
  const char* env = getenv("FLJSD_GEMM_MULTICAST");
  const bool env_off = env != nullptr && env[0] == '0';
  const bool mc = mblocks >= 2 && !g.no_multicast && !env_off;
  CUtensorMap ma, mb;
  bool ok;
  if (g.a_mn)  // A stored [k x m]
    ok = make_map(&ma, g.a, g.m, g.k, g.lda, 64, 64);
  else  // A stored [m x k]
    ok = make_map(&ma, g.a, g.k, g.m, g.lda, BK, BM);
  if (!ok) return cudaErrorInvalidValue;
  if (g.b_mn)  // B stored [k x n]
    ok = make_map(&mb, g.b, g.n, g.k, g.ldb, 64, 64);
  else  // B stored [n x k]; with multicast each CTA fetches half the tile's rows
    ok = make_map(&mb, g.b, g.k, g.n, g.ldb, BK, mc ? BN / 2 : BN);
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
  p.m_units = mc ? (p.num_m_blocks + 1) / 2 : p.num_m_blocks;
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
    const int64_t per_unit = (int64_t)BM * (mc ? 2 : 1) * g.k * 2;
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
  // split-K when the output has too few tiles for the GPU (one-CTA schedule,
  // plain stores only); the partials go to the caller's scratch.
  // FLJSD_GEMM_SPLITK=0 in the environment turns it off.
  p.k_splits = 1;
  p.kb_per_split = p.num_k_blocks;
  p.partial = nullptr;
  const char* senv = getenv("FLJSD_GEMM_SPLITK");
  const bool split_off = senv != nullptr && senv[0] == '0';
  if (!mc && !split_off && g.splitk_ws != nullptr && !g.accumulate && g.d32 == nullptr &&
      g.stats == nullptr) {
    int s_ = splitk_factor(g.m, g.n, g.k, num_sms());
    while (s_ > 1 && (size_t)s_ * (size_t)g.m * (size_t)g.ldd * sizeof(float) > g.splitk_ws_bytes)
      --s_;
    if (s_ > 1) {
      p.kb_per_split = (p.num_k_blocks + s_ - 1) / s_;
      p.k_splits = (p.num_k_blocks + p.kb_per_split - 1) / p.kb_per_split;
      p.partial = g.splitk_ws;
      p.num_units = p.num_tiles * p.k_splits;
    }
  }
  if (p.k_splits > 1) {
    cudaError_t e;
    if (!g.a_mn && !g.b_mn) e = launch_t<false, false, false>(ma, mb, d, p, st);
    else if (!g.a_mn && g.b_mn) e = launch_t<false, true, false>(ma, mb, d, p, st);
    else if (g.a_mn && g.b_mn) e = launch_t<true, true, false>(ma, mb, d, p, st);
    else e = launch_t<true, false, false>(ma, mb, d, p, st);
    if (e != cudaSuccess) return e;
    k_splitk_reduce<<<num_sms() * 4, 256, 0, st>>>(p.partial, p.k_splits, g.m, g.n, g.ldd, d);
    count_extra_launch();
    return cudaGetLastError();
  }
  if (mc) {
    if (!g.a_mn && !g.b_mn) return launch_t<false, false, true>(ma, mb, d, p, st);
    if (!g.a_mn && g.b_mn) return launch_t<false, true, true>(ma, mb, d, p, st);
    if (g.a_mn && g.b_mn) return launch_t<true, true, true>(ma, mb, d, p, st);
    return launch_t<true, false, true>(ma, mb, d, p, st);
  }
  if (!g.a_mn && !g.b_mn) return launch_t<false, false, false>(ma, mb, d, p, st);
  if (!g.a_mn && g.b_mn) return launch_t<false, true, false>(ma, mb, d, p, st);
  if (g.a_mn && g.b_mn) return launch_t<true, true, false>(ma, mb, d, p, st);
  return launch_t<true, false, false>(ma, mb, d, p, st);
}

}  // namespace fljsd
