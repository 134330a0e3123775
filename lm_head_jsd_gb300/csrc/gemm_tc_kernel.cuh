// bf16 GEMM on the 5th-generation tensor cores (sm_103a): D (+)= A . B^T.
//
// Persistent, warp-specialised kernel, one CTA per SM:
//   warp 0      TMA producer: 128B-swizzled tiles of A and B into a ring of
//               up to 4 shared-memory stages (mbarrier complete_tx).
//   warp 1      MMA issuer: tcgen05.mma kind::f16 (bf16 x bf16 -> fp32), tile
//               128 x 256 x 16, accumulating in tensor memory; two 256-column
//               accumulators so the epilogue of tile i overlaps the main loop
//               of tile i+1. Warp 1 also allocates / frees the 512 TMEM columns.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, rounding to bf16
//               into shared-memory staging buffers written out by TMA stores
//               (measured 2.3x the write rate of 16-byte stores per row and
//               thread on a short-K contraction), or a read-modify-write of the
//               stored value (bf16 or an fp32 side accumulator) for
//               accumulation, and optionally the per-row (max, sum 2^(x - max))
//               partials of every 128 columns (pass 1 of the online softmax).
//   warp 6      for an accumulating epilogue: TMA copies of the old output
//               values, 128 rows x 128 bytes per slab, into a slab ring ahead
//               of the epilogue, which adds the product in place and writes
//               each slab back with one TMA store per warp. (A row-per-thread
//               read-modify-write through plain loads keeps too few bytes in
//               flight to reach HBM bandwidth.)
//   warps 7..10 a second epilogue group for short contractions, where the
//               epilogue sets the pace: warps 2..5 take columns 0..127 of each
//               tile, warps 7..10 columns 128..255 (one epilogue warp per
//               scheduler cannot hide its own instruction latencies).
// Contractions with too few output tiles for the GPU split K: fp32 partials
// per split, summed in a fixed order by a second kernel.
// Operands may be K-major (the contraction dimension contiguous) or MN-major;
// the three contractions of the fused-linear JSD need: logits = X . W^T
// (both K-major), grad_input = dZ . W (B MN-major), grad_weight = dZ^T . X
// (both MN-major).
//
// CTA pairs: two CTAs of a 2-CTA cluster compute a 256 x 256 tile together
// with tcgen05.mma.cta_group::2. Each CTA copies its own 128 rows of A and its
// own 128 rows (half) of the B tile into its own shared memory; the MMA of the
// leader CTA reads both CTAs' halves, so each SM pulls 32 KB per 64-deep
// k-block from L2 instead of 48 KB. Both CTAs' copies complete on the
// leader's stage barrier, the leader's MMA thread issues for both and each
// CTA drains its own 128 accumulator rows from its own tensor memory. The
// leader hands each freed stage and each finished accumulator to the other
// CTA with a plain remote mbarrier arrive; every copy has one destination.
//
// Tile orders: bands of m-blocks sweeping all n-blocks (the band of A stays in
// L2 while B streams), or n-blocks fastest.
//
// Every wait on an mbarrier is bounded in time; on expiry the kernel records
// FLJSD_ERR_TIMEOUT in a device status word, stops issuing work, drains what
// it issued (again bounded) and frees its tensor memory.
//
// This header holds the kernel and its launcher template; the instantiations
// are spread over one translation unit per operand layout (gemm_tc_kk.cu,
// gemm_tc_kmn.cu, gemm_tc_mnmn.cu, gemm_tc_mnk.cu) so that they compile in
// parallel, and gemm_tc.cu holds the host side (tensor maps, schedule choice).
#pragma once

#include "internal.cuh"
#include "gemm_tc.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>

namespace fljsd {
namespace tcgemm {


constexpr int BM = 128, BN = 256, BK = 64, UMMA_K = 16;
constexpr int STAGES = 6;  // operand stages (at most; see KParams::nst)
constexpr int MAX_SLABS = 8;                    // prefetched slabs of the stored output
constexpr int SLAB_BYTES = BM * 128;            // 128 rows x 128 bytes (64 bf16 / 32 fp32)
constexpr int OUT_BUF_BYTES = 32 * 128;  // one warp's staging buffer: 32 rows x 128 B
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int ACC_COLS = BN;                    // fp32 accumulator columns per tile
constexpr int TMEM_COLS = 2 * ACC_COLS;         // double-buffered accumulator
constexpr int EPI_STAGE = 0, EPI_SLAB16 = 1, EPI_GENERIC = 2;
constexpr int CTRL_BYTES = 512;

// One operand stage of a CTA: the A tile (128 rows) and the B tile (256 rows),
// or in a CTA pair (see the kernel) the CTA's half of the B tile (128 rows).
__host__ __device__ constexpr int stage_bytes(bool pair) {
  return A_BYTES + (pair ? B_BYTES / 2 : B_BYTES);
}

// 7 warps (roles at the kernel), 11 with the second epilogue group
__host__ __device__ constexpr int threads_for(int groups) { return groups == 2 ? 352 : 224; }
constexpr int SMEM_MAX = 232448;  // opt-in shared memory per CTA on sm_103
// operand stages + slab ring + alignment slack + control block
// bufs: staging buffers of all epilogue warps together (0 without stage_out)
__host__ __device__ constexpr int smem_bytes(int nst, int nslab, int bufs, bool pair) {
  return nst * stage_bytes(pair) + nslab * SLAB_BYTES + bufs * OUT_BUF_BYTES + 1024 + CTRL_BYTES;
}
static_assert(smem_bytes(2, 8, 0, false) <= SMEM_MAX && smem_bytes(3, 5, 0, false) <= SMEM_MAX &&
                  smem_bytes(4, 2, 0, false) <= SMEM_MAX && smem_bytes(4, 0, 8, false) <= SMEM_MAX &&
                  smem_bytes(3, 0, 16, false) <= SMEM_MAX,
              "shared memory");
static_assert(smem_bytes(6, 0, 8, true) <= SMEM_MAX && smem_bytes(5, 0, 16, true) <= SMEM_MAX &&
                  smem_bytes(4, 5, 0, true) <= SMEM_MAX && smem_bytes(6, 2, 0, true) <= SMEM_MAX &&
                  smem_bytes(3, 8, 0, true) <= SMEM_MAX,
              "shared memory (pairs)");
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
// CL: acquire at cluster scope (the phase completes through arrivals of
// threads in the other CTA of a pair).
template <bool CL = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if (CL)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  return ok != 0;
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive (relaxed, cluster scope) on an mbarrier of another CTA of the
// cluster, given its shared::cluster address (map_to_cta): for hand-overs that
// order only asynchronous work (see the kernel's barrier notes).
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
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

// Shared-memory control block (barrier use per CTA of a pair in the kernel).
struct Ctrl {
  unsigned long long full[STAGES];
  unsigned long long empty[STAGES];
  unsigned long long cfull[MAX_SLABS];   // slab of the stored output landed
  unsigned long long cempty[MAX_SLABS];  // slab read by the four epilogue warps
  unsigned long long tmem_full[2];
  unsigned long long tmem_empty[2];
  unsigned long long drain;
  unsigned long long timeout_ns;
  uint32_t tmem_base;
  volatile int abort;
};
static_assert(sizeof(Ctrl) <= CTRL_BYTES, "control block");

// Bounded wait: true when the phase completed, false on timeout or abort
// (then the abort flag is set and the status word records the timeout).
template <bool CL = false>
__device__ __forceinline__ bool wait_bar(Ctrl* cb, uint32_t bar, uint32_t parity, int* status) {
  if (mbar_try_wait<CL>(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait<CL>(bar, parity)) return true;
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
// Operand copies. In a CTA pair (PAIR) the copy lands in this CTA's shared
// memory and completes (complete_tx) on the mbarrier at shared::cluster
// address `bar`, which may be the other CTA's (the leader's).
template <bool PAIR>
__device__ __forceinline__ void tma_operand(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  if (PAIR)
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
  else
    tma_load_2d(dst, map, bar, x, y);
}
// Shared -> global tensor copy (clipped at the tensor's bounds), tracked by
// bulk groups of the issuing thread.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// all but the most recent bulk group have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// at most `keep` (1, 3 or 7) of the most recent bulk groups still read shared memory
__device__ __forceinline__ void bulk_wait_read_keep(int keep) {
  if (keep >= 7)
    asm volatile("cp.async.bulk.wait_group.read 7;" ::: "memory");
  else if (keep >= 3)
    asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory");
  else
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// generic-proxy writes to shared memory become visible to later TMA reads
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
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
// N >> 3 at [17,23), M >> 4 at [24,29). M is 128 on one CTA and 256 on a CTA
// pair (128 rows in each CTA's tensor memory).
__host__ __device__ constexpr uint32_t instr_desc(bool a_mn, bool b_mn, bool pair) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)((pair ? 2 * BM : BM) >> 4) << 24);
}

// tcgen05 instructions of one kernel all name the same CTA group: ::1 for one
// CTA per tile, ::2 for a CTA pair.
template <bool PAIR>
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  if (PAIR)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// Arrive on this CTA's mbarrier `bar` once every MMA this thread issued has
// completed (for a pair: in both CTAs).
template <bool PAIR>
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  if (PAIR)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
  else
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// Tensor-memory allocation: one warp per CTA (for a pair, one warp in each CTA,
// together).
template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t cols) {
  if (PAIR) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  } else {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
}
template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  if (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols));
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols));
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
  // scheduling units: m-blocks (one CTA per tile) or pairs of m-blocks (a CTA
  // pair per 256 x 256 tile)
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
  // operand stages in use (<= STAGES), and the stored-output prefetch of an
  // accumulating epilogue: warp 6 copies the old values of each tile with TMA
  // into a ring of nslab slabs (slab_cols columns each, cps 32-column chunks
  // per slab) ahead of the epilogue; nslab = 0 reads them with plain loads.
  int nst, nslab, slab_cols, cps;
  // slab_store: the new values go back into the slab and out with one TMA
  // store per epilogue warp (its 32 rows); slab_f32: the slab holds fp32
  int slab_store, slab_f32;
  // stage_out (plain bf16 output, no slabs): each epilogue warp rounds its 32
  // rows x 64 columns into one of nbuf (2, 4 or 8) shared-memory buffers and
  // writes them with a TMA store (whole lines instead of 16 bytes per row and
  // thread)
  int stage_out, nbuf;
  // epilogue warps: one group of four (warps 2-5: all 256 columns of a tile),
  // or two (warps 7-10 take columns 128-255) where the epilogue is the bound
  int epi_groups;
  // epilogue mode, also the kernel's template parameter (so that the common
  // paths carry no runtime branches on it): EPI_STAGE staging + TMA stores
  // (plain bf16 output, optional pass-1 partials), EPI_SLAB16 bf16 slab
  // read-modify-write, EPI_GENERIC everything else (split-K partials, the fp32
  // side accumulator, plain or read-modify-write stores from registers)
  int epi_mode;
  int stat_tiles;  // pass-1 partials per row: one per 128 columns
  int* status;
};

// The remaining ways of storing one 32-column chunk of a row: read-modify-write
// through global memory (bf16 D or the fp32 side accumulator, or from a slab
// that is not written back), plain 16-byte stores per row and thread, and the
// ragged right edge. Kept out of line so that the epilogue loop's common paths
// (staging for TMA stores, the slab read-modify-write) stay compact in the
// instruction cache, which the other warps' loops share.
static __device__ __noinline__ void store_chunk_generic(const KParams& p, float* v, int64_t row,
                                                        int64_t col0, __nv_bfloat16* drow,
                                                        const uint8_t* crow, int c, int lane) {
  // Read-modify-write of the stored value: issue the reads of the whole
  // 32-column chunk before using any of them (they are independent).
  const bool full_chunk = col0 + 32 <= p.n;
  const bool rmw16 = p.accumulate && p.d32 == nullptr;
  const bool rmw32 = p.d32 != nullptr && (p.accumulate || p.finalize);
  if (full_chunk && (rmw16 || rmw32)) {
    if (rmw16) {
      uint4 o[4];
      if (crow != nullptr) {
        // 16-byte units of the swizzled slab row: unit u sits at u ^ (row & 7)
        const int h = (c % p.cps) * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          o[q] = *reinterpret_cast<const uint4*>(crow + (((h + q) ^ (lane & 7)) << 4));
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(drow + col0);
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = src[q];
      }
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
      float4 o[8];
      if (crow != nullptr) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          o[q] = *reinterpret_cast<const float4*>(crow + ((q ^ (lane & 7)) << 4));
      } else {
        const float4* src = reinterpret_cast<const float4*>(p.d32 + row * p.ldd + col0);
#pragma unroll
        for (int q = 0; q < 8; ++q) o[q] = src[q];
      }
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
    return;
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

// Barrier use (one CTA per tile | CTA pair: leader, i.e. cluster rank 0 | other CTA):
//   full[s]        copies of stage s landed | both CTAs' copies (the leader
//                  expects the bytes of both) | unused
//   empty[s]       the MMA read stage s | same | the leader handed stage s on (remote
//                  arrive, once per fill, after expecting both CTAs' bytes)
//   tmem_full[a]   accumulator a complete | same | relayed by the leader's epilogue
//   tmem_empty[a]  4G epilogue warps drained accumulator a | 4G warps of each CTA | unused
// Every hand-over between the two CTAs orders only asynchronous work (TMA
// writes and MMA reads of a stage; MMA writes and tcgen05.ld reads of the
// accumulator, the latter completed by tcgen05.wait::ld before the arrive),
// so the remote arrives are relaxed: a release at cluster scope waits for the
// arriving thread's earlier global stores and cost ~0.5 us per arrive
// (measured: it halved the pair's throughput as the stage hand-over and
// slowed epilogue-bound contractions by 60% as the accumulator hand-offs).
template <bool A_MN, bool B_MN, bool PAIR, int G, int EPI>
__global__ void __launch_bounds__(threads_for(G), 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmS,
              __nv_bfloat16* __restrict__ D, KParams p) {
  constexpr int SB = stage_bytes(PAIR);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t cslabs = base + p.nst * SB;  // slab ring (1024-aligned)
  uint8_t* stg = gbase + p.nst * SB + p.nslab * SLAB_BYTES;  // output staging
  Ctrl* cb = reinterpret_cast<Ctrl*>(stg + (p.stage_out ? 4 * G * p.nbuf * OUT_BUF_BYTES : 0));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&cb->full[s]), 1);
      mbar_init(smem_u32(&cb->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&cb->tmem_full[a]), 1);
      mbar_init(smem_u32(&cb->tmem_empty[a]), PAIR ? 8 * G : 4 * G);
    }
    for (int s = 0; s < MAX_SLABS; ++s) {
      mbar_init(smem_u32(&cb->cfull[s]), 1);
      mbar_init(smem_u32(&cb->cempty[s]), 4);
    }
    mbar_init(smem_u32(&cb->drain), 1);
    cb->abort = 0;
    cb->timeout_ns = p.timeout_ns;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // bring the tensor maps into the TMA unit's descriptor cache up front
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if (p.nslab > 0) prefetch_tensormap(&tmC);
    if (p.slab_store || p.stage_out) prefetch_tensormap(&tmS);
  }
  // the other CTA's copies and arrivals target this CTA's barriers: they must
  // be initialised cluster-wide before anyone issues
  if (PAIR) cluster_sync_all();
  if (warp == 1) tmem_alloc<PAIR>(smem_u32(&cb->tmem_base), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = cb->tmem_base;
  const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int unit_step = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

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
    mb = PAIR ? 2 * mu + (int)rank : mu;
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
      // A pair's other CTA fills a stage only when the leader hands it on:
      // the k-th hand-over of stage s completes phase k of its empty[s], so
      // it waits for the parity of the current round, where the leader (and
      // a single CTA) waits for the MMA to have released the previous round.
      const uint32_t flip = (PAIR && !leader) ? 0u : 1u;
      for (int t = unit0; ok && t < p.num_units; t += unit_step) {
        int mb, nb, tile, split, kb0, kb1;
        unit_split(t, tile, split, kb0, kb1);
        tile_coords(tile, mb, nb);
        const int m0 = mb * BM, n0 = nb * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bar(cb, smem_u32(&cb->empty[stage]), phase ^ flip, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * SB;
          const uint32_t sb = sa + A_BYTES;
          const int k0 = kb * BK;
          uint32_t fb;
          int nh, nb_rows;  // this CTA's rows of the B tile
          if (PAIR) {
            // both CTAs' copies complete on the leader's barrier, which
            // expects the bytes of both before the other CTA may copy (the
            // MMA has read both halves of the previous round by now)
            fb = map_to_cta(smem_u32(&cb->full[stage]), 0);
            if (leader) {
              mbar_arrive_expect_tx(smem_u32(&cb->full[stage]), 2 * SB);
              mbar_arrive_remote_relaxed(map_to_cta(smem_u32(&cb->empty[stage]), 1));
            }
            nh = n0 + (int)rank * (BN / 2);
            nb_rows = BN / 2;
          } else {
            fb = smem_u32(&cb->full[stage]);
            mbar_arrive_expect_tx(fb, SB);
            nh = n0;
            nb_rows = BN;
          }
          if (A_MN) {
            tma_operand<PAIR>(sa, &tmA, fb, m0, k0);
            tma_operand<PAIR>(sa + 8192, &tmA, fb, m0 + 64, k0);
          } else {
            tma_operand<PAIR>(sa, &tmA, fb, k0, m0);
          }
          if (B_MN) {
            for (int j = 0; j < nb_rows / 64; ++j)
              tma_operand<PAIR>(sb + j * 8192, &tmB, fb, nh + 64 * j, k0);
          } else {
            tma_operand<PAIR>(sb, &tmB, fb, k0, nh);
          }
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == p.nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: every issued copy has landed before the CTA may exit. A pair's
      // leader waits for both CTAs' copies (they complete on its barriers;
      // the other CTA copies into a stage only after the leader has expected
      // its bytes), and the cluster barrier at the exit keeps the other CTA
      // resident until then.
      if (!PAIR || leader)
        for (int s = 0; s < STAGES; ++s)
          if (issued[s]) wait_bar(cb, smem_u32(&cb->full[s]), issued_parity[s], p.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (a pair's leader issues for both CTAs) ----------------
    if (lane == 0 && (!PAIR || leader)) {
      constexpr uint32_t idesc = instr_desc(A_MN, B_MN, PAIR);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      bool any = false;
      for (int t = unit0; ok && t < p.num_units; t += unit_step, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!wait_bar<PAIR>(cb, smem_u32(&cb->tmem_empty[acc]), acc_phase ^ 1u, p.status)) break;
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
          const uint32_t sa = base + stage * SB;
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
            mma_bf16<PAIR>(tmem_d, ad, bd, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          }
          // frees the stage once read (in a pair: both CTAs' halves)
          mma_commit<PAIR>(smem_u32(&cb->empty[stage]));
          any = true;
          if (++stage == p.nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit<PAIR>(smem_u32(&cb->tmem_full[acc]));
      }
      if (any) {
        // all issued MMAs have completed before tensor memory is released
        mma_commit<PAIR>(smem_u32(&cb->drain));
        wait_bar(cb, smem_u32(&cb->drain), 0, p.status);
      }
    }
  } else if (warp == 6) {
    // ---------------- stored-output prefetch ----------------
    // The old values of each tile (bf16 D or the fp32 side accumulator), in
    // slabs of 128 rows x 128 bytes, 128B-swizzled, in the epilogue's order.
    if (lane == 0 && p.nslab > 0) {
      int slot = 0;
      uint32_t phase = 0;
      uint32_t issued_parity[MAX_SLABS];
      bool issued[MAX_SLABS];
      for (int s = 0; s < MAX_SLABS; ++s) issued[s] = false;
      bool ok = true;
      for (int t = unit0; ok && t < p.num_units; t += unit_step) {
        int mb, nb, tile, split, kb0, kb1;
        unit_split(t, tile, split, kb0, kb1);
        tile_coords(tile, mb, nb);
        const int n0 = nb * BN;
        const int ncols = (int)min((int64_t)BN, p.n - n0);
        const int nsl = (ncols + p.slab_cols - 1) / p.slab_cols;
        for (int j = 0; j < nsl; ++j) {
          if (!wait_bar(cb, smem_u32(&cb->cempty[slot]), phase ^ 1u, p.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&cb->cfull[slot]);
          mbar_arrive_expect_tx(fb, SLAB_BYTES);
          tma_load_2d(cslabs + slot * SLAB_BYTES, &tmC, fb, n0 + j * p.slab_cols, mb * BM);
          issued[slot] = true;
          issued_parity[slot] = phase;
          if (++slot == p.nslab) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < MAX_SLABS; ++s)
        if (issued[s]) wait_bar(cb, smem_u32(&cb->cfull[s]), issued_parity[s], p.status);
    }
  } else if (warp <= 5 || G == 2) {
    // ---------------- epilogue (warps 2..5, and 7..10 with two groups) ----------------
    const int sub = warp & 3;  // TMEM lane quarter this warp may access
    const int grp = warp >= 7 ? 1 : 0;
    const int ew = grp * 4 + sub;  // epilogue warp index (staging buffers)
    // chunks of 32 columns this group handles: all 8, or one half each
    const int c_lo = G == 2 ? grp * 4 : 0;
    const int c_hi = G == 2 ? c_lo + 4 : 8;
    int local = 0;
    // ring position (slot, phase) of slab 0 of the current tile: the slabs of
    // all earlier tiles of this CTA come first (the prefetch warp's order)
    int tslot = 0;
    uint32_t tphase = 0;
    // the mode's paths, fixed at compile time where the mode fixes them
    constexpr bool kStage = EPI == EPI_STAGE;
    const bool kSlabStore = EPI == EPI_SLAB16 || (EPI == EPI_GENERIC && p.slab_store);
    const bool kSlabs = EPI == EPI_SLAB16 || (EPI == EPI_GENERIC && p.nslab > 0);
    int pend = -1;  // slab whose TMA store may still be reading it (lane 0)
    int sbuf = 0;   // staging buffer of this warp in use (stage_out)
    bool dead = false;
    for (int t = unit0; t < p.num_units; t += unit_step, ++local) {
      int mb, nb, tile, split, kb0, kb1;
      unit_split(t, tile, split, kb0, kb1);
      tile_coords(tile, mb, nb);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      bool ok = true;
      if (lane == 0) {
        ok = wait_bar<PAIR>(cb, smem_u32(&cb->tmem_full[acc]), acc_phase, p.status);
        // the leader's first epilogue warp tells the other CTA that its rows
        // of the accumulator are complete too (the MMAs were issued here)
        if (PAIR && ok && leader && ew == 0)
          mbar_arrive_remote_relaxed(map_to_cta(smem_u32(&cb->tmem_full[acc]), 1));
      }
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
      const int ncols = (int)min((int64_t)BN, p.n - (int64_t)nb * BN);
      const int nch = (ncols + 31) / 32;
      int cslot = 0;  // ring slot of the current slab
      // not unrolled: eight copies of this body would crowd the instruction
      // cache that the other warps' loops share (measured: the logits GEMM
      // 9.0 -> 14.2 ms when the bounds became compile-time constants)
#pragma unroll 1
      for (int c = c_lo; c < c_hi; ++c) {
        if (c >= nch) break;  // columns past the output: nothing to store, no slab
        float v[32];
        tmem_ld32(tmem_base + ((uint32_t)(sub * 32) << 16) + acc * ACC_COLS + c * 32, v);
        uint8_t* crow = nullptr;  // this row's 128 bytes of the current slab
        if (kSlabs) {
          cslot = tslot + (p.cps == 2 ? c >> 1 : c);
          uint32_t cphase = tphase;
          while (cslot >= p.nslab) {
            cslot -= p.nslab;
            cphase ^= 1u;
          }
          if ((c & (p.cps - 1)) == 0) {
            const bool got = wait_bar(cb, smem_u32(&cb->cfull[cslot]), cphase, p.status);
            if (!__all_sync(0xffffffffu, got)) {
              dead = true;
              break;
            }
          }
          crow = gbase + p.nst * SB + cslot * SLAB_BYTES + (sub * 32 + lane) * 128;
        }
        if (kStage && (c & 1) == 0) {
          // the store that last used this staging buffer has read it
          if (lane == 0) bulk_wait_read_keep(p.nbuf - 1);
          __syncwarp();
        }
        if (kSlabStore) {
          // old + product, written back in place (16-byte unit u of the
          // swizzled row sits at u ^ (row & 7)); rows and columns past the
          // output are zero-filled here and clipped by the store
          if (EPI == EPI_GENERIC) {  // the fp32 side accumulator
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float4* u = reinterpret_cast<float4*>(crow + ((q ^ (lane & 7)) << 4));
              const float4 o = *u;
              *u = make_float4(o.x + v[4 * q], o.y + v[4 * q + 1], o.z + v[4 * q + 2],
                               o.w + v[4 * q + 3]);
            }
          } else {
            const int h = (c % p.cps) * 4;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4* u = reinterpret_cast<uint4*>(crow + (((h + q) ^ (lane & 7)) << 4));
              const uint4 o = *u;
              const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
              float x[8];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                x[2 * e] = v[q * 8 + 2 * e] + bf16_lo(ow[e]);
                x[2 * e + 1] = v[q * 8 + 2 * e + 1] + bf16_hi(ow[e]);
              }
              *u = make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                              pack_bf16(x[6], x[7]));
            }
          }
        } else do {  // `continue` ends this chunk's work; the slab is released below
          if (!row_ok) continue;
          const int64_t col0 = (int64_t)nb * BN + c * 32;
          if (EPI == EPI_GENERIC && p.k_splits > 1) {
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
          if (kStage) {
            // rounded to bf16 into this warp's staging buffer (16-byte unit u
            // of the swizzled 128-byte row sits at u ^ (row & 7))
            uint8_t* srow = stg + ((ew * p.nbuf + sbuf) * 32 + lane) * 128;
            const int h = (c & 1) * 4;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(srow + (((h + q) ^ (lane & 7)) << 4)) =
                  make_uint4(pack_bf16(v[q * 8], v[q * 8 + 1]), pack_bf16(v[q * 8 + 2], v[q * 8 + 3]),
                             pack_bf16(v[q * 8 + 4], v[q * 8 + 5]),
                             pack_bf16(v[q * 8 + 6], v[q * 8 + 7]));
            continue;
          }
          if constexpr (EPI == EPI_GENERIC) {
            float vv[32];  // the out-of-line path takes the values through memory
#pragma unroll
            for (int e = 0; e < 32; ++e) vv[e] = v[e];
            store_chunk_generic(p, vv, row, col0, drow, crow, c, lane);
          }
        } while (0);
        if (kStage && ((c & 1) || c == nch - 1)) {
          // 32 rows x 64 columns staged: one TMA store (clipped at the output's
          // bounds)
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int64_t r0 = (int64_t)mb * BM + sub * 32;
            if (r0 < p.m)
              tma_store_2d(&tmS, smem_u32(stg + (ew * p.nbuf + sbuf) * OUT_BUF_BYTES),
                           nb * BN + (c >> 1) * 64, (int32_t)r0);
            bulk_commit();
          }
          if (++sbuf == p.nbuf) sbuf = 0;
        }
        if (kSlabs && ((c + 1) % p.cps == 0 || c == nch - 1)) {
          // this warp is done with the slab
          if (kSlabStore) {
            // its 32 rows go out with one TMA store; the slab is handed back
            // to the prefetch warp once the store has read it (one behind)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int64_t r0 = (int64_t)mb * BM + sub * 32;
              if (r0 < p.m)
                tma_store_2d(&tmS, smem_u32(crow - lane * 128),
                             nb * BN + (c / p.cps) * p.slab_cols, (int32_t)r0);
              bulk_commit();
              bulk_wait_read_1();
              if (pend >= 0) mbar_arrive(smem_u32(&cb->cempty[pend]));
            }
            pend = cslot;
          } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&cb->cempty[cslot]));
          }
        }
        if (p.stats && ((c & 3) == 3 || c == nch - 1)) {
          // the partial of this row over one 128-column half of the tile
          if (row_ok) p.stats[row * p.stat_tiles + nb * 2 + (c >> 2)] = make_float2(st_m, st_d);
          st_m = -INFINITY;
          st_d = 0.f;
        }
      }
      if (dead) break;
      if (kSlabs) {
        tslot += (ncols + p.slab_cols - 1) / p.slab_cols;
        while (tslot >= p.nslab) {
          tslot -= p.nslab;
          tphase ^= 1u;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // the accumulator's MMAs are the leader's: its barrier counts the
        // epilogue warps of both CTAs
        if (PAIR && !leader)
          mbar_arrive_remote_relaxed(map_to_cta(smem_u32(&cb->tmem_empty[acc]), 0));
        else
          mbar_arrive(smem_u32(&cb->tmem_empty[acc]));
      }
    }
    if ((kSlabStore || kStage) && lane == 0) {
      // every store of this warp has completed before the CTA may exit
      bulk_wait_all();
      if (pend >= 0) mbar_arrive(smem_u32(&cb->cempty[pend]));
    }
  }

  tc_fence_before();
  __syncthreads();
  // no CTA of a pair leaves while the other may still read its shared memory
  // (the leader's MMAs), land copies on its barriers or arrive on them
  if (PAIR) cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<PAIR>(tmem_base, TMEM_COLS);
  }
}

template <bool A_MN, bool B_MN, bool PAIR, int G, int EPI>
cudaError_t launch_g(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mcm,
                     const CUtensorMap& msm, __nv_bfloat16* d, KParams p, cudaStream_t st) {
  constexpr int THREADS = threads_for(G);
  const int smem = smem_bytes(p.nst, p.nslab, p.stage_out ? 4 * G * p.nbuf : 0, PAIR);
  static int max_clusters[64] = {0};
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cache = dev >= 0 && dev < 64;
  auto kern = k_gemm_tc<A_MN, B_MN, PAIR, G, EPI>;
  if (!cache || !attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
    if (e != cudaSuccess) return e;
    if (cache) attr_set[dev] = true;
  }
  if (!PAIR) {
    const int grid = p.num_units < num_sms() ? p.num_units : num_sms();
    kern<<<grid, THREADS, smem, st>>>(ma, mb, mcm, msm, d, p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, mcm, msm, d, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Every (epilogue groups, epilogue mode) variant of one layout and schedule.
template <bool A_MN, bool B_MN, bool PAIR>
cudaError_t launch_modes(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mcm,
                         const CUtensorMap& msm, __nv_bfloat16* d, const KParams& p,
                         cudaStream_t st) {
  if (p.epi_groups == 2) {
    if (p.epi_mode == EPI_STAGE) return launch_g<A_MN, B_MN, PAIR, 2, EPI_STAGE>(ma, mb, mcm, msm, d, p, st);
    if (p.epi_mode == EPI_SLAB16) return launch_g<A_MN, B_MN, PAIR, 2, EPI_SLAB16>(ma, mb, mcm, msm, d, p, st);
    return launch_g<A_MN, B_MN, PAIR, 2, EPI_GENERIC>(ma, mb, mcm, msm, d, p, st);
  }
  if (p.epi_mode == EPI_STAGE) return launch_g<A_MN, B_MN, PAIR, 1, EPI_STAGE>(ma, mb, mcm, msm, d, p, st);
  if (p.epi_mode == EPI_SLAB16) return launch_g<A_MN, B_MN, PAIR, 1, EPI_SLAB16>(ma, mb, mcm, msm, d, p, st);
  return launch_g<A_MN, B_MN, PAIR, 1, EPI_GENERIC>(ma, mb, mcm, msm, d, p, st);
}

// Launchers of one operand layout (A K-major or MN-major, B likewise), each
// defined in its own translation unit: every schedule (CTA pairs or one CTA
// per tile) and epilogue variant (one or two epilogue groups, from
// p.epi_groups).
#define FLJSD_TC_LAUNCHER(name)                                                    \
  cudaError_t name(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mcm, \
                   const CUtensorMap& msm, __nv_bfloat16* d, const KParams& p, bool pair, \
                   cudaStream_t st)
FLJSD_TC_LAUNCHER(launch_kk);
FLJSD_TC_LAUNCHER(launch_kmn);
FLJSD_TC_LAUNCHER(launch_mnmn);
FLJSD_TC_LAUNCHER(launch_mnk);

}  // namespace tcgemm
}  // namespace fljsd
