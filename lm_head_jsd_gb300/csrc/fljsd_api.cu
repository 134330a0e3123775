// C ABI of libfljsd.so: argument checks, the chunk planner, the chunk loop
// of the forward pass, the backward scaling, status strings, launch
// accounting and per-kernel event timing. Declarations and semantics are in
// include/fljsd.h.
#include "internal.cuh"
#include "gemm_tc.cuh"

#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

namespace fljsd {

// ---------------------------------------------------------------------------
// launch accounting and tracing
// ---------------------------------------------------------------------------
namespace {
std::atomic<int64_t> g_launches{0};

struct Trace {
  std::mutex mu;
  int max = 0;
  int used = 0;
  int open = -1;  // index of the launch whose start event was recorded
  std::vector<cudaEvent_t> start, stop;
  std::vector<int> kind;
} g_trace;

void trace_release() {
  for (auto e : g_trace.start) cudaEventDestroy(e);
  for (auto e : g_trace.stop) cudaEventDestroy(e);
  g_trace.start.clear();
  g_trace.stop.clear();
  g_trace.kind.clear();
  g_trace.max = g_trace.used = 0;
  g_trace.open = -1;
}
}  // namespace

void trace_begin(int kind, cudaStream_t st) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_trace.max == 0) return;
  std::lock_guard<std::mutex> lk(g_trace.mu);
  if (g_trace.used >= g_trace.max) return;
  const int i = g_trace.used;
  g_trace.kind[i] = kind;
  cudaEventRecord(g_trace.start[i], st);
  g_trace.open = i;
}

void count_extra_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void trace_end(int kind, cudaStream_t st) {
  if (g_trace.max == 0) return;
  std::lock_guard<std::mutex> lk(g_trace.mu);
  if (g_trace.open < 0 || g_trace.kind[g_trace.open] != kind) return;
  cudaEventRecord(g_trace.stop[g_trace.open], st);
  g_trace.used = g_trace.open + 1;
  g_trace.open = -1;
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
inline size_t dtype_size(int dt) { return dt == FLJSD_BF16 ? 2 : 4; }

struct Layout {
  int64_t ld, ntiles;
  size_t zs, zt, stats_s, stats_t, loss_rows, misc, acc32, total, logits_bytes, stats_bytes;
  bool use_acc32;
};

Layout layout_for(const fljsd_problem& p, int64_t chunk_rows) {
  Layout L{};
  L.ld = (p.v + 7) / 8 * 8;
  const size_t s = dtype_size(p.dtype);
  const size_t zbytes = align_up((size_t)chunk_rows * (size_t)L.ld * s);
  // per-row pass-1 partials of every 128 columns, written by the logits GEMMs
  L.ntiles = (p.v + TC_STATS_COLS - 1) / TC_STATS_COLS;
  const size_t sbytes = align_up((size_t)chunk_rows * (size_t)L.ntiles * sizeof(float2));
  L.zs = 0;
  L.zt = zbytes;
  L.stats_s = 2 * zbytes;
  L.stats_t = L.stats_s + sbytes;
  L.loss_rows = L.stats_t + sbytes;
  L.misc = L.loss_rows + align_up((size_t)p.bt * sizeof(float));
  // fp32 grad_weight accumulator: only when it changes anything
  L.use_acc32 = (p.flags & FLJSD_FLAG_ACCUM_FP32) && p.dtype == FLJSD_BF16 && chunk_rows < p.bt;
  L.acc32 = L.misc + kAlign;
  L.total = L.acc32 + (L.use_acc32 ? align_up((size_t)p.v * (size_t)p.h_s * sizeof(float)) : 0);
  L.logits_bytes = 2 * (size_t)chunk_rows * (size_t)L.ld * s;
  L.stats_bytes = 2 * sbytes + align_up((size_t)p.bt * sizeof(float)) + kAlign;
  return L;
}

fljsd_status check_problem(const fljsd_problem* p) {
  if (p == nullptr) return FLJSD_ERR_INVALID_ARG;
  if (p->bt <= 0 || p->h_s <= 0 || p->h_t <= 0 || p->v <= 0) return FLJSD_ERR_INVALID_ARG;
  if (p->dtype != FLJSD_F32 && p->dtype != FLJSD_BF16) return FLJSD_ERR_INVALID_ARG;
  if (p->reduction < FLJSD_RED_NONE || p->reduction > FLJSD_RED_BATCHMEAN)
    return FLJSD_ERR_INVALID_ARG;
  if (!(p->beta >= 0.f && p->beta <= 1.f)) return FLJSD_ERR_INVALID_ARG;  // also rejects NaN
  if (!(p->temperature > 0.f) || !std::isfinite(p->temperature)) return FLJSD_ERR_INVALID_ARG;
  if (p->chunk_rows < 0) return FLJSD_ERR_INVALID_ARG;
  if ((p->flags & ~(FLJSD_FLAG_T2 | FLJSD_FLAG_ACCUM_FP32)) != 0 || p->reserved != 0)
    return FLJSD_ERR_INVALID_ARG;
  // grid limits of the kernels (rows of a chunk and vocabulary tiles)
  if (p->v > (int64_t)1 << 30 || p->bt > (int64_t)1 << 30) return FLJSD_ERR_UNSUPPORTED;
  if (p->h_s > (int64_t)1 << 20 || p->h_t > (int64_t)1 << 20) return FLJSD_ERR_UNSUPPORTED;
  return FLJSD_OK;
}

inline bool aligned16(const void* q) { return ((uintptr_t)q & 15u) == 0; }

// One contraction D (+)= A . B^T of the path. Operand storage as in
// TcGemmArgs: a_mn / b_mn select an operand stored with the contraction
// dimension as its outer (row) dimension. bf16 goes to the tensor cores
// whenever the strides allow TMA (multiples of 8 elements); fp32 and the
// remaining bf16 shapes use the CUDA-core kernel.
// `stats` (optional) receives the per-row pass-1 partials of the output;
// *stats_done tells whether they were produced (the tensor-core path only).
cudaError_t run_gemm(int dtype, int kind, const void* a, int64_t lda, int a_mn, const void* b,
                     int64_t ldb, int b_mn, void* d, int64_t ldd, int64_t m, int64_t n, int64_t k,
                     int accumulate, int raster_n_fastest, int* status, cudaStream_t st,
                     float2* stats = nullptr, float stats_scale = 0.f,
                     bool* stats_done = nullptr, float* d32 = nullptr, int finalize = 0,
                     void* splitk_ws = nullptr, size_t splitk_bytes = 0) {
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

const char* fljsd_status_string(fljsd_status s) {
  switch (s) {
    case FLJSD_OK: return "ok";
    case FLJSD_ERR_INVALID_ARG: return "invalid argument";
    case FLJSD_ERR_UNSUPPORTED: return "unsupported problem";
    case FLJSD_ERR_WORKSPACE: return "workspace too small";
    case FLJSD_ERR_CUDA: return "CUDA error";
    case FLJSD_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

fljsd_status fljsd_plan(const fljsd_problem* p, size_t free_hbm_bytes, fljsd_plan_t* out) {
  fljsd_status st = check_problem(p);
  if (st != FLJSD_OK) return st;
  if (out == nullptr) return FLJSD_ERR_INVALID_ARG;
  int64_t c = 0;
  if (p->chunk_rows > 0) {
    c = p->chunk_rows < p->bt ? p->chunk_rows : p->bt;
  } else if (free_hbm_bytes == 0) {
    c = p->bt;
  } else {
    const size_t budget = free_hbm_bytes / 2;
    // One chunk first: it needs no fp32 grad_weight accumulator, which the
    // estimate below charges to every multi-chunk plan.
    int64_t fit = p->bt;
    if (layout_for(*p, p->bt).total > budget) {
      const Layout one = layout_for(*p, 1);
      const Layout zero = layout_for(*p, 0);
      const size_t per_row = one.total - zero.total;  // upper bound per row (alignment included)
      if (budget < one.total) return FLJSD_ERR_WORKSPACE;
      fit = (int64_t)((budget - zero.total) / (per_row > 0 ? per_row : 1));
      if (fit >= p->bt) fit = p->bt - 1;  // the one-chunk plan did not fit
    }
    if (fit >= p->bt) {
      c = p->bt;
    } else {
      c = fit / 128 * 128;
      if (c == 0) c = fit;
      while (c > 0 && layout_for(*p, c).total > budget) c -= (c > 128 ? 128 : 1);
      if (c <= 0) return FLJSD_ERR_WORKSPACE;
    }
  }
  const Layout L = layout_for(*p, c);
  out->chunk_rows = c;
  out->num_chunks = (p->bt + c - 1) / c;
  out->ld = L.ld;
  out->workspace_bytes = L.total;
  out->logits_bytes = L.logits_bytes;
  out->stats_bytes = L.stats_bytes;
  out->status_offset = L.misc + sizeof(int);
  return FLJSD_OK;
}

fljsd_status fljsd_forward(const fljsd_problem* p, const fljsd_plan_t* plan, const void* x_s,
                           const void* w_s, const void* x_t, const void* w_t,
                           const int64_t* labels, const float* row_grad, float* loss,
                           void* grad_input, void* grad_weight, void* workspace,
                           size_t workspace_bytes, fljsd_stream_t stream_) {
  fljsd_status st = check_problem(p);
  if (st != FLJSD_OK) return st;
  if (plan == nullptr) return FLJSD_ERR_INVALID_ARG;
  if (!x_s || !w_s || !x_t || !w_t || !loss || !grad_input || !grad_weight || !workspace)
    return FLJSD_ERR_INVALID_ARG;
  const void* ptrs[] = {x_s, w_s, x_t, w_t, loss, grad_input, grad_weight, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return FLJSD_ERR_INVALID_ARG;
  if ((labels && !aligned16(labels)) || (row_grad && !aligned16(row_grad)))
    return FLJSD_ERR_INVALID_ARG;
  const int64_t c = plan->chunk_rows;
  if (c <= 0 || c > p->bt || (p->chunk_rows > 0 && c != (p->chunk_rows < p->bt ? p->chunk_rows : p->bt)))
    return FLJSD_ERR_INVALID_ARG;
  const Layout L = layout_for(*p, c);
  if (plan->ld != L.ld || plan->workspace_bytes != L.total ||
      plan->num_chunks != (p->bt + c - 1) / c)
    return FLJSD_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return FLJSD_ERR_WORKSPACE;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  char* ws = static_cast<char*>(workspace);
  void* zs = ws + L.zs;
  void* zt = ws + L.zt;
  float* loss_rows = p->reduction == FLJSD_RED_NONE ? loss : reinterpret_cast<float*>(ws + L.loss_rows);
  int* n_valid = reinterpret_cast<int*>(ws + L.misc);
  int* status = n_valid + 1;  // device status word, reset by the row-count kernel
  float2* stats_s = reinterpret_cast<float2*>(ws + L.stats_s);
  float2* stats_t = reinterpret_cast<float2*>(ws + L.stats_t);
  float* acc32 = reinterpret_cast<float*>(ws + L.acc32);
  const size_t s = dtype_size(p->dtype);

  cudaError_t e = launch_count_valid(labels, p->bt, p->ignore_index, n_valid, stream);
  if (e != cudaSuccess) return FLJSD_ERR_CUDA;

  for (int64_t chunk = 0; chunk * c < p->bt; ++chunk) {
    const int64_t r0 = chunk * c;
    const int64_t rows = (p->bt - r0) < c ? (p->bt - r0) : c;
    const char* xs_c = static_cast<const char*>(x_s) + (size_t)r0 * p->h_s * s;
    const char* xt_c = static_cast<const char*>(x_t) + (size_t)r0 * p->h_t * s;

    // student and teacher logits, rounded to the input dtype (X . W^T, both K-major),
    // with the pass-1 partials of each row folded in the epilogue
    const float c2 = (float)(1.4426950408889634 / (double)p->temperature);
    bool st_s = false, st_t = false;
    e = run_gemm(p->dtype, FLJSD_KERNEL_GEMM_LOGITS, xs_c, p->h_s, 0, w_s, p->h_s, 0, zs, L.ld,
                 rows, p->v, p->h_s, 0, 0, status, stream, stats_s, c2, &st_s);
    if (e != cudaSuccess) return FLJSD_ERR_CUDA;
    e = run_gemm(p->dtype, FLJSD_KERNEL_GEMM_LOGITS, xt_c, p->h_t, 0, w_t, p->h_t, 0, zt, L.ld,
                 rows, p->v, p->h_t, 0, 0, status, stream, stats_t, c2, &st_t);
    if (e != cudaSuccess) return FLJSD_ERR_CUDA;

    // three passes over V; dlogits overwrite the student logits
    JsdRowArgs ra{};
    ra.zs = zs; ra.zt = zt; ra.ld = L.ld; ra.v = p->v; ra.rows = rows; ra.row0 = r0;
    ra.labels = labels; ra.ignore_index = p->ignore_index;
    ra.row_grad = p->reduction == FLJSD_RED_NONE ? row_grad : nullptr;
    ra.n_valid = n_valid; ra.loss_rows = loss_rows; ra.reduction = p->reduction;
    ra.beta = p->beta; ra.inv_temperature = 1.0f / p->temperature; ra.scale_log2 = c2;
    ra.loss_scale = (p->flags & FLJSD_FLAG_T2) ? p->temperature * p->temperature : 1.0f;
    // the partials are used only when both GEMMs produced them (same code path
    // for student and teacher, so equal logits give equal statistics)
    ra.stats_s = (st_s && st_t) ? stats_s : nullptr;
    ra.stats_t = (st_s && st_t) ? stats_t : nullptr;
    ra.ntiles = L.ntiles;
    e = launch_jsd_rows(p->dtype, ra, stream);
    if (e != cudaSuccess) return FLJSD_ERR_CUDA;

    // grad_input rows of this chunk = dZ . W_s (W_s stored [V x H]: B is N-major).
    // A chunk with too few output tiles for the GPU splits the V contraction;
    // the teacher logits are dead by now and hold the fp32 partials.
    e = run_gemm(p->dtype, FLJSD_KERNEL_GEMM_GRAD_INPUT, zs, L.ld, 0, w_s, p->h_s, 1,
                 static_cast<char*>(grad_input) + (size_t)r0 * p->h_s * s, p->h_s, rows, p->h_s,
                 p->v, 0, 1, status, stream, nullptr, 0.f, nullptr, nullptr, 0, zt,
                 L.logits_bytes / 2);
    if (e != cudaSuccess) return FLJSD_ERR_CUDA;

    // grad_weight (+)= dZ^T . X_s: both operands stored with the chunk rows as
    // the outer dimension (M-major A, N-major B); the first chunk overwrites
    const bool last = (r0 + rows >= p->bt);
    if (L.use_acc32) {
      // fp32 accumulator across chunks, rounded to the input dtype once
      e = run_gemm(p->dtype, FLJSD_KERNEL_GEMM_GRAD_WEIGHT, zs, L.ld, 1, xs_c, p->h_s, 1,
                   grad_weight, p->h_s, p->v, p->h_s, rows, chunk > 0 ? 1 : 0, 1, status, stream,
                   nullptr, 0.f, nullptr, acc32, last ? 1 : 0);
    } else {
      e = run_gemm(p->dtype, FLJSD_KERNEL_GEMM_GRAD_WEIGHT, zs, L.ld, 1, xs_c, p->h_s, 1,
                   grad_weight, p->h_s, p->v, p->h_s, rows, chunk > 0 ? 1 : 0, 1, status, stream);
    }
    if (e != cudaSuccess) return FLJSD_ERR_CUDA;
  }

  if (p->reduction != FLJSD_RED_NONE) {
    e = launch_reduce_loss(loss_rows, p->bt, p->v, p->reduction, n_valid, loss, stream);
    if (e != cudaSuccess) return FLJSD_ERR_CUDA;
  }
  return FLJSD_OK;
}

fljsd_status fljsd_backward(const fljsd_problem* p, const float* grad_output, void* grad_input,
                            void* grad_weight, fljsd_stream_t stream_) {
  fljsd_status st = check_problem(p);
  if (st != FLJSD_OK) return st;
  if (!grad_output || !grad_input || !grad_weight) return FLJSD_ERR_INVALID_ARG;
  if (!aligned16(grad_input) || !aligned16(grad_weight) || ((uintptr_t)grad_output & 3u))
    return FLJSD_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (launch_scale(p->dtype, grad_input, p->bt * p->h_s, grad_output, stream) != cudaSuccess)
    return FLJSD_ERR_CUDA;
  if (launch_scale(p->dtype, grad_weight, p->v * p->h_s, grad_output, stream) != cudaSuccess)
    return FLJSD_ERR_CUDA;
  return FLJSD_OK;
}

fljsd_status fljsd_workspace_status(const fljsd_plan_t* plan, const void* workspace,
                                    fljsd_stream_t stream_, int32_t* device_status) {
  if (!plan || !workspace || !device_status || plan->status_offset + 4 > plan->workspace_bytes)
    return FLJSD_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, static_cast<const char*>(workspace) + plan->status_offset, sizeof(v),
                      cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return FLJSD_ERR_CUDA;
  *device_status = v;
  return FLJSD_OK;
}

fljsd_status fljsd_gemm_bf16(const void* a, int64_t lda, int32_t a_mn, const void* b,
                             int64_t ldb, int32_t b_mn, void* d, int64_t ldd, int64_t m,
                             int64_t n, int64_t k, int32_t accumulate, int32_t* status,
                             int32_t flags, fljsd_stream_t stream_) {
  if ((flags & ~(FLJSD_GEMM_SINGLE_CTA | FLJSD_GEMM_TEST_STALL)) != 0)
    return FLJSD_ERR_INVALID_ARG;
  if (!a || !b || !d || m <= 0 || n <= 0 || k <= 0) return FLJSD_ERR_INVALID_ARG;
  if ((a_mn != 0 && a_mn != 1) || (b_mn != 0 && b_mn != 1) || (accumulate != 0 && accumulate != 1))
    return FLJSD_ERR_INVALID_ARG;
  if (lda < (a_mn ? m : k) || ldb < (b_mn ? n : k) || ldd < n) return FLJSD_ERR_INVALID_ARG;
  const bool stall = (flags & FLJSD_GEMM_TEST_STALL) != 0;
  TcGemmArgs t{a,       lda,  a_mn, b, ldb, b_mn, d, ldd, m, n, k, accumulate, 1, status,
               nullptr, 0.f,  nullptr, 0, stall ? 50ull * 1000 * 1000 : 0ull, stall ? 1 : 0};
  t.single_cta = (flags & FLJSD_GEMM_SINGLE_CTA) ? 1 : 0;
  if (!tc_gemm_supported(t)) return FLJSD_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  trace_begin(FLJSD_KERNEL_SMALL, stream);
  cudaError_t e = launch_gemm_tc(t, stream);
  trace_end(FLJSD_KERNEL_SMALL, stream);
  return e == cudaSuccess ? FLJSD_OK : FLJSD_ERR_CUDA;
}

size_t fljsd_rows_workspace_bytes(int64_t rows) {
  if (rows <= 0) return 0;
  return align_up((size_t)rows * sizeof(float)) + kAlign;
}

static fljsd_status dist_common(int64_t rows, int64_t v, int32_t dtype, int32_t reduction,
                                const void* x, const void* y, float* loss, void* grad,
                                void* workspace, size_t workspace_bytes) {
  if (rows <= 0 || v <= 0) return FLJSD_ERR_INVALID_ARG;
  if (rows > (int64_t)1 << 31 || v > (int64_t)1 << 31) return FLJSD_ERR_UNSUPPORTED;
  if (dtype != FLJSD_F32 && dtype != FLJSD_BF16) return FLJSD_ERR_INVALID_ARG;
  if (reduction < FLJSD_RED_NONE || reduction > FLJSD_RED_BATCHMEAN) return FLJSD_ERR_INVALID_ARG;
  if (!x || !y || !loss || !grad || !workspace) return FLJSD_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(grad) || !aligned16(workspace) ||
      ((uintptr_t)loss & 3u))
    return FLJSD_ERR_INVALID_ARG;
  if (workspace_bytes < fljsd_rows_workspace_bytes(rows)) return FLJSD_ERR_WORKSPACE;
  return FLJSD_OK;
}

fljsd_status fljsd_jsd_logspace(int64_t rows, int64_t v, int32_t dtype, float beta,
                                int32_t reduction, int64_t ignore_index, const void* input,
                                const void* target, const int64_t* labels, float* loss,
                                void* grad_input, void* workspace, size_t workspace_bytes,
                                fljsd_stream_t stream_) {
  fljsd_status st = dist_common(rows, v, dtype, reduction, input, target, loss, grad_input,
                                workspace, workspace_bytes);
  if (st != FLJSD_OK) return st;
  if (!(beta >= 0.f && beta <= 1.f)) return FLJSD_ERR_INVALID_ARG;
  if (labels && !aligned16(labels)) return FLJSD_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  char* ws = static_cast<char*>(workspace);
  float* loss_rows = reduction == FLJSD_RED_NONE ? loss : reinterpret_cast<float*>(ws);
  int* n_valid = reinterpret_cast<int*>(ws + align_up((size_t)rows * sizeof(float)));
  if (launch_count_valid(labels, rows, ignore_index, n_valid, stream) != cudaSuccess)
    return FLJSD_ERR_CUDA;
  DistArgs a{input, target, grad_input, rows, v, labels, ignore_index, n_valid, loss_rows,
             nullptr, reduction, beta};
  if (launch_jsd_logspace(dtype, a, stream) != cudaSuccess) return FLJSD_ERR_CUDA;
  if (reduction != FLJSD_RED_NONE &&
      launch_reduce_loss(loss_rows, rows, v, reduction, n_valid, loss, stream) != cudaSuccess)
    return FLJSD_ERR_CUDA;
  return FLJSD_OK;
}

fljsd_status fljsd_tvd(int64_t rows, int64_t v, int32_t dtype, int32_t reduction,
                       int64_t ignore_index, const void* p, const void* q, const int64_t* labels,
                       float* loss, void* grad_p, void* workspace, size_t workspace_bytes,
                       fljsd_stream_t stream_) {
  fljsd_status st = dist_common(rows, v, dtype, reduction, p, q, loss, grad_p, workspace,
                                workspace_bytes);
  if (st != FLJSD_OK) return st;
  if (labels && !aligned16(labels)) return FLJSD_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  char* ws = static_cast<char*>(workspace);
  float* loss_rows = reinterpret_cast<float*>(ws);
  int* n_valid = reinterpret_cast<int*>(ws + align_up((size_t)rows * sizeof(float)));
  if (launch_count_valid(labels, rows, ignore_index, n_valid, stream) != cudaSuccess)
    return FLJSD_ERR_CUDA;
  DistArgs a{p, q, grad_p, rows, v, labels, ignore_index, n_valid, loss_rows,
             reduction == FLJSD_RED_NONE ? loss : nullptr, reduction, 0.f};
  if (launch_tvd(dtype, a, stream) != cudaSuccess) return FLJSD_ERR_CUDA;
  if (reduction != FLJSD_RED_NONE &&
      launch_reduce_loss(loss_rows, rows, v, reduction, n_valid, loss, stream) != cudaSuccess)
    return FLJSD_ERR_CUDA;
  return FLJSD_OK;
}

fljsd_status fljsd_scale(int32_t dtype, void* x, int64_t n, const float* grad_output,
                         fljsd_stream_t stream_) {
  if ((dtype != FLJSD_F32 && dtype != FLJSD_BF16) || !x || !grad_output || n < 0)
    return FLJSD_ERR_INVALID_ARG;
  if (!aligned16(x) || ((uintptr_t)grad_output & 3u)) return FLJSD_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  return launch_scale(dtype, x, n, grad_output, stream) == cudaSuccess ? FLJSD_OK
                                                                      : FLJSD_ERR_CUDA;
}

int64_t fljsd_launch_count(void) { return g_launches.load(); }
void fljsd_launch_count_reset(void) { g_launches.store(0); }

fljsd_status fljsd_trace_enable(int32_t max_launches) {
  std::lock_guard<std::mutex> lk(g_trace.mu);
  trace_release();
  if (max_launches < 0) return FLJSD_ERR_INVALID_ARG;
  if (max_launches == 0) return FLJSD_OK;
  g_trace.start.resize(max_launches);
  g_trace.stop.resize(max_launches);
  g_trace.kind.assign(max_launches, -1);
  for (int i = 0; i < max_launches; ++i) {
    if (cudaEventCreate(&g_trace.start[i]) != cudaSuccess ||
        cudaEventCreate(&g_trace.stop[i]) != cudaSuccess) {
      g_trace.start.resize(i);
      g_trace.stop.resize(i);
      trace_release();
      return FLJSD_ERR_CUDA;
    }
  }
  g_trace.max = max_launches;
  return FLJSD_OK;
}

fljsd_status fljsd_trace_reset(void) {
  std::lock_guard<std::mutex> lk(g_trace.mu);
  g_trace.used = 0;
  g_trace.open = -1;
  return FLJSD_OK;
}

fljsd_status fljsd_trace_read(int32_t kind, double* total_ms, int64_t* launches) {
  if (!total_ms || !launches || kind < 0 || kind >= FLJSD_KERNEL_NUM_KINDS)
    return FLJSD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_trace.mu);
  double tot = 0.0;
  int64_t n = 0;
  for (int i = 0; i < g_trace.used; ++i) {
    if (g_trace.kind[i] != kind) continue;
    if (cudaEventSynchronize(g_trace.stop[i]) != cudaSuccess) return FLJSD_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_trace.start[i], g_trace.stop[i]) != cudaSuccess)
      return FLJSD_ERR_CUDA;
    tot += ms;
    ++n;
  }
  *total_ms = tot;
  *launches = n;
  return FLJSD_OK;
}

}  // extern "C"
