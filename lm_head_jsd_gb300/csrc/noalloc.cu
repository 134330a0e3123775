// fljsd_forward_noalloc: the fused-linear JSD forward for callers that cannot
// allocate device memory -- for example code running inside a host framework
// that owns every device allocation and hands a plugin only its input and
// output buffers, so there is nowhere to get a workspace from. The scratch the
// forward needs (the two logits buffers of one chunk, the per-row losses, the
// valid-row count and the status word) lives in a file-scope device array of
// fixed size instead of a caller-provided workspace.
//
// Costs and limits, for the user of this entry point:
//  - the array is kNoAllocScratchBytes (64 MiB) on every GPU that loads the
//    library, held until the process exits, whether or not this entry point
//    is ever called;
//  - every call shares that one array, so calls whose work overlaps on the
//    GPU (on different streams, or from different host threads) race and
//    corrupt each other's results; serialise them;
//  - the chunk is limited to what fits: rows of 2 * ceil8(V) * sizeof(dtype)
//    bytes each, plus 4 bytes per row of the whole batch for the losses;
//    problems that do not fit even one row are rejected.
// Nothing in the array needs to start at zero: every byte a call reads is
// written earlier in the same call (the first kernel resets the count and the
// status word), so the contents a previous call left behind do no harm.
#include "internal.cuh"

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;

static __device__ __align__(256) unsigned char g_fljsd_scratch[kNoAllocScratchBytes];

// In host code g_fljsd_scratch names a host-side stand-in, not device memory,
// so its device address is looked up once per device, with that device
// current, and cached.
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

fljsd_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLJSD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FLJSD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fljsd_scratch) != cudaSuccess || p == nullptr)
      return FLJSD_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FLJSD_OK;
}

bool aligned16(const void* q) { return ((uintptr_t)q & 15u) == 0; }

}  // namespace

extern "C" fljsd_status fljsd_forward_noalloc(const fljsd_problem* problem, const void* x_s,
                                              const void* w_s, const void* x_t, const void* w_t,
                                              const int64_t* labels, const float* row_grad,
                                              float* loss, void* grad_input, void* grad_weight,
                                              fljsd_stream_t stream) {
  if (problem == nullptr) return FLJSD_ERR_INVALID_ARG;
  if (!x_s || !w_s || !x_t || !w_t || !loss || !grad_input || !grad_weight)
    return FLJSD_ERR_INVALID_ARG;
  const void* ptrs[] = {x_s, w_s, x_t, w_t, loss, grad_input, grad_weight};
  for (const void* q : ptrs)
    if (!aligned16(q)) return FLJSD_ERR_INVALID_ARG;

  // Chunk geometry that fits the fixed array: the planner given twice the
  // array size uses at most the array size.
  fljsd_plan_t plan;
  fljsd_status st;
  if (problem->chunk_rows > 0) {
    st = fljsd_plan(problem, 0, &plan);
    if (st == FLJSD_OK && plan.workspace_bytes > kNoAllocScratchBytes) return FLJSD_ERR_WORKSPACE;
  } else {
    st = fljsd_plan(problem, 2 * kNoAllocScratchBytes, &plan);
  }
  if (st != FLJSD_OK) return st;  // FLJSD_ERR_WORKSPACE: not even one row fits

  void* scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != FLJSD_OK) return st;
  fljsd_problem p = *problem;
  p.chunk_rows = plan.chunk_rows;
  return fljsd_forward(&p, &plan, x_s, w_s, x_t, w_t, labels, row_grad, loss, grad_input,
                       grad_weight, scratch, kNoAllocScratchBytes, stream);
}
