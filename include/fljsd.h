/*
 * fljsd.h -- C ABI of the GB300 (sm_103a) fused-linear Jensen-Shannon
 * distillation loss.
 *
 * What the library computes (Liger-Kernel pull requests, cited by title):
 *
 *  - "[Perf] Fuse log-softmax into fused_linear_jsd kernel" (PR 1352),
 *    "Summary" and "Details": for a chunk of C rows, the student logits
 *    Z_s = X_s . W_s^T and the teacher logits Z_t = X_t . W_t^T are formed in
 *    the input dtype; the temperature-scaled log-softmaxes of both come from a
 *    three-pass online softmax over V (pass 1: running max m and denominator d
 *    for student and teacher together; pass 2: per-row loss and the
 *    cross-column term dX_sum; pass 3: the logit gradient dZ written in place
 *    over the student logits buffer). All math after the GEMM is fp32.
 *  - Same page, "Testing Done": beta == 0 is forward KL(P||Q), beta == 1 is
 *    reverse KL(Q||P), anything between is the generalized JSD
 *    beta*KL(P||M) + (1-beta)*KL(Q||M), M = beta*P + (1-beta)*Q, with P the
 *    teacher and Q the student distribution.
 *  - Same page, "Open questions" 2: the temperature divides the logits once.
 *  - "Fix TVD gradient at p == q" (PR 1374), "Summary": an element where the
 *    student and teacher log-probabilities tie contributes exactly zero.
 *  - "perf(flce): write the weight-gradient product directly into
 *    grad_weight" (PR 1429), "Summary" and "Changes": grad_input = dZ . W_s per
 *    chunk and grad_weight = sum over chunks of dZ^T . X_s, written straight
 *    into grad_weight; the first chunk overwrites (beta = 0), later chunks add
 *    the fp32 product to the stored value and round once; the outputs may be
 *    uninitialised (empty_like) because every element is written.
 *
 * Conventions for every entry point:
 *  - Matrices are dense, row-major, contiguous. Element type is given by
 *    fljsd_problem.dtype for X_s, W_s, X_t, W_t, grad_input and grad_weight.
 *  - Device pointers are caller-owned; the library allocates and frees no
 *    device memory. Every device pointer must be 16-byte aligned.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream). Argument checks are synchronous: on any error status
 *    nothing has been launched, except FLJSD_ERR_CUDA, which reports a launch
 *    failure after earlier launches of the same call may have been queued.
 *  - Not re-entrant across threads for the same workspace; distinct
 *    workspaces on distinct streams may run concurrently.
 */
#ifndef FLJSD_H
#define FLJSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st* fljsd_stream_t;

typedef enum {
  FLJSD_OK = 0,
  FLJSD_ERR_INVALID_ARG = 1, /* null pointer, bad size, beta or temperature, misalignment */
  FLJSD_ERR_UNSUPPORTED = 2, /* valid but beyond the kernels' size limits (stated per call) */
  FLJSD_ERR_WORKSPACE = 3,   /* workspace smaller than the plan requires */
  FLJSD_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  FLJSD_ERR_TIMEOUT = 5      /* a bounded device-side wait expired */
} fljsd_status;

typedef enum { FLJSD_F32 = 0, FLJSD_BF16 = 1 } fljsd_dtype;

/* Reductions. The pages name four (PR 1374, "Details") and fix "batchmean"
 * as division by the number of rows (PR 1374, tie table). n = number of rows
 * whose label != ignore_index (BT when labels is NULL).
 *   NONE:      loss[r] = L_r (0 for ignored rows); gradients are those of
 *              sum_r row_grad[r] * L_r (row_grad NULL means all ones).
 *   SUM:       loss = sum_r L_r.
 *   MEAN:      loss = sum_r L_r / (n * V).
 *   BATCHMEAN: loss = sum_r L_r / n.
 * With n == 0 the loss and both gradients are 0. */
typedef enum {
  FLJSD_RED_NONE = 0,
  FLJSD_RED_SUM = 1,
  FLJSD_RED_MEAN = 2,
  FLJSD_RED_BATCHMEAN = 3
} fljsd_reduction;

typedef struct {
  int64_t bt;           /* rows (batch * sequence) */
  int64_t h_s;          /* student hidden size */
  int64_t h_t;          /* teacher hidden size */
  int64_t v;            /* vocabulary size */
  int32_t dtype;        /* fljsd_dtype of X_s, W_s, X_t, W_t and the gradients */
  int32_t reduction;    /* fljsd_reduction */
  float beta;           /* in [0, 1]; 0 and 1 select the KL endpoints exactly */
  float temperature;    /* > 0 and finite; logits are divided by it once */
  int64_t ignore_index; /* label value of rows that are skipped (Liger: -100) */
  int64_t chunk_rows;   /* rows per chunk; 0 lets fljsd_plan choose */
  int32_t flags;        /* FLJSD_FLAG_* bits, 0 for the pages' behaviour */
  int32_t reserved;     /* must be 0 */
} fljsd_problem;

/* Opt-in behaviours (none of them is the pages' default).
 * FLJSD_FLAG_T2: multiply the loss and both gradients by T^2 (Hinton et al.
 *   2015); the pages divide by T once and leave this to the caller
 *   ("[Perf] Fuse log-softmax into fused_linear_jsd kernel", Open questions 2).
 * FLJSD_FLAG_ACCUM_FP32: with bf16 inputs and more than one chunk, accumulate
 *   grad_weight across chunks in an fp32 buffer inside the workspace
 *   (V * h_s * 4 bytes) and round it to bf16 once after the last chunk, as
 *   the accum_dtype=float32 option of "perf(flce): write the weight-gradient
 *   product directly into grad_weight" (PR 1429) does; without it every chunk
 *   after the first rounds the running sum to bf16. */
#define FLJSD_FLAG_T2 1
#define FLJSD_FLAG_ACCUM_FP32 2

typedef struct {
  int64_t chunk_rows;     /* C: rows of one chunk */
  int64_t num_chunks;     /* ceil(bt / C) */
  int64_t ld;             /* row stride (elements) of the logits buffers, >= v */
  size_t workspace_bytes; /* device bytes fljsd_forward needs */
  size_t logits_bytes;    /* 2 * C * ld * sizeof(dtype): the two logits buffers */
  size_t stats_bytes;     /* per-row and per-tile statistics */
  size_t status_offset;   /* byte offset of the int32 device status word in the workspace */
} fljsd_plan_t;

/*
 * fljsd_plan -- choose the chunk geometry and size the workspace.
 *
 * If problem->chunk_rows > 0 it is used (clamped to bt). Otherwise the largest
 * chunk whose workspace fits in half of `free_hbm_bytes` is taken (a multiple
 * of 128 rows unless it is all of bt); free_hbm_bytes == 0 means "no limit",
 * i.e. one chunk. The pages found one chunk fastest and the fixed
 * cdiv(V, H) heuristic mis-tuned for JSD (PR 1352, "Open questions" 4); live
 * memory per chunk is the two logits tensors, 2 * C * V * s bytes (PR 1352,
 * "Details", memory table), plus O(C) statistics and the (BT,) loss vector.
 * Host only; launches nothing. Returns FLJSD_ERR_INVALID_ARG for a bad
 * problem, FLJSD_ERR_UNSUPPORTED for shapes the kernels do not handle (bt or
 * v above 2^30, h_s or h_t above 2^20), and FLJSD_ERR_WORKSPACE if not even
 * one row fits.
 */
fljsd_status fljsd_plan(const fljsd_problem* problem, size_t free_hbm_bytes,
                        fljsd_plan_t* out);

/*
 * fljsd_forward -- loss and both gradients (upstream gradient 1).
 *
 *   x_s [bt x h_s], w_s [v x h_s], x_t [bt x h_t], w_t [v x h_t]: inputs
 *       (device, dtype; never modified). The teacher is frozen: no teacher
 *       gradient is produced.
 *   labels [bt] int64 (device) or NULL: rows with label == ignore_index are
 *       skipped.
 *   row_grad [bt] fp32 (device) or NULL: upstream per-row gradient, used only
 *       with FLJSD_RED_NONE (NULL = ones).
 *   loss (device fp32): [1] for SUM, MEAN, BATCHMEAN; [bt] for NONE.
 *   grad_input [bt x h_s] (device, dtype): d loss / d x_s.
 *   grad_weight [v x h_s] (device, dtype): d loss / d w_s.
 *   workspace (device), workspace_bytes >= plan->workspace_bytes.
 *
 * Every element of loss, grad_input and grad_weight is written. `plan` must
 * come from fljsd_plan for the same problem.
 */
fljsd_status fljsd_forward(const fljsd_problem* problem, const fljsd_plan_t* plan,
                           const void* x_s, const void* w_s, const void* x_t,
                           const void* w_t, const int64_t* labels, const float* row_grad,
                           float* loss, void* grad_input, void* grad_weight,
                           void* workspace, size_t workspace_bytes, fljsd_stream_t stream);

/*
 * fljsd_forward_noalloc -- fljsd_forward for callers that cannot allocate
 * device memory (e.g. a plugin inside a host framework that owns every
 * device allocation and passes in only input and output buffers). The pages
 * have no counterpart of this entry point; it is an addition of this library.
 *
 * Arguments are those of fljsd_forward without plan and workspace: the
 * scratch lives in a fixed 64 MiB device array inside the library, which
 * every GPU that loads the library holds until the process exits.
 *   - The chunk rows are chosen to fit that array (problem->chunk_rows, if
 *     > 0, must fit it). A problem whose scratch does not fit even one row
 *     (2 * ceil8(v) * sizeof(dtype) bytes per row, plus 4 * bt bytes) returns
 *     FLJSD_ERR_WORKSPACE before anything is launched.
 *   - Every call shares the one array: calls whose work overlaps on the GPU
 *     (different streams, different host threads) race; serialise them.
 *     Nothing in the array has to start at zero: a call writes every byte it
 *     reads, so what the previous call left there does not matter.
 *   - The first call on a device (the current device) looks up the array's
 *     device address with the CUDA runtime and caches it; make that first
 *     call before any stream capture. It calls no cudaMalloc or cudaFree.
 * Returns what fljsd_forward returns, and FLJSD_ERR_CUDA if the address
 * lookup fails.
 */
fljsd_status fljsd_forward_noalloc(const fljsd_problem* problem, const void* x_s,
                                   const void* w_s, const void* x_t, const void* w_t,
                                   const int64_t* labels, const float* row_grad, float* loss,
                                   void* grad_input, void* grad_weight, fljsd_stream_t stream);

/*
 * fljsd_backward -- scale the gradients computed by fljsd_forward by the
 * upstream scalar gradient *grad_output (device fp32), in place, on `stream`.
 * The forward already holds the gradients for an upstream gradient of 1
 * (PR 1352, "Details": the gradient is written during the forward pass), so
 * this is one elementwise pass over grad_input [bt x h_s] and grad_weight
 * [v x h_s] that does nothing when *grad_output == 1.
 */
fljsd_status fljsd_backward(const fljsd_problem* problem, const float* grad_output,
                            void* grad_input, void* grad_weight, fljsd_stream_t stream);

/*
 * fljsd_workspace_status -- the device status word of the last fljsd_forward
 * that used `workspace` (FLJSD_OK, or FLJSD_ERR_TIMEOUT if a bounded wait
 * inside a kernel expired). Synchronises `stream`, then copies 4 bytes to
 * the host into *device_status. Returns FLJSD_ERR_CUDA if the copy fails.
 */
fljsd_status fljsd_workspace_status(const fljsd_plan_t* plan, const void* workspace,
                                    fljsd_stream_t stream, int32_t* device_status);

/*
 * fljsd_gemm_bf16 -- the tensor-core contraction used by the path, exposed
 * as a building block: D[m x n] = A . B^T (accumulate == 0) or
 * D = D + A . B^T (accumulate == 1; the stored value and the fp32 product
 * are added and rounded once, as for grad_weight in PR 1429, "Summary").
 *   a_mn == 0: A stored [m x k] row-major with row stride lda (k contiguous);
 *   a_mn == 1: A stored [k x m] row-major with row stride lda (m contiguous);
 *   b_mn == 0: B stored [n x k]; b_mn == 1: B stored [k x n] (stride ldb);
 *   D stored [m x ldd]. All bf16, device, 16-byte aligned; lda, ldb, ldd
 *   multiples of 8; m, n, k >= 1.
 * status: device int32 that receives FLJSD_ERR_TIMEOUT if a bounded wait
 * expires (may be NULL). flags: 0, FLJSD_GEMM_SINGLE_CTA or
 * FLJSD_GEMM_TEST_STALL (below).
 * Asynchronous on `stream`. FLJSD_ERR_INVALID_ARG for
 * shapes or alignments outside the above.
 */
fljsd_status fljsd_gemm_bf16(const void* a, int64_t lda, int32_t a_mn, const void* b,
                             int64_t ldb, int32_t b_mn, void* d, int64_t ldd, int64_t m,
                             int64_t n, int64_t k, int32_t accumulate, int32_t* status,
                             int32_t flags, fljsd_stream_t stream);
/* flags of fljsd_gemm_bf16: by default, for contractions at least 256 deep,
 * pairs of 128-row blocks of D run as CTA pairs (2-CTA clusters,
 * tcgen05.mma.cta_group::2) that compute a 256 x 256 tile together, each CTA
 * copying only its own rows of A and half of the B tile, unless the pairs
 * would need more than 12% more waves of tiles over the GPU than one CTA per
 * tile (an odd block count leaves a pair half empty; few tiles can add a
 * wave);
 * FLJSD_GEMM_SINGLE_CTA runs one CTA per 128 x 256 tile. The results are
 * identical. The environment variable FLJSD_GEMM_PAIR (read at each launch)
 * selects for every GEMM of the library: 0 one CTA per tile, 2 CTA pairs at
 * any contraction depth. */
#define FLJSD_GEMM_SINGLE_CTA 1
/* Test of the failure path: the kernel's copy warp issues nothing, so its
 * first bounded wait expires after 50 ms; *status then holds
 * FLJSD_ERR_TIMEOUT, D is not written, and the context stays usable. */
#define FLJSD_GEMM_TEST_STALL 2

/*
 * Distances over given distributions (no GEMM). Both take [rows x v] row-major
 * tensors of `dtype`, optional int64 labels [rows] (rows whose label equals
 * ignore_index give loss 0 and gradient 0; n = the other rows), a reduction
 * as for fljsd_forward (none / sum / mean = / (n v) / batchmean = / n), and a
 * device workspace of fljsd_rows_workspace_bytes(rows) bytes. They return the
 * gradient for an upstream gradient of 1 (fljsd_scale applies another).
 *
 * fljsd_jsd_logspace -- the generalized JSD on log-probabilities, the public
 * contract of Liger's _jsd_kernel ("[Perf] Fuse log-softmax into
 * fused_linear_jsd kernel", PR 1352, Open questions 3): input = X = log Q
 * (student), target = Y = log P (teacher); per element beta*P*(Y - log M) +
 * (1-beta)*Q*(X - log M) with M = beta*P + (1-beta)*Q, forward KL P*(Y - X) at
 * beta == 0, reverse KL Q*(X - Y) at beta == 1; ties (X == Y) contribute 0.
 * grad_input = d loss / d X element by element (inputs are not renormalised,
 * so no softmax Jacobian): (1-beta)*Q*(X - log M), -P at beta == 0,
 * Q*(X - Y + 1) at beta == 1, times the reduction weight. loss: [1], or [rows]
 * for reduction none.
 *
 * fljsd_tvd -- total variation distance with the tie fix of "Fix TVD
 * gradient at p == q" (PR 1374, Summary): per element 0.5*|p - q|, gradient
 * in p = 0.5 * sign(p - q) * (reduction weight) with sign(0) = 0. loss: [1],
 * or [rows x v] fp32 per element for reduction none.
 *
 * fljsd_scale -- x *= *grad_output in place (device fp32 scalar), skipped on
 * the device when it is 1: the backward of the two functions above.
 *
 * Errors (checked on the host before anything is launched):
 * FLJSD_ERR_INVALID_ARG for rows or v <= 0, an unknown dtype or reduction, beta
 * outside [0, 1], a null input, target, loss, gradient or workspace pointer, or
 * one not 16-byte aligned (loss: 4 bytes; labels, when given: 16 bytes);
 * FLJSD_ERR_UNSUPPORTED for rows or v above 2^31; FLJSD_ERR_WORKSPACE for a
 * workspace below fljsd_rows_workspace_bytes(rows); FLJSD_ERR_CUDA when a
 * launch fails. fljsd_scale: FLJSD_ERR_INVALID_ARG for an unknown dtype, n < 0,
 * or a null or unaligned pointer.
 */
size_t fljsd_rows_workspace_bytes(int64_t rows);
fljsd_status fljsd_jsd_logspace(int64_t rows, int64_t v, int32_t dtype, float beta,
                                int32_t reduction, int64_t ignore_index, const void* input,
                                const void* target, const int64_t* labels, float* loss,
                                void* grad_input, void* workspace, size_t workspace_bytes,
                                fljsd_stream_t stream);
fljsd_status fljsd_tvd(int64_t rows, int64_t v, int32_t dtype, int32_t reduction,
                       int64_t ignore_index, const void* p, const void* q, const int64_t* labels,
                       float* loss, void* grad_p, void* workspace, size_t workspace_bytes,
                       fljsd_stream_t stream);
fljsd_status fljsd_scale(int32_t dtype, void* x, int64_t n, const float* grad_output,
                         fljsd_stream_t stream);

/*
 * Fused linear cross-entropy (FLCE): loss = CE(x . w^T, labels) and its
 * gradients in x and w, on the same GEMMs, chunk planner and grad_weight
 * contract as fljsd_forward ("perf(flce): write the weight-gradient product
 * directly into grad_weight", PR 1429: first chunk overwrites, later chunks add
 * in fp32 and round once, or accumulate in fp32 with FLJSD_FLAG_ACCUM_FP32).
 * Per row with label y and logits z (c = softcap * tanh(z / softcap) when
 * softcap > 0, else c = z), lse = log sum_j e^{c_j}:
 *   L = lse - (1 - eps) c_y - (eps / V) sum_j c_j + lse_square_scale * lse^2
 * (eps = label_smoothing). Reductions: none -> [bt] per-row losses; sum;
 * mean and batchmean -> divided by the number of rows whose label is not
 * ignore_index. Labels are required (int64 [bt], device); a label outside
 * [0, v) that is not ignore_index makes its row contribute 0 and sets the
 * workspace status word to FLJSD_ERR_INVALID_ARG (fljsd_workspace_status).
 * x [bt x h], w [v x h], grad_input [bt x h], grad_weight [v x h] in dtype.
 * Gradients are for an upstream gradient of 1 (fljsd_scale applies another).
 *
 * fljsd_ce_plan / fljsd_ce_forward follow fljsd_plan / fljsd_forward: every
 * pointer is caller-owned device memory, 16-byte aligned (loss 4 bytes);
 * grad_input and grad_weight are written in full and may be uninitialised; the
 * workspace (plan->workspace_bytes, device, caller-owned) holds the logits of
 * one chunk and the per-row statistics; the forward is asynchronous on
 * `stream`. Errors, checked on the host before anything is launched:
 * FLJSD_ERR_INVALID_ARG for a dimension <= 0, an unknown dtype, reduction or
 * flag, label_smoothing outside [0, 1], a negative or non-finite
 * lse_square_scale or softcap, or a null or unaligned pointer;
 * FLJSD_ERR_UNSUPPORTED for bt or v above 2^30 or h above 2^20;
 * FLJSD_ERR_WORKSPACE when the workspace is smaller than the plan's (or, in
 * fljsd_ce_plan, when not even one row fits the budget); FLJSD_ERR_CUDA when a
 * launch fails.
 */
typedef struct {
  int64_t bt, h, v;
  int32_t dtype;          /* fljsd_dtype */
  int32_t reduction;      /* fljsd_reduction */
  int64_t ignore_index;
  int64_t chunk_rows;     /* 0 lets fljsd_ce_plan choose */
  float label_smoothing;  /* in [0, 1] */
  float lse_square_scale; /* z-loss coefficient, >= 0 */
  float softcap;          /* 0 disables the tanh cap */
  int32_t flags;          /* FLJSD_FLAG_ACCUM_FP32 or 0 */
} fljsd_ce_problem;

fljsd_status fljsd_ce_plan(const fljsd_ce_problem* problem, size_t free_hbm_bytes,
                           fljsd_plan_t* out);
fljsd_status fljsd_ce_forward(const fljsd_ce_problem* problem, const fljsd_plan_t* plan,
                              const void* x, const void* w, const int64_t* labels, float* loss,
                              void* grad_input, void* grad_weight, void* workspace,
                              size_t workspace_bytes, fljsd_stream_t stream);

/* Static, human-readable name of a status code. Never NULL. */
const char* fljsd_status_string(fljsd_status status);

/*
 * Launch accounting and per-kernel timing (for benchmarks).
 *
 * fljsd_launch_count returns the number of kernels this library has launched
 * in the process (all devices, all streams) since load or the last
 * fljsd_launch_count_reset.
 *
 * fljsd_trace_enable(max_launches) turns on per-launch CUDA-event timing on
 * the launching stream for up to max_launches launches (events are created on
 * the current device); fljsd_trace_enable(0) turns it off and releases the
 * events. fljsd_trace_read synchronises the recorded events and returns, for
 * kernel class `kind` (FLJSD_KERNEL_*), the summed milliseconds and the number
 * of recorded launches; fljsd_trace_reset forgets the recorded launches.
 * These are process-global and not thread-safe.
 */
typedef enum {
  FLJSD_KERNEL_GEMM_LOGITS = 0,      /* Z = X . W^T, student and teacher */
  FLJSD_KERNEL_JSD_ROWS = 1,         /* the three passes over V */
  FLJSD_KERNEL_GEMM_GRAD_INPUT = 2,  /* dZ . W_s */
  FLJSD_KERNEL_GEMM_GRAD_WEIGHT = 3, /* dZ^T . X_s into grad_weight */
  FLJSD_KERNEL_SMALL = 4,            /* row count, loss reduction, scaling */
  FLJSD_KERNEL_NUM_KINDS = 5
} fljsd_kernel_kind;

int64_t fljsd_launch_count(void);
void fljsd_launch_count_reset(void);
fljsd_status fljsd_trace_enable(int32_t max_launches);
fljsd_status fljsd_trace_reset(void);
fljsd_status fljsd_trace_read(int32_t kind, double* total_ms, int64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* FLJSD_H */
