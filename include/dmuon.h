/*
 * dmuon.h -- C ABI of the DMuon owner-side Muon step on one GB300 (sm_103a).
 *
 * What the library computes (DMuon home page, "What DMuon Can Do" / "LLM
 * Pretraining"; "Z2 vs Z3 Modes", "The two packed-buffer lifecycles"): the
 * owner of a set of 2-D projection matrices runs, once per step,
 *   1. Nesterov momentum on each gradient and packs the result (bf16) into one
 *      contiguous per-owner buffer;
 *   2. one Newton-Schulz orthogonalisation of every packed matrix (home page,
 *      owner section: each matrix is orthogonalised once, by its owner);
 *   3. the scaled weight update.
 * The pages name Muon and Newton-Schulz but do not write them out; the library
 * uses the standard Muon forms:
 *   M <- beta*M + (1-beta)*G,   U = (1-beta)*G + beta*M
 *   X = U^T if rows > cols else U,   X0 = X / (||X||_F + eps)
 *   ns_steps times: A = X X^T;  B = b*A + c*A*A;  X = a*X + B*X
 *   O = X^T if transposed else X
 *   W <- W - lr * sqrt(max(1, rows/cols)) * O
 * with (a, b, c) = (3.4445, -4.7750, 2.0315) and eps = 1e-7 by default.
 * The Gram variant (home page, "VLA and VLM": Gram Newton-Schulz) iterates on
 * the m x m Gram matrix and gives the same result in exact arithmetic.
 *
 * Conventions shared by every call:
 *  - A matrix is a PyTorch parameter of shape (rows, cols) = (out, in),
 *    row-major and contiguous.  m = min(rows, cols), n = max(rows, cols).
 *  - Every tensor pointer is a DEVICE pointer owned by the caller.  The
 *    arrays that hold those pointers (grad[], momentum[], weight[]) and the
 *    shape / offset arrays are HOST arrays, read during the call only.
 *  - The library allocates no memory.  All scratch lives in the caller's
 *    `workspace` (size from dmuon_workspace_bytes, 256-byte aligned); the
 *    library writes its tables there with a small kernel on `stream` whose
 *    parameters carry the bytes (no host staging buffer, no pageable copy).
 *  - Calls are asynchronous on `stream`.  Arguments are checked on the host
 *    before anything is enqueued; a bad argument returns an error and
 *    launches nothing.  A call that launches work first clears a pending
 *    (non-sticky) CUDA error left by earlier work of the calling thread, so
 *    that DMUON_ERR_CUDA reports only its own failures.  Device-side failures (a bounded wait that gave up)
 *    are recorded in the workspace and reported by dmuon_stream_status.
 *  - Results are deterministic: the same inputs give bit-identical outputs
 *    (no floating-point atomics; fixed reduction orders).
 *  - NaN / Inf in the inputs propagate; nothing is clamped.  An all-zero
 *    gradient gives O = 0, so W is unchanged.
 *  - Calls that share a workspace must not overlap on the GPU.
 *  - Tensors of one call must not overlap each other (gradients, momenta,
 *    weights, the packed buffer and the workspace are distinct memory).
 */
#ifndef DMUON_H
#define DMUON_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every call. */
typedef enum {
  DMUON_OK = 0,
  DMUON_ERR_INVALID_ARG = -1,  /* null pointer, bad size, bad enum, ns_steps < 0 ... */
  DMUON_ERR_ALIGNMENT = -2,    /* packed / workspace not 256-byte aligned */
  DMUON_ERR_WORKSPACE = -3,    /* ws_bytes < dmuon_workspace_bytes(...) */
  DMUON_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed */
  DMUON_ERR_TIMEOUT = -5,      /* a bounded device wait gave up (dmuon_stream_status) */
  DMUON_ERR_UNSUPPORTED = -6   /* device is not sm_103 / shape beyond limits */
} dmuon_status;

/* Element types of caller tensors. */
typedef enum { DMUON_F32 = 0, DMUON_BF16 = 1 } dmuon_dtype;

/*
 * Newton-Schulz variant.
 *   DMUON_NS_STANDARD  the standard iteration on every matrix.
 *   DMUON_NS_GRAM      the Gram iteration on each matrix where it saves work
 *                      (n > m, ns_steps >= 2) AND the library's accuracy rule
 *                      admits it for that aspect ratio n/m and step count (see
 *                      dmuon_ns_variant_for); the standard one elsewhere.
 *   DMUON_NS_GRAM_ALL  the Gram iteration on every matrix with n > m, without
 *                      the accuracy rule -- for measuring that rule.  Near-square
 *                      matrices can come out far outside the Newton-Schulz
 *                      tolerance (bf16 loses the squared small singular values).
 */
typedef enum { DMUON_NS_STANDARD = 0, DMUON_NS_GRAM = 1, DMUON_NS_GRAM_ALL = 2 } dmuon_ns_variant;

/* Shape of one parameter: PyTorch (out, in) = (rows, cols). */
typedef struct { int64_t rows, cols; } dmuon_shape;

/* Largest accepted m = min(rows, cols) and n = max(rows, cols). */
#define DMUON_MAX_M 32768
#define DMUON_MAX_N 1048576
/* Element alignment of packed segments: 256 bytes of bf16. */
#define DMUON_PACK_ALIGN_ELEMS 128

/*
 * dmuon_plan -- host-only owner assignment and packing offsets.
 * Home page, "MoE": each matrix gets one owner and the partition is balanced
 * so that no rank straggles; "Z2 vs Z3 Modes": the matrices of one owner share
 * one contiguous buffer.  Reading: greedy LPT by element count (descending
 * size, ties to the lower index; least-loaded owner, ties to the lower owner),
 * then, owner by owner, segments in parameter order, each starting on a
 * DMUON_PACK_ALIGN_ELEMS boundary, the owner buffers back to back in one
 * allocation.
 *   n            number of matrices (>= 1)
 *   shp[n]       shapes (host)
 *   n_owners     number of owner buffers (>= 1)
 *   owner_of[n]  out: owner of each matrix (host)
 *   offset[n]    out: element offset of each segment in the packed allocation
 *   owner_elems[n_owners] out: elements of each owner buffer (padded)
 * Returns DMUON_OK or DMUON_ERR_INVALID_ARG.  Touches no GPU.
 */
int dmuon_plan(int n, const dmuon_shape* shp, int n_owners, int* owner_of,
               int64_t* offset, int64_t* owner_elems);

/*
 * dmuon_ns_variant_for -- the form (DMUON_NS_STANDARD or DMUON_NS_GRAM) that a
 * call with `ns_variant` runs on a (rows, cols) matrix at `ns_steps` steps.
 * Home page, "VLA and VLM" and the closing credits name Gram Newton-Schulz;
 * the pages give no rule for when to use it.  This library's rule: Gram only
 * where it saves work (n > m, ns_steps >= 2) and, for DMUON_NS_GRAM, only
 * inside a band of aspect ratios n/m, per step count from 2 to 10, in which
 * the bf16 Gram iteration was measured to stay below 0.9 x the Newton-Schulz
 * tolerance (2e-2 up to 5 steps, 4e-2 above) on seeded Gaussian inputs of
 * several sizes; e.g. n/m in [1.75, 7] at 5 steps, [1.5, 8] at 8 steps.  The
 * calibration assumes well-spread singular values, as Gaussian inputs have.
 * Returns DMUON_ERR_INVALID_ARG for a bad shape, step count or variant.
 * Touches no GPU.
 */
int dmuon_ns_variant_for(int64_t rows, int64_t cols, int ns_steps, int ns_variant);

/*
 * dmuon_workspace_bytes -- scratch bytes that dmuon_pack / dmuon_ns_batched /
 * dmuon_unpack_update / dmuon_muon_step need for this shape list and variant.
 * dmuon_pack and dmuon_unpack_update use only the leading part of it (tables
 * and norm partial sums), which is laid out the same for both variants, so one
 * workspace sized for the variant in use serves all four calls.
 * Returns 0 for invalid arguments.  Touches no GPU.
 */
size_t dmuon_workspace_bytes(int n, const dmuon_shape* shp, int ns_variant);

/*
 * dmuon_pack -- Nesterov momentum + pack (step 1 above).
 * For each matrix i: M_i <- beta*M_i + (1-beta)*G_i (fp32, in place) and
 * packed[offset[i] + k] = bf16_rne(U_i[k]) with U_i = (1-beta)*G_i + beta*M_i,
 * in the parameter's own (rows, cols) row-major order.  Also records
 * ||U_i||_F^2 partial sums (fp32, fixed order) in the workspace; a following
 * dmuon_ns_batched(..., use_pack_norms=1) uses them as the norm of the fp32 U.
 *   grad[n]      device pointers, dtype grad_dt (F32 or BF16)
 *   momentum[n]  device pointers, fp32, updated in place
 *   packed_bf16  device, 256-byte aligned, >= max(offset[i] + rows*cols) bf16
 *   offset[n]    element offsets (multiples of DMUON_PACK_ALIGN_ELEMS)
 */
int dmuon_pack(int n, const dmuon_shape* shp, const void* const* grad, int grad_dt,
               float* const* momentum, float beta, void* packed_bf16,
               const int64_t* offset, void* workspace, size_t ws_bytes,
               cudaStream_t stream);

/*
 * dmuon_ns_batched -- Newton-Schulz orthogonalisation of every packed matrix,
 * in place (step 2 above).  packed[offset[i] ...] holds U_i (bf16, (rows, cols)
 * row-major) on entry and O_i (bf16, same layout) on return.
 *   ns_steps       >= 0; 0 returns X0 = U / (||U||_F + eps)
 *   ns_variant     DMUON_NS_STANDARD, DMUON_NS_GRAM or DMUON_NS_GRAM_ALL
 *   abc            host float[3] (a, b, c), or NULL for (3.4445, -4.7750, 2.0315)
 *   eps            norm epsilon (the standard value is 1e-7)
 *   use_pack_norms 1: take ||U_i|| from the partial sums of the preceding
 *                  dmuon_pack on this workspace (fp32 U); 0: compute it from
 *                  the bf16 values in `packed`.
 * Products run on the tcgen05 tensor cores with bf16 operands and fp32
 * accumulation; A and B are stored bf16.
 */
int dmuon_ns_batched(int n, const dmuon_shape* shp, void* packed_bf16,
                     const int64_t* offset, int ns_steps, int ns_variant,
                     const float* abc, float eps, int use_pack_norms,
                     void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * dmuon_unpack_update -- scaled weight update (step 3 above):
 * W_i <- W_i - lr * sqrt(max(1, rows/cols)) * O_i, O_i read from packed.
 * fp32 arithmetic; a bf16 W is rounded to nearest even.
 *   weight[n]   device pointers, dtype weight_dt (F32 or BF16), in place
 */
int dmuon_unpack_update(int n, const dmuon_shape* shp, void* const* weight,
                        int weight_dt, float lr, const void* packed_bf16,
                        const int64_t* offset, void* workspace, size_t ws_bytes,
                        cudaStream_t stream);

/*
 * dmuon_muon_step -- the whole owner-side Muon step: dmuon_pack, then
 * dmuon_ns_batched(use_pack_norms = 1) with the default coefficients and
 * eps = 1e-7, then dmuon_unpack_update, enqueued on `stream`.
 * With ns_steps >= 1 and two or more distinct working shapes (or
 * orientations, or forms under the Gram variant), the step overlaps its
 * memory-bound kernels with the tensor-core products: it visits groups of
 * shapes in turn (an order and grouping a time model of the launches picks),
 * and while one group is orthogonalised, later groups are packed and relaid
 * out and earlier groups' weights are updated, in pieces that each start
 * together with one long product launch and are sized to finish inside it;
 * what does not fit -- the first group's pack, the part of a later group's
 * pack that the products before it cannot hide (run just before that group),
 * the last group's update -- runs alone on `stream`.  The overlapped work runs on a
 * lowest-priority companion stream that the library creates for `stream` on
 * its first call with it (one per caller stream, up to 16 per device; past
 * that, and while `stream` is being captured, a companion shared by the device
 * serves), ordered against `stream` with events; when the call returns, all of
 * it is ordered before any later work on `stream`.  Owners that step on
 * different caller streams therefore run concurrently.  Results are identical
 * to the three separate calls.
 * The call can be captured into a CUDA graph (stream capture on `stream`) and
 * replayed: its tables are written by a kernel, and the second stream joins
 * the capture through the events.  Make one call on the device before the
 * first capture (it sets the library up for the device); the graph then reads
 * the buffers that were passed at capture time.
 */
int dmuon_muon_step(int n, const dmuon_shape* shp, const void* const* grad, int grad_dt,
                    float* const* momentum, void* const* weight, int weight_dt,
                    float lr, float beta, int ns_steps, int ns_variant,
                    void* packed_bf16, const int64_t* offset, void* workspace,
                    size_t ws_bytes, cudaStream_t stream);

/*
 * dmuon_adamw -- AdamW step for the parameters Muon does not own (home page,
 * "LLM Pretraining": AdamW learning rate 1e-3 in the usage example; "VLA and VLM":
 * embeddings, norms and heads stay outside the Muon set).  The pages give only
 * the learning rate; the update is the usual AdamW with decoupled weight decay:
 *   p <- p * (1 - lr*wd)
 *   m <- beta1*m + (1-beta1)*g;   v <- beta2*v + (1-beta2)*g^2
 *   p <- p - lr/(1-beta1^t) * m / (sqrt(v)/sqrt(1-beta2^t) + eps)
 * fp32 arithmetic; the hyper-parameters arrive in double and the per-step
 * scalars (1-beta1, 1-beta2, the bias corrections, 1-lr*wd) are formed in
 * double on the host and rounded to fp32 once.  A bf16 p is rounded to
 * nearest even.  Typical values: beta1 0.9, beta2 0.999, eps 1e-8,
 * weight_decay 0.01.
 *   n            number of tensors (0 is a no-op)
 *   numel[n]     host: elements of each tensor (any shape, contiguous)
 *   param[n]     device, dtype param_dt (F32 or BF16), updated in place
 *   grad[n]      device, dtype grad_dt (F32 or BF16)
 *   exp_avg[n], exp_avg_sq[n]   device, fp32, updated in place
 *   step         1-based step number t
 *   workspace    device, 256-byte aligned, >= dmuon_adamw_workspace_bytes(n)
 * One kernel launch for all tensors; 16-byte vector access where all four
 * pointers of a tensor are 16-byte aligned.
 */
size_t dmuon_adamw_workspace_bytes(int n);
int dmuon_adamw(int n, const int64_t* numel, void* const* param, int param_dt,
                const void* const* grad, int grad_dt, float* const* exp_avg,
                float* const* exp_avg_sq, double lr, double beta1, double beta2, double eps,
                double weight_decay, int step, void* workspace, size_t ws_bytes,
                cudaStream_t stream);

/*
 * dmuon_stream_status -- synchronises `stream`, then reports (and clears) the
 * device error word kept in `workspace`: DMUON_OK, DMUON_ERR_TIMEOUT when a
 * bounded device wait gave up, DMUON_ERR_CUDA when the stream holds a CUDA
 * error.  workspace may be NULL (then only the stream is checked).
 */
int dmuon_stream_status(cudaStream_t stream, void* workspace);

/*
 * dmuon_debug_wait_timeout -- test hook for the device failure path: launches
 * one block that waits on a shared-memory barrier nobody signals, with a
 * limit of `budget_us` microseconds (1..1000000).  The wait gives up, the
 * kernel records DMUON_ERR_TIMEOUT in the workspace error word and returns,
 * leaving the context usable.  Needs ws_bytes >= 256.  workspace == NULL
 * targets the error word of the built-in scratch array of
 * dmuon_ns_batched_noalloc instead (read it with dmuon_noalloc_status).
 */
int dmuon_debug_wait_timeout(void* workspace, size_t ws_bytes, int budget_us,
                             cudaStream_t stream);

/* Bytes of the library's built-in scratch array (see dmuon_ns_batched_noalloc). */
#define DMUON_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * dmuon_ns_batched_noalloc -- dmuon_ns_batched without a caller workspace, for
 * callers that cannot allocate device memory at all: code that runs where
 * cudaMalloc is forbidden or would stall (inside a host framework that owns
 * every device allocation, a plugin that may only use the buffers it is
 * handed, a latency-critical loop where cudaMalloc's implicit device
 * synchronisation is not acceptable).  The DMuon pages have no counterpart to
 * this call; it is a convenience of this library.
 *
 * Scratch comes from one file-scope __device__ array of
 * DMUON_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library.  Every GPU that
 * loads the library holds that array until the process exits.  The call
 * allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * The caller still passes the packed input/output buffer and the offsets,
 * with the same meaning and layout as for dmuon_ns_batched; the norms are taken
 * from the bf16 packed values (use_pack_norms = 0).
 *
 *  - Set-up: the first call on a device (with that device current) looks up
 *    the array's device address once and keeps it; make that first call
 *    before any stream capture.
 *  - Size limit: a shape list whose dmuon_workspace_bytes exceeds
 *    DMUON_NOALLOC_SCRATCH_BYTES is rejected with DMUON_ERR_WORKSPACE before
 *    anything is enqueued (e.g. 1024 x 4096 fits, 4096 x 4096 does not).
 *  - Sharing: every call on a device uses the same array, which keeps the last
 *    call's contents.  Calls whose work overlaps on the GPU (two streams, two
 *    host threads without ordering) race on it and give wrong results; order
 *    them on one stream.
 *  - Failures: the array holds its own device error word.  Each call clears it
 *    when it starts; a bounded wait that gives up inside the call leaves the
 *    outputs incomplete and records DMUON_ERR_TIMEOUT there, which
 *    dmuon_noalloc_status reports.  Read it before the next call.
 */
int dmuon_ns_batched_noalloc(int n, const dmuon_shape* shp, void* packed_bf16,
                             const int64_t* offset, int ns_steps, int ns_variant,
                             const float* abc, float eps, cudaStream_t stream);

/*
 * dmuon_noalloc_status -- dmuon_stream_status for the built-in scratch array
 * of dmuon_ns_batched_noalloc on the current device: synchronises `stream`,
 * then reports (and clears) the array's device error word: DMUON_OK,
 * DMUON_ERR_TIMEOUT when a bounded wait inside a call gave up, DMUON_ERR_CUDA
 * when the stream holds a CUDA error.  Like the call itself it allocates
 * nothing; on a device where no call has run yet it first looks up the
 * array's address (the same one-time set-up).  The DMuon pages have no
 * counterpart to it.
 */
int dmuon_noalloc_status(cudaStream_t stream);

/*
 * Tracing of the Newton-Schulz product launches, for measuring what happens
 * between and around them (launch gaps, last-wave tails, pipeline fill and
 * drain).  Between dmuon_trace_begin and dmuon_trace_end, every product launch
 * made on the device that was current at dmuon_trace_begin writes one record
 * per CTA into `records` (device memory of that device, 16-byte aligned), in
 * launch order, until `bytes` is used up; later launches are not traced.
 * Times are %globaltimer nanoseconds.  In a CTA pair only the first CTA
 * issues MMAs, so the second CTA's MMA stamps are 0 (also in a CTA that had no
 * tile).  Tracing costs a few stores per CTA; it changes no result.  Process-
 * wide: one trace at a time.  dmuon_trace_end returns the number of records
 * handed out; they are valid once the traced work has completed.
 */
typedef struct {
  uint32_t launch;           /* launch sequence number since dmuon_trace_begin */
  uint32_t cta;              /* blockIdx.x (CTAs 2k and 2k+1 form pair k) */
  uint32_t kind;             /* product kind: 0 sym K-major, 1 sym MN-major, 2 full wide, 3 full tall */
  uint32_t tiles;            /* 256 x 256 tiles of the whole launch */
  uint64_t t_entry_ns, t_mma_first_ns, t_mma_last_ns, t_exit_ns;
  /* first CTA of a pair, in SM cycles: its MMA thread's span (its start to the
     drain of its last MMA), and within it the waits for operand stages and for the
     epilogue to free an accumulator (0 elsewhere).  With the MMAs queued ahead of
     the tensor pipe, operand waits include the normal run-ahead of the thread, so
     they bound, not measure, operand starvation */
  uint64_t mma_span_cycles, wait_operand_cycles, wait_accum_cycles;
} dmuon_trace_record;
int dmuon_trace_begin(void* records, size_t bytes);
long long dmuon_trace_end(void);

/* Human-readable text for a status code (static storage). */
const char* dmuon_status_string(int status);

/* Library version: major*10000 + minor*100 + patch. */
int dmuon_version(void);

/*
 * dmuon_launch_count -- number of kernels the library has launched from the
 * calling host thread (every call above counts its own launches) since the
 * last reset; reset != 0 clears the count after reading it.
 */
long long dmuon_launch_count(int reset);

#ifdef __cplusplus
}
#endif
#endif /* DMUON_H */
