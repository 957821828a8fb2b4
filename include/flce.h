/*
 * flce.h -- C ABI of the GB300 (sm_103a) fused linear cross-entropy library.
 *
 * Fused linear cross-entropy (FLCE) computes the cross-entropy loss of
 * softmax(X @ W) for hidden states X [N,D] and a vocabulary projection W [D,V]
 * without ever holding the N x V logits in memory, and its gradients dX and dW.
 *
 * Sources, cited by page title and section:
 *   [P1] "Cutting LLM Memory by 84%: A Deep Dive into Fused Kernels" (blog post):
 *        "The Logit Bottleneck" (shapes), "Definition and Forward Pass" (loss =
 *        lse - target logit, online softmax), "Backward Pass" ("Matrix
 *        Multiplication", "Cross-Entropy", "Fused Linear Cross-Entropy"), "Setup
 *        and Target Logit Pre-computation" (ignore_index, default -100), "Path to
 *        Production" (no atomics on dX; a dW pass that writes each block once).
 *   [P3] NVIDIA TransformerEngine pull request #995 (label-smoothing rule of the
 *        backward kernel; entry points that release the Python GIL).
 *   [P4] Liger-Kernel pull request #1291, "[CuteDSL] FLCE: 2-SM online-softmax fast
 *        path (Blackwell)", "Summary": store-free forward that keeps only the
 *        per-row LSE and target logit; a backward that recomputes the softmax per
 *        vocabulary tile and contracts dW over the token dimension; feature list
 *        (label_smoothing, z-loss "lse_square_scale", ignore_index, mean/sum,
 *        forward-only reduction 'none', refusal of 'none' with a gradient).
 *
 * Definitions (eps = label_smoothing, s = zloss_scale, valid(i) <=> y_i != ignore_index):
 *   z_ij   = sum_k X_ik W_kj
 *   lse_i  = log sum_j exp(z_ij)
 *   l_i    = (1-eps)(lse_i - z_{i,y_i}) + eps (lse_i - (1/V) sum_j z_ij) + s lse_i^2   (valid rows)
 *   l_i    = 0                                                                         (ignored rows)
 *   loss   = sum_i l_i  (SUM) | sum_i l_i / n_valid (MEAN, 0 if n_valid == 0) | l (NONE)
 *   dZ_ij  = g [exp(z_ij - lse_i)(1 + 2 s lse_i) - (1-eps) delta_{j,y_i} - eps/V],
 *            g = grad_out (SUM) or grad_out / n_valid (MEAN); dZ_i = 0 for ignored rows
 *   dX     = dZ W^T,   dW = X^T dZ
 * eps follows torch's convention: the target class keeps 1 - eps + eps/V of the
 * probability mass, every other class eps/V. (TransformerEngine's label_smoothing
 * alpha equals eps = alpha V / (V - 1).)
 *
 * Data layout (all row-major, contiguous, device memory):
 *   X        bf16  [N, D]      row stride D elements
 *   W        bf16  [D, V]      row stride V elements (nn.Linear's [V, D] and f16 inputs:
 *                              flce_options.weight_layout and .input_dtype)
 *   targets  int32 [N]
 *   lse      fp32  [N]
 *   loss     fp32  [1] (MEAN, SUM) or [N] (NONE)
 *   dX       bf16  [N, D]      (the type of X)
 *   dW       fp32  [D, V]      (the layout of W)
 *
 * Ownership and execution: the caller owns every buffer, including the
 * workspace; the library never allocates or frees memory. All calls are
 * asynchronous on `stream` and never synchronise, except
 * flce_check_device_error. The library keeps no state between calls other than
 * per-device launch attributes, a launch counter and a per-thread error detail;
 * separate workspaces make calls independent.
 *
 * Errors: host-side argument checks return a status synchronously and launch
 * nothing. Conditions found on the device (a target outside [0, V) that is not
 * the ignore index; a pipeline wait that exceeded its time limit) set an error
 * word inside the workspace and poison the affected results with NaN (a bad target:
 * its row's loss and gradient rows; a timeout: every lse and loss value of the
 * forward, every element of a 16-bit dX of the backward, while dW is then undefined);
 * no kernel traps. flce_check_device_error reads that word.
 *
 * Requirements: a compute capability 10.3 device (GB300); D % 8 == 0 and
 * V % 8 == 0 (16-byte row strides for the tensor-memory-access unit); X, W, dX,
 * dW and the workspace 16-byte aligned; targets, lse and loss 4-byte aligned.
 * Every buffer, workspace and option array included, is device memory of the
 * current device or managed memory: host memory (pinned or pageable) and another
 * device's memory are refused with FLCE_ERR_INVALID_ARG before anything is
 * launched, and flce_last_error_detail names the buffer.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *`; NULL means the legacy default stream */

typedef enum {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARG = 1,          /* null pointer, size < 1, eps outside [0,1), s < 0, bad enum,
                                        a buffer that is not memory of the current device */
  FLCE_ERR_ALIGNMENT = 2,            /* D or V not a multiple of 8, or a misaligned pointer */
  FLCE_ERR_UNSUPPORTED_DEVICE = 3,   /* the current device is not compute capability 10.3 */
  FLCE_ERR_WORKSPACE_TOO_SMALL = 4,  /* ws_bytes < flce_workspace_size(...) */
  FLCE_ERR_REDUCTION_NONE_GRAD = 5,  /* flce_backward with FLCE_REDUCTION_NONE (refused by design) */
  FLCE_ERR_CUDA = 6,                 /* a CUDA runtime or driver call failed */
  FLCE_ERR_BAD_TARGET = 7,           /* device: a target outside [0,V) that is not ignore_index */
  FLCE_ERR_TIMEOUT = 8,              /* device: a pipeline wait exceeded its limit; results invalid */
  FLCE_ERR_TOO_LARGE = 9,            /* a size exceeds the library's index range */
  FLCE_ERR_F16_RANGE = 10            /* device, f16 inputs: a row's scaled gradient coefficient
                                        exceeds the f16 range (class weights too large) */
} flce_status;

typedef enum {
  FLCE_REDUCTION_MEAN = 0,
  FLCE_REDUCTION_SUM = 1,
  FLCE_REDUCTION_NONE = 2
} flce_reduction;

/* Bytes of workspace that flce_forward (for_backward == 0), flce_backward
 * (for_backward == 1) or flce_forward_backward (for_backward == 2) needs for this
 * shape. Returns 0 for invalid sizes. The backward workspace holds a 16-bit gradient
 * band of N x Vc columns (Vc a multiple of 512, at most 16384, and below V once V
 * exceeds 512) and an fp32 [N, D] dX accumulator; no buffer has N x V elements.
 * for_backward == 3 gives the size from which flce_forward (without the argmax and
 * epilogue options, N >= 2048) runs its GEMM on the valid rows only, gathered into the workspace:
 * the forward's own size plus the row list and the valid rows of X (N x D 16-bit values).
 * Any backward or fused workspace has that room. The results are the same either way,
 * bit for bit; only the time differs. */
size_t flce_workspace_size(int64_t N, int64_t D, int64_t V, int for_backward);

/* Forward pass. [P1] "Definition and Forward Pass" and "Kernel Implementation"
 * (online softmax over vocabulary tiles, target logit, lse - z_y); [P4] "Summary"
 * (store-free: only the per-row LSE and target logit leave the GEMM epilogue).
 *   X, W, targets : inputs as laid out above (device pointers).
 *   ignore_index  : rows whose target equals it have loss 0 (default -100 in [P1]).
 *   label_smoothing in [0,1), zloss_scale >= 0, red : see the definitions above.
 *   loss          : out, fp32 [1] (MEAN/SUM) or [N] (NONE).
 *   lse           : out, fp32 [N], log-sum-exp of every valid row; 0 for a row whose
 *                   target is the ignore index (its loss needs no lse; [P1]'s kernel
 *                   returns early for such rows).
 *   workspace     : device scratch of at least flce_workspace_size(N,D,V,0) bytes; from
 *                   flce_workspace_size(N,D,V,3) bytes the GEMM skips the ignored rows.
 * Returns FLCE_OK or a host-side error; nothing is launched on error. */
flce_status flce_forward(const void* X, const void* W, const int32_t* targets,
                         int64_t N, int64_t D, int64_t V, int32_t ignore_index,
                         float label_smoothing, float zloss_scale, flce_reduction red,
                         float* loss, float* lse,
                         void* workspace, size_t ws_bytes, struct CUstream_st* stream);

/* Backward pass. [P1] "Backward Pass" and "Path to Production"; [P3] backward
 * kernel (smoothing rule); [P4] "Summary" (recompute the softmax per vocabulary
 * tile; dW contracts over the token dimension and each dW block is written once).
 *   lse       : fp32 [N] from flce_forward with the same inputs.
 *   grad_out  : device fp32 scalar, the upstream gradient of the reduced loss.
 *   dX        : out, bf16 [N, D] (overwritten). Until the call's last kernel writes
 *               it, the buffer serves as scratch: the backward gathers the valid rows
 *               of X there and runs its GEMMs on them alone (an ignored row's gradient
 *               is zero). A dX that overlaps an input (X itself, say) is computed in
 *               place without that compaction.
 *   dW        : out, fp32 [D, V] (overwritten, each element written once).
 *   workspace : device scratch of at least flce_workspace_size(N,D,V,1) bytes.
 * The options must equal the forward call's. FLCE_REDUCTION_NONE is refused
 * (FLCE_ERR_REDUCTION_NONE_GRAD), as in [P4]: a per-row upstream gradient is not
 * supported by the fused reduction. */
flce_status flce_backward(const void* X, const void* W, const int32_t* targets, const float* lse,
                          int64_t N, int64_t D, int64_t V, int32_t ignore_index,
                          float label_smoothing, float zloss_scale, flce_reduction red,
                          const float* grad_out, void* dX, float* dW,
                          void* workspace, size_t ws_bytes, struct CUstream_st* stream);

/* Optional features of the extended entry points below. [P4] "Summary" names them
 * (softcap, bias, ce_weight, token accuracy, predicted tokens, vocabulary-parallel
 * use through the Megatron path of [P3]) without defining them; the semantics are
 * torch's, as [P4] claims parity with torch:
 *   z_ij = sum_k X_ik W_kj + bias_j,   u_ij = softcap * tanh(z_ij / softcap) (softcap > 0) else z_ij,
 *   l_i  = (1-eps) w_{y_i} (lse_i - u_{i,y_i}) + (eps/V) sum_j w_j (lse_i - u_ij) + s lse_i^2,
 *   MEAN divides by sum over valid rows of w_{y_i} (the valid-row count when w == 1),
 *   dU_ij = g [p_ij ((1-eps) w_{y_i} + (eps/V) sum_j w_j + 2 s lse_i) - (eps/V) w_j - (1-eps) w_{y_i} delta],
 *   dZ = dU (1 - (u/softcap)^2) with a softcap,  dbias = sum_i dZ_i,
 *   predicted_i = argmax_j u_ij (smallest index on ties), accuracy = matches / valid rows.
 * Zero-initialise the struct and set what you need; NULL means "no options". */
/* Storage of W and dW. FLCE_WEIGHT_DV: W [D, V] and dW [D, V], row-major (the default,
 * the layout of "Cutting LLM Memory by 84%", "The Logit Bottleneck"). FLCE_WEIGHT_VD:
 * W [V, D] and dW [V, D], row-major -- the weight of an nn.Linear(D, V) language-model
 * head, taken as it is stored (no transposed copy). Not a part of the pages' method. */
typedef enum { FLCE_WEIGHT_DV = 0, FLCE_WEIGHT_VD = 1 } flce_weight_layout;

/* Element type of X and W (and of dX; dW is fp32 either way). The tensor cores multiply
 * both at the same rate. With f16 the gradient band holds G/g scaled by 2^10 (so that
 * probabilities near 1/V stay normal f16 numbers) and dX, dW are scaled back in fp32; this
 * needs (1 - eps) w_y + (eps/V) sum_j w_j + 2 s lse < 64 on every row (class weights below
 * ~60 in practice); a row above it is reported by flce_check_device_error as
 * FLCE_ERR_F16_RANGE (its gradient would overflow the band). dX is rounded once from its
 * fp32 accumulator to f16, so entries below f16's normal range (6.1e-5) keep only
 * absolute precision: scale the loss (grad_out) or ask for the fp32 dX (dX_f32) when
 * gradients are that small. Not a part of the pages' method, whose kernels take 16-bit
 * inputs ([P4] "Summary"). */
typedef enum { FLCE_INPUT_BF16 = 0, FLCE_INPUT_F16 = 1 } flce_input_dtype;

typedef struct flce_options {
  float softcap;             /* > 0: cap the logits with softcap*tanh(z/softcap); 0: off */
  const float* bias;         /* device fp32 [V] added to every row's logits, or NULL */
  const float* class_weight; /* device fp32 [V] per-class weights (all >= 0), or NULL */
  int32_t* predicted;        /* forward out: device int32 [N] argmax of each row, or NULL */
  float* accuracy;           /* forward out: device fp32 [1] argmax == target over valid rows, or NULL */
  float* dbias;              /* backward out: device fp32 [V] (needs bias), or NULL */
  float* dX_f32;             /* backward out: device fp32 [N, D] dX written instead of the bf16 dX, or NULL */
  int64_t v_offset;          /* vocabulary shard: global index of W's first column (0 if unsharded) */
  int64_t v_total;           /* vocabulary shard: size of the full vocabulary (0 means V: unsharded) */
  int64_t row_band;          /* backward: > 0 processes rows in bands of this many ([P1] "Path to
                                Production": micro-batching along N), so the workspace is
                                flce_workspace_size(row_band, D, V, 1) whatever N is; dW then
                                accumulates across bands (fp32 adds in a fixed order). 0: all rows. */
  int32_t weight_layout;     /* flce_weight_layout of W and dW (FLCE_WEIGHT_DV if 0) */
  int32_t input_dtype;       /* flce_input_dtype of X, W and dX (FLCE_INPUT_BF16 if 0) */
  int32_t accumulate_grads;  /* backward: 1 adds this call's dW (and dbias) into the caller's
                                buffers instead of overwriting them, for gradient accumulation
                                over micro-batches ([P1] "Path to Production"); the adds are
                                fp32 element-wise, in a fixed order. dX is always overwritten. */
} flce_options;

/* flce_forward with options (NULL behaves exactly like flce_forward). Vocabulary
 * shards (v_total > V) are not accepted here: use flce_shard_stats. */
flce_status flce_forward_ex(const void* X, const void* W, const int32_t* targets,
                            int64_t N, int64_t D, int64_t V, int32_t ignore_index,
                            float label_smoothing, float zloss_scale, flce_reduction red,
                            const flce_options* opt, float* loss, float* lse,
                            void* workspace, size_t ws_bytes, struct CUstream_st* stream);

/* flce_backward with options. With opt->v_total > V, W holds the columns
 * [v_offset, v_offset + V) of a vocabulary of v_total, lse is the full-vocabulary
 * log-sum-exp (flce_combine_shards), dW is this shard's [D, V] block and dX (or dX_f32)
 * this shard's partial dX, to be summed over shards by the caller (e.g. an
 * all-reduce). Shards support label smoothing and z-loss, not the other options. */
flce_status flce_backward_ex(const void* X, const void* W, const int32_t* targets, const float* lse,
                             int64_t N, int64_t D, int64_t V, int32_t ignore_index,
                             float label_smoothing, float zloss_scale, flce_reduction red,
                             const flce_options* opt, const float* grad_out, void* dX, float* dW,
                             void* workspace, size_t ws_bytes, struct CUstream_st* stream);

/* Forward and backward in one call, for a loss that is the last layer ([P1] "Kernel
 * Implementation" fuses both passes for that reason). Same outputs as flce_forward_ex
 * followed by flce_backward_ex; workspace: flce_workspace_size(N, D, V, 2) bytes. */
flce_status flce_forward_backward(const void* X, const void* W, const int32_t* targets,
                                  int64_t N, int64_t D, int64_t V, int32_t ignore_index,
                                  float label_smoothing, float zloss_scale, flce_reduction red,
                                  const flce_options* opt, const float* grad_out,
                                  float* loss, float* lse, void* dX, float* dW,
                                  void* workspace, size_t ws_bytes, struct CUstream_st* stream);

/* Vocabulary-parallel forward, one shard: W holds columns [v_offset, v_offset + V)
 * of the full vocabulary. Writes stats, device fp32 [4][N]: the shard's log-sum-exp,
 * the sum of the shard's logits, the target logit if the target is in the shard
 * (else 0) and 1/0 for whether it is. Gather the shards' stats (e.g. all-gather,
 * 16 bytes per row per shard) and call flce_combine_shards. Workspace:
 * flce_workspace_size(N, D, V, 0). */
flce_status flce_shard_stats(const void* X, const void* W, const int32_t* targets,
                             int64_t N, int64_t D, int64_t V, int64_t v_offset, int32_t ignore_index,
                             float* stats, void* workspace, size_t ws_bytes, struct CUstream_st* stream);

/* flce_shard_stats for W stored [V, D] (the shard is rows [v_offset, v_offset + V) of the
 * full weight) or f16 inputs: opt may set weight_layout and input_dtype, every other
 * field must be zero (FLCE_ERR_INVALID_ARG otherwise). NULL behaves like flce_shard_stats. */
flce_status flce_shard_stats_ex(const void* X, const void* W, const int32_t* targets,
                                int64_t N, int64_t D, int64_t V, int64_t v_offset, int32_t ignore_index,
                                const flce_options* opt, float* stats, void* workspace, size_t ws_bytes,
                                struct CUstream_st* stream);

/* Combine K shards' stats (device fp32 [K][4][N], shard order irrelevant) into the
 * full-vocabulary lse [N] and the loss, as flce_forward would for the whole
 * vocabulary of v_total classes. Workspace: flce_workspace_size(N, 8, 8, 0). */
flce_status flce_combine_shards(const float* stats, int32_t K, const int32_t* targets, int64_t N,
                                int64_t v_total, int32_t ignore_index, float label_smoothing,
                                float zloss_scale, flce_reduction red, float* loss, float* lse,
                                void* workspace, size_t ws_bytes, struct CUstream_st* stream);

/* Synchronises `stream`, then reads and clears the device error word of the
 * most recent call that used `workspace`. Returns FLCE_OK, FLCE_ERR_TIMEOUT,
 * FLCE_ERR_BAD_TARGET, FLCE_ERR_F16_RANGE (in that order of precedence), or
 * FLCE_ERR_CUDA if the copy itself failed. */
flce_status flce_check_device_error(void* workspace, struct CUstream_st* stream);

/* A static, human-readable name for a status. */
const char* flce_status_string(flce_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH: 300 (0.3.0). 0.2 grew flce_options
 * (weight_layout, input_dtype, accumulate_grads at its end): code built against 0.1's
 * header must be rebuilt. 0.3: the forward writes lse 0 for ignored rows (it may skip
 * them), and flce_workspace_size takes for_backward == 3. */
int flce_version(void);

/* Which call failed the last time an entry point returned FLCE_ERR_CUDA on the calling
 * thread: the CUDA runtime or driver call and its error name, e.g.
 * "cudaMemsetAsync(...): cudaErrorInvalidValue"; or, after FLCE_ERR_INVALID_ARG for a
 * buffer outside the current device's memory, that buffer's name and why, e.g.
 * "X: is host memory, not device memory". Empty if that never happened on this
 * thread; later successful calls do not clear it. The string is thread-local, owned by
 * the library and valid until the thread's next library call. Diagnostics only: the
 * pages have no counterpart. */
const char* flce_last_error_detail(void);

/* Number of kernels this library has launched in the process so far, over every thread
 * and device (a relaxed atomic counter; each launch counts itself when it is issued).
 * For profiling and launch accounting; the pages have no counterpart. */
unsigned long long flce_kernel_launches(void);

/* Diagnostic device timing of the tensor-core GEMMs. With flce_profile_gemms(1), every
 * later GEMM launch of any thread is bracketed by two CUDA events recorded on the call's
 * stream (created per launch; not for use under stream capture); flce_profile_gemms(0)
 * stops that. flce_profile_read waits for the events recorded so far, adds their elapsed
 * times and counts per GEMM kind into ms[4] and launches[4] (0 forward, 1 gradient,
 * 2 dW, 3 dX), releases them, and returns FLCE_OK (FLCE_ERR_CUDA if an event failed).
 * For measuring each kernel's share of a step live; the pages have no counterpart. */
void flce_profile_gemms(int enable);
flce_status flce_profile_read(double* ms, unsigned long long* launches);

/* Width (vocabulary columns) of the gradient bands flce_backward uses for this shape on
 * the current device: a multiple of 512 at most the workspace's band capacity, chosen so
 * that the dW GEMM's launches fill the device's resident clusters evenly. opt may be
 * NULL (only weight_layout and row_band matter). Returns 0 for invalid sizes or without
 * a supported device. Diagnostics and launch accounting; the pages have no counterpart. */
int64_t flce_backward_band_width(int64_t N, int64_t D, int64_t V, const flce_options* opt);

/* Self-test of failure detection: launches one small kernel whose pipeline wait (the
 * bounded mbarrier wait every GEMM uses) waits for an arrival that never comes, gives up
 * after the wait limit (2 s) and records FLCE_DEVERR_TIMEOUT in the workspace header
 * instead of hanging. Asynchronous like every call; flce_check_device_error then returns
 * FLCE_ERR_TIMEOUT, and the context stays usable. workspace: at least 256 bytes.
 * Diagnostics only; the pages have no counterpart. */
flce_status flce_selftest_wait_timeout(void* workspace, size_t ws_bytes, struct CUstream_st* stream);

/* Forward pass without a workspace, for callers that cannot allocate device memory
 * (code inside an allocator or memory-pool callback, runtimes that give a fixed
 * device arena and forbid further allocation). The source pages have no
 * counterpart: this is a library convenience. Arguments, outputs and results are
 * those of flce_forward; the scratch is a 64 MiB device array inside the library,
 * taken on every GPU where this entry point is used until the process exits (under
 * CUDA's default lazy module loading; with CUDA_MODULE_LOADING=EAGER it is taken on
 * every device the process uses).
 *  - The first call on a device (with that device current) looks up the array's
 *    device address and keeps it; make that first call before any stream capture,
 *    and do not use this entry point after a device reset (the kept address would be
 *    stale).
 *  - All calls share the array: calls that overlap on the GPU race; serialise them.
 *    Each call clears the parts that must start at zero.
 *  - Shapes needing more than 64 MiB of forward scratch (flce_workspace_size(N, D,
 *    V, 0)) return FLCE_ERR_WORKSPACE_TOO_SMALL and launch nothing.
 *  - It never calls cudaMalloc, cudaFree or any allocating routine.
 *  - Its device error word is internal, so device findings show in the results: a bad
 *    target makes its row's loss (and the reduced loss) NaN, and a pipeline wait that
 *    ran out makes every lse and loss value of the call NaN. */
flce_status flce_forward_noalloc(const void* X, const void* W, const int32_t* targets,
                                 int64_t N, int64_t D, int64_t V, int32_t ignore_index,
                                 float label_smoothing, float zloss_scale, flce_reduction red,
                                 float* loss, float* lse, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H_ */
