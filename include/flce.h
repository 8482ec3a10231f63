/*
 * flce.h - fused linear cross-entropy (LM head) on GB300 (sm_103a).
 *
 * The operation ("efficient-llm-anatomy" README, section "Fused cross-entropy
 * computes backward during forward", and the "Per-component memory savings"
 * table, row "Cross-entropy"): the LM-head matmul, softmax and negative
 * log-likelihood are computed chunk by chunk over tokens, so the N x V logits
 * are never materialised, and grad_input / grad_weight are produced in the
 * same call as the loss.
 *
 * Notation:
 *   X  = hidden      [N, H] bf16, row-major (row n is token n)
 *   W  = weight      [V, H] bf16, row-major (PyTorch Linear layout: forward
 *                    is X @ W^T; "Alisa's book of LLMs", "Neural net basics",
 *                    linear-layer backprop paragraph)
 *   t  = targets     [N] int32; t[n] == ignore_index marks an ignored token.
 *                    Targets are NOT shifted inside the library: t[n] labels
 *                    row n (the shift is the caller's business, as in the
 *                    "implementing the loss" code of the same page).
 *   z  = X W^T, lse_n = log sum_v exp(z_nv), loss_n = lse_n - z_{n,t_n}
 *   loss = sum over valid n of loss_n / n_valid          (FLCE_REDUCE_MEAN)
 *        = sum over valid n of loss_n                    (FLCE_REDUCE_SUM)
 *   dz_nv = (softmax(z_n)_v - [v == t_n]) * s,  s = 1/n_valid (mean) or 1
 *           ("gradient of softmax + CE loss" section; the 1/n from the
 *           linearity of the mean, "Backpropagation" section)
 *   grad_hidden = dz W    (bf16 [N, H]; rows of ignored tokens are +0.0)
 *   grad_weight = dz^T X  (fp32 [V, H]; gradients accumulate in fp32, the
 *                          mixed-precision convention of the same page)
 *   When no token is valid (n_valid == 0) the loss and both gradients are 0.
 *
 * Memory and ownership.  The caller allocates every buffer, including the
 * workspace; the library never allocates device memory.  Inputs are only
 * read.  Outputs are fully overwritten (never accumulated into).  All device
 * pointers must be 16-byte aligned and must not alias one another.
 *
 * Streams.  Each call only enqueues kernels on `stream` (a cudaStream_t
 * passed as void*, NULL = legacy default stream) and returns; nothing
 * synchronises the host.  Errors that the host can see (bad sizes, NULL or
 * misaligned pointers, a workspace that is too small, a failed launch) are
 * returned at once and nothing is enqueued.  Errors that only the device can
 * see (a target outside [0, V) that is not ignore_index, a stalled pipeline
 * stage) are recorded in a status word inside the workspace: read it with
 * flce_query_status().  The loss of a call whose device status is not FLCE_OK is
 * written as NaN, so a caller that never reads the status still sees that the
 * outputs of that call are not valid.  Device code never traps.
 *
 * Concurrency.  Calls are reentrant; concurrent calls need separate
 * workspaces.
 */
#ifndef FLCE_H
#define FLCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum flce_status {
  FLCE_OK = 0,
  FLCE_EINVAL = 1,        /* NULL pointer, N/H/V < 1, unknown flag          */
  FLCE_EUNSUPPORTED = 2,  /* H % 8 != 0, pointer not 16-byte aligned,       */
                          /* size beyond the supported range, no sm_100+ GPU */
  FLCE_EWORKSPACE = 3,    /* workspace_bytes below the minimum plan          */
  FLCE_EBADTARGET = 4,    /* (device) a target outside [0,V), not ignored    */
  FLCE_ETIMEOUT = 5,      /* (device) a pipeline wait ran out of time        */
  FLCE_ECUDA = 6          /* a CUDA runtime call or launch failed            */
} flce_status;

/* Reduction flags (bit 0). */
#define FLCE_REDUCE_MEAN 0x0u  /* mean over non-ignored tokens (default)       */
#define FLCE_REDUCE_SUM  0x1u  /* unscaled sum; grads without the 1/n_valid   */
/*
 * Output precision of grad_weight (bit 1), flce_fwd_bwd and
 * flce_rmsnorm_fwd_bwd only.  With FLCE_GW_BF16, grad_weight is a bf16
 * [V,H] array: the gradient still accumulates in fp32 over the token chunks
 * ("Alisa's book of LLMs", "Precision": bf16 compute, fp32 accumulation of
 * gradients) in a V*H*4-byte region of the workspace, and the finished sum is
 * rounded once (nearest even) into grad_weight.  The workspace functions
 * include that region when the flag is passed, so this workspace is larger
 * than 5% of the bf16 logits at every large vocabulary (V*H*4 alone is
 * 2.1 GB at H=4096, V=128256).
 */
#define FLCE_GW_BF16     0x2u

/* Description of how a call is carried out for a given workspace size. */
typedef struct flce_plan_info {
  int64_t chunk_rows;       /* C: valid tokens processed per chunk            */
  int64_t max_chunks;       /* chunks launched (ceil(N / C)); empty ones exit  */
  int64_t logits_row_stride;/* elements per row of the bf16 chunk logits buffer*/
  int32_t gemm_launches_per_chunk; /* 2 (logits; grad_hidden + grad_weight), 1 fwd */
  int32_t dx_splits;        /* vocabulary splits of the grad_hidden GEMM        */
  int32_t vocab_tiles;      /* ceil(V / 256): logits tiles per 256 tokens      */
  size_t workspace_bytes;   /* bytes the plan uses (<= the bytes offered)      */
} flce_plan_info;

/*
 * Workspace sizes.  The workspace holds one chunk of tokens at a time: the
 * chunked processing of the "efficient-llm-anatomy" README ("Fused
 * cross-entropy computes backward during forward", and the memory the
 * "Per-component memory savings" table measures for the cross-entropy row).
 * flce_workspace_bytes: the default plan, sized so that the extra device
 *   memory stays below 5% of the N*V*2 bytes that bf16 logits would take
 *   (never below one 128-row chunk).
 * flce_workspace_bytes_for_chunk: the plan with a given chunk size
 *   (chunk_rows is rounded up to a multiple of 128).
 * flce_loss_workspace_bytes: the same for the forward-only flce_loss.
 * Return 0 for invalid sizes.
 */
size_t flce_workspace_bytes(int64_t N, int64_t H, int64_t V, uint32_t flags);
size_t flce_workspace_bytes_for_chunk(int64_t N, int64_t H, int64_t V,
                                      uint32_t flags, int64_t chunk_rows);
size_t flce_loss_workspace_bytes(int64_t N, int64_t H, int64_t V, uint32_t flags);

/*
 * The plan flce_fwd_bwd (forward_only = 0) or flce_loss (forward_only = 1)
 * would use with `workspace_bytes` of workspace: the largest chunk that fits.
 */
flce_status flce_plan(int64_t N, int64_t H, int64_t V, uint32_t flags,
                      int forward_only, size_t workspace_bytes,
                      flce_plan_info* out);

/*
 * Forward + backward in one call.
 *   hidden       [N,H] bf16 (device)          read
 *   weight       [V,H] bf16 (device)          read
 *   targets      [N] int32 (device)           read
 *   loss         [1] fp32 (device)            written
 *   n_valid      [1] int32 (device)           written: tokens with t != ignore_index
 *   row_loss     [N] fp32 (device) or NULL    written: loss_n (unscaled), 0 when ignored
 *   grad_hidden  [N,H] bf16 (device)          written
 *   grad_weight  [V,H] fp32 (device)          written (bf16 with FLCE_GW_BF16)
 *   workspace    device scratch of workspace_bytes (>= flce_workspace_bytes_for_chunk
 *                with chunk 128); its contents need no initialisation and
 *                hold the device status word afterwards.
 * Supported sizes: 1 <= N < 2^31, 8 <= H <= 2^20 with H % 8 == 0,
 * 1 <= V < 2^31.
 */
flce_status flce_fwd_bwd(const void* hidden, const void* weight,
                         const int32_t* targets, int64_t N, int64_t H,
                         int64_t V, int32_t ignore_index, uint32_t flags,
                         float* loss, int32_t* n_valid, float* row_loss,
                         void* grad_hidden, float* grad_weight,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward only: loss (and optionally row_loss) without gradients, 2*N*H*V
 * flops instead of 6*N*H*V: the masked mean of the per-token negative
 * log-likelihoods ("Alisa's book of LLMs", "cross-entropy loss" and
 * "implementing the loss"), each from a max-shifted log-sum-exp ("Numerical
 * stability and other tricks").  Same argument rules as flce_fwd_bwd.
 */
flce_status flce_loss(const void* hidden, const void* weight,
                      const int32_t* targets, int64_t N, int64_t H, int64_t V,
                      int32_t ignore_index, uint32_t flags, float* loss,
                      int32_t* n_valid, float* row_loss, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * The final RMSNorm fused in front of the LM head ("Alisa's book of LLMs",
 * transformer section: final norm, then unembedding; RMSNorm divides every
 * element of the hidden state by its RMS and multiplies by a learned
 * per-dimension gain).  With h = hidden (pre-norm, bf16 [N,H]) and
 * g = gain (bf16 [H]):
 *   x_n = h_n * r_n * g,   r_n = 1 / sqrt(mean_h(h_nh^2) + eps)
 * then the fused linear cross-entropy of x (rounded to bf16) against weight.
 * Outputs: loss, n_valid, row_loss as flce_fwd_bwd; grad_hidden (bf16
 * [N,H]) is the gradient with respect to the PRE-norm hidden states,
 *   dh_n = r_n (g * dx_n - xhat_n * mean_h(g * dx_n * xhat_n)),  xhat_n = h_n r_n,
 * grad_gain (fp32 [H]) = sum_n dx_n * xhat_n (summed over chunks in a fixed
 * order), grad_weight (fp32 [V,H]) as flce_fwd_bwd.  eps >= 0.  Workspace:
 * flce_rmsnorm_workspace_bytes (the 5% rule plus 4 bytes per chunk row and
 * per chunk and hidden unit).
 */
size_t flce_rmsnorm_workspace_bytes(int64_t N, int64_t H, int64_t V, uint32_t flags);
flce_status flce_rmsnorm_fwd_bwd(const void* hidden, const void* gain, float eps,
                                 const void* weight, const int32_t* targets,
                                 int64_t N, int64_t H, int64_t V,
                                 int32_t ignore_index, uint32_t flags,
                                 float* loss, int32_t* n_valid, float* row_loss,
                                 void* grad_hidden, float* grad_gain,
                                 float* grad_weight, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Vocabulary-parallel LM head (the weight split by rows over P ranks, as a
 * column-parallel linear layer; "Alisa's book of LLMs", parallelism sections:
 * sharded matmul whose output dimension is split, and tensor parallelism).
 * Rank r holds weight rows [v0, v0 + V_shard) of a V_total-row weight and
 * the whole batch.  One step:
 *  1. flce_vocab_shard_stats: per token, over the shard's logits, the max,
 *     the sum of exp(z - max) and the target logit (0 when the target is not
 *     in the shard); ignored tokens give 0, 0, 0.
 *  2. all-reduce MAX of row_max over ranks; flce_vocab_rescale rescales the
 *     local sums to the global max (the online-softmax merge, "Numerical
 *     stability and other tricks"); all-reduce SUM of row_sumexp and of
 *     row_target_logit.
 *  3. flce_vocab_finish (any rank): lse = max + log(sum), per-token loss
 *     lse - z_t, loss = mean (or sum) over valid tokens, n_valid.
 *  4. flce_vocab_shard_bwd with the global lse: the shard's logits are
 *     computed again chunk by chunk, dz = (exp(z - lse) - onehot) * s, the
 *     shard's grad_weight (fp32 [V_shard, H], complete) and this shard's fp32
 *     part of grad_hidden ([N, H]); all-reduce SUM of the parts gives
 *     grad_hidden.
 * The collectives are the caller's (e.g. NCCL); all arrays are device
 * arrays; targets hold ids in [0, V_total).  Workspaces as flce_fwd_bwd
 * with V = V_shard (flce_vocab_shard_workspace_bytes).
 */
size_t flce_vocab_shard_workspace_bytes(int64_t N, int64_t H, int64_t V_shard, uint32_t flags);
flce_status flce_vocab_shard_stats(const void* hidden, const void* weight_shard,
                                   const int32_t* targets, int64_t N, int64_t H,
                                   int64_t V_shard, int64_t v0, int64_t V_total,
                                   int32_t ignore_index, float* row_max,
                                   float* row_sumexp, float* row_target_logit,
                                   int32_t* n_valid, void* workspace,
                                   size_t workspace_bytes, void* stream);
flce_status flce_vocab_rescale(const float* row_max_local, const float* row_max_global,
                               float* row_sumexp, int64_t N, void* stream);
flce_status flce_vocab_finish(const float* row_max, const float* row_sumexp,
                              const float* row_target_logit, const int32_t* targets,
                              int64_t N, int32_t ignore_index, uint32_t flags,
                              float* lse, float* row_loss, float* loss,
                              int32_t* n_valid, void* stream);
flce_status flce_vocab_shard_bwd(const void* hidden, const void* weight_shard,
                                 const int32_t* targets, int64_t N, int64_t H,
                                 int64_t V_shard, int64_t v0, int64_t V_total,
                                 int32_t ignore_index, uint32_t flags, const float* lse,
                                 float* grad_hidden_partial, float* grad_weight_shard,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * grad_hidden (bf16 [N,H]) and grad_weight (fp32 [V,H]) multiplied in place by
 * the fp32 scalar at device address `scale` (read on the device, so the call
 * does not synchronise).  This is the backward of the fused op inside an
 * autograd graph: flce_fwd_bwd already produced the gradients of the loss, and
 * the backward pass only scales them by the incoming gradient of the loss
 * ("efficient-llm-anatomy" README, "Fused cross-entropy computes backward
 * during forward": the backward pass just distributes them).  H % 8 == 0;
 * pointers 16-byte aligned (scale 4-byte).
 */
flce_status flce_scale_grads(void* grad_hidden, float* grad_weight, int64_t N,
                             int64_t H, int64_t V, const float* scale,
                             void* stream);

/*
 * Error reporting of this library (the pages specify none).
 * Synchronises `stream`, then reads the device status word of the last call
 * that used `workspace`: FLCE_OK, FLCE_EBADTARGET or FLCE_ETIMEOUT (or
 * FLCE_ECUDA if the stream reports an error).
 */
flce_status flce_query_status(const void* workspace, void* stream);

/*
 * Where the first pipeline wait of the last call on `workspace` ran out of
 * time (after FLCE_ETIMEOUT).  Synchronises `stream`.  info[0] = wait site
 * (0 = none; 10 = an epilogue waiting for its accumulator, 6 = the MMA
 * issuer waiting for a free accumulator, 7 = the MMA issuer waiting for
 * operands, 3 = the TMA producer waiting for a free stage; the others are
 * the scheduler hand-offs), info[1] = CTA rank in its pair, info[2] = block
 * index, info[3] = number of waits that ran out.
 */
flce_status flce_query_stall(const void* workspace, int32_t* info /* [4] */, void* stream);

/*
 * Test hook for the failure path of the GEMM pipeline: arms the next tcgen05
 * GEMM launch of this process (a one-shot, process-wide switch) so that its
 * MMA issuer withholds the accumulator-ready signal of the first tile of every
 * CTA pair.  The epilogue's bounded wait for that signal then runs out after
 * timeout_ns (<= 10 s); the kernel raises its abort flag, lets the copies in
 * flight land, waits for its MMAs, frees TMEM and returns.  The call's status
 * becomes FLCE_ETIMEOUT and its loss NaN; the CUDA context stays usable.
 */
flce_status flce_debug_arm_stall(uint64_t timeout_ns);

/*
 * Diagnostic: enqueue one kernel that waits on a pipeline barrier nothing
 * will ever signal, bounded by timeout_ns, so that the timeout path (status
 * word set to FLCE_ETIMEOUT, kernel returns normally) can be exercised
 * without hanging the GPU.  Needs >= 256 bytes of workspace.
 */
flce_status flce_selftest_timeout(void* workspace, uint64_t timeout_ns,
                                  void* stream);

/*
 * flce_fwd_bwd without a workspace argument, for callers that cannot
 * allocate device memory (code inside a CUDA graph capture or an allocator
 * hook, plugins whose host framework owns every cudaMalloc, fixed memory
 * budgets).  The pages have no counterpart: it is a deployment variant of
 * flce_fwd_bwd with the same arguments, outputs and tolerances.
 *   Scratch: a static device array of FLCE_NOALLOC_WORKSPACE_BYTES (64 MiB)
 *     inside the library.  A GPU holds it from the moment it loads the
 *     array's module until the process exits: with CUDA's lazy module loading
 *     (the default under PyTorch) that is this entry point's first call on the
 *     device, with eager loading the loading of the library.  The call itself
 *     allocates nothing.
 *   Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   Limits: sizes whose smallest plan (one 128-token chunk) does not fit in
 *     the array are rejected with FLCE_EWORKSPACE; larger problems run with
 *     smaller chunks than flce_fwd_bwd's default plan.
 *   Sharing: every call on a device uses the same array.  Calls that overlap
 *     on the GPU (other streams, other threads) race and give wrong results;
 *     serialise them.  The array needs no clearing between calls.
 *   Device-side status (bad targets, time-outs) is written into the array
 *     and cannot be read back through flce_query_status; such a call writes
 *     a NaN loss.
 */
#define FLCE_NOALLOC_WORKSPACE_BYTES (64u * 1024u * 1024u)
flce_status flce_fwd_bwd_noalloc(const void* hidden, const void* weight,
                                 const int32_t* targets, int64_t N, int64_t H,
                                 int64_t V, int32_t ignore_index, uint32_t flags,
                                 float* loss, int32_t* n_valid, float* row_loss,
                                 void* grad_hidden, float* grad_weight,
                                 void* stream);

/*
 * Launch profiling (for benchmarks).  Between flce_profile_begin() and
 * flce_profile_end(), every call records a pair of CUDA events around each
 * of its tcgen05 GEMM launches on the call's stream and counts every kernel
 * it launches.  flce_profile_end() synchronises those events and returns, per
 * GEMM launch kind (0 = logits, 1 = backward: grad_hidden and grad_weight
 * tiles in one launch, 2 = unused), the summed device time in milliseconds
 * and the number of launches, plus the total number of kernels launched.  Any output pointer may be NULL.  Profiling is
 * process-wide and not meant to be used from several threads at once.
 */
flce_status flce_profile_begin(void);
flce_status flce_profile_end(double* gemm_ms /* [3] */, int64_t* gemm_launches /* [3] */,
                             int64_t* kernel_launches);

/* Static English description of a status code (error reporting of this
 * library; the pages specify none). */
const char* flce_status_string(flce_status s);

/* Library version, e.g. "0.1.0" (no counterpart in the pages). */
const char* flce_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H */
