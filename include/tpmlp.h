/*
 * tpmlp -- the Megatron tensor-parallel MLP sublayer on one GB300 (sm_103a).
 *
 * The sublayer (page "Megatron tensor-parallel MLP", synapticradio.com,
 * section "Start with the dense block"):
 *
 *     n  = RMSNorm(x) * norm_w                       (pre-norm)
 *     G  = n W_g^T, U = n W_u^T                      (column-parallel, W_gate_up [2,F,H])
 *     A  = SiLU(G) * U                                (per FFN shard, no reduction)
 *     y  = x + sum_{s=0}^{t-1} A_s W_d,s^T + b_down   (row-parallel + the g reduction)
 *
 * or, with TPMLP_GELU (page "Megatron-LM walkthrough", Part II, and page
 * "Megatron-LM Explained", "The MLP block: column-parallel, then row-parallel"):
 *
 *     A  = GeLU(n W_1^T + b_1),  W_1 [F,H], b_1 [F]
 *
 * plus the mirrored backward (the f reduction of the normed-input gradient,
 * section "Put the other collective in backward"), a mean-squared-error loss
 * and one SGD update.  The tensor-parallel degree t is a logical split of the
 * FFN axis inside one process: rank r owns channels [r F/t, (r+1) F/t) of the
 * gate rows, the up rows and the down columns alike (the fixture's shared
 * interval, "Start with the dense block").  Both reductions are summed on the
 * device inside the GEMM accumulators, in shard order 0..t-1.
 *
 * Conventions for every entry point:
 *  - All tensors are row-major and contiguous, in device memory owned by the
 *    caller.  The library never allocates or frees device memory: scratch
 *    lives in a caller-provided workspace (tpmlp_bind_workspace).
 *  - Element type: TPMLP_F32 -> every tensor is float.  TPMLP_BF16 -> x, y,
 *    dy, dx, target and the parameters are bfloat16; all parameter
 *    gradients and master weights are float (fp32 accumulate everywhere).
 *  - Calls are asynchronous on the context's CUDA stream.  They return after
 *    validating arguments and enqueuing kernels.  Device-side failures
 *    (a bounded wait that gave up) are reported by tpmlp_sync.
 *  - No call throws; each returns a tpmlp_status.  On error nothing is
 *    enqueued, and tpmlp_last_error() holds a one-line message.
 *  - Pointers must be 16-byte aligned.  H and F must be multiples of 8.
 */
#ifndef TPMLP_H_
#define TPMLP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TPMLP_API __attribute__((visibility("default")))
#else
#define TPMLP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tpmlp_ctx tpmlp_ctx;

typedef enum {
  TPMLP_OK = 0,
  TPMLP_ERR_ARG = 1,          /* null / misaligned pointer, bad value */
  TPMLP_ERR_SHAPE = 2,        /* F % t != 0, H or F not a multiple of 8, tokens > max_tokens */
  TPMLP_ERR_UNSUPPORTED = 3,  /* dtype/activation value, or device is not sm_103 */
  TPMLP_ERR_ORDER = 4,        /* no workspace; backward before forward; sgd before backward */
  TPMLP_ERR_CUDA = 5,         /* a CUDA runtime call failed */
  TPMLP_ERR_TIMEOUT = 6       /* a bounded device-side wait gave up (reported by tpmlp_sync) */
} tpmlp_status;

typedef enum { TPMLP_F32 = 0, TPMLP_BF16 = 1 } tpmlp_dtype;
typedef enum { TPMLP_SWIGLU = 0, TPMLP_GELU = 1 } tpmlp_act;

/* Debug flags (tpmlp_set_debug).  The two SKIP flags reproduce the broken
 * variants of section "Remove each collective" as seen by one rank `shard`:
 *  SKIP_FWD_REDUCE: the g reduction is replaced by shard `shard`'s own
 *    partial, y = x + A_s W_d,s^T + b_down; the backward then runs from that
 *    output's dy for every shard.
 *  SKIP_BWD_REDUCE: the f reduction is replaced by shard `shard`'s own
 *    normed-input gradient.
 *  FORCE_TIMEOUT: the next forward's first GEMM waits on an event that never
 *    happens, gives up after ~2 ms and records TPMLP_ERR_TIMEOUT (tests the
 *    bounded-wait path without a hang).
 *  GEMM_SINGLE_CTA: run the bf16 GEMMs with single-CTA 128x256 tiles instead
 *    of CTA-pair 256x256 tiles (same results up to rounding; for testing). */
enum {
  TPMLP_DBG_SKIP_FWD_REDUCE = 1u,
  TPMLP_DBG_SKIP_BWD_REDUCE = 2u,
  TPMLP_DBG_FORCE_TIMEOUT = 4u,
  TPMLP_DBG_GEMM_SINGLE_CTA = 8u,
  /* Sequence parallelism without the all-reduce of the norm-weight and
   * output-bias gradients ("Megatron-LM walkthrough", "Stage 7:
   * finalize_model_grads"): dnorm_w and db_down are the debug shard's sums
   * over its own tokens. */
  TPMLP_DBG_SKIP_SP_GRAD_SYNC = 16u
};

typedef struct {
  int64_t max_tokens; /* N upper bound (tokens = batch * seq) for workspace sizing */
  int64_t hidden;     /* H */
  int64_t ffn;        /* F */
  int32_t max_t;      /* largest logical TP degree that will be passed to forward */
  int32_t dtype;      /* tpmlp_dtype */
  int32_t act;        /* tpmlp_act */
  int32_t reserved;   /* must be 0 */
} tpmlp_config;

/* Validate `cfg` and create a context bound to `cuda_stream` (a cudaStream_t,
 * NULL = legacy default stream) on the current device.  Host-only checks run
 * first, so a bad config is rejected without touching the GPU. */
TPMLP_API tpmlp_status tpmlp_create(const tpmlp_config* cfg, void* cuda_stream, tpmlp_ctx** out);

/* Bytes of device workspace a context with `cfg` needs (saved activations
 * n/rstd/G,U/A, the backward intermediates dGU and dN, reduction partials,
 * the device status word and, for bf16, 40 MB of scratch for the partial sums
 * of GEMM tiles whose contraction is split along K in a launch's last wave).
 * 0 if `cfg` is invalid. */
TPMLP_API size_t tpmlp_workspace_bytes(const tpmlp_config* cfg);

/* Hand the context `bytes` of device memory at `dev` (256-byte aligned).  The
 * caller owns it and keeps it alive until tpmlp_destroy.  Zeroes the status
 * word and the split GEMMs' arrival flags (enqueued on the stream); the rest
 * of the workspace needs no initial contents. */
TPMLP_API tpmlp_status tpmlp_bind_workspace(tpmlp_ctx* ctx, void* dev, size_t bytes);

/* Change the stream later calls enqueue on. */
TPMLP_API tpmlp_status tpmlp_set_stream(tpmlp_ctx* ctx, void* cuda_stream);

/* Forward of the sublayer for `tokens` rows (0 <= tokens <= max_tokens).
 *  x [tokens,H], norm_w [H], w_gate_up [2,F,H] (SwiGLU; GeLU: W_1 [F,H]),
 *  b_1 [F] (GeLU only, NULL for SwiGLU), w_down [H,F], b_down [H] -> y [tokens,H].
 *  eps: RMSNorm epsilon, inside the square root.  t: logical TP degree,
 *  1 <= t <= max_t and F % t == 0 (the fixture's divisibility assertion).
 * The pointers of x and of the parameters are remembered: backward reads x,
 * and the updates write the parameters in place, so they must stay valid
 * until then. */
TPMLP_API tpmlp_status tpmlp_forward(tpmlp_ctx* ctx, int64_t tokens, const void* x, const void* norm_w,
                           const void* w_gate_up, const void* b_1, const void* w_down,
                           const void* b_down, float eps, int32_t t, void* y);

/* loss = 0.5 * mean((y - target)^2) over tokens*H elements, written as one
 * float to device memory `loss_dev`; dy = (y - target) / (tokens*H).
 * y, target, dy: [tokens,H] in the activation dtype.  tokens from the last forward. */
TPMLP_API tpmlp_status tpmlp_mse_loss_grad(tpmlp_ctx* ctx, const void* y, const void* target, void* dy,
                                 float* loss_dev);

/* Backward of the last forward, given dy [tokens,H].  Outputs: dx [tokens,H]
 * (activation dtype); float gradients dnorm_w [H], dw_gate_up [2,F,H]
 * (GeLU: dW_1 [F,H]), db_1 [F] (GeLU only, else NULL), dw_down [H,F],
 * db_down [H].  Gradients are overwritten, not accumulated. */
TPMLP_API tpmlp_status tpmlp_backward(tpmlp_ctx* ctx, const void* dy, void* dx, float* dnorm_w,
                            float* dw_gate_up, float* db_1, float* dw_down, float* db_down);

/* Bind float master copies of the parameters (same shapes) for the bf16
 * dtype.  When bound, sgd_step updates the masters and rewrites the bf16
 * parameters as their round-to-nearest-even copies.  All or none (b_1 only
 * for GeLU).  Passing all NULL unbinds. */
TPMLP_API tpmlp_status tpmlp_bind_master(tpmlp_ctx* ctx, float* norm_w, float* w_gate_up, float* b_1,
                               float* w_down, float* b_down);

/* One plain SGD update, w <- w - lr * g, of every parameter of the last
 * forward with the gradients of the last backward.  F32: in place on the
 * parameters.  BF16 with masters: masters updated, parameters re-rounded.
 * BF16 without masters: parameters updated through float and re-rounded. */
TPMLP_API tpmlp_status tpmlp_sgd_step(tpmlp_ctx* ctx, float lr);

/* One fp32 tensor per parameter, each laid out like that parameter
 * (b_1 is the GeLU first-projection bias; NULL for SwiGLU). */
typedef struct {
  float* norm_w;
  float* w_gate_up;
  float* b_1;
  float* w_down;
  float* b_down;
} tpmlp_param_set;

/* Hyperparameters of one AdamW step ("Megatron-LM walkthrough", "Stage 8",
 * whose launch example uses lr 1.5e-4, weight decay 0.1, clip 1.0). */
typedef struct {
  float lr;            /* learning rate, finite */
  float beta1, beta2;  /* moment decay rates, each in [0, 1) */
  float eps;           /* added to the root of the corrected second moment, >= 0 */
  float weight_decay;  /* decoupled decay, applied to w_gate_up (or W_1) and w_down only */
  float max_grad_norm; /* clip the global L2 gradient norm to this; <= 0 turns clipping off */
  int64_t step;        /* 1-based index of this update, for the bias corrections */
} tpmlp_adamw_params;

/* Bind the first (m) and second (v) moment estimates of AdamW: device fp32
 * tensors owned by the caller, zero before the first step and carried from
 * step to step by the caller.  They must stay valid while adamw_step runs.
 * Every pointer is 16-byte aligned; b_1 is set exactly for GeLU.  Passing
 * two NULL sets unbinds.  TPMLP_ERR_ARG on a missing or misaligned tensor. */
TPMLP_API tpmlp_status tpmlp_bind_adam_state(tpmlp_ctx* ctx, const tpmlp_param_set* m, const tpmlp_param_set* v);

/* One AdamW update of every parameter of the last forward, with the
 * gradients of the last backward, after clipping them by their global norm
 * (the walkthrough's optimizer step, "Stage 8"):
 *   c = min(1, max_grad_norm / (||g|| + 1e-6))   (1 if max_grad_norm <= 0)
 *   m <- b1 m + (1 - b1) c g;   v <- b2 v + (1 - b2) (c g)^2
 *   w <- w - lr wd w - lr (m / (1 - b1^step)) / (sqrt(v / (1 - b2^step)) + eps)
 * ||g|| runs over every parameter gradient; wd is weight_decay for the
 * projection matrices and 0 for norm_w and the biases.  Parameters follow
 * sgd_step's rules (f32 in place; bf16 through the bound fp32 masters, bf16
 * copies re-rounded; bf16 without masters through float).  `grad_norm`, if
 * not NULL, is a device float that receives ||g|| before clipping.
 * Two kernels: a norm pass over the gradients, then the update.
 * TPMLP_ERR_ORDER before a backward; TPMLP_ERR_ARG without bound moments or
 * with hyperparameters out of range. */
TPMLP_API tpmlp_status tpmlp_adamw_step(tpmlp_ctx* ctx, const tpmlp_adamw_params* hp, float* grad_norm);

/* GEMM operand precision of the bf16 dtype. */
typedef enum { TPMLP_PREC_BF16 = 0, TPMLP_PREC_FP8 = 1 } tpmlp_precision;

/* Bytes of the extra device workspace the FP8 precision needs (E4M3 copies
 * of every GEMM operand, row-major and transposed, and their scales); 0 for
 * the f32 dtype or an invalid config. */
TPMLP_API size_t tpmlp_fp8_workspace_bytes(const tpmlp_config* cfg);

/* Hand the context the FP8 workspace (256-byte aligned, caller-owned, kept
 * alive until tpmlp_destroy).  TPMLP_ERR_UNSUPPORTED for the f32 dtype. */
TPMLP_API tpmlp_status tpmlp_bind_fp8_workspace(tpmlp_ctx* ctx, void* dev, size_t bytes);

/* Select the GEMM operand precision (page "Megatron-Core Architecture: 5D
 * Distributed Parallelism, ... FP8 Transformer Engine", its list of
 * Megatron-Core subsystems, item 6).  TPMLP_PREC_FP8: before each of the six
 * GEMMs its two operands are cast to E4M3 with one scale per tensor (448 /
 * the tensor's current absolute maximum; tpmlp_fp8_quantize), row-major and
 * transposed so that every GEMM reads K-major codes; the tensor cores
 * multiply the codes with fp32 accumulation and the epilogue divides by both
 * scales before its element-wise step.  Activations, gradients and the
 * optimizer stay as in TPMLP_PREC_BF16.  Needs the bf16 dtype
 * (TPMLP_ERR_UNSUPPORTED) and a bound FP8 workspace (TPMLP_ERR_ORDER); the
 * shard restrictions of the SKIP flags must fall on 128-element blocks.
 * Changing the precision requires a new forward. */
TPMLP_API tpmlp_status tpmlp_set_precision(tpmlp_ctx* ctx, int32_t precision);

/* Sequence-parallel form ("Megatron-LM walkthrough", "Deep dive: sequence
 * parallelism, memory for free"): shard s of t owns the contiguous tokens
 * [s N/t, (s+1) N/t) outside the tensor-parallel region.  On one GPU the
 * all-gather into that region and the reduce-scatter out of it are the
 * identity on the token-major layout, so forward outputs and the projection
 * gradients are those of the plain form; dnorm_w and db_down are taken per
 * shard and then summed across the shards in shard order (the all-reduce of
 * the sequence-parallel norm gradients).  While enabled, forward needs
 * tokens % t == 0 and t <= 64 (TPMLP_ERR_SHAPE) and rejects the
 * SKIP_FWD/BWD_REDUCE flags (TPMLP_ERR_UNSUPPORTED).  Changing the mode
 * requires a new forward. */
TPMLP_API tpmlp_status tpmlp_set_sequence_parallel(tpmlp_ctx* ctx, int32_t enable);

/* The SGD update applied by backward (bf16 dtype with fp32 masters bound;
 * "Megatron-LM walkthrough", "Stage 8: the optimizer step").  While enabled,
 * tpmlp_backward still writes every gradient, and also applies
 * w <- w - lr * g to the fp32 masters and bf16 copies of the parameters of
 * the last forward.  With at least 8192 tokens, W_gate_up (W_1) and W_down
 * are updated inside the epilogues of the GEMMs that produce their
 * gradients (their contraction over the tokens then hides the masters' reads
 * and writes); with fewer, and for the other parameters, the update kernel
 * runs at the end of backward.  The arithmetic is tpmlp_sgd_step's, so
 * masters and copies are bit-identical to backward followed by
 * tpmlp_sgd_step(lr).  The data-gradient GEMM into the normed input runs
 * before the gate/up weight gradient, so every read of a weight precedes its
 * update.  After such a
 * backward, tpmlp_sgd_step and tpmlp_adamw_step return TPMLP_ERR_ORDER until
 * the next forward.  Errors: TPMLP_ERR_UNSUPPORTED for the fp32 dtype,
 * TPMLP_ERR_ARG for a non-finite lr, and TPMLP_ERR_ORDER from backward when
 * no masters are bound.  enable = 0 turns it off (lr is then ignored). */
TPMLP_API tpmlp_status tpmlp_set_update_in_backward(tpmlp_ctx* ctx, int32_t enable, float lr);

/* 1 if the last backward updated W_gate_up (W_1) and W_down inside their
 * weight-gradient epilogues, 0 otherwise (no update in backward, fewer than
 * 8192 tokens, or a NULL context).  Never fails. */
TPMLP_API int32_t tpmlp_update_in_epilogue(const tpmlp_ctx* ctx);

/* Debug flags (TPMLP_DBG_*) and the shard whose view the SKIP flags take. */
TPMLP_API tpmlp_status tpmlp_set_debug(tpmlp_ctx* ctx, uint32_t flags, int32_t shard);

/* Wait for the stream, then report an asynchronous CUDA error or a device
 * status word set by a bounded wait (TPMLP_ERR_TIMEOUT; the word is cleared). */
TPMLP_API tpmlp_status tpmlp_sync(tpmlp_ctx* ctx);

/* Per-kernel CUDA-event timing on the context's stream: enable/disable, then
 * read the summed milliseconds and launch counts per kernel id since the last
 * read (this call synchronises the stream).  `n` = array capacity; returns
 * the number of kernel ids written. */
TPMLP_API tpmlp_status tpmlp_set_timing(tpmlp_ctx* ctx, int32_t enable);
TPMLP_API int32_t tpmlp_read_kernel_times(tpmlp_ctx* ctx, float* ms, int64_t* launches, int32_t n);
/* Name of kernel id `id` (0 <= id < tpmlp_num_kernel_ids()), or NULL. */
TPMLP_API const char* tpmlp_kernel_name(int32_t id);
TPMLP_API int32_t tpmlp_num_kernel_ids(void);

/* Number of kernels this context has launched since creation. */
TPMLP_API uint64_t tpmlp_launch_count(const tpmlp_ctx* ctx);

/* Static text for a status code; the last error message of a context
 * (or of the calling thread when ctx is NULL, e.g. after a failed create). */
TPMLP_API const char* tpmlp_status_string(tpmlp_status s);
TPMLP_API const char* tpmlp_last_error(const tpmlp_ctx* ctx);

/* Free the host-side context.  Does not touch caller memory. */
TPMLP_API void tpmlp_destroy(tpmlp_ctx* ctx);

/* ---------------------------------------------------------------- FP8 building blocks
 * The FP8 GEMMs of page "Megatron-Core Architecture: 5D Distributed
 * Parallelism, ... FP8 Transformer Engine" (its subsystem list, item 6):
 * E4M3 operands with one scale per tensor.  The FP8 training step
 * (tpmlp_set_precision) is built from these two operations. */

/* Device scratch that tpmlp_fp8_quantize needs (partial maxima). */
#define TPMLP_FP8_SCRATCH_BYTES 4096

/* Cast a bf16 tensor src [rows, cols] (row-major, contiguous, cols % 8 == 0)
 * to E4M3 with its current per-tensor scale s = 448 / max|src| (float32;
 * s = 1 when src is all zero): code = round-to-nearest-even(src * s),
 * saturated to +-448.  Writes the codes row-major to dst [rows, cols] (pitch
 * ld_dst bytes) and/or transposed to dst_t [cols, rows] (pitch ld_dst_t
 * bytes); either may be NULL, not both.  Pitches are multiples of 16 and
 * pointers 16-byte aligned.  *inv_scale (device float) receives 1 / s.
 * scratch: TPMLP_FP8_SCRATCH_BYTES of device memory.  Asynchronous on
 * `stream`.  TPMLP_ERR_SHAPE / TPMLP_ERR_ARG on bad sizes or pointers. */
TPMLP_API tpmlp_status tpmlp_fp8_quantize(const void* src, int64_t rows, int64_t cols, uint8_t* dst, int64_t ld_dst,
                                          uint8_t* dst_t, int64_t ld_dst_t, float* inv_scale, void* scratch,
                                          void* stream);

/* c [M, N] (float, pitch ldc elements) = (a b^T) * (*inv_scale_a) *
 * (*inv_scale_b), with a [M, K] and b [N, K] E4M3 codes (K-major, pitches
 * lda, ldb bytes, multiples of 16): the tcgen05 kind::f8f6f4 tensor-core
 * GEMM with fp32 accumulation.  N % 4 == 0.  `status` is a device word the
 * caller zeroes; a bounded wait that gives up sets it nonzero.
 * Asynchronous on `stream`. */
TPMLP_API tpmlp_status tpmlp_fp8_gemm(const uint8_t* a, int64_t lda, const uint8_t* b, int64_t ldb, int64_t M,
                                      int64_t N, int64_t K, const float* inv_scale_a, const float* inv_scale_b,
                                      float* c, int64_t ldc, uint32_t* status, void* stream);

/* ---------------------------------------------------------------- attention sublayer
 * The tensor-parallel attention sublayer ("Megatron-LM Explained",
 * "Self-attention: split across heads"; page "Megatron-Core Architecture: 5D
 * Distributed Parallelism, ...": W_QKV split column-wise, W_out row-wise, one
 * all-reduce; page "Megatron tensor-parallel MLP", closing note: grouped-query
 * attention keeping complete query/KV head groups per rank):
 *
 *     n = RMSNorm(x) * norm_w
 *     [Q | K | V] = n W_qkv^T,  W_qkv [(n_q + 2 n_kv) d, H] (query, key, value rows)
 *     Z_h = softmax_causal(Q_h K_g^T / sqrt(d)) V_g  for query head h, group g = h / (n_q / n_kv)
 *     y = x + sum over ranks of Z_r W_o,r^T + b_o,  W_o [H, n_q d]
 *
 * Tokens are `batch` sequences of `seq` rows each (token-major, [batch*seq, H]);
 * the mask is causal within each sequence.  Rank r of t owns KV groups
 * [r n_kv/t, (r+1) n_kv/t) and their query heads; on one GPU the ranks'
 * partial outputs and normed-input gradients are summed on chip in head
 * order.  bf16 storage, fp32 accumulation.  Two kernel paths compute the
 * same function: the fused one (default where head_dim == 128 and seq % 128
 * == 0) streams key/value blocks through tensor memory with an online
 * softmax and never stores scores (the backward recomputes them from each
 * query row's log-sum-exp); the unfused one materialises the scores and their
 * gradient per (sequence, head) in the workspace (fp32 scores, bf16
 * probabilities).  Loss: tpmlp_mse_loss_grad_noalloc.  Same conventions as
 * the MLP calls above (caller-owned memory, asynchronous, status codes). */
typedef struct tpattn_ctx tpattn_ctx;
typedef struct {
  int64_t max_tokens; /* batch * seq upper bound */
  int64_t hidden;     /* H, a multiple of 8, at most 8192 */
  int32_t n_heads;    /* query heads n_q, a multiple of n_kv_heads */
  int32_t n_kv_heads; /* key/value heads n_kv (groups) */
  int32_t head_dim;   /* d: 64, 128, 192 or 256 */
  int32_t max_seq;    /* largest seq, a multiple of 64, at most 4096 (TPATTN_FUSED_ONLY: 128, 32768) */
  int32_t max_t;      /* largest logical TP degree; must divide n_kv_heads */
  int32_t dtype;      /* TPMLP_BF16 */
  int32_t flags;      /* 0, or TPATTN_FUSED_ONLY */
} tpattn_config;

/* flags: only the fused attention kernels run.  The workspace then holds no
 * score square (batch * n_q * seq^2 * 6 bytes on the unfused path), which
 * lets max_seq go up to 32768 (a multiple of 128); head_dim must be 128,
 * every forward's seq a multiple of 128 (else TPMLP_ERR_SHAPE), and
 * tpattn_set_fused(ctx, 0) returns TPMLP_ERR_UNSUPPORTED. */
#define TPATTN_FUSED_ONLY 1

TPMLP_API size_t tpattn_workspace_bytes(const tpattn_config* cfg);
TPMLP_API tpmlp_status tpattn_create(const tpattn_config* cfg, void* cuda_stream, tpattn_ctx** out);
/* As tpmlp_bind_workspace, for the attention context (tpattn_workspace_bytes). */
TPMLP_API tpmlp_status tpattn_bind_workspace(tpattn_ctx* ctx, void* dev, size_t bytes);
/* batch sequences of seq tokens (seq % 64 == 0, seq <= max_seq); t divides n_kv_heads.
 * x [batch*seq, H], norm_w [H], w_qkv [(n_q+2n_kv) d, H], w_o [H, n_q d], b_o [H] -> y.
 * The pointers of x and of the parameters are remembered: backward reads x,
 * and the updates write the parameters in place, so they must stay valid
 * until then. */
TPMLP_API tpmlp_status tpattn_forward(tpattn_ctx* ctx, int64_t batch, int64_t seq, const void* x, const void* norm_w,
                                      const void* w_qkv, const void* w_o, const void* b_o, float eps, int32_t t,
                                      void* y);
/* dx (bf16) and float gradients dnorm_w [H], dw_qkv, dw_o, db_o. */
TPMLP_API tpmlp_status tpattn_backward(tpattn_ctx* ctx, const void* dy, void* dx, float* dnorm_w, float* dw_qkv,
                                       float* dw_o, float* db_o);
TPMLP_API tpmlp_status tpattn_bind_master(tpattn_ctx* ctx, float* norm_w, float* w_qkv, float* w_o, float* b_o);
/* enable != 0 (the default): forwards whose shape allows it (head_dim 128,
 * seq % 128 == 0) run the fused attention kernels; 0: always the unfused
 * path.  Takes effect at the next tpattn_forward; a backward follows the path
 * of its forward. */
TPMLP_API tpmlp_status tpattn_set_fused(tpattn_ctx* ctx, int32_t enable);
/* 1 if the last tpattn_forward ran the fused kernels, 0 if not (or no forward yet). */
TPMLP_API int32_t tpattn_fused_active(const tpattn_ctx* ctx);
TPMLP_API tpmlp_status tpattn_sgd_step(tpattn_ctx* ctx, float lr);

/* Have tpattn_backward apply the SGD update itself, as tpmlp_set_update_in_backward
 * does for the MLP ("Megatron-LM walkthrough", "Stage 8: the optimizer step").
 * While enabled, tpattn_backward still writes every gradient, and also applies
 * w <- w - lr * g to the bound fp32 masters and bf16 copies of the parameters
 * of the last forward.  With at least 8192 tokens (batch * seq), W_qkv and W_o
 * are updated inside the epilogues of the GEMMs that produce their gradients;
 * with fewer, and for norm_w and b_o, the update kernel runs at the end of
 * backward.  Masters and copies are bit-identical to backward followed by
 * tpattn_sgd_step(lr).  The data-gradient GEMM into the normed input runs
 * before the QKV weight gradient, and dZ = dy W_o before the output
 * projection's weight gradient, so every read of a weight precedes its
 * update.  After such a backward, tpattn_sgd_step and tpattn_adamw_step
 * return TPMLP_ERR_ORDER until the next forward.  Errors: TPMLP_ERR_ARG for a
 * non-finite lr, and TPMLP_ERR_ORDER from backward when no masters are bound.
 * enable = 0 turns it off (lr is then ignored). */
TPMLP_API tpmlp_status tpattn_set_update_in_backward(tpattn_ctx* ctx, int32_t enable, float lr);

/* 1 if the last tpattn_backward updated W_qkv and W_o inside their
 * weight-gradient epilogues, 0 otherwise (no update in backward, fewer than
 * 8192 tokens, or a NULL context).  Never fails. */
TPMLP_API int32_t tpattn_update_in_epilogue(const tpattn_ctx* ctx);

/* The attention sublayer's four parameters, one fp32 device tensor each
 * (shapes as in tpattn_forward); used for the AdamW moments. */
typedef struct {
  float* norm_w; /* [H] */
  float* w_qkv;  /* [(n_q + 2 n_kv) d, H] */
  float* w_o;    /* [H, n_q d] */
  float* b_o;    /* [H] */
} tpattn_param_set;

/* Bind the AdamW moments m and v of the attention parameters: caller-owned
 * fp32 device tensors, zero before the first step, 16-byte aligned, valid
 * while tpattn_adamw_step runs.  Two NULL sets unbind.  TPMLP_ERR_ARG on a
 * missing or misaligned tensor. */
TPMLP_API tpmlp_status tpattn_bind_adam_state(tpattn_ctx* ctx, const tpattn_param_set* m, const tpattn_param_set* v);

/* One clipped AdamW update of the attention parameters with the gradients of
 * the last tpattn_backward: the rule of tpmlp_adamw_step (global-norm
 * clipping over all four gradients, bias-corrected moments, decoupled
 * weight decay on w_qkv and w_o only).  bf16 parameters are updated through
 * the bound fp32 masters (tpattn_bind_master) and re-rounded, or through
 * float when none are bound.  `grad_norm`, if not NULL, is a device float
 * that receives the norm before clipping.  Two kernels (norm pass, update).
 * TPMLP_ERR_ORDER before a backward; TPMLP_ERR_ARG without bound moments or
 * with hyperparameters out of range. */
TPMLP_API tpmlp_status tpattn_adamw_step(tpattn_ctx* ctx, const tpmlp_adamw_params* hp, float* grad_norm);
TPMLP_API tpmlp_status tpattn_sync(tpattn_ctx* ctx);
TPMLP_API tpmlp_status tpattn_set_timing(tpattn_ctx* ctx, int32_t enable);
TPMLP_API int32_t tpattn_read_kernel_times(tpattn_ctx* ctx, float* ms, int64_t* launches, int32_t n);
TPMLP_API const char* tpattn_kernel_name(int32_t id);
TPMLP_API int32_t tpattn_num_kernel_ids(void);
TPMLP_API uint64_t tpattn_launch_count(const tpattn_ctx* ctx);
TPMLP_API const char* tpattn_last_error(const tpattn_ctx* ctx);
TPMLP_API void tpattn_destroy(tpattn_ctx* ctx);

/* Loss and loss gradient without any device allocation or workspace.
 *
 * The method itself has no such call: this entry point exists for callers that
 * cannot call cudaMalloc -- code whose device memory is owned by a host
 * framework's pool and budget, or a latency-bound loop where an allocation
 * (which may synchronise the device) is not acceptable.  It computes the same
 * result as tpmlp_mse_loss_grad, without a context:
 *   loss = 0.5 * mean((y - target)^2) over n elements -> *loss_dev (float),
 *   dy   = (y - target) / n,
 * with y, target, dy of `dtype` (TPMLP_F32 or TPMLP_BF16), n >= 0 a multiple
 * of 8, pointers 16-byte aligned, enqueued on `cuda_stream`.
 * Its per-block partial sums live in a fixed array inside the library
 * (TPMLP_NOALLOC_LOSS_MAX_BLOCKS doubles, 8 KiB, held by every GPU that
 * loads the library until the process exits).  The loss kernel's grid is
 * capped at that many blocks, which stride over all n elements, so the array
 * bounds the number of partial sums and no n is refused for its sake.
 * The first call on a device looks up that array's device address (with the
 * device current) and keeps it for the life of the process: make that first
 * call before any stream capture, and do not use this entry point on a device
 * after cudaDeviceReset.  All calls share the array: calls whose kernels
 * overlap on the GPU race on it.  Each call writes every partial sum it reads.
 * Errors: TPMLP_ERR_UNSUPPORTED (dtype), TPMLP_ERR_SHAPE (n < 0 or not a
 * multiple of 8), TPMLP_ERR_ARG (NULL / misaligned), TPMLP_ERR_CUDA; the
 * message is in tpmlp_last_error(NULL). */
#define TPMLP_NOALLOC_LOSS_MAX_BLOCKS 1024
TPMLP_API tpmlp_status tpmlp_mse_loss_grad_noalloc(int32_t dtype, int64_t n, const void* y, const void* target,
                                                   void* dy, float* loss_dev, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* TPMLP_H_ */
