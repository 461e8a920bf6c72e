// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "epilogue.cuh"

namespace tpmlp {

// Device status word bits (written by kernels, read by tpmlp_sync).
constexpr uint32_t STATUS_TIMEOUT = 1u;

// C[M, N] = sum over the contraction segments of A(m, k) B(k, n).
//  A K-major : A(m,k) = a[m * lda + k]  (tensor [M, K_extent])
//  A MN-major: A(m,k) = a[k * lda + m]  (tensor [K_extent, M])
//  B K-major : B(k,n) = b[n * ldb + k]  (tensor [b_rows, K_extent])
//  B MN-major: B(k,n) = b[k * ldb + n]  (tensor [K_extent, N])
// paired (K-major B only): output channel n takes B rows n (gate) and
// pair_off + n (up); the epilogue receives both sums.
// Contraction segments [k0, k1) and [k2, k3) (k2 == k3 for one segment).
// Batched GEMMs (tensor-core path): one problem of M x N x K per batch index
// z = (z0, z1, z2) < dims, all with the same tensor maps.  Each operand's
// coordinates are shifted by base + z0 s0 + z1 s1 + z2 s2, separately for its
// contiguous ("col") and strided ("row") coordinate: for a K-major operand
// col = k and row = m or n; for an MN-major operand col = m or n and row = k.
// The output (and epilogue-input) coordinates shift by o.  Offsets of
// MN-major operands' columns are multiples of 64; M and N of a batched
// problem are multiples of 32, K of 64.
struct BatchOffsets {
  int64_t col[4] = {0, 0, 0, 0};  // base, s0, s1, s2
  int64_t row[4] = {0, 0, 0, 0};
};
struct BatchDesc {
  int dims[3] = {1, 1, 1};
  BatchOffsets a, b, o;
};

enum CausalMode { CAUSAL_NONE = 0, CAUSAL_SKIP_UPPER = 1, CAUSAL_K_UPTO = 2, CAUSAL_K_FROM = 3 };

struct GemmDesc {
  int M = 0, N = 0;
  int64_t k_extent = 0;  // K extent of the A/B tensors
  const void* a = nullptr;
  int64_t lda = 0;
  bool a_mn = false;
  const void* b = nullptr;
  int64_t ldb = 0;
  bool b_mn = false;
  int64_t b_rows = 0;  // rows of a K-major B tensor
  // Operand tensor extents (contiguous, strided) when they exceed the
  // problem's own (batched problems); 0 = the problem's extents.
  int64_t a_ext_col = 0, a_ext_row = 0, b_ext_col = 0, b_ext_row = 0;
  bool paired = false;
  int64_t pair_off = 0;
  int64_t kseg[4] = {0, 0, 0, 0};
  int epi = EPI_STORE_F32;
  EpiParams ep{};
  int tile_mode = 0;  // tensor-core path: 0 automatic, 1 single-CTA tiles, 2 CTA-pair tiles
  // FP8: A and B are E4M3 codes (K-major only, pitches in bytes, multiples of
  // 16); the accumulator is multiplied by (*deq_a) * (*deq_b) before the
  // epilogue (the inverse per-tensor scales, device floats).
  bool f8 = false;
  const float* deq_a = nullptr;
  const float* deq_b = nullptr;
  BatchDesc batch;
  // Attention problems (one segment, M = one sequence's queries or keys):
  // SKIP_UPPER leaves out output tiles wholly above the diagonal; K_UPTO
  // contracts only over K < the tile's last row + 1; K_FROM only over
  // K >= the tile's first row (all at tile granularity; the entries beyond
  // the causal boundary inside a tile must be zero in A).
  int causal = CAUSAL_NONE;
  // Tail split along K (tensor-core path): the tiles of the last, partial
  // wave of the persistent grid are cut into up to four contiguous K parts
  // run by otherwise idle CTAs; the parts after the first leave their f32
  // accumulators in `split_scratch` and count their arrival in
  // `split_counters` by writing the launch's epoch there, and the first
  // part adds the partials in part order.  NULL disables the split.  The
  // flags are zeroed when the workspace is bound and epochs are unique in
  // the process (so workspaces shared between contexts stay safe); a 32-bit
  // epoch repeats after 2^32 - 1 split launches, and a stale flag could then
  // match only if its slot had gone unwritten for all of them.
  float* split_scratch = nullptr;
  size_t split_scratch_bytes = 0;
  uint32_t* split_counters = nullptr;
  int split_counter_words = 0;
};

// Workspace regions for the tail split: partial accumulators of up to
// SPLIT_SLOTS tiles of 256 x 256 f32 (or twice as many 128 x 256 single-CTA
// tiles), and an arrival flag per later part of a split tile, CTA of the pair
// and epilogue warp (8 per slot, 16 per slot for single-CTA tiles).
constexpr int SPLIT_SLOTS = 160;
constexpr size_t SPLIT_SCRATCH_BYTES = (size_t)SPLIT_SLOTS * 256 * 256 * 4;
constexpr int SPLIT_COUNTER_WORDS = SPLIT_SLOTS * 16;

// tcgen05/TMA GEMM for bf16 operands (f32 accumulation in tensor memory), or
// E4M3 operands with f8 set.  Segment boundaries must be multiples of 64
// elements (128 for E4M3), except an end equal to k_extent.
cudaError_t launch_gemm_tc(const GemmDesc& g, cudaStream_t st, int num_sms, uint32_t* status, int force_timeout);

// fp32 SIMT GEMM (exact fp32 path), any segments.
cudaError_t launch_gemm_simt_f32(const GemmDesc& g, cudaStream_t st);

// Bounded wait on a flag nothing sets; records STATUS_TIMEOUT (debug aid).
cudaError_t launch_timeout_probe(uint32_t* status, cudaStream_t st);

// Row-wise and reduction kernels (dtype: 0 = f32, 1 = bf16).
// amax (optional): largest stored |normed value|, float bits, atomicMax (zeroed by the caller).
cudaError_t launch_rmsnorm_fwd(int dtype, const void* x, const void* w, float eps, void* nrm, float* rstd,
                               int64_t N, int64_t H, cudaStream_t st, uint32_t* amax = nullptr);
// RMSNorm backward blocks: a multiple of `shards` (N % shards == 0); each block
// covers rows of one token shard only, so the per-block partials of dnorm_w
// and db_down sum per shard.
int rmsnorm_bwd_blocks(int64_t N, int num_sms, int shards);
cudaError_t launch_rmsnorm_bwd(int dtype, const float* dnrm, const void* x, const float* rstd, const void* w,
                               const void* dy, void* dx, float* part_dw, float* part_db, int64_t N, int64_t H,
                               int shards, int nblocks, cudaStream_t st);
// out0[g][c] = sum_{p < nparts} part0[g * nparts + p][c] for g < groups (and the
// same for part1/out1 when part1 != nullptr); sums in a fixed order.
cudaError_t launch_colsum_finalize(const float* part0, float* out0, const float* part1, float* out1, int nparts,
                                   int64_t C, cudaStream_t st, int groups = 1);
int colsum_blocks(int64_t N, int num_sms);
cudaError_t launch_colsum_partials(int dtype, const void* in, int64_t ld, float* part, int64_t N, int64_t C,
                                   int nblocks, cudaStream_t st);
int loss_blocks(int64_t n, int num_sms);
cudaError_t launch_mse_loss_grad(int dtype, const void* y, const void* target, void* dy, double* part,
                                 int nblocks, int64_t n, float inv_count, cudaStream_t st);
cudaError_t launch_loss_finalize(const double* part, int nblocks, double scale, float* loss, cudaStream_t st);

struct SgdSeg {
  float* master;      // float master copy (or nullptr)
  const float* grad;  // float gradient
  void* w;            // parameter in the activation dtype
  int64_t n;          // elements (multiple of 4)
};
constexpr int SGD_MAX_SEGS = 6;
struct SgdArgs {
  SgdSeg seg[SGD_MAX_SEGS];
  int nseg;
  float lr;
};
cudaError_t launch_sgd(int dtype, const SgdArgs& a, int num_sms, cudaStream_t st);

// AdamW with global-norm clipping: one segment per parameter.
struct AdamSeg {
  float* master;      // float master copy (or nullptr)
  const float* grad;  // float gradient
  void* w;            // parameter in the activation dtype
  float* m;           // first moment
  float* v;           // second moment
  int64_t n;          // elements (multiple of 4)
  float lr_wd;        // lr * weight_decay for this parameter (0: no decay)
};
constexpr int ADAM_MAX_SEGS = 6;
constexpr int MAX_NORM_PARTS = 2048;
struct AdamArgs {
  AdamSeg seg[ADAM_MAX_SEGS];
  int nseg;
  float beta1, beta2;      // moment rates
  float one_m_beta1, one_m_beta2;
  float step_size;         // lr / (1 - beta1^step)
  float inv_sqrt_bc2;      // 1 / sqrt(1 - beta2^step)
  float eps;
  float max_norm;          // <= 0: no clipping
  double* part;            // per-block partial sums of g^2 (MAX_NORM_PARTS)
  float* grad_norm;        // optional device output
};
// Number of blocks (= norm partials) both AdamW kernels use.
int adam_blocks(const AdamArgs& a, int num_sms);
cudaError_t launch_grad_sqnorm(const AdamArgs& a, int nblocks, cudaStream_t st);
cudaError_t launch_adamw(int dtype, const AdamArgs& a, int nblocks, cudaStream_t st);

// FP8 casts: amax partials (at most FP8_MAX_PARTS floats in `part`), then
// E4M3 codes row-major (dst, pitch ld bytes) and/or transposed (dst_t, pitch
// ld_t bytes) with the scale 448 / amax; 1 / scale goes to *inv_scale.
constexpr int FP8_MAX_PARTS = 1024;
int fp8_blocks(int64_t elems, int num_sms);
cudaError_t launch_fp8_quantize(const void* src, int64_t rows, int64_t cols, uint8_t* dst, int64_t ld,
                                uint8_t* dst_t, int64_t ld_t, float* part, float* inv_scale, int num_sms,
                                cudaStream_t st);
// The two kernels of launch_fp8_quantize: nparts = fp8_blocks(rows * cols) partial maxima, then the cast.
cudaError_t launch_fp8_amax(const void* src, int64_t n, float* part, int nparts, cudaStream_t st);
cudaError_t launch_fp8_cast(const void* src, int64_t rows, int64_t cols, uint8_t* dst, int64_t ld, uint8_t* dst_t,
                            int64_t ld_t, const float* part, int nparts, float* inv_scale, int num_sms,
                            cudaStream_t st);

// Attention rows: P = causal softmax(scale * S) (bf16, zeros above the
// diagonal), dS = scale * P (dP - rowsum(P dP)) written over P, and the sum
// of per-query-head K/V gradients over each group into the QKV gradient.
// Rows of S floats (S % 4 == 0, S <= 4096), row r at query r % S.
cudaError_t launch_attn_softmax_fwd(const float* s, void* p, int64_t rows, int S, float scale, cudaStream_t st);
cudaError_t launch_attn_softmax_bwd(void* p, const float* dp, int64_t rows, int S, float scale, cudaStream_t st);
cudaError_t launch_attn_group_sum(const float* in, void* out, int batch, int S, int n_q, int n_kv, int d,
                                  int64_t ld_out, int64_t col0, int num_sms, cudaStream_t st);

// Fused causal attention (head_dim 128, sequence a multiple of 128): the
// forward writes Z and the base-2 log-sum-exp of every query row
// ([batch * n_q * S], row (b n_q + h) S + i); the backward takes D =
// rowsum(dZ o Z) and a cleared f32 dQ accumulator from flash_bwd_prep, writes
// the K and V columns of dqkv and adds dQ into the accumulator, which
// flash_dq_cast converts into dqkv's query columns.
cudaError_t launch_flash_attn_fwd(const void* qkv, int batch, int S, int nq, int nkv, int d, void* z, float* lse2,
                                  uint32_t* status, cudaStream_t st);
cudaError_t launch_flash_bwd_prep(const void* dz, const void* z, float* dsum, float* dq_acc, int batch, int S, int nq,
                                  int d, int num_sms, cudaStream_t st);
cudaError_t launch_flash_attn_bwd(const void* qkv, const void* dz, const float* lse2, const float* dsum, float* dq_acc,
                                  void* dqkv, int batch, int S, int nq, int nkv, int d, uint32_t* status,
                                  cudaStream_t st);
cudaError_t launch_flash_dq_cast(const float* dq_acc, void* dqkv, int64_t N, int64_t Zc, int64_t ld, int num_sms,
                                 cudaStream_t st);

// Message returned by tpmlp_last_error(NULL) on this host thread.
void set_thread_error(const std::string& msg);

}  // namespace tpmlp
