// C ABI of the tensor-parallel attention sublayer ("Megatron-LM Explained",
// "Self-attention: split across heads"; the W_QKV column split and W_out row
// split with one all-reduce on the architecture page; grouped-query attention
// with complete head groups per rank, the TP-MLP page's closing note).
//
//   forward : rmsnorm_fwd -> gemm_qkv -> gemm_scores (batched Q K^T)
//             -> softmax_fwd (causal) -> gemm_pv (batched P V) -> gemm_out_proj
//             (the head-ordered K sum is the all-reduce, + bias + residual)
//   backward: gemm_dz (dy W_o) -> gemm_wgrad_out -> gemm_dp (batched dZ V^T)
//             -> gemm_dv (batched P^T dZ per query head) -> group_sum ->
//             softmax_bwd -> gemm_dq (batched dS K) -> gemm_dk (batched
//             dS^T Q per query head) -> group_sum -> gemm_wgrad_qkv ->
//             gemm_dgrad_norm (every head's contribution summed on chip: the
//             f all-reduce) -> rmsnorm_bwd_residual -> colsum_finalize
//   sgd     : sgd_update
//   adamw   : grad_sqnorm -> adamw_update
// Fused path (head_dim 128, seq % 128 == 0; the default): gemm_scores ->
// softmax_fwd -> gemm_pv become flash_attn_fwd (Z and each row's log-sum-exp),
// and gemm_dp .. group_sum become flash_bwd_prep (D = rowsum(dZ o Z), dQ
// accumulator cleared) -> flash_attn_bwd (dK, dV per group into dqkv, dQ added
// into the accumulator) -> flash_dq_cast.
// The logical degree t fixes which heads a rank owns (complete KV groups);
// on one GPU the ranks' work is the same set of GEMMs in head order.  The
// causal mask is used at tile granularity: score tiles above the diagonal are
// never computed, and the products with P or dS contract only over the causal
// part of each tile row or column.
#include <cuda_runtime.h>

#include <cmath>
#include <string>
#include <vector>

#include "../../include/tpmlp.h"
#include "tpmlp_internal.h"

using namespace tpmlp;

namespace {

enum AttnKernel {
  A_RMSNORM_FWD = 0,
  A_GEMM_QKV,
  A_GEMM_SCORES,
  A_SOFTMAX_FWD,
  A_GEMM_PV,
  A_GEMM_OUT,
  A_GEMM_DZ,
  A_GEMM_WGRAD_OUT,
  A_GEMM_DP,
  A_GEMM_DV,
  A_GROUP_SUM,
  A_SOFTMAX_BWD,
  A_GEMM_DQ,
  A_GEMM_DK,
  A_GEMM_WGRAD_QKV,
  A_GEMM_DGRAD_NORM,
  A_RMSNORM_BWD,
  A_COLSUM,
  A_SGD,
  A_FLASH_FWD,
  A_FLASH_BWD_PREP,
  A_FLASH_BWD,
  A_FLASH_DQ_CAST,
  A_GRAD_NORM,
  A_ADAMW,
  A_COUNT
};
const char* const kAttnNames[A_COUNT] = {
    "rmsnorm_fwd",     "gemm_qkv",        "gemm_scores",     "softmax_fwd",      "gemm_pv",
    "gemm_out_proj",   "gemm_dz",         "gemm_wgrad_out",  "gemm_dp",          "gemm_dv",
    "group_sum",       "softmax_bwd",     "gemm_dq",         "gemm_dk",          "gemm_wgrad_qkv",
    "gemm_dgrad_norm", "rmsnorm_bwd_residual", "colsum_finalize", "sgd_update",
    "flash_attn_fwd",  "flash_bwd_prep",  "flash_attn_bwd",  "flash_dq_cast",   "grad_sqnorm",
    "adamw_update"};

constexpr int MAX_PARTS = 1024;
thread_local std::string g_attn_err;

size_t al256(size_t v) { return (v + 255) & ~size_t(255); }
bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct AttnLayout {
  size_t status, split_ctr, nrm, rstd, qkv, z, dz, dqkv, dnrm, scores, probs, dkv_head, lse2, dsum, part_dw, part_db,
      norm_part, split_scratch, total;
};

bool attn_config_error(const tpattn_config* c, std::string* why) {
  auto fail = [&](const char* m) {
    if (why) *why = m;
    return true;
  };
  if (!c) return fail("config is NULL");
  if (c->dtype != TPMLP_BF16) return fail("the attention sublayer runs in bf16");
  if (c->flags & ~TPATTN_FUSED_ONLY) return fail("unknown flags");
  const bool fused_only = (c->flags & TPATTN_FUSED_ONLY) != 0;
  if (c->max_tokens < 0 || c->hidden <= 0 || c->hidden % 8 != 0 || c->hidden > 8192)
    return fail("hidden must be a positive multiple of 8, at most 8192");
  if (c->n_heads < 1 || c->n_kv_heads < 1 || c->n_heads % c->n_kv_heads != 0)
    return fail("n_heads must be a positive multiple of n_kv_heads");
  if (c->head_dim < 64 || c->head_dim % 64 != 0 || c->head_dim > 256) return fail("head_dim must be 64, 128, 192 or 256");
  if (fused_only) {
    if (c->head_dim != 128) return fail("TPATTN_FUSED_ONLY needs head_dim 128");
    if (c->max_seq < 128 || c->max_seq % 128 != 0 || c->max_seq > 32768)
      return fail("with TPATTN_FUSED_ONLY, max_seq must be a multiple of 128, at most 32768");
  } else if (c->max_seq < 64 || c->max_seq % 64 != 0 || c->max_seq > 4096) {
    return fail("max_seq must be a multiple of 64, at most 4096");
  }
  if (c->max_t < 1 || c->n_kv_heads % c->max_t != 0) return fail("max_t must divide n_kv_heads");
  if (c->max_tokens > (int64_t)1 << 24) return fail("max_tokens too large");
  return false;
}

AttnLayout attn_layout(const tpattn_config& c) {
  AttnLayout L{};
  const size_t N = (size_t)c.max_tokens, H = (size_t)c.hidden, d = (size_t)c.head_dim;
  const size_t W = (size_t)(c.n_heads + 2 * c.n_kv_heads) * d, Z = (size_t)c.n_heads * d;
  // score elements, batch * n_q * S * S (none when only the fused kernels run)
  const size_t SS = (c.flags & TPATTN_FUSED_ONLY) ? 0 : N * (size_t)c.max_seq * (size_t)c.n_heads;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = al256(off + bytes);
    return o;
  };
  L.status = take(256);
  L.split_ctr = take(SPLIT_COUNTER_WORDS * sizeof(uint32_t));  // split GEMMs' arrival flags (epoch-tagged)
  L.nrm = take(N * H * 2);
  L.rstd = take(N * 4);
  L.qkv = take(N * W * 2);
  L.z = take(N * Z * 2);
  L.dz = take(N * Z * 2);
  L.dqkv = take(N * W * 2);
  L.dnrm = take(N * H * 4);
  L.scores = take(SS * 4);   // S, then dP
  L.probs = take(SS * 2);    // P, then dS
  L.dkv_head = take(N * Z * 4);  // per-query-head dK or dV; the fused path's f32 dQ accumulator
  L.lse2 = take(N * (size_t)c.n_heads * 4);  // fused path: base-2 log-sum-exp per (sequence, head, query)
  L.dsum = take(N * (size_t)c.n_heads * 4);  // fused path: rowsum(dZ o Z), same layout
  L.part_dw = take((size_t)MAX_PARTS * H * 4);
  L.part_db = take((size_t)MAX_PARTS * H * 4);
  L.norm_part = take((size_t)MAX_NORM_PARTS * sizeof(double));  // AdamW: per-block partial sums of g^2
  L.split_scratch = take(SPLIT_SCRATCH_BYTES);  // tail-split partial accumulators of the GEMMs
  L.total = off;
  return L;
}

}  // namespace

struct tpattn_ctx {
  tpattn_config cfg{};
  cudaStream_t stream = nullptr;
  int num_sms = 0;
  uint8_t* ws = nullptr;
  AttnLayout L{};
  bool fwd_done = false, bwd_done = false;
  // SGD applied by backward (tpattn_set_update_in_backward) and what the last backward did
  bool upd_in_bwd = false, upd_done = false, upd_epi = false;
  float upd_lr = 0.0f;
  bool fused = true, fwd_fused = false;
  int64_t batch = 0, seq = 0;
  const void *x = nullptr, *norm_w = nullptr, *w_qkv = nullptr, *w_o = nullptr, *b_o = nullptr;
  float *g_norm_w = nullptr, *g_w_qkv = nullptr, *g_w_o = nullptr, *g_b_o = nullptr;
  float *m_norm_w = nullptr, *m_w_qkv = nullptr, *m_w_o = nullptr, *m_b_o = nullptr;
  tpattn_param_set adam_m{}, adam_v{};
  bool adam_bound = false;
  bool timing = false;
  struct Rec {
    int id;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> spare;
  uint64_t launches = 0;
  std::string err;

  template <typename P>
  P* wsp(size_t off) const {
    return reinterpret_cast<P*>(ws + off);
  }
  tpmlp_status fail(tpmlp_status s, const std::string& m) {
    err = m;
    return s;
  }
  cudaEvent_t event() {
    if (!spare.empty()) {
      cudaEvent_t e = spare.back();
      spare.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
  template <typename Fn>
  tpmlp_status run(int id, Fn&& fn) {
    cudaEvent_t a = nullptr, b = nullptr;
    if (timing) {
      a = event();
      b = event();
      cudaEventRecord(a, stream);
    }
    const cudaError_t e = fn();
    if (timing) {
      cudaEventRecord(b, stream);
      recs.push_back({id, a, b});
    }
    ++launches;
    if (e != cudaSuccess) return fail(TPMLP_ERR_CUDA, std::string(kAttnNames[id]) + ": " + cudaGetErrorString(e));
    return TPMLP_OK;
  }
  tpmlp_status gemm(int id, const GemmDesc& desc) {
    GemmDesc g = desc;
    g.split_scratch = wsp<float>(L.split_scratch);
    g.split_scratch_bytes = SPLIT_SCRATCH_BYTES;
    g.split_counters = wsp<uint32_t>(L.split_ctr);
    g.split_counter_words = SPLIT_COUNTER_WORDS;
    return run(id, [&] { return launch_gemm_tc(g, stream, num_sms, wsp<uint32_t>(L.status), 0); });
  }
};

#define ATTN_TRY(expr)                 \
  do {                                 \
    const tpmlp_status s_ = (expr);    \
    if (s_ != TPMLP_OK) return s_;     \
  } while (0)

namespace {

// Batch index (b, g, hq) over sequences, KV groups and the query heads of a group.
BatchDesc head_batch(int B, int n_kv, int hpg) {
  BatchDesc bd;
  bd.dims[0] = B;
  bd.dims[1] = n_kv;
  bd.dims[2] = hpg;
  return bd;
}

// Unfused attention core: scores, causal softmax and P V as batched GEMMs
// and a row kernel, with the scores materialised.
tpmlp_status attn_core_unfused(tpattn_ctx* c, int B, int S, void* qkv, float* sc, void* pr, void* z) {
  const tpattn_config& cf = c->cfg;
  const int N = B * S, d = cf.head_dim;
  const int nq = cf.n_heads, nkv = cf.n_kv_heads, hpg = nq / nkv, W = (nq + 2 * nkv) * d, Zc = nq * d;
  // S[b, h] = Q_h K_g^T  (batched over sequence b, group g, head hq of the group)
  GemmDesc s;
  s.M = S;
  s.N = S;
  s.k_extent = d;
  s.a = qkv;
  s.lda = W;
  s.a_ext_col = W;
  s.a_ext_row = N;
  s.b = qkv;
  s.ldb = W;
  s.b_rows = S;
  s.b_ext_col = W;
  s.b_ext_row = N;
  s.kseg[1] = d;
  s.batch = head_batch(B, nkv, hpg);
  s.batch.a.col[2] = (int64_t)hpg * d;  // Q head g hpg + hq
  s.batch.a.col[3] = d;
  s.batch.a.row[1] = S;                 // sequence b
  s.batch.b.col[0] = (int64_t)nq * d;   // K group g
  s.batch.b.col[2] = d;
  s.batch.b.row[1] = S;
  s.batch.o.row[1] = (int64_t)nq * S;   // score block (b nq + g hpg + hq) S
  s.batch.o.row[2] = (int64_t)hpg * S;
  s.batch.o.row[3] = S;
  s.causal = CAUSAL_SKIP_UPPER;
  s.epi = EPI_STORE_F32;
  s.ep.out0 = sc;
  s.ep.ld_out0 = S;
  s.ep.out_rows = (int64_t)B * nq * S;
  s.ep.out_cols = S;
  ATTN_TRY(c->gemm(A_GEMM_SCORES, s));
  const int64_t rows = (int64_t)B * nq * S;
  const float scale = 1.0f / std::sqrt((float)d);
  ATTN_TRY(c->run(A_SOFTMAX_FWD, [&] { return launch_attn_softmax_fwd(sc, pr, rows, S, scale, c->stream); }));
  // Z[:, head h] = P[b, h] V_g
  GemmDesc pv;
  pv.M = S;
  pv.N = d;
  pv.k_extent = S;
  pv.a = pr;
  pv.lda = S;
  pv.a_ext_col = S;
  pv.a_ext_row = rows;
  pv.b = qkv;
  pv.ldb = W;
  pv.b_mn = true;
  pv.b_ext_col = W;
  pv.b_ext_row = N;
  pv.kseg[1] = S;
  pv.batch = head_batch(B, nkv, hpg);
  pv.batch.a.row[1] = (int64_t)nq * S;
  pv.batch.a.row[2] = (int64_t)hpg * S;
  pv.batch.a.row[3] = S;
  pv.batch.b.col[0] = (int64_t)(nq + nkv) * d;  // V group g
  pv.batch.b.col[2] = d;
  pv.batch.b.row[1] = S;
  pv.batch.o.col[2] = (int64_t)hpg * d;
  pv.batch.o.col[3] = d;
  pv.batch.o.row[1] = S;
  pv.causal = CAUSAL_K_UPTO;
  pv.epi = EPI_STORE_BF16;
  pv.ep.out0 = z;
  pv.ep.ld_out0 = Zc;
  pv.ep.out_rows = N;
  pv.ep.out_cols = Zc;
  return c->gemm(A_GEMM_PV, pv);
}

// Unfused attention core backward: dP, dV, the softmax backward, dQ and dK
// as batched GEMMs and row kernels over the materialised P.
tpmlp_status attn_core_bwd_unfused(tpattn_ctx* c, int B, int S, void* qkv, void* dz, void* dqkv, float* dp, void* pr,
                                   float* dkv) {
  const tpattn_config& cf = c->cfg;
  const int N = B * S, d = cf.head_dim;
  const int nq = cf.n_heads, nkv = cf.n_kv_heads, hpg = nq / nkv, W = (nq + 2 * nkv) * d, Zc = nq * d;
  const int64_t rows = (int64_t)B * nq * S;
  // dP[b, h] = dZ_h V_g^T  (into the score buffer)
  GemmDesc g;
  g.M = S;
  g.N = S;
  g.k_extent = d;
  g.a = dz;
  g.lda = Zc;
  g.a_ext_col = Zc;
  g.a_ext_row = N;
  g.b = qkv;
  g.ldb = W;
  g.b_rows = S;
  g.b_ext_col = W;
  g.b_ext_row = N;
  g.kseg[1] = d;
  g.batch = head_batch(B, nkv, hpg);
  g.batch.a.col[2] = (int64_t)hpg * d;
  g.batch.a.col[3] = d;
  g.batch.a.row[1] = S;
  g.batch.b.col[0] = (int64_t)(nq + nkv) * d;
  g.batch.b.col[2] = d;
  g.batch.b.row[1] = S;
  g.batch.o.row[1] = (int64_t)nq * S;
  g.batch.o.row[2] = (int64_t)hpg * S;
  g.batch.o.row[3] = S;
  g.causal = CAUSAL_SKIP_UPPER;
  g.epi = EPI_STORE_F32;
  g.ep.out0 = dp;
  g.ep.ld_out0 = S;
  g.ep.out_rows = rows;
  g.ep.out_cols = S;
  ATTN_TRY(c->gemm(A_GEMM_DP, g));
  // Per query head: dV_h = P^T dZ_h (f32), then the sum over each group's heads.
  GemmDesc v;
  v.M = S;
  v.N = d;
  v.k_extent = S;
  v.a = pr;
  v.lda = S;
  v.a_mn = true;
  v.a_ext_col = S;
  v.a_ext_row = rows;
  v.b = dz;
  v.ldb = Zc;
  v.b_mn = true;
  v.b_ext_col = Zc;
  v.b_ext_row = N;
  v.kseg[1] = S;
  v.batch = head_batch(B, nkv, hpg);
  v.batch.a.row[1] = (int64_t)nq * S;
  v.batch.a.row[2] = (int64_t)hpg * S;
  v.batch.a.row[3] = S;
  v.batch.b.col[2] = (int64_t)hpg * d;
  v.batch.b.col[3] = d;
  v.batch.b.row[1] = S;
  v.batch.o.row[1] = (int64_t)nq * S;
  v.batch.o.row[2] = (int64_t)hpg * S;
  v.batch.o.row[3] = S;
  v.causal = CAUSAL_K_FROM;
  v.epi = EPI_STORE_F32;
  v.ep.out0 = dkv;
  v.ep.ld_out0 = d;
  v.ep.out_rows = rows;
  v.ep.out_cols = d;
  ATTN_TRY(c->gemm(A_GEMM_DV, v));
  ATTN_TRY(c->run(A_GROUP_SUM, [&] {
    return launch_attn_group_sum(dkv, dqkv, B, S, nq, nkv, d, W, (int64_t)(nq + nkv) * d, c->num_sms, c->stream);
  }));
  // dS = P (dP - rowsum(P dP)) / sqrt(d), over P
  const float scale = 1.0f / std::sqrt((float)d);
  ATTN_TRY(c->run(A_SOFTMAX_BWD, [&] { return launch_attn_softmax_bwd(pr, dp, rows, S, scale, c->stream); }));
  // dQ_h = dS K_g  (into dqkv's query columns)
  GemmDesc q;
  q.M = S;
  q.N = d;
  q.k_extent = S;
  q.a = pr;
  q.lda = S;
  q.a_ext_col = S;
  q.a_ext_row = rows;
  q.b = qkv;
  q.ldb = W;
  q.b_mn = true;
  q.b_ext_col = W;
  q.b_ext_row = N;
  q.kseg[1] = S;
  q.batch = head_batch(B, nkv, hpg);
  q.batch.a.row[1] = (int64_t)nq * S;
  q.batch.a.row[2] = (int64_t)hpg * S;
  q.batch.a.row[3] = S;
  q.batch.b.col[0] = (int64_t)nq * d;  // K group g
  q.batch.b.col[2] = d;
  q.batch.b.row[1] = S;
  q.batch.o.col[2] = (int64_t)hpg * d;
  q.batch.o.col[3] = d;
  q.batch.o.row[1] = S;
  q.causal = CAUSAL_K_UPTO;
  q.epi = EPI_STORE_BF16;
  q.ep.out0 = dqkv;
  q.ep.ld_out0 = W;
  q.ep.out_rows = N;
  q.ep.out_cols = W;
  ATTN_TRY(c->gemm(A_GEMM_DQ, q));
  // Per query head: dK_h = dS^T Q_h (f32), then the sum over each group's heads.
  GemmDesc k = v;
  k.a = pr;
  k.b = qkv;
  k.ldb = W;
  k.b_ext_col = W;
  k.b_ext_row = N;
  k.batch.b.col[0] = 0;  // Q head g hpg + hq
  k.batch.b.col[2] = (int64_t)hpg * d;
  k.batch.b.col[3] = d;
  ATTN_TRY(c->gemm(A_GEMM_DK, k));
  return c->run(A_GROUP_SUM, [&] {
    return launch_attn_group_sum(dkv, dqkv, B, S, nq, nkv, d, W, (int64_t)nq * d, c->num_sms, c->stream);
  });
}

}  // namespace

extern "C" {

size_t tpattn_workspace_bytes(const tpattn_config* cfg) {
  if (attn_config_error(cfg, nullptr)) return 0;
  return attn_layout(*cfg).total;
}

tpmlp_status tpattn_create(const tpattn_config* cfg, void* stream, tpattn_ctx** out) {
  if (!out) return TPMLP_ERR_ARG;
  *out = nullptr;
  std::string why;
  if (attn_config_error(cfg, &why)) {
    g_attn_err = why;
    return TPMLP_ERR_SHAPE;
  }
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) {
    g_attn_err = "no CUDA device";
    return TPMLP_ERR_CUDA;
  }
  if (major != 10 || minor != 3) {
    g_attn_err = "needs an sm_103 device";
    return TPMLP_ERR_UNSUPPORTED;
  }
  tpattn_ctx* c = new tpattn_ctx();
  c->cfg = *cfg;
  c->stream = static_cast<cudaStream_t>(stream);
  c->num_sms = sms;
  c->L = attn_layout(*cfg);
  *out = c;
  return TPMLP_OK;
}

tpmlp_status tpattn_bind_workspace(tpattn_ctx* c, void* dev, size_t bytes) {
  if (!c) return TPMLP_ERR_ARG;
  if (!dev || (reinterpret_cast<uintptr_t>(dev) & 255u)) return c->fail(TPMLP_ERR_ARG, "workspace must be 256-byte aligned");
  if (bytes < c->L.total) return c->fail(TPMLP_ERR_ARG, "workspace too small");
  c->ws = static_cast<uint8_t*>(dev);
  // the status word and the split GEMMs' arrival flags (epoch-tagged: stale values must not match)
  cudaError_t e = cudaMemsetAsync(c->ws + c->L.status, 0, 256, c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->ws + c->L.split_ctr, 0, SPLIT_COUNTER_WORDS * sizeof(uint32_t), c->stream);
  return e == cudaSuccess ? TPMLP_OK : c->fail(TPMLP_ERR_CUDA, cudaGetErrorString(e));
}

tpmlp_status tpattn_forward(tpattn_ctx* c, int64_t batch, int64_t seq, const void* x, const void* norm_w,
                            const void* w_qkv, const void* w_o, const void* b_o, float eps, int32_t t, void* y) {
  if (!c) return TPMLP_ERR_ARG;
  if (!c->ws) return c->fail(TPMLP_ERR_ORDER, "no workspace bound");
  const tpattn_config& cf = c->cfg;
  if (batch < 1 || seq < 64 || seq % 64 != 0 || seq > cf.max_seq || batch * seq > cf.max_tokens)
    return c->fail(TPMLP_ERR_SHAPE, "seq must be a multiple of 64 within max_seq, batch * seq within max_tokens");
  if (t < 1 || t > cf.max_t || cf.n_kv_heads % t != 0) return c->fail(TPMLP_ERR_SHAPE, "t must divide n_kv_heads");
  if ((cf.flags & TPATTN_FUSED_ONLY) && seq % 128 != 0)
    return c->fail(TPMLP_ERR_SHAPE, "a fused-only context needs seq to be a multiple of 128");
  if (!x || !norm_w || !w_qkv || !w_o || !b_o || !y) return c->fail(TPMLP_ERR_ARG, "NULL tensor");
  for (const void* p : {x, norm_w, w_qkv, w_o, b_o, (const void*)y})
    if (!a16(p)) return c->fail(TPMLP_ERR_ARG, "tensor not 16-byte aligned");
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return c->fail(TPMLP_ERR_ARG, "eps must be finite and >= 0");
  const int B = (int)batch, S = (int)seq, N = B * S, H = (int)cf.hidden, d = cf.head_dim;
  const int nq = cf.n_heads, nkv = cf.n_kv_heads, W = (nq + 2 * nkv) * d, Zc = nq * d;
  c->fwd_done = c->bwd_done = false;
  c->batch = batch;
  c->seq = seq;
  c->x = x;
  c->norm_w = norm_w;
  c->w_qkv = w_qkv;
  c->w_o = w_o;
  c->b_o = b_o;
  void* nrm = c->wsp<void>(c->L.nrm);
  void* qkv = c->wsp<void>(c->L.qkv);
  void* z = c->wsp<void>(c->L.z);
  float* sc = c->wsp<float>(c->L.scores);
  void* pr = c->wsp<void>(c->L.probs);
  c->fwd_fused = c->fused && d == 128 && S % 128 == 0;
  ATTN_TRY(c->run(A_RMSNORM_FWD, [&] {
    return launch_rmsnorm_fwd(1, x, norm_w, eps, nrm, c->wsp<float>(c->L.rstd), N, H, c->stream);
  }));
  // qkv = n W_qkv^T
  GemmDesc g;
  g.M = N;
  g.N = W;
  g.k_extent = H;
  g.a = nrm;
  g.lda = H;
  g.b = w_qkv;
  g.ldb = H;
  g.b_rows = W;
  g.kseg[1] = H;
  g.epi = EPI_STORE_BF16;
  g.ep.out0 = qkv;
  g.ep.ld_out0 = W;
  ATTN_TRY(c->gemm(A_GEMM_QKV, g));
  if (c->fwd_fused) {
    ATTN_TRY(c->run(A_FLASH_FWD, [&] {
      return launch_flash_attn_fwd(qkv, B, S, nq, nkv, d, z, c->wsp<float>(c->L.lse2), c->wsp<uint32_t>(c->L.status),
                                   c->stream);
    }));
  } else {
    ATTN_TRY(attn_core_unfused(c, B, S, qkv, sc, pr, z));
  }
  // y = x + Z W_o^T + b_o; the K loop runs over the heads in order: the
  // ranks' partial outputs summed on chip.
  GemmDesc o;
  o.M = N;
  o.N = H;
  o.k_extent = Zc;
  o.a = z;
  o.lda = Zc;
  o.b = w_o;
  o.ldb = Zc;
  o.b_rows = H;
  o.kseg[1] = Zc;
  o.epi = EPI_DOWN_RESID;
  o.ep.out0 = y;
  o.ep.ld_out0 = H;
  o.ep.in0 = x;
  o.ep.ld_in0 = H;
  o.ep.vec = b_o;
  ATTN_TRY(c->gemm(A_GEMM_OUT, o));
  c->fwd_done = true;
  c->upd_done = false;
  return TPMLP_OK;
}


constexpr int64_t ATTN_UPDATE_IN_EPILOGUE_MIN_TOKENS = 8192;

// SGD w <- w - lr g over the parameters of the last forward with the gradients
// of the last backward; the two projection matrices only when `matrices`.
static tpmlp_status attn_run_sgd(tpattn_ctx* c, float lr, bool matrices) {
  const tpattn_config& cf = c->cfg;
  const int64_t H = cf.hidden, d = cf.head_dim, W = (int64_t)(cf.n_heads + 2 * cf.n_kv_heads) * d,
                Zc = (int64_t)cf.n_heads * d;
  SgdArgs a{};
  a.lr = lr;
  a.seg[a.nseg++] = SgdSeg{c->m_norm_w, c->g_norm_w, const_cast<void*>(c->norm_w), H};
  if (matrices) {
    a.seg[a.nseg++] = SgdSeg{c->m_w_qkv, c->g_w_qkv, const_cast<void*>(c->w_qkv), W * H};
    a.seg[a.nseg++] = SgdSeg{c->m_w_o, c->g_w_o, const_cast<void*>(c->w_o), H * Zc};
  }
  a.seg[a.nseg++] = SgdSeg{c->m_b_o, c->g_b_o, const_cast<void*>(c->b_o), H};
  return c->run(A_SGD, [&] { return launch_sgd(1, a, c->num_sms, c->stream); });
}

tpmlp_status tpattn_backward(tpattn_ctx* c, const void* dy, void* dx, float* dnorm_w, float* dw_qkv, float* dw_o,
                             float* db_o) {
  if (!c) return TPMLP_ERR_ARG;
  if (!c->fwd_done) return c->fail(TPMLP_ERR_ORDER, "backward before forward");
  if (!dy || !dx || !dnorm_w || !dw_qkv || !dw_o || !db_o) return c->fail(TPMLP_ERR_ARG, "NULL tensor");
  for (const void* p : {dy, (const void*)dx, (const void*)dnorm_w, (const void*)dw_qkv, (const void*)dw_o,
                        (const void*)db_o})
    if (!a16(p)) return c->fail(TPMLP_ERR_ARG, "tensor not 16-byte aligned");
  const tpattn_config& cf = c->cfg;
  const int B = (int)c->batch, S = (int)c->seq, N = B * S, H = (int)cf.hidden, d = cf.head_dim;
  const int nq = cf.n_heads, nkv = cf.n_kv_heads, W = (nq + 2 * nkv) * d, Zc = nq * d;
  const bool upd = c->upd_in_bwd;
  if (upd && (!c->m_norm_w || !c->m_w_qkv || !c->m_w_o || !c->m_b_o))
    return c->fail(TPMLP_ERR_ORDER, "the update in backward needs bound fp32 masters");
  // W_qkv and W_o are updated in their weight-gradient epilogues from 8192
  // tokens (as in the MLP), otherwise by the update kernel after backward
  const bool fuse = upd && N >= ATTN_UPDATE_IN_EPILOGUE_MIN_TOKENS;
  c->bwd_done = false;
  c->upd_done = false;
  c->upd_epi = false;
  c->g_norm_w = dnorm_w;
  c->g_w_qkv = dw_qkv;
  c->g_w_o = dw_o;
  c->g_b_o = db_o;
  void* nrm = c->wsp<void>(c->L.nrm);
  void* qkv = c->wsp<void>(c->L.qkv);
  void* z = c->wsp<void>(c->L.z);
  void* dz = c->wsp<void>(c->L.dz);
  void* dqkv = c->wsp<void>(c->L.dqkv);
  float* dnrm = c->wsp<float>(c->L.dnrm);
  float* dp = c->wsp<float>(c->L.scores);
  void* pr = c->wsp<void>(c->L.probs);
  float* dkv = c->wsp<float>(c->L.dkv_head);
  // dZ = dy W_o
  GemmDesc a;
  a.M = N;
  a.N = Zc;
  a.k_extent = H;
  a.a = dy;
  a.lda = H;
  a.b = c->w_o;
  a.ldb = Zc;
  a.b_mn = true;
  a.kseg[1] = H;
  a.epi = EPI_STORE_BF16;
  a.ep.out0 = dz;
  a.ep.ld_out0 = Zc;
  ATTN_TRY(c->gemm(A_GEMM_DZ, a));
  // dW_o = dy^T Z
  GemmDesc wo;
  wo.M = H;
  wo.N = Zc;
  wo.k_extent = N;
  wo.a = dy;
  wo.lda = H;
  wo.a_mn = true;
  wo.b = z;
  wo.ldb = Zc;
  wo.b_mn = true;
  wo.kseg[1] = N;
  wo.epi = EPI_STORE_F32;
  wo.ep.out0 = dw_o;
  wo.ep.ld_out0 = Zc;
  if (fuse) {  // W_o was last read by the dZ GEMM above
    wo.ep.sgd_master = c->m_w_o;
    wo.ep.sgd_w = static_cast<__nv_bfloat16*>(const_cast<void*>(c->w_o));
    wo.ep.sgd_ld = Zc;
    wo.ep.sgd_lr = c->upd_lr;
  }
  ATTN_TRY(c->gemm(A_GEMM_WGRAD_OUT, wo));
  if (c->fwd_fused) {
    float* dq_acc = c->wsp<float>(c->L.dkv_head);
    float* dsum = c->wsp<float>(c->L.dsum);
    ATTN_TRY(c->run(A_FLASH_BWD_PREP,
                    [&] { return launch_flash_bwd_prep(dz, z, dsum, dq_acc, B, S, nq, d, c->num_sms, c->stream); }));
    ATTN_TRY(c->run(A_FLASH_BWD, [&] {
      return launch_flash_attn_bwd(qkv, dz, c->wsp<float>(c->L.lse2), dsum, dq_acc, dqkv, B, S, nq, nkv, d,
                                   c->wsp<uint32_t>(c->L.status), c->stream);
    }));
    ATTN_TRY(c->run(A_FLASH_DQ_CAST,
                    [&] { return launch_flash_dq_cast(dq_acc, dqkv, N, Zc, W, c->num_sms, c->stream); }));
  } else {
    ATTN_TRY(attn_core_bwd_unfused(c, B, S, qkv, dz, dqkv, dp, pr, dkv));
  }
  // dN = dqkv W_qkv: every head's contribution summed on chip (the f all-reduce);
  // it runs before the QKV weight gradient, which may update W_qkv
  GemmDesc dn;
  dn.M = N;
  dn.N = H;
  dn.k_extent = W;
  dn.a = dqkv;
  dn.lda = W;
  dn.b = c->w_qkv;
  dn.ldb = H;
  dn.b_mn = true;
  dn.kseg[1] = W;
  dn.epi = EPI_STORE_F32;
  dn.ep.out0 = dnrm;
  dn.ep.ld_out0 = H;
  ATTN_TRY(c->gemm(A_GEMM_DGRAD_NORM, dn));
  // dW_qkv = dqkv^T n
  GemmDesc wq;
  wq.M = W;
  wq.N = H;
  wq.k_extent = N;
  wq.a = dqkv;
  wq.lda = W;
  wq.a_mn = true;
  wq.b = nrm;
  wq.ldb = H;
  wq.b_mn = true;
  wq.kseg[1] = N;
  wq.epi = EPI_STORE_F32;
  wq.ep.out0 = dw_qkv;
  wq.ep.ld_out0 = H;
  if (fuse) {  // W_qkv was last read by the dN GEMM above
    wq.ep.sgd_master = c->m_w_qkv;
    wq.ep.sgd_w = static_cast<__nv_bfloat16*>(const_cast<void*>(c->w_qkv));
    wq.ep.sgd_ld = H;
    wq.ep.sgd_lr = c->upd_lr;
  }
  ATTN_TRY(c->gemm(A_GEMM_WGRAD_QKV, wq));
  const int nb = rmsnorm_bwd_blocks(N, c->num_sms, 1);
  float* pdw = c->wsp<float>(c->L.part_dw);
  float* pdb = c->wsp<float>(c->L.part_db);
  ATTN_TRY(c->run(A_RMSNORM_BWD, [&] {
    return launch_rmsnorm_bwd(1, dnrm, c->x, c->wsp<float>(c->L.rstd), c->norm_w, dy, dx, pdw, pdb, N, H, 1, nb,
                              c->stream);
  }));
  ATTN_TRY(c->run(A_COLSUM, [&] { return launch_colsum_finalize(pdw, dnorm_w, pdb, db_o, nb, H, c->stream); }));
  c->bwd_done = true;
  if (upd) {
    // the matrices too unless their weight-gradient epilogues updated them
    ATTN_TRY(attn_run_sgd(c, c->upd_lr, !fuse));
    c->upd_done = true;
    c->upd_epi = fuse;
  }
  return TPMLP_OK;
}

tpmlp_status tpattn_bind_master(tpattn_ctx* c, float* norm_w, float* w_qkv, float* w_o, float* b_o) {
  if (!c) return TPMLP_ERR_ARG;
  const bool none = !norm_w && !w_qkv && !w_o && !b_o;
  if (!none && (!norm_w || !w_qkv || !w_o || !b_o)) return c->fail(TPMLP_ERR_ARG, "bind all master tensors or none");
  for (const void* p : {(const void*)norm_w, (const void*)w_qkv, (const void*)w_o, (const void*)b_o})
    if (!a16(p)) return c->fail(TPMLP_ERR_ARG, "tensor not 16-byte aligned");
  c->m_norm_w = norm_w;
  c->m_w_qkv = w_qkv;
  c->m_w_o = w_o;
  c->m_b_o = b_o;
  return TPMLP_OK;
}

tpmlp_status tpattn_set_fused(tpattn_ctx* c, int32_t enable) {
  if (!c) return TPMLP_ERR_ARG;
  if (!enable && (c->cfg.flags & TPATTN_FUSED_ONLY))
    return c->fail(TPMLP_ERR_UNSUPPORTED, "a fused-only context has no workspace for the unfused path");
  c->fused = enable != 0;
  return TPMLP_OK;
}

int32_t tpattn_fused_active(const tpattn_ctx* c) { return c && c->fwd_done && c->fwd_fused ? 1 : 0; }

tpmlp_status tpattn_sgd_step(tpattn_ctx* c, float lr) {
  if (!c) return TPMLP_ERR_ARG;
  if (!c->bwd_done) return c->fail(TPMLP_ERR_ORDER, "sgd_step before backward");
  if (c->upd_done) return c->fail(TPMLP_ERR_ORDER, "the last backward already applied the update");
  if (!std::isfinite(lr)) return c->fail(TPMLP_ERR_ARG, "lr must be finite");
  return attn_run_sgd(c, lr, true);
}

tpmlp_status tpattn_set_update_in_backward(tpattn_ctx* c, int32_t enable, float lr) {
  if (!c) return TPMLP_ERR_ARG;
  if (enable && !std::isfinite(lr)) return c->fail(TPMLP_ERR_ARG, "lr must be finite");
  c->upd_in_bwd = enable != 0;
  c->upd_lr = enable ? lr : 0.0f;
  return TPMLP_OK;
}

int32_t tpattn_update_in_epilogue(const tpattn_ctx* c) { return c && c->upd_done && c->upd_epi ? 1 : 0; }

tpmlp_status tpattn_bind_adam_state(tpattn_ctx* c, const tpattn_param_set* m, const tpattn_param_set* v) {
  if (!c) return TPMLP_ERR_ARG;
  if (!m && !v) {
    c->adam_m = tpattn_param_set{};
    c->adam_v = tpattn_param_set{};
    c->adam_bound = false;
    return TPMLP_OK;
  }
  if (!m || !v) return c->fail(TPMLP_ERR_ARG, "bind both moment sets or neither");
  for (const tpattn_param_set* s : {m, v}) {
    if (!s->norm_w || !s->w_qkv || !s->w_o || !s->b_o) return c->fail(TPMLP_ERR_ARG, "a moment tensor is missing");
    for (const void* p : {(const void*)s->norm_w, (const void*)s->w_qkv, (const void*)s->w_o, (const void*)s->b_o})
      if (!a16(p)) return c->fail(TPMLP_ERR_ARG, "moment tensor not 16-byte aligned");
  }
  c->adam_m = *m;
  c->adam_v = *v;
  c->adam_bound = true;
  return TPMLP_OK;
}

// The MLP's clipped AdamW (norm pass over every gradient, then the update)
// over the attention sublayer's four parameters; weight decay on the two
// projection matrices only.
tpmlp_status tpattn_adamw_step(tpattn_ctx* c, const tpmlp_adamw_params* hp, float* grad_norm) {
  if (!c) return TPMLP_ERR_ARG;
  if (!hp) return c->fail(TPMLP_ERR_ARG, "hyperparameters are NULL");
  if (!c->bwd_done) return c->fail(TPMLP_ERR_ORDER, "adamw_step before backward");
  if (c->upd_done) return c->fail(TPMLP_ERR_ORDER, "the last backward already applied the update");
  if (!c->adam_bound) return c->fail(TPMLP_ERR_ARG, "AdamW moments are not bound");
  if (!std::isfinite(hp->lr) || !std::isfinite(hp->weight_decay) || !std::isfinite(hp->max_grad_norm) ||
      !(hp->beta1 >= 0.f && hp->beta1 < 1.f) || !(hp->beta2 >= 0.f && hp->beta2 < 1.f) ||
      !(hp->eps >= 0.f && std::isfinite(hp->eps)) || hp->step < 1)
    return c->fail(TPMLP_ERR_ARG, "AdamW hyperparameter out of range");
  if (grad_norm && (reinterpret_cast<uintptr_t>(grad_norm) & 3u))
    return c->fail(TPMLP_ERR_ARG, "grad_norm not 4-byte aligned");
  const tpattn_config& cf = c->cfg;
  const int64_t H = cf.hidden, d = cf.head_dim, W = (int64_t)(cf.n_heads + 2 * cf.n_kv_heads) * d,
                Zc = (int64_t)cf.n_heads * d;
  const double bc1 = 1.0 - std::pow((double)hp->beta1, (double)hp->step);
  const double bc2 = 1.0 - std::pow((double)hp->beta2, (double)hp->step);
  AdamArgs a{};
  a.beta1 = hp->beta1;
  a.beta2 = hp->beta2;
  a.one_m_beta1 = (float)(1.0 - (double)hp->beta1);
  a.one_m_beta2 = (float)(1.0 - (double)hp->beta2);
  a.step_size = (float)((double)hp->lr / bc1);
  a.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
  a.eps = hp->eps;
  a.max_norm = hp->max_grad_norm;
  a.part = c->wsp<double>(c->L.norm_part);
  a.grad_norm = grad_norm;
  const float lr_wd = (float)((double)hp->lr * (double)hp->weight_decay);
  const tpattn_param_set &M = c->adam_m, &V = c->adam_v;
  a.seg[a.nseg++] = AdamSeg{c->m_norm_w, c->g_norm_w, const_cast<void*>(c->norm_w), M.norm_w, V.norm_w, H, 0.0f};
  a.seg[a.nseg++] = AdamSeg{c->m_w_qkv, c->g_w_qkv, const_cast<void*>(c->w_qkv), M.w_qkv, V.w_qkv, W * H, lr_wd};
  a.seg[a.nseg++] = AdamSeg{c->m_w_o, c->g_w_o, const_cast<void*>(c->w_o), M.w_o, V.w_o, H * Zc, lr_wd};
  a.seg[a.nseg++] = AdamSeg{c->m_b_o, c->g_b_o, const_cast<void*>(c->b_o), M.b_o, V.b_o, H, 0.0f};
  const int nb = adam_blocks(a, c->num_sms);
  ATTN_TRY(c->run(A_GRAD_NORM, [&] { return launch_grad_sqnorm(a, nb, c->stream); }));
  return c->run(A_ADAMW, [&] { return launch_adamw(1, a, nb, c->stream); });
}

tpmlp_status tpattn_sync(tpattn_ctx* c) {
  if (!c) return TPMLP_ERR_ARG;
  cudaError_t e = cudaStreamSynchronize(c->stream);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return c->fail(TPMLP_ERR_CUDA, cudaGetErrorString(e));
  if (!c->ws) return TPMLP_OK;
  uint32_t st = 0;
  e = cudaMemcpy(&st, c->wsp<uint32_t>(c->L.status), sizeof st, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return c->fail(TPMLP_ERR_CUDA, cudaGetErrorString(e));
  if (st) {
    cudaMemsetAsync(c->wsp<uint32_t>(c->L.status), 0, sizeof st, c->stream);
    return c->fail(TPMLP_ERR_TIMEOUT, "a bounded device wait gave up");
  }
  return TPMLP_OK;
}

tpmlp_status tpattn_set_timing(tpattn_ctx* c, int32_t enable) {
  if (!c) return TPMLP_ERR_ARG;
  c->timing = enable != 0;
  return TPMLP_OK;
}

int32_t tpattn_read_kernel_times(tpattn_ctx* c, float* ms, int64_t* launches, int32_t n) {
  if (!c || !ms || !launches || n < A_COUNT) return -1;
  cudaStreamSynchronize(c->stream);
  for (int i = 0; i < A_COUNT; ++i) {
    ms[i] = 0.0f;
    launches[i] = 0;
  }
  for (const auto& r : c->recs) {
    float t = 0.0f;
    cudaEventElapsedTime(&t, r.a, r.b);
    ms[r.id] += t;
    launches[r.id] += 1;
    c->spare.push_back(r.a);
    c->spare.push_back(r.b);
  }
  c->recs.clear();
  return A_COUNT;
}

const char* tpattn_kernel_name(int32_t id) { return id >= 0 && id < A_COUNT ? kAttnNames[id] : nullptr; }
int32_t tpattn_num_kernel_ids(void) { return A_COUNT; }
uint64_t tpattn_launch_count(const tpattn_ctx* c) { return c ? c->launches : 0; }
const char* tpattn_last_error(const tpattn_ctx* c) { return c ? c->err.c_str() : g_attn_err.c_str(); }

void tpattn_destroy(tpattn_ctx* c) {
  if (!c) return;
  for (auto& r : c->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : c->spare) cudaEventDestroy(e);
  delete c;
}

}  // extern "C"
