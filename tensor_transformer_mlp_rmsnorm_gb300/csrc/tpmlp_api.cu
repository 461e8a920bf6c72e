// C ABI of the tensor-parallel MLP sublayer: argument checks, workspace
// layout, and the kernel sequence of each call.  See include/tpmlp.h.
//
// Step order (page "Megatron tensor-parallel MLP"):
//   forward : rmsnorm_fwd -> gemm_gateup_act (column-parallel expansion,
//             "Split the expansion") -> gemm_down_reduce (row-parallel
//             contraction with the shard sum, bias and residual, "Split the
//             contraction")
//   loss    : mse_loss_grad -> loss_finalize
//   backward: gemm_dgrad_act (g backward is the identity) -> gemm_wgrad_down
//             -> gemm_wgrad_gateup -> gemm_dgrad_norm_reduce (the f
//             all-reduce, "Put the other collective in backward") ->
//             rmsnorm_bwd_residual -> colsum_finalize
//   sgd     : sgd_update
//   adamw   : grad_sqnorm -> adamw_update (walkthrough, "Stage 8")
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <utility>
#include <vector>

#include "../../include/tpmlp.h"
#include "tpmlp_internal.h"

using namespace tpmlp;

namespace {

enum KernelId {
  K_RMSNORM_FWD = 0,
  K_GEMM_GATEUP,
  K_GEMM_DOWN,
  K_LOSS,
  K_LOSS_FINAL,
  K_GEMM_DGRAD_ACT,
  K_GEMM_WGRAD_DOWN,
  K_GEMM_WGRAD_GATEUP,
  K_GEMM_DGRAD_NORM,
  K_RMSNORM_BWD,
  K_COLSUM_FINAL,
  K_COLSUM_B1,
  K_SGD,
  K_GRAD_NORM,
  K_ADAMW,
  K_FP8_AMAX,
  K_FP8_CAST,
  K_PROBE,
  K_COUNT
};

const char* const kKernelNames[K_COUNT] = {
    "rmsnorm_fwd",        "gemm_gateup_act",     "gemm_down_reduce",     "mse_loss_grad",
    "loss_finalize",      "gemm_dgrad_act",      "gemm_wgrad_down",      "gemm_wgrad_gateup",
    "gemm_dgrad_norm_reduce", "rmsnorm_bwd_residual", "colsum_finalize", "colsum_b1",
    "sgd_update",         "grad_sqnorm",         "adamw_update",         "fp8_amax",
    "fp8_cast",           "timeout_probe"};

constexpr int MAX_BWD_PARTS = 1024;
constexpr int MAX_B1_PARTS = 256;
constexpr int MAX_LOSS_PARTS = 1024;
constexpr int64_t MAX_HIDDEN = 8192;
constexpr int MAX_SP_SHARDS = 64;

thread_local std::string g_thread_err;

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct Layout {
  size_t status, split_ctr, loss_part, norm_part, nrm, rstd, gu, act, dgu, dnrm, part_dw, part_db, part_b1, shard_sums,
      split_scratch, total;
};

bool config_error(const tpmlp_config* c, std::string* why, tpmlp_status* st) {
  auto fail = [&](tpmlp_status s, const char* m) {
    if (why) *why = m;
    if (st) *st = s;
    return true;
  };
  if (!c) return fail(TPMLP_ERR_ARG, "config is NULL");
  if (c->dtype != TPMLP_F32 && c->dtype != TPMLP_BF16) return fail(TPMLP_ERR_UNSUPPORTED, "unknown dtype");
  if (c->act != TPMLP_SWIGLU && c->act != TPMLP_GELU) return fail(TPMLP_ERR_UNSUPPORTED, "unknown activation");
  if (c->reserved != 0) return fail(TPMLP_ERR_ARG, "reserved field must be 0");
  if (c->max_tokens < 0) return fail(TPMLP_ERR_SHAPE, "max_tokens must be >= 0");
  if (c->hidden <= 0 || c->ffn <= 0) return fail(TPMLP_ERR_SHAPE, "hidden and ffn must be positive");
  if (c->hidden % 8 != 0 || c->ffn % 8 != 0) return fail(TPMLP_ERR_SHAPE, "hidden and ffn must be multiples of 8");
  if (c->hidden > MAX_HIDDEN) return fail(TPMLP_ERR_SHAPE, "hidden > 8192 is not supported");
  if (c->max_t < 1 || c->max_t > c->ffn) return fail(TPMLP_ERR_SHAPE, "max_t must be in [1, ffn]");
  if (c->max_tokens > (int64_t)1 << 30 || c->ffn > (int64_t)1 << 24)
    return fail(TPMLP_ERR_SHAPE, "tokens or ffn too large");
  return false;
}

Layout make_layout(const tpmlp_config& c) {
  Layout L{};
  const size_t E = c.dtype == TPMLP_BF16 ? 2 : 4;
  const size_t N = (size_t)c.max_tokens, H = (size_t)c.hidden, F = (size_t)c.ffn;
  const size_t guw = c.act == TPMLP_SWIGLU ? 2 * F : F;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.status = take(256);
  L.split_ctr = take(SPLIT_COUNTER_WORDS * sizeof(uint32_t));  // split GEMMs' arrival flags (epoch-tagged)
  L.loss_part = take(MAX_LOSS_PARTS * sizeof(double));
  L.norm_part = take(MAX_NORM_PARTS * sizeof(double));
  L.nrm = take(N * H * E);
  L.rstd = take(N * 4);
  L.gu = take(N * guw * E);
  L.act = take(N * F * E);
  L.dgu = take(N * guw * E);
  L.dnrm = take(N * H * 4);
  L.part_dw = take((size_t)MAX_BWD_PARTS * H * 4);
  L.part_db = take((size_t)MAX_BWD_PARTS * H * 4);
  L.part_b1 = c.act == TPMLP_GELU ? take((size_t)MAX_B1_PARTS * F * 4) : off;
  L.shard_sums = take((size_t)2 * (c.max_t < MAX_SP_SHARDS ? c.max_t : MAX_SP_SHARDS) * H * 4);
  L.split_scratch = c.dtype == TPMLP_BF16 ? take(SPLIT_SCRATCH_BYTES) : off;  // tensor-core GEMMs only
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t pitch16(int64_t n) { return (n + 15) / 16 * 16; }

// FP8 operand buffers (E4M3 codes, pitches rounded up to 16 bytes): each
// tensor that feeds a GEMM row-major (q) and transposed (t), with one inverse
// scale per tensor.  Transposed copies of token-major tensors are sized for
// max_tokens and used with the pitch of the actual token count.
enum Fp8Tensor { F8_NRM = 0, F8_WGU, F8_ACT, F8_WD, F8_DY, F8_DGU, F8_COUNT };
struct Fp8Layout {
  size_t inv, amax, part, q[F8_COUNT], t[F8_COUNT], total;
};

Fp8Layout make_fp8_layout(const tpmlp_config& c) {
  Fp8Layout L{};
  const size_t N = (size_t)c.max_tokens, H = (size_t)c.hidden, F = (size_t)c.ffn;
  const size_t guw = c.act == TPMLP_SWIGLU ? 2 * F : F;
  const size_t rows[F8_COUNT] = {N, guw, N, H, N, N};  // row-major shape [rows, cols]
  const size_t cols[F8_COUNT] = {H, H, F, F, H, guw};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.inv = take(F8_COUNT * sizeof(float));
  L.amax = take(F8_COUNT * sizeof(float));  // maxima that producers fold in with atomicMax
  L.part = take(FP8_MAX_PARTS * sizeof(float));
  for (int i = 0; i < F8_COUNT; ++i) {
    L.q[i] = take(rows[i] * (size_t)pitch16((int64_t)cols[i]));
    L.t[i] = take(cols[i] * (size_t)pitch16((int64_t)rows[i]));
  }
  L.total = off;
  return L;
}

}  // namespace

void tpmlp::set_thread_error(const std::string& msg) { g_thread_err = msg; }

struct tpmlp_ctx {
  tpmlp_config cfg{};
  cudaStream_t stream = nullptr;
  int device = 0, num_sms = 0;
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  Layout L{};
  // state of the last forward / backward
  bool fwd_done = false, bwd_done = false;
  int64_t tokens = 0;
  int t = 1;
  const void *x = nullptr, *norm_w = nullptr, *w_gu = nullptr, *b_1 = nullptr, *w_down = nullptr,
             *b_down = nullptr;
  float *g_norm_w = nullptr, *g_w_gu = nullptr, *g_b_1 = nullptr, *g_w_down = nullptr, *g_b_down = nullptr;
  float *m_norm_w = nullptr, *m_w_gu = nullptr, *m_b_1 = nullptr, *m_w_down = nullptr, *m_b_down = nullptr;
  bool sp = false;  // sequence-parallel form: token shards of N / t rows
  bool fp8 = false;  // E4M3 GEMM operands (needs the FP8 workspace)
  // SGD applied by backward (tpmlp_set_update_in_backward), and whether the
  // last backward did so (sgd_step / adamw_step are then refused)
  bool upd_in_bwd = false, upd_done = false, upd_epi = false;
  float upd_lr = 0.0f;
  uint8_t* ws8 = nullptr;
  Fp8Layout L8{};
  tpmlp_param_set adam_m{}, adam_v{};
  bool adam_bound = false;
  uint32_t dbg_flags = 0;
  int dbg_shard = 0;
  // timing
  bool timing = false;
  std::vector<cudaEvent_t> free_events;
  struct Rec {
    int id;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  uint64_t launches = 0;
  std::string err;

  int E() const { return cfg.dtype == TPMLP_BF16 ? 2 : 4; }
  bool swiglu() const { return cfg.act == TPMLP_SWIGLU; }
  template <typename P>
  P* wsp(size_t off) const {
    return reinterpret_cast<P*>(ws + off);
  }
  uint32_t* status() const { return wsp<uint32_t>(L.status); }

  tpmlp_status fail(tpmlp_status s, const std::string& m) {
    err = m;
    return s;
  }
  cudaEvent_t event() {
    if (!free_events.empty()) {
      cudaEvent_t e = free_events.back();
      free_events.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
  // Run one kernel launcher, with optional CUDA-event timing around it.
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
    if (e != cudaSuccess) return fail(TPMLP_ERR_CUDA, std::string(kKernelNames[id]) + ": " + cudaGetErrorString(e));
    ++launches;
    return TPMLP_OK;
  }
};

#define TPMLP_TRY(expr)                 \
  do {                                  \
    const tpmlp_status _s = (expr);     \
    if (_s != TPMLP_OK) return _s;      \
  } while (0)

namespace {

tpmlp_status run_gemm(tpmlp_ctx* c, int id, const GemmDesc& desc, int force_timeout = 0) {
  if (c->cfg.dtype == TPMLP_BF16) {
    GemmDesc g = desc;
    if (c->dbg_flags & TPMLP_DBG_GEMM_SINGLE_CTA) g.tile_mode = 1;
    g.split_scratch = c->wsp<float>(c->L.split_scratch);
    g.split_scratch_bytes = SPLIT_SCRATCH_BYTES;
    g.split_counters = c->wsp<uint32_t>(c->L.split_ctr);
    g.split_counter_words = SPLIT_COUNTER_WORDS;
    return c->run(id, [&] { return launch_gemm_tc(g, c->stream, c->num_sms, c->status(), force_timeout); });
  }
  const GemmDesc& g = desc;
  return c->run(id, [&] { return launch_gemm_simt_f32(g, c->stream); });
}

// Contraction segments in elements for a shard restriction; the tensor-core
// path needs 64-element block boundaries (128 for E4M3 operands).
bool seg_ok(const tpmlp_ctx* c, int64_t b, int64_t e, int64_t extent) {
  if (c->cfg.dtype != TPMLP_BF16) return true;
  const int64_t blk = c->fp8 ? 128 : 64;
  return b % blk == 0 && (e % blk == 0 || e == extent);
}

uint32_t* fp8_amax_slot(const tpmlp_ctx* c, int tensor) {
  return reinterpret_cast<uint32_t*>(c->ws8 + c->L8.amax) + tensor;
}

// Zero the fused maxima of the listed tensors before their producers run.
tpmlp_status fp8_clear_amax(tpmlp_ctx* c, int first, int count) {
  const cudaError_t e = cudaMemsetAsync(fp8_amax_slot(c, first), 0, count * sizeof(uint32_t), c->stream);
  return e == cudaSuccess ? TPMLP_OK : c->fail(TPMLP_ERR_CUDA, cudaGetErrorString(e));
}

// E4M3 copies (row-major and transposed) of a bf16 tensor [rows, cols] with
// its per-tensor scale.  With fused_amax the producer already folded the
// tensor's maximum into its slot; otherwise an amax pass runs first.
tpmlp_status fp8_cast(tpmlp_ctx* c, int tensor, const void* src, int64_t rows, int64_t cols,
                      bool fused_amax = false) {
  float* part = reinterpret_cast<float*>(c->ws8 + c->L8.part);
  float* inv = reinterpret_cast<float*>(c->ws8 + c->L8.inv) + tensor;
  uint8_t* q = c->ws8 + c->L8.q[tensor];
  uint8_t* t = c->ws8 + c->L8.t[tensor];
  const int64_t n = rows * cols;
  int nb = 1;
  if (fused_amax) {
    part = reinterpret_cast<float*>(fp8_amax_slot(c, tensor));
  } else {
    nb = n > 0 ? fp8_blocks(n, c->num_sms) : 1;
    TPMLP_TRY(c->run(K_FP8_AMAX, [&] { return launch_fp8_amax(src, n, part, nb, c->stream); }));
  }
  return c->run(K_FP8_CAST, [&] {
    return launch_fp8_cast(src, rows, cols, q, pitch16(cols), t, pitch16(rows), part, nb, inv, c->num_sms, c->stream);
  });
}

// Point a GEMM at E4M3 operands: A = tensor ta (row-major copy, or the
// transposed one with ta_t), B = tensor tb likewise, both K-major.
void use_fp8(const tpmlp_ctx* c, GemmDesc& g, int ta, bool ta_t, int64_t lda, int tb, bool tb_t, int64_t ldb,
             int64_t b_rows) {
  const float* inv = reinterpret_cast<const float*>(c->ws8 + c->L8.inv);
  g.f8 = true;
  g.a = c->ws8 + (ta_t ? c->L8.t[ta] : c->L8.q[ta]);
  g.lda = lda;
  g.a_mn = false;
  g.b = c->ws8 + (tb_t ? c->L8.t[tb] : c->L8.q[tb]);
  g.ldb = ldb;
  g.b_mn = false;
  g.b_rows = b_rows;
  g.deq_a = inv + ta;
  g.deq_b = inv + tb;
}

}  // namespace

extern "C" {

const char* tpmlp_status_string(tpmlp_status s) {
  switch (s) {
    case TPMLP_OK: return "ok";
    case TPMLP_ERR_ARG: return "invalid argument";
    case TPMLP_ERR_SHAPE: return "invalid shape";
    case TPMLP_ERR_UNSUPPORTED: return "unsupported";
    case TPMLP_ERR_ORDER: return "call out of order";
    case TPMLP_ERR_CUDA: return "CUDA error";
    case TPMLP_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* tpmlp_last_error(const tpmlp_ctx* ctx) { return ctx ? ctx->err.c_str() : g_thread_err.c_str(); }

size_t tpmlp_workspace_bytes(const tpmlp_config* cfg) {
  if (config_error(cfg, nullptr, nullptr)) return 0;
  return make_layout(*cfg).total;
}

tpmlp_status tpmlp_create(const tpmlp_config* cfg, void* cuda_stream, tpmlp_ctx** out) {
  if (!out) {
    g_thread_err = "out is NULL";
    return TPMLP_ERR_ARG;
  }
  *out = nullptr;
  std::string why;
  tpmlp_status st = TPMLP_OK;
  if (config_error(cfg, &why, &st)) {
    g_thread_err = why;
    return st;
  }
  int dev = 0, major = 0, minor = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    g_thread_err = std::string("no usable CUDA device: ") + cudaGetErrorString(e);
    return TPMLP_ERR_CUDA;
  }
  if (major != 10 || minor != 3) {
    char buf[96];
    snprintf(buf, sizeof buf, "device is sm_%d%d; this library is built for sm_103a", major, minor);
    g_thread_err = buf;
    return TPMLP_ERR_UNSUPPORTED;
  }
  tpmlp_ctx* c = new tpmlp_ctx();
  c->cfg = *cfg;
  c->stream = static_cast<cudaStream_t>(cuda_stream);
  c->device = dev;
  c->num_sms = sms;
  c->L = make_layout(*cfg);
  *out = c;
  return TPMLP_OK;
}

tpmlp_status tpmlp_bind_workspace(tpmlp_ctx* c, void* dev, size_t bytes) {
  if (!c) return TPMLP_ERR_ARG;
  if (!dev || (reinterpret_cast<uintptr_t>(dev) & 255u)) return c->fail(TPMLP_ERR_ARG, "workspace must be 256-byte aligned");
  if (bytes < c->L.total) return c->fail(TPMLP_ERR_ARG, "workspace too small");
  c->ws = static_cast<uint8_t*>(dev);
  c->ws_bytes = bytes;
  // the status word, and the split GEMMs' arrival flags: a flag counts when it
  // holds its launch's epoch, so whatever the memory held before must not
  cudaError_t e = cudaMemsetAsync(c->ws + c->L.status, 0, 256, c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->ws + c->L.split_ctr, 0, SPLIT_COUNTER_WORDS * sizeof(uint32_t), c->stream);
  if (e != cudaSuccess) return c->fail(TPMLP_ERR_CUDA, cudaGetErrorString(e));
  return TPMLP_OK;
}

size_t tpmlp_fp8_workspace_bytes(const tpmlp_config* cfg) {
  if (config_error(cfg, nullptr, nullptr) || cfg->dtype != TPMLP_BF16) return 0;
  return make_fp8_layout(*cfg).total;
}

tpmlp_status tpmlp_bind_fp8_workspace(tpmlp_ctx* c, void* dev, size_t bytes) {
  if (!c) return TPMLP_ERR_ARG;
  if (c->cfg.dtype != TPMLP_BF16) return c->fail(TPMLP_ERR_UNSUPPORTED, "FP8 operands are for the bf16 dtype");
  if (!dev || (reinterpret_cast<uintptr_t>(dev) & 255u))
    return c->fail(TPMLP_ERR_ARG, "FP8 workspace must be 256-byte aligned");
  c->L8 = make_fp8_layout(c->cfg);
  if (bytes < c->L8.total) return c->fail(TPMLP_ERR_ARG, "FP8 workspace too small");
  c->ws8 = static_cast<uint8_t*>(dev);
  return TPMLP_OK;
}

tpmlp_status tpmlp_set_precision(tpmlp_ctx* c, int32_t precision) {
  if (!c) return TPMLP_ERR_ARG;
  if (precision != TPMLP_PREC_BF16 && precision != TPMLP_PREC_FP8)
    return c->fail(TPMLP_ERR_ARG, "unknown precision");
  if (precision == TPMLP_PREC_FP8) {
    if (c->cfg.dtype != TPMLP_BF16) return c->fail(TPMLP_ERR_UNSUPPORTED, "FP8 GEMMs are for the bf16 dtype");
    if (!c->ws8) return c->fail(TPMLP_ERR_ORDER, "no FP8 workspace bound");
  }
  c->fp8 = precision == TPMLP_PREC_FP8;
  c->fwd_done = c->bwd_done = false;
  return TPMLP_OK;
}

tpmlp_status tpmlp_set_stream(tpmlp_ctx* c, void* s) {
  if (!c) return TPMLP_ERR_ARG;
  c->stream = static_cast<cudaStream_t>(s);
  return TPMLP_OK;
}

tpmlp_status tpmlp_set_debug(tpmlp_ctx* c, uint32_t flags, int32_t shard) {
  if (!c) return TPMLP_ERR_ARG;
  if (flags & ~31u) return c->fail(TPMLP_ERR_ARG, "unknown debug flag");
  if (shard < 0) return c->fail(TPMLP_ERR_ARG, "shard must be >= 0");
  c->dbg_flags = flags;
  c->dbg_shard = shard;
  return TPMLP_OK;
}

tpmlp_status tpmlp_set_sequence_parallel(tpmlp_ctx* c, int32_t enable) {
  if (!c) return TPMLP_ERR_ARG;
  c->sp = enable != 0;
  c->fwd_done = c->bwd_done = false;
  return TPMLP_OK;
}

tpmlp_status tpmlp_forward(tpmlp_ctx* c, int64_t tokens, const void* x, const void* norm_w, const void* w_gate_up,
                           const void* b_1, const void* w_down, const void* b_down, float eps, int32_t t, void* y) {
  if (!c) return TPMLP_ERR_ARG;
  if (!c->ws) return c->fail(TPMLP_ERR_ORDER, "no workspace bound");
  const tpmlp_config& cf = c->cfg;
  // With zero tokens the activations may be empty (NULL) buffers.
  if (!norm_w || !w_gate_up || !w_down || !b_down || (tokens != 0 && (!x || !y)))
    return c->fail(TPMLP_ERR_ARG, "NULL tensor");
  if (c->swiglu() ? b_1 != nullptr : b_1 == nullptr)
    return c->fail(TPMLP_ERR_ARG, "b_1 is required for GeLU and must be NULL for SwiGLU");
  for (const void* p : {x, norm_w, w_gate_up, w_down, b_down, (const void*)y})
    if (!aligned16(p)) return c->fail(TPMLP_ERR_ARG, "tensor not 16-byte aligned");
  if (b_1 && !aligned16(b_1)) return c->fail(TPMLP_ERR_ARG, "tensor not 16-byte aligned");
  if (tokens < 0 || tokens > cf.max_tokens) return c->fail(TPMLP_ERR_SHAPE, "tokens outside [0, max_tokens]");
  if (t < 1 || t > cf.max_t) return c->fail(TPMLP_ERR_SHAPE, "t outside [1, max_t]");
  if (cf.ffn % t != 0) return c->fail(TPMLP_ERR_SHAPE, "ffn is not divisible by t");
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return c->fail(TPMLP_ERR_ARG, "eps must be finite and >= 0");
  const int64_t H = cf.hidden, F = cf.ffn, Fs = F / t;
  const bool skip_g = (c->dbg_flags & TPMLP_DBG_SKIP_FWD_REDUCE) != 0;
  const bool skip_f = (c->dbg_flags & TPMLP_DBG_SKIP_BWD_REDUCE) != 0;
  const bool skip_sp = (c->dbg_flags & TPMLP_DBG_SKIP_SP_GRAD_SYNC) != 0;
  if ((skip_g || skip_f || skip_sp) && c->dbg_shard >= t) return c->fail(TPMLP_ERR_ARG, "debug shard >= t");
  if (c->sp) {
    if (t > MAX_SP_SHARDS) return c->fail(TPMLP_ERR_SHAPE, "sequence parallelism supports t <= 64");
    if (tokens % t != 0) return c->fail(TPMLP_ERR_SHAPE, "tokens are not divisible by t (sequence parallelism)");
    if (skip_g || skip_f)
      return c->fail(TPMLP_ERR_UNSUPPORTED, "the skip-reduction variants are defined without sequence parallelism");
  } else if (skip_sp) {
    return c->fail(TPMLP_ERR_ARG, "SKIP_SP_GRAD_SYNC needs sequence parallelism");
  }
  const int64_t lo = c->dbg_shard * Fs, hi = lo + Fs;
  if (skip_g && !seg_ok(c, lo, hi, F)) return c->fail(TPMLP_ERR_SHAPE, "shard bounds not on 64-element blocks");
  if (skip_f && !(seg_ok(c, lo, hi, F) && (c->swiglu() ? seg_ok(c, F + lo, F + hi, 2 * F) : true)))
    return c->fail(TPMLP_ERR_SHAPE, "shard bounds not on 64-element blocks");

  c->fwd_done = c->bwd_done = false;
  c->tokens = tokens;
  c->t = t;
  c->x = x;
  c->norm_w = norm_w;
  c->w_gu = w_gate_up;
  c->b_1 = b_1;
  c->w_down = w_down;
  c->b_down = b_down;
  const int dt = cf.dtype == TPMLP_BF16 ? 1 : 0;
  const int force_timeout = (c->dbg_flags & TPMLP_DBG_FORCE_TIMEOUT) != 0;
  if (tokens > 0) {
    void* nrm = c->wsp<void>(c->L.nrm);
    float* rstd = c->wsp<float>(c->L.rstd);
    if (c->fp8) TPMLP_TRY(fp8_clear_amax(c, 0, F8_COUNT));
    uint32_t* nrm_amax = c->fp8 ? fp8_amax_slot(c, F8_NRM) : nullptr;
    TPMLP_TRY(c->run(K_RMSNORM_FWD, [&] {
      return launch_rmsnorm_fwd(dt, x, norm_w, eps, nrm, rstd, tokens, H, c->stream, nrm_amax);
    }));
    if (force_timeout && dt == 0) TPMLP_TRY(c->run(K_PROBE, [&] { return launch_timeout_probe(c->status(), c->stream); }));
    GemmDesc g;
    g.M = (int)tokens;
    g.N = (int)F;
    g.k_extent = H;
    g.a = nrm;
    g.lda = H;
    g.b = w_gate_up;
    g.ldb = H;
    g.kseg[0] = 0;
    g.kseg[1] = H;
    if (c->swiglu()) {
      g.b_rows = 2 * F;
      g.paired = true;
      g.pair_off = F;
      g.epi = EPI_GATEUP_SWIGLU;
      g.ep.out0 = c->wsp<void>(c->L.gu);
      g.ep.ld_out0 = 2 * F;
      g.ep.pair_off = F;
    } else {
      g.b_rows = F;
      g.epi = EPI_FC1_GELU;
      g.ep.out0 = c->wsp<void>(c->L.gu);
      g.ep.ld_out0 = F;
      g.ep.vec = b_1;
    }
    g.ep.out1 = c->wsp<void>(c->L.act);
    g.ep.ld_out1 = F;
    const int64_t guw = c->swiglu() ? 2 * F : F;
    if (c->fp8) {
      TPMLP_TRY(fp8_cast(c, F8_NRM, nrm, tokens, H, true));
      TPMLP_TRY(fp8_cast(c, F8_WGU, w_gate_up, guw, H));
      TPMLP_TRY(fp8_cast(c, F8_WD, w_down, H, F));
      use_fp8(c, g, F8_NRM, false, pitch16(H), F8_WGU, false, pitch16(H), guw);
      g.ep.amax = fp8_amax_slot(c, F8_ACT);
    }
    TPMLP_TRY(run_gemm(c, K_GEMM_GATEUP, g, force_timeout && dt == 1));

    GemmDesc d;
    d.M = (int)tokens;
    d.N = (int)H;
    d.k_extent = F;
    d.a = c->wsp<void>(c->L.act);
    d.lda = F;
    d.b = w_down;
    d.ldb = F;
    d.b_rows = H;
    d.kseg[0] = skip_g ? lo : 0;
    d.kseg[1] = skip_g ? hi : F;
    d.epi = EPI_DOWN_RESID;
    d.ep.out0 = y;
    d.ep.ld_out0 = H;
    d.ep.in0 = x;
    d.ep.ld_in0 = H;
    d.ep.vec = b_down;
    if (c->fp8) {
      TPMLP_TRY(fp8_cast(c, F8_ACT, c->wsp<void>(c->L.act), tokens, F, true));
      use_fp8(c, d, F8_ACT, false, pitch16(F), F8_WD, false, pitch16(F), H);
    }
    TPMLP_TRY(run_gemm(c, K_GEMM_DOWN, d));
  }
  c->fwd_done = true;
  c->upd_done = false;
  return TPMLP_OK;
}

tpmlp_status tpmlp_mse_loss_grad(tpmlp_ctx* c, const void* y, const void* target, void* dy, float* loss_dev) {
  if (!c) return TPMLP_ERR_ARG;
  if (!c->fwd_done) return c->fail(TPMLP_ERR_ORDER, "mse_loss_grad before forward");
  const int64_t n = c->tokens * c->cfg.hidden;
  if (!loss_dev || (n != 0 && (!y || !target || !dy))) return c->fail(TPMLP_ERR_ARG, "NULL tensor");
  if (!aligned16(y) || !aligned16(target) || !aligned16(dy)) return c->fail(TPMLP_ERR_ARG, "tensor not 16-byte aligned");
  if (n == 0) {
    const cudaError_t e = cudaMemsetAsync(loss_dev, 0, sizeof(float), c->stream);
    return e == cudaSuccess ? TPMLP_OK : c->fail(TPMLP_ERR_CUDA, cudaGetErrorString(e));
  }
  const int dt = c->cfg.dtype == TPMLP_BF16 ? 1 : 0;
  const int nb = loss_blocks(n, c->num_sms);
  double* part = c->wsp<double>(c->L.loss_part);
  const float inv = (float)(1.0 / (double)n);
  TPMLP_TRY(c->run(K_LOSS, [&] { return launch_mse_loss_grad(dt, y, target, dy, part, nb, n, inv, c->stream); }));
  TPMLP_TRY(c->run(K_LOSS_FINAL, [&] { return launch_loss_finalize(part, nb, 0.5 / (double)n, loss_dev, c->stream); }));
  return TPMLP_OK;
}

// SGD w <- w - lr g over the parameters of the last forward with the gradients
// of the last backward; the two projection matrices only when `matrices`.
constexpr int64_t UPDATE_IN_EPILOGUE_MIN_TOKENS = 8192;

static tpmlp_status run_sgd(tpmlp_ctx* c, float lr, bool matrices) {
  const int64_t H = c->cfg.hidden, F = c->cfg.ffn;
  const bool sw = c->swiglu();
  SgdArgs a{};
  a.lr = lr;
  auto add = [&](float* m, const float* g, const void* w, int64_t n) {
    a.seg[a.nseg++] = SgdSeg{m, g, const_cast<void*>(w), n};
  };
  add(c->m_norm_w, c->g_norm_w, c->norm_w, H);
  if (matrices) add(c->m_w_gu, c->g_w_gu, c->w_gu, (sw ? 2 * F : F) * H);
  if (!sw) add(c->m_b_1, c->g_b_1, c->b_1, F);
  if (matrices) add(c->m_w_down, c->g_w_down, c->w_down, H * F);
  add(c->m_b_down, c->g_b_down, c->b_down, H);
  const int dt = c->cfg.dtype == TPMLP_BF16 ? 1 : 0;
  return c->run(K_SGD, [&] { return launch_sgd(dt, a, c->num_sms, c->stream); });
}

tpmlp_status tpmlp_backward(tpmlp_ctx* c, const void* dy, void* dx, float* dnorm_w, float* dw_gate_up, float* db_1,
                            float* dw_down, float* db_down) {
  if (!c) return TPMLP_ERR_ARG;
  if (!c->fwd_done) return c->fail(TPMLP_ERR_ORDER, "backward before forward");
  if (!dnorm_w || !dw_gate_up || !dw_down || !db_down || (c->tokens != 0 && (!dy || !dx)))
    return c->fail(TPMLP_ERR_ARG, "NULL tensor");
  if (c->swiglu() ? db_1 != nullptr : db_1 == nullptr)
    return c->fail(TPMLP_ERR_ARG, "db_1 is required for GeLU and must be NULL for SwiGLU");
  for (const void* p : {dy, (const void*)dx, (const void*)dnorm_w, (const void*)dw_gate_up, (const void*)dw_down,
                        (const void*)db_down})
    if (!aligned16(p)) return c->fail(TPMLP_ERR_ARG, "tensor not 16-byte aligned");
  if (db_1 && !aligned16(db_1)) return c->fail(TPMLP_ERR_ARG, "tensor not 16-byte aligned");
  const tpmlp_config& cf = c->cfg;
  const int64_t N = c->tokens, H = cf.hidden, F = cf.ffn, Fs = F / c->t;
  const bool sw = c->swiglu();
  const int64_t guw = sw ? 2 * F : F;
  const int dt = cf.dtype == TPMLP_BF16 ? 1 : 0;
  const bool upd = c->upd_in_bwd;
  if (upd && (!c->m_norm_w || !c->m_w_gu || !c->m_w_down || !c->m_b_down))
    return c->fail(TPMLP_ERR_ORDER, "the update in backward needs bound fp32 masters");
  // The weight matrices are updated in their gradient GEMMs' epilogues when
  // the contraction over tokens is long enough to hide the masters' extra
  // reads and writes there (measured: K = 8192 and 16384 steps 1.5-2.2%
  // faster, K = 4096 even, K = 512 19% slower, where the epilogue's stores
  // already set the pace); otherwise by the update kernel after backward.
  const bool fuse = upd && N >= UPDATE_IN_EPILOGUE_MIN_TOKENS;
  c->bwd_done = false;
  c->upd_done = false;
  c->upd_epi = false;
  c->g_norm_w = dnorm_w;
  c->g_w_gu = dw_gate_up;
  c->g_b_1 = db_1;
  c->g_w_down = dw_down;
  c->g_b_down = db_down;
  if (N == 0) {
    // No tokens: every parameter gradient is an empty sum.
    cudaError_t e = cudaSuccess;
    for (auto pr : {std::make_pair((void*)dnorm_w, H), std::make_pair((void*)dw_gate_up, guw * H),
                    std::make_pair((void*)dw_down, H * F), std::make_pair((void*)db_down, H)})
      if (e == cudaSuccess) e = cudaMemsetAsync(pr.first, 0, (size_t)pr.second * 4, c->stream);
    if (e == cudaSuccess && db_1) e = cudaMemsetAsync(db_1, 0, (size_t)F * 4, c->stream);
    if (e != cudaSuccess) return c->fail(TPMLP_ERR_CUDA, cudaGetErrorString(e));
    c->bwd_done = true;
    if (upd) {
      TPMLP_TRY(run_sgd(c, c->upd_lr, true));
      c->upd_done = true;
    }
    return TPMLP_OK;
  }
  void* gu = c->wsp<void>(c->L.gu);
  void* act = c->wsp<void>(c->L.act);
  void* dgu = c->wsp<void>(c->L.dgu);
  void* nrm = c->wsp<void>(c->L.nrm);
  float* dnrm = c->wsp<float>(c->L.dnrm);

  // dA = dy W_d, then the activation derivative (g backward is the identity).
  GemmDesc a;
  a.M = (int)N;
  a.N = (int)F;
  a.k_extent = H;
  a.a = dy;
  a.lda = H;
  a.b = c->w_down;
  a.ldb = F;
  a.b_mn = true;
  a.kseg[1] = H;
  a.epi = sw ? EPI_DGRAD_SWIGLU : EPI_DGRAD_GELU;
  a.ep.in0 = gu;
  a.ep.ld_in0 = guw;
  a.ep.out0 = dgu;
  a.ep.ld_out0 = guw;
  a.ep.pair_off = F;
  if (c->fp8) {
    TPMLP_TRY(fp8_cast(c, F8_DY, dy, N, H));
    use_fp8(c, a, F8_DY, false, pitch16(H), F8_WD, true, pitch16(H), F);
    TPMLP_TRY(fp8_clear_amax(c, F8_DGU, 1));
    a.ep.amax = fp8_amax_slot(c, F8_DGU);
  }
  TPMLP_TRY(run_gemm(c, K_GEMM_DGRAD_ACT, a));

  // dW_d = dy^T A (contraction over tokens).
  GemmDesc wd;
  wd.M = (int)H;
  wd.N = (int)F;
  wd.k_extent = N;
  wd.a = dy;
  wd.lda = H;
  wd.a_mn = true;
  wd.b = act;
  wd.ldb = F;
  wd.b_mn = true;
  wd.kseg[1] = N;
  wd.epi = EPI_STORE_F32;
  wd.ep.out0 = dw_down;
  wd.ep.ld_out0 = F;
  if (fuse) {  // W_down was last read by the dA GEMM above
    wd.ep.sgd_master = c->m_w_down;
    wd.ep.sgd_w = static_cast<__nv_bfloat16*>(const_cast<void*>(c->w_down));
    wd.ep.sgd_ld = F;
    wd.ep.sgd_lr = c->upd_lr;
  }
  if (c->fp8) use_fp8(c, wd, F8_DY, true, pitch16(N), F8_ACT, true, pitch16(N), F);
  TPMLP_TRY(run_gemm(c, K_GEMM_WGRAD_DOWN, wd));

  if (c->fp8) TPMLP_TRY(fp8_cast(c, F8_DGU, dgu, N, guw, true));
  // dN = sum over shards of dGU_s W_gu,s -- the f all-reduce, summed on chip.
  // It runs before the gate/up weight gradient, which may update W_gate_up.
  GemmDesc dn;
  dn.M = (int)N;
  dn.N = (int)H;
  dn.k_extent = guw;
  dn.a = dgu;
  dn.lda = guw;
  dn.b = c->w_gu;
  dn.ldb = H;
  dn.b_mn = true;
  if (c->dbg_flags & TPMLP_DBG_SKIP_BWD_REDUCE) {
    const int64_t lo = c->dbg_shard * Fs, hi = lo + Fs;
    dn.kseg[0] = lo;
    dn.kseg[1] = hi;
    dn.kseg[2] = sw ? F + lo : 0;
    dn.kseg[3] = sw ? F + hi : 0;
  } else {
    dn.kseg[1] = guw;
  }
  dn.epi = EPI_STORE_F32;
  dn.ep.out0 = dnrm;
  dn.ep.ld_out0 = H;
  if (c->fp8) use_fp8(c, dn, F8_DGU, false, pitch16(guw), F8_WGU, true, pitch16(guw), H);
  TPMLP_TRY(run_gemm(c, K_GEMM_DGRAD_NORM, dn));

  // dW_gate_up = dGU^T n  ([2F, H]; GeLU: dW_1 [F, H]).
  GemmDesc wg;
  wg.M = (int)guw;
  wg.N = (int)H;
  wg.k_extent = N;
  wg.a = dgu;
  wg.lda = guw;
  wg.a_mn = true;
  wg.b = nrm;
  wg.ldb = H;
  wg.b_mn = true;
  wg.kseg[1] = N;
  wg.epi = EPI_STORE_F32;
  wg.ep.out0 = dw_gate_up;
  wg.ep.ld_out0 = H;
  if (fuse) {  // W_gate_up was last read by the dN GEMM above
    wg.ep.sgd_master = c->m_w_gu;
    wg.ep.sgd_w = static_cast<__nv_bfloat16*>(const_cast<void*>(c->w_gu));
    wg.ep.sgd_ld = H;
    wg.ep.sgd_lr = c->upd_lr;
  }
  if (c->fp8) use_fp8(c, wg, F8_DGU, true, pitch16(N), F8_NRM, true, pitch16(N), H);
  TPMLP_TRY(run_gemm(c, K_GEMM_WGRAD_GATEUP, wg));

  if (!sw) {
    const int nb = colsum_blocks(N, c->num_sms);
    float* part = c->wsp<float>(c->L.part_b1);
    TPMLP_TRY(c->run(K_COLSUM_B1, [&] { return launch_colsum_partials(dt, dgu, F, part, N, F, nb, c->stream); }));
    TPMLP_TRY(c->run(K_COLSUM_FINAL, [&] { return launch_colsum_finalize(part, db_1, nullptr, nullptr, nb, F, c->stream); }));
  }

  const int shards = c->sp ? c->t : 1;
  const int nb = rmsnorm_bwd_blocks(N, c->num_sms, shards);
  float* pdw = c->wsp<float>(c->L.part_dw);
  float* pdb = c->wsp<float>(c->L.part_db);
  TPMLP_TRY(c->run(K_RMSNORM_BWD, [&] {
    return launch_rmsnorm_bwd(dt, dnrm, c->x, c->wsp<float>(c->L.rstd), c->norm_w, dy, dx, pdw, pdb, N, H, shards,
                              nb, c->stream);
  }));
  if (!c->sp) {
    TPMLP_TRY(c->run(K_COLSUM_FINAL, [&] { return launch_colsum_finalize(pdw, dnorm_w, pdb, db_down, nb, H, c->stream); }));
  } else {
    // Sequence parallelism: each shard's sums of dN * xhat and dy over its own
    // tokens, then their all-reduce across the shards (walkthrough, "Stage 7:
    // finalize_model_grads"), summed in shard order.  SKIP_SP_GRAD_SYNC keeps
    // the debug shard's own sums instead.
    float* ss_dw = c->wsp<float>(c->L.shard_sums);
    float* ss_db = ss_dw + (int64_t)shards * H;
    TPMLP_TRY(c->run(K_COLSUM_FINAL, [&] {
      return launch_colsum_finalize(pdw, ss_dw, pdb, ss_db, nb / shards, H, c->stream, shards);
    }));
    const bool skip = (c->dbg_flags & TPMLP_DBG_SKIP_SP_GRAD_SYNC) != 0;
    const int64_t off = skip ? (int64_t)c->dbg_shard * H : 0;
    TPMLP_TRY(c->run(K_COLSUM_FINAL, [&] {
      return launch_colsum_finalize(ss_dw + off, dnorm_w, ss_db + off, db_down, skip ? 1 : shards, H, c->stream);
    }));
  }
  c->bwd_done = true;
  if (upd) {
    // the matrices too unless their weight-gradient epilogues updated them
    TPMLP_TRY(run_sgd(c, c->upd_lr, !fuse));
    c->upd_done = true;
    c->upd_epi = fuse;
  }
  return TPMLP_OK;
}

tpmlp_status tpmlp_bind_master(tpmlp_ctx* c, float* norm_w, float* w_gate_up, float* b_1, float* w_down,
                               float* b_down) {
  if (!c) return TPMLP_ERR_ARG;
  const bool none = !norm_w && !w_gate_up && !b_1 && !w_down && !b_down;
  if (none) {
    c->m_norm_w = c->m_w_gu = c->m_b_1 = c->m_w_down = c->m_b_down = nullptr;
    return TPMLP_OK;
  }
  if (c->cfg.dtype != TPMLP_BF16) return c->fail(TPMLP_ERR_UNSUPPORTED, "master weights are for the bf16 dtype");
  if (!norm_w || !w_gate_up || !w_down || !b_down || (c->swiglu() ? b_1 != nullptr : b_1 == nullptr))
    return c->fail(TPMLP_ERR_ARG, "bind all master tensors or none");
  for (const void* p : {(const void*)norm_w, (const void*)w_gate_up, (const void*)w_down, (const void*)b_down})
    if (!aligned16(p)) return c->fail(TPMLP_ERR_ARG, "tensor not 16-byte aligned");
  if (b_1 && !aligned16(b_1)) return c->fail(TPMLP_ERR_ARG, "tensor not 16-byte aligned");
  c->m_norm_w = norm_w;
  c->m_w_gu = w_gate_up;
  c->m_b_1 = b_1;
  c->m_w_down = w_down;
  c->m_b_down = b_down;
  return TPMLP_OK;
}

tpmlp_status tpmlp_sgd_step(tpmlp_ctx* c, float lr) {
  if (!c) return TPMLP_ERR_ARG;
  if (!c->bwd_done) return c->fail(TPMLP_ERR_ORDER, "sgd_step before backward");
  if (c->upd_done) return c->fail(TPMLP_ERR_ORDER, "the last backward already applied the update");
  if (!std::isfinite(lr)) return c->fail(TPMLP_ERR_ARG, "lr must be finite");
  return run_sgd(c, lr, true);
}

int32_t tpmlp_update_in_epilogue(const tpmlp_ctx* c) { return c && c->upd_done && c->upd_epi ? 1 : 0; }

tpmlp_status tpmlp_set_update_in_backward(tpmlp_ctx* c, int32_t enable, float lr) {
  if (!c) return TPMLP_ERR_ARG;
  if (enable && c->cfg.dtype != TPMLP_BF16)
    return c->fail(TPMLP_ERR_UNSUPPORTED, "the update in backward is for the bf16 dtype with fp32 masters");
  if (enable && !std::isfinite(lr)) return c->fail(TPMLP_ERR_ARG, "lr must be finite");
  c->upd_in_bwd = enable != 0;
  c->upd_lr = enable ? lr : 0.0f;
  return TPMLP_OK;
}

tpmlp_status tpmlp_bind_adam_state(tpmlp_ctx* c, const tpmlp_param_set* m, const tpmlp_param_set* v) {
  if (!c) return TPMLP_ERR_ARG;
  if (!m && !v) {
    c->adam_m = tpmlp_param_set{};
    c->adam_v = tpmlp_param_set{};
    c->adam_bound = false;
    return TPMLP_OK;
  }
  if (!m || !v) return c->fail(TPMLP_ERR_ARG, "bind both moment sets or neither");
  for (const tpmlp_param_set* s : {m, v}) {
    if (!s->norm_w || !s->w_gate_up || !s->w_down || !s->b_down || (c->swiglu() ? s->b_1 != nullptr : !s->b_1))
      return c->fail(TPMLP_ERR_ARG, "a moment tensor is missing (b_1 exactly for GeLU)");
    for (const void* p : {(const void*)s->norm_w, (const void*)s->w_gate_up, (const void*)s->b_1,
                          (const void*)s->w_down, (const void*)s->b_down})
      if (p && !aligned16(p)) return c->fail(TPMLP_ERR_ARG, "moment tensor not 16-byte aligned");
  }
  c->adam_m = *m;
  c->adam_v = *v;
  c->adam_bound = true;
  return TPMLP_OK;
}

tpmlp_status tpmlp_adamw_step(tpmlp_ctx* c, const tpmlp_adamw_params* hp, float* grad_norm) {
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
  const int64_t H = c->cfg.hidden, F = c->cfg.ffn;
  const bool sw = c->swiglu();
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
  auto add = [&](float* master, const float* g, const void* w, float* m, float* v, int64_t n, bool decay) {
    a.seg[a.nseg++] = AdamSeg{master, g, const_cast<void*>(w), m, v, n, decay ? lr_wd : 0.0f};
  };
  const tpmlp_param_set &M = c->adam_m, &V = c->adam_v;
  add(c->m_norm_w, c->g_norm_w, c->norm_w, M.norm_w, V.norm_w, H, false);
  add(c->m_w_gu, c->g_w_gu, c->w_gu, M.w_gate_up, V.w_gate_up, (sw ? 2 * F : F) * H, true);
  if (!sw) add(c->m_b_1, c->g_b_1, c->b_1, M.b_1, V.b_1, F, false);
  add(c->m_w_down, c->g_w_down, c->w_down, M.w_down, V.w_down, H * F, true);
  add(c->m_b_down, c->g_b_down, c->b_down, M.b_down, V.b_down, H, false);
  const int nb = adam_blocks(a, c->num_sms);
  const int dt = c->cfg.dtype == TPMLP_BF16 ? 1 : 0;
  TPMLP_TRY(c->run(K_GRAD_NORM, [&] { return launch_grad_sqnorm(a, nb, c->stream); }));
  return c->run(K_ADAMW, [&] { return launch_adamw(dt, a, nb, c->stream); });
}

tpmlp_status tpmlp_sync(tpmlp_ctx* c) {
  if (!c) return TPMLP_ERR_ARG;
  cudaError_t e = cudaStreamSynchronize(c->stream);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return c->fail(TPMLP_ERR_CUDA, cudaGetErrorString(e));
  if (!c->ws) return TPMLP_OK;
  uint32_t st = 0;
  e = cudaMemcpy(&st, c->status(), sizeof st, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return c->fail(TPMLP_ERR_CUDA, cudaGetErrorString(e));
  if (st != 0) {
    cudaMemset(c->status(), 0, sizeof st);
    if (st & STATUS_TIMEOUT) return c->fail(TPMLP_ERR_TIMEOUT, "a bounded device wait gave up");
  }
  return TPMLP_OK;
}

tpmlp_status tpmlp_set_timing(tpmlp_ctx* c, int32_t enable) {
  if (!c) return TPMLP_ERR_ARG;
  c->timing = enable != 0;
  return TPMLP_OK;
}

int32_t tpmlp_read_kernel_times(tpmlp_ctx* c, float* ms, int64_t* launches, int32_t n) {
  if (!c || n < 0) return -1;
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return -1;
  const int m = n < K_COUNT ? n : K_COUNT;
  for (int i = 0; i < m; ++i) {
    if (ms) ms[i] = 0.0f;
    if (launches) launches[i] = 0;
  }
  for (auto& r : c->recs) {
    float t = 0.0f;
    cudaEventElapsedTime(&t, r.a, r.b);
    if (r.id < m) {
      if (ms) ms[r.id] += t;
      if (launches) launches[r.id] += 1;
    }
    c->free_events.push_back(r.a);
    c->free_events.push_back(r.b);
  }
  c->recs.clear();
  return m;
}

const char* tpmlp_kernel_name(int32_t id) { return (id >= 0 && id < K_COUNT) ? kKernelNames[id] : nullptr; }

int32_t tpmlp_num_kernel_ids(void) { return K_COUNT; }

uint64_t tpmlp_launch_count(const tpmlp_ctx* c) { return c ? c->launches : 0; }

void tpmlp_destroy(tpmlp_ctx* c) {
  if (!c) return;
  for (auto& r : c->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : c->free_events) cudaEventDestroy(e);
  delete c;
}

}  // extern "C"
