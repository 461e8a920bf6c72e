// Fused causal attention on the sm_103a tensor cores, for the tensor-parallel
// attention sublayer ("Megatron-LM Explained", "Self-attention: split across
// heads"): softmax(Q K^T / sqrt(d)) V per (sequence, query head) with the
// scores kept on chip, and its backward from each query row's log-sum-exp.
//
// Forward.  One CTA owns two 128-query tiles (A, B) of one (sequence, query
// head) and streams the key/value blocks of its KV group up to the diagonal;
// both tiles share every K_j / V_j load:
//
//   warp 0     : TMA producer -- Q_A, Q_B once; K_j and V_j into two-stage rings.
//   warp 1     : owns tensor memory -- per tile a 128-column score buffer
//                S (later overwritten by P as packed bf16) and a 128-column
//                output accumulator O -- and issues tcgen05.mma:
//                S_X = Q_X K_j^T, then O_X += P_X V_j with P_X read straight
//                from tensor memory, alternating the tiles so one tile's
//                softmax runs under the other tile's products.
//   warps 2..5 : online softmax of tile A, one query row per thread;
//   warps 6..9 : the same for tile B.  Per key block: one read of the score
//                row, the row maximum, P = exp2(s - m) written back as bf16,
//                the running sum l.  The running maximum m is only moved
//                (and O rescaled in tensor memory) when a block's maximum
//                exceeds it by more than 2^8, so most blocks touch O not at
//                all; P stays below 2^8 in the stale frame.  Finally O / l as
//                bf16 (TMA store) and the base-2 log-sum-exp m + log2(l).
//
// Scores are scaled by 1/sqrt(d); exponentials run in base 2 with log2(e)
// folded into the scale.  The diagonal block masks keys above the query.
// Every wait is bounded (1 s); a wait that gives up sets the status word,
// and the CTA drains and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "f32x2.cuh"
#include "ptx_sm103.cuh"
#include "tma_maps.cuh"
#include "tpmlp_internal.h"
#include "vec.cuh"

namespace tpmlp {
namespace {

constexpr int FB = 128;  // queries per tile = keys per block
constexpr int FD = 128;  // head dimension
constexpr int FTHREADS = 320;
constexpr uint32_t FCOLS = 512;
constexpr uint64_t FWAIT_NS = 1000000000ull;
constexpr uint64_t FDRAIN_NS = 200000000ull;
constexpr uint32_t TILE_BYTES = FB * 64 * 2;     // one [128 x 64] bf16 SW128 tile, 16 KB
constexpr uint32_t OPND_BYTES = 2 * TILE_BYTES;  // a [128 x 128] operand: two tiles
constexpr float RESCALE_LOG2 = 8.0f;             // move the running maximum only past 2^8
// shared memory: Q_A, Q_B (each reused as its tile's output staging), K ring, V ring
constexpr uint32_t SQ = 0;
constexpr uint32_t SK = SQ + 2 * OPND_BYTES;
constexpr uint32_t SV = SK + 2 * OPND_BYTES;
constexpr uint32_t FSMEM = SV + 2 * OPND_BYTES + 1024;

struct FaParams {
  int S, nq, nkv, hpg, nqblk;  // nqblk: 256-query blocks per sequence
  int k_col0, v_col0;          // first key / value column of the QKV tensor
  float scale_log2;            // log2(e) / sqrt(d)
  float* lse2;                 // [batch * nq * S] base-2 log-sum-exp of the scaled scores
  uint32_t* status;
};

// Row r of a [32 x 32] bf16 box with the 64-byte swizzle (TMA store staging).
__device__ __forceinline__ void stage_row_bf16_fa(uint8_t* tile, int r, const float* v) {
  uint8_t* rowp = tile + r * 64;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 w;
    __nv_bfloat162 h;
    h = __floats2bfloat162_rn(v[8 * c], v[8 * c + 1]);
    w.x = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(v[8 * c + 2], v[8 * c + 3]);
    w.y = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(v[8 * c + 4], v[8 * c + 5]);
    w.z = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(v[8 * c + 6], v[8 * c + 7]);
    w.w = *reinterpret_cast<uint32_t*>(&h);
    *reinterpret_cast<uint4*>(rowp + ((c ^ ((r >> 1) & 3)) << 4)) = w;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(FTHREADS, 1)
    flash_fwd_kernel(const __grid_constant__ CUtensorMap map_qkv, const __grid_constant__ CUtensorMap map_z,
                     const FaParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2],
      o_full[2], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile int* abort_flag = &abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // block -> (256-query block, head, sequence), the longest (diagonal-most)
  // query blocks of every head first: CTAs start in block order, so the last
  // ones to start are the shortest.  (Ordered per head instead, a 16-key-block
  // CTA started last; a list-scheduling model of 152 SMs puts that order 15%
  // over the balanced time and this one within 3%.)  The K and V blocks of all
  // groups (32 MB at 4 x 2048 tokens) stay in L2 either way.
  const int nbh = (int)(gridDim.x / p.nqblk);
  const int qb = p.nqblk - 1 - (int)(blockIdx.x / nbh);
  const int bh = (int)(blockIdx.x % nbh);
  const int h = bh % p.nq, b = bh / p.nq;
  const int g = h / p.hpg;
  const int q0 = qb * 2 * FB;           // first query of tile A
  const bool has_b = q0 + FB < p.S;     // tile B exists (S % 256 == 128 leaves the last CTA one tile)
  const int nk_a = 2 * qb + 1;          // key blocks seen by tile A (its diagonal is the last)
  const int nk_b = has_b ? 2 * qb + 2 : 0;
  const int nk = has_b ? nk_b : nk_a;
  const int row_seq = b * p.S;

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&o_full[i], 1);
    }
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_qkv);
    tma_prefetch_desc(&map_z);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, FCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t armed_k = 0, par_k = 0, armed_v = 0, par_v = 0;
      bool ok = true;
      mbar_arrive_expect_tx(&q_full, (has_b ? 2 : 1) * OPND_BYTES);
      for (int x = 0; x < (has_b ? 2 : 1); ++x)
        for (int t = 0; t < 2; ++t)
          tma_load_2d(smem + SQ + x * OPND_BYTES + t * TILE_BYTES, &map_qkv, &q_full, h * FD + 64 * t,
                      row_seq + q0 + x * FB);
      for (int j = 0; ok && j < nk; ++j) {
        const int s = j & 1;
        const uint32_t par = (uint32_t)((j >> 1) & 1);
        const int row_k = row_seq + j * FB;
        if (!mbar_wait(&k_empty[s], par ^ 1u, abort_flag, p.status, STATUS_TIMEOUT, FWAIT_NS)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&k_full[s], OPND_BYTES);
        armed_k |= 1u << s;
        par_k = (par_k & ~(1u << s)) | (par << s);
        for (int t = 0; t < 2; ++t)
          tma_load_2d(smem + SK + s * OPND_BYTES + t * TILE_BYTES, &map_qkv, &k_full[s], p.k_col0 + g * FD + 64 * t,
                      row_k);
        if (!mbar_wait(&v_empty[s], par ^ 1u, abort_flag, p.status, STATUS_TIMEOUT, FWAIT_NS)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&v_full[s], OPND_BYTES);
        armed_v |= 1u << s;
        par_v = (par_v & ~(1u << s)) | (par << s);
        for (int t = 0; t < 2; ++t)
          tma_load_2d(smem + SV + s * OPND_BYTES + t * TILE_BYTES, &map_qkv, &v_full[s], p.v_col0 + g * FD + 64 * t,
                      row_k);
      }
      if (!ok || *abort_flag) {
        // copies still in flight land on the full barriers of the phases armed last
        int no_abort = 0;
        mbar_wait(&q_full, 0, &no_abort, p.status, 0u, FDRAIN_NS);
        for (int s = 0; s < 2; ++s) {
          if (armed_k & (1u << s)) mbar_wait(&k_full[s], (par_k >> s) & 1u, &no_abort, p.status, 0u, FDRAIN_NS / 4);
          if (armed_v & (1u << s)) mbar_wait(&v_full[s], (par_v >> s) & 1u, &no_abort, p.status, 0u, FDRAIN_NS / 4);
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    constexpr uint32_t IDESC_S = idesc_bf16_f32(FB, FB, false, false);
    constexpr uint32_t IDESC_PV = idesc_bf16_f32(FB, FD, false, true);
    // The warp runs this role in warp-uniform control flow; one lane, elected
    // at each issue point, issues the MMAs and commits.  Descriptors are
    // built once and advanced by constant offsets, so an MMA costs an add and
    // the instruction: a 128-wide product keeps the tensor core busy for only
    // about 64 cycles, less than rebuilding two descriptors per MMA took.
    const uint64_t q_desc = sw128_desc(smem_u32(smem + SQ), 16, 1024);
    const uint64_t k_desc = sw128_desc(smem_u32(smem + SK), 16, 1024);
    const uint64_t v_desc = sw128_desc(smem_u32(smem + SV), TILE_BYTES, 1024);
    auto wait_all = [&](uint64_t* bar, uint32_t par) -> int {
      return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag, p.status, STATUS_TIMEOUT, FWAIT_NS));
    };
    // S_x = Q_x K_j^T into tile x's score columns (issued by the elected lane)
    auto mma_s = [&](int x, int j) {
      const uint64_t qa = desc_advance(q_desc, x * OPND_BYTES), kb = desc_advance(k_desc, (j & 1) * OPND_BYTES);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc_mma_f16(tmem_base + x * FB, desc_advance(qa, (kk >> 2) * TILE_BYTES + (kk & 3) * 32),
                   desc_advance(kb, (kk >> 2) * TILE_BYTES + (kk & 3) * 32), IDESC_S, kk > 0 ? 1u : 0u);
      tc_commit(&s_full[x]);
    };
    // O_x += P_x V_j, P_x from tile x's score columns (bf16 pairs, 8 columns per K = 16)
    auto mma_pv = [&](int x, int j, bool last) {
      const uint64_t vb = desc_advance(v_desc, (j & 1) * OPND_BYTES);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc_mma_f16_ts(tmem_base + 256 + x * FD, tmem_base + x * FB + kk * 8, desc_advance(vb, kk * 2048), IDESC_PV,
                      (j > 0 || kk > 0) ? 1u : 0u);
      if (last) tc_commit(&o_full[x]);
    };
    auto issue_s = [&](int x, int j) {
      if (elect_one()) mma_s(x, j);
      __syncwarp();
    };
    auto issue_pv = [&](int x, int j, bool last) {
      if (elect_one()) mma_pv(x, j, last);
      __syncwarp();
    };
    int ok = wait_all(&q_full, 0) && wait_all(&k_full[0], 0);
    if (ok) {
      tc_fence_after();
      issue_s(0, 0);
      if (has_b) issue_s(1, 0);
      if (elect_one()) tc_commit(&k_empty[0]);
      __syncwarp();
    }
    for (int j = 0; ok && j < nk; ++j) {
      const int s = j & 1;
      if (!(ok = wait_all(&v_full[s], (j >> 1) & 1))) break;
      const bool next = j + 1 < nk;
      if (j < nk_a) {
        if (!(ok = wait_all(&p_full[0], j & 1))) break;
        tc_fence_after();
        issue_pv(0, j, j + 1 == nk_a);
      }
      if (next && !(ok = wait_all(&k_full[(j + 1) & 1], ((j + 1) >> 1) & 1))) break;
      tc_fence_after();
      if (j + 1 < nk_a) issue_s(0, j + 1);
      if (has_b) {
        if (!(ok = wait_all(&p_full[1], j & 1))) break;
        tc_fence_after();
      }
      // tile B's products and the ring releases in one elected issue (one
      // issue point fewer per key block: 2% on the 2048-token workload)
      if (elect_one()) {
        if (has_b) {
          mma_pv(1, j, j + 1 == nk_b);
          if (j + 1 < nk_b) mma_s(1, j + 1);
        }
        tc_commit(&v_empty[s]);
        if (next) tc_commit(&k_empty[(j + 1) & 1]);
      }
      __syncwarp();
    }
    if (elect_one()) tc_commit(&drain_bar);
    __syncwarp();
    int no_abort = 0;
    mbar_wait(&drain_bar, 0, &no_abort, p.status, STATUS_TIMEOUT, FDRAIN_NS);
  } else {
    // --------------------------------------------------------- softmax warps
    const int x = (warp - 2) >> 2;  // tile
    const int q4 = warp & 3;        // TMEM lane quarter of this warp
    const int r = q4 * 32 + lane;   // query row within the tile
    const int nkx = x ? nk_b : nk_a;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t t_s = tmem_base + lane_off + x * FB;
    const uint32_t t_o = tmem_base + lane_off + 256 + x * FD;
    float m_run = -INFINITY, l = 0.0f;  // running maximum (log2 units, possibly stale) and sum
    int ok = nkx > 0;                   // tile B may be absent
    for (int j = 0; ok && j < nkx; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[x], j & 1, abort_flag, p.status, STATUS_TIMEOUT, FWAIT_NS));
      if (!ok) break;
      tc_fence_after();
      uint32_t v[128];
      tmem_ld_32x32b_x32(t_s, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_32x32b_x32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_32x32b_x32(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(v + 64));
      tmem_ld_32x32b_x32(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(v + 96));
      tmem_ld_wait();
      const bool diag = j == nkx - 1;  // keys above the query are masked (-> P = 0)
      if (diag) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > r) v[c] = __float_as_uint(-INFINITY);
      }
      // row maximum over eight independent chains (column c in chain c % 8)
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float m = __uint_as_float(v[k]);
#pragma unroll
        for (int i = 1; i < 15; i += 2) m = fmax3(m, __uint_as_float(v[k + 8 * i]), __uint_as_float(v[k + 8 * i + 8]));
        mx[k] = fmaxf(m, __uint_as_float(v[k + 120]));
      }
      float mb = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
      mb *= p.scale_log2;
      const bool move = __any_sync(0xffffffffu, mb > m_run + RESCALE_LOG2);
      float alpha = 1.0f;
      if (move) {
        const float m_new = fmaxf(m_run, mb);
        alpha = ex2_fast(m_run - m_new);  // 0 on the first block
        l *= alpha;
        m_run = m_new;
      }
      // P = 2^(s scale - m) a column pair at a time; the row sum in four
      // independent pair accumulators
      const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nm2 = f2_pack(-m_run, -m_run);
      uint64_t ps2[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) ps2[k] = f2_pack(0.0f, 0.0f);
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        float a0, a1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), sc2, nm2), a0, a1);
        const float p0 = ex2_fast(a0), p1 = ex2_fast(a1);
        ps2[(c >> 1) & 3] = f2_add(ps2[(c >> 1) & 3], f2_pack(p0, p1));
        v[c >> 1] = pack_bf16x2(p0, p1);
      }
      {
        float s0, s1, s2, s3, s4, s5, s6, s7;
        f2_unpack(ps2[0], s0, s1);
        f2_unpack(ps2[1], s2, s3);
        f2_unpack(ps2[2], s4, s5);
        f2_unpack(ps2[3], s6, s7);
        l += ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
      }
      tmem_st_32x32b_x32(t_s, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_st_32x32b_x32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      if (move && j > 0) {
        // O holds blocks < j (the score MMA of block j was issued after the
        // output MMA of block j - 1, so that one has completed too); the
        // output MMA of block j waits for p_full below
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_o + 32 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st_32x32b_x32(t_o + 32 * c, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[x]);
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&o_full[x], 0, abort_flag, p.status, STATUS_TIMEOUT, FWAIT_NS));
      if (ok) {
        tc_fence_after();
        const float inv = 1.0f / l;
        const int row = q0 + x * FB + r;
        p.lse2[(size_t)bh * p.S + row] = m_run + log2f(l);
        // output rows [q0 + x FB + 32 q4, +32): this warp's 8 KB of the tile's
        // (now idle) Q buffer, four [32 x 32] boxes
        uint8_t* stg = smem + SQ + x * OPND_BYTES + q4 * 8192;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_o + 32 * c, o);
          tmem_ld_wait();
          float f[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(o[e]) * inv;
          stage_row_bf16_fa(stg + c * 2048, lane, f);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int c = 0; c < 4; ++c) tma_store_2d(&map_z, stg + c * 2048, h * FD + c * 32, row_seq + q0 + x * FB + q4 * 32);
          bulk_commit_group();
          bulk_wait_all();
        }
        __syncwarp();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, FCOLS);
  }
}

// ---------------------------------------------------------------- backward
// One CTA per (sequence b, KV group g, 128-key block j) accumulates dK_j and
// dV_j of the group in tensor memory over every query head of the group and
// every 64-query block i that sees the keys (i >= 2 j), and adds each
// dQ_i contribution into an f32 accumulator with reductions.  With P
// recomputed from the forward's log-sum-exp and D_i = rowsum(dO_i o O_i):
//
//   S^T  = K_j Q_i^T               dP^T = V_j dO_i^T
//   P^T  = exp2(S^T log2(e)/sqrt(d) - lse2_i)    (keys above a query masked)
//   dS^T = P^T o (dP^T - D_i) / sqrt(d)
//   dV_j += P^T dO_i               dK_j += dS^T Q_i      dQ_i^T = K_j^T dS^T
//
//   warp 0      : TMA producer -- K_j, V_j once; Q_i, dO_i, lse2_i per
//                 step into a four-stage ring (the row warps read D_i from
//                 global memory).  Steps run over the query
//                 blocks from the last one down, the heads of the group
//                 inner, so the CTAs of one (sequence, group) read the same
//                 Q / dO blocks at about the same time.
//   warp 1      : tensor memory owner; issues the score-side products
//                 S^T and dP^T.
//   warp 14     : issues the accumulating products dV, dQ^T and dK.
//                 Two issuers keep products queued while either one waits
//                 on a barrier: each wait costs an issue gap, and with one
//                 issuer every gap reached the tensor pipe.
//   warps 2..5  : row group 0, the even steps; warps 6..9: row group 1, the
//                 odd steps.  One key row per thread: P^T (bf16, written
//                 over its scores in tensor memory, where the dV product
//                 reads it) and dS^T (bf16, into the group's shared-memory
//                 tile in the K-major layout the MMAs read); at the end
//                 group 0 writes the dV rows and group 1 the dK rows.
//   warps 10..13: dQ^T epilogue, one head-dim row per thread: tensor memory
//                 to registers, then reductions into the f32 dQ accumulator.
// Every step-indexed buffer has two slots, step n using slot n & 1, so the
// two row groups work on consecutive steps at the same time and one group's
// element-wise work runs under the products of the other group's step:
// tensor memory holds S^T / P^T per slot, dP^T per slot (overwritten by the
// step's dQ^T once the group has read dP^T), dV_j and dK_j.  Per step n the
// score issuer issues dP^T_{n+1} and S^T_{n+2}; the accumulating issuer
// dV_n, dQ^T_n and dK_n.  Products of one issuer run in issue order; across
// the two, every reuse of a buffer waits on a barrier: S^T_{n+2} overwrites
// slot n & 1 only after dV_n has read P^T_n (pv_done) and the row group has
// read it back for dS (ds_full).
// The same shared-memory tile of Q, dO, K or dS^T serves as a K-major operand
// of one product and an MN-major operand of another: a 128-byte swizzled tile
// of 64-element rows is both.
constexpr int BKB = 128;  // keys per CTA
constexpr int BQB = 64;   // queries per step
constexpr int BTHREADS = 480;
constexpr int B_ISSUER = 14;  // warp index of the second MMA issuer
constexpr int GROUP_WARPS = 4;  // warps per row group: one per TMEM lane quarter
constexpr uint32_t KT_BYTES = BKB * 64 * 2;   // [128 keys x 64 d] tile, 16 KB
constexpr uint32_t QT_BYTES = BQB * 64 * 2;   // [64 queries x 64 d] tile, 8 KB
// shared memory
constexpr uint32_t B_SK = 0;                          // K_j: two 16 KB tiles
constexpr uint32_t B_SV = B_SK + 2 * KT_BYTES;        // V_j
constexpr int QST = 4;                                // Q / dO / lse2 ring stages
constexpr uint32_t B_SQ = B_SV + 2 * KT_BYTES;        // Q_i ring: QST stages x two 8 KB tiles
constexpr uint32_t B_SDO = B_SQ + 2 * QST * QT_BYTES; // dO_i ring
constexpr uint32_t B_SDS = B_SDO + 2 * QST * QT_BYTES; // dS^T: 2 slots x [128 keys x 64 queries], 16 KB each
constexpr uint32_t B_SLD = B_SDS + 2 * KT_BYTES;      // lse2 ring: QST stages x 64 floats
constexpr uint32_t BSMEM = B_SLD + QST * BQB * 4 + 1024;
static_assert(BSMEM <= 232448 - 256, "shared memory budget");
constexpr uint32_t IN_TX = 4 * QT_BYTES + BQB * 4;
// tensor memory columns
constexpr uint32_t T_S = 0;     // S^T: 2 slots x 64 (P^T over the first 32 columns of its slot)
constexpr uint32_t T_PQ = 128;  // dP^T, then dQ^T: 2 slots x 64
constexpr uint32_t T_DV = 256;  // dV_j: 128
constexpr uint32_t T_DK = 384;  // dK_j: 128

struct FbParams {
  int S, nq, nkv, hpg;
  int q64;  // S / 64
  int k_col0, v_col0;
  float scale_log2, scale;
  const float* lse2;  // [batch * nq * S]
  const float* dsum;  // D, same layout
  __nv_bfloat16* dqkv;
  int64_t ld_dqkv;
  float* dq_acc;  // [batch S, nq d] f32 dQ accumulator
  int64_t ld_dq;
  uint32_t* status;
};

// *addr += v in global memory, no value returned
__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

__global__ void __launch_bounds__(BTHREADS, 1)
    flash_bwd_kernel(const __grid_constant__ CUtensorMap map_kv, const __grid_constant__ CUtensorMap map_q,
                     const __grid_constant__ CUtensorMap map_do, const FbParams p, int batch) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t kv_full, in_full[QST], in_empty[QST], s_full[2], p_full[2], dp_full[2],
      ds_full[2], ds_empty[2], dq_full[2], dq_empty[2], pv_done[2], acc_full, drain_bar, drain_b;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile int* abort_flag = &abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // block -> (key block j, sequence b, group g); the key blocks with the most query blocks first
  const int nbg = batch * p.nkv;
  const int j = (int)(blockIdx.x / nbg);
  const int bg = (int)(blockIdx.x % nbg);
  const int b = bg / p.nkv, g = bg % p.nkv;
  const int i0 = 2 * j;                 // first 64-query block that sees key block j
  const int per_head = p.q64 - i0;
  const int nsteps = p.hpg * per_head;  // >= 2
  const int row_k = b * p.S + j * BKB;
  // step n -> 64-query block i (from the last down) and query head h of the group
  auto step_i = [&](int n) { return p.q64 - 1 - n / p.hpg; };
  auto step_h = [&](int n) { return g * p.hpg + n % p.hpg; };

  if (threadIdx.x == 0) {
    mbar_init(&kv_full, 1);
    for (int i = 0; i < QST; ++i) {
      mbar_init(&in_full[i], 1);
      mbar_init(&in_empty[i], 1 + GROUP_WARPS);  // the MMA commit and the step's row group (lse2 / D reads)
    }

    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], GROUP_WARPS);
      mbar_init(&dp_full[i], 1);
      mbar_init(&ds_full[i], GROUP_WARPS);
      mbar_init(&ds_empty[i], 1);
      mbar_init(&dq_full[i], 1);
      mbar_init(&dq_empty[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&drain_bar, 1);
    mbar_init(&drain_b, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_kv);
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_do);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, FCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  auto wait_all = [&](uint64_t* bar, uint32_t par) -> int {
    return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag, p.status, STATUS_TIMEOUT, FWAIT_NS));
  };
  auto arrive = [&](uint64_t* bar) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      mbar_arrive_expect_tx(&kv_full, 4 * KT_BYTES);
      for (int t = 0; t < 2; ++t) {
        tma_load_2d(smem + B_SK + t * KT_BYTES, &map_kv, &kv_full, p.k_col0 + g * FD + 64 * t, row_k);
        tma_load_2d(smem + B_SV + t * KT_BYTES, &map_kv, &kv_full, p.v_col0 + g * FD + 64 * t, row_k);
      }
      for (int n = 0; ok && n < nsteps; ++n) {
        const int s = n % QST;
        const uint32_t par = (uint32_t)((n / QST) & 1);
        if (!mbar_wait(&in_empty[s], par ^ 1u, abort_flag, p.status, STATUS_TIMEOUT, FWAIT_NS)) {
          ok = false;
          break;
        }
        const int h = step_h(n), i = step_i(n);
        const int row_q = b * p.S + i * BQB;
        mbar_arrive_expect_tx(&in_full[s], IN_TX);
        armed |= 1u << s;
        armed_par = (armed_par & ~(1u << s)) | (par << s);
        for (int t = 0; t < 2; ++t) {
          tma_load_2d(smem + B_SQ + (2 * s + t) * QT_BYTES, &map_q, &in_full[s], h * FD + 64 * t, row_q);
          tma_load_2d(smem + B_SDO + (2 * s + t) * QT_BYTES, &map_do, &in_full[s], h * FD + 64 * t, row_q);
        }
        const size_t li = ((size_t)(b * p.nq + h)) * p.S + (size_t)i * BQB;
        bulk_load_1d(smem + B_SLD + s * 256, p.lse2 + li, BQB * 4, &in_full[s]);
      }
      if (!ok || *abort_flag) {
        int no_abort = 0;
        mbar_wait(&kv_full, 0, &no_abort, p.status, 0u, FDRAIN_NS);
        for (int s = 0; s < QST; ++s)
          if (armed & (1u << s)) mbar_wait(&in_full[s], (armed_par >> s) & 1u, &no_abort, p.status, 0u, FDRAIN_NS / 4);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    constexpr uint32_t IDESC_SP = idesc_bf16_f32(BKB, BQB, false, false);  // S^T, dP^T
    constexpr uint32_t IDESC_KV = idesc_bf16_f32(BKB, FD, false, true);    // dV, dK
    constexpr uint32_t IDESC_DQ = idesc_bf16_f32(FD, BQB, true, true);     // dQ^T
    // Warp-uniform control flow; one lane, elected at each issue point,
    // issues the MMAs and commits.  Descriptors are built once and advanced
    // by constant offsets, so an MMA costs an add and the instruction.
    const uint64_t k_kdesc = sw128_desc(smem_u32(smem + B_SK), 16, 1024);        // K, K-major
    const uint64_t v_kdesc = sw128_desc(smem_u32(smem + B_SV), 16, 1024);        // V, K-major
    const uint64_t k_mdesc = sw128_desc(smem_u32(smem + B_SK), KT_BYTES, 1024);  // K^T, MN-major
    const uint64_t q_kdesc = sw128_desc(smem_u32(smem + B_SQ), 16, 1024);        // Q ring, K-major
    const uint64_t q_mdesc = sw128_desc(smem_u32(smem + B_SQ), QT_BYTES, 1024);  // Q ring, MN-major
    const uint64_t o_kdesc = sw128_desc(smem_u32(smem + B_SDO), 16, 1024);       // dO ring, K-major
    const uint64_t o_mdesc = sw128_desc(smem_u32(smem + B_SDO), QT_BYTES, 1024); // dO ring, MN-major
    const uint64_t ds_kdesc = sw128_desc(smem_u32(smem + B_SDS), 16, 1024);      // dS^T slots, K-major
    const uint64_t ds_mdesc = sw128_desc(smem_u32(smem + B_SDS), KT_BYTES, 1024);// dS^T slots, MN-major
    // S^T_n = K Q_n^T or dP^T_n = V dO_n^T, then a commit to `done`
    auto issue_nt = [&](uint32_t d_tmem, uint64_t a, uint64_t bq, uint64_t* done) {
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16(d_tmem, desc_advance(a, (kk >> 2) * KT_BYTES + (kk & 3) * 32),
                     desc_advance(bq, (kk >> 2) * QT_BYTES + (kk & 3) * 32), IDESC_SP, kk > 0 ? 1u : 0u);
        tc_commit(done);
      }
      __syncwarp();
    };
    // S^T_n into slot n & 1, where P^T_{n-2} was read by dV_{n-2}: issued before it, in order
    auto issue_s = [&](int n) -> int {
      const int q = n % QST;
      if (!wait_all(&in_full[q], (n / QST) & 1)) return 0;
      tc_fence_after();
      issue_nt(tmem_base + T_S + (n & 1) * BQB, k_kdesc, desc_advance(q_kdesc, 2 * q * QT_BYTES), &s_full[n & 1]);
      return 1;
    };
    // dP^T_n into slot n & 1 once dQ^T_{n-2} has been read out of it; dO_n is
    // in place since S^T_n was issued
    auto issue_dp = [&](int n) -> int {
      if (!wait_all(&dq_empty[n & 1], ((n >> 1) & 1) ^ 1u)) return 0;
      tc_fence_after();
      issue_nt(tmem_base + T_PQ + (n & 1) * BQB, v_kdesc, desc_advance(o_kdesc, 2 * (n % QST) * QT_BYTES),
               &dp_full[n & 1]);
      return 1;
    };
    int ok = wait_all(&kv_full, 0);
    if (ok) ok = issue_s(0);
    if (ok && nsteps > 1) ok = issue_s(1);
    if (ok) ok = issue_dp(0);
    for (int n = 0; ok && n < nsteps; ++n) {
      if (n + 1 < nsteps && !(ok = issue_dp(n + 1))) break;
      if (n + 2 < nsteps) {
        // slot n & 1 holds P^T_n until dV_n has read it and the row group
        // has read it back for dS_n
        const uint32_t par = (uint32_t)((n >> 1) & 1);
        if (!(ok = wait_all(&pv_done[n & 1], par))) break;
        if (!(ok = wait_all(&ds_full[n & 1], par))) break;
        if (!(ok = issue_s(n + 2))) break;
      }
    }
    if (elect_one()) tc_commit(&drain_bar);
    __syncwarp();
    int no_abort = 0;
    mbar_wait(&drain_bar, 0, &no_abort, p.status, STATUS_TIMEOUT, FDRAIN_NS);
  } else if (warp == B_ISSUER) {
    // ------------------------------------------------- accumulating issuer
    constexpr uint32_t IDESC_KV = idesc_bf16_f32(BKB, FD, false, true);    // dV, dK
    constexpr uint32_t IDESC_DQ = idesc_bf16_f32(FD, BQB, true, true);     // dQ^T
    const uint64_t k_mdesc = sw128_desc(smem_u32(smem + B_SK), KT_BYTES, 1024);  // K^T, MN-major
    const uint64_t q_mdesc = sw128_desc(smem_u32(smem + B_SQ), QT_BYTES, 1024);  // Q ring, MN-major
    const uint64_t o_mdesc = sw128_desc(smem_u32(smem + B_SDO), QT_BYTES, 1024); // dO ring, MN-major
    const uint64_t ds_kdesc = sw128_desc(smem_u32(smem + B_SDS), 16, 1024);      // dS^T slots, K-major
    const uint64_t ds_mdesc = sw128_desc(smem_u32(smem + B_SDS), KT_BYTES, 1024);// dS^T slots, MN-major
    int ok = 1;
    for (int n = 0; ok && n < nsteps; ++n) {
      const int s = n & 1, q = n % QST;
      const uint32_t par = (uint32_t)((n >> 1) & 1);
      const uint64_t sq = desc_advance(q_mdesc, 2 * q * QT_BYTES), sdo = desc_advance(o_mdesc, 2 * q * QT_BYTES);
      const uint64_t sds_k = desc_advance(ds_kdesc, s * KT_BYTES), sds_m = desc_advance(ds_mdesc, s * KT_BYTES);
      // dV += P^T dO_n, P^T from tensor memory (bf16 pairs, 8 columns per K = 16).
      // p_full implies S^T_n, issued after dO_n landed, has been read.
      if (!(ok = wait_all(&p_full[s], par))) break;
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_f16_ts(tmem_base + T_DV, tmem_base + T_S + s * BQB + kk * 8, desc_advance(sdo, kk * 2048), IDESC_KV,
                        (n > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&pv_done[s]);
      }
      __syncwarp();
      // dQ^T_n = K^T dS^T over the slot's dP^T, which the group has read; then
      // dK += dS^T Q_n.  dQ^T goes first so that its slot, which dP^T_{n+2}
      // needs next, is read out while dK_n keeps the tensor core busy.
      if (!(ok = wait_all(&ds_full[s], par))) break;
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16(tmem_base + T_PQ + s * BQB, desc_advance(k_mdesc, kk * 2048), desc_advance(sds_m, kk * 2048),
                     IDESC_DQ, kk > 0 ? 1u : 0u);
        tc_commit(&dq_full[s]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_f16(tmem_base + T_DK, desc_advance(sds_k, kk * 32), desc_advance(sq, kk * 2048), IDESC_KV,
                     (n > 0 || kk > 0) ? 1u : 0u);
        // the stage's readers are done: S^T_n and dP^T_n (the score issuer's)
        // were read by the row group before p_full and ds_full, dV_n and dK_n
        // are this thread's
        tc_commit(&ds_empty[s]);
        tc_commit(&in_empty[q]);
        if (n + 1 == nsteps) tc_commit(&acc_full);
      }
      __syncwarp();
    }
    if (elect_one()) tc_commit(&drain_b);
    __syncwarp();
    int no_abort = 0;
    mbar_wait(&drain_b, 0, &no_abort, p.status, STATUS_TIMEOUT, FDRAIN_NS);
  } else if (warp < 2 + 2 * GROUP_WARPS) {
    // ------------------------------------------------------------ row groups
    const int grp = (warp - 2) / GROUP_WARPS;  // steps n with n & 1 == grp, slot grp
    const int q = warp & 3;
    const int r = q * 32 + lane;  // key row of P^T, dS^T, dK, dV
    const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16);
    const int key = j * BKB + r;
    const uint32_t t_s = tl + T_S + grp * BQB, t_dp = tl + T_PQ + grp * BQB;
    uint8_t* rowp = smem + B_SDS + grp * KT_BYTES + r * 128;
    int ok = 1;
    for (int n = grp; n < nsteps; n += 2) {
      const int q3 = n % QST;
      const uint32_t par = (uint32_t)((n >> 1) & 1);
      const int i = step_i(n);
      if (!(ok = wait_all(&in_full[q3], (n / QST) & 1))) break;
      if (!(ok = wait_all(&s_full[grp], par))) break;
      tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(smem + B_SLD + q3 * 256);
      {
        // P^T row (bf16 pairs) over the first 32 columns of the scores, read
        // in two 32-column halves; the half written (columns 0..15, then
        // 16..31) has been read already
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_s + 32 * hh, v);
          tmem_ld_wait();
          float pr[32];
#pragma unroll
          for (int c = 0; c < 32; ++c)
            pr[c] = ex2_fast(fmaf(__uint_as_float(v[c]), p.scale_log2, -lse2[32 * hh + c]));
          if (i < i0 + 2) {  // the two query blocks that cross the diagonal
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (i * BQB + 32 * hh + c < key) pr[c] = 0.0f;
          }
          uint32_t w[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) w[c >> 1] = pack_bf16x2(pr[c], pr[c + 1]);
          tmem_st_32x32b_x16(t_s + 16 * hh, w);
          tmem_st_wait();
        }
      }
      tc_fence_before();
      arrive(&p_full[grp]);
      // D of this step's 64 queries, from global memory (every lane reads the
      // same values); the loads are in flight while dP^T is awaited
      float dsum[64];
      {
        const float4* d4 = reinterpret_cast<const float4*>(
            p.dsum + ((size_t)(b * p.nq + step_h(n))) * p.S + (size_t)i * BQB);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float4 t4 = __ldg(d4 + k);
          dsum[4 * k] = t4.x;
          dsum[4 * k + 1] = t4.y;
          dsum[4 * k + 2] = t4.z;
          dsum[4 * k + 3] = t4.w;
        }
      }
      if (!(ok = wait_all(&dp_full[grp], par))) break;
      // dS^T row into the group's slot, once step n - 2's products have read it
      if (!(ok = wait_all(&ds_empty[grp], par ^ 1u))) break;
      tc_fence_after();
      // dS = P (dP - D) / sqrt(d) in four 16-column quarters, with P the
      // bf16 values the dV product uses, read back from tensor memory; each
      // quarter is packed straight into its two 16-byte chunks of the
      // swizzled row
      const uint64_t sc2 = f2_pack(p.scale, p.scale);
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        uint32_t v[16], pk[8];
        tmem_ld_32x32b_x16(t_dp + 16 * hh, v);
        tmem_ld_32x32b_x8(t_s + 8 * hh, pk);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; c += 2) {
          const int cc = 16 * hh + c;
          const uint32_t pw = pk[c >> 1];
          const uint64_t d2 = f2_add(f2_pack(__uint_as_float(v[c]), __uint_as_float(v[c + 1])),
                                     f2_pack(-dsum[cc], -dsum[cc + 1]));
          const uint64_t p2 = f2_pack(__uint_as_float(pw << 16), __uint_as_float(pw & 0xffff0000u));
          float d0, d1;
          f2_unpack(f2_mul(f2_mul(p2, sc2), d2), d0, d1);
          v[c >> 1] = pack_bf16x2(d0, d1);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k)
          *reinterpret_cast<uint4*>(rowp + (((2 * hh + k) ^ (r & 7)) << 4)) =
              make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
      }
      // the dP^T reads are complete (waited above); dQ^T_n may overwrite them
      tc_fence_before();
      fence_proxy_async_smem();
      arrive(&ds_full[grp]);
      arrive(&in_empty[q3]);
    }
    if (ok && (ok = wait_all(&acc_full, 0))) {
      tc_fence_after();
      // group 0: the dV_j row, group 1: the dK_j row (bf16) in the group's V / K columns of dqkv
      __nv_bfloat16* dst = p.dqkv + (size_t)(b * p.S + key) * p.ld_dqkv + (grp ? p.k_col0 : p.v_col0) + g * FD;
      const uint32_t col = grp ? T_DK : T_DV;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tl + col + 32 * c, v);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          reinterpret_cast<uint4*>(dst + 32 * c)[k] =
              make_uint4(pack_bf16x2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1])),
                         pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
                         pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
                         pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
      }
    }
  } else {
    // --------------------------------------------------------- dQ epilogue
    // Thread (warp quarter q, lane) owns head-dim column d = 32 q + lane of
    // dQ^T: it reads its 64 query values out of tensor memory, frees the
    // slot, and adds them into the f32 accumulator with one reduction per
    // query (each warp instruction covers 32 consecutive floats of a row).
    const int q = warp & 3;
    const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16);
    for (int m = 0; m < nsteps; ++m) {
      const int s = m & 1;
      if (!wait_all(&dq_full[s], (m >> 1) & 1)) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld_32x32b_x32(tl + T_PQ + s * BQB, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_32x32b_x32(tl + T_PQ + s * BQB + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_wait();
      tc_fence_before();
      arrive(&dq_empty[s]);
      float* dst = p.dq_acc + (size_t)(b * p.S + step_i(m) * BQB) * p.ld_dq + step_h(m) * FD + q * 32 + lane;
#pragma unroll
      for (int c = 0; c < 64; ++c) red_add_f32(dst + (size_t)c * p.ld_dq, __uint_as_float(v[c]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, FCOLS);
  }
}

// D[(b nq + h) S + q] = sum_c dO[b S + q, h d + c] O[b S + q, h d + c], and
// the f32 dQ accumulator cleared alongside.  d = 128: a block walks whole
// token rows (nq d contiguous elements); each half-warp takes one head of
// the row, a lane 8 elements (16-byte loads), and sums the products with
// four shuffles.  Two chunks per thread per pass keep four loads in flight.
__global__ void __launch_bounds__(256) flash_bwd_prep_kernel(const __nv_bfloat16* __restrict__ dz,
                                                             const __nv_bfloat16* __restrict__ z,
                                                             float* __restrict__ dsum, float* __restrict__ dq_acc,
                                                             int64_t N, int S, int nq) {
  const int chunks = nq * 16;  // 8-element chunks per token row
  for (int64_t tok = blockIdx.x; tok < N; tok += gridDim.x) {
    const int64_t row0 = tok * (int64_t)chunks * 8;
    const int b = (int)(tok / S), qi = (int)(tok % S);
    // the loop runs warp-uniformly (the shuffles need every lane); chunks is a
    // multiple of 16, so each half-warp is wholly in or out of range
    for (int base = threadIdx.x & ~31; base < chunks; base += 2 * blockDim.x) {
      const int k0 = base + (threadIdx.x & 31), k1 = k0 + blockDim.x;
      const bool has0 = k0 < chunks, has1 = k1 < chunks;
      float a0[8], o0[8], a1[8], o1[8];
      if (has0) {
        Vec<__nv_bfloat16>::load(dz + row0 + 8 * k0, a0);
        Vec<__nv_bfloat16>::load(z + row0 + 8 * k0, o0);
      }
      if (has1) {
        Vec<__nv_bfloat16>::load(dz + row0 + 8 * k1, a1);
        Vec<__nv_bfloat16>::load(z + row0 + 8 * k1, o1);
      }
      const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      float s0 = 0.0f, s1 = 0.0f;
      if (has0) {
        store4(dq_acc + row0 + 8 * k0, zero);
        store4(dq_acc + row0 + 8 * k0 + 4, zero);
#pragma unroll
        for (int i = 0; i < 8; ++i) s0 = fmaf(a0[i], o0[i], s0);
      }
      if (has1) {
        store4(dq_acc + row0 + 8 * k1, zero);
        store4(dq_acc + row0 + 8 * k1 + 4, zero);
#pragma unroll
        for (int i = 0; i < 8; ++i) s1 = fmaf(a1[i], o1[i], s1);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      }
      if (has0 && (k0 & 15) == 0) dsum[((int64_t)b * nq + (k0 >> 4)) * S + qi] = s0;
      if (has1 && (k1 & 15) == 0) dsum[((int64_t)b * nq + (k1 >> 4)) * S + qi] = s1;
    }
  }
}

// dqkv[:, 0 : Zc] = bf16(dQ accumulator): a block walks whole rows, a
// thread 8 floats (two 16-byte loads, one 16-byte store), two chunks per pass.
__global__ void __launch_bounds__(256) flash_dq_cast_kernel(const float* __restrict__ dq_acc,
                                                            __nv_bfloat16* __restrict__ dqkv, int64_t N, int64_t Zc,
                                                            int64_t ld) {
  const int chunks = (int)(Zc / 8);
  for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
    const float* src = dq_acc + row * Zc;
    __nv_bfloat16* dst = dqkv + row * ld;
    for (int k0 = threadIdx.x; k0 < chunks; k0 += 2 * blockDim.x) {
      const int k1 = k0 + blockDim.x;
      float v0[8], v1[8];
      load4(src + 8 * k0, v0);
      load4(src + 8 * k0 + 4, v0 + 4);
      if (k1 < chunks) {
        load4(src + 8 * k1, v1);
        load4(src + 8 * k1 + 4, v1 + 4);
      }
      Vec<__nv_bfloat16>::store(dst + 8 * k0, v0);
      if (k1 < chunks) Vec<__nv_bfloat16>::store(dst + 8 * k1, v1);
    }
  }
}

}  // namespace

cudaError_t launch_flash_attn_fwd(const void* qkv, int batch, int S, int nq, int nkv, int d, void* z, float* lse2,
                                  uint32_t* status, cudaStream_t st) {
  if (d != FD || S % FB != 0 || nq % nkv != 0) return cudaErrorInvalidValue;
  const int64_t N = (int64_t)batch * S;
  const int64_t W = (int64_t)(nq + 2 * nkv) * d;
  CUtensorMap map_qkv, map_z;
  if (!make_map(&map_qkv, qkv, (uint64_t)W, (uint64_t)N, (uint64_t)W, FB) ||
      !make_out_map(&map_z, z, false, (uint64_t)nq * d, (uint64_t)N, (uint64_t)nq * d))
    return cudaErrorInvalidValue;
  static bool attr_done = false;
  if (!attr_done) {
    const cudaError_t e = cudaFuncSetAttribute(flash_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FSMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  FaParams p{};
  p.S = S;
  p.nq = nq;
  p.nkv = nkv;
  p.hpg = nq / nkv;
  p.nqblk = (S + 2 * FB - 1) / (2 * FB);
  p.k_col0 = nq * d;
  p.v_col0 = (nq + nkv) * d;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)d);
  p.lse2 = lse2;
  p.status = status;
  const unsigned blocks = (unsigned)((int64_t)batch * nq * p.nqblk);
  flash_fwd_kernel<<<blocks, FTHREADS, FSMEM, st>>>(map_qkv, map_z, p);
  return cudaGetLastError();
}

cudaError_t launch_flash_bwd_prep(const void* dz, const void* z, float* dsum, float* dq_acc, int batch, int S, int nq,
                                  int d, int num_sms, cudaStream_t st) {
  if (d != FD) return cudaErrorInvalidValue;
  const int64_t N = (int64_t)batch * S;
  if (N <= 0 || nq <= 0) return cudaSuccess;
  const int64_t blocks = N < 8LL * num_sms ? N : 8LL * num_sms;
  flash_bwd_prep_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(dz),
                                                          static_cast<const __nv_bfloat16*>(z), dsum, dq_acc, N, S,
                                                          nq);
  return cudaGetLastError();
}

cudaError_t launch_flash_attn_bwd(const void* qkv, const void* dz, const float* lse2, const float* dsum, float* dq_acc,
                                  void* dqkv, int batch, int S, int nq, int nkv, int d, uint32_t* status,
                                  cudaStream_t st) {
  if (d != FD || S % BKB != 0 || nq % nkv != 0) return cudaErrorInvalidValue;
  const int64_t N = (int64_t)batch * S;
  const int64_t W = (int64_t)(nq + 2 * nkv) * d, Zc = (int64_t)nq * d;
  CUtensorMap map_kv, map_q, map_do;
  if (!make_map(&map_kv, qkv, (uint64_t)W, (uint64_t)N, (uint64_t)W, BKB) ||
      !make_map(&map_q, qkv, (uint64_t)W, (uint64_t)N, (uint64_t)W, BQB) ||
      !make_map(&map_do, dz, (uint64_t)Zc, (uint64_t)N, (uint64_t)Zc, BQB))
    return cudaErrorInvalidValue;
  static bool attr_done = false;
  if (!attr_done) {
    const cudaError_t e = cudaFuncSetAttribute(flash_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BSMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  FbParams p{};
  p.S = S;
  p.nq = nq;
  p.nkv = nkv;
  p.hpg = nq / nkv;
  p.q64 = S / BQB;
  p.k_col0 = nq * d;
  p.v_col0 = (nq + nkv) * d;
  p.scale = 1.0f / sqrtf((float)d);
  p.scale_log2 = 1.4426950408889634f * p.scale;
  p.lse2 = lse2;
  p.dsum = dsum;
  p.dqkv = static_cast<__nv_bfloat16*>(dqkv);
  p.ld_dqkv = W;
  p.dq_acc = dq_acc;
  p.ld_dq = Zc;
  p.status = status;
  const unsigned blocks = (unsigned)((int64_t)(S / BKB) * batch * nkv);
  flash_bwd_kernel<<<blocks, BTHREADS, BSMEM, st>>>(map_kv, map_q, map_do, p, batch);
  return cudaGetLastError();
}

cudaError_t launch_flash_dq_cast(const float* dq_acc, void* dqkv, int64_t N, int64_t Zc, int64_t ld, int num_sms,
                                 cudaStream_t st) {
  if (Zc % 8 != 0 || ld % 8 != 0 || Zc / 8 > (1LL << 30)) return cudaErrorInvalidValue;
  if (N <= 0 || Zc <= 0) return cudaSuccess;
  const int64_t blocks = N < 8LL * num_sms ? N : 8LL * num_sms;
  flash_dq_cast_kernel<<<(unsigned)blocks, 256, 0, st>>>(dq_acc, static_cast<__nv_bfloat16*>(dqkv), N, Zc, ld);
  return cudaGetLastError();
}

}  // namespace tpmlp
