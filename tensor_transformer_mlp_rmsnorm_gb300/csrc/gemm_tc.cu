// Persistent, warp-specialised bf16 GEMM on the sm_103a tensor cores.
//
//   warp 0      : TMA producer -- one thread streams A and B tiles (128-byte
//                 swizzle) into a shared-memory ring.
//   warp 1      : owns tensor memory (512 columns = two 128x256 f32
//                 accumulators); one thread issues tcgen05.mma, committing
//                 each stage back to the producer and each finished tile to
//                 the epilogue.
//   warps 2..5  : epilogue -- tcgen05.ld the accumulator (lane = row), apply
//                 the fused element-wise step, store to global memory.  The
//                 two accumulators let tile i's epilogue overlap tile i+1's
//                 main loop.
//
// Two tile shapes share the code:
//   * CTA pair (cluster of 2, cta_group::2): a 256x256 tile per pair.  Each
//     CTA loads 128 rows of A and 128 of the 256 B columns per 64-deep stage
//     (32 KB, 6 stages), the even CTA issues M=256 MMAs for both, and each
//     CTA's tensor memory holds its 128 rows.  Per SM this halves the B bytes
//     per flop and leaves room for a deeper ring -- the default.
//   * single CTA (cta_group::1): a 128x256 tile, 4 stages of 48 KB; used when
//     the problem has a single 128-row block.
//
// The contraction runs over up to two K segments in order.  For the
// row-parallel down projection the K axis is the FFN axis, so shard s's
// partial product A_s W_d,s^T is accumulated in shard order 0..t-1 into the
// same tensor-memory tile: that *is* the g all-reduce of the page "Megatron
// tensor-parallel MLP" ("Split the contraction"), done on-chip.  The normed-
// input gradient GEMM likewise sums every shard's dN_s (the f all-reduce,
// "Put the other collective in backward").  Restricting the segments to one
// shard reproduces the broken variants of "Remove each collective".
//
// Every wait is bounded (1 s); a wait that gives up raises a CTA-wide abort
// flag and a bit in the device status word, in-flight TMA copies and MMAs are
// drained, tensor memory is released and the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include <atomic>

#include "epilogue.cuh"
#include "ptx_sm103.cuh"
#include "tma_maps.cuh"
#include "tpmlp_internal.h"

namespace tpmlp {
namespace {

constexpr int BM = 128;  // accumulator rows per CTA (TMEM lanes)
constexpr int BN = 256;  // accumulator columns (MMA N)
constexpr int BK = 64;   // K depth of one stage in bf16 elements (one 128-byte swizzle row)
constexpr int UMMA_K = 16;
// E4M3 operands: the same 128-byte rows hold 128 elements, and one MMA takes K = 32.
template <bool F8>
struct KDepth {
  static constexpr int STAGE = F8 ? 128 : BK;  // elements per stage row
  static constexpr int MMA = F8 ? 32 : UMMA_K;
};
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;   // 1 s per wait
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;   // 0.2 s for draining after an abort
constexpr uint64_t PEER_DRAIN_NS = 5000000ull;      // 5 ms: a CTA-pair peer's loads land long before this
constexpr uint64_t FORCED_LIMIT_NS = 2000000ull;    // 2 ms for the forced-timeout debug wait
constexpr int SPLIT_MIN_KBLOCKS = 64;               // shortest contraction whose tail is split

// Epilogues that read global inputs (the residual x, or G and U, or Z) bring
// them into shared memory with TMA as well.
template <int EPI>
__host__ __device__ constexpr bool epi_has_in() {
  return EPI == EPI_DOWN_RESID || EPI == EPI_DGRAD_SWIGLU || EPI == EPI_DGRAD_GELU;
}

constexpr int NUM_THREADS = 192;

// Whether the epilogue warps stage with single (rather than double) input
// and output buffers.  The SwiGLU backward's main loop contracts over only
// H with an MN-major W_down: it needs the sixth ring stage more than its
// epilogue needs double buffers (measured: 4% faster).
template <int EPI>
__host__ __device__ constexpr bool epi_single() {
  return EPI == EPI_DGRAD_SWIGLU;
}

template <bool PAIR, bool HAS_IN, bool SB = false>
struct TileCfg {
  // Operand ring depth: double-buffered staging of epilogue inputs takes one
  // stage's room.
  static constexpr int STAGES = PAIR ? (HAS_IN && !SB ? 5 : 6) : (HAS_IN ? 3 : 4);
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // B columns held by this CTA per stage
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // Epilogue staging per epilogue warp: outputs in two 4 KB buffers used
  // alternately (each up to two 32x32 bf16 tiles or one 32x32 f32 tile) or,
  // for the three-output gate/up epilogue, one 6 KB buffer; inputs in two
  // 4 KB buffers (up to two 32x32 bf16 tiles each).
  // With single buffers each warp has one 4 KB buffer of each kind.
  static constexpr int EPI_OUT_BYTES = SB ? 4096 : 8192;
  static constexpr int EPI_IN_BYTES = HAS_IN ? (SB ? 4096 : 8192) : 0;
  static constexpr int EPI_WARP_BYTES = EPI_OUT_BYTES + EPI_IN_BYTES;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 4 * EPI_WARP_BYTES + 1024;  // + alignment
  static constexpr int TILE_M = PAIR ? 2 * BM : BM;  // output rows per tile (per pair)
  static constexpr uint32_t TX_BYTES = PAIR ? 2 * STAGE_BYTES : STAGE_BYTES;
  static constexpr uint32_t EPI_ARRIVALS = PAIR ? 8 : 4;  // one per epilogue warp, both CTAs
};

struct TcParams {
  int M, N;
  int num_m_blk, num_n_blk, num_tiles, group_m;
  int kb[4];  // two k-block segments [kb0, kb1), [kb2, kb3)
  int paired;
  int pair_off;
  EpiParams ep;
  uint32_t* status;
  int force_timeout;
  int a3d, b3d;  // MN-major operand loaded as one 3-D box per stage
  const float* deq_a;  // FP8: inverse operand scales
  const float* deq_b;
  int tiles_per_batch;  // num_m_blk * num_n_blk
  BatchDesc batch;
  int causal;  // CAUSAL_* restriction for attention problems
  // Work units: tiles [0, split_first) whole, then `split` K parts of each
  // tile in [split_first, num_tiles); num_units in all.  kb_total is the
  // k-blocks of one tile's contraction (both segments).
  int num_units, split_first, split, kb_total;
  float* scratch;      // partial accumulators of the parts after the first
  uint32_t* counters;  // arrival flags: per split tile, CTA of the pair, epilogue warp and later part
  size_t scratch_bytes;
  int counter_words;
  uint32_t epoch;  // value a later part's flag takes in this launch (never 0, unique per launch)
};

// One work unit: a tile, which of its K parts, and the range [vb, ve) of
// k-blocks it contracts, counted over the tile's segments in order.
struct Unit {
  int tile, part, vb, ve;
};
__device__ __forceinline__ Unit unit_of(const TcParams& p, int u) {
  Unit w;
  if (u < p.split_first) {
    w.tile = u;
    w.part = 0;
    w.vb = 0;
    w.ve = 0x7fffffff;
    return w;
  }
  const int i = u - p.split_first;
  w.tile = p.split_first + i / p.split;
  w.part = i % p.split;
  w.vb = (int)((int64_t)w.part * p.kb_total / p.split);
  w.ve = (int)((int64_t)(w.part + 1) * p.kb_total / p.split);
  return w;
}

// Bounded wait until *flag == epoch (acquire at GPU scope).  On a timeout it
// raises the CTA's abort flag and ORs `code` into the status word.
__device__ __forceinline__ bool wait_flag(const uint32_t* flag, uint32_t epoch, volatile int* abort,
                                          uint32_t* status, uint32_t code, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v == epoch) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort = 1;
      atomicOr(status, code);
      return false;
    }
    __nanosleep(256);
  }
}

// Causal restrictions of attention problems (M = queries or keys of one
// sequence): tiles wholly above the diagonal skipped (score GEMMs), or the
// contraction over keys cut at the tile's last query (P V, dS K), or over
// queries started at the tile's first key (P^T dZ, dS^T Q).
__device__ __forceinline__ bool tile_active(const TcParams& p, int mb, int nb, int tile_m) {
  return p.causal != CAUSAL_SKIP_UPPER || nb * BN <= (mb + 1) * tile_m - 1;
}
__device__ __forceinline__ void seg_range(const TcParams& p, int mb, int seg, int tile_m, int bke, int& lo, int& hi) {
  lo = p.kb[2 * seg];
  hi = p.kb[2 * seg + 1];
  if (p.causal == CAUSAL_K_UPTO) hi = min(hi, ((mb + 1) * tile_m + bke - 1) / bke);
  if (p.causal == CAUSAL_K_FROM) lo = max(lo, (mb * tile_m) / bke);
}

// The k-blocks of segment `seg` of tile row block mb that unit `un` contracts:
// [lo, hi), with v0 the count of the tile's k-blocks in earlier segments
// (advanced past this segment on return).
__device__ __forceinline__ void unit_seg_range(const TcParams& p, const Unit& un, int mb, int seg, int tile_m, int bke,
                                               int& v0, int& lo, int& hi) {
  int a, b;
  seg_range(p, mb, seg, tile_m, bke, a, b);
  const int n = b > a ? b - a : 0;
  lo = a + max(0, min(n, un.vb - v0));
  hi = a + max(0, min(n, un.ve - v0));
  v0 += n;
}

// Coordinate shift of one operand for batch index z.
struct Shift {
  int col, row;
};
__device__ __forceinline__ Shift batch_shift(const BatchDesc& b, const BatchOffsets& o, int z) {
  const int z2 = z % b.dims[2];
  const int z1 = (z / b.dims[2]) % b.dims[1];
  const int z0 = z / (b.dims[2] * b.dims[1]);
  return Shift{(int)(o.col[0] + z0 * o.col[1] + z1 * o.col[2] + z2 * o.col[3]),
               (int)(o.row[0] + z0 * o.row[1] + z1 * o.row[2] + z2 * o.row[3])};
}

// Tile -> (batch index, row block, column block); the raster runs inside a batch.
__device__ __forceinline__ void tile_coords(const TcParams& p, int tile, int& mb, int& nb, int& z) {
  z = tile / p.tiles_per_batch;
  tile -= z * p.tiles_per_batch;
  const int per_group = p.group_m * p.num_n_blk;
  const int g = tile / per_group;
  const int first_m = g * p.group_m;
  const int gm = min(p.num_m_blk - first_m, p.group_m);
  const int r = tile - g * per_group;
  mb = first_m + r % gm;
  nb = r / gm;
}

__device__ __forceinline__ uint4 pack8_bf16(const float* f) {
  uint4 r;
  __nv_bfloat162 h;
  h = __floats2bfloat162_rn(f[0], f[1]);
  r.x = *reinterpret_cast<uint32_t*>(&h);
  h = __floats2bfloat162_rn(f[2], f[3]);
  r.y = *reinterpret_cast<uint32_t*>(&h);
  h = __floats2bfloat162_rn(f[4], f[5]);
  r.z = *reinterpret_cast<uint32_t*>(&h);
  h = __floats2bfloat162_rn(f[6], f[7]);
  r.w = *reinterpret_cast<uint32_t*>(&h);
  return r;
}

__device__ __forceinline__ void unpack8_bf16(uint4 v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    float2 t = __bfloat1622float2(h);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// Partial accumulators of a split tile.  A warp's 32 rows x BN columns of one
// later K part are one 32 KB block, laid out lane-minor so that every warp
// access covers 512 contiguous bytes: float4 number (cc * 8 + k) * 32 + lane
// holds columns cc * 32 + 4 k .. + 3 of the lane's row.  The same thread
// (same CTA rank, warp quarter and lane) writes a block and reads it back.
__device__ __forceinline__ void dump32_to(float4* blk, int cc, int lane, const uint32_t (&r)[32]) {
#pragma unroll
  for (int k = 0; k < 8; ++k)
    __stcg(blk + (cc * 8 + k) * 32 + lane, make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                                       __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3])));
}

// r += the later parts' columns cc * 32 .. + 31 of this lane's row, added in
// part order (read past L1: other CTAs wrote them during this launch).  Two
// parts' loads are in flight at a time.
__device__ __forceinline__ void add_parts(uint32_t (&r)[32], const float4* blk1, size_t part_stride4, int split,
                                          int cc, int lane) {
#pragma unroll 1
  for (int p0 = 1; p0 < split; p0 += 2) {
    float4 v[2][8];
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (p0 + j < split) {
        const float4* b = blk1 + (size_t)(p0 + j - 1) * part_stride4 + cc * 256 + lane;
#pragma unroll
        for (int k = 0; k < 8; ++k) v[j][k] = __ldcg(b + k * 32);
      }
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (p0 + j < split) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          r[4 * k] = __float_as_uint(__uint_as_float(r[4 * k]) + v[j][k].x);
          r[4 * k + 1] = __float_as_uint(__uint_as_float(r[4 * k + 1]) + v[j][k].y);
          r[4 * k + 2] = __float_as_uint(__uint_as_float(r[4 * k + 2]) + v[j][k].z);
          r[4 * k + 3] = __float_as_uint(__uint_as_float(r[4 * k + 3]) + v[j][k].w);
        }
      }
  }
}

// The SGD update of 32 consecutive parameters of one row (nv of them valid),
// where their gradient g is produced, in two halves so that the masters'
// loads are issued a chunk ahead: sgd_load reads the fp32 masters into
// registers; sgd_apply forms the separate update kernel's
// master = fmaf(-lr, g, master), stores it, and stores its bf16 rounding
// (nearest even) into the parameter copy.  Loops are fully unrolled so that
// the chunk stays in registers.
__device__ __forceinline__ void sgd_load(const EpiParams& e, int row, int col, int nv, float (&v)[32]) {
  const float* m = e.sgd_master + (size_t)row * e.sgd_ld + col;
  if (nv >= 32) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 t = reinterpret_cast<const float4*>(m)[k];
      v[4 * k] = t.x;
      v[4 * k + 1] = t.y;
      v[4 * k + 2] = t.z;
      v[4 * k + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = i < nv ? m[i] : 0.0f;
  }
}
__device__ __forceinline__ void sgd_apply(const EpiParams& e, int row, int col, int nv, const float* g,
                                          float (&v)[32]) {
  float* m = e.sgd_master + (size_t)row * e.sgd_ld + col;
  __nv_bfloat16* w = e.sgd_w + (size_t)row * e.sgd_ld + col;
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = fmaf(-e.sgd_lr, g[i], v[i]);
  if (nv >= 32) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      reinterpret_cast<float4*>(m)[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
#pragma unroll
    for (int k = 0; k < 4; ++k) reinterpret_cast<uint4*>(w)[k] = pack8_bf16(v + 8 * k);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < nv) {
        m[i] = v[i];
        w[i] = __float2bfloat16_rn(v[i]);
      }
  }
}

// Raw bf16 inputs of one epilogue chunk (32 consecutive values of one row,
// two tensors at most), loaded ahead of the math that uses them.
struct EpiIn {
  uint4 a[4];
  uint4 b[4];
};

// 32 consecutive bf16 values starting at src, of which the first n are read
// (n <= 0: none); the rest are zero.
__device__ __forceinline__ void load32_raw(const __nv_bfloat16* src, int n, uint4 (&o)[4]) {
  if (n >= 32) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = s4[i];
    return;
  }
  const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src);
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t lo = 2 * i < n ? s16[2 * i] : 0u;
    const uint32_t hi = 2 * i + 1 < n ? s16[2 * i + 1] : 0u;
    w[i] = lo | (hi << 16);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

__device__ __forceinline__ void unpack32(const uint4 (&v)[4], float* f) {
#pragma unroll
  for (int i = 0; i < 4; ++i) unpack8_bf16(v[i], f + 8 * i);
}

// Load n (<= 32) consecutive bf16 values as floats; the rest read as 0.
__device__ __forceinline__ void load32_bf16_guard(const __nv_bfloat16* src, int n, float* f) {
  uint4 v[4];
  load32_raw(src, n, v);
  unpack32(v, f);
}

// Row r of a 32x32 bf16 input tile loaded by TMA with the 64-byte swizzle.
__device__ __forceinline__ void read_row_bf16(const uint8_t* tile, int r, uint4 (&o)[4]) {
  const uint8_t* rowp = tile + r * 64;
#pragma unroll
  for (int c = 0; c < 4; ++c) o[c] = *reinterpret_cast<const uint4*>(rowp + ((c ^ ((r >> 1) & 3)) << 4));
}

// Row r of a 32x32 staging tile in the layout the TMA store expects:
// bf16 rows are 64 bytes with the 64-byte swizzle (16-byte chunk c of row r
// at c ^ ((r >> 1) & 3)); f32 rows are 128 bytes with the 128-byte swizzle
// (chunk c at c ^ (r & 7)).  Both are free of shared-memory bank conflicts
// when the 32 lanes of a warp each write their own row.
__device__ __forceinline__ void stage_row_bf16(uint8_t* tile, int r, const float* v) {
  uint8_t* rowp = tile + r * 64;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(rowp + ((c ^ ((r >> 1) & 3)) << 4)) = pack8_bf16(v + 8 * c);
}

__device__ __forceinline__ void stage_row_f32(uint8_t* tile, int r, const float* v) {
  uint8_t* rowp = tile + r * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<float4*>(rowp + ((c ^ (r & 7)) << 4)) =
        make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

// Number of 32x32 output tiles the epilogue of each kind stores per chunk.
template <int EPI>
struct EpiOut {
  static constexpr int N = EPI == EPI_GATEUP_SWIGLU ? 3 : (EPI == EPI_FC1_GELU || EPI == EPI_DGRAD_SWIGLU) ? 2 : 1;
  static constexpr int NBUF = N == 3 ? 1 : 2;  // staging buffers per warp
};

// Epilogue of one thread's row for output columns [col, col+32): fused math
// on the accumulator values v (and u, the second half, for the paired
// layouts), results written into the warp's staging tiles (row r).  Inputs
// outside the matrix read as zero; the TMA store clips the outputs.
// Largest |o[i]| over the first n (<= 32 or more) columns.
__device__ __forceinline__ float max_abs32(const float* o, int n) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) m = i < n ? fmaxf(m, fabsf(o[i])) : m;
  return m;
}

// Returns, when `want_max`, the largest magnitude among the activation
// outputs of this row's valid columns (A; dG and dU; dZ), else 0.
template <int EPI>
__device__ __forceinline__ float epi_stage(const EpiParams& ep, int col, const float* v, const float* u,
                                           const EpiIn& in, uint8_t* st, int r, bool want_max) {
  typedef __nv_bfloat16 T;
  const int ncols = ep.N - col;  // valid columns of this chunk (may exceed 32)
  float o[32];
  float mx = 0.0f;
  if (EPI == EPI_GATEUP_SWIGLU) {
    stage_row_bf16(st, r, v);
    stage_row_bf16(st + 2048, r, u);
#pragma unroll
    for (int i = 0; i < 32; i += 2) swiglu_fwd_fast2(v[i], v[i + 1], u[i], u[i + 1], o[i], o[i + 1]);
    stage_row_bf16(st + 4096, r, o);
    if (want_max) mx = max_abs32(o, ncols);
  } else if (EPI == EPI_FC1_GELU) {
    float b[32];
    load32_bf16_guard(static_cast<const T*>(ep.vec) + col, ncols, b);
#pragma unroll
    for (int i = 0; i < 32; ++i) b[i] += v[i];
    stage_row_bf16(st, r, b);
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = gelu_fast(b[i]);
    stage_row_bf16(st + 2048, r, o);
    if (want_max) mx = max_abs32(o, ncols);
  } else if (EPI == EPI_DOWN_RESID) {
    float x[32], b[32];
    unpack32(in.a, x);
    load32_bf16_guard(static_cast<const T*>(ep.vec) + col, ncols, b);
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = x[i] + v[i] + b[i];
    stage_row_bf16(st, r, o);
  } else if (EPI == EPI_DGRAD_SWIGLU) {
    float g[32], uu[32];
    unpack32(in.a, g);
    unpack32(in.b, uu);
#pragma unroll
    for (int i = 0; i < 32; i += 2)
      swiglu_bwd_fast2(v[i], v[i + 1], g[i], g[i + 1], uu[i], uu[i + 1], o[i], o[i + 1], uu[i], uu[i + 1]);
    stage_row_bf16(st, r, o);
    stage_row_bf16(st + 2048, r, uu);
    if (want_max) mx = fmaxf(max_abs32(o, ncols), max_abs32(uu, ncols));
  } else if (EPI == EPI_DGRAD_GELU) {
    float z[32];
    unpack32(in.a, z);
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = v[i] * gelu_grad_fast(z[i]);
    stage_row_bf16(st, r, o);
    if (want_max) mx = max_abs32(o, ncols);
  } else if (EPI == EPI_STORE_BF16) {
    stage_row_bf16(st, r, v);
  } else {
    stage_row_f32(st, r, v);
  }
  return mx;
}

template <bool PAIR, bool A_MN, bool B_MN, int EPI, bool F8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_o0, const __grid_constant__ CUtensorMap map_o1,
                   const __grid_constant__ CUtensorMap map_o2, const __grid_constant__ CUtensorMap map_i0,
                   const __grid_constant__ CUtensorMap map_i1, const TcParams p) {
  constexpr bool HAS_IN = epi_has_in<EPI>();
  constexpr bool SB = epi_single<EPI>();
  using C = TileCfg<PAIR, HAS_IN, SB>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::STAGES];
  __shared__ __align__(8) uint64_t empty_bar[C::STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t never_bar;
  __shared__ __align__(8) uint64_t in_bar[4][2];  // epilogue input tiles, per warp and buffer
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  uint8_t* sE = smem + C::STAGES * C::STAGE_BYTES;  // epilogue staging
  volatile int* abort_flag = &abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int worker = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int num_workers = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  constexpr uint32_t IDESC = F8 ? idesc_e4m3_f32(C::TILE_M, BN) : idesc_bf16_f32(C::TILE_M, BN, A_MN, B_MN);
  static_assert(!F8 || (!A_MN && !B_MN), "E4M3 operands are K-major");

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], C::EPI_ARRIVALS);
    }
    mbar_init(&drain_bar, 1);
    mbar_init(&never_bar, 1);
    for (int w = 0; w < 4; ++w)
      for (int b = 0; b < 2; ++b) mbar_init(&in_bar[w][b], 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
    tma_prefetch_desc(&map_o0);
    if (HAS_IN) tma_prefetch_desc(&map_i0);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(&tmem_base_sh, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&tmem_base_sh, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer's barriers exist before anything targets them
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;

  if (p.force_timeout) {
    // Debug: a wait on a barrier nobody arrives on gives up and aborts the CTA.
    if (threadIdx.x == 0) mbar_wait(&never_bar, 0, abort_flag, p.status, STATUS_TIMEOUT, FORCED_LIMIT_NS);
    __syncthreads();
  }

  if (warp == 0) {
    if (lane == 0 && !*abort_flag) {
      // ------------------------------------------------------------ producer
      uint32_t stage = 0, phase = 0;
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      for (int u = worker; ok && u < p.num_units; u += num_workers) {
        const Unit un = unit_of(p, u);
        int mb, nb, z;
        tile_coords(p, un.tile, mb, nb, z);
        if (!tile_active(p, mb, nb, C::TILE_M)) continue;
        const Shift sa = batch_shift(p.batch, p.batch.a, z), sbt = batch_shift(p.batch, p.batch.b, z);
        const int m0 = mb * C::TILE_M + (int)rank * BM + (A_MN ? sa.col : sa.row);
        int brow0, brow1;  // first B row (K-major) / column (MN-major) of each 128-wide half
        if (p.paired) {
          brow0 = nb * (BN / 2);
          brow1 = p.pair_off + nb * (BN / 2);
        } else {
          brow0 = nb * BN;
          brow1 = nb * BN + BN / 2;
        }
        if (PAIR) brow0 = rank ? brow1 : brow0;  // each CTA of the pair holds one half
        brow0 += B_MN ? sbt.col : sbt.row;
        brow1 += B_MN ? sbt.col : sbt.row;
        int v0 = 0;
        for (int seg = 0; ok && seg < 2; ++seg) {
          int kb_lo, kb_hi;
          unit_seg_range(p, un, mb, seg, C::TILE_M, KDepth<F8>::STAGE, v0, kb_lo, kb_hi);
          for (int kb = kb_lo; kb < kb_hi; ++kb) {
            if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(&full_bar[stage], C::TX_BYTES);
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
            const int ka = kb * KDepth<F8>::STAGE + (A_MN ? sa.row : sa.col);  // A's K coordinate
            const int k0 = kb * KDepth<F8>::STAGE + (B_MN ? sbt.row : sbt.col);  // B's K coordinate
            uint8_t* a_dst = sA + stage * C::A_BYTES;
            uint8_t* b_dst = sB + stage * C::B_BYTES;
            if (PAIR) {
              const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);  // the leader's barrier
              if (!A_MN) {
                tma_load_2d_pair(a_dst, &map_a, fb, ka, m0);
              } else if (p.a3d) {
                tma_load_3d_pair(a_dst, &map_a, fb, 0, ka, m0 >> 6);
              } else {
                tma_load_2d_pair(a_dst, &map_a, fb, m0, ka);
                tma_load_2d_pair(a_dst + 8192, &map_a, fb, m0 + 64, ka);
              }
              if (!B_MN) {
                tma_load_2d_pair(b_dst, &map_b, fb, k0, brow0);
              } else if (p.b3d) {
                tma_load_3d_pair(b_dst, &map_b, fb, 0, k0, brow0 >> 6);
              } else {
                tma_load_2d_pair(b_dst, &map_b, fb, brow0, k0);
                tma_load_2d_pair(b_dst + 8192, &map_b, fb, brow0 + 64, k0);
              }
            } else {
              if (!A_MN) {
                tma_load_2d(a_dst, &map_a, &full_bar[stage], ka, m0);
              } else if (p.a3d) {
                tma_load_3d(a_dst, &map_a, &full_bar[stage], 0, ka, m0 >> 6);
              } else {
                tma_load_2d(a_dst, &map_a, &full_bar[stage], m0, ka);
                tma_load_2d(a_dst + 8192, &map_a, &full_bar[stage], m0 + 64, ka);
              }
              if (!B_MN) {
                tma_load_2d(b_dst, &map_b, &full_bar[stage], k0, brow0);
                tma_load_2d(b_dst + C::B_BYTES / 2, &map_b, &full_bar[stage], k0, brow1);
              } else if (p.b3d) {
                tma_load_3d(b_dst, &map_b, &full_bar[stage], 0, k0, brow0 >> 6);
              } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  tma_load_2d(b_dst + j * 8192, &map_b, &full_bar[stage], brow0 + 64 * j, k0);
              }
            }
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok || *abort_flag) {
        // Let the copies this CTA started land before it may exit.  The
        // leader sees them (and the peer's) complete on its stage barriers;
        // the peer waits until its stages are consumed or a short time passes.
        int no_abort = 0;
        for (int s = 0; s < C::STAGES; ++s) {
          if (!(armed & (1u << s))) continue;
          const uint32_t par = (armed_par >> s) & 1u;
          if (leader)
            mbar_wait(&full_bar[s], par, &no_abort, p.status, STATUS_TIMEOUT, DRAIN_LIMIT_NS);
          else
            mbar_wait(&empty_bar[s], par, &no_abort, p.status, 0u, PEER_DRAIN_NS);
        }
      }
    }
  } else if (warp == 1) {
    if (leader) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs this loop in warp-uniform control flow (waits are
      // folded with __all_sync) and one elected lane issues the MMAs: that
      // keeps the descriptors in uniform registers and the issue cost of a
      // tcgen05.mma well below the 128 cycles it keeps the tensor core busy.
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      int ok = !*abort_flag;
      for (int u = worker; ok && u < p.num_units; u += num_workers) {
        const Unit un = unit_of(p, u);
        int mb, nb, z;
        tile_coords(p, un.tile, mb, nb, z);
        if (!tile_active(p, mb, nb, C::TILE_M)) continue;
        ok = __all_sync(0xffffffffu, mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort_flag, p.status,
                                               STATUS_TIMEOUT, WAIT_LIMIT_NS));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        uint32_t accumulate = 0;
        int v0 = 0;
        for (int seg = 0; ok && seg < 2; ++seg) {
          int kb_lo, kb_hi;
          unit_seg_range(p, un, mb, seg, C::TILE_M, KDepth<F8>::STAGE, v0, kb_lo, kb_hi);
          for (int kb = kb_lo; kb < kb_hi; ++kb) {
            ok = __all_sync(0xffffffffu, mbar_wait(&full_bar[stage], phase, abort_flag, p.status, STATUS_TIMEOUT,
                                                   WAIT_LIMIT_NS));
            if (!ok) break;
            tc_fence_after();
            const uint32_t a_base = smem_u32(sA + stage * C::A_BYTES);
            const uint32_t b_base = smem_u32(sB + stage * C::B_BYTES);
            if (elect_one()) {
#pragma unroll
              for (int k = 0; k < KDepth<F8>::STAGE / KDepth<F8>::MMA; ++k) {
                const uint64_t a_desc =
                    A_MN ? sw128_desc(a_base + k * 2048, 8192, 1024) : sw128_desc(a_base + k * 32, 16, 1024);
                const uint64_t b_desc =
                    B_MN ? sw128_desc(b_base + k * 2048, 8192, 1024) : sw128_desc(b_base + k * 32, 16, 1024);
                if (F8) {
                  if (PAIR)
                    tc_mma_f8_pair(d_tmem, a_desc, b_desc, IDESC, accumulate | (uint32_t)k);
                  else
                    tc_mma_f8(d_tmem, a_desc, b_desc, IDESC, accumulate | (uint32_t)k);
                } else {
                  if (PAIR)
                    tc_mma_f16_pair(d_tmem, a_desc, b_desc, IDESC, accumulate | (uint32_t)k);
                  else
                    tc_mma_f16(d_tmem, a_desc, b_desc, IDESC, accumulate | (uint32_t)k);
                }
              }
              // Free the stage for the producers once these MMAs complete.
              if (PAIR)
                tc_commit_pair(&empty_bar[stage], 0x3);
              else
                tc_commit(&empty_bar[stage]);
            }
            __syncwarp();
            accumulate = 1;
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) break;
        if (elect_one()) {
          if (PAIR)
            tc_commit_pair(&tfull_bar[acc], 0x3);
          else
            tc_commit(&tfull_bar[acc]);
        }
        __syncwarp();
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // No MMA may still be running when tensor memory is released.
      if (elect_one()) {
        if (PAIR)
          tc_commit_pair(&drain_bar, 0x3);
        else
          tc_commit(&drain_bar);
      }
      __syncwarp();
      int no_abort = 0;
      mbar_wait(&drain_bar, 0, &no_abort, p.status, STATUS_TIMEOUT, DRAIN_LIMIT_NS);
    } else if (lane == 0 && PAIR) {
      // Peer CTA: its tensor memory is written by the leader's MMAs; wait for
      // the leader's final commit (bounded, so an aborted leader cannot hold it).
      int no_abort = 0;
      mbar_wait(&drain_bar, 0, &no_abort, p.status, 0u, DRAIN_LIMIT_NS);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    // Warp ew handles every 32-column chunk of its TMEM lane quarter.  With
    // double buffers the next chunk's inputs are requested before the current
    // one is read; with single buffers once every lane has read the current
    // chunk's rows, and the output buffer is rewritten once the previous
    // store has read it.
    constexpr int NIN = SB ? 1 : 2;          // input buffers per warp
    constexpr int NOUT = SB ? 1 : EpiOut<EPI>::NBUF;  // output buffers per warp
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int ew = warp - 2;
    uint8_t* st = sE + ew * C::EPI_WARP_BYTES;  // output staging
    uint8_t* si = st + C::EPI_OUT_BYTES;        // input staging
    constexpr uint32_t IN_BYTES = EPI == EPI_DGRAD_SWIGLU ? 4096u : 2048u;
    uint32_t acc = 0, acc_phase = 0, n_stored = 0;
    uint32_t n_in = 0, n_used = 0, in_par = 0;  // input tiles issued / consumed, parity per buffer
    const float deq = F8 ? __ldg(p.deq_a) * __ldg(p.deq_b) : 1.0f;
    const bool want_max = p.ep.amax != nullptr;
    float amax_acc = 0.0f;
    // Input tiles of chunk [col, col+32) of this warp's 32 rows -> buffer n_in % NIN.
    // Every lane must have executed fence.proxy.async after its last generic
    // reads of that buffer before the refill is issued: with double buffers
    // the staging fence of the chunk that read it lies in between; with a
    // single buffer the chunk loop fences explicitly.
    auto issue_in = [&](int col, int row0) {
      if (!HAS_IN) return;
      const uint32_t b = NIN == 2 ? (n_in & 1u) : 0u;
      if (lane == 0) {
        mbar_arrive_expect_tx(&in_bar[ew][b], IN_BYTES);
        tma_load_2d(si + b * 4096, &map_i0, &in_bar[ew][b], col, row0);
        if (EPI == EPI_DGRAD_SWIGLU) tma_load_2d(si + b * 4096 + 2048, &map_i1, &in_bar[ew][b], col, row0);
      }
      ++n_in;
    };
    for (int u = worker; u < p.num_units; u += num_workers) {
      const Unit un = unit_of(p, u);
      int mb, nb, z;
      tile_coords(p, un.tile, mb, nb, z);
      if (!tile_active(p, mb, nb, C::TILE_M)) continue;
      const Shift so = batch_shift(p.batch, p.batch.o, z);  // output / input coordinate shift
      const int row0 = mb * C::TILE_M + (int)rank * BM + q * 32;  // first row of this warp
      constexpr int CHUNKS = EPI == EPI_GATEUP_SWIGLU ? BN / 2 / 32 : BN / 32;
      const int col_base = EPI == EPI_GATEUP_SWIGLU ? nb * (BN / 2) : nb * BN;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      // Split tiles: this warp's arrival flags (one per later part), and its
      // block in the first later part's scratch slot (one slot of TILE_M x BN
      // floats per later part, part_stride4 float4s apart).
      const bool split = un.tile >= p.split_first;
      const int ti = un.tile - p.split_first;
      uint32_t* flags = split ? p.counters + (((size_t)ti * 2 + rank) * 4 + q) * (p.split - 1) : nullptr;
      constexpr size_t part_stride4 = (size_t)C::TILE_M * BN / 4;
      float4* blk1 = split ? reinterpret_cast<float4*>(p.scratch) +
                                 ((size_t)ti * (p.split - 1) * C::TILE_M + (size_t)rank * BM + q * 32) * (BN / 4)
                           : nullptr;
      if (split && un.part > 0) {
        // A later K part: leave the raw accumulator rows of this warp in its
        // slot, then raise this warp's flag (release) for the first part.
        int ok = __all_sync(0xffffffffu, mbar_wait(&tfull_bar[acc], acc_phase, abort_flag, p.status,
                                                   STATUS_TIMEOUT, WAIT_LIMIT_NS));
        if (!ok) break;
        tc_fence_after();
        if (row0 < p.M) {
          float4* blk = blk1 + (size_t)(un.part - 1) * part_stride4;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tbase + c * 32, r);
            tmem_ld_wait();
            dump32_to(blk, c, lane, r);
          }
        }
        __threadfence();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flags + un.part - 1), "r"(p.epoch) : "memory");
          if (PAIR)
            mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
          else
            mbar_arrive(&tempty_bar[acc]);
        }
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
        continue;
      }
      // The first chunk's inputs are fetched while the tile's main loop runs,
      // each later chunk's while the previous one is computed.
      if (col_base < p.N && row0 < p.M) issue_in(col_base + so.col, row0 + so.row);
      // Weight gradients with the update applied here: the first chunk's
      // masters are read while the tile's main loop runs.
      const bool sgd = EPI == EPI_STORE_F32 && p.ep.sgd_master && row0 + lane < p.M && col_base < p.N;
      float sgdm[32];
      if (sgd) sgd_load(p.ep, row0 + lane, col_base, p.N - col_base, sgdm);
      int ok = mbar_wait(&tfull_bar[acc], acc_phase, abort_flag, p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      if (split) {
        // The first K part of a split tile: wait for the later parts of this
        // warp's rows.
        int wok = 1;
        if (lane == 0)
          for (int part = 1; part < p.split && wok; ++part)
            wok = wait_flag(flags + part - 1, p.epoch, abort_flag, p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
        ok = __all_sync(0xffffffffu, wok);
        if (!ok) break;
      }
      uint32_t r0[32], r1[32];
#pragma unroll 1
      for (int c = 0; c < CHUNKS; ++c) {
        const int col = col_base + c * 32;
        // Chunks wholly outside the output are skipped by the whole warp.
        if (col >= p.N || row0 >= p.M) break;
        const bool more = c + 1 < CHUNKS && col + 32 < p.N;
        if (NIN == 2 && more) issue_in(col + 32 + so.col, row0 + so.row);
        tmem_ld_32x32b_x32(tbase + c * 32, r0);
        if (EPI == EPI_GATEUP_SWIGLU) tmem_ld_32x32b_x32(tbase + BN / 2 + c * 32, r1);
        EpiIn in;
        if (HAS_IN) {
          const uint32_t b = NIN == 2 ? (n_used & 1u) : 0u;
          int iok = mbar_wait(&in_bar[ew][b], (in_par >> b) & 1u, abort_flag, p.status, STATUS_TIMEOUT,
                              WAIT_LIMIT_NS);
          iok = __all_sync(0xffffffffu, iok);
          if (!iok) {  // the load stays counted as in flight for the drain below
            ok = 0;
            break;
          }
          in_par ^= 1u << b;
          ++n_used;
          read_row_bf16(si + b * 4096, lane, in.a);
          if (EPI == EPI_DGRAD_SWIGLU) read_row_bf16(si + b * 4096 + 2048, lane, in.b);
          if (NIN == 1) {
            // The refill is an async-proxy (TMA) write into the buffer these
            // generic loads read.  __syncwarp orders memory only within the
            // generic proxy, so without the proxy fence neither the compiler
            // nor the hardware keeps the loads before the refill, and lanes
            // could read some 16-byte granules of the next chunk's inputs.
            fence_proxy_async_smem();
            __syncwarp();  // every lane has read its input row before the buffer is refilled
            if (more) issue_in(col + 32 + so.col, row0 + so.row);
          }
        }
        // Stores alternate between the output buffers (counting stored
        // chunks, not chunk indices); a buffer is rewritten once the stores
        // issued from it NOUT chunks ago have read it.
        uint8_t* sb = st + (NOUT == 2 ? (n_stored & 1u) * 4096 : 0);
        if (lane == 0) {
          if (NOUT == 2)
            bulk_wait_read_but_last();
          else
            bulk_wait_read_all();
        }
        __syncwarp();  // also: every lane has read its input row before the buffer is refilled
        tmem_ld_wait();
        if (split) {
          // the later parts' partial sums, added in part order
          add_parts(r0, blk1, part_stride4, p.split, c, lane);
          if (EPI == EPI_GATEUP_SWIGLU) add_parts(r1, blk1, part_stride4, p.split, BN / 64 + c, lane);
        }
        if (F8) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            r0[i] = __float_as_uint(__uint_as_float(r0[i]) * deq);
            if (EPI == EPI_GATEUP_SWIGLU) r1[i] = __float_as_uint(__uint_as_float(r1[i]) * deq);
          }
        }
        const float cm = epi_stage<EPI>(p.ep, col, reinterpret_cast<const float*>(r0),
                                        reinterpret_cast<const float*>(r1), in, sb, lane, want_max);
        if (row0 + lane < p.M) amax_acc = fmaxf(amax_acc, cm);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&map_o0, sb, col + so.col, row0 + so.row);
          if (EpiOut<EPI>::N > 1) tma_store_2d(&map_o1, sb + 2048, col + so.col, row0 + so.row);
          if (EpiOut<EPI>::N > 2) tma_store_2d(&map_o2, sb + 4096, col + so.col, row0 + so.row);
          bulk_commit_group();
        }
        if (EPI == EPI_STORE_F32 && sgd) {
          // the next chunk's masters are requested before this chunk's are written
          float nxt[32];
          if (more) sgd_load(p.ep, row0 + lane, col + 32, p.N - col - 32, nxt);
          sgd_apply(p.ep, row0 + lane, col, p.N - col, reinterpret_cast<const float*>(r0), sgdm);
          if (more) {
#pragma unroll
            for (int i = 0; i < 32; ++i) sgdm[i] = nxt[i];
          }
        }
        ++n_stored;
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
        else
          mbar_arrive(&tempty_bar[acc]);
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    // Input tiles still in flight (after an abort) land before the CTA may exit.
    int no_abort = 0;
    while (n_used < n_in) {
      const uint32_t b = NIN == 2 ? (n_used & 1u) : 0u;
      mbar_wait(&in_bar[ew][b], (in_par >> b) & 1u, &no_abort, p.status, 0u, DRAIN_LIMIT_NS);
      in_par ^= 1u << b;
      ++n_used;
    }
    if (want_max) {
      // The stored values are the bf16 roundings; rounding is monotone, so the
      // largest stored magnitude is the rounding of the largest value.
      float m = amax_acc;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) atomicMax(p.ep.amax, __float_as_uint(__bfloat162float(__float2bfloat16_rn(m))));
    }
    if (lane == 0) bulk_wait_all();  // the stores complete before the CTA may exit
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // neither CTA leaves while the other may still signal it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

struct Maps {
  CUtensorMap a, b, o[3], i[2];
};

// Epoch of a split launch: unique within the process (every context's GEMMs
// draw from it), never 0.
uint32_t next_split_epoch() {
  static std::atomic<uint32_t> last{0};
  uint32_t e = last.fetch_add(1, std::memory_order_relaxed) + 1;
  while (e == 0) e = last.fetch_add(1, std::memory_order_relaxed) + 1;
  return e;
}

template <bool PAIR, bool A_MN, bool B_MN, int EPI, bool F8 = false>
cudaError_t launch_inst(const Maps& mp, const TcParams& p, int num_sms, cudaStream_t st) {
  using C = TileCfg<PAIR, epi_has_in<EPI>(), epi_single<EPI>()>;
  auto kfn = gemm_tc_kernel<PAIR, A_MN, B_MN, EPI, F8>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_workers = 0;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    max_workers = num_sms;
    if (attr_err == cudaSuccess && PAIR) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
      cfg.blockDim = dim3(NUM_THREADS, 1, 1);
      cfg.dynamicSmemBytes = C::SMEM_BYTES;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      attr_err = cudaOccupancyMaxActiveClusters(&clusters, kfn, &cfg);
      max_workers = clusters;
    }
  });
  if (attr_err != cudaSuccess) return attr_err;
  if (max_workers <= 0) return cudaErrorInvalidConfiguration;
  // Tail split: the r tiles of the last, partial round of the persistent grid
  // (r of W workers busy) are cut into S = min(W / r, 4) contiguous K parts,
  // so that the round takes about 1/S of a tile's time.  The tail units
  // [T - r, T - r + r S) all fall in the last round (T - r is a multiple of
  // W), one per worker and after its whole tiles, so a first part only ever
  // waits on workers that wait on nobody.  Contractions shorter than 64
  // k-blocks are not split: there the partial sums' round trip through L2
  // and the counter reset cost more than the shorter round saves (measured:
  // K = 2048 GEMMs 5% slower split three ways; K >= 4096 ones 1-5% faster).
  TcParams q = p;
  const int W = max_workers;
  if (q.scratch && q.counters && q.causal == CAUSAL_NONE && q.tiles_per_batch == q.num_tiles &&
      q.kb_total >= SPLIT_MIN_KBLOCKS) {
    const int r = q.num_tiles % W;
    int S = r > 0 ? W / r : 1;
    if (S > 4) S = 4;
    if (S > q.kb_total) S = q.kb_total;
    while (S > 1 && ((size_t)r * (S - 1) * C::TILE_M * BN * sizeof(float) > q.scratch_bytes ||
                     (size_t)r * 8 * (S - 1) > (size_t)q.counter_words))
      --S;
    if (S >= 2) {
      q.split = S;
      q.split_first = q.num_tiles - r;
      q.num_units = q.split_first + r * S;
      // Arrival flags are not reset: a flag counts only when it holds this
      // launch's epoch, which no earlier launch wrote.
      q.epoch = next_split_epoch();
    }
  }
  const int workers = q.num_units < W ? q.num_units : W;
  if (!PAIR) {
    kfn<<<workers, NUM_THREADS, C::SMEM_BYTES, st>>>(mp.a, mp.b, mp.o[0], mp.o[1], mp.o[2], mp.i[0], mp.i[1], q);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * workers, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kfn, mp.a, mp.b, mp.o[0], mp.o[1], mp.o[2], mp.i[0], mp.i[1], q);
}

template <bool PAIR>
cudaError_t launch_shape(const GemmDesc& g, cudaStream_t st, int num_sms, uint32_t* status, int force_timeout) {
  const int BKE = g.f8 ? 128 : BK;  // elements per stage row
  const int esz = g.f8 ? 1 : 2;
  if (g.f8 && (g.a_mn || g.b_mn || !g.deq_a || !g.deq_b)) return cudaErrorInvalidValue;
  using C = TileCfg<PAIR, false>;  // tile shape only (the ring depth does not matter here)
  TcParams p{};
  p.M = g.M;
  p.N = g.N;
  p.num_m_blk = (g.M + C::TILE_M - 1) / C::TILE_M;
  p.num_n_blk = g.paired ? (g.N + BN / 2 - 1) / (BN / 2) : (g.N + BN - 1) / BN;
  p.tiles_per_batch = p.num_m_blk * p.num_n_blk;
  const int64_t nbatch = (int64_t)g.batch.dims[0] * g.batch.dims[1] * g.batch.dims[2];
  if (nbatch < 1 || (int64_t)p.tiles_per_batch * nbatch > (1ll << 30)) return cudaErrorInvalidValue;
  if (nbatch > 1 && (g.M % 32 != 0 || g.N % 32 != 0 || g.k_extent % BKE != 0)) return cudaErrorInvalidValue;
  p.num_tiles = (int)(p.tiles_per_batch * nbatch);
  p.batch = g.batch;
  p.causal = g.causal;
  if (g.causal != CAUSAL_NONE && (g.paired || g.kseg[0] != 0 || g.kseg[3] > g.kseg[2])) return cudaErrorInvalidValue;
  // Tiles run in groups of group_m row blocks sweeping every column block, so
  // a group's A rows (about 32 MB) stay in L2 while B streams past them.  For
  // long contractions, where that rule gives few rows, the group is at least
  // sqrt(concurrent tiles) high: the tiles in flight then form a square and
  // share the most operand blocks.
  const int64_t a_block_bytes = (int64_t)C::TILE_M * g.k_extent * esz;
  int gm = (int)((32ll << 20) / (a_block_bytes > 0 ? a_block_bytes : 1));
  int gmin = 1;
  while (gmin * gmin < (PAIR ? num_sms / 2 : num_sms)) ++gmin;
  gm = gm < gmin ? gmin : (gm > 64 ? 64 : gm);
  p.group_m = p.num_m_blk < gm ? p.num_m_blk : gm;
  for (int s = 0; s < 2; ++s) {
    const int64_t k0 = g.kseg[2 * s], k1 = g.kseg[2 * s + 1];
    if (k1 < k0 || k0 % BKE != 0 || (k1 % BKE != 0 && k1 != g.k_extent) || k1 > g.k_extent)
      return cudaErrorInvalidValue;
    p.kb[2 * s] = (int)(k0 / BKE);
    p.kb[2 * s + 1] = (int)((k1 + BKE - 1) / BKE);
  }
  if (p.kb[1] - p.kb[0] + p.kb[3] - p.kb[2] <= 0) return cudaErrorInvalidValue;
  p.kb_total = p.kb[1] - p.kb[0] + p.kb[3] - p.kb[2];
  p.num_units = p.num_tiles;  // whole tiles unless the launch splits the tail
  p.split_first = p.num_tiles;
  p.split = 1;
  p.scratch = g.split_scratch;
  p.scratch_bytes = g.split_scratch_bytes;
  p.counters = g.split_counters;
  p.counter_words = g.split_counter_words;
  p.paired = g.paired ? 1 : 0;
  p.pair_off = (int)g.pair_off;
  p.ep = g.ep;
  p.ep.M = g.M;
  p.ep.N = g.N;
  p.status = status;
  p.force_timeout = force_timeout;
  p.deq_a = g.deq_a;
  p.deq_b = g.deq_b;

  // Box heights: K-major A = this CTA's 128 rows; K-major B = 128 rows per
  // box; MN-major operands move in 64 (MN) x 64 (K) boxes.
  // MN-major operands whose MN extent is a multiple of 64 move as one 3-D box
  // per stage (fewer TMA instructions); otherwise as 64x64 2-D boxes.
  Maps mp;
  bool ok;
  // Extents of the operand tensors (contiguous x strided); a batched problem
  // reads blocks of larger tensors.
  const uint64_t a_col = g.a_ext_col ? g.a_ext_col : (uint64_t)(g.a_mn ? g.M : g.k_extent);
  const uint64_t a_row = g.a_ext_row ? g.a_ext_row : (uint64_t)(g.a_mn ? g.k_extent : g.M);
  const uint64_t b_col = g.b_ext_col ? g.b_ext_col : (uint64_t)(g.b_mn ? g.N : g.k_extent);
  const uint64_t b_row = g.b_ext_row ? g.b_ext_row : (uint64_t)(g.b_mn ? g.k_extent : g.b_rows);
  p.a3d = g.a_mn && a_col % 64 == 0 && g.M % 64 == 0;
  p.b3d = g.b_mn && b_col % 64 == 0 && g.N % 64 == 0;
  if (g.f8)
    ok = make_map_u8(&mp.a, g.a, a_col, a_row, (uint64_t)g.lda, BM);
  else if (!g.a_mn)
    ok = make_map(&mp.a, g.a, a_col, a_row, (uint64_t)g.lda, BM);
  else if (p.a3d)
    ok = make_mn_map3(&mp.a, g.a, a_col, a_row, (uint64_t)g.lda, BM / 64);
  else
    ok = make_map(&mp.a, g.a, a_col, a_row, (uint64_t)g.lda, 64);
  if (!ok) return cudaErrorInvalidValue;
  if (g.f8)
    ok = make_map_u8(&mp.b, g.b, b_col, b_row, (uint64_t)g.ldb, BN / 2);
  else if (!g.b_mn)
    ok = make_map(&mp.b, g.b, b_col, b_row, (uint64_t)g.ldb, BN / 2);
  else if (p.b3d)
    ok = make_mn_map3(&mp.b, g.b, b_col, b_row, (uint64_t)g.ldb, C::B_ROWS / 64);
  else
    ok = make_map(&mp.b, g.b, b_col, b_row, (uint64_t)g.ldb, 64);
  if (!ok) return cudaErrorInvalidValue;
  // Output maps; the paired layouts get one map per half so that stores clip
  // at the half's last channel (F) rather than at 2F.
  const uint64_t M = (uint64_t)g.M, N = (uint64_t)g.N;
  const EpiParams& e = g.ep;
  const __nv_bfloat16* o0 = static_cast<const __nv_bfloat16*>(e.out0);
  switch (g.epi) {
    case EPI_GATEUP_SWIGLU:
      ok = make_out_map(&mp.o[0], o0, false, N, M, e.ld_out0) &&
           make_out_map(&mp.o[1], o0 + e.pair_off, false, N, M, e.ld_out0) &&
           make_out_map(&mp.o[2], e.out1, false, N, M, e.ld_out1);
      break;
    case EPI_FC1_GELU:
      ok = make_out_map(&mp.o[0], o0, false, N, M, e.ld_out0) && make_out_map(&mp.o[1], e.out1, false, N, M, e.ld_out1);
      mp.o[2] = mp.o[1];
      break;
    case EPI_DGRAD_SWIGLU:
      ok = make_out_map(&mp.o[0], o0, false, N, M, e.ld_out0) &&
           make_out_map(&mp.o[1], o0 + e.pair_off, false, N, M, e.ld_out0);
      mp.o[2] = mp.o[1];
      break;
    case EPI_STORE_F32:
    case EPI_STORE_BF16:
      // batched problems store into one tensor holding every batch's block
      ok = make_out_map(&mp.o[0], e.out0, g.epi == EPI_STORE_F32, e.out_cols ? (uint64_t)e.out_cols : N,
                        e.out_rows ? (uint64_t)e.out_rows : M, e.ld_out0);
      mp.o[1] = mp.o[2] = mp.o[0];
      break;
    default:  // DOWN_RESID, DGRAD_GELU
      ok = make_out_map(&mp.o[0], o0, false, N, M, e.ld_out0);
      mp.o[1] = mp.o[2] = mp.o[0];
      break;
  }
  if (!ok) return cudaErrorInvalidValue;
  // Epilogue inputs (same 32x32 box format as the outputs).
  const __nv_bfloat16* i0 = static_cast<const __nv_bfloat16*>(e.in0);
  mp.i[0] = mp.i[1] = mp.o[0];
  if (g.epi == EPI_DOWN_RESID || g.epi == EPI_DGRAD_GELU)
    ok = make_out_map(&mp.i[0], i0, false, N, M, e.ld_in0);
  else if (g.epi == EPI_DGRAD_SWIGLU)
    ok = make_out_map(&mp.i[0], i0, false, N, M, e.ld_in0) &&
         make_out_map(&mp.i[1], i0 + e.pair_off, false, N, M, e.ld_in0);
  if (!ok) return cudaErrorInvalidValue;

  if (g.f8) {
    switch (g.epi) {
      case EPI_GATEUP_SWIGLU:
        if (!g.paired) return cudaErrorInvalidValue;
        return launch_inst<PAIR, false, false, EPI_GATEUP_SWIGLU, true>(mp, p, num_sms, st);
      case EPI_FC1_GELU:
        return launch_inst<PAIR, false, false, EPI_FC1_GELU, true>(mp, p, num_sms, st);
      case EPI_DOWN_RESID:
        return launch_inst<PAIR, false, false, EPI_DOWN_RESID, true>(mp, p, num_sms, st);
      case EPI_DGRAD_SWIGLU:
        return launch_inst<PAIR, false, false, EPI_DGRAD_SWIGLU, true>(mp, p, num_sms, st);
      case EPI_DGRAD_GELU:
        return launch_inst<PAIR, false, false, EPI_DGRAD_GELU, true>(mp, p, num_sms, st);
      case EPI_STORE_F32:
        return launch_inst<PAIR, false, false, EPI_STORE_F32, true>(mp, p, num_sms, st);
      default:
        return cudaErrorNotSupported;
    }
  }
  const int key = (g.a_mn ? 100 : 0) + (g.b_mn ? 10 : 0) + g.epi;
  switch (key) {
    case 0 + EPI_GATEUP_SWIGLU:
      if (!g.paired) return cudaErrorInvalidValue;
      return launch_inst<PAIR, false, false, EPI_GATEUP_SWIGLU>(mp, p, num_sms, st);
    case 0 + EPI_FC1_GELU:
      return launch_inst<PAIR, false, false, EPI_FC1_GELU>(mp, p, num_sms, st);
    case 0 + EPI_DOWN_RESID:
      return launch_inst<PAIR, false, false, EPI_DOWN_RESID>(mp, p, num_sms, st);
    case 10 + EPI_DGRAD_SWIGLU:
      return launch_inst<PAIR, false, true, EPI_DGRAD_SWIGLU>(mp, p, num_sms, st);
    case 10 + EPI_DGRAD_GELU:
      return launch_inst<PAIR, false, true, EPI_DGRAD_GELU>(mp, p, num_sms, st);
    case 110 + EPI_STORE_F32:
      return launch_inst<PAIR, true, true, EPI_STORE_F32>(mp, p, num_sms, st);
    case 10 + EPI_STORE_F32:
      return launch_inst<PAIR, false, true, EPI_STORE_F32>(mp, p, num_sms, st);
    case 0 + EPI_STORE_F32:
      return launch_inst<PAIR, false, false, EPI_STORE_F32>(mp, p, num_sms, st);
    case 0 + EPI_STORE_BF16:
      return launch_inst<PAIR, false, false, EPI_STORE_BF16>(mp, p, num_sms, st);
    case 10 + EPI_STORE_BF16:
      return launch_inst<PAIR, false, true, EPI_STORE_BF16>(mp, p, num_sms, st);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace

cudaError_t launch_gemm_tc(const GemmDesc& g, cudaStream_t st, int num_sms, uint32_t* status, int force_timeout) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  // CTA pairs unless the problem has a single 128-row block (or 1-CTA tiles are forced).
  const bool pair = g.tile_mode == 2 || (g.tile_mode == 0 && g.M > BM);
  if (pair) return launch_shape<true>(g, st, num_sms, status, force_timeout);
  return launch_shape<false>(g, st, num_sms, status, force_timeout);
}

}  // namespace tpmlp
