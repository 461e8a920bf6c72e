// FP8 (E4M3) operands for the tensor-core GEMMs: per-tensor scaling from the
// tensor's current absolute maximum (the FP8 Transformer Engine GEMMs of
// "Megatron-Core Architecture: 5D Distributed Parallelism, ... FP8 Transformer
// Engine"), written as HBM-bound kernels:
//
//   amax_partials : per-block maxima of |x| over a bf16 tensor (integer max
//                   on the magnitude bits, so order-independent and exact);
//   quantize_e4m3 : every block folds the partials into the same amax and
//                   scale s = 448 / amax (float32; 1 for an all-zero tensor),
//                   then casts 128x128 tiles: codes = RN_satfinite(x * s),
//                   written row-major (dst) and/or transposed (dst_t) through
//                   shared memory; block 0 stores 1 / s for the GEMM epilogue.
//
// The GEMMs take only K-major E4M3 operands, so every operand that a GEMM
// contracts along its rows (weights in the data-gradient GEMMs, activations
// and gradients in the weight-gradient GEMMs) gets a transposed copy here.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/tpmlp.h"
#include "tpmlp_internal.h"

namespace tpmlp {
namespace {

constexpr int THREADS = 256;

__global__ void __launch_bounds__(THREADS) amax_partials_kernel(const __nv_bfloat16* __restrict__ x, int64_t n8,
                                                                float* __restrict__ part) {
  const int64_t stride = (int64_t)gridDim.x * THREADS;
  uint32_t m = 0;  // two bf16 magnitudes per 32-bit word, compared as unsigned halves
  for (int64_t i = (int64_t)blockIdx.x * THREADS + threadIdx.x; i < n8; i += stride) {
    const uint4 v = reinterpret_cast<const uint4*>(x)[i];
    m = __vmaxu2(m, v.x & 0x7fff7fffu);
    m = __vmaxu2(m, v.y & 0x7fff7fffu);
    m = __vmaxu2(m, v.z & 0x7fff7fffu);
    m = __vmaxu2(m, v.w & 0x7fff7fffu);
  }
  uint32_t h = max(m & 0xffffu, m >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) h = max(h, __shfl_xor_sync(0xffffffffu, h, o));
  __shared__ uint32_t red[THREADS / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = h;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int w = 0; w < THREADS / 32; ++w) r = max(r, red[w]);
    part[blockIdx.x] = __uint_as_float(r << 16);  // bf16 bits -> float
  }
}

__device__ __forceinline__ uint32_t cvt4_e4m3(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// 8 bf16 -> 8 codes (two 32-bit words), scaled by s.
__device__ __forceinline__ uint2 quant8(const uint4 v, float s) {
  float f[8];
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    f[2 * i] = t.x * s;
    f[2 * i + 1] = t.y * s;
  }
  return make_uint2(cvt4_e4m3(f[0], f[1], f[2], f[3]), cvt4_e4m3(f[4], f[5], f[6], f[7]));
}

struct QuantArgs {
  const __nv_bfloat16* src;  // [rows, cols], contiguous
  int64_t rows, cols;
  uint8_t* dst;  // [rows, cols] codes, pitch ld (or nullptr)
  int64_t ld;
  uint8_t* dst_t;  // [cols, rows] codes, pitch ld_t (or nullptr)
  int64_t ld_t;
  const float* part;  // amax partials
  int nparts;
  float* inv_scale;  // out: 1 / s
};

// One block casts 128x128 tiles.  Phase 1: each thread converts 16-element
// row segments (row-major codes go straight to dst) and parks the codes
// row-major in shared memory.  Phase 2: each thread takes a 16-row x 4-column
// block of codes (16 word reads; a warp reads 32 consecutive words of one
// row, so no bank conflicts), transposes it as 4x4 byte blocks with
// __byte_perm, and writes four 16-byte rows of dst_t.
constexpr int QT = 128;

__device__ __forceinline__ void transpose4x4(uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  // rows a..d hold bytes [x0 x1 x2 x3] (x0 lowest); afterwards a..d hold the columns
  const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(a, b, 0x7362);
  const uint32_t t2 = __byte_perm(c, d, 0x5140), t3 = __byte_perm(c, d, 0x7362);
  a = __byte_perm(t0, t2, 0x5410);
  b = __byte_perm(t0, t2, 0x7632);
  c = __byte_perm(t1, t3, 0x5410);
  d = __byte_perm(t1, t3, 0x7632);
}

__global__ void __launch_bounds__(THREADS) quantize_e4m3_kernel(const QuantArgs q) {
  __shared__ __align__(16) uint32_t tile[QT][QT / 4];  // codes, row-major, 4 per word
  __shared__ float red[THREADS / 32];
  __shared__ float s_scale;
  float m = 0.0f;
  for (int i = threadIdx.x; i < q.nparts; i += THREADS) m = fmaxf(m, q.part[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.0f;
    for (int w = 0; w < THREADS / 32; ++w) a = fmaxf(a, red[w]);
    const float s = (a > 0.0f && a <= 3.4e38f) ? __fdiv_rn(448.0f, a) : 1.0f;
    s_scale = s;
    if (blockIdx.x == 0) *q.inv_scale = __fdiv_rn(1.0f, s);
  }
  __syncthreads();
  const float s = s_scale;
  const int64_t tiles_c = (q.cols + QT - 1) / QT;
  const int64_t ntiles = ((q.rows + QT - 1) / QT) * tiles_c;
  // phase 1: 8 threads per row, 16 codes each; 32 rows per pass, 4 passes
  const int seg = threadIdx.x & 7, prow = threadIdx.x >> 3;
  // phase 2: a warp per 16-row group, a lane per 4-column group
  const int cg = threadIdx.x & 31, rg = threadIdx.x >> 5;
  for (int64_t tile_i = blockIdx.x; tile_i < ntiles; tile_i += gridDim.x) {
    const int64_t r0 = (tile_i / tiles_c) * QT, c0 = (tile_i % tiles_c) * QT;
    const int64_t c = c0 + seg * 16;
    // all eight 16-byte loads of this thread first, then the casts and stores
    uint4 raw[4][2];
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
      const int64_t r = r0 + pass * 32 + prow;
      const __nv_bfloat16* src = q.src + r * q.cols + c;
      raw[pass][0] = (r < q.rows && c < q.cols) ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0, 0, 0, 0);
      raw[pass][1] =
          (r < q.rows && c + 8 < q.cols) ? __ldg(reinterpret_cast<const uint4*>(src + 8)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
      const int tr = pass * 32 + prow;
      const int64_t r = r0 + tr;
      const uint2 lo = quant8(raw[pass][0], s), hi = quant8(raw[pass][1], s);
      if (r < q.rows) {
        if (q.dst) {
          uint8_t* d = q.dst + r * q.ld + c;
          if (c + 8 < q.cols)
            *reinterpret_cast<uint4*>(d) = make_uint4(lo.x, lo.y, hi.x, hi.y);
          else if (c < q.cols)
            *reinterpret_cast<uint2*>(d) = lo;
        }
      }
      if (q.dst_t) *reinterpret_cast<uint4*>(&tile[tr][seg * 4]) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
    if (q.dst_t) {
      __syncthreads();
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) w[k] = tile[rg * 16 + k][cg];
#pragma unroll
      for (int k = 0; k < 16; k += 4) transpose4x4(w[k], w[k + 1], w[k + 2], w[k + 3]);
      // w[4 j + i] now holds rows 4j..4j+3 of source column 4 cg + i
      const int64_t rr = r0 + rg * 16;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t col = c0 + cg * 4 + i;  // source column = destination row
        if (col < q.cols && rr < q.rows) {
          uint8_t* out = q.dst_t + col * q.ld_t + rr;
          const uint4 v = make_uint4(w[i], w[4 + i], w[8 + i], w[12 + i]);
          if (rr + 16 <= q.rows) {
            *reinterpret_cast<uint4*>(out) = v;
          } else {
            const uint8_t* b = reinterpret_cast<const uint8_t*>(&v);
            for (int j = 0; j < 16 && rr + j < q.rows; ++j) out[j] = b[j];
          }
        }
      }
      __syncthreads();
    }
  }
}

}  // namespace

int fp8_blocks(int64_t elems, int num_sms) {
  int64_t b = (elems / 8 + THREADS - 1) / THREADS;
  if (b > 4LL * num_sms) b = 4LL * num_sms;
  if (b > FP8_MAX_PARTS) b = FP8_MAX_PARTS;
  return (int)(b < 1 ? 1 : b);
}

cudaError_t launch_fp8_amax(const void* src, int64_t n, float* part, int nparts, cudaStream_t st) {
  if (n <= 0) return cudaMemsetAsync(part, 0, sizeof(float), st);
  amax_partials_kernel<<<nparts, THREADS, 0, st>>>(static_cast<const __nv_bfloat16*>(src), n / 8, part);
  return cudaGetLastError();
}

cudaError_t launch_fp8_cast(const void* src, int64_t rows, int64_t cols, uint8_t* dst, int64_t ld, uint8_t* dst_t,
                            int64_t ld_t, const float* part, int nparts, float* inv_scale, int num_sms,
                            cudaStream_t st) {
  QuantArgs q{static_cast<const __nv_bfloat16*>(src), rows, cols, dst, ld, dst_t, ld_t, part, nparts, inv_scale};
  const int64_t tiles = ((rows + QT - 1) / QT) * ((cols + QT - 1) / QT);
  int64_t qb = tiles < 4LL * num_sms ? tiles : 4LL * num_sms;
  if (qb < 1) qb = 1;
  quantize_e4m3_kernel<<<(unsigned)qb, THREADS, 0, st>>>(q);
  return cudaGetLastError();
}

cudaError_t launch_fp8_quantize(const void* src, int64_t rows, int64_t cols, uint8_t* dst, int64_t ld,
                                uint8_t* dst_t, int64_t ld_t, float* part, float* inv_scale, int num_sms,
                                cudaStream_t st) {
  const int64_t n = rows * cols;
  const int nb = n > 0 ? fp8_blocks(n, num_sms) : 1;
  const cudaError_t e = launch_fp8_amax(src, n, part, nb, st);
  if (e != cudaSuccess) return e;
  return launch_fp8_cast(src, rows, cols, dst, ld, dst_t, ld_t, part, nb, inv_scale, num_sms, st);
}

}  // namespace tpmlp

using namespace tpmlp;

extern "C" {

TPMLP_API tpmlp_status tpmlp_fp8_quantize(const void* src, int64_t rows, int64_t cols, uint8_t* dst, int64_t ld_dst,
                                          uint8_t* dst_t, int64_t ld_dst_t, float* inv_scale, void* scratch,
                                          void* stream) {
  auto aligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  if (rows < 0 || cols < 0 || cols % 8 != 0) return TPMLP_ERR_SHAPE;
  const bool empty = rows * cols == 0;  // NULL tensors are allowed then
  if (!inv_scale || !scratch || (!empty && (!src || (!dst && !dst_t)))) return TPMLP_ERR_ARG;
  if (!aligned(src, 16) || !aligned(scratch, 16) || !aligned(inv_scale, 4)) return TPMLP_ERR_ARG;
  if (dst && (!aligned(dst, 16) || ld_dst < cols || ld_dst % 16 != 0)) return TPMLP_ERR_ARG;
  if (dst_t && (!aligned(dst_t, 16) || ld_dst_t < rows || ld_dst_t % 16 != 0)) return TPMLP_ERR_ARG;
  if (empty) dst = dst_t = nullptr;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    return TPMLP_ERR_CUDA;
  const cudaError_t e = launch_fp8_quantize(src, rows, cols, dst, ld_dst, dst_t, ld_dst_t,
                                            static_cast<float*>(scratch), inv_scale, sms,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TPMLP_OK : TPMLP_ERR_CUDA;
}

TPMLP_API tpmlp_status tpmlp_fp8_gemm(const uint8_t* a, int64_t lda, const uint8_t* b, int64_t ldb, int64_t M,
                                      int64_t N, int64_t K, const float* inv_scale_a, const float* inv_scale_b,
                                      float* c, int64_t ldc, uint32_t* status, void* stream) {
  auto aligned = [](const void* p, uintptr_t al) { return (reinterpret_cast<uintptr_t>(p) & (al - 1)) == 0; };
  if (M < 0 || N < 0 || K < 1 || M > (1 << 30) || N > (1 << 30)) return TPMLP_ERR_SHAPE;
  if (N % 4 != 0) return TPMLP_ERR_SHAPE;
  if (!a || !b || !c || !inv_scale_a || !inv_scale_b || !status) return TPMLP_ERR_ARG;
  if (!aligned(a, 16) || !aligned(b, 16) || !aligned(c, 16) || !aligned(status, 4)) return TPMLP_ERR_ARG;
  if (lda < K || ldb < K || lda % 16 != 0 || ldb % 16 != 0 || ldc < N || ldc % 4 != 0) return TPMLP_ERR_ARG;
  if (M == 0 || N == 0) return TPMLP_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    return TPMLP_ERR_CUDA;
  GemmDesc g;
  g.M = (int)M;
  g.N = (int)N;
  g.k_extent = K;
  g.a = a;
  g.lda = lda;
  g.b = b;
  g.ldb = ldb;
  g.b_rows = N;
  g.kseg[1] = K;
  g.epi = EPI_STORE_F32;
  g.ep.out0 = c;
  g.ep.ld_out0 = ldc;
  g.f8 = true;
  g.deq_a = inv_scale_a;
  g.deq_b = inv_scale_b;
  const cudaError_t e = launch_gemm_tc(g, static_cast<cudaStream_t>(stream), sms, status, 0);
  return e == cudaSuccess ? TPMLP_OK : (e == cudaErrorInvalidValue ? TPMLP_ERR_ARG : TPMLP_ERR_CUDA);
}

}  // extern "C"
