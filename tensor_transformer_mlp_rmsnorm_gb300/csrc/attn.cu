// Row kernels of the tensor-parallel attention sublayer ("Megatron-LM
// Explained", "Self-attention: split across heads"): the causal softmax of the
// score rows and its backward, and the sum of per-query-head K/V gradients
// over the heads of a group (grouped-query attention).  The contractions
// around them run on the tensor-core GEMM as batched problems.
//
// Scores are rows of S floats, one row per (sequence, query head, query i);
// keys j > i are masked.  128 threads own a row, with its values in
// registers, 16-byte accesses and warp-shuffle plus shared-memory reductions.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tpmlp_internal.h"
#include "vec.cuh"

namespace tpmlp {
namespace {

constexpr int MAX_SEQ = 4096;
constexpr int MAX_V4 = MAX_SEQ / 4 / 128;  // float4 per thread at 128 threads per row

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Causal rows are only read up to the diagonal and written up to the end of
// the diagonal's 256-column block: the GEMMs that consume P and dS contract
// over the causal part at 256-row tile granularity, so the zeros inside the
// diagonal block are read and the columns beyond it never are.
constexpr int CAUSAL_BLOCK = 256;

// 128 threads own a row (two rows per 256-thread block); thread t holds the
// float4 vectors at columns 4 (t + 128 k), so a row of S <= 4096 floats sits
// in at most 8 registers x 4 per thread.  Row maxima and sums combine the four
// warps through shared memory.
constexpr int ROW_THREADS = 128;
constexpr int ROWS_PER_BLOCK = 2;

__device__ __forceinline__ float row_reduce(float v, bool is_max, float (*red)[ROW_THREADS / 32]) {
  v = is_max ? warp_max(v) : warp_sum(v);
  const int slot = threadIdx.x / ROW_THREADS, w = (threadIdx.x % ROW_THREADS) >> 5;
  if ((threadIdx.x & 31) == 0) red[slot][w] = v;
  __syncthreads();
  float r = red[slot][0];
#pragma unroll
  for (int k = 1; k < ROW_THREADS / 32; ++k) r = is_max ? fmaxf(r, red[slot][k]) : r + red[slot][k];
  __syncthreads();  // red is reused by the next reduction
  return r;
}

// P[r, j] = exp(scale (s[r, j] - max)) / sum over j <= i, zero for i < j < the
// end of i's 256-column block, where i = r % S.
template <int NV>
__global__ void __launch_bounds__(ROW_THREADS * ROWS_PER_BLOCK) softmax_fwd_kernel(const float* __restrict__ s,
                                                                                   __nv_bfloat16* __restrict__ p,
                                                                                   int64_t rows, int S,
                                                                                   float scale_log2) {
  __shared__ float red[ROWS_PER_BLOCK][ROW_THREADS / 32];
  const int t = threadIdx.x % ROW_THREADS;
  const int64_t r = (int64_t)blockIdx.x * ROWS_PER_BLOCK + threadIdx.x / ROW_THREADS;
  const bool valid = r < rows;
  const int i = valid ? (int)(r % S) : -1;
  const int lim = valid ? min(S, (i / CAUSAL_BLOCK + 1) * CAUSAL_BLOCK) : 0;
  const float* sr = s + r * S;
  float v[NV][4];
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = 4 * (t + ROW_THREADS * k);
    if (c <= i) {
      load4(sr + c, v[k]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (c + e > i) v[k][e] = -INFINITY;
        m = fmaxf(m, v[k][e]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[k][e] = -INFINITY;
    }
  }
  m = row_reduce(m, true, red);  // finite for a valid row: column 0 is always kept
  float sum = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[k][e] = valid ? exp2f((v[k][e] - m) * scale_log2) : 0.0f;  // masked -> 0
      sum += v[k][e];
    }
  sum = row_reduce(sum, false, red);
  if (!valid) return;
  const float inv = 1.0f / sum;
  __nv_bfloat16* pr = p + r * S;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = 4 * (t + ROW_THREADS * k);
    if (c < lim) {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[k][e] *= inv;
      store4(pr + c, v[k]);
    }
  }
}

// dS[r, j] = scale * P[r, j] (dP[r, j] - sum_j P dP), written over P (zeros
// past the diagonal up to the end of its 256-column block).
template <int NV>
__global__ void __launch_bounds__(ROW_THREADS * ROWS_PER_BLOCK) softmax_bwd_kernel(__nv_bfloat16* __restrict__ p,
                                                                                   const float* __restrict__ dp,
                                                                                   int64_t rows, int S, float scale) {
  __shared__ float red[ROWS_PER_BLOCK][ROW_THREADS / 32];
  const int t = threadIdx.x % ROW_THREADS;
  const int64_t r = (int64_t)blockIdx.x * ROWS_PER_BLOCK + threadIdx.x / ROW_THREADS;
  const bool valid = r < rows;
  const int i = valid ? (int)(r % S) : -1;
  const int lim = valid ? min(S, (i / CAUSAL_BLOCK + 1) * CAUSAL_BLOCK) : 0;
  __nv_bfloat16* pr = p + r * S;
  const float* dr = dp + r * S;
  float pv[NV][4], dv[NV][4];
  float dot = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = 4 * (t + ROW_THREADS * k);
    if (c <= i) {  // P is zero past the diagonal; dP is only computed up to the diagonal's tile
      load4(pr + c, pv[k]);
      load4(dr + c, dv[k]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (c + e > i) pv[k][e] = dv[k][e] = 0.0f;
        dot = fmaf(pv[k][e], dv[k][e], dot);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) pv[k][e] = dv[k][e] = 0.0f;
    }
  }
  dot = row_reduce(dot, false, red);
  if (!valid) return;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = 4 * (t + ROW_THREADS * k);
    if (c < lim) {
      float o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = scale * pv[k][e] * (dv[k][e] - dot);
      store4(pr + c, o);
    }
  }
}

// out[b S + j, col0 + g d + c] = sum_{h < hpg} in[((b n_q + g hpg + h) S + j) d + c]
// (bf16), for the K or V section of the QKV gradient.
__global__ void __launch_bounds__(256) group_sum_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out,
                                                        int batch, int S, int n_q, int n_kv, int d, int64_t ld_out,
                                                        int64_t col0) {
  const int hpg = n_q / n_kv;
  const int64_t n4 = (int64_t)batch * n_kv * S * d / 4;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n4; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = 4 * t;
    const int c = (int)(e % d);
    const int64_t rest = e / d;
    const int j = (int)(rest % S);
    const int64_t bg = rest / S;
    const int g = (int)(bg % n_kv);
    const int b = (int)(bg / n_kv);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int h = 0; h < hpg; ++h) {
      float v[4];
      load4(in + (((int64_t)b * n_q + (int64_t)g * hpg + h) * S + j) * d + c, v);
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] += v[k];
    }
    store4(out + ((int64_t)b * S + j) * ld_out + col0 + (int64_t)g * d + c, acc);
  }
}

template <template <int> class K, typename... A>
cudaError_t launch_rows(int S, int64_t rows, cudaStream_t st, A... args) {
  const unsigned blocks = (unsigned)((rows + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK);
  const int nv = (S / 4 + ROW_THREADS - 1) / ROW_THREADS;  // float4 per thread
  if (nv <= 1)
    K<1>::launch(blocks, st, args...);
  else if (nv <= 2)
    K<2>::launch(blocks, st, args...);
  else if (nv <= 4)
    K<4>::launch(blocks, st, args...);
  else if (nv <= MAX_V4)
    K<MAX_V4>::launch(blocks, st, args...);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

template <int NV>
struct FwdL {
  static void launch(unsigned blocks, cudaStream_t st, const float* s, __nv_bfloat16* p, int64_t rows, int S,
                     float sl2) {
    softmax_fwd_kernel<NV><<<blocks, ROW_THREADS * ROWS_PER_BLOCK, 0, st>>>(s, p, rows, S, sl2);
  }
};
template <int NV>
struct BwdL {
  static void launch(unsigned blocks, cudaStream_t st, __nv_bfloat16* p, const float* dp, int64_t rows, int S,
                     float scale) {
    softmax_bwd_kernel<NV><<<blocks, ROW_THREADS * ROWS_PER_BLOCK, 0, st>>>(p, dp, rows, S, scale);
  }
};

}  // namespace

cudaError_t launch_attn_softmax_fwd(const float* s, void* p, int64_t rows, int S, float scale, cudaStream_t st) {
  if (S % 4 != 0 || S > MAX_SEQ) return cudaErrorInvalidValue;
  if (rows <= 0) return cudaSuccess;
  return launch_rows<FwdL>(S, rows, st, s, static_cast<__nv_bfloat16*>(p), rows, S, scale * 1.4426950408889634f);
}

cudaError_t launch_attn_softmax_bwd(void* p, const float* dp, int64_t rows, int S, float scale, cudaStream_t st) {
  if (S % 4 != 0 || S > MAX_SEQ) return cudaErrorInvalidValue;
  if (rows <= 0) return cudaSuccess;
  return launch_rows<BwdL>(S, rows, st, static_cast<__nv_bfloat16*>(p), dp, rows, S, scale);
}

cudaError_t launch_attn_group_sum(const float* in, void* out, int batch, int S, int n_q, int n_kv, int d,
                                  int64_t ld_out, int64_t col0, int num_sms, cudaStream_t st) {
  if (d % 4 != 0) return cudaErrorInvalidValue;
  const int64_t n4 = (int64_t)batch * n_kv * S * d / 4;
  if (n4 <= 0) return cudaSuccess;
  int64_t blocks = (n4 + 255) / 256;
  if (blocks > 8LL * num_sms) blocks = 8LL * num_sms;
  group_sum_kernel<<<(unsigned)blocks, 256, 0, st>>>(in, static_cast<__nv_bfloat16*>(out), batch, S, n_q, n_kv, d,
                                                     ld_out, col0);
  return cudaGetLastError();
}

}  // namespace tpmlp
