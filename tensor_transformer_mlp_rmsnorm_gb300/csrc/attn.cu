// Row kernels of the tensor-parallel attention sublayer ("Megatron-LM
// Explained", "Self-attention: split across heads"): the causal softmax of the
// score rows and its backward, and the sum of per-query-head K/V gradients
// over the heads of a group (grouped-query attention).  The contractions
// around them run on the tensor-core GEMM as batched problems.
//
// Scores are rows of S floats, one row per (sequence, query head, query i);
// keys j > i are masked.  One warp owns a row: S / 32 values per lane in
// registers, 16-byte accesses, warp-shuffle max and sums.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tpmlp_internal.h"
#include "vec.cuh"

namespace tpmlp {
namespace {

constexpr int WARPS = 8;
constexpr int MAX_SEQ = 4096;              // 128 floats per lane
constexpr int MAX_V4 = MAX_SEQ / 32 / 4;  // float4 per lane

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

// P[r, j] = exp(scale (s[r, j] - max)) / sum over j <= i, zero for j > i,
// where i = r % S.  Lane l holds columns 4 (l + 32 v) .. +3.
template <int NV>
__global__ void __launch_bounds__(WARPS * 32) softmax_fwd_kernel(const float* __restrict__ s,
                                                                 __nv_bfloat16* __restrict__ p, int64_t rows,
                                                                 int S, float scale_log2) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int i = (int)(r % S);
  const float* sr = s + r * S;
  float v[NV][4];
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = 4 * (lane + 32 * k);
    if (c < S) {
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
  m = warp_max(m);  // finite: column 0 is always kept
  float sum = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[k][e] = exp2f((v[k][e] - m) * scale_log2);  // masked -> 0
      sum += v[k][e];
    }
  const float inv = 1.0f / warp_sum(sum);
  __nv_bfloat16* pr = p + r * S;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = 4 * (lane + 32 * k);
    if (c < S) {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[k][e] *= inv;
      store4(pr + c, v[k]);
    }
  }
}

// dS[r, j] = scale * P[r, j] (dP[r, j] - sum_j P dP), written over P.
template <int NV>
__global__ void __launch_bounds__(WARPS * 32) softmax_bwd_kernel(__nv_bfloat16* __restrict__ p,
                                                                 const float* __restrict__ dp, int64_t rows, int S,
                                                                 float scale) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (r >= rows) return;
  __nv_bfloat16* pr = p + r * S;
  const float* dr = dp + r * S;
  float pv[NV][4], dv[NV][4];
  float dot = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = 4 * (lane + 32 * k);
    if (c < S) {
      load4(pr + c, pv[k]);
      load4(dr + c, dv[k]);
#pragma unroll
      for (int e = 0; e < 4; ++e) dot = fmaf(pv[k][e], dv[k][e], dot);
    }
  }
  dot = warp_sum(dot);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = 4 * (lane + 32 * k);
    if (c < S) {
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
  const unsigned blocks = (unsigned)((rows + WARPS - 1) / WARPS);
  const int nv = (S / 4 + 31) / 32;
  if (nv <= 4)
    K<4>::launch(blocks, st, args...);
  else if (nv <= 16)
    K<16>::launch(blocks, st, args...);
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
    softmax_fwd_kernel<NV><<<blocks, WARPS * 32, 0, st>>>(s, p, rows, S, sl2);
  }
};
template <int NV>
struct BwdL {
  static void launch(unsigned blocks, cudaStream_t st, __nv_bfloat16* p, const float* dp, int64_t rows, int S,
                     float scale) {
    softmax_bwd_kernel<NV><<<blocks, WARPS * 32, 0, st>>>(p, dp, rows, S, scale);
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
