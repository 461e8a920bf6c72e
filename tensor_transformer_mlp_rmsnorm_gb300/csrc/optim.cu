// AdamW with global gradient-norm clipping, the optimizer step of the
// "Megatron-LM walkthrough" ("Stage 8"): the norm of every gradient taken
// together, a clip factor from it, then the AdamW update of the fp32 masters
// (or of the parameters in place for fp32).
//
// Two HBM-bound kernels over the same fixed grid:
//   grad_sqnorm : each block sums g^2 over its grid-stride share of all
//                 gradients (fp64 accumulation) into one partial;
//   adamw_update: each block first sums all partials in the same fixed order
//                 (so every block derives the identical norm and clip factor),
//                 then updates its share: reads g, m, v, master and writes m,
//                 v, master and the parameter copy (30 B per bf16 parameter).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "tpmlp_internal.h"
#include "vec.cuh"

namespace tpmlp {
namespace {

constexpr int THREADS = 256;
constexpr double CLIP_EPS = 1e-6;

// Sum over the block in a fixed order; result valid in thread 0.
__device__ double block_sum(double s) {
  __shared__ double warp_part[THREADS / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = s;
  __syncthreads();
  double r = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < THREADS / 32; ++w) r += warp_part[w];
  return r;
}

__device__ __forceinline__ float sq4(const float* v) { return (v[0] * v[0] + v[1] * v[1]) + (v[2] * v[2] + v[3] * v[3]); }

// FP64 is a slow pipe on this part: squares are summed in float over 16
// elements (a balanced tree, relative error a few 1e-7) and only those
// partial sums are accumulated in double.
__global__ void __launch_bounds__(THREADS) grad_sqnorm_kernel(const AdamArgs a) {
  const int64_t stride = (int64_t)gridDim.x * THREADS;
  const int64_t tid = (int64_t)blockIdx.x * THREADS + threadIdx.x;
  double s = 0.0;
  for (int k = 0; k < a.nseg; ++k) {
    const float* g = a.seg[k].grad;
    const int64_t n4 = a.seg[k].n / 4;
    int64_t i = tid;
    for (; i + 3 * stride < n4; i += 4 * stride) {
      float v0[4], v1[4], v2[4], v3[4];
      load4(g + 4 * i, v0);
      load4(g + 4 * (i + stride), v1);
      load4(g + 4 * (i + 2 * stride), v2);
      load4(g + 4 * (i + 3 * stride), v3);
      s += (double)((sq4(v0) + sq4(v1)) + (sq4(v2) + sq4(v3)));
    }
    for (; i < n4; i += stride) {
      float v[4];
      load4(g + 4 * i, v);
      s += (double)sq4(v);
    }
  }
  s = block_sum(s);
  if (threadIdx.x == 0) a.part[blockIdx.x] = s;
}

template <typename T>
__global__ void __launch_bounds__(THREADS) adamw_kernel(const AdamArgs a) {
  __shared__ float s_clip;
  double s = 0.0;
  for (int i = threadIdx.x; i < (int)gridDim.x; i += THREADS) s += a.part[i];
  s = block_sum(s);
  if (threadIdx.x == 0) {
    const double norm = sqrt(s);
    float clip = 1.0f;
    if (a.max_norm > 0.0f) {
      const double c = (double)a.max_norm / (norm + CLIP_EPS);
      if (c < 1.0) clip = (float)c;
    }
    s_clip = clip;
    if (blockIdx.x == 0 && a.grad_norm) *a.grad_norm = (float)norm;
  }
  __syncthreads();
  const float clip = s_clip;
  const int64_t stride = (int64_t)gridDim.x * THREADS;
  const int64_t tid = (int64_t)blockIdx.x * THREADS + threadIdx.x;
  for (int k = 0; k < a.nseg; ++k) {
    const AdamSeg sg = a.seg[k];
    T* w = static_cast<T*>(sg.w);
    const int64_t n4 = sg.n / 4;
    for (int64_t i = tid; i < n4; i += stride) {
      float g[4], m[4], v[4], p[4];
      load4(sg.grad + 4 * i, g);
      load4(sg.m + 4 * i, m);
      load4(sg.v + 4 * i, v);
      if (sg.master)
        load4(sg.master + 4 * i, p);
      else
        load4(w + 4 * i, p);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float gc = g[j] * clip;
        m[j] = fmaf(a.beta1, m[j], a.one_m_beta1 * gc);
        v[j] = fmaf(a.beta2, v[j], a.one_m_beta2 * gc * gc);
        const float denom = sqrtf(v[j]) * a.inv_sqrt_bc2 + a.eps;
        p[j] = fmaf(-sg.lr_wd, p[j], p[j]) - a.step_size * m[j] / denom;
      }
      store4(sg.m + 4 * i, m);
      store4(sg.v + 4 * i, v);
      if (sg.master) store4(sg.master + 4 * i, p);
      store4(w + 4 * i, p);
    }
  }
}

}  // namespace

int adam_blocks(const AdamArgs& a, int num_sms) {
  int64_t tot = 0;
  for (int k = 0; k < a.nseg; ++k) tot += a.seg[k].n / 4;
  int64_t b = (tot + THREADS - 1) / THREADS;
  if (b > 8LL * num_sms) b = 8LL * num_sms;
  if (b > MAX_NORM_PARTS) b = MAX_NORM_PARTS;
  return (int)(b < 1 ? 1 : b);
}

cudaError_t launch_grad_sqnorm(const AdamArgs& a, int nblocks, cudaStream_t st) {
  grad_sqnorm_kernel<<<nblocks, THREADS, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_adamw(int dtype, const AdamArgs& a, int nblocks, cudaStream_t st) {
  if (dtype == 0)
    adamw_kernel<float><<<nblocks, THREADS, 0, st>>>(a);
  else
    adamw_kernel<__nv_bfloat16><<<nblocks, THREADS, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tpmlp
