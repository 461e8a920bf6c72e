// Memory-bound kernels of the sublayer step: RMSNorm forward and backward
// (with the residual gradient and the token-axis sums of the replicated
// parameters' gradients), the MSE loss and its gradient, column sums, and the
// SGD update.  All use 16-byte vector accesses and fp32 arithmetic;
// reductions over tokens go through per-block partials summed in a fixed
// order, so results are deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "tpmlp_internal.h"
#include "vec.cuh"

namespace tpmlp {
namespace {

// ------------------------------------------------------------- RMSNorm fwd
// A block of 256 threads walks rows r = blockIdx.x, + gridDim.x, ...; each
// thread holds NVT 16-byte vectors of the row (and of w, loaded once).  The
// next row's vectors are loaded before the current row's block-wide sum of
// squares, so two rows of loads are in flight per block.  With `amax`, the
// largest stored |normed value| of the block is combined into *amax (float
// bits, atomicMax; rounding to T is monotone, so the rounding of the largest
// value is the largest stored value).
template <typename T, int NVT>
__global__ void __launch_bounds__(256) rmsnorm_fwd_kernel(const T* __restrict__ x, const T* __restrict__ w, float eps,
                                                          T* __restrict__ nrm, float* __restrict__ rstd, int64_t N,
                                                          int H, uint32_t* __restrict__ amax) {
  constexpr int V = Vec<T>::N;
  __shared__ float red[2][8];
  const int nvec = H / V;
  float wv[NVT][V];
  uint4 nx[NVT];  // next row, raw
#pragma unroll
  for (int i = 0; i < NVT; ++i) {
    const int v = threadIdx.x + 256 * i;
    if (v < nvec) Vec<T>::load(w + v * V, wv[i]);
  }
  auto prefetch = [&](int64_t row) {
#pragma unroll
    for (int i = 0; i < NVT; ++i) {
      const int v = threadIdx.x + 256 * i;
      if (v < nvec) nx[i] = __ldg(reinterpret_cast<const uint4*>(x + row * H + v * V));
    }
  };
  float m = 0.0f;
  int par = 0;
  if ((int64_t)blockIdx.x < N) prefetch(blockIdx.x);
  for (int64_t row = blockIdx.x; row < N; row += gridDim.x, par ^= 1) {
    float xs[NVT][V];
#pragma unroll
    for (int i = 0; i < NVT; ++i) {
      const int v = threadIdx.x + 256 * i;
      if (v < nvec)
        Vec<T>::load(reinterpret_cast<const T*>(&nx[i]), xs[i]);
      else
#pragma unroll
        for (int j = 0; j < V; ++j) xs[i][j] = 0.0f;
    }
    if (row + gridDim.x < N) prefetch(row + gridDim.x);
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < NVT; ++i)
#pragma unroll
      for (int j = 0; j < V; ++j) ss = fmaf(xs[i][j], xs[i][j], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[par][threadIdx.x >> 5] = ss;
    __syncthreads();
    ss = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) ss += red[par][k];
    const float r = 1.0f / sqrtf(ss / (float)H + eps);
    T* nr = nrm + row * H;
#pragma unroll
    for (int i = 0; i < NVT; ++i) {
      const int v = threadIdx.x + 256 * i;
      if (v < nvec) {
        float o[V];
#pragma unroll
        for (int j = 0; j < V; ++j) {
          o[j] = xs[i][j] * r * wv[i][j];
          m = fmaxf(m, fabsf(o[j]));
        }
        Vec<T>::store(nr + v * V, o);
      }
    }
    if (threadIdx.x == 0) rstd[row] = r;
  }
  if (amax) {
    __shared__ float redm[8];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) redm[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int k = 1; k < 8; ++k) m = fmaxf(m, redm[k]);
      atomicMax(amax, __float_as_uint(to_f(from_f<T>(m))));
    }
  }
}

template <typename T, int NVT>
cudaError_t rmsnorm_fwd_nvt(const T* x, const T* w, float eps, T* nrm, float* rstd, int64_t N, int H,
                            uint32_t* amax, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = 4LL * (sms > 0 ? sms : 1);  // one wave
  if (blocks > N) blocks = N;
  rmsnorm_fwd_kernel<T, NVT><<<(unsigned)blocks, 256, 0, st>>>(x, w, eps, nrm, rstd, N, H, amax);
  return cudaGetLastError();
}

template <typename T>
cudaError_t rmsnorm_fwd_t(const T* x, const T* w, float eps, T* nrm, float* rstd, int64_t N, int64_t H,
                          uint32_t* amax, cudaStream_t st) {
  const int64_t nvec = H / Vec<T>::N;
  if (nvec <= 256) return rmsnorm_fwd_nvt<T, 1>(x, w, eps, nrm, rstd, N, (int)H, amax, st);
  if (nvec <= 512) return rmsnorm_fwd_nvt<T, 2>(x, w, eps, nrm, rstd, N, (int)H, amax, st);
  if (nvec <= 1024) return rmsnorm_fwd_nvt<T, 4>(x, w, eps, nrm, rstd, N, (int)H, amax, st);
  if (nvec <= 2048) return rmsnorm_fwd_nvt<T, 8>(x, w, eps, nrm, rstd, N, (int)H, amax, st);
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------- RMSNorm bwd
// Block b owns rows [b*R, (b+1)*R).  Per row: g = dN * w, xhat = x * rstd,
// c = mean_h(g * xhat), dx = dy + rstd * (g - xhat * c).  Each thread also
// keeps running column sums of dN * xhat (norm weight gradient) and dy (down
// bias gradient) for its columns; they are written as the block's partials.
// The next row's dN, x, dy and rstd are loaded (as raw 16/8-byte vectors)
// before the current row's reduction, so a block keeps two rows of loads in
// flight; w is re-read from L1 each row to leave room in the register file.
template <typename T>
struct Raw4;  // 4 consecutive elements as loaded
template <>
struct Raw4<float> {
  float4 v;
  __device__ void load(const float* p) { v = __ldg(reinterpret_cast<const float4*>(p)); }
  __device__ void get(float* f) const { f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w; }
};
template <>
struct Raw4<__nv_bfloat16> {
  uint2 v;
  __device__ void load(const __nv_bfloat16* p) { v = __ldg(reinterpret_cast<const uint2*>(p)); }
  __device__ void get(float* f) const {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  }
};

template <typename T, int MAXV>
__global__ void __launch_bounds__(256) rmsnorm_bwd_kernel(const float* __restrict__ dnrm, const T* __restrict__ x,
                                                          const float* __restrict__ rstd, const T* __restrict__ w,
                                                          const T* __restrict__ dy, T* __restrict__ dx,
                                                          float* __restrict__ part_dw, float* __restrict__ part_db,
                                                          int64_t N, int H, int64_t shard_rows, int blocks_per_shard,
                                                          int rows_per_block) {
  __shared__ float red[2][8];
  const int nv = H / 4;
  float adw[MAXV][4], adb[MAXV][4];
#pragma unroll
  for (int i = 0; i < MAXV; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) adw[i][j] = adb[i][j] = 0.0f;
  // Blocks tile each token shard separately, so no block's partial mixes two
  // shards (one shard spanning all N rows when the tokens are not split).
  const int64_t shard = blockIdx.x / blocks_per_shard;
  const int64_t s0 = shard * shard_rows;
  const int64_t r0 = s0 + (int64_t)(blockIdx.x % blocks_per_shard) * rows_per_block;
  const int64_t r1 = min(min(N, s0 + shard_rows), r0 + rows_per_block);
  float4 dn_n[MAXV];
  Raw4<T> x_n[MAXV], dy_n[MAXV];
  float rs_n = 0.0f;
  auto prefetch = [&](int64_t row) {
    rs_n = __ldg(rstd + row);
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int v = threadIdx.x + 256 * i;
      if (v < nv) {
        dn_n[i] = __ldg(reinterpret_cast<const float4*>(dnrm + row * H) + v);
        x_n[i].load(x + row * H + 4 * v);
        dy_n[i].load(dy + row * H + 4 * v);
      }
    }
  };
  if (r0 < r1) prefetch(r0);
  int par = 0;
  for (int64_t row = r0; row < r1; ++row, par ^= 1) {
    float4 dn_c[MAXV];
    Raw4<T> x_c[MAXV], dy_c[MAXV];
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      dn_c[i] = dn_n[i];
      x_c[i] = x_n[i];
      dy_c[i] = dy_n[i];
    }
    const float rs = rs_n;
    if (row + 1 < r1) prefetch(row + 1);
    float dot = 0.0f;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int v = threadIdx.x + 256 * i;
      if (v < nv) {
        float xv[4], wv[4];
        x_c[i].get(xv);
        Raw4<T> wr;
        wr.load(w + 4 * v);
        wr.get(wv);
        const float dn[4] = {dn_c[i].x, dn_c[i].y, dn_c[i].z, dn_c[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) dot = fmaf(dn[j] * wv[j], xv[j] * rs, dot);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if ((threadIdx.x & 31) == 0) red[par][threadIdx.x >> 5] = dot;
    __syncthreads();
    dot = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) dot += red[par][k];
    const float c = dot / (float)H;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int v = threadIdx.x + 256 * i;
      if (v < nv) {
        float xv[4], wv[4], d[4], o[4];
        x_c[i].get(xv);
        dy_c[i].get(d);
        Raw4<T> wr;
        wr.load(w + 4 * v);
        wr.get(wv);
        const float dn[4] = {dn_c[i].x, dn_c[i].y, dn_c[i].z, dn_c[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float xh = xv[j] * rs;
          const float g = dn[j] * wv[j];
          o[j] = d[j] + rs * (g - xh * c);
          adw[i][j] = fmaf(dn[j], xh, adw[i][j]);
          adb[i][j] += d[j];
        }
        store4(dx + row * H + 4 * v, o);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int v = threadIdx.x + 256 * i;
    if (v < nv) {
      store4(part_dw + (int64_t)blockIdx.x * H + 4 * v, adw[i]);
      store4(part_db + (int64_t)blockIdx.x * H + 4 * v, adb[i]);
    }
  }
}

template <typename T>
cudaError_t rmsnorm_bwd_t(const float* dnrm, const T* x, const float* rstd, const T* w, const T* dy, T* dx,
                          float* part_dw, float* part_db, int64_t N, int64_t H, int shards, int nblocks,
                          cudaStream_t st) {
  const int64_t shard_rows = N / shards;
  const int bps = nblocks / shards;
  const int rpb = (int)((shard_rows + bps - 1) / bps);
  const int nv = (int)(H / 4);
#define TPMLP_BWD(MV)                                                                                            \
  rmsnorm_bwd_kernel<T, MV><<<nblocks, 256, 0, st>>>(dnrm, x, rstd, w, dy, dx, part_dw, part_db, N, (int)H, \
                                                    shard_rows, bps, rpb)
  if (nv <= 256) TPMLP_BWD(1);
  else if (nv <= 512) TPMLP_BWD(2);
  else if (nv <= 1024) TPMLP_BWD(4);
  else if (nv <= 2048) TPMLP_BWD(8);
  else return cudaErrorInvalidValue;
#undef TPMLP_BWD
  return cudaGetLastError();
}

// ------------------------------------------------------------- column sums
// out[g][c] = sum_p part[g * nparts + p][c] for up to two (part, out) pairs
// (blockIdx.y) and `groups` groups of partial rows (blockIdx.z).
// A block covers 32 columns; its 8 warps each sum a strided subset of the
// partial rows, then the 8 warp sums are added in warp order (deterministic).
__global__ void __launch_bounds__(256) colsum_finalize_kernel(const float* __restrict__ part0, float* __restrict__ out0,
                                                              const float* __restrict__ part1, float* __restrict__ out1,
                                                              int nparts, int64_t C) {
  __shared__ float red[8][33];
  // blockIdx.z: group of nparts consecutive partial rows -> output row z
  const float* part = (blockIdx.y ? part1 : part0) + (int64_t)blockIdx.z * nparts * C;
  float* out = (blockIdx.y ? out1 : out0) + (int64_t)blockIdx.z * C;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 32 + lane;
  float s = 0.0f;
  if (c < C)
    for (int p = wid; p < nparts; p += 8) s += part[(int64_t)p * C + c];
  red[wid][lane] = s;
  __syncthreads();
  if (wid == 0 && c < C) {
    float t = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) t += red[k][lane];
    out[c] = t;
  }
}

// Block (x, y): columns [1024 x, 1024 x + 1024) (4 per thread), rows of chunk y.
template <typename T>
__global__ void colsum_partials_kernel(const T* __restrict__ in, int64_t ld, float* __restrict__ part, int64_t N,
                                       int64_t C, int rows_per_block) {
  const int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (c >= C) return;
  const int64_t r0 = (int64_t)blockIdx.y * rows_per_block;
  const int64_t r1 = min(N, r0 + rows_per_block);
  float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int64_t r = r0; r < r1; ++r) {
    float v[4];
    load4(in + r * ld + c, v);
#pragma unroll
    for (int j = 0; j < 4; ++j) s[j] += v[j];
  }
  store4(part + (int64_t)blockIdx.y * C + c, s);
}

// ------------------------------------------------------------- loss
template <typename T>
__global__ void __launch_bounds__(256) mse_loss_grad_kernel(const T* __restrict__ y, const T* __restrict__ tg,
                                                            T* __restrict__ dy, double* __restrict__ part, int64_t n,
                                                            float inv_count) {
  constexpr int V = Vec<T>::N;
  __shared__ double red[8];
  const int64_t nv = n / V;
  double acc = 0.0;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nv; v += (int64_t)gridDim.x * blockDim.x) {
    float a[V], b[V], o[V];
    Vec<T>::load(y + v * V, a);
    Vec<T>::load(tg + v * V, b);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const float d = a[j] - b[j];
      s = fmaf(d, d, s);
      o[j] = d * inv_count;
    }
    Vec<T>::store(dy + v * V, o);
    acc += (double)s;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int k = 0; k < 8; ++k) s += red[k];
    part[blockIdx.x] = s;
  }
}

__global__ void loss_finalize_kernel(const double* __restrict__ part, int nblocks, double scale,
                                     float* __restrict__ loss) {
  __shared__ double red[256];
  double s = 0.0;
  for (int i = threadIdx.x; i < nblocks; i += 256) s += part[i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = (float)(red[0] * scale);
}

// ------------------------------------------------------------- SGD
template <typename T>
__global__ void __launch_bounds__(256) sgd_kernel(const SgdArgs a) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int s = 0; s < a.nseg; ++s) {
    const SgdSeg sg = a.seg[s];
    const int64_t n4 = sg.n / 4;
    T* w = static_cast<T*>(sg.w);
    for (int64_t i = tid; i < n4; i += stride) {
      float g[4], v[4];
      load4(sg.grad + 4 * i, g);
      if (sg.master) {
        load4(sg.master + 4 * i, v);
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = fmaf(-a.lr, g[j], v[j]);
        store4(sg.master + 4 * i, v);
      } else {
        load4(w + 4 * i, v);
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = fmaf(-a.lr, g[j], v[j]);
      }
      store4(w + 4 * i, v);
    }
  }
}

}  // namespace

cudaError_t launch_rmsnorm_fwd(int dtype, const void* x, const void* w, float eps, void* nrm, float* rstd, int64_t N,
                               int64_t H, cudaStream_t st, uint32_t* amax) {
  if (N <= 0) return cudaSuccess;
  if (dtype == 0)
    return rmsnorm_fwd_t<float>((const float*)x, (const float*)w, eps, (float*)nrm, rstd, N, H, amax, st);
  return rmsnorm_fwd_t<__nv_bfloat16>((const __nv_bfloat16*)x, (const __nv_bfloat16*)w, eps, (__nv_bfloat16*)nrm,
                                      rstd, N, H, amax, st);
}

int rmsnorm_bwd_blocks(int64_t N, int num_sms, int shards) {
  int64_t b = 2LL * num_sms;  // one wave at two resident blocks per SM
  if (b > 1024) b = 1024;
  int64_t bps = b / shards;
  if (bps > N / shards) bps = N / shards;
  if (bps < 1) bps = 1;
  return (int)(bps * shards);
}

cudaError_t launch_rmsnorm_bwd(int dtype, const float* dnrm, const void* x, const float* rstd, const void* w,
                               const void* dy, void* dx, float* part_dw, float* part_db, int64_t N, int64_t H,
                               int shards, int nblocks, cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  if (shards < 1 || N % shards != 0 || nblocks % shards != 0) return cudaErrorInvalidValue;
  if (dtype == 0)
    return rmsnorm_bwd_t<float>(dnrm, (const float*)x, rstd, (const float*)w, (const float*)dy, (float*)dx, part_dw,
                                part_db, N, H, shards, nblocks, st);
  return rmsnorm_bwd_t<__nv_bfloat16>(dnrm, (const __nv_bfloat16*)x, rstd, (const __nv_bfloat16*)w,
                                      (const __nv_bfloat16*)dy, (__nv_bfloat16*)dx, part_dw, part_db, N, H, shards,
                                      nblocks, st);
}

cudaError_t launch_colsum_finalize(const float* part0, float* out0, const float* part1, float* out1, int nparts,
                                   int64_t C, cudaStream_t st, int groups) {
  if (C <= 0) return cudaSuccess;
  dim3 grid((unsigned)((C + 31) / 32), part1 ? 2u : 1u, (unsigned)groups);
  colsum_finalize_kernel<<<grid, 256, 0, st>>>(part0, out0, part1, out1, nparts, C);
  return cudaGetLastError();
}

int colsum_blocks(int64_t N, int num_sms) {
  int64_t b = num_sms;
  if (b > 256) b = 256;
  if (b > N) b = N;
  return (int)(b < 1 ? 1 : b);
}

cudaError_t launch_colsum_partials(int dtype, const void* in, int64_t ld, float* part, int64_t N, int64_t C,
                                   int nblocks, cudaStream_t st) {
  if (N <= 0 || C <= 0) return cudaSuccess;
  const int rpb = (int)((N + nblocks - 1) / nblocks);
  dim3 grid((unsigned)((C / 4 + 255) / 256), (unsigned)nblocks);
  if (dtype == 0)
    colsum_partials_kernel<float><<<grid, 256, 0, st>>>((const float*)in, ld, part, N, C, rpb);
  else
    colsum_partials_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)in, ld, part, N, C, rpb);
  return cudaGetLastError();
}

int loss_blocks(int64_t n, int num_sms) {
  int64_t b = (n / 8 + 255) / 256;
  if (b > 6LL * num_sms) b = 6LL * num_sms;
  if (b > 1024) b = 1024;
  return (int)(b < 1 ? 1 : b);
}

cudaError_t launch_mse_loss_grad(int dtype, const void* y, const void* target, void* dy, double* part, int nblocks,
                                 int64_t n, float inv_count, cudaStream_t st) {
  if (dtype == 0)
    mse_loss_grad_kernel<float><<<nblocks, 256, 0, st>>>((const float*)y, (const float*)target, (float*)dy, part, n,
                                                        inv_count);
  else
    mse_loss_grad_kernel<__nv_bfloat16><<<nblocks, 256, 0, st>>>(
        (const __nv_bfloat16*)y, (const __nv_bfloat16*)target, (__nv_bfloat16*)dy, part, n, inv_count);
  return cudaGetLastError();
}

cudaError_t launch_loss_finalize(const double* part, int nblocks, double scale, float* loss, cudaStream_t st) {
  loss_finalize_kernel<<<1, 256, 0, st>>>(part, nblocks, scale, loss);
  return cudaGetLastError();
}

cudaError_t launch_sgd(int dtype, const SgdArgs& a, int num_sms, cudaStream_t st) {
  int64_t tot = 0;
  for (int s = 0; s < a.nseg; ++s) tot += a.seg[s].n / 4;
  int64_t blocks = (tot + 255) / 256;
  if (blocks > 8LL * num_sms) blocks = 8LL * num_sms;
  if (blocks < 1) blocks = 1;
  if (dtype == 0)
    sgd_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(a);
  else
    sgd_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tpmlp
