// Element-wise math fused into the GEMM epilogues.
//
// Page "Megatron tensor-parallel MLP" ("Split the expansion"): the SwiGLU
// product SiLU(gate) * up is taken per FFN channel on the shard that owns it,
// so it needs no communication and sits in the column-parallel GEMM's
// epilogue.  ("Split the contraction"): bias and residual are added once,
// after the shard sum, in the row-parallel GEMM's epilogue.  The backward
// epilogues apply the derivative of the activation to dA = dy W_d.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "f32x2.cuh"

namespace tpmlp {

enum EpiKind : int {
  EPI_GATEUP_SWIGLU = 0,  // acc = [G | U] of 128 channels: store G, U, A = SiLU(G) * U
  EPI_FC1_GELU = 1,       // Z = acc + b_1: store Z, A = GeLU(Z)
  EPI_DOWN_RESID = 2,     // y = x + acc + b_down
  EPI_DGRAD_SWIGLU = 3,   // dA = acc: store dG = dA U SiLU'(G), dU = dA SiLU(G)
  EPI_DGRAD_GELU = 4,     // dZ = acc * GeLU'(Z)
  EPI_STORE_F32 = 5,      // out = acc (float)
  EPI_STORE_BF16 = 6      // out = acc (bf16)
};

// Pointers and leading dimensions (in elements) of the epilogue's operands.
//  GATEUP_SWIGLU: out0 = GU [M, 2F] (G in [0,F), U in [F,2F)), out1 = A [M, F]
//  FC1_GELU     : out0 = Z [M, F], out1 = A [M, F], vec = b_1 [F]
//  DOWN_RESID   : out0 = y [M, H], in0 = x [M, H], vec = b_down [H]
//  DGRAD_SWIGLU : in0 = GU [M, 2F], out0 = dGU [M, 2F]
//  DGRAD_GELU   : in0 = Z [M, F], out0 = dZ [M, F]
//  STORE_F32    : out0 = float [M, N]
//  STORE_BF16   : out0 = bf16 [M, N] (tensor-core path only)
struct EpiParams {
  void* out0;
  void* out1;
  const void* in0;
  const void* vec;
  int64_t ld_out0, ld_out1, ld_in0;
  int64_t pair_off;  // F: column offset of U / dU in the paired layouts
  int M, N;          // valid output rows / columns (channels for the paired layouts)
  // STORE_F32 / STORE_BF16: extent of the whole output tensor (rows x cols),
  // which a batched problem fills block by block; 0 = M x N.
  int64_t out_rows, out_cols;
  // Optional (tensor-core path): the largest magnitude of the activation
  // output (A, or dG and dU, or dZ) after bf16 rounding, as float bits,
  // combined with atomicMax (the caller zeroes it first).
  uint32_t* amax;
  // Optional (tensor-core STORE_F32 of a weight gradient): the SGD update
  // applied where the gradient is produced.  Each output element g also sets
  // master = fmaf(-sgd_lr, g, master) and writes the new master rounded to
  // bf16 (nearest even) into sgd_w; both are row-major with leading dimension
  // sgd_ld and indexed like the output.
  float* sgd_master;
  __nv_bfloat16* sgd_w;
  int64_t sgd_ld;
  float sgd_lr;
};

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }
__device__ __forceinline__ float silu_f(float z) { return z * sigmoid_f(z); }
// Exact (erf) GeLU and its derivative Phi(z) + z phi(z).
__device__ __forceinline__ float gelu_f(float z) { return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f)); }
__device__ __forceinline__ float gelu_grad_f(float z) {
  return 0.5f * (1.0f + erff(z * 0.70710678118654752f)) + z * expf(-0.5f * z * z) * 0.39894228040143268f;
}
// SwiGLU backward for one channel: (dG, dU) from dA, G, U.
__device__ __forceinline__ void swiglu_bwd(float da, float g, float u, float& dg, float& du) {
  const float s = sigmoid_f(g);
  dg = da * u * s * (1.0f + g * (1.0f - s));
  du = da * g * s;
}

// Fast variants for the bf16 tensor-core epilogues, whose results are stored
// in bf16 (relative rounding 2^-9): __expf and the approximate division
// (errors of a few ulp of float) are far inside that; for z -> -inf the
// sigmoid is 0, not NaN.  The fp32 path keeps expf and IEEE division.
__device__ __forceinline__ float sigmoid_fast(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }
__device__ __forceinline__ float silu_fast(float z) { return z * sigmoid_fast(z); }
__device__ __forceinline__ void swiglu_bwd_fast(float da, float g, float u, float& dg, float& du) {
  const float s = sigmoid_fast(g);
  dg = da * u * s * (1.0f + g * (1.0f - s));
  du = da * g * s;
}

// The same two formulas for a pair of channels with two-lane arithmetic:
// sigma(g) = 1 / (1 + 2^(-g log2 e)) from one ex2 and one rcp per channel,
// then dG = dA sigma U (1 + g (1 - sigma)) and dU = dA sigma g.  For
// g -> -inf sigma is 0 and for g -> +inf it is 1, as above.
__device__ __forceinline__ void swiglu_bwd_fast2(float da0, float da1, float g0, float g1, float u0, float u1,
                                                 float& dg0, float& dg1, float& du0, float& du1) {
  const uint64_t one = f2_pack(1.0f, 1.0f);
  const uint64_t g = f2_pack(g0, g1);
  float t0, t1;
  f2_unpack(f2_mul(g, f2_pack(-1.4426950408889634f, -1.4426950408889634f)), t0, t1);
  float d0, d1;
  f2_unpack(f2_add(f2_pack(ex2_fast(t0), ex2_fast(t1)), one), d0, d1);
  const uint64_t s = f2_pack(rcp_fast(d0), rcp_fast(d1));
  const uint64_t das = f2_mul(f2_pack(da0, da1), s);
  f2_unpack(f2_mul(das, g), du0, du1);
  const uint64_t w = f2_fma(g, f2_fma(s, f2_pack(-1.0f, -1.0f), one), one);  // 1 + g (1 - sigma)
  f2_unpack(f2_mul(f2_mul(das, f2_pack(u0, u1)), w), dg0, dg1);
}

// Phi(z) and exp(-z^2/2) for the bf16 tensor-core epilogues.  erf comes from
// the rational approximation of Abramowitz & Stegun, Handbook of
// Mathematical Functions, eq. 7.1.26: for x >= 0, erf(x) = 1 - t P(t)
// e^(-x^2) with t = 1 / (1 + p x), |error| <= 1.5e-7, extended to x < 0 by
// oddness; here x = |z| / sqrt(2), so e^(-x^2) = e^(-z^2/2) serves the
// density too.  Results are stored in bf16 (2^-9 relative), far coarser
// than the approximation.  The fp32 path keeps erff / expf.
__device__ __forceinline__ void gauss_fast(float z, float& Phi, float& e) {
  const float x = fabsf(z) * 0.70710678118654752f;
  const float t = rcp_fast(fmaf(0.3275911f, x, 1.0f));
  const float tp =
      t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f), -0.284496736f),
               0.254829592f);
  e = ex2_fast(-1.4426950408889634f * x * x);
  Phi = fmaf(0.5f, copysignf(fmaf(-tp, e, 1.0f), z), 0.5f);
}
// GeLU(z) = z Phi(z) and GeLU'(z) = Phi(z) + z phi(z), phi(z) = e^(-z^2/2) / sqrt(2 pi).
__device__ __forceinline__ float gelu_fast(float z) {
  float P, e;
  gauss_fast(z, P, e);
  return z * P;
}
__device__ __forceinline__ float gelu_grad_fast(float z) {
  float P, e;
  gauss_fast(z, P, e);
  return fmaf(z * 0.39894228040143268f, e, P);
}

// SiLU(g) u for a pair of channels: g sigma(g) u.
__device__ __forceinline__ void swiglu_fwd_fast2(float g0, float g1, float u0, float u1, float& a0, float& a1) {
  const uint64_t g = f2_pack(g0, g1);
  float t0, t1;
  f2_unpack(f2_mul(g, f2_pack(-1.4426950408889634f, -1.4426950408889634f)), t0, t1);
  float d0, d1;
  f2_unpack(f2_add(f2_pack(ex2_fast(t0), ex2_fast(t1)), f2_pack(1.0f, 1.0f)), d0, d1);
  f2_unpack(f2_mul(f2_mul(g, f2_pack(u0, u1)), f2_pack(rcp_fast(d0), rcp_fast(d1))), a0, a1);
}

// One output element (m, n) of the fp32 SIMT path.  For GATEUP_SWIGLU, `acc`
// is G and `acc2` is U of channel n.
template <int EPI, typename T>
__device__ __forceinline__ void epi_elem(const EpiParams& p, int m, int n, float acc, float acc2) {
  const int64_t mm = m;
  if (EPI == EPI_GATEUP_SWIGLU) {
    T* gu = static_cast<T*>(p.out0);
    gu[mm * p.ld_out0 + n] = from_f<T>(acc);
    gu[mm * p.ld_out0 + p.pair_off + n] = from_f<T>(acc2);
    static_cast<T*>(p.out1)[mm * p.ld_out1 + n] = from_f<T>(silu_f(acc) * acc2);
  } else if (EPI == EPI_FC1_GELU) {
    const float z = acc + to_f(static_cast<const T*>(p.vec)[n]);
    static_cast<T*>(p.out0)[mm * p.ld_out0 + n] = from_f<T>(z);
    static_cast<T*>(p.out1)[mm * p.ld_out1 + n] = from_f<T>(gelu_f(z));
  } else if (EPI == EPI_DOWN_RESID) {
    const float x = to_f(static_cast<const T*>(p.in0)[mm * p.ld_in0 + n]);
    const float b = to_f(static_cast<const T*>(p.vec)[n]);
    static_cast<T*>(p.out0)[mm * p.ld_out0 + n] = from_f<T>(x + acc + b);
  } else if (EPI == EPI_DGRAD_SWIGLU) {
    const T* gu = static_cast<const T*>(p.in0);
    float dg, du;
    swiglu_bwd(acc, to_f(gu[mm * p.ld_in0 + n]), to_f(gu[mm * p.ld_in0 + p.pair_off + n]), dg, du);
    T* o = static_cast<T*>(p.out0);
    o[mm * p.ld_out0 + n] = from_f<T>(dg);
    o[mm * p.ld_out0 + p.pair_off + n] = from_f<T>(du);
  } else if (EPI == EPI_DGRAD_GELU) {
    const float z = to_f(static_cast<const T*>(p.in0)[mm * p.ld_in0 + n]);
    static_cast<T*>(p.out0)[mm * p.ld_out0 + n] = from_f<T>(acc * gelu_grad_f(z));
  } else {
    static_cast<float*>(p.out0)[mm * p.ld_out0 + n] = acc;
  }
}

}  // namespace tpmlp
