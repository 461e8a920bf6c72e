// Exact-fp32 GEMM on the CUDA cores for the float configuration of the
// sublayer (tf32 tensor cores cannot meet a 1e-5 relative tolerance).  Same
// operand conventions, contraction segments and fused epilogues as the
// tensor-core path, so the float and bf16 configurations compute the same
// steps in the same order.
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "ptx_sm103.cuh"
#include "tpmlp_internal.h"

namespace tpmlp {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

struct SimtParams {
  const float* a;
  const float* b;
  int64_t lda, ldb;
  int a_mn, b_mn;
  int M, N;
  int paired;
  int64_t pair_off;
  int64_t kseg[4];
  EpiParams ep;
};

template <int EPI>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const SimtParams p) {
  __shared__ float As[TK][TM + 1];
  __shared__ float Bs[TK][TN + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * TM;
  // paired: a tile covers 32 channels, B columns [0,32) are gate rows and
  // [32,64) the matching up rows.
  const int ch0 = p.paired ? blockIdx.x * (TN / 2) : blockIdx.x * TN;
  float acc[4][4] = {};
  for (int s = 0; s < 2; ++s) {
    for (int64_t k0 = p.kseg[2 * s]; k0 < p.kseg[2 * s + 1]; k0 += TK) {
      const int64_t kend = p.kseg[2 * s + 1];
      for (int e = threadIdx.x; e < TK * TM; e += 256) {
        const int kk = e / TM, mm = e % TM;
        const int64_t k = k0 + kk;
        const int m = m0 + mm;
        float v = 0.0f;
        if (k < kend && m < p.M) v = p.a_mn ? p.a[k * p.lda + m] : p.a[(int64_t)m * p.lda + k];
        As[kk][mm] = v;
      }
      for (int e = threadIdx.x; e < TK * TN; e += 256) {
        const int kk = e / TN, c = e % TN;
        const int64_t k = k0 + kk;
        int64_t brow;
        bool valid;
        if (p.paired) {
          const int ch = ch0 + (c & (TN / 2 - 1));
          valid = ch < p.N;
          brow = (c < TN / 2 ? 0 : p.pair_off) + ch;
        } else {
          brow = ch0 + c;
          valid = brow < p.N;
        }
        float v = 0.0f;
        if (k < kend && valid) v = p.b_mn ? p.b[k * p.ldb + brow] : p.b[brow * p.ldb + k];
        Bs[kk][c] = v;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < TK; ++kk) {
        float av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = As[kk][ty + 16 * i];
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx + 16 * j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= p.M) continue;
    if (p.paired) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int ch = ch0 + tx + 16 * j;
        if (ch < p.N) epi_elem<EPI, float>(p.ep, m, ch, acc[i][j], acc[i][j + 2]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = ch0 + tx + 16 * j;
        if (n < p.N) epi_elem<EPI, float>(p.ep, m, n, acc[i][j], 0.0f);
      }
    }
  }
}

__global__ void timeout_probe_kernel(uint32_t* status) {
  // Waits for status[1] to become non-zero, which nothing does, then gives up.
  volatile uint32_t* flag = status + 1;
  const uint64_t t0 = global_timer_ns();
  while (*flag == 0) {
    if (global_timer_ns() - t0 > 2000000ull) {
      atomicOr(status, STATUS_TIMEOUT);
      return;
    }
  }
}

}  // namespace

cudaError_t launch_gemm_simt_f32(const GemmDesc& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  SimtParams p{};
  p.a = static_cast<const float*>(g.a);
  p.b = static_cast<const float*>(g.b);
  p.lda = g.lda;
  p.ldb = g.ldb;
  p.a_mn = g.a_mn;
  p.b_mn = g.b_mn;
  p.M = g.M;
  p.N = g.N;
  p.paired = g.paired;
  p.pair_off = g.pair_off;
  for (int i = 0; i < 4; ++i) p.kseg[i] = g.kseg[i];
  p.ep = g.ep;
  p.ep.M = g.M;
  p.ep.N = g.N;
  const int tn = g.paired ? TN / 2 : TN;
  dim3 grid((g.N + tn - 1) / tn, (g.M + TM - 1) / TM);
  switch (g.epi) {
    case EPI_GATEUP_SWIGLU: gemm_simt_kernel<EPI_GATEUP_SWIGLU><<<grid, 256, 0, st>>>(p); break;
    case EPI_FC1_GELU: gemm_simt_kernel<EPI_FC1_GELU><<<grid, 256, 0, st>>>(p); break;
    case EPI_DOWN_RESID: gemm_simt_kernel<EPI_DOWN_RESID><<<grid, 256, 0, st>>>(p); break;
    case EPI_DGRAD_SWIGLU: gemm_simt_kernel<EPI_DGRAD_SWIGLU><<<grid, 256, 0, st>>>(p); break;
    case EPI_DGRAD_GELU: gemm_simt_kernel<EPI_DGRAD_GELU><<<grid, 256, 0, st>>>(p); break;
    default: gemm_simt_kernel<EPI_STORE_F32><<<grid, 256, 0, st>>>(p); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_timeout_probe(uint32_t* status, cudaStream_t st) {
  timeout_probe_kernel<<<1, 1, 0, st>>>(status);
  return cudaGetLastError();
}

}  // namespace tpmlp
