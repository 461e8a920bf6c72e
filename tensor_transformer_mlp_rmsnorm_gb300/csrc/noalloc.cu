// MSE loss and its gradient for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a host framework may own every byte of
// device memory through its own pool and budget (a raw allocation would count
// outside it or fail), and cudaMalloc may synchronise the device, which a
// latency-bound serving loop cannot afford.  Such callers can still hand over
// their inputs and outputs.  This entry point runs the same loss kernels as
// tpmlp_mse_loss_grad, but keeps the per-block partial sums in a fixed array
// that lives in the library itself, so no workspace is needed.
//
// The array belongs to every GPU that loads the library, until the process
// exits.  All calls share it: two calls whose kernels overlap on the GPU
// (different streams, or different host threads) race on it.  Each call
// writes every partial it later reads, so nothing has to be cleared between
// calls.  Its device address is looked up once per device and kept for the
// life of the process, so the entry point must not be used on a device after
// cudaDeviceReset.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/tpmlp.h"
#include "tpmlp_internal.h"

namespace {

// One double per block of the loss kernel's grid.  The grid is capped at
// kMaxBlocks blocks that stride over all n elements, so the array bounds the
// number of partial sums, not n.
constexpr int64_t kMaxBlocks = TPMLP_NOALLOC_LOSS_MAX_BLOCKS;
static __device__ __align__(256) double g_loss_partials[kMaxBlocks];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
double* g_partials_addr[kMaxDevices] = {};

// Device address of g_loss_partials on the current device.  In host code the
// symbol is only a host-side stand-in, never a device address, so it is looked
// up once per device with that device current.
tpmlp_status partials_on_current_device(double** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    tpmlp::set_thread_error(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    return TPMLP_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    tpmlp::set_thread_error("device index out of range");
    return TPMLP_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_partials_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_loss_partials);
    if (e != cudaSuccess || !p) {
      tpmlp::set_thread_error(std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
      return TPMLP_ERR_CUDA;
    }
    g_partials_addr[dev] = static_cast<double*>(p);
  }
  *out = g_partials_addr[dev];
  return TPMLP_OK;
}

}  // namespace

extern "C" tpmlp_status tpmlp_mse_loss_grad_noalloc(int32_t dtype, int64_t n, const void* y, const void* target,
                                                    void* dy, float* loss_dev, void* cuda_stream) {
  if (dtype != TPMLP_F32 && dtype != TPMLP_BF16) {
    tpmlp::set_thread_error("unknown dtype");
    return TPMLP_ERR_UNSUPPORTED;
  }
  if (n < 0 || n % 8 != 0) {
    tpmlp::set_thread_error("n must be >= 0 and a multiple of 8");
    return TPMLP_ERR_SHAPE;
  }
  // One block per 256 vectors of 16 bytes, capped at the array's size; the
  // loss kernel strides over the vectors, so the capped grid covers any n.
  const int64_t per_block = 256LL * (dtype == TPMLP_BF16 ? 8 : 4);
  const int64_t blocks = (n + per_block - 1) / per_block;
  const int grid = (int)(blocks < kMaxBlocks ? blocks : kMaxBlocks);
  if (!loss_dev || (n > 0 && (!y || !target || !dy))) {
    tpmlp::set_thread_error("NULL tensor");
    return TPMLP_ERR_ARG;
  }
  for (const void* p : {y, target, (const void*)dy})
    if (reinterpret_cast<uintptr_t>(p) & 15u) {
      tpmlp::set_thread_error("tensor not 16-byte aligned");
      return TPMLP_ERR_ARG;
    }
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e;
  if (n == 0) {
    e = cudaMemsetAsync(loss_dev, 0, sizeof(float), st);
  } else {
    double* part = nullptr;
    const tpmlp_status s = partials_on_current_device(&part);
    if (s != TPMLP_OK) return s;
    const int dt = dtype == TPMLP_BF16 ? 1 : 0;
    e = tpmlp::launch_mse_loss_grad(dt, y, target, dy, part, grid, n, (float)(1.0 / (double)n), st);
    if (e == cudaSuccess) e = tpmlp::launch_loss_finalize(part, grid, 0.5 / (double)n, loss_dev, st);
  }
  if (e != cudaSuccess) {
    tpmlp::set_thread_error(std::string("tpmlp_mse_loss_grad_noalloc: ") + cudaGetErrorString(e));
    return TPMLP_ERR_CUDA;
  }
  return TPMLP_OK;
}
