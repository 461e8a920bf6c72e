// Host-side TMA tensor-map encoding for the tcgen05 kernels (2-D K-major
// operand boxes with the 128-byte swizzle, 3-D MN-major boxes, 32x32 epilogue
// boxes).  The driver entry point is looked up once through the runtime.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace tpmlp {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

enum ElemKind { EK_BF16 = 0, EK_F32 = 1, EK_U8 = 2 };

// 2-D tensor [outer, inner] with row pitch `ld` elements.
inline bool encode_map(CUtensorMap* m, const void* ptr, int ek, uint64_t inner, uint64_t outer, uint64_t ld,
                uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const uint64_t esz = ek == EK_F32 ? 4 : (ek == EK_U8 ? 1 : 2);
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * esz};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = ek == EK_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : (ek == EK_U8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  CUresult r = enc(m, dt, 2,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 operand: boxes of 64 (one 128-byte swizzle row) x box_outer.
inline bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_outer) {
  return encode_map(m, ptr, EK_BF16, inner, outer, ld, 64, box_outer, CU_TENSOR_MAP_SWIZZLE_128B);
}

// E4M3 K-major operand: boxes of 128 codes (one 128-byte swizzle row) x box_outer.
inline bool make_map_u8(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_outer) {
  return encode_map(m, ptr, EK_U8, inner, outer, ld, 128, box_outer, CU_TENSOR_MAP_SWIZZLE_128B);
}

// MN-major bf16 operand [k_extent, mn] (pitch ld, mn a multiple of 64) as a
// 3-D tensor {64, k_extent, mn / 64}: one box of `chunks` 64-element MN
// chunks x 64 K rows lands in shared memory exactly as `chunks` 2-D boxes
// placed 8 KB apart would.
inline bool make_mn_map3(CUtensorMap* m, const void* ptr, uint64_t mn, uint64_t k_extent, uint64_t ld, uint32_t chunks) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc || mn % 64 != 0) return false;
  cuuint64_t dims[3] = {64, k_extent, mn / 64};
  cuuint64_t strides[2] = {ld * 2, 128};
  cuuint32_t box[3] = {64, 64, chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Epilogue output [rows, cols] (pitch ld): 32x32 boxes, 64-byte swizzle for
// bf16 rows, 128-byte swizzle for f32 rows (the staging-tile layouts).
inline bool make_out_map(CUtensorMap* m, const void* ptr, bool f32, uint64_t cols, uint64_t rows, uint64_t ld) {
  return encode_map(m, ptr, f32 ? EK_F32 : EK_BF16, cols, rows, ld, 32, 32,
                    f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

}  // namespace tpmlp
