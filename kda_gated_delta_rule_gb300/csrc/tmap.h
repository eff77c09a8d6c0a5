// Host-side encoding of TMA tensor maps for token-major [rows][H][128] tensors (bf16 or fp32).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace kda {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [rows][H][128] tensor; box = 128 channels x 1 head x box_rows rows, no swizzle, zero fill outside.
// Returns false when the driver entry point is missing or rejects the description.
inline bool encode_token_map(CUtensorMap* map, const void* base, bool f32, long long rows, int H, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t es = f32 ? 4 : 2, D = 128;
  const cuuint64_t dims[3] = {D, (cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {D * es, (cuuint64_t)H * D * es};
  const cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [rows][H][128] tensor; box = 64 channels x 1 head x box_rows rows with the 128-byte swizzle: a load at
// x = 0 (channels 0..63) or x = 64 lands as a [box_rows][64] tile whose row r sits at r * 128 bytes with its
// 16-byte chunks permuted by r % 8 (the tensor cores' 128-byte-swizzled operand layout; the destination
// must be 1024-byte aligned).  Zero fill outside the tensor.
inline bool encode_token_map_sw128(CUtensorMap* map, const void* base, long long rows, int H, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t es = 2, D = 128;
  const cuuint64_t dims[3] = {D, (cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {D * es, (cuuint64_t)H * D * es};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace kda
