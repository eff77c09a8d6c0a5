// Shared device helpers of the KDA CUDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

using bf16 = __nv_bfloat16;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// Reports a device-detected problem into the optional status word.
__device__ __forceinline__ void flag_status(int32_t* st, int32_t f) {
  if (st) atomicOr(st, f);
}
__device__ __forceinline__ void add_work(int32_t* st, int32_t n) {
  if (st && n) atomicAdd(reinterpret_cast<unsigned int*>(st + 1), static_cast<unsigned int>(n));
}

// Streaming (evict-first) 128-bit global accesses for state tiles that are touched once per launch.
__device__ __forceinline__ float4 ld_stream(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st_stream(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }

}  // namespace kda
