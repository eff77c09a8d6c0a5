// Slot-to-slot state copies: copy-on-write restore and standalone snapshots.
//
// Source: "SGLang and Miles: day-0 support for Kimi K3", section "hybrid KDA memory management",
// "three state movements on the forward stream": every state copy is a kernel on the serial forward
// stream, between the forward passes that produce and consume the state, so stream order provides the
// happens-before relation.
//
// Each CTA moves 16 KB of one slot pair with 128-bit streaming loads issued before the stores.
#include "common.cuh"
#include "launch.h"

namespace kda {

constexpr int COPY_NT = 256;
constexpr int COPY_VEC_PER_THREAD = 4;
constexpr int COPY_VEC_PER_CTA = COPY_NT * COPY_VEC_PER_THREAD;

__global__ void __launch_bounds__(COPY_NT) state_copy_kernel(const float* __restrict__ src, int src_num_slots,
                                                             const int32_t* __restrict__ src_slots,
                                                             float* __restrict__ dst, int dst_num_slots,
                                                             const int32_t* __restrict__ dst_slots,
                                                             int64_t state_vec4, int32_t* status) {
  const int i = blockIdx.y;
  const int ss = src_slots[i], ds = dst_slots[i];
  if (ss < 0 || ss >= src_num_slots || ds < 0 || ds >= dst_num_slots) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag_status(status, KDA_DEV_SLOT_OOB);
    return;
  }
  const float4* s4 = reinterpret_cast<const float4*>(src) + (size_t)ss * state_vec4;
  float4* d4 = reinterpret_cast<float4*>(dst) + (size_t)ds * state_vec4;
  const int64_t base = (int64_t)blockIdx.x * COPY_VEC_PER_CTA + threadIdx.x;
  float4 buf[COPY_VEC_PER_THREAD];
#pragma unroll
  for (int u = 0; u < COPY_VEC_PER_THREAD; ++u) {
    const int64_t e = base + (int64_t)u * COPY_NT;
    if (e < state_vec4) buf[u] = __ldcs(s4 + e);
  }
#pragma unroll
  for (int u = 0; u < COPY_VEC_PER_THREAD; ++u) {
    const int64_t e = base + (int64_t)u * COPY_NT;
    if (e < state_vec4) __stcs(d4 + e, buf[u]);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) add_work(status, 1);
}

cudaError_t launch_state_copy(const CopyArgs& a, cudaStream_t s) {
  if (a.n == 0) return cudaSuccess;
  const int64_t vec4 = a.state_elems / 4;
  const int64_t gx = (vec4 + COPY_VEC_PER_CTA - 1) / COPY_VEC_PER_CTA;
  if (gx > 0x7fffffff) return cudaErrorInvalidValue;
  for (int off = 0; off < a.n; off += 65535) {  // grid.y is limited to 65535 pairs per launch
    const int cnt = (a.n - off) < 65535 ? (a.n - off) : 65535;
    dim3 grid((unsigned)gx, (unsigned)cnt);
    state_copy_kernel<<<grid, COPY_NT, 0, s>>>(a.src, a.src_num_slots, a.src_slots + off, a.dst, a.dst_num_slots,
                                               a.dst_slots + off, vec4, a.status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kda
