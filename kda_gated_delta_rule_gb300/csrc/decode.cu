// Decode step, speculative verify and replay fold.
//
// Sources: "Kimi K3: Architecture and SGLang Day-0 Support", KDA math box (the per-token update);
// "SGLang and Miles: day-0 support for Kimi K3", section "ReplaySSM: raw-input replay for KDA state"
// (verify reads the committed checkpoint and never writes it, storing each step's raw inputs
// (v, k, gk, beta); the fold replays only the accepted prefix in place with the stored gate values, so
// the rebuilt state is bit-identical to the recurrence baseline).
//
// One CTA per (request, head) holds the whole D x D state in registers (D/16 warps, each owning 16 value
// columns; 128-bit loads of row segments), so each 64 KB state (D = 128) is read once and written at most
// once per launch.  The window's inputs are staged in shared memory before the dependent token steps.
#include "device.h"
#include "launch.h"
#include "tc_ptx.cuh"
#include "wstep.cuh"

namespace kda {

// Tokens of a window staged in shared memory at once (processed in groups of WGRP) by all threads, so
// the dependent per-token steps never wait on global memory; one block barrier per group.
constexpr int WGRP = 8;

// Raw bits of a group of window tokens, as loaded from global memory.
template <int D, typename Tin>
struct __align__(16) RawGroup {
  alignas(16) Tin k[WGRP][D];
  alignas(16) Tin q[WGRP][D];
  alignas(16) Tin v[WGRP][D];
  alignas(16) float g[WGRP][D];
  float beta[WGRP];
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Issues asynchronous copies of tokens row0 + u * rstride, u < cnt (element offset row * D), into `raw`.
// No registers are held while the copies are in flight.
template <int D, typename Tin, bool WITH_Q>
__device__ __forceinline__ void fetch_tokens(RawGroup<D, Tin>* raw, const Tin* k, const Tin* q, const Tin* v,
                                             const float* g, const float* beta, size_t row0, size_t rstride,
                                             int cnt, int tid, int nt) {
  constexpr int CH = D * (int)sizeof(Tin) / 16;  // 16-byte chunks per row of k, q, v
  constexpr int CG = D * 4 / 16;                 // per row of g
  for (int e = tid; e < cnt * (3 * CH + CG); e += nt) {
    const int u = e / (3 * CH + CG), r = e % (3 * CH + CG);
    const size_t off = (row0 + (size_t)u * rstride) * D;
    if (r < CH) {
      cp_async16(reinterpret_cast<uint8_t*>(raw->k[u]) + 16 * r, reinterpret_cast<const uint8_t*>(k + off) + 16 * r);
    } else if (r < 2 * CH) {
      if (WITH_Q)
        cp_async16(reinterpret_cast<uint8_t*>(raw->q[u]) + 16 * (r - CH),
                   reinterpret_cast<const uint8_t*>(q + off) + 16 * (r - CH));
    } else if (r < 3 * CH) {
      cp_async16(reinterpret_cast<uint8_t*>(raw->v[u]) + 16 * (r - 2 * CH),
                 reinterpret_cast<const uint8_t*>(v + off) + 16 * (r - 2 * CH));
    } else {
      cp_async16(reinterpret_cast<uint8_t*>(raw->g[u]) + 16 * (r - 3 * CH),
                 reinterpret_cast<const uint8_t*>(g + off) + 16 * (r - 3 * CH));
    }
  }
  if (tid < cnt) cp_async4(&raw->beta[tid], beta + row0 + (size_t)tid * rstride);
}

// Converts a fetched group into the step's fp32 token layout and, with RECORD, writes the raw bits of
// (k, v, g, beta) to the replay record.  Call after cp_async_wait_all and a barrier.
template <int D, typename Tin, bool WITH_Q, bool RECORD>
__device__ __forceinline__ void unpack_tokens(WTok<D>* tok, const RawGroup<D, Tin>* raw, size_t row0, size_t rstride,
                                              int cnt, int tid, const ReplayPtrs* rec) {
  if (tid < D) {
    const int pj = wperm(tid, D);  // lane order of the warp step
#pragma unroll
    for (int u = 0; u < WGRP; ++u) {
      if (u < cnt) {
        const Tin kv = raw->k[u][tid], vv = raw->v[u][tid];
        const float gv = raw->g[u][tid];
        tok[u].k[pj] = to_f32(kv);
        if (WITH_Q) tok[u].q[pj] = to_f32(raw->q[u][tid]);
        tok[u].a[pj] = expf(gv);
        tok[u].v[tid] = to_f32(vv);
        if (RECORD) {
          const size_t e = (row0 + u * rstride) * D + tid;
          static_cast<Tin*>(rec->k)[e] = kv;
          static_cast<Tin*>(rec->v)[e] = vv;
          rec->g[e] = gv;
        }
      }
    }
  } else if (tid < D + WGRP) {
    const int u = tid - D;
    if (u < cnt) {
      tok[u].beta = raw->beta[u];
      if (RECORD) rec->beta[row0 + u * rstride] = raw->beta[u];
    }
  }
}

template <int D, typename Tin, typename Tout>
__global__ void __launch_bounds__(WCfg<D>::NT, 2) decode_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                                 const Tin* __restrict__ v,
                                                                 const float* __restrict__ g,
                                                                 const float* __restrict__ beta, int H, float* pool,
                                                                 int num_slots, const int32_t* __restrict__ slot_ids,
                                                                 Tout* __restrict__ out, int32_t* status) {
  __shared__ WTok<D> tok[1];
  __shared__ RawGroup<D, Tin> raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int slot = slot_ids[b];
  if (slot < 0 || slot >= num_slots) {
    if (tid == 0) flag_status(status, KDA_DEV_SLOT_OOB);
    return;
  }
  float* Sg = pool + ((size_t)slot * H + h) * D * D;
  const size_t row = (size_t)b * H + h;
  fetch_tokens<D, Tin, true>(&raw, k, q, v, g, beta, row, 0, 1, tid, WCfg<D>::NT);
  float2 S[WRows<D>::P][4];
  wload<D>(S, Sg, warp, lane);
  cp_async_wait_all();
  __syncthreads();
  unpack_tokens<D, Tin, true, false>(tok, &raw, row, 0, 1, tid, nullptr);
  __syncthreads();
  const float o = wstep<D, true>(S, tok[0], warp, lane);
  if (((lane >> 2) & 1) == 0) out[row * D + wstep_out_col(warp, lane)] = from_f32<Tout>(o);
  wstore<D>(S, Sg, warp, lane);
  if (tid == 0) add_work(status, 1);
}

template <int D, typename Tin, typename Tout>
__global__ void __launch_bounds__(WCfg<D>::NT, 2) verify_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                                 const Tin* __restrict__ v,
                                                                 const float* __restrict__ g,
                                                                 const float* __restrict__ beta, int W, int H,
                                                                 const float* __restrict__ pool, int num_slots,
                                                                 const int32_t* __restrict__ slot_ids,
                                                                 Tout* __restrict__ out, ReplayPtrs rec,
                                                                 float* __restrict__ snapshot_out, int32_t* status) {
  __shared__ WTok<D> tok[WGRP];
  __shared__ RawGroup<D, Tin> raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int slot = slot_ids[b];
  if (slot < 0 || slot >= num_slots) {
    if (tid == 0) flag_status(status, KDA_DEV_SLOT_OOB);
    return;
  }
  float2 S[WRows<D>::P][4];
  for (int w0 = 0; w0 < W; w0 += WGRP) {
    const int cnt = W - w0 < WGRP ? W - w0 : WGRP;
    if (w0 > 0) __syncthreads();  // the previous group's steps have finished reading tok[]
    const size_t row0 = ((size_t)b * W + w0) * H + h;
    fetch_tokens<D, Tin, true>(&raw, k, q, v, g, beta, row0, H, cnt, tid, WCfg<D>::NT);
    if (w0 == 0) wload<D>(S, pool + ((size_t)slot * H + h) * D * D, warp, lane);
    cp_async_wait_all();
    __syncthreads();
    // the group's inputs, and their raw-input record: the exact stored bits the fold consumes
    unpack_tokens<D, Tin, true, true>(tok, &raw, row0, H, cnt, tid, &rec);
    __syncthreads();
    for (int u = 0; u < cnt; ++u) {
      const size_t row = row0 + (size_t)u * H;
      const float o = wstep<D, true>(S, tok[u], warp, lane);
      if (((lane >> 2) & 1) == 0) out[row * D + wstep_out_col(warp, lane)] = from_f32<Tout>(o);
      if (snapshot_out) wstore<D>(S, snapshot_out + row * D * D, warp, lane);
    }
  }
  if (tid == 0) add_work(status, W);
}

template <int D, typename Tin>
__global__ void __launch_bounds__(WCfg<D>::NT, 2) fold_kernel(float* pool, int num_slots,
                                                               const int32_t* __restrict__ slot_ids, int W, int H,
                                                               ReplayPtrs rec, const int32_t* __restrict__ accepted,
                                                               int32_t* status) {
  __shared__ WTok<D> tok[WGRP];
  __shared__ RawGroup<D, Tin> raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int n = accepted[b];
  if (n < 0 || n > W) {
    if (tid == 0) flag_status(status, KDA_DEV_ACCEPT_OOB);
    return;
  }
  if (n == 0) return;  // nothing accepted: the committed state stays as it is
  const int slot = slot_ids[b];
  if (slot < 0 || slot >= num_slots) {
    if (tid == 0) flag_status(status, KDA_DEV_SLOT_OOB);
    return;
  }
  float* Sg = pool + ((size_t)slot * H + h) * D * D;
  float2 S[WRows<D>::P][4];
  const Tin* rk = static_cast<const Tin*>(rec.k);
  const Tin* rv = static_cast<const Tin*>(rec.v);
  for (int w0 = 0; w0 < n; w0 += WGRP) {
    const int cnt = n - w0 < WGRP ? n - w0 : WGRP;
    if (w0 > 0) __syncthreads();
    const size_t row0 = ((size_t)b * W + w0) * H + h;
    fetch_tokens<D, Tin, false>(&raw, rk, nullptr, rv, rec.g, rec.beta, row0, H, cnt, tid, WCfg<D>::NT);
    if (w0 == 0) wload<D>(S, Sg, warp, lane);
    cp_async_wait_all();
    __syncthreads();
    unpack_tokens<D, Tin, false, false>(tok, &raw, row0, H, cnt, tid, nullptr);
    __syncthreads();
    for (int u = 0; u < cnt; ++u) wstep<D, false>(S, tok[u], warp, lane);
  }
  wstore<D>(S, Sg, warp, lane);
  if (tid == 0) add_work(status, n);
}

// The fold as a stream: two persistent CTAs per SM walk the (request, head) units with stride gridDim.x,
// skipping units with nothing accepted.  While a unit replays from registers, the next unit's state is on
// its way into shared memory (one bulk copy) and its recorded tokens follow with cp.async, so every SM
// keeps a state load in flight instead of starting each one cold.  The per-token arithmetic is the same
// wstep as decode and the one-unit-per-CTA fold, so the committed state stays bit-identical to n decode
// steps.  Windows of up to WGRP tokens, bf16 record.
template <int D, typename Tin>
struct FoldStreamSmem {
  static constexpr size_t STAGE = (size_t)D * D * 4;
  static constexpr size_t RAW = STAGE;
  static constexpr size_t TOK = RAW + 2 * sizeof(RawGroup<D, Tin>);
  static constexpr size_t BAR = TOK + WGRP * sizeof(WTok<D>);
  static constexpr size_t BYTES = BAR + 16;
};

template <int D, typename Tin>
__global__ void __launch_bounds__(WCfg<D>::NT, 2) fold_stream_kernel(float* pool, int num_slots,
                                                                      const int32_t* __restrict__ slot_ids, int W,
                                                                      int H, ReplayPtrs rec,
                                                                      const int32_t* __restrict__ accepted,
                                                                      int32_t* status, int units) {
  using L = FoldStreamSmem<D, Tin>;
  extern __shared__ __align__(128) uint8_t smem[];
  float* stage = reinterpret_cast<float*>(smem);
  RawGroup<D, Tin>* raw = reinterpret_cast<RawGroup<D, Tin>*>(smem + L::RAW);
  WTok<D>* tok = reinterpret_cast<WTok<D>*>(smem + L::TOK);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Tin* rk = static_cast<const Tin*>(rec.k);
  const Tin* rv = static_cast<const Tin*>(rec.v);
  // the first unit at or after u that has accepted tokens and a valid slot (every thread computes it)
  auto next_unit = [&](int u) {
    for (; u < units; u += (int)gridDim.x) {
      const int b = u / H, n = accepted[b];
      if (n < 0 || n > W) {
        if (tid == 0) flag_status(status, KDA_DEV_ACCEPT_OOB);
        continue;
      }
      if (n == 0) continue;
      const int slot = slot_ids[b];
      if (slot < 0 || slot >= num_slots) {
        if (tid == 0) flag_status(status, KDA_DEV_SLOT_OOB);
        continue;
      }
      break;
    }
    return u;
  };
  // requests unit u's state (thread 0) and its recorded tokens into raw[buf]
  auto prefetch = [&](int u, int buf) {
    const int b = u / H, h = u % H;
    if (tid == 0) {
      tc::bar_arrive_expect_tx(bar, (uint32_t)L::STAGE);
      tc::bulk_g2s(stage, pool + ((size_t)slot_ids[b] * H + h) * D * D, (uint32_t)L::STAGE, bar);
    }
    fetch_tokens<D, Tin, false>(raw + buf, rk, nullptr, rv, rec.g, rec.beta, ((size_t)b * W) * H + h, H, accepted[b],
                                tid, WCfg<D>::NT);
  };
  if (tid == 0) {
    tc::bar_init(bar, 1);
    tc::bar_fence_init();
  }
  __syncthreads();
  int u = next_unit((int)blockIdx.x);
  if (u < units) prefetch(u, 0);
  bool ok = true;
  float2 S[WRows<D>::P][4];
#pragma unroll 1
  for (int it = 0; u < units; ++it) {
    const int b = u / H, h = u % H, n = accepted[b];
    const int buf = it & 1;
    const bool landed = tc::bar_wait(bar, (uint32_t)it & 1u);
    cp_async_wait_all();
    ok = __syncthreads_and(landed) != 0;
    if (!ok) break;
    wload_shared<D>(S, stage, warp, lane);
    unpack_tokens<D, Tin, false, false>(tok, raw + buf, 0, 0, n, tid, nullptr);
    __syncthreads();  // the stage has been read and the tokens unpacked
    const int un = next_unit(u + (int)gridDim.x);
    if (un < units) prefetch(un, buf ^ 1);
    for (int t = 0; t < n; ++t) wstep<D, false>(S, tok[t], warp, lane);
    wstore<D>(S, pool + ((size_t)slot_ids[b] * H + h) * D * D, warp, lane);
    if (tid == 0) add_work(status, n);
    u = un;
  }
  if (!ok) {  // the state copy did not land in time: report it and give the copy one more bounded wait
    if (tid == 0) flag_status(status, KDA_DEV_TIMEOUT);
    tc::bar_wait(bar, 0u);
    tc::bar_wait(bar, 1u);
  }
}

// Decode as a stream, the same scheme as the fold stream: two persistent CTAs per SM walk the
// (request, head) units with stride gridDim.x; the next unit's state is bulk-copied into shared memory and
// its token follows with cp.async while the current unit steps and stores from registers.  The step is the
// same wstep as the one-unit-per-CTA decode, so outputs and state bits do not depend on which ran.
template <int D, typename Tin>
struct DecodeStreamSmem {
  static constexpr size_t STAGE = (size_t)D * D * 4;
  static constexpr size_t RAW = STAGE;
  static constexpr size_t TOK = RAW + 2 * sizeof(RawGroup<D, Tin>);
  static constexpr size_t BAR = TOK + sizeof(WTok<D>);
  static constexpr size_t BYTES = BAR + 16;
};

template <int D, typename Tin, typename Tout>
__global__ void __launch_bounds__(WCfg<D>::NT, 2) decode_stream_kernel(const Tin* __restrict__ q,
                                                                        const Tin* __restrict__ k,
                                                                        const Tin* __restrict__ v,
                                                                        const float* __restrict__ g,
                                                                        const float* __restrict__ beta, int H,
                                                                        float* pool, int num_slots,
                                                                        const int32_t* __restrict__ slot_ids,
                                                                        Tout* __restrict__ out, int32_t* status,
                                                                        int units) {
  using L = DecodeStreamSmem<D, Tin>;
  extern __shared__ __align__(128) uint8_t smem[];
  float* stage = reinterpret_cast<float*>(smem);
  RawGroup<D, Tin>* raw = reinterpret_cast<RawGroup<D, Tin>*>(smem + L::RAW);
  WTok<D>* tok = reinterpret_cast<WTok<D>*>(smem + L::TOK);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the first unit at or after u whose request has a valid slot (every thread computes it)
  auto next_unit = [&](int u) {
    for (; u < units; u += (int)gridDim.x) {
      const int slot = slot_ids[u / H];
      if (slot >= 0 && slot < num_slots) break;
      if (tid == 0) flag_status(status, KDA_DEV_SLOT_OOB);
    }
    return u;
  };
  // requests unit u's state (thread 0) and its token (row u of the [B, H] inputs) into raw[buf]
  auto prefetch = [&](int u, int buf) {
    if (tid == 0) {
      tc::bar_arrive_expect_tx(bar, (uint32_t)L::STAGE);
      tc::bulk_g2s(stage, pool + ((size_t)slot_ids[u / H] * H + u % H) * D * D, (uint32_t)L::STAGE, bar);
    }
    fetch_tokens<D, Tin, true>(raw + buf, k, q, v, g, beta, (size_t)u, 0, 1, tid, WCfg<D>::NT);
  };
  if (tid == 0) {
    tc::bar_init(bar, 1);
    tc::bar_fence_init();
  }
  __syncthreads();
  int u = next_unit((int)blockIdx.x);
  if (u < units) prefetch(u, 0);
  bool ok = true;
  float2 S[WRows<D>::P][4];
#pragma unroll 1
  for (int it = 0; u < units; ++it) {
    const int buf = it & 1;
    const bool landed = tc::bar_wait(bar, (uint32_t)it & 1u);
    cp_async_wait_all();
    ok = __syncthreads_and(landed) != 0;
    if (!ok) break;
    wload_shared<D>(S, stage, warp, lane);
    unpack_tokens<D, Tin, true, false>(tok, raw + buf, 0, 0, 1, tid, nullptr);
    __syncthreads();  // the stage has been read and the token unpacked
    const int un = next_unit(u + (int)gridDim.x);
    if (un < units) prefetch(un, buf ^ 1);
    const float o = wstep<D, true>(S, tok[0], warp, lane);
    if (((lane >> 2) & 1) == 0) out[(size_t)u * D + wstep_out_col(warp, lane)] = from_f32<Tout>(o);
    wstore<D>(S, pool + ((size_t)slot_ids[u / H] * H + u % H) * D * D, warp, lane);
    if (tid == 0) add_work(status, 1);
    u = un;
  }
  if (!ok) {  // the state copy did not land in time: report it and give the copy one more bounded wait
    if (tid == 0) flag_status(status, KDA_DEV_TIMEOUT);
    tc::bar_wait(bar, 0u);
    tc::bar_wait(bar, 1u);
  }
}

// ---------------------------------------------------------------- launchers

template <int D, typename Tin, typename Tout>
static cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
  decode_kernel<D, Tin, Tout><<<a.B * a.H, WCfg<D>::NT, 0, s>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v), a.g, a.beta, a.H,
      a.pool, a.num_slots, a.slot_ids, static_cast<Tout*>(a.out), a.status);
  return cudaGetLastError();
}

template <int D, typename Tin, typename Tout>
static cudaError_t launch_decode_stream_t(const DecodeArgs& a, cudaStream_t s) {
  using L = DecodeStreamSmem<D, Tin>;
  cudaError_t e = cudaFuncSetAttribute(decode_stream_kernel<D, Tin, Tout>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
  if (e != cudaSuccess) return e;
  const int units = a.B * a.H, sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = units < 2 * sms ? units : 2 * sms;
  decode_stream_kernel<D, Tin, Tout><<<grid, WCfg<D>::NT, L::BYTES, s>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v), a.g, a.beta, a.H,
      a.pool, a.num_slots, a.slot_ids, static_cast<Tout*>(a.out), a.status, units);
  return cudaGetLastError();
}

template <int D, typename Tin, typename Tout>
static cudaError_t launch_verify_t(const VerifyArgs& a, cudaStream_t s) {
  verify_kernel<D, Tin, Tout><<<a.B * a.H, WCfg<D>::NT, 0, s>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v), a.g, a.beta, a.W, a.H,
      a.pool, a.num_slots, a.slot_ids, static_cast<Tout*>(a.out), a.rec, a.snapshot_out, a.status);
  return cudaGetLastError();
}

template <int D, typename Tin>
static cudaError_t launch_fold_stream_t(const FoldArgs& a, cudaStream_t s) {
  using L = FoldStreamSmem<D, Tin>;
  cudaError_t e = cudaFuncSetAttribute(fold_stream_kernel<D, Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L::BYTES);
  if (e != cudaSuccess) return e;
  const int units = a.B * a.H, sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = units < 2 * sms ? units : 2 * sms;
  fold_stream_kernel<D, Tin><<<grid, WCfg<D>::NT, L::BYTES, s>>>(a.pool, a.num_slots, a.slot_ids, a.W, a.H, a.rec,
                                                                 a.accepted, a.status, units);
  return cudaGetLastError();
}

template <int D, typename Tin>
static cudaError_t launch_fold_t(const FoldArgs& a, cudaStream_t s) {
  fold_kernel<D, Tin><<<a.B * a.H, WCfg<D>::NT, 0, s>>>(a.pool, a.num_slots, a.slot_ids, a.W, a.H, a.rec, a.accepted,
                                                  a.status);
  return cudaGetLastError();
}

template <typename Tin, typename Tout>
static cudaError_t decode_d(const DecodeArgs& a, cudaStream_t s) {
  switch (a.d) {
    case 16: return launch_decode_t<16, Tin, Tout>(a, s);
    case 32: return launch_decode_t<32, Tin, Tout>(a, s);
    case 64: return launch_decode_t<64, Tin, Tout>(a, s);
    case 128: return launch_decode_stream_t<128, Tin, Tout>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename Tin, typename Tout>
static cudaError_t verify_d(const VerifyArgs& a, cudaStream_t s) {
  switch (a.d) {
    case 16: return launch_verify_t<16, Tin, Tout>(a, s);
    case 32: return launch_verify_t<32, Tin, Tout>(a, s);
    case 64: return launch_verify_t<64, Tin, Tout>(a, s);
    case 128: return launch_verify_t<128, Tin, Tout>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename Tin>
static cudaError_t fold_d(const FoldArgs& a, cudaStream_t s) {
  switch (a.d) {
    case 16: return launch_fold_t<16, Tin>(a, s);
    case 32: return launch_fold_t<32, Tin>(a, s);
    case 64: return launch_fold_t<64, Tin>(a, s);
    case 128: return launch_fold_t<128, Tin>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  if (a.in_bf16) return a.out_bf16 ? decode_d<bf16, bf16>(a, s) : decode_d<bf16, float>(a, s);
  return a.out_bf16 ? decode_d<float, bf16>(a, s) : decode_d<float, float>(a, s);
}

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s) {
  if (verify_tc_supported(a)) return launch_verify_tc(a, s);
  if (a.in_bf16) return a.out_bf16 ? verify_d<bf16, bf16>(a, s) : verify_d<bf16, float>(a, s);
  return a.out_bf16 ? verify_d<float, bf16>(a, s) : verify_d<float, float>(a, s);
}

cudaError_t launch_fold(const FoldArgs& a, cudaStream_t s) {
  if (a.in_bf16 && a.d == 128 && a.W <= WGRP) return launch_fold_stream_t<128, bf16>(a, s);
  return a.in_bf16 ? fold_d<bf16>(a, s) : fold_d<float>(a, s);
}

}  // namespace kda
