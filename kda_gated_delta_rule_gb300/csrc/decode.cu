// Decode step, speculative verify and replay fold.
//
// Sources: "Kimi K3: Architecture and SGLang Day-0 Support", KDA math box (the per-token update);
// "SGLang and Miles: day-0 support for Kimi K3", section "ReplaySSM: raw-input replay for KDA state"
// (verify reads the committed checkpoint and never writes it, storing each step's raw inputs
// (v, k, gk, beta); the fold replays only the accepted prefix in place with the stored gate values, so
// the rebuilt state is bit-identical to the recurrence baseline).
//
// One CTA per (request, head) holds the whole D x D state in registers (2*D threads, 128-bit loads of
// row segments), so each 64 KB state (D = 128) is read once and written at most once per launch.
#include "launch.h"
#include "step.cuh"

namespace kda {

// Loads one token of one head (element offset `base` for the D-vectors, `bidx` for beta) into smem.
template <int D, typename Tin, bool WITH_Q>
__device__ __forceinline__ void load_token(TokenSmem<D, D>& tok, const Tin* k, const Tin* q, const Tin* v,
                                           const float* g, const float* beta, size_t base, size_t bidx, int tid) {
  if (tid < D) {
    tok.k[tid] = to_f32(k[base + tid]);
    if (WITH_Q) tok.q[tid] = to_f32(q[base + tid]);
    tok.a[tid] = expf(g[base + tid]);
    tok.v[tid] = to_f32(v[base + tid]);
  }
  if (tid == 0) tok.beta = beta[bidx];
}

template <int D, typename Tin, typename Tout>
__global__ void __launch_bounds__(2 * D, 2) decode_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                       const Tin* __restrict__ v, const float* __restrict__ g,
                                                       const float* __restrict__ beta, int H, float* pool,
                                                       int num_slots, const int32_t* __restrict__ slot_ids,
                                                       Tout* __restrict__ out, int32_t* status) {
  constexpr int NT = 2 * D;
  using TL = Tile<D, D, NT>;
  __shared__ TokenSmem<D, D> tok;
  __shared__ StepSmem<D, D, NT> sm;
  const int tid = threadIdx.x;
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int slot = slot_ids[b];
  if (slot < 0 || slot >= num_slots) {
    if (tid == 0) flag_status(status, KDA_DEV_SLOT_OOB);
    return;
  }
  float* Sg = pool + ((size_t)slot * H + h) * D * D;
  float S[TL::ROWS][4];
  load_tile<D, D, NT>(S, Sg, D, 0, tid);
  const size_t base = ((size_t)b * H + h) * D;
  load_token<D, Tin, true>(tok, k, q, v, g, beta, base, (size_t)b * H + h, tid);
  __syncthreads();
  const float o = step<D, D, NT, true>(S, tok, sm, tid);
  if (tid < D) out[base + tid] = from_f32<Tout>(o);
  store_tile<D, D, NT>(S, Sg, D, 0, tid);
  if (tid == 0) add_work(status, 1);
}

template <int D, typename Tin, typename Tout>
__global__ void __launch_bounds__(2 * D, 2) verify_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                       const Tin* __restrict__ v, const float* __restrict__ g,
                                                       const float* __restrict__ beta, int W, int H,
                                                       const float* __restrict__ pool, int num_slots,
                                                       const int32_t* __restrict__ slot_ids, Tout* __restrict__ out,
                                                       ReplayPtrs rec, float* __restrict__ snapshot_out,
                                                       int32_t* status) {
  constexpr int NT = 2 * D;
  using TL = Tile<D, D, NT>;
  __shared__ TokenSmem<D, D> tok[2];
  __shared__ StepSmem<D, D, NT> sm;
  const int tid = threadIdx.x;
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int slot = slot_ids[b];
  if (slot < 0 || slot >= num_slots) {
    if (tid == 0) flag_status(status, KDA_DEV_SLOT_OOB);
    return;
  }
  float S[TL::ROWS][4];
  load_tile<D, D, NT>(S, pool + ((size_t)slot * H + h) * D * D, D, 0, tid);
  Tin* rk = static_cast<Tin*>(rec.k);
  Tin* rv = static_cast<Tin*>(rec.v);
  for (int w = 0; w < W; ++w) {
    const size_t row = ((size_t)b * W + w) * H + h;
    const size_t base = row * D;
    TokenSmem<D, D>& t = tok[w & 1];
    load_token<D, Tin, true>(t, k, q, v, g, beta, base, row, tid);
    // raw-input record: the exact stored bits the fold will consume
    if (tid < D) {
      rk[base + tid] = k[base + tid];
      rv[base + tid] = v[base + tid];
      rec.g[base + tid] = g[base + tid];
    }
    if (tid == 0) rec.beta[row] = beta[row];
    __syncthreads();
    const float o = step<D, D, NT, true>(S, t, sm, tid);
    if (tid < D) out[base + tid] = from_f32<Tout>(o);
    if (snapshot_out) store_tile<D, D, NT>(S, snapshot_out + row * D * D, D, 0, tid);
  }
  if (tid == 0) add_work(status, W);
}

template <int D, typename Tin>
__global__ void __launch_bounds__(2 * D, 2) fold_kernel(float* pool, int num_slots, const int32_t* __restrict__ slot_ids,
                                                     int W, int H, ReplayPtrs rec,
                                                     const int32_t* __restrict__ accepted, int32_t* status) {
  constexpr int NT = 2 * D;
  using TL = Tile<D, D, NT>;
  __shared__ TokenSmem<D, D> tok[2];
  __shared__ StepSmem<D, D, NT> sm;
  const int tid = threadIdx.x;
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
  float S[TL::ROWS][4];
  load_tile<D, D, NT>(S, Sg, D, 0, tid);
  const Tin* rk = static_cast<const Tin*>(rec.k);
  const Tin* rv = static_cast<const Tin*>(rec.v);
  for (int w = 0; w < n; ++w) {
    const size_t row = ((size_t)b * W + w) * H + h;
    TokenSmem<D, D>& t = tok[w & 1];
    load_token<D, Tin, false>(t, rk, nullptr, rv, rec.g, rec.beta, row * D, row, tid);
    __syncthreads();
    step<D, D, NT, false>(S, t, sm, tid);
  }
  store_tile<D, D, NT>(S, Sg, D, 0, tid);
  if (tid == 0) add_work(status, n);
}

// ---------------------------------------------------------------- launchers

template <int D, typename Tin, typename Tout>
static cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
  decode_kernel<D, Tin, Tout><<<a.B * a.H, 2 * D, 0, s>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v), a.g, a.beta, a.H,
      a.pool, a.num_slots, a.slot_ids, static_cast<Tout*>(a.out), a.status);
  return cudaGetLastError();
}

template <int D, typename Tin, typename Tout>
static cudaError_t launch_verify_t(const VerifyArgs& a, cudaStream_t s) {
  verify_kernel<D, Tin, Tout><<<a.B * a.H, 2 * D, 0, s>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v), a.g, a.beta, a.W, a.H,
      a.pool, a.num_slots, a.slot_ids, static_cast<Tout*>(a.out), a.rec, a.snapshot_out, a.status);
  return cudaGetLastError();
}

template <int D, typename Tin>
static cudaError_t launch_fold_t(const FoldArgs& a, cudaStream_t s) {
  fold_kernel<D, Tin><<<a.B * a.H, 2 * D, 0, s>>>(a.pool, a.num_slots, a.slot_ids, a.W, a.H, a.rec, a.accepted,
                                                  a.status);
  return cudaGetLastError();
}

template <typename Tin, typename Tout>
static cudaError_t decode_d(const DecodeArgs& a, cudaStream_t s) {
  switch (a.d) {
    case 16: return launch_decode_t<16, Tin, Tout>(a, s);
    case 32: return launch_decode_t<32, Tin, Tout>(a, s);
    case 64: return launch_decode_t<64, Tin, Tout>(a, s);
    case 128: return launch_decode_t<128, Tin, Tout>(a, s);
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
  if (a.in_bf16) return a.out_bf16 ? verify_d<bf16, bf16>(a, s) : verify_d<bf16, float>(a, s);
  return a.out_bf16 ? verify_d<float, bf16>(a, s) : verify_d<float, float>(a, s);
}

cudaError_t launch_fold(const FoldArgs& a, cudaStream_t s) { return a.in_bf16 ? fold_d<bf16>(a, s) : fold_d<float>(a, s); }

}  // namespace kda
