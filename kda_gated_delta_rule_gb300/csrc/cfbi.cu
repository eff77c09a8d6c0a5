// Batch-invariant prefill / decode: one row-level computation contract for both paths.
//
// Source: "Kimi K3.1 inference zero mismatch" (LLMNews), section 6.1 (CF-BI): prefill and decode follow
// one row-level contract -- the output of a position depends on the entry state of its chunk and the
// rows before it in that chunk, prefill computes the rows in bulk and decode computes the new row, both in
// the same operation order; besides the recurrent state, the open chunk's row cache and position are kept.
// The current contract uses 16-token chunks with an fp32 row cache per head.  The arithmetic of a row is
// the KDA update of "Kimi K3: Architecture and SGLang Day-0 Support" (KDA math box) unrolled over the open
// chunk from its entry state S_c (rows u = 0 .. t of the chunk, G_u the in-chunk cumulative log-decay):
//   A_tu = beta_t sum_j k_t[j] k_u[j] exp(G_t[j] - G_u[j])  (u < t),
//   P_tu =        sum_j q_t[j] k_u[j] exp(G_t[j] - G_u[j])  (u <= t),
//   R_t  = row t of P (I + A)^-1 diag(beta)  (rows of (I + A)^-1 extended one per row and cached),
//   o_t  = S_c^T (q_t o e^{G_t} - sum_u R_tu k_u o e^{G_u}) + sum_u R_tu v_u,
// and when the chunk is full the entry state advances:
//   U = (I + A)^-1 diag(beta) (V - (K o e^G) S_c),   S_{c+1} = Diag(e^{G_15}) S_c + (K o e^{G_15 - G})^T U.
// Every operation is an explicit round-to-nearest fp32 intrinsic in a fixed order and the two kernels run
// the same device functions with the same thread mapping, so a token's output and the state bits are the
// same whichever path (or batch, or split of a sequence into prefill and decode) computed them.
#include "cfbi_rows.h"
#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace kda {
namespace {

using cfbi::CH;
using cfbi::D;
using cfbi::R_A;
using cfbi::R_BETA;
using cfbi::R_G;
using cfbi::R_K;
using cfbi::R_T;
using cfbi::R_V;
using cfbi::RF;
constexpr int NT = 256;
#ifndef CFBI_DECODE_CTAS
#define CFBI_DECODE_CTAS 3  // decode CTAs resident per SM
#endif

struct RowScratch {
  alignas(16) float q[D];  // q_t (fp32)
  float qh[D];          // q_t o e^{G_t} - sum_u R_tu k_u o e^{G_u}
  float oh[D];          // sum_u R_tu v_u
  float part[2][D];     // partial sums of the read-out over the two key halves
  float p[CH];          // P_t[u]
  float r[CH];          // R_t[u]
};
// 24 KB: kp, ws and u live one after another in one region (barriers between a last read and the next
// first write), so the scratch fits in one row buffer.
struct FoldScratch {
  float kh[CH][D];          // k_u o e^{G_15 - G_u}
  union {
    float kp[CH][D];        // k_u o e^{G_u}
    float ws[2][CH][D];     // partial (K o e^G) S_c over the two key halves
    float u[CH][D];         // U
  };
};
static_assert(sizeof(FoldScratch) <= (size_t)CH * RF * 4, "fold scratch fits a row buffer");

// Row t of the open chunk, steps 1-4 (rows[0 .. t-1] cached; rows[t] holds k_t, v_t, g_t in the G slot and
// beta_t; scr.q holds q_t): completes rows[t] (G_t, A_t, T_t) and leaves qh and oh in scr.
__device__ __forceinline__ void cfbi_row_front(float* rows, RowScratch& scr, int t, int tid) {
  float* rt = rows + t * RF;
  const int warp = tid >> 5, lane = tid & 31;
  // 1. G_t = G_{t-1} + g_t; the slots of row t that no step below writes (A_t[u] for u >= t, the padding)
  //    are set to zero, so the cached row's bytes are a function of the chunk's tokens alone
  if (tid < D) rt[R_G + tid] = __fadd_rn(t > 0 ? rows[(t - 1) * RF + R_G + tid] : 0.f, rt[R_G + tid]);
  else if (tid < D + CH && tid - D >= t) rt[R_A + tid - D] = 0.f;
  else if (tid >= D + CH && tid < D + CH + (RF - R_T - CH)) rt[R_T + CH + tid - D - CH] = 0.f;
  __syncthreads();
  // 2. A_t[u] (u < t) and P_t[u] (u <= t): warp w takes u = w, w + 8; lane l channels 4l .. 4l+3 in order,
  //    then a fixed xor butterfly; lane 0's sum is the value
  {
    const float4 kt = *reinterpret_cast<const float4*>(rt + R_K + 4 * lane);
    const float4 gt = *reinterpret_cast<const float4*>(rt + R_G + 4 * lane);
    const float4 qt = *reinterpret_cast<const float4*>(scr.q + 4 * lane);
  for (int u = warp; u <= t; u += NT / 32) {
    const float* ru = rows + u * RF;
    const float4 ku = *reinterpret_cast<const float4*>(ru + R_K + 4 * lane);
    const float4 gu = *reinterpret_cast<const float4*>(ru + R_G + 4 * lane);
    float a = 0.f, p = 0.f;
    const float kc[4] = {ku.x, ku.y, ku.z, ku.w}, gc[4] = {gu.x, gu.y, gu.z, gu.w};
    const float ktc[4] = {kt.x, kt.y, kt.z, kt.w}, gtc[4] = {gt.x, gt.y, gt.z, gt.w};
    const float qc[4] = {qt.x, qt.y, qt.z, qt.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float kk = __fmul_rn(kc[i], __expf(__fsub_rn(gtc[i], gc[i])));
      a = __fmaf_rn(ktc[i], kk, a);
      p = __fmaf_rn(qc[i], kk, p);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, m));
      p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, m));
    }
    if (lane == 0) {
      if (u < t) rt[R_A + u] = __fmul_rn(rt[R_BETA], a);
      scr.p[u] = p;
    }
  }
  }
  __syncthreads();
  // 3. row t of T = (I + A)^-1 from the cached rows (lane v: T_t[v] = [v == t] - sum_{u=v}^{t-1} A_tu T_u[v],
  //    zero for v > t), then z = P_t T (lane v: sum_{w=v}^{t} P_t[w] T_w[v]) and R_t = z diag(beta)
  if (warp == 0 && lane < CH) {
    const int v = lane;
    float acc = v == t ? 1.f : 0.f;
#pragma unroll
    for (int u = 0; u < CH - 1; ++u)
      if (u >= v && u < t) acc = __fmaf_rn(-rt[R_A + u], rows[u * RF + R_T + v], acc);
    rt[R_T + v] = acc;
  }
  __syncwarp();
  if (warp == 0 && lane < CH) {
    const int v = lane;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < CH; ++w)
      if (w >= v && w <= t) acc = __fmaf_rn(scr.p[w], rows[w * RF + R_T + v], acc);
    scr.r[v] = v <= t ? __fmul_rn(acc, rows[v * RF + R_BETA]) : 0.f;
  }
  __syncthreads();
  // 4. qh (key channel j = tid) and oh (value column c = tid - 128)
  if (tid < D) {
    const int j = tid;
    float acc = __fmul_rn(scr.q[j], __expf(rt[R_G + j]));
#pragma unroll
    for (int u = 0; u < CH; ++u)
      if (u <= t) acc = __fmaf_rn(-scr.r[u], __fmul_rn(rows[u * RF + R_K + j], __expf(rows[u * RF + R_G + j])), acc);
    scr.qh[j] = acc;
  } else {
    const int c = tid - D;
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < CH; ++u)
      if (u <= t) acc = __fmaf_rn(scr.r[u], rows[u * RF + R_V + c], acc);
    scr.oh[c] = acc;
  }
  __syncthreads();
}

// Step 5, o_t = S_c^T qh + oh: thread (c, half) sums its 64 key rows in order, then part0 + part1 + oh;
// returns o_t[c] on threads c < 128.  sv(e) is this thread's part of the entry state, S_c[64 * half + e][c]
// for e < 64 (c = tid % 128, half = tid / 128), from registers or from shared memory.
template <int UE, typename StateAt>
__device__ __forceinline__ float cfbi_readout(RowScratch& scr, StateAt sv, int tid) {
  const int c = tid & (D - 1), half = tid >> 7;
  float acc = 0.f;
#pragma unroll UE
  for (int e = 0; e < 64; ++e) acc = __fmaf_rn(scr.qh[64 * half + e], sv(e), acc);
  scr.part[half][c] = acc;
  __syncthreads();
  return tid < D ? __fadd_rn(__fadd_rn(scr.part[0][tid], scr.part[1][tid]), scr.oh[tid]) : 0.f;
}

// The whole row with the entry state part in registers; returns o_t[c] on threads c < 128.
__device__ __forceinline__ float cfbi_row(float* rows, RowScratch& scr, int t, const float (&sv)[64], int tid) {
  cfbi_row_front(rows, scr, t, tid);
  return cfbi_readout<64>(scr, [&](int e) { return sv[e]; }, tid);
}

// Advances the entry state (this thread's part sv, as in cfbi_row) over the full chunk in rows[0 .. 15].
// ld(e) reads and st(e, x) writes this thread's part of the state, S_c[64 * half + e][c] (registers, or
// global memory); each element is read (twice) before it is written, by its own thread only.
// UE: unroll of the passes over the 64 state elements (64 when the state is in registers).
template <int UE, typename Ld, typename St>
__device__ __forceinline__ void cfbi_fold(const float* rows, FoldScratch& scr, Ld ld, St st, int tid) {
  const float* last = rows + (CH - 1) * RF;
  for (int e = tid; e < CH * D; e += NT) {
    const int u = e / D, j = e % D;
    const float* ru = rows + u * RF;
    scr.kp[u][j] = __fmul_rn(ru[R_K + j], __expf(ru[R_G + j]));
    scr.kh[u][j] = __fmul_rn(ru[R_K + j], __expf(__fsub_rn(last[R_G + j], ru[R_G + j])));
  }
  __syncthreads();
  // (K o e^G) S_c: thread (c, half) over its 64 key rows in order, for every row u
  {
    const int c = tid & (D - 1), half = tid >> 7;
    float acc[CH];
#pragma unroll
    for (int u = 0; u < CH; ++u) acc[u] = 0.f;
#pragma unroll UE
    for (int e = 0; e < 64; ++e) {
      const int j = 64 * half + e;
      const float s = ld(e);
#pragma unroll
      for (int u = 0; u < CH; ++u) acc[u] = __fmaf_rn(scr.kp[u][j], s, acc[u]);
    }
    __syncthreads();  // kp has been read; ws takes its place
#pragma unroll
    for (int u = 0; u < CH; ++u) scr.ws[half][u][c] = acc[u];
  }
  __syncthreads();
  // U = T diag(beta) (V - (K o e^G) S_c): value column c; thread (c, half) forms rows u of its half
  {
    const int c = tid & (D - 1), half = tid >> 7;
    float y[CH];
#pragma unroll
    for (int w = 0; w < CH; ++w) {
      const float* rw = rows + w * RF;
      y[w] = __fmul_rn(rw[R_BETA], __fsub_rn(rw[R_V + c], __fadd_rn(scr.ws[0][w][c], scr.ws[1][w][c])));
    }
    __syncthreads();  // ws has been read; u takes its place
#pragma unroll
    for (int uu = 0; uu < CH / 2; ++uu) {
      const int u = (CH / 2) * half + uu;
      const float* ru = rows + u * RF;
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < CH; ++w)
        if (w <= u) acc = __fmaf_rn(ru[R_T + w], y[w], acc);
      scr.u[u][c] = acc;
    }
  }
  __syncthreads();
  // S_{c+1}[j][c] = e^{G_15[j]} S_c[j][c] + sum_u k_u[j] e^{G_15[j] - G_u[j]} U[u][c]
  {
    const int c = tid & (D - 1), half = tid >> 7;
    float uc[CH];
#pragma unroll
    for (int u = 0; u < CH; ++u) uc[u] = scr.u[u][c];
#pragma unroll UE
    for (int e = 0; e < 64; ++e) {
      const int j = 64 * half + e;
      float s = __fmul_rn(__expf(last[R_G + j]), ld(e));
#pragma unroll
      for (int u = 0; u < CH; ++u) s = __fmaf_rn(scr.kh[u][j], uc[u], s);
      st(e, s);
    }
  }
  __syncthreads();
}

// The new token's inputs into rows[t] (k, v, g in the G slot, beta) and scr.q.
template <typename Tin>
__device__ __forceinline__ void cfbi_load_token(float* rows, RowScratch& scr, int t, const Tin* q, const Tin* k,
                                                const Tin* v, const float* g, const float* beta, size_t row, int tid) {
  float* rt = rows + t * RF;
  if (tid < D) {
    rt[R_K + tid] = to_f32(k[row * D + tid]);
    rt[R_G + tid] = g[row * D + tid];
    scr.q[tid] = to_f32(q[row * D + tid]);
  } else {
    const int c = tid - D;
    rt[R_V + c] = to_f32(v[row * D + c]);
    if (c == 0) rt[R_BETA] = beta[row];
  }
  __syncthreads();
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}

struct CfbiSmem {
  alignas(16) float rows[CH * RF];
  RowScratch scr;
  FoldScratch fold;
};

// this thread's part of a [128][128] state: rows 64 * half .. +63 of column c
__device__ __forceinline__ void load_part(float (&sv)[64], const float* S, int tid) {
  const float* p = S + (size_t)64 * (tid >> 7) * D + (tid & (D - 1));
#pragma unroll
  for (int e = 0; e < 64; ++e) sv[e] = p[(size_t)e * D];
}
__device__ __forceinline__ void store_part(const float (&sv)[64], float* S, int tid) {
  float* p = S + (size_t)64 * (tid >> 7) * D + (tid & (D - 1));
#pragma unroll
  for (int e = 0; e < 64; ++e) p[(size_t)e * D] = sv[e];
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(NT, 1) cfbi_prefill_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                             const Tin* __restrict__ v, const float* __restrict__ g,
                                                             const float* __restrict__ beta, const int32_t* cu,
                                                             int64_t T, int max_seqlen, int H, float* pool,
                                                             float* cache, int32_t* counts, int num_slots,
                                                             const int32_t* __restrict__ slot_ids,
                                                             Tout* __restrict__ out, int32_t* status) {
  extern __shared__ float4 smem4[];
  CfbiSmem& s = *reinterpret_cast<CfbiSmem*>(smem4);
  const int tid = threadIdx.x, h = blockIdx.x, i = blockIdx.y;
  const int64_t s0 = cu[i], s1 = cu[i + 1];
  if (s0 < 0 || s1 < s0 || s1 > T || s1 - s0 > (int64_t)max_seqlen) {
    if (tid == 0) flag_status(status, KDA_DEV_SEQ_OOB);
    return;
  }
  const int slot = slot_ids[i];
  if (slot < 0 || slot >= num_slots) {
    if (tid == 0) flag_status(status, KDA_DEV_SLOT_OOB);
    return;
  }
  float* Sg = pool + ((size_t)slot * H + h) * D * D;
  float* cg = cache + ((size_t)slot * H + h) * CH * RF;
  int32_t* cnt = counts + (size_t)slot * H + h;
  int L = *cnt;
  if (L < 0 || L >= CH) {
    if (tid == 0) flag_status(status, KDA_DEV_SLOT_OOB);
    return;
  }
  float sv[64];
  load_part(sv, Sg, tid);
  for (int e = tid; e < L * RF / 4; e += NT) reinterpret_cast<float4*>(s.rows)[e] = reinterpret_cast<const float4*>(cg)[e];
  __syncthreads();
  for (int64_t t = s0; t < s1; ++t) {
    const size_t row = (size_t)t * H + h;
    cfbi_load_token(s.rows, s.scr, L, q, k, v, g, beta, row, tid);
    const float o = cfbi_row(s.rows, s.scr, L, sv, tid);
    if (tid < D) out[row * D + tid] = from_f32<Tout>(o);
    if (++L == CH) {
      cfbi_fold<64>(s.rows, s.fold, [&](int e) { return sv[e]; }, [&](int e, float x) { sv[e] = x; }, tid);
      L = 0;
    }
  }
  store_part(sv, Sg, tid);
  for (int e = tid; e < L * RF / 4; e += NT) reinterpret_cast<float4*>(cg)[e] = reinterpret_cast<const float4*>(s.rows)[e];
  if (tid == 0) {
    *cnt = L;
    add_work(status, (int32_t)(s1 - s0));
  }
}

// Decode: one CTA per (request, head), three resident per SM (the hardware scheduler balances the units
// that complete a chunk, which cost several plain ones).  The token's inputs are loaded first (they do not
// depend on the slot); once the slot is known, thread 0 asks L2 for the whole 64 KB entry state with one
// bulk prefetch, then the row count and the cached rows follow.  The read-out (and the fold, when the
// token completes a chunk) read the state from global memory, where the prefetch has brought it into L2,
// so no thread holds the state in registers.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(NT, CFBI_DECODE_CTAS) cfbi_decode_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v, const float* __restrict__ g,
    const float* __restrict__ beta, int H, float* pool, float* cache, int32_t* counts, int num_slots,
    const int32_t* __restrict__ slot_ids, Tout* __restrict__ out, int32_t* status) {
  extern __shared__ float4 smem4[];
  CfbiSmem& s = *reinterpret_cast<CfbiSmem*>(smem4);
  const int tid = threadIdx.x, b = blockIdx.x / H, h = blockIdx.x % H;
  const int c = tid & (D - 1), half = tid >> 7;
  const size_t row = (size_t)b * H + h;
  float x0, x1, x2 = 0.f, xb = 0.f;
  if (tid < D) {
    x0 = to_f32(k[row * D + c]);
    x1 = g[row * D + c];
    x2 = to_f32(q[row * D + c]);
  } else {
    x0 = to_f32(v[row * D + c]);
    x1 = 0.f;
    if (c == 0) xb = beta[row];
  }
  const int slot = slot_ids[b];
  if (slot < 0 || slot >= num_slots) {
    if (tid == 0) flag_status(status, KDA_DEV_SLOT_OOB);
    return;
  }
  const size_t sh = (size_t)slot * H + h;
  float* Sg = pool + sh * D * D;
  if (tid == 0) tc::bulk_prefetch_l2(Sg, (uint32_t)(D * D * 4));
  float* cg = cache + sh * CH * RF;
  const int L = counts[sh];
  if (L < 0 || L >= CH) {
    if (tid == 0) flag_status(status, KDA_DEV_SLOT_OOB);
    return;
  }
  for (int e = tid; e < L * RF / 4; e += NT) cp_async16(reinterpret_cast<float4*>(s.rows) + e, reinterpret_cast<const float4*>(cg) + e);
  asm volatile("cp.async.commit_group;" ::: "memory");
  {
    float* rt = s.rows + L * RF;
    if (tid < D) {
      rt[R_K + c] = x0;
      rt[R_G + c] = x1;
      s.scr.q[c] = x2;
    } else {
      rt[R_V + c] = x0;
      if (c == 0) rt[R_BETA] = xb;
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  cfbi_row_front(s.rows, s.scr, L, tid);
  float* sp = Sg + (size_t)64 * half * D + c;  // this thread's part: rows 64 * half + e of column c
  const float o = cfbi_readout<64>(s.scr, [&](int e) { return __ldcg(sp + (size_t)e * D); }, tid);
  if (tid < D) out[row * D + tid] = from_f32<Tout>(o);
  if (L + 1 == CH) {
    cfbi_fold<16>(s.rows, s.fold, [&](int e) { return __ldcg(sp + (size_t)e * D); },
                  [&](int e, float x) { sp[(size_t)e * D] = x; }, tid);
    if (tid == 0) counts[sh] = 0;
  } else {
    for (int e = tid; e < RF / 4; e += NT)
      reinterpret_cast<float4*>(cg + L * RF)[e] = reinterpret_cast<const float4*>(s.rows + L * RF)[e];
    if (tid == 0) counts[sh] = L + 1;
  }
  if (tid == 0) add_work(status, 1);
}

constexpr size_t PREFILL_SMEM = sizeof(CfbiSmem);

template <typename Tin, typename Tout>
cudaError_t launch_prefill_t(const CfbiArgs& a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(cfbi_prefill_kernel<Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)PREFILL_SMEM);
  if (e != cudaSuccess) return e;
  cfbi_prefill_kernel<Tin, Tout><<<dim3(a.H, a.N), NT, PREFILL_SMEM, st>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v), a.g, a.beta, a.cu,
      a.T, a.max_seqlen, a.H, a.pool, a.cache, a.counts, a.num_slots, a.slot_ids, static_cast<Tout*>(a.out),
      a.status);
  return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_decode_t(const CfbiArgs& a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(cfbi_decode_kernel<Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(CfbiSmem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(cfbi_decode_kernel<Tin, Tout>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  cfbi_decode_kernel<Tin, Tout><<<a.B * a.H, NT, sizeof(CfbiSmem), st>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v), a.g, a.beta, a.H,
      a.pool, a.cache, a.counts, a.num_slots, a.slot_ids, static_cast<Tout*>(a.out), a.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cfbi_prefill(const CfbiArgs& a, cudaStream_t st) {
  if (a.in_bf16) return a.out_bf16 ? launch_prefill_t<bf16, bf16>(a, st) : launch_prefill_t<bf16, float>(a, st);
  return a.out_bf16 ? launch_prefill_t<float, bf16>(a, st) : launch_prefill_t<float, float>(a, st);
}

cudaError_t launch_cfbi_decode(const CfbiArgs& a, cudaStream_t st) {
  if (a.in_bf16) return a.out_bf16 ? launch_decode_t<bf16, bf16>(a, st) : launch_decode_t<bf16, float>(a, st);
  return a.out_bf16 ? launch_decode_t<float, bf16>(a, st) : launch_decode_t<float, float>(a, st);
}

}  // namespace kda
