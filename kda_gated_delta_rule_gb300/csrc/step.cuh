// The per-token KDA update on a register-resident state tile.
//
// Source: "Kimi K3: Architecture and SGLang Day-0 Support" (AI-Infra-Visualized lesson), section
// "attention mechanism explained: KDA", math box: gate S~ = Diag(alpha) S, read r_old = S~^T k, delta
// write S = S~ + beta k (v - r_old)^T; read-out o = S^T q after the write (linear-attention section).
// The read-out is evaluated as o = S~^T q + (q . k) u with u = beta (v - r_old), which is S^T q.
//
// A CTA of NT threads holds a D x DVT tile of S (rows = key channels, columns = value channels).  Thread
// (rg, lane) owns rows rg*ROWS .. rg*ROWS+ROWS-1 and the four columns 4*lane .. 4*lane+3.  Loads and
// stores of a row segment are 128-bit and coalesced across the lanes.  The reductions over rows are
// partial sums per thread (fixed row order), combined across row groups through shared memory in a fixed
// group order.  Every floating-point operation is an explicit round-to-nearest intrinsic (scalar, or the
// packed fp32x2 form, which rounds each lane the same way), so decode, verify, replay and the sequential
// prefill produce bit-identical states from identical inputs.
#pragma once

#include "common.cuh"

namespace kda {

template <int D, int DVT, int NT>
struct Tile {
  static constexpr int LANES = DVT / 4;  // threads across the columns of the tile
  static constexpr int RG = NT / LANES;  // row groups
  static constexpr int ROWS = D / RG;    // rows per thread
  static_assert(DVT % 4 == 0 && NT % LANES == 0 && D % RG == 0 && ROWS >= 1, "bad tile");
  static_assert(DVT <= NT, "one thread per column is needed for the combine step");
};

// Inputs of one token for the tile (fp32), double-buffered by the callers.
template <int D, int DVT>
struct __align__(16) TokenSmem {
  float k[D];
  float q[D];
  float a[D];  // alpha = exp(g)
  float v[DVT];
  float beta;
};

// 16-byte aligned: the partial sums and u are read and written with 128-bit shared-memory accesses.
template <int D, int DVT, int NT>
struct __align__(16) StepSmem {
  alignas(16) float red_r[Tile<D, DVT, NT>::RG][DVT];
  alignas(16) float red_q[Tile<D, DVT, NT>::RG][DVT];
  alignas(16) float red_qk[Tile<D, DVT, NT>::RG];
  alignas(16) float u[DVT];
};

// One token.  Returns, in threads tid < DVT, the output of column tid (only meaningful when WANT_O).
// Must be called by all NT threads; contains three __syncthreads().  The token inputs in `tok` must be
// visible to all threads on entry (the caller synchronises after writing them).
template <int D, int DVT, int NT, bool WANT_O>
__device__ __forceinline__ float step(float (&S)[Tile<D, DVT, NT>::ROWS][4], const TokenSmem<D, DVT>& tok,
                                      StepSmem<D, DVT, NT>& sm, int tid) {
  using TL = Tile<D, DVT, NT>;
  const int lane = tid % TL::LANES;
  const int rg = tid / TL::LANES;
  // column pairs (0,1) and (2,3) use the packed fp32x2 pipe; every lane rounds like the scalar op
  float2 r01 = make_float2(0.f, 0.f), r23 = r01, q01 = r01, q23 = r01;
  float qk = 0.f;
#pragma unroll
  for (int i = 0; i < TL::ROWS; ++i) {
    const int j = rg * TL::ROWS + i;
    const float2 a2 = make_float2(tok.a[j], tok.a[j]);
    const float2 k2 = make_float2(tok.k[j], tok.k[j]);
    float2 s01 = __fmul2_rn(a2, make_float2(S[i][0], S[i][1]));
    float2 s23 = __fmul2_rn(a2, make_float2(S[i][2], S[i][3]));
    r01 = __ffma2_rn(s01, k2, r01);
    r23 = __ffma2_rn(s23, k2, r23);
    if (WANT_O) {
      const float qj = tok.q[j];
      const float2 q2 = make_float2(qj, qj);
      q01 = __ffma2_rn(s01, q2, q01);
      q23 = __ffma2_rn(s23, q2, q23);
      qk = __fmaf_rn(qj, tok.k[j], qk);
    }
    S[i][0] = s01.x;
    S[i][1] = s01.y;
    S[i][2] = s23.x;
    S[i][3] = s23.y;
  }
  *reinterpret_cast<float4*>(&sm.red_r[rg][4 * lane]) = make_float4(r01.x, r01.y, r23.x, r23.y);
  if (WANT_O) {
    *reinterpret_cast<float4*>(&sm.red_q[rg][4 * lane]) = make_float4(q01.x, q01.y, q23.x, q23.y);
    if (lane == 0) sm.red_qk[rg] = qk;
  }
  __syncthreads();
  float o = 0.f;
  if (tid < DVT) {
    float R = 0.f, Q = 0.f, QK = 0.f;
#pragma unroll 8
    for (int g = 0; g < TL::RG; ++g) {
      R = __fadd_rn(R, sm.red_r[g][tid]);
      if (WANT_O) {
        Q = __fadd_rn(Q, sm.red_q[g][tid]);
        QK = __fadd_rn(QK, sm.red_qk[g]);
      }
    }
    const float u = __fmul_rn(tok.beta, __fsub_rn(tok.v[tid], R));
    sm.u[tid] = u;
    if (WANT_O) o = __fmaf_rn(QK, u, Q);
  }
  __syncthreads();
  const float4 u4 = *reinterpret_cast<const float4*>(&sm.u[4 * lane]);
  const float2 u01 = make_float2(u4.x, u4.y), u23 = make_float2(u4.z, u4.w);
#pragma unroll
  for (int i = 0; i < TL::ROWS; ++i) {
    const float kj = tok.k[rg * TL::ROWS + i];
    const float2 k2 = make_float2(kj, kj);
    const float2 s01 = __ffma2_rn(k2, u01, make_float2(S[i][0], S[i][1]));
    const float2 s23 = __ffma2_rn(k2, u23, make_float2(S[i][2], S[i][3]));
    S[i][0] = s01.x;
    S[i][1] = s01.y;
    S[i][2] = s23.x;
    S[i][3] = s23.y;
  }
  return o;
}

// Loads / stores the tile rows of S from a row-major [D][ld] fp32 matrix (tile columns start at `col0`).
template <int D, int DVT, int NT>
__device__ __forceinline__ void load_tile(float (&S)[Tile<D, DVT, NT>::ROWS][4], const float* src, int ld, int col0,
                                          int tid) {
  using TL = Tile<D, DVT, NT>;
  const int lane = tid % TL::LANES, rg = tid / TL::LANES;
#pragma unroll
  for (int i = 0; i < TL::ROWS; ++i) {
    const float4 x = ld_stream(src + (size_t)(rg * TL::ROWS + i) * ld + col0 + 4 * lane);
    S[i][0] = x.x;
    S[i][1] = x.y;
    S[i][2] = x.z;
    S[i][3] = x.w;
  }
}

template <int D, int DVT, int NT>
__device__ __forceinline__ void store_tile(const float (&S)[Tile<D, DVT, NT>::ROWS][4], float* dst, int ld, int col0,
                                           int tid) {
  using TL = Tile<D, DVT, NT>;
  const int lane = tid % TL::LANES, rg = tid / TL::LANES;
#pragma unroll
  for (int i = 0; i < TL::ROWS; ++i)
    st_stream(dst + (size_t)(rg * TL::ROWS + i) * ld + col0 + 4 * lane, make_float4(S[i][0], S[i][1], S[i][2], S[i][3]));
}

template <int D, int DVT, int NT>
__device__ __forceinline__ void zero_tile(float (&S)[Tile<D, DVT, NT>::ROWS][4]) {
#pragma unroll
  for (int i = 0; i < Tile<D, DVT, NT>::ROWS; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) S[i][c] = 0.f;
}

}  // namespace kda
