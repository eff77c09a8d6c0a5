// The per-token KDA update for decode, verify and replay, on a warp-owned column block of the state.
//
// Source: "Kimi K3: Architecture and SGLang Day-0 Support" (AI-Infra-Visualized lesson), section
// "attention mechanism explained: KDA", math box: gate S~ = Diag(alpha) S, read r_old = S~^T k, delta
// write S = S~ + beta k (v - r_old)^T; read-out o = S^T q after the write (linear-attention section),
// evaluated as o = S~^T q + (q . k) u with u = beta (v - r_old).
//
// Layout: a CTA of D/16 warps holds one D x D head state in registers.  Warp w owns value columns
// 16w .. 16w+15 (columns evolve independently).  Lane l covers the 4 columns 16w + 4(l%4) .. +3 of the key
// rows l/4 + 8m, m = 0 .. D/8-1, so one 128-bit load instruction of the warp reads 8 full 64-byte row
// segments.  Registers pair rows m = 2i and 2i+1 of one column, so the packed fp32x2 pipe processes two
// rows per instruction and each row-pair's gate, key and query arrive with one 64-bit shared load (tokens
// are staged with their channels permuted to match).  The two sums over rows (S~^T k and S~^T q) first
// combine the pair halves, then reduce across the 8 lanes that share a column chunk with a fixed-order
// butterfly of warp shuffles; u is broadcast back the same way.  No block-wide barrier is needed per
// token.  Every operation rounds to nearest (scalar or packed fp32x2 intrinsics, each lane rounding like
// the scalar op), so decode, verify and replay produce bit-identical states from identical inputs.
#pragma once

#include "common.cuh"

namespace kda {

template <int D>
struct WCfg {
  static constexpr int NW = D / 16;  // warps per head state
  static constexpr int NT = 32 * NW; // threads per CTA
  static constexpr int R = D / 8;    // key rows per lane
  static_assert(D % 16 == 0 && D >= 16 && D <= 128, "head size");
};

// Column (within the head) whose output and u a lane holds after the row sums; lanes with bit 2 clear
// write the output.
__device__ __forceinline__ int wstep_out_col(int warp, int lane) {
  return 16 * warp + 4 * (lane & 3) + 2 * ((lane >> 4) & 1) + ((lane >> 3) & 1);
}

// Inputs of one token (fp32) in shared memory.  a, k, q are stored in lane order: channel j sits at index
// (j % 8) * (D / 8) + j / 8; v is in channel order.
template <int D>
struct __align__(16) WTok {
  alignas(16) float a[D];  // alpha = exp(g)
  alignas(16) float k[D];
  alignas(16) float q[D];
  alignas(16) float v[D];
  float beta;
};

__device__ __forceinline__ constexpr int wperm(int j, int D) { return (j % 8) * (D / 8) + j / 8; }

// Sum over the 8 lanes that share lane % 4, of 4 per-lane column partials (x: columns 0,1 / 2,3 of the
// chunk).  Returns the full sum of column 2*bit4 + bit3 of the chunk; lanes l and l ^ 4 return identical
// values.
__device__ __forceinline__ float reduce_rows(float2 x01, float2 x23, int lane) {
  const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1;
  const float2 keep = b4 ? x23 : x01, give = b4 ? x01 : x23;
  const float2 n = __fadd2_rn(keep, make_float2(__shfl_xor_sync(0xffffffffu, give.x, 16),
                                                __shfl_xor_sync(0xffffffffu, give.y, 16)));
  const float m1 = __fadd_rn(b3 ? n.y : n.x, __shfl_xor_sync(0xffffffffu, b3 ? n.x : n.y, 8));
  return __fadd_rn(m1, __shfl_xor_sync(0xffffffffu, m1, 4));
}

// Number of row pairs per lane.
template <int D>
struct WRows {
  static constexpr int P = D / 16;
};

// One token.  S[i][c] = (S[rg + 16i][col c], S[rg + 16i + 8][col c]) with rg = lane / 4 and col c the c-th
// of the lane's 4 columns.  Returns the output of column 16*warp + 4*(lane%4) + 2*bit4 + bit3 of the lane
// (meaningful when WANT_O).  Warp-synchronous; no block barrier.
template <int D, bool WANT_O>
__device__ __forceinline__ float wstep(float2 (&S)[WRows<D>::P][4], const WTok<D>& tok, int warp, int lane) {
  constexpr int P = WRows<D>::P;
  const int base = (lane >> 2) * (D / 8);
  float2 r[4], sq[4], k2[P];
#pragma unroll
  for (int c = 0; c < 4; ++c) r[c] = sq[c] = make_float2(0.f, 0.f);
  float2 qk2 = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const float2 a2 = *reinterpret_cast<const float2*>(tok.a + base + 2 * i);
    k2[i] = *reinterpret_cast<const float2*>(tok.k + base + 2 * i);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      S[i][c] = __fmul2_rn(a2, S[i][c]);
      r[c] = __ffma2_rn(S[i][c], k2[i], r[c]);
    }
    if (WANT_O) {
      const float2 q2 = *reinterpret_cast<const float2*>(tok.q + base + 2 * i);
#pragma unroll
      for (int c = 0; c < 4; ++c) sq[c] = __ffma2_rn(S[i][c], q2, sq[c]);
      qk2 = __ffma2_rn(q2, k2[i], qk2);
    }
  }
  const float rc = reduce_rows(make_float2(__fadd_rn(r[0].x, r[0].y), __fadd_rn(r[1].x, r[1].y)),
                               make_float2(__fadd_rn(r[2].x, r[2].y), __fadd_rn(r[3].x, r[3].y)), lane);
  const int c = wstep_out_col(warp, lane);
  const float u = __fmul_rn(tok.beta, __fsub_rn(tok.v[c], rc));
  float o = 0.f;
  if (WANT_O) {
    const float sqc = reduce_rows(make_float2(__fadd_rn(sq[0].x, sq[0].y), __fadd_rn(sq[1].x, sq[1].y)),
                                  make_float2(__fadd_rn(sq[2].x, sq[2].y), __fadd_rn(sq[3].x, sq[3].y)), lane);
    float qk = __fadd_rn(qk2.x, qk2.y);
#pragma unroll
    for (int msk = 4; msk <= 16; msk <<= 1) qk = __fadd_rn(qk, __shfl_xor_sync(0xffffffffu, qk, msk));
    o = __fmaf_rn(qk, u, sqc);
  }
  // u of the lane's 4 columns: column e of chunk (lane % 4) sits in lane (lane % 4) + 8*(e & 1) + 16*(e >> 1)
  const int q4 = lane & 3;
  float2 uu[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float ue = __shfl_sync(0xffffffffu, u, q4 + 8 * (e & 1) + 16 * (e >> 1));
    uu[e] = make_float2(ue, ue);
  }
#pragma unroll
  for (int i = 0; i < P; ++i)
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) S[i][cc] = __ffma2_rn(k2[i], uu[cc], S[i][cc]);
  return o;
}

// Loads / stores a lane's rows of the warp's 16 columns from a row-major [D][D] fp32 state.
template <int D>
__device__ __forceinline__ void wload(float2 (&S)[WRows<D>::P][4], const float* src, int warp, int lane) {
  const float* p = src + (size_t)(lane >> 2) * D + 16 * warp + 4 * (lane & 3);
#pragma unroll
  for (int i = 0; i < WRows<D>::P; ++i) {
    const float4 x0 = ld_stream(p + (size_t)16 * i * D);
    const float4 x1 = ld_stream(p + (size_t)(16 * i + 8) * D);
    S[i][0] = make_float2(x0.x, x1.x);
    S[i][1] = make_float2(x0.y, x1.y);
    S[i][2] = make_float2(x0.z, x1.z);
    S[i][3] = make_float2(x0.w, x1.w);
  }
}

// Loads a lane's rows of the warp's 16 columns from a row-major [D][D] fp32 state in shared memory.
template <int D>
__device__ __forceinline__ void wload_shared(float2 (&S)[WRows<D>::P][4], const float* src, int warp, int lane) {
  const float* p = src + (lane >> 2) * D + 16 * warp + 4 * (lane & 3);
#pragma unroll
  for (int i = 0; i < WRows<D>::P; ++i) {
    const float4 x0 = *reinterpret_cast<const float4*>(p + 16 * i * D);
    const float4 x1 = *reinterpret_cast<const float4*>(p + (16 * i + 8) * D);
    S[i][0] = make_float2(x0.x, x1.x);
    S[i][1] = make_float2(x0.y, x1.y);
    S[i][2] = make_float2(x0.z, x1.z);
    S[i][3] = make_float2(x0.w, x1.w);
  }
}

template <int D>
__device__ __forceinline__ void wstore(const float2 (&S)[WRows<D>::P][4], float* dst, int warp, int lane) {
  float* p = dst + (size_t)(lane >> 2) * D + 16 * warp + 4 * (lane & 3);
#pragma unroll
  for (int i = 0; i < WRows<D>::P; ++i) {
    st_stream(p + (size_t)16 * i * D, make_float4(S[i][0].x, S[i][1].x, S[i][2].x, S[i][3].x));
    st_stream(p + (size_t)(16 * i + 8) * D, make_float4(S[i][0].y, S[i][1].y, S[i][2].y, S[i][3].y));
  }
}

}  // namespace kda
