// Inverse of a unit lower-triangular 64 x 64 system, T = (I + A)^-1 with A strictly lower, in fp32 by a
// 256-thread CTA (the WY/UT form's per-chunk solve; its blocked order is derived from block forward
// substitution, not taken from the pages).  Diagonal 16 x 16 blocks by forward substitution (threads 0..63,
// one column each); then, with M_ik = T_ii A_ik, block row i of (I + A) T = I gives
// T_ij = -sum_{k=j}^{i-1} M_ik T_kj, computed in four rounds one 16 x 16 block product deep (one warp per
// product: lane (rp, cg) owns rows rp and rp + 8, columns 4 cg .. 4 cg + 3; per step two conflict-free
// scalar loads, a warp's eight rows sitting in eight bank groups at a row stride of LS = 4 mod 32 floats,
// and one 16-byte load feed eight FMAs):
//   1. M_ik for all six pairs (kept in the upper block (k, i) of T);
//   2. T_10, T_21, T_32 (one term each);
//   3. the six products M_20 T_00, M_21 T_10, M_31 T_11, M_32 T_21, M_30 T_00, M_31 T_10 (into A's storage);
//   4. T_20 and T_31 as sums of two of them, and T_30 = -(M_30 T_00 + M_31 T_10) + M_32 (M_20 T_00 + M_21 T_10).
// A is overwritten (scratch); T's upper blocks hold the M_ik afterwards (the diagonal blocks' upper
// triangles are zero).  Every thread of the CTA calls it; the caller synchronises the CTA before reading T
// (the last round writes T_20, T_31 and T_30).
#pragma once
#include <cstdint>

namespace kda {

template <int LS>
__device__ __forceinline__ void inv_mac16(const float* m, const float* b, float (&a0)[4], float (&a1)[4]) {
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const float m0 = m[u], m1 = m[8 * LS + u];
    const float4 b4 = *reinterpret_cast<const float4*>(b + u * LS);
    a0[0] = fmaf(m0, b4.x, a0[0]); a0[1] = fmaf(m0, b4.y, a0[1]); a0[2] = fmaf(m0, b4.z, a0[2]); a0[3] = fmaf(m0, b4.w, a0[3]);
    a1[0] = fmaf(m1, b4.x, a1[0]); a1[1] = fmaf(m1, b4.y, a1[1]); a1[2] = fmaf(m1, b4.z, a1[2]); a1[3] = fmaf(m1, b4.w, a1[3]);
  }
}

template <int LS>
__device__ __forceinline__ void unit_lower_inverse64(float* sA, float* sT, int tid) {
  static_assert(LS % 32 == 4, "row stride: 8 consecutive rows in 8 bank groups");
  if (tid < 64) {
    const int b = tid >> 4, cc = tid & 15;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < r; ++u) acc = fmaf(sA[(16 * b + r) * LS + 16 * b + u], x[u], acc);
      x[r] = r == cc ? 1.f : (r < cc ? 0.f : -acc);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) sT[(16 * b + r) * LS + 16 * b + cc] = x[r];
  }
  __syncthreads();
  const int rp = (tid >> 2) & 7, cg = tid & 3, wv = tid >> 5;
  auto mac = [&](const float* mb, const float* bb, float (&a0)[4], float (&a1)[4]) {
    inv_mac16<LS>(mb + rp * LS, bb + 4 * cg, a0, a1);
  };
  auto tblk = [&](int r, int c) { return sT + 16 * r * LS + 16 * c; };  // block (r, c) of T
  constexpr int PLD = 20;                                               // row stride of the partial products
  auto pblk = [&](int s) { return sA + s * 16 * PLD; };
  auto put = [&](float* dst, int ld, const float (&a0)[4], const float (&a1)[4], float sg) {
    *reinterpret_cast<float4*>(dst + rp * ld + 4 * cg) = make_float4(sg * a0[0], sg * a0[1], sg * a0[2], sg * a0[3]);
    *reinterpret_cast<float4*>(dst + (rp + 8) * ld + 4 * cg) = make_float4(sg * a1[0], sg * a1[1], sg * a1[2], sg * a1[3]);
  };
  if (wv < 6) {  // round 1: M_ik = T_ii A_ik; pairs (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
    const int bi = wv == 0 ? 1 : (wv < 3 ? 2 : 3);
    const int bk = wv == 0 ? 0 : (wv < 3 ? wv - 1 : wv - 3);
    float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
    mac(tblk(bi, bi), sA + 16 * bi * LS + 16 * bk, a0, a1);
    put(tblk(bk, bi), LS, a0, a1, 1.f);
  }
  __syncthreads();
  if (wv < 3) {  // round 2: T_{w+1,w} = -M_{w+1,w} T_ww
    float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
    mac(tblk(wv, wv + 1), tblk(wv, wv), a0, a1);
    put(tblk(wv + 1, wv), LS, a0, a1, -1.f);
  }
  __syncthreads();
  if (wv < 6) {  // round 3: (i, j, k) = (2,0,0) (2,0,1) (3,1,1) (3,1,2) (3,0,0) (3,0,1): M_ik T_kj into slot wv
    const int bi = wv < 2 ? 2 : 3, bj = wv < 2 ? 0 : (wv < 4 ? 1 : 0);
    const int bk = wv == 0 ? 0 : (wv == 1 ? 1 : (wv == 2 ? 1 : (wv == 3 ? 2 : (wv == 4 ? 0 : 1))));
    float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
    mac(tblk(bk, bi), tblk(bk, bj), a0, a1);
    put(pblk(wv), PLD, a0, a1, 1.f);
  }
  __syncthreads();
  if (wv < 3) {  // round 4
    float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
    if (wv == 2) {  // M_32 (M_20 T_00 + M_21 T_10): the second operand summed on the fly
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float m0 = tblk(2, 3)[rp * LS + u], m1 = tblk(2, 3)[(rp + 8) * LS + u];
        const float4 p0 = *reinterpret_cast<const float4*>(pblk(0) + u * PLD + 4 * cg);
        const float4 p1 = *reinterpret_cast<const float4*>(pblk(1) + u * PLD + 4 * cg);
        const float4 b4 = make_float4(p0.x + p1.x, p0.y + p1.y, p0.z + p1.z, p0.w + p1.w);
        a0[0] = fmaf(m0, b4.x, a0[0]); a0[1] = fmaf(m0, b4.y, a0[1]); a0[2] = fmaf(m0, b4.z, a0[2]); a0[3] = fmaf(m0, b4.w, a0[3]);
        a1[0] = fmaf(m1, b4.x, a1[0]); a1[1] = fmaf(m1, b4.y, a1[1]); a1[2] = fmaf(m1, b4.z, a1[2]); a1[3] = fmaf(m1, b4.w, a1[3]);
      }
    }
    // wv 0: T_20 = -(slot 0 + slot 1); wv 1: T_31 = -(slot 2 + slot 3); wv 2: T_30 = acc - (slot 4 + slot 5)
    const int sa = 2 * wv, dr = wv == 1 ? 3 : (wv == 0 ? 2 : 3), dc = wv == 1 ? 1 : 0;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int row = rp + 8 * h2;
      const float4 x0 = *reinterpret_cast<const float4*>(pblk(sa) + row * PLD + 4 * cg);
      const float4 x1 = *reinterpret_cast<const float4*>(pblk(sa + 1) + row * PLD + 4 * cg);
      const float* ac = h2 ? a1 : a0;
      *reinterpret_cast<float4*>(tblk(dr, dc) + row * LS + 4 * cg) =
          make_float4(ac[0] - (x0.x + x1.x), ac[1] - (x0.y + x1.y), ac[2] - (x0.z + x1.z), ac[3] - (x0.w + x1.w));
    }
  }
}

}  // namespace kda
