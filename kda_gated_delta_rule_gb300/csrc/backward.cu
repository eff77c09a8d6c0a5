// Chunked backward (vector-Jacobian product) of the KDA recurrence, dk = dv = 128, 64-token chunks.
//
// The forward recurrence is the KDA math box of "Kimi K3: Architecture and SGLang Day-0 Support"
// (gate, read along the key, delta write; o = S^T q after the write); the training side that needs its
// gradient is "Kimi K3 training and serving infra" (marsggbo blog), section 7.  The chunk algebra below is
// derived from the recurrence by induction over a chunk (it is not printed on the pages).  Per chunk with
// entry state S and in-chunk cumulative log-decay G (G_C its last row):
//   K+ = K o e^G,  Q+ = Q o e^G,  K^ = K o e^(G_C - G),  a_ts = sum_j k_t k_s e^(G_t - G_s) (s < t),
//   P_ts = sum_j q_t k_s e^(G_t - G_s) (s <= t),  T = (I + diag(beta) a)^-1,
//   W = T diag(beta) K+,  U~ = T diag(beta) V,  U = U~ - W S,
//   O = Q+ S + P U,  S' = Diag(e^G_C) S + K^^T U.
// Its reverse, with dS' the gradient at the chunk's exit state:
//   dU = P^T dO + K^ dS',   dS = Q+^T dO + Diag(e^G_C) dS' - W^T dU          (the carry, chunk to chunk)
//   dQ+ = dO S^T,  dW = -dU S^T,  dK^ = U dS'^T,  dP = tril(dO U^T),  d(e^G_C) = rowsum(dS' o S)
//   dT = dW (diag(beta) K+)^T + dU (diag(beta) V)^T,  dA = -T^T dT T^T (strictly lower)
//   dK+ = diag(beta) T^T dW,  dv = diag(beta) T^T dU
// and the chain rule through beta, the e^G factors and the pair decays e^(G_t - G_s); dg is the in-chunk
// reverse cumulative sum of dG.  Pair decays are split at a reference token r, e^(G_t - G_s) =
// e^(G_t - G_r) e^(G_r - G_s): the chunk's last token when the chunk's decay span stays within e^80, else the
// last token of s's 16-token block while every factor stays below e^80 (always when g >= -5, the pages'
// floor); a block that would exceed it takes the pair decays one by one.
//
// Kernels handing over through a per-(chunk, head) fp32 workspace (tiles move into shared memory by
// asynchronous 16-byte copies):
//   prep (chunk-parallel) -> forward pass (entry states, U) -> reverse chain (dS', dU)
//   -> state products -> WY backward -> per-channel assembly (chunk-parallel).
// With bf16 inputs the forward pass is the tensor-core segmented prefill (operand records, segment
// fragments, the fragment scan, then every segment from its exact entry state, writing each chunk's entry
// state and U into this workspace); otherwise it is the CUDA-core chain below.  With bf16 inputs the prep
// also flags each (sequence, head) holding a 16-token block whose decay span passes e^80 (g below the
// floor), where the tensor-core pass's block references overflow; the CUDA-core chain then runs for the
// flagged (sequence, head)s only and overwrites their entry states and U.  The reverse chain likewise: on
// the tensor cores over the same operand records (segmented, the fragment scan run from dL/dS_T), with the
// CUDA-core reverse chain below for fp32 inputs and the flagged (sequence, head)s.  The state products run on
// the tensor cores (split-bf16 tcgen05 MMAs, fp32 accumulation); the remaining kernels are fp32 on the
// CUDA cores.
#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"
#include "wy_inverse.cuh"

namespace kda {
namespace {

constexpr int C = 64;      // chunk length
constexpr int D = 128;     // dk = dv
constexpr int NT = 256;    // threads per CTA
constexpr int NTC = 512;   // threads per CTA of the chain kernels
constexpr int LD = D + 4;  // shared row stride of [rows][128] tiles (16-byte rows; 8 consecutive rows hit distinct banks)
constexpr int LC = C + 4;  // shared row stride of [64][64] tiles
constexpr int HC = 64;     // channels per CTA of the assembly kernel
constexpr int CB = 16;     // value columns per CTA of the chain kernels
constexpr float SPAN_MAX = 80.f;

// Workspace record of one (chunk, head), fp32 element offsets.  All [64][128] / [128][128] / [64][64] tiles
// are dense row-major.
constexpr uint32_t BW_G = 0;                    // G [64][128]
constexpr uint32_t BW_W = BW_G + C * D;         // W = T diag(beta) K+
constexpr uint32_t BW_UT = BW_W + C * D;        // U~ = T diag(beta) V
constexpr uint32_t BW_KH = BW_UT + C * D;       // K^ = K o e^(G_C - G)
constexpr uint32_t BW_QP = BW_KH + C * D;       // Q+ = Q o e^G
constexpr uint32_t BW_P = BW_QP + C * D;        // P [64][64] (s <= t)
constexpr uint32_t BW_T = BW_P + C * C;         // T = (I + diag(beta) a)^-1 [64][64]
constexpr uint32_t BW_A = BW_T + C * C;         // a [64][64] (s < t)
constexpr uint32_t BW_GAM = BW_A + C * C;       // e^(G_C) [128]
constexpr uint32_t BW_H = BW_GAM + D;           // entry state S [128][128]
constexpr uint32_t BW_U = BW_H + D * D;         // U [64][128]
constexpr uint32_t BW_DS = BW_U + C * D;        // dS' (gradient at the exit state) [128][128]
constexpr uint32_t BW_DU = BW_DS + D * D;       // dU [64][128]
constexpr uint32_t BW_DQP = BW_DU + C * D;      // dQ+ [64][128]
constexpr uint32_t BW_DW = BW_DQP + C * D;      // dW [64][128]
constexpr uint32_t BW_DKH = BW_DW + C * D;      // dK^ [64][128]
constexpr uint32_t BW_DP = BW_DKH + C * D;      // dP [64][64]
constexpr uint32_t BW_DGAM = BW_DP + C * C;     // d(e^G_C) [128]
constexpr uint32_t BW_DKP = BW_DGAM + D;        // dK+ [64][128]
constexpr uint32_t BW_DA = BW_DKP + C * D;      // dA [64][64]
constexpr uint32_t BW_DBETA = BW_DA + C * C;    // dbeta through W and U~ [64]
constexpr uint32_t BW_FLOATS = BW_DBETA + C;

__device__ __forceinline__ void ld4(const float* p, float (&x)[4]) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
}
__device__ __forceinline__ void ld4(const bf16* p, float (&x)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  x[0] = a.x, x[1] = a.y, x[2] = b.x, x[3] = b.y;
}

// 16-byte asynchronous global -> shared copy; src_bytes = 0 writes zeros (the source is not read)
__device__ __forceinline__ void cp_async16(float* dst, const float* src, int src_bytes) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// rows [0, rows) x columns [c0, c0 + ncols) of a row-major source (row r at src + r * stride) into shared
// memory as fp32 with row stride ld (a multiple of 4); rows >= n are zero.  fp32 sources are copied
// asynchronously (complete with cp_async_commit / cp_async_wait); bf16 sources are widened through
// registers, all of a thread's loads issued before its stores.
template <int NTH>
__device__ __forceinline__ void load_rows(float* dst, int ld, const float* src, int64_t stride, int rows, int n,
                                          int c0, int ncols) {
  const int q4 = ncols / 4;
  for (int e = threadIdx.x; e < rows * q4; e += NTH) {
    const int r = e / q4, c = (e % q4) * 4;
    cp_async16(dst + r * ld + c, src + (r < n ? r : 0) * stride + c0 + c, r < n ? 16 : 0);
  }
}
template <int NTH>
__device__ __forceinline__ void load_rows(float* dst, int ld, const bf16* src, int64_t stride, int rows, int n,
                                          int c0, int ncols) {
  constexpr int MAXIT = 8;
  const int q4 = ncols / 4, total = rows * q4;
  for (int base = 0; base < total; base += MAXIT * NTH) {
    float x[MAXIT][4];
#pragma unroll
    for (int it = 0; it < MAXIT; ++it) {
      const int e = base + it * NTH + threadIdx.x;
      const int r = e / q4, c = (e % q4) * 4;
      x[it][0] = x[it][1] = x[it][2] = x[it][3] = 0.f;
      if (e < total && r < n) ld4(src + r * stride + c0 + c, x[it]);
    }
#pragma unroll
    for (int it = 0; it < MAXIT; ++it) {
      const int e = base + it * NTH + threadIdx.x;
      if (e < total) {
        const int r = e / q4, c = (e % q4) * 4;
        *reinterpret_cast<float4*>(dst + r * ld + c) = make_float4(x[it][0], x[it][1], x[it][2], x[it][3]);
      }
    }
  }
}

// acc += sum_{r < 8} x[r * xs] * y4[r * ys .. + 3]: the 8 scalar and 8 16-byte shared loads are issued
// before the FMAs, so one group of a loop waits on shared-memory latency once
__device__ __forceinline__ void dot8x4(const float* x, int xs, const float* y, int ys, float (&acc)[4]) {
  float xv[8];
  float4 yv[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    xv[r] = x[r * xs];
    yv[r] = *reinterpret_cast<const float4*>(y + r * ys);
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    acc[0] = fmaf(xv[r], yv[r].x, acc[0]);
    acc[1] = fmaf(xv[r], yv[r].y, acc[1]);
    acc[2] = fmaf(xv[r], yv[r].z, acc[2]);
    acc[3] = fmaf(xv[r], yv[r].w, acc[3]);
  }
}

struct Seq {
  int bos, eos;
};

// Bounds of sequence i; false (and the flag) when cu_seqlens is malformed.
__device__ __forceinline__ bool seq_bounds(const BackwardArgs& a, int i, Seq& s, bool report) {
  s.bos = a.cu[i];
  s.eos = a.cu[i + 1];
  if (s.bos < 0 || s.eos < s.bos || s.eos > a.T || s.eos - s.bos > a.max_seqlen) {
    if (report && threadIdx.x == 0) flag_status(a.status, KDA_DEV_SEQ_OOB);
    return false;
  }
  return true;
}

__device__ __forceinline__ float* record(const BackwardArgs& a, int t0, int i, int h) {
  return a.ws + ((size_t)(t0 / C + i) * a.H + h) * BW_FLOATS;
}

// ---------------------------------------------------------------------------------------------------
// 1. prep: G, a, P, T, W, U~, K^, Q+, e^G_C of one (chunk, head)
// ---------------------------------------------------------------------------------------------------
constexpr size_t PREP_SMEM = (5 * C * LD + 16 * LD + 3 * C * LC + C) * sizeof(float);

template <typename Tin>
__global__ void __launch_bounds__(NT, 1) bwd_prep_kernel(BackwardArgs a) {
  const int c = blockIdx.x, h = blockIdx.y, i = blockIdx.z, tid = threadIdx.x;
  Seq sq;
  if (!seq_bounds(a, i, sq, c == 0 && h == 0)) return;
  const int t0 = sq.bos + c * C;
  if (t0 >= sq.eos) return;
  const int n = min(C, sq.eos - t0);
  float* w = record(a, t0, i, h);
  extern __shared__ float sm[];
  float* sK = sm;              // k [64][LD]
  float* sQ = sK + C * LD;     // q
  float* sG = sQ + C * LD;     // g, then G
  float* sX = sG + C * LD;     // k o e^(G_t - G_r) of the current block; later diag(beta) K+, then diag(beta) V
  float* sY = sX + C * LD;     // q o e^(G_t - G_r) of the current block
  float* sM = sY + C * LD;     // k o e^(G_r - G_s) of the current block [16][LD]
  float* sA = sM + 16 * LD;    // a [64][LC]
  float* sP = sA + C * LC;     // P [64][LC]
  float* sT = sP + C * LC;     // T [64][LC]
  float* sB = sT + C * LC;     // beta [64]
  const int64_t rs = (int64_t)a.H * D;
  load_rows<NT>(sK, LD, reinterpret_cast<const Tin*>(a.k) + ((int64_t)t0 * a.H + h) * D, rs, C, n, 0, D);
  load_rows<NT>(sQ, LD, reinterpret_cast<const Tin*>(a.q) + ((int64_t)t0 * a.H + h) * D, rs, C, n, 0, D);
  load_rows<NT>(sG, LD, a.g + ((int64_t)t0 * a.H + h) * D, rs, C, n, 0, D);
  if (tid < C) sB[tid] = tid < n ? a.beta[(int64_t)(t0 + tid) * a.H + h] : 0.f;
  for (int e = tid; e < C * LC; e += NT) sA[e] = 0.f, sP[e] = 0.f;
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  float gspan = 0.f;  // the channel's decay span over the chunk (including its start, G = 0)
  if (tid < D) {  // in-chunk cumulative sum, one thread per channel
    float acc = 0.f, gmin = 0.f, gmax = 0.f;
    for (int t = 0; t < C; ++t) {
      acc += sG[t * LD + tid];
      sG[t * LD + tid] = acc;
      gmin = fminf(gmin, acc);
      gmax = fmaxf(gmax, acc);
    }
    gspan = gmax - gmin;
  }
  const bool chunk_wide = __syncthreads_or(gspan > SPAN_MAX);
  if (tid == 0) add_work(a.status, n);

  if (!chunk_wide) {
    // Common case: one reference token, the chunk's last, for every pair: a = X Y^T and P = Xq Y^T with
    // X = k o e^(G - G_C), Xq = q o e^(G - G_C) and Y = k o e^(G_C - G) (the record's K^), every factor within
    // e^SPAN_MAX.  The records' G, K^ and Q+ are written on the way; Y takes q's place.
    for (int e = tid; e < C * D / 4; e += NT) {
      const int t = e >> 5, j = (e & 31) * 4;
      const float4 k4 = *reinterpret_cast<const float4*>(sK + t * LD + j);
      const float4 q4 = *reinterpret_cast<const float4*>(sQ + t * LD + j);
      const float4 g4 = *reinterpret_cast<const float4*>(sG + t * LD + j);
      const float4 c4 = *reinterpret_cast<const float4*>(sG + (C - 1) * LD + j);
      const float kk[4] = {k4.x, k4.y, k4.z, k4.w}, qq[4] = {q4.x, q4.y, q4.z, q4.w};
      const float gg[4] = {g4.x, g4.y, g4.z, g4.w}, gc[4] = {c4.x, c4.y, c4.z, c4.w};
      float x[4], xq[4], y[4], qp[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float e1 = __expf(gg[u] - gc[u]);
        x[u] = kk[u] * e1;
        xq[u] = qq[u] * e1;
        y[u] = kk[u] * __expf(gc[u] - gg[u]);
        qp[u] = qq[u] * __expf(gg[u]);
      }
      *reinterpret_cast<float4*>(sX + t * LD + j) = make_float4(x[0], x[1], x[2], x[3]);
      *reinterpret_cast<float4*>(sY + t * LD + j) = make_float4(xq[0], xq[1], xq[2], xq[3]);
      *reinterpret_cast<float4*>(sQ + t * LD + j) = make_float4(y[0], y[1], y[2], y[3]);
      *reinterpret_cast<float4*>(w + BW_G + t * D + j) = g4;
      *reinterpret_cast<float4*>(w + BW_KH + t * D + j) = make_float4(y[0], y[1], y[2], y[3]);
      *reinterpret_cast<float4*>(w + BW_QP + t * D + j) = make_float4(qp[0], qp[1], qp[2], qp[3]);
    }
    __syncthreads();
    // thread (tr, tc): rows t = 4 tr + r, columns s = tc + 16 r' (a warp's Y rows in eight bank groups)
    const int tr = tid >> 4, tc = tid & 15;
    float aa[4][4] = {}, pp[4][4] = {};
#pragma unroll 2
    for (int j = 0; j < D; j += 4) {
      float4 x[4], xq[4], y[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        x[r] = *reinterpret_cast<const float4*>(sX + (4 * tr + r) * LD + j);
        xq[r] = *reinterpret_cast<const float4*>(sY + (4 * tr + r) * LD + j);
        y[r] = *reinterpret_cast<const float4*>(sQ + (tc + 16 * r) * LD + j);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          aa[r][q] = fmaf(x[r].w, y[q].w, fmaf(x[r].z, y[q].z, fmaf(x[r].y, y[q].y, fmaf(x[r].x, y[q].x, aa[r][q]))));
          pp[r][q] = fmaf(xq[r].w, y[q].w, fmaf(xq[r].z, y[q].z, fmaf(xq[r].y, y[q].y, fmaf(xq[r].x, y[q].x, pp[r][q]))));
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int t = 4 * tr + r, s = tc + 16 * q;
        sA[t * LC + s] = s < t ? aa[r][q] : 0.f;
        sP[t * LC + s] = s <= t ? pp[r][q] : 0.f;
      }
    __syncthreads();
  }

  // a and P when the chunk's span is wider: one 16-column block of s at a time, each at its own reference
  for (int b0 = 0; chunk_wide && b0 < n; b0 += 16) {
    const int r = min(b0 + 15, n - 1);
    bool wide = false;
    if (tid < D) {
      const float gr = sG[r * LD + tid];
      for (int t = b0; t < C; ++t) wide |= sG[t * LD + tid] - gr > SPAN_MAX;
      for (int s = b0; s <= r; ++s) wide |= gr - sG[s * LD + tid] > SPAN_MAX;
    }
    wide = __syncthreads_or(wide);
    if (wide && tid == 0 && a.steep) atomicOr(a.steep + (size_t)i * a.H + h, 1);
    // thread -> row t = b0 + tid / 4, columns s = b0 + tid % 4 + 4m
    const int t = b0 + (tid >> 2), sl = tid & 3;
    if (!wide) {
      for (int e = tid; e < 16 * D; e += NT) {
        const int s = e / D, j = e % D;
        sM[s * LD + j] = sK[(b0 + s) * LD + j] * __expf(sG[r * LD + j] - sG[(b0 + s) * LD + j]);
      }
      for (int e = tid; e < (C - b0) * D; e += NT) {
        const int tt = b0 + e / D, j = e % D;
        const float f = __expf(sG[tt * LD + j] - sG[r * LD + j]);
        sX[tt * LD + j] = sK[tt * LD + j] * f;
        sY[tt * LD + j] = sQ[tt * LD + j] * f;
      }
      __syncthreads();
      if (t < C) {
        float ac[4] = {0.f, 0.f, 0.f, 0.f}, pc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < D; ++j) {
          const float x = sX[t * LD + j], y = sY[t * LD + j];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float km = sM[(sl + 4 * m) * LD + j];
            ac[m] = fmaf(x, km, ac[m]);
            pc[m] = fmaf(y, km, pc[m]);
          }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int s = b0 + sl + 4 * m;
          sA[t * LC + s] = s < t ? ac[m] : 0.f;
          sP[t * LC + s] = s <= t ? pc[m] : 0.f;
        }
      }
    } else if (t < C) {
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        const int s = b0 + sl + 4 * m;
        float ac = 0.f, pc = 0.f;
        if (s <= t)
          for (int j = 0; j < D; ++j) {
            const float e = __expf(sG[t * LD + j] - sG[s * LD + j]) * sK[s * LD + j];
            ac = fmaf(sK[t * LD + j], e, ac);
            pc = fmaf(sQ[t * LD + j], e, pc);
          }
        sA[t * LC + s] = s < t ? ac : 0.f;
        sP[t * LC + s] = s <= t ? pc : 0.f;
      }
    }
    __syncthreads();
  }

  // the chunk's v into sY (free once a and P are formed), asynchronously, while the inverse and W run: fp32
  // inputs as they are (row stride LD), bf16 inputs as raw bf16 rows (widened before U~); rows past n zero
  {
    const Tin* vsrc = reinterpret_cast<const Tin*>(a.v) + ((int64_t)t0 * a.H + h) * D;
    constexpr int Q16 = D * (int)sizeof(Tin) / 16;  // 16-byte pieces of a row
    for (int e = tid; e < C * Q16; e += NT) {
      const int r = e / Q16, qq = e % Q16;
      float* dst = sizeof(Tin) == 4 ? sY + r * LD + 4 * qq : sY + r * (D / 2) + 4 * qq;
      cp_async16(dst, reinterpret_cast<const float*>(vsrc + (r < n ? r : 0) * rs) + 4 * qq, r < n ? 16 : 0);
    }
    cp_async_commit();
  }

  // the record's a; then A = diag(beta) a in place (the inverse's scratch) and T = (I + A)^-1, blocked by
  // 16 (T's upper blocks, the inverse's scratch, cleared after); then diag(beta) K+ in sX
  for (int e = tid; e < C * C; e += NT) w[BW_A + e] = sA[(e / C) * LC + e % C];
  __syncthreads();
  for (int e = tid; e < C * C; e += NT) sA[(e / C) * LC + e % C] *= sB[e / C];
  __syncthreads();
  unit_lower_inverse64<LC>(sA, sT, tid);
  __syncthreads();
  for (int e = tid; e < 6 * 256; e += NT) {  // upper blocks (r, c), r < c: (0,1) (0,2) (1,2) (0,3) (1,3) (2,3)
    const int blk = e >> 8, r = blk == 0 ? 0 : (blk < 3 ? blk - 1 : blk - 3), cb = blk == 0 ? 1 : (blk < 3 ? 2 : 3);
    sT[(16 * r + ((e >> 4) & 15)) * LC + 16 * cb + (e & 15)] = 0.f;
  }
  for (int e = tid; e < C * D; e += NT) {
    const int s = e / D, j = e % D;
    sX[s * LD + j] = sB[s] * sK[s * LD + j] * __expf(sG[s * LD + j]);
  }
  __syncthreads();

  // records: G, a, P, T, e^G_C, K^, Q+ (elementwise; G, K^ and Q+ already in the common case), then
  // W = T diag(beta) K+ and U~ = T diag(beta) V
  for (int e = tid; chunk_wide && e < C * D; e += NT) {
    const int t = e / D, j = e % D;
    const float G = sG[t * LD + j], GC = sG[(n - 1) * LD + j];
    w[BW_G + e] = G;
    w[BW_KH + e] = sK[t * LD + j] * __expf(GC - G);
    w[BW_QP + e] = sQ[t * LD + j] * __expf(G);
  }
  for (int e = tid; e < C * C; e += NT) {
    const int t = e / C, s = e % C;
    w[BW_P + e] = sP[t * LC + s];
    w[BW_T + e] = sT[t * LC + s];
  }
  if (tid < D) w[BW_GAM + tid] = __expf(sG[(n - 1) * LD + tid]);
  // W = T (diag(beta) K+) and U~ = T diag(beta) V: rows t = 4 ty + i, columns 4 tx + 64 mm + u; T's rows read
  // four columns s per 16-byte load; T is lower, so s runs to the thread's last row
  const int ty = tid >> 4, tx = tid & 15;
  auto t_product = [&](const float* sRhs, bool scale_beta, float* dst) {
    float acc[4][8] = {};
#pragma unroll 1
    for (int sb = 0; sb < 4 * ty + 4; sb += 4) {
      float x[4][4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const float4 v = *reinterpret_cast<const float4*>(sT + (4 * ty + ii) * LC + sb);
        x[ii][0] = v.x, x[ii][1] = v.y, x[ii][2] = v.z, x[ii][3] = v.w;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int s = sb + e;
        const float bs = scale_beta ? sB[s] : 1.f;
        const float4 y0 = *reinterpret_cast<const float4*>(sRhs + s * LD + 4 * tx);
        const float4 y1 = *reinterpret_cast<const float4*>(sRhs + s * LD + 4 * tx + 64);
        const float y[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
          const float xs = x[ii][e] * bs;
#pragma unroll
          for (int m = 0; m < 8; ++m) acc[ii][m] = fmaf(xs, y[m], acc[ii][m]);
        }
      }
    }
#pragma unroll
    for (int ii = 0; ii < 4; ++ii)
#pragma unroll
      for (int mm = 0; mm < 2; ++mm)
        *reinterpret_cast<float4*>(dst + (4 * ty + ii) * D + 4 * tx + 64 * mm) =
            make_float4(acc[ii][4 * mm], acc[ii][4 * mm + 1], acc[ii][4 * mm + 2], acc[ii][4 * mm + 3]);
  };
  t_product(sX, false, w + BW_W);
  cp_async_wait<0>();  // v
  __syncthreads();
  if constexpr (sizeof(Tin) == 4) {
    t_product(sY, true, w + BW_UT);
  } else {  // widen the raw bf16 rows into sX (free: W is done)
    for (int e = tid; e < C * D / 8; e += NT) {
      const int r = e / (D / 8), cc = e % (D / 8);
      const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(sY) + r * D + 8 * cc);
      const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
      float x[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // bf16 pairs, the lower element in the low half
        x[2 * q] = __uint_as_float(wv[q] << 16);
        x[2 * q + 1] = __uint_as_float(wv[q] & 0xFFFF0000u);
      }
      *reinterpret_cast<float4*>(sX + r * LD + 8 * cc) = make_float4(x[0], x[1], x[2], x[3]);
      *reinterpret_cast<float4*>(sX + r * LD + 8 * cc + 4) = make_float4(x[4], x[5], x[6], x[7]);
    }
    __syncthreads();
    t_product(sX, true, w + BW_UT);
  }
}

// ---------------------------------------------------------------------------------------------------
// 2. forward chain over the chunks of one (sequence, head, 16 value columns): entry states and U.
//    The next chunk's operands are copied in while the current one is processed (two stages).
// ---------------------------------------------------------------------------------------------------
constexpr int FS_STAGE = 2 * C * LD + C * CB + D;  // W, K^, U~ columns, e^G_C
constexpr int FS_PART = 20;                        // row stride of the partial sums (16 columns, padded)
constexpr size_t FWD_SMEM = (2 * FS_STAGE + D * CB + C * CB + 4 * D * FS_PART) * sizeof(float);

__global__ void __launch_bounds__(NTC, 1) bwd_fwd_chain_kernel(BackwardArgs a) {
  const int cb = blockIdx.x, h = blockIdx.y, i = blockIdx.z, tid = threadIdx.x, c0 = cb * CB;
  if (a.steep && !a.steep[(size_t)i * a.H + h]) return;  // the tensor-core forward pass covered it
  Seq sq;
  if (!seq_bounds(a, i, sq, false)) return;
  extern __shared__ float sm[];
  float* sS = sm + 2 * FS_STAGE;  // state columns [128][CB]
  float* sU = sS + D * CB;        // U columns [64][CB]
  float* sPart = sU + C * CB;     // K^^T U over four 16-token quarters [4][128][FS_PART]
  const float* s0 = nullptr;
  if (!a.init_zero) {
    const int slot = a.slot_ids[i];
    if (slot < 0 || slot >= a.num_slots) {
      if (tid == 0 && cb == 0) flag_status(a.status, KDA_DEV_SLOT_OOB);
    } else {
      s0 = a.pool + ((size_t)slot * a.H + h) * D * D;
    }
  }
  for (int e = tid; e < D * CB; e += NTC) sS[e] = s0 ? s0[(e / CB) * D + c0 + e % CB] : 0.f;
  const int nc = (sq.eos - sq.bos + C - 1) / C;
  auto issue = [&](int c) {
    float* st = sm + (c & 1) * FS_STAGE;
    const float* w = record(a, sq.bos + c * C, i, h);
    load_rows<NTC>(st, LD, w + BW_W, D, C, C, 0, D);
    load_rows<NTC>(st + C * LD, LD, w + BW_KH, D, C, C, 0, D);
    load_rows<NTC>(st + 2 * C * LD, CB, w + BW_UT, D, C, C, c0, CB);
    load_rows<NTC>(st + 2 * C * LD + C * CB, D, w + BW_GAM, D, 1, 1, 0, D);
    cp_async_commit();
  };
  if (nc > 0) issue(0);
  for (int c = 0; c < nc; ++c) {
    if (c + 1 < nc) {
      issue(c + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float* sW = sm + (c & 1) * FS_STAGE;
    const float* sKh = sW + C * LD;
    const float* sUt = sKh + C * LD;
    const float* sGam = sUt + C * CB;
    float* w = record(a, sq.bos + c * C, i, h);
    {  // the entry state, 16-byte stores
      const int j = tid >> 2, c4 = (tid & 3) * 4;
      *reinterpret_cast<float4*>(w + BW_H + j * D + c0 + c4) = *reinterpret_cast<const float4*>(sS + j * CB + c4);
    }
    // register tiles of 4 contiguous columns (16-byte shared loads of the state / U rows)
    if (tid < 256) {  // U = U~ - W S: row t = tid / 4
      const int t = tid >> 2, c4 = (tid & 3) * 4;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int j = 0; j < D; j += 8) dot8x4(sW + t * LD + j, 1, sS + j * CB + c4, CB, acc);
      const float4 ut = *reinterpret_cast<const float4*>(sUt + t * CB + c4);
      const float4 u = make_float4(ut.x - acc[0], ut.y - acc[1], ut.z - acc[2], ut.w - acc[3]);
      *reinterpret_cast<float4*>(sU + t * CB + c4) = u;
      *reinterpret_cast<float4*>(w + BW_U + t * D + c0 + c4) = u;
    }
    __syncthreads();
    {  // K^^T U: lane = row j of a 32-row group, all 16 columns in registers, tokens split in four quarters
       // (each token's U row is read once per warp, as a broadcast)
      const int warp = tid >> 5, lane = tid & 31;
      const int j = 32 * (warp & 3) + lane, tq = warp >> 2;
      float acc[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) acc[m] = 0.f;
#pragma unroll 4
      for (int t = 16 * tq; t < 16 * tq + 16; ++t) {
        const float x = sKh[t * LD + j];
        const float4* u = reinterpret_cast<const float4*>(sU + t * CB);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 y = u[q];
          acc[4 * q] = fmaf(x, y.x, acc[4 * q]);
          acc[4 * q + 1] = fmaf(x, y.y, acc[4 * q + 1]);
          acc[4 * q + 2] = fmaf(x, y.z, acc[4 * q + 2]);
          acc[4 * q + 3] = fmaf(x, y.w, acc[4 * q + 3]);
        }
      }
      float4* dst = reinterpret_cast<float4*>(sPart + (tq * D + j) * FS_PART);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
    }
    __syncthreads();
    {  // S = Diag(e^G_C) S + the four quarters: row j = tid / 4 (own elements only: in place)
      const int j = tid >> 2, c4 = (tid & 3) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int tq = 0; tq < 4; ++tq) {
        const float4 p = *reinterpret_cast<const float4*>(sPart + (tq * D + j) * FS_PART + c4);
        acc.x += p.x, acc.y += p.y, acc.z += p.z, acc.w += p.w;
      }
      const float gm = sGam[j];
      float4* sp = reinterpret_cast<float4*>(sS + j * CB + c4);
      const float4 sv = *sp;
      *sp = make_float4(fmaf(gm, sv.x, acc.x), fmaf(gm, sv.y, acc.y), fmaf(gm, sv.z, acc.z), fmaf(gm, sv.w, acc.w));
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------------------------------
// 3. reverse chain: dS' at every chunk exit, dU, and dS_0.  Stage A (P, K^, Q+, dO columns, e^G_C) is
//    double-buffered and copied in a chunk ahead; stage B (W) is copied in during the previous chunk's
//    dU step.  Threads 0-255 form dU while threads 256-511 form Q+^T dO for rows j and j + 64, and then
//    finish dS for those rows; register tiles of 4 contiguous columns read 16-byte rows of dS', dU, dO.
// ---------------------------------------------------------------------------------------------------
constexpr int RS_A = C * LC + 2 * C * LD + C * CB + D;  // P, K^, Q+, raw dO columns (<= 64 x 16 fp32), e^G_C
constexpr int RS_B = C * LD;                            // W
constexpr size_t REV_SMEM = (2 * RS_A + RS_B + D * CB + C * CB) * sizeof(float);

template <typename Tin>
__global__ void __launch_bounds__(NTC, 1) bwd_rev_chain_kernel(BackwardArgs a) {
  const int cb = blockIdx.x, h = blockIdx.y, i = blockIdx.z, tid = threadIdx.x, c0 = cb * CB;
  if (a.steep && !a.steep[(size_t)i * a.H + h]) return;  // the tensor-core reverse pass covered it
  Seq sq;
  if (!seq_bounds(a, i, sq, false)) return;
  extern __shared__ float sm[];
  float* sW = sm + 2 * RS_A;     // W
  float* sdS = sW + RS_B;        // dS columns [128][CB]
  float* sdU = sdS + D * CB;     // dU columns [64][CB]
  const float* dfin = a.d_final ? a.d_final + ((size_t)i * a.H + h) * D * D : nullptr;
  for (int e = tid; e < D * CB; e += NTC) sdS[e] = dfin ? dfin[(e / CB) * D + c0 + e % CB] : 0.f;
  const int nc = (sq.eos - sq.bos + C - 1) / C;
  const int64_t rs = (int64_t)a.H * D;
  constexpr int DO_Q = CB * (int)sizeof(Tin) / 16;  // 16-byte pieces of one dO row slice
  auto issue_a = [&](int c, int buf) {
    float* st = sm + buf * RS_A;
    const int t0 = sq.bos + c * C, n = min(C, sq.eos - t0);
    const float* w = record(a, t0, i, h);
    load_rows<NTC>(st, LC, w + BW_P, C, C, C, 0, C);
    load_rows<NTC>(st + C * LC, LD, w + BW_KH, D, C, C, 0, D);
    load_rows<NTC>(st + C * LC + C * LD, LD, w + BW_QP, D, C, C, 0, D);
    const Tin* src = reinterpret_cast<const Tin*>(a.d_out) + ((int64_t)t0 * a.H + h) * D + c0;
    Tin* dst = reinterpret_cast<Tin*>(st + C * LC + 2 * C * LD);
    for (int e = tid; e < C * DO_Q; e += NTC) {
      const int r = e / DO_Q, q = e % DO_Q;
      cp_async16(reinterpret_cast<float*>(dst + r * CB + q * (16 / (int)sizeof(Tin))),
                 reinterpret_cast<const float*>(src + (r < n ? r : 0) * rs + q * (16 / (int)sizeof(Tin))),
                 r < n ? 16 : 0);
    }
    load_rows<NTC>(st + C * LC + 2 * C * LD + C * CB, D, w + BW_GAM, D, 1, 1, 0, D);
    cp_async_commit();
  };
  auto issue_b = [&](int c) {
    const float* w = record(a, sq.bos + c * C, i, h);
    load_rows<NTC>(sW, LD, w + BW_W, D, C, C, 0, D);
    cp_async_commit();
  };
  if (nc > 0) {
    issue_a(nc - 1, 0);
    issue_b(nc - 1);
  }
  auto fma4 = [](float x, const float (&y)[4], float (&acc)[4]) {
#pragma unroll
    for (int m = 0; m < 4; ++m) acc[m] = fmaf(x, y[m], acc[m]);
  };
  for (int c = nc - 1, k = 0; c >= 0; --c, ++k) {
    cp_async_wait<1>();  // stage A of chunk c has landed (stage B may still be in flight)
    __syncthreads();
    if (c > 0) issue_a(c - 1, (k + 1) & 1);
    const float* sP = sm + (k & 1) * RS_A;
    const float* sKh = sP + C * LC;
    const float* sQp = sKh + C * LD;
    const Tin* sDO = reinterpret_cast<const Tin*>(sQp + C * LD);
    const float* sGam = sQp + C * LD + C * CB;
    float* w = record(a, sq.bos + c * C, i, h);
    {  // dS' of this chunk, 16-byte stores
      const int j = tid >> 2, c4 = (tid & 3) * 4;
      *reinterpret_cast<float4*>(w + BW_DS + j * D + c0 + c4) = *reinterpret_cast<const float4*>(sdS + j * CB + c4);
    }
    const int c4 = (tid & 3) * 4;
    float y0[4] = {0.f, 0.f, 0.f, 0.f}, y1[4] = {0.f, 0.f, 0.f, 0.f};
    if (tid < 256) {  // dU = P^T dO + K^ dS': row t = tid / 4
      const int t = tid >> 2;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int s = t & ~7; s < C; s += 8) {  // P[s][t] = 0 for s < t
        float pv[8], ov[8][4];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          pv[r] = sP[(s + r) * LC + t];
          ld4(sDO + (s + r) * CB + c4, ov[r]);
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) fma4(pv[r], ov[r], acc);
      }
#pragma unroll 1
      for (int j = 0; j < D; j += 8) dot8x4(sKh + t * LD + j, 1, sdS + j * CB + c4, CB, acc);
      const float4 u = make_float4(acc[0], acc[1], acc[2], acc[3]);
      *reinterpret_cast<float4*>(sdU + t * CB + c4) = u;
      *reinterpret_cast<float4*>(w + BW_DU + t * D + c0 + c4) = u;
    } else {  // Q+^T dO for rows j and j + 64
      const int j = (tid - 256) >> 2;
#pragma unroll 1
      for (int t = 0; t < C; t += 8) {
        float q0[8], q1[8], ov[8][4];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          q0[r] = sQp[(t + r) * LD + j];
          q1[r] = sQp[(t + r) * LD + j + 64];
          ld4(sDO + (t + r) * CB + c4, ov[r]);
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          fma4(q0[r], ov[r], y0);
          fma4(q1[r], ov[r], y1);
        }
      }
    }
    if (c > 0)
      cp_async_wait<1>();  // stage B of chunk c has landed (the next stage A may still be in flight)
    else
      cp_async_wait<0>();
    __syncthreads();
    if (tid >= 256) {  // dS = Q+^T dO + Diag(e^G_C) dS' - W^T dU for rows j and j + 64 (in place)
      const int j = (tid - 256) >> 2;
#pragma unroll 1
      for (int t = 0; t < C; t += 8) {
        float w0[8], w1[8], uv[8][4];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          w0[r] = -sW[(t + r) * LD + j];
          w1[r] = -sW[(t + r) * LD + j + 64];
          ld4(sdU + (t + r) * CB + c4, uv[r]);
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          fma4(w0[r], uv[r], y0);
          fma4(w1[r], uv[r], y1);
        }
      }
      float* s0p = sdS + j * CB + c4;
      float* s1p = sdS + (j + 64) * CB + c4;
      const float g0 = sGam[j], g1 = sGam[j + 64];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        s0p[m] = fmaf(g0, s0p[m], y0[m]);
        s1p[m] = fmaf(g1, s1p[m], y1[m]);
      }
    }
    __syncthreads();
    if (c > 0) issue_b(c - 1);
  }
  __syncthreads();  // (a sequence without chunks: the fill above used another thread mapping)
  if (a.d_init) {
    float* dst = a.d_init + ((size_t)i * a.H + h) * D * D;
    const int j = tid >> 2, c4 = (tid & 3) * 4;
    *reinterpret_cast<float4*>(dst + j * D + c0 + c4) = *reinterpret_cast<const float4*>(sdS + j * CB + c4);
  }
}

// ---------------------------------------------------------------------------------------------------
// 4. state products of one (chunk, head): dQ+ = dO S^T, dW = -dU S^T, d(e^G_C), dP = tril(dO U^T), dK^ = U dS'^T,
// as two split-bf16 tcgen05 MMAs:
//   set 1: D1 = S [dO; dU]^T          (M = 128 key channels j, N = 128, K = 128 value channels)
//          columns 0..63 = dQ+^T [j][t], columns 64..127 = (dU S^T)^T = -dW^T [j][t]
//   set 2: D2 = [U; dO] [dS'; U]^T    (M = 128, N = 192, K = 128)
//          rows 0..63, columns 0..127 = U dS'^T = dK^ [s][j]; rows 64..127, columns 128..191 = dO U^T -> dP
// Every fp32 operand enters as bf16 hi + lo and the products hi*hi + hi*lo + lo*hi accumulate in fp32
// (relative operand error ~2^-16; the gradients are held to 1e-4 of their rms).  d(e^G_C) stays on the CUDA
// cores, read from the same loads that build the operands.
// ---------------------------------------------------------------------------------------------------
constexpr uint32_t SG_A = 0;            // A1 = S (hi, lo), later A2 = [U; dO]: [128][128] bf16, two 16 KB K-blocks each
constexpr uint32_t SG_B1 = 65536;       // B1 = [dO; dU] (hi, lo): [128][128]
constexpr uint32_t SG_B2 = 131072;      // B2 = [dS'; U] (hi, lo): [192][128], two 24 KB K-blocks each
constexpr uint32_t SG_BAR = 229376;
constexpr size_t STATE_TC_SMEM = SG_BAR + 64 + 1024;

// offset of the 16-byte chunk cc (channels 8cc .. 8cc + 7) of row r in a [rows][128] K-major tile
__device__ __forceinline__ uint32_t kt_off(int r, int cc, int rows) {
  return (uint32_t)(cc >> 3) * (uint32_t)(rows * 128) + tc::sw128_chunk(r, cc & 7);
}
__device__ __forceinline__ void split8(uint8_t* hi, uint8_t* lo, const float* v) {
  uint4 h, l;
  tc::split_pair(v[0], v[1], h.x, l.x);
  tc::split_pair(v[2], v[3], h.y, l.y);
  tc::split_pair(v[4], v[5], h.z, l.z);
  tc::split_pair(v[6], v[7], h.w, l.w);
  *reinterpret_cast<uint4*>(hi) = h;
  *reinterpret_cast<uint4*>(lo) = l;
}
__device__ __forceinline__ void load8(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const bf16* p, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = __uint_as_float(w[e] << 16);
    v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

// D (tensor memory) = sum over the three split products of A [128][128] and B [N][128], both K-major
__device__ __forceinline__ void issue_split(uint32_t d, uint32_t a, uint32_t b, int brows, uint32_t idesc) {
  const uint32_t ablk = 128 * 128, bblk = (uint32_t)brows * 128;
#pragma unroll
  for (int part = 0; part < 3; ++part) {
    const uint32_t aa = a + (part == 2 ? 2 * ablk : 0), bb = b + (part == 1 ? 2 * bblk : 0);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_ss(d, tc::sdesc(aa + (uint32_t)(ks >> 2) * ablk + (uint32_t)(ks & 3) * 32u),
                 tc::sdesc(bb + (uint32_t)(ks >> 2) * bblk + (uint32_t)(ks & 3) * 32u), idesc, (part | ks) != 0);
  }
}

template <typename Tin>
__global__ void __launch_bounds__(NT, 1) bwd_state_grads_tc_kernel(BackwardArgs a) {
  const int c = blockIdx.x, h = blockIdx.y, i = blockIdx.z, tid = threadIdx.x, warp = tid >> 5;
  Seq sq;
  if (!seq_bounds(a, i, sq, false)) return;
  const int t0 = sq.bos + c * C;
  if (t0 >= sq.eos) return;
  const int n = min(C, sq.eos - t0);
  float* w = record(a, t0, i, h);
  extern __shared__ uint8_t sgraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sgraw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + SG_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SG_BAR + 16);
  const Tin* dO = reinterpret_cast<const Tin*>(a.d_out) + ((int64_t)t0 * a.H + h) * D;
  const int64_t ldo = (int64_t)a.H * D;
  constexpr uint32_t AH = 2 * 16384, B1H = 2 * 16384, B2H = 2 * 24576;  // bytes of a hi (or lo) tile
  if (warp == 0) tc::tmem_alloc(tslot, 512);
  if (tid == 0) {
    tc::bar_init(bar, 1);
    tc::bar_fence_init();
  }
  // set 1 and set 2's B operand: S and dS' rows j (with d(e^G_C)_j = sum_l dS'_jl S_jl), dU, dO, U.  Each
  // thread's global loads go out in groups of four rows before any of them is split (one memory latency
  // per group instead of one per row)
  {
    const int cc = tid & 15;
#pragma unroll 1
    for (int jb = tid >> 4; jb < D; jb += 4 * (NT / 16)) {
      float x[4][8], y[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = jb + u * (NT / 16);
        load8(w + BW_H + j * D + 8 * cc, x[u]);
        load8(w + BW_DS + j * D + 8 * cc, y[u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = jb + u * (NT / 16);
        split8(sm + SG_A + kt_off(j, cc, 128), sm + SG_A + AH + kt_off(j, cc, 128), x[u]);
        split8(sm + SG_B2 + kt_off(j, cc, 192), sm + SG_B2 + B2H + kt_off(j, cc, 192), y[u]);
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) s = fmaf(x[u][e], y[u][e], s);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (cc == 0) w[BW_DGAM + j] = s;
      }
    }
    {  // rows t = tid / 16 + 16 u, u < 4: all of C = 64
      float x[4][8], y[4][8], z[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = (tid >> 4) + u * (NT / 16);
        if (t < n) load8(dO + t * ldo + 8 * cc, x[u]);
        else for (int e = 0; e < 8; ++e) x[u][e] = 0.f;
        load8(w + BW_DU + t * D + 8 * cc, y[u]);
        load8(w + BW_U + t * D + 8 * cc, z[u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = (tid >> 4) + u * (NT / 16);
        split8(sm + SG_B1 + kt_off(t, cc, 128), sm + SG_B1 + B1H + kt_off(t, cc, 128), x[u]);
        split8(sm + SG_B1 + kt_off(64 + t, cc, 128), sm + SG_B1 + B1H + kt_off(64 + t, cc, 128), y[u]);
        split8(sm + SG_B2 + kt_off(128 + t, cc, 192), sm + SG_B2 + B2H + kt_off(128 + t, cc, 192), z[u]);
      }
    }
  }
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = *tslot;
  const uint32_t base = tc::smem_u32(sm);
  if (tid == 0) {
    issue_split(tm, base + SG_A, base + SG_B1, 128, tc::idesc_bf16(128, 128));
    tc::commit(bar);
  }
  bool ok = __syncthreads_and(tc::bar_wait(bar, 0u)) != 0;
  // set 2's A operand over set 1's: [U; dO] (loads grouped as above)
  if (ok) {
    tc::fence_after_sync();
    const int cc = tid & 15;
    float x[4][8], z[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = (tid >> 4) + u * (NT / 16);
      if (t < n) load8(dO + t * ldo + 8 * cc, x[u]);
      else for (int e = 0; e < 8; ++e) x[u][e] = 0.f;
      load8(w + BW_U + t * D + 8 * cc, z[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = (tid >> 4) + u * (NT / 16);
      split8(sm + SG_A + kt_off(t, cc, 128), sm + SG_A + AH + kt_off(t, cc, 128), z[u]);
      split8(sm + SG_A + kt_off(64 + t, cc, 128), sm + SG_A + AH + kt_off(64 + t, cc, 128), x[u]);
    }
    tc::fence_proxy_async();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (ok && tid == 0) {
    issue_split(tm + 128, base + SG_A, base + SG_B2, 192, tc::idesc_bf16(128, 192));
    tc::commit(bar);
  }
  const int q = warp & 3, g = warp >> 2, r = 32 * q + (tid & 31);
  const uint32_t trow = tm + ((uint32_t)(q * 32) << 16);
  if (ok) {  // set 1 (complete): dQ+ [t][j] and dW [t][j], one coalesced row per warp store
    float v[32];
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      tc::tmem_ld32(trow + 64 * g + 32 * half, v);
      float* dst = w + (g ? BW_DW : BW_DQP) + (size_t)(32 * half) * D + r;
#pragma unroll
      for (int e = 0; e < 32; ++e) dst[(size_t)e * D] = g ? -v[e] : v[e];
    }
  }
  ok = __syncthreads_and(ok && tc::bar_wait(bar, 1u)) != 0;
  if (ok) {  // set 2: dK^ rows (lanes 0..63), dP rows (lanes 64..127)
    tc::fence_after_sync();
    float v[32];
    if (q < 2) {
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        tc::tmem_ld32(trow + 128 + 64 * g + 32 * half, v);
        float4* dst = reinterpret_cast<float4*>(w + BW_DKH + (size_t)r * D + 64 * g + 32 * half);
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
      }
    } else {
      const int t = r - 64;
      tc::tmem_ld32(trow + 256 + 32 * g, v);
      float4* dst = reinterpret_cast<float4*>(w + BW_DP + (size_t)t * C + 32 * g);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int s0 = 32 * g + 4 * e;
        dst[e] = make_float4(s0 <= t ? v[4 * e] : 0.f, s0 + 1 <= t ? v[4 * e + 1] : 0.f, s0 + 2 <= t ? v[4 * e + 2] : 0.f,
                             s0 + 3 <= t ? v[4 * e + 3] : 0.f);
      }
    }
  } else if (tid == 0) {
    flag_status(a.status, KDA_DEV_TIMEOUT);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tm, 512);
}

// ---------------------------------------------------------------------------------------------------
// 5. WY backward of one (chunk, head): dT, dA, dK+ = diag(beta) T^T dW, dv = diag(beta) T^T dU, dbeta part
// ---------------------------------------------------------------------------------------------------
constexpr size_t WY_SMEM = (2 * C * LC + 5 * C * LD + C) * sizeof(float);

template <typename Tin>
__global__ void __launch_bounds__(NT, 1) bwd_wy_grads_kernel(BackwardArgs a) {
  const int c = blockIdx.x, h = blockIdx.y, i = blockIdx.z, tid = threadIdx.x;
  Seq sq;
  if (!seq_bounds(a, i, sq, false)) return;
  const int t0 = sq.bos + c * C;
  if (t0 >= sq.eos) return;
  const int n = min(C, sq.eos - t0);
  float* w = record(a, t0, i, h);
  extern __shared__ float sm[];
  float* sT = sm;                // T [64][LC]
  float* sM = sT + C * LC;       // dT [64][LC]
  float* sKp = sM + C * LC;      // K+ [64][LD]; later T^T dT [64][LC]
  float* sV = sKp + C * LD;      // V [64][LD]
  float* sDW = sV + C * LD;      // dW [64][LD]
  float* sDU = sDW + C * LD;     // dU [64][LD]
  float* sGw = sDU + C * LD;     // G [64][LD] (for K+ = K o e^G)
  float* sB = sGw + C * LD;      // beta [64]
  const int64_t rs = (int64_t)a.H * D;
  load_rows<NT>(sT, LC, w + BW_T, C, C, C, 0, C);
  load_rows<NT>(sKp, LD, reinterpret_cast<const Tin*>(a.k) + ((int64_t)t0 * a.H + h) * D, rs, C, n, 0, D);
  load_rows<NT>(sV, LD, reinterpret_cast<const Tin*>(a.v) + ((int64_t)t0 * a.H + h) * D, rs, C, n, 0, D);
  load_rows<NT>(sDW, LD, w + BW_DW, D, C, C, 0, D);
  load_rows<NT>(sDU, LD, w + BW_DU, D, C, C, 0, D);
  load_rows<NT>(sGw, LD, w + BW_G, D, C, C, 0, D);
  if (tid < C) sB[tid] = tid < n ? a.beta[(int64_t)(t0 + tid) * a.H + h] : 0.f;
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  for (int e = tid; e < C * D; e += NT) sKp[(e / D) * LD + e % D] *= __expf(sGw[(e / D) * LD + e % D]);
  __syncthreads();
  const int ty = tid >> 4, tx = tid & 15;
  {  // dT_ts = beta_s (dW_t . K+_s + dU_t . V_s), 16-byte loads along j
    float acc[4][4] = {};
#pragma unroll 2
    for (int j = 0; j < D; j += 4) {
      float4 x[4], y[4], p[4], q[4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        x[ii] = *reinterpret_cast<const float4*>(sDW + (ty + 16 * ii) * LD + j);
        y[ii] = *reinterpret_cast<const float4*>(sDU + (ty + 16 * ii) * LD + j);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        p[m] = *reinterpret_cast<const float4*>(sKp + (tx + 16 * m) * LD + j);
        q[m] = *reinterpret_cast<const float4*>(sV + (tx + 16 * m) * LD + j);
      }
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float v = acc[ii][m];
          v = fmaf(x[ii].x, p[m].x, fmaf(y[ii].x, q[m].x, v));
          v = fmaf(x[ii].y, p[m].y, fmaf(y[ii].y, q[m].y, v));
          v = fmaf(x[ii].z, p[m].z, fmaf(y[ii].z, q[m].z, v));
          acc[ii][m] = fmaf(x[ii].w, p[m].w, fmaf(y[ii].w, q[m].w, v));
        }
    }
#pragma unroll
    for (int ii = 0; ii < 4; ++ii)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int s = tx + 16 * m;
        sM[(ty + 16 * ii) * LC + s] = sB[s] * acc[ii][m];
      }
  }
  {  // dB_K = T^T dW, dB_V = T^T dU (rows s = 4 ty + i, columns j = 4 tx + 64 (m / 4) + m % 4, T lower:
     // t >= s); dK+ = beta dB_K, dv = beta dB_V, dbeta part
    float bk[4][8] = {}, bv[4][8] = {};
    for (int t = 4 * ty; t < C; ++t) {
      float4 y[2], z[2];
      const float4 x4 = *reinterpret_cast<const float4*>(sT + t * LC + 4 * ty);
      const float x[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        y[mm] = *reinterpret_cast<const float4*>(sDW + t * LD + 4 * tx + 64 * mm);
        z[mm] = *reinterpret_cast<const float4*>(sDU + t * LD + 4 * tx + 64 * mm);
      }
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
          bk[ii][4 * mm + 0] = fmaf(x[ii], y[mm].x, bk[ii][4 * mm + 0]);
          bk[ii][4 * mm + 1] = fmaf(x[ii], y[mm].y, bk[ii][4 * mm + 1]);
          bk[ii][4 * mm + 2] = fmaf(x[ii], y[mm].z, bk[ii][4 * mm + 2]);
          bk[ii][4 * mm + 3] = fmaf(x[ii], y[mm].w, bk[ii][4 * mm + 3]);
          bv[ii][4 * mm + 0] = fmaf(x[ii], z[mm].x, bv[ii][4 * mm + 0]);
          bv[ii][4 * mm + 1] = fmaf(x[ii], z[mm].y, bv[ii][4 * mm + 1]);
          bv[ii][4 * mm + 2] = fmaf(x[ii], z[mm].z, bv[ii][4 * mm + 2]);
          bv[ii][4 * mm + 3] = fmaf(x[ii], z[mm].w, bv[ii][4 * mm + 3]);
        }
    }
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const int s = 4 * ty + ii;
      const float b = sB[s];
      float part = 0.f;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int j = 4 * tx + 64 * (m >> 2) + (m & 3);
        part = fmaf(bk[ii][m], sKp[s * LD + j], part);
        part = fmaf(bv[ii][m], sV[s * LD + j], part);
        w[BW_DKP + s * D + j] = b * bk[ii][m];
        if (s < n) a.dv[((int64_t)(t0 + s) * a.H + h) * D + j] = b * bv[ii][m];
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (tx == 0) w[BW_DBETA + s] = part;
    }
  }
  __syncthreads();
  float* sN = sKp;  // T^T dT [64][LC]
  {  // T^T dT: rows s = 4 ty + i (T lower: t >= s), columns tx + 16 m
    float acc[4][4] = {};
    for (int t = 4 * ty; t < C; ++t) {
      float y[4];
      const float4 x4 = *reinterpret_cast<const float4*>(sT + t * LC + 4 * ty);
      const float x[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) y[m] = sM[t * LC + tx + 16 * m];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int m = 0; m < 4; ++m) acc[ii][m] = fmaf(x[ii], y[m], acc[ii][m]);
    }
    __syncthreads();
#pragma unroll
    for (int ii = 0; ii < 4; ++ii)
#pragma unroll
      for (int m = 0; m < 4; ++m) sN[(4 * ty + ii) * LC + tx + 16 * m] = acc[ii][m];
  }
  __syncthreads();
  {  // dA = -(T^T dT) T^T, strictly lower: rows s = 4 ty + i, columns u = tx + 16 m, four t per 16-byte load
    float acc[4][4] = {};
#pragma unroll 2
    for (int tb = 0; tb < C; tb += 4) {
      float x[4][4], y[4][4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const float4 v = *reinterpret_cast<const float4*>(sN + (4 * ty + ii) * LC + tb);
        x[ii][0] = v.x, x[ii][1] = v.y, x[ii][2] = v.z, x[ii][3] = v.w;
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 v = *reinterpret_cast<const float4*>(sT + (tx + 16 * m) * LC + tb);
        y[m][0] = v.x, y[m][1] = v.y, y[m][2] = v.z, y[m][3] = v.w;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int ii = 0; ii < 4; ++ii)
#pragma unroll
          for (int m = 0; m < 4; ++m) acc[ii][m] = fmaf(x[ii][e], y[m][e], acc[ii][m]);
    }
#pragma unroll
    for (int ii = 0; ii < 4; ++ii)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int s = 4 * ty + ii, u = tx + 16 * m;
        w[BW_DA + s * C + u] = u < s ? -acc[ii][m] : 0.f;
      }
  }
}

// ---------------------------------------------------------------------------------------------------
// 6. assembly of one (chunk, head, 64 channels): pair-decay terms, dq, dk, dg, dbeta
// ---------------------------------------------------------------------------------------------------
constexpr int NTA = 512;  // threads of the assembly kernel
constexpr size_t ASM_SMEM = (11 * C * LC + 2 * 16 * LC + 2 * C) * sizeof(float);

template <typename Tin>
__global__ void __launch_bounds__(NTA, 1) bwd_assemble_kernel(BackwardArgs a) {
  const int c = blockIdx.x, h = blockIdx.y >> 1, half = blockIdx.y & 1, i = blockIdx.z, tid = threadIdx.x;
  Seq sq;
  if (!seq_bounds(a, i, sq, false)) return;
  const int t0 = sq.bos + c * C;
  if (t0 >= sq.eos) return;
  const int n = min(C, sq.eos - t0);
  const int j0 = half * HC;
  float* w = record(a, t0, i, h);
  extern __shared__ float sm[];
  float* sK = sm;               // k [64][LC] (this CTA's 64 channels)
  float* sQ = sK + C * LC;      // q
  float* sG = sQ + C * LC;      // G
  float* sEp = sG + C * LC;     // e^(G_t - G_r) of the current block; later dG
  float* sDP = sEp + C * LC;    // dP; later the G_C terms dK^ o K^
  float* sDA = sDP + C * LC;    // dA (beta not folded in)
  float* sDKC = sDA + C * LC;   // the sums over t >= s of dk_s (each row written by its own block)
  float* sKm = sDKC + C * LC;   // k o e^(G_r - G_s) of the current block [16][LC]
  float* sEm = sKm + 16 * LC;   // e^(G_r - G_s) [16][LC]
  float* sYc = sEm + 16 * LC;   // common case: k o e^(G_C - G) [64][LC]
  float* sGQ = sYc + C * LC;    // the records' dQ+, dK+, dK^ of this CTA's 64 channels [64][LC] each
  float* sGK = sGQ + C * LC;
  float* sGH = sGK + C * LC;
  float* sB = sGH + C * LC;     // beta [64]
  float* sDiag = sB + C;        // dP_tt [64] (the diagonal is kept out of the pair sums: in dG its two
                                // contributions, through q_t and through k_t, cancel exactly)
  const int64_t rs = (int64_t)a.H * D;
  const int64_t in0 = ((int64_t)t0 * a.H + h) * D;
  load_rows<NTA>(sK, LC, reinterpret_cast<const Tin*>(a.k) + in0, rs, C, n, j0, HC);
  load_rows<NTA>(sQ, LC, reinterpret_cast<const Tin*>(a.q) + in0, rs, C, n, j0, HC);
  load_rows<NTA>(sG, LC, w + BW_G, D, C, C, j0, HC);
  load_rows<NTA>(sDP, LC, w + BW_DP, C, C, C, 0, C);
  load_rows<NTA>(sDA, LC, w + BW_DA, C, C, C, 0, C);
  if (tid < C) sB[tid] = tid < n ? a.beta[(int64_t)(t0 + tid) * a.H + h] : 0.f;
  cp_async_commit();
  load_rows<NTA>(sGQ, LC, w + BW_DQP, D, C, C, j0, HC);  // used at the end: left in flight until then
  load_rows<NTA>(sGK, LC, w + BW_DKP, D, C, C, j0, HC);
  load_rows<NTA>(sGH, LC, w + BW_DKH, D, C, C, j0, HC);
  cp_async_commit();
  cp_async_wait<1>();
  __syncthreads();
  if (tid < C) {
    sDiag[tid] = sDP[tid * LC + tid];
    sDP[tid * LC + tid] = 0.f;
  }
  {  // each channel's decay span over the chunk (with its start, G = 0): eight tokens per thread, then per channel
    const int jj = tid & (HC - 1), part = tid / HC;
    float gmin = 0.f, gmax = 0.f;
#pragma unroll
    for (int u = 0; u < C / 8; ++u) {
      const float g = sG[(8 * part + u) * LC + jj];
      gmin = fminf(gmin, g), gmax = fmaxf(gmax, g);
    }
    sKm[part * HC + jj] = gmin;
    sEm[part * HC + jj] = gmax;
  }
  __syncthreads();
  const int ty = tid >> 4, tx = tid & 15;    // own elements: rows ty + 32 ii, channels (own_col)
  const int orow = tid >> 5, ocol = tid & 31;  // in block b0: row b0 + orow, channels ocol + 32 mm
  float dqp[2][4] = {}, dkr[2][4] = {}, dkc[2][4] = {};
  bool chunk_wide = false;  // some channel's decay span over the chunk above SPAN_MAX
  if (tid < HC) {
    float gmin = 0.f, gmax = 0.f;
#pragma unroll
    for (int part = 0; part < NTA / HC; ++part) gmin = fminf(gmin, sKm[part * HC + tid]), gmax = fmaxf(gmax, sEm[part * HC + tid]);
    chunk_wide = gmax - gmin > SPAN_MAX;
  }
  chunk_wide = __syncthreads_or(chunk_wide);
  // own elements: rows 2 ty + ii and channels 4 tx + m in the common case (16-byte loads), rows ty + 32 ii and
  // channels tx + 16 m when the blocks take their own references
  auto own_col = [&](int m) { return chunk_wide ? tx + 16 * m : 4 * tx + m; };
  auto own_row = [&](int ii) { return chunk_wide ? ty + 32 * ii : 2 * ty + ii; };
  if (!chunk_wide) {
    // Common case: every pair decay through the chunk's last token, e^(G_t - G_s) = e^(G_t - G_C) e^(G_C - G_s):
    //   dq~_t = e^(G_t - G_C) (dP Y)_t,  dk_r,t = beta_t e^(G_t - G_C) (dA Y)_t,
    //   dk_c,s = e^(G_C - G_s) (dP^T Xq + (diag(beta) dA)^T X)_s
    // with X = k o e^(G - G_C), Xq = q o e^(G - G_C), Y = k o e^(G_C - G) (dP without its diagonal, dA strictly
    // lower: the sums run over s < t and t > s).
    float* sXc = sEp;    // X
    float* sXq = sDKC;   // Xq
    for (int e = tid; e < C * HC / 4; e += NTA) {
      const int t = e >> 4, j = (e & 15) * 4;
      const float4 k4 = *reinterpret_cast<const float4*>(sK + t * LC + j);
      const float4 q4 = *reinterpret_cast<const float4*>(sQ + t * LC + j);
      const float4 g4 = *reinterpret_cast<const float4*>(sG + t * LC + j);
      const float4 c4 = *reinterpret_cast<const float4*>(sG + (C - 1) * LC + j);
      const float kk[4] = {k4.x, k4.y, k4.z, k4.w}, qq[4] = {q4.x, q4.y, q4.z, q4.w};
      const float gg[4] = {g4.x, g4.y, g4.z, g4.w}, gc[4] = {c4.x, c4.y, c4.z, c4.w};
      float x[4], xq[4], y[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float e1 = __expf(gg[u] - gc[u]);
        x[u] = kk[u] * e1;
        xq[u] = qq[u] * e1;
        y[u] = kk[u] * __expf(gc[u] - gg[u]);
      }
      *reinterpret_cast<float4*>(sXc + t * LC + j) = make_float4(x[0], x[1], x[2], x[3]);
      *reinterpret_cast<float4*>(sXq + t * LC + j) = make_float4(xq[0], xq[1], xq[2], xq[3]);
      *reinterpret_cast<float4*>(sYc + t * LC + j) = make_float4(y[0], y[1], y[2], y[3]);
    }
    __syncthreads();
    // own rows r0 = 2 ty, r1 = 2 ty + 1: their dP and dA entries come four columns (row sums) or two rows
    // (column sums) per 16-byte or 8-byte load
    const int jc = 4 * tx, r0 = 2 * ty, r1 = r0 + 1;
    const int send = (r1 + 4) & ~3;  // row sums over s < t, in steps of four (entries at s >= t are zero)
#pragma unroll 2
    for (int sb = 0; sb < send; sb += 4) {
      const float4 p04 = *reinterpret_cast<const float4*>(sDP + r0 * LC + sb);
      const float4 p14 = *reinterpret_cast<const float4*>(sDP + r1 * LC + sb);
      const float4 q04 = *reinterpret_cast<const float4*>(sDA + r0 * LC + sb);
      const float4 q14 = *reinterpret_cast<const float4*>(sDA + r1 * LC + sb);
      const float p0[4] = {p04.x, p04.y, p04.z, p04.w}, p1[4] = {p14.x, p14.y, p14.z, p14.w};
      const float q0[4] = {q04.x, q04.y, q04.z, q04.w}, q1[4] = {q14.x, q14.y, q14.z, q14.w};
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float4 y4 = *reinterpret_cast<const float4*>(sYc + (sb + v) * LC + jc);
        const float y[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          dqp[0][u] = fmaf(p0[v], y[u], dqp[0][u]);
          dqp[1][u] = fmaf(p1[v], y[u], dqp[1][u]);
          dkr[0][u] = fmaf(q0[v], y[u], dkr[0][u]);
          dkr[1][u] = fmaf(q1[v], y[u], dkr[1][u]);
        }
      }
    }
#pragma unroll 4
    for (int t = r0 + 1; t < C; ++t) {  // column sums (entries at t <= s are zero)
      const float4 x4 = *reinterpret_cast<const float4*>(sXc + t * LC + jc);
      const float4 z4 = *reinterpret_cast<const float4*>(sXq + t * LC + jc);
      const float x[4] = {x4.x, x4.y, x4.z, x4.w}, xq[4] = {z4.x, z4.y, z4.z, z4.w};
      const float bt = sB[t];
      const float2 pp = *reinterpret_cast<const float2*>(sDP + t * LC + r0);
      const float2 qq = *reinterpret_cast<const float2*>(sDA + t * LC + r0);
      const float p0 = pp.x, p1 = pp.y, q0 = bt * qq.x, q1 = bt * qq.y;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        dkc[0][u] = fmaf(p0, xq[u], fmaf(q0, x[u], dkc[0][u]));
        dkc[1][u] = fmaf(p1, xq[u], fmaf(q1, x[u], dkc[1][u]));
      }
    }
#pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
      const int t = r0 + ii;
      const float bt = sB[t];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float gt = sG[t * LC + jc + u], gcu = sG[(C - 1) * LC + jc + u];
        const float ep = __expf(gt - gcu), em = __expf(gcu - gt);
        dqp[ii][u] *= ep;
        dkr[ii][u] *= bt * ep;
        dkc[ii][u] *= em;
      }
    }
  }
  for (int bi = 0; chunk_wide && bi * 16 < n; ++bi) {
    const int b0 = bi * 16, r = min(b0 + 15, n - 1);
    bool wide = false;
    if (tid < HC) {
      const float gr = sG[r * LC + tid];
      for (int t = b0; t < C; ++t) wide |= sG[t * LC + tid] - gr > SPAN_MAX;
      for (int s = b0; s <= r; ++s) wide |= gr - sG[s * LC + tid] > SPAN_MAX;
    }
    wide = __syncthreads_or(wide);
    if (!wide) {
      for (int e = tid; e < (C - b0) * HC; e += NTA) {
        const int t = b0 + e / HC, j = e % HC;
        sEp[t * LC + j] = __expf(sG[t * LC + j] - sG[r * LC + j]);
      }
      for (int e = tid; e < 16 * HC; e += NTA) {
        const int s = e / HC, j = e % HC;
        const float em = __expf(sG[r * LC + j] - sG[(b0 + s) * LC + j]);
        sEm[s * LC + j] = em;
        sKm[s * LC + j] = sK[(b0 + s) * LC + j] * em;
      }
      __syncthreads();
#pragma unroll
      for (int ii = 0; ii < 2; ++ii) {
        const int t = ty + 32 * ii;
        if (t >= b0) {  // rows t: sum over s in the block (dP, dA masked below the diagonal already)
          float r1[4] = {}, r2[4] = {};
          for (int s = 0; s < 16; ++s) {
            const float p = sDP[t * LC + b0 + s], q = sDA[t * LC + b0 + s];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const float km = sKm[s * LC + tx + 16 * m];
              r1[m] = fmaf(p, km, r1[m]);
              r2[m] = fmaf(q, km, r2[m]);
            }
          }
          const float bt = sB[t];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float ep = sEp[t * LC + tx + 16 * m];
            dqp[ii][m] = fmaf(r1[m], ep, dqp[ii][m]);
            dkr[ii][m] = fmaf(bt * r2[m], ep, dkr[ii][m]);
          }
        }
      }
      {  // rows s of this block: sums over t >= b0
        const int s = b0 + orow;
        float r3[2] = {};
        for (int t = b0; t < C; ++t) {
          const float p = sDP[t * LC + s], q = sB[t] * sDA[t * LC + s];
#pragma unroll
          for (int mm = 0; mm < 2; ++mm) {
            const int j = ocol + 32 * mm;
            const float ep = sEp[t * LC + j];
            r3[mm] = fmaf(p, sQ[t * LC + j] * ep, fmaf(q, sK[t * LC + j] * ep, r3[mm]));
          }
        }
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) sDKC[s * LC + ocol + 32 * mm] = r3[mm] * sEm[orow * LC + ocol + 32 * mm];
      }
      __syncthreads();
    } else {  // pair decays one by one
#pragma unroll
      for (int ii = 0; ii < 2; ++ii) {
        const int t = ty + 32 * ii;
        if (t >= b0) {
          const float bt = sB[t];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int j = tx + 16 * m;
            float r1 = 0.f, r2 = 0.f;
            for (int s = b0; s < b0 + 16 && s <= t; ++s) {
              const float e = __expf(sG[t * LC + j] - sG[s * LC + j]) * sK[s * LC + j];
              r1 = fmaf(sDP[t * LC + s], e, r1);
              r2 = fmaf(sDA[t * LC + s], e, r2);
            }
            dqp[ii][m] += r1;
            dkr[ii][m] = fmaf(bt, r2, dkr[ii][m]);
          }
        }
      }
      const int s = b0 + orow;
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        const int j = ocol + 32 * mm;
        float r3 = 0.f;
        for (int t = s; t < C; ++t) {
          const float e = __expf(sG[t * LC + j] - sG[s * LC + j]);
          r3 = fmaf(sDP[t * LC + s], sQ[t * LC + j] * e, fmaf(sB[t] * sDA[t * LC + s], sK[t * LC + j] * e, r3));
        }
        sDKC[s * LC + j] = r3;
      }
      __syncthreads();
    }
  }
  // final values of the own elements; dG and the G_C terms go to shared memory for the reverse cumsum
  float* sDG = sEp;
  float* sXC = sDP;
  cp_async_wait<0>();  // the records' dQ+, dK+, dK^
  __syncthreads();
  if (!chunk_wide) {  // own channels 4 tx .. 4 tx + 3: every operand by 16-byte loads, dq and dk by 16-byte stores
    const int jc = 4 * tx;
#pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
      const int t = own_row(ii);
      float dGv[4] = {0.f, 0.f, 0.f, 0.f}, xcv[4] = {0.f, 0.f, 0.f, 0.f};
      if (t < n) {
        auto ld = [&](const float* base) {
          const float4 v = *reinterpret_cast<const float4*>(base + t * LC + jc);
          return v;
        };
        const float4 g4 = ld(sG), k4 = ld(sK), q4 = ld(sQ), gq4 = ld(sGQ), gk4 = ld(sGK), gh4 = ld(sGH);
        const float4 c4 = *reinterpret_cast<const float4*>(sG + (n - 1) * LC + jc);
        const float Gv[4] = {g4.x, g4.y, g4.z, g4.w}, Cv[4] = {c4.x, c4.y, c4.z, c4.w};
        const float kv[4] = {k4.x, k4.y, k4.z, k4.w}, qv[4] = {q4.x, q4.y, q4.z, q4.w};
        const float gqv[4] = {gq4.x, gq4.y, gq4.z, gq4.w}, gkv[4] = {gk4.x, gk4.y, gk4.z, gk4.w};
        const float ghv[4] = {gh4.x, gh4.y, gh4.z, gh4.w};
        const float dpt = sDiag[t];
        float dqo[4], dko[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float e0 = __expf(Gv[u]), ec = __expf(Cv[u] - Gv[u]);
          const float kk = kv[u], qq = qv[u], gq = gqv[u], gk = gkv[u], gh = ghv[u], dkcv = dkc[ii][u];
          dqo[u] = fmaf(dpt, kk, fmaf(gq, e0, dqp[ii][u]));
          dko[u] = fmaf(dpt, qq, fmaf(gk, e0, fmaf(gh, ec, dkr[ii][u] + dkcv)));
          xcv[u] = gh * kk * ec;
          dGv[u] = (gq * qq + gk * kk) * e0 + qq * dqp[ii][u] + kk * (dkr[ii][u] - dkcv);
        }
        const int64_t o = ((int64_t)(t0 + t) * a.H + h) * D + j0 + jc;
        *reinterpret_cast<float4*>(a.dq + o) = make_float4(dqo[0], dqo[1], dqo[2], dqo[3]);
        *reinterpret_cast<float4*>(a.dk + o) = make_float4(dko[0], dko[1], dko[2], dko[3]);
      }
      *reinterpret_cast<float4*>(sDG + t * LC + jc) = make_float4(dGv[0], dGv[1], dGv[2], dGv[3]);
      *reinterpret_cast<float4*>(sXC + t * LC + jc) = make_float4(xcv[0], xcv[1], xcv[2], xcv[3]);
    }
  }
#pragma unroll
  for (int ii = 0; chunk_wide && ii < 2; ++ii) {
    const int t = own_row(ii);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int jl = own_col(m), j = j0 + jl;
      float dG = 0.f, xc = 0.f;
      if (t < n) {
        const float dkcv = chunk_wide ? sDKC[t * LC + jl] : dkc[ii][m];
        const float G = sG[t * LC + jl], GC = sG[(n - 1) * LC + jl];
        const float e0 = __expf(G), ec = __expf(GC - G);
        const float kk = sK[t * LC + jl], qq = sQ[t * LC + jl];
        const float gq = sGQ[t * LC + jl], gk = sGK[t * LC + jl], gh = sGH[t * LC + jl];
        const int64_t o = ((int64_t)(t0 + t) * a.H + h) * D + j;
        const float dpt = sDiag[t];
        a.dq[o] = fmaf(dpt, kk, fmaf(gq, e0, dqp[ii][m]));
        a.dk[o] = fmaf(dpt, qq, fmaf(gk, e0, fmaf(gh, ec, dkr[ii][m] + dkcv)));
        xc = gh * kk * ec;
        dG = (gq * qq + gk * kk) * e0 + qq * dqp[ii][m] + kk * (dkr[ii][m] - dkcv);
      }
      sDG[t * LC + jl] = dG;
      sXC[t * LC + jl] = xc;
    }
  }
  __syncthreads();
  {
    // dg_u = sum_{t >= u} (dG_t - X_t) + dG_C with X_t = dK^_t K^_t and dG_C = sum_t X_t + d(e^G_C) e^G_C;
    // the X terms are summed directly as sum_{t < u} X_t (a prefix, not the total minus a suffix), and
    // sDG holds dG_t without -X_t.  Thread (channel jj, part): tokens 8 part .. 8 part + 7, the parts'
    // totals combined through shared memory (the block scratch is free).
    const int jj = tid & (HC - 1), part = tid / HC, j = j0 + jj, tb = 8 * part;
    float xs = 0.f, ds = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) xs += sXC[(tb + u) * LC + jj];
#pragma unroll
    for (int u = 7; u >= 0; --u) ds += sDG[(tb + u) * LC + jj];
    sKm[part * HC + jj] = xs;
    sEm[part * HC + jj] = ds;
    __syncthreads();
    float pre = 0.f, run = w[BW_DGAM + j] * w[BW_GAM + j];
    for (int pp = 0; pp < part; ++pp) pre += sKm[pp * HC + jj];
    for (int pp = NTA / HC - 1; pp > part; --pp) run += sEm[pp * HC + jj];
    float px[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      px[u] = pre;
      pre += sXC[(tb + u) * LC + jj];
    }
#pragma unroll
    for (int u = 7; u >= 0; --u) {
      const int t = tb + u;
      run += sDG[t * LC + jj];
      if (t < n) a.dg[((int64_t)(t0 + t) * a.H + h) * D + j] = run + px[u];
    }
  }
  if (half == 0) {  // dbeta_t = (W, U~ part) + sum_s dA_ts a_ts: thread (row t, eight columns), lanes summed
    const int t = tid >> 3, part = tid & 7;
    float s = 0.f;
#pragma unroll
    for (int u = 8 * part; u < 8 * part + 8; ++u)
      if (u < t) s = fmaf(sDA[t * LC + u], w[BW_A + t * C + u], s);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (part == 0 && t < n) a.dbeta[(int64_t)(t0 + t) * a.H + h] = w[BW_DBETA + t] + s;
  }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// The tensor-core passes' layout after the per-chunk records: operand records, fragments and entry states
// (used by the forward pass, then by the reverse one), and the steep flags.
struct FwdLayout {
  int P;
  size_t rec_off, frag_off, entry_off, steep_off, total;
};
// segments per (sequence, head) of the tensor-core passes: the per-segment passes run H P CTAs, one per SM of
// a 152-SM GPU (the fragment phases two waves); a constant, so that the workspace size depends on the
// problem alone
int fwd_segments_target(int H) { return H >= 152 ? 1 : 152 / H; }
FwdLayout fwd_layout(int64_t T, int N, int H) {
  FwdLayout L{};
  L.P = fwd_segments_target(H);
  const size_t heads = (size_t)N * L.P * H;
  L.rec_off = ((size_t)((T + C - 1) / C + N) * H * BW_FLOATS * sizeof(float) + 1023) & ~(size_t)1023;
  L.frag_off = L.rec_off + ((tc_record_bytes(T, N, H) + 1023) & ~(size_t)1023);
  L.entry_off = L.frag_off + heads * D * 2 * D * sizeof(float);
  L.steep_off = L.entry_off + heads * D * D * sizeof(float);
  L.total = L.steep_off + (((size_t)N * H * sizeof(int32_t) + 255) & ~(size_t)255);
  return L;
}

// The forward and reverse passes on the tensor cores (bf16 inputs): operand records -> fragments -> scan ->
// every chunk's entry state and U; then over the same records the state gradient's per-segment maps ->
// their scan from dL/dS_T -> every chunk's dS' and dU, and dL/dS_0.
cudaError_t chain_passes_tc(const BackwardArgs& a, cudaStream_t s) {
  const FwdLayout L = fwd_layout(a.T, a.N, a.H);
  const int pt = L.P;
  int seg = (int)((((int64_t)a.max_seqlen + pt - 1) / pt + C - 1) / C * C);
  if (seg < C) seg = C;
  PrefillArgs p{};
  p.q = a.q, p.k = a.k, p.v = a.v, p.g = a.g, p.beta = a.beta;
  p.in_bf16 = true, p.out_bf16 = false;
  p.T = a.T, p.H = a.H, p.d = D, p.N = a.N, p.cu = a.cu, p.max_seqlen = a.max_seqlen;
  p.pool = const_cast<float*>(a.pool), p.num_slots = a.num_slots, p.slot_ids = a.slot_ids;
  p.init_zero = a.init_zero;
  p.status = a.status;
  p.seg_len = seg;
  p.P = (int)(((int64_t)a.max_seqlen + seg - 1) / seg);
  if (p.P < 1) p.P = 1;
  uint8_t* base = reinterpret_cast<uint8_t*>(a.ws);
  p.records = base + L.rec_off;
  p.frag = reinterpret_cast<float*>(base + L.frag_off);
  p.entry = reinterpret_cast<float*>(base + L.entry_off);
  p.bw_ws = a.ws, p.bw_rec_floats = (int)BW_FLOATS, p.bw_off_h = (int)BW_H, p.bw_off_u = (int)BW_U;
  p.no_work_count = true;
  p.zero_bad_slot = true;  // this call's contract: a bad slot is flagged and differentiated from zero
  cudaError_t e = launch_tc_prep(p, p.records, s);
  if (e == cudaSuccess) e = launch_tc_chain_frag(p, p.records, s);
  if (e == cudaSuccess) e = launch_seg_scan(p, s);
  if (e == cudaSuccess) e = launch_tc_chain_states(p, p.records, s);
  p.d_out = a.d_out, p.d_final = a.d_final, p.d_init = a.d_init;
  p.bw_off_ds = (int)BW_DS, p.bw_off_du = (int)BW_DU;
  p.scan_init = a.d_final;  // the reverse scan starts from dL/dS_T (zero when not given)
  p.init_zero = a.d_final == nullptr;
  if (e == cudaSuccess) e = launch_tc_rev_frag(p, p.records, s);
  if (e == cudaSuccess) e = launch_seg_scan(p, s);
  if (e == cudaSuccess) e = launch_tc_rev_pass(p, p.records, s);
  return e;
}

template <typename Tin>
cudaError_t launch_backward_t(const BackwardArgs& a_in, cudaStream_t s) {
  cudaError_t e;
  BackwardArgs a = a_in;
  a.steep = nullptr;
  if (a.in_bf16) {  // the tensor-core forward pass, with the CUDA-core chain for steep (sequence, head)s
    a.steep = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(a.ws) + fwd_layout(a.T, a.N, a.H).steep_off);
    if ((e = cudaMemsetAsync(a.steep, 0, (size_t)a.N * a.H * sizeof(int32_t), s)) != cudaSuccess) return e;
  }
  if ((e = set_smem(bwd_prep_kernel<Tin>, PREP_SMEM)) != cudaSuccess) return e;
  if ((e = set_smem(bwd_fwd_chain_kernel, FWD_SMEM)) != cudaSuccess) return e;
  if ((e = set_smem(bwd_rev_chain_kernel<Tin>, REV_SMEM)) != cudaSuccess) return e;
  if ((e = set_smem(bwd_state_grads_tc_kernel<Tin>, STATE_TC_SMEM)) != cudaSuccess) return e;
  if ((e = set_smem(bwd_wy_grads_kernel<Tin>, WY_SMEM)) != cudaSuccess) return e;
  if ((e = set_smem(bwd_assemble_kernel<Tin>, ASM_SMEM)) != cudaSuccess) return e;
  const int nch = (a.max_seqlen + C - 1) / C;
  const dim3 chunks(nch, a.H, a.N), halves(nch, 2 * a.H, a.N), chains(D / CB, a.H, a.N);
  if (nch > 0) {
    bwd_prep_kernel<Tin><<<chunks, NT, PREP_SMEM, s>>>(a);
    if (a.in_bf16) {
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      if ((e = chain_passes_tc(a, s)) != cudaSuccess) return e;
    }
    bwd_fwd_chain_kernel<<<chains, NTC, FWD_SMEM, s>>>(a);  // (bf16: only the steep (sequence, head)s)
  }
  bwd_rev_chain_kernel<Tin><<<chains, NTC, REV_SMEM, s>>>(a);  // (bf16: only the steep (sequence, head)s)
  if (nch > 0) {
    bwd_state_grads_tc_kernel<Tin><<<chunks, NT, STATE_TC_SMEM, s>>>(a);
    bwd_wy_grads_kernel<Tin><<<chunks, NT, WY_SMEM, s>>>(a);
    bwd_assemble_kernel<Tin><<<halves, NTA, ASM_SMEM, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

size_t backward_ws_bytes(int64_t T, int N, int H) {
  // the per-chunk records, then (the bf16 inputs' tensor-core forward pass) operand records, fragments and
  // entry states
  return fwd_layout(T, N, H).total;
}

cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  return a.in_bf16 ? launch_backward_t<bf16>(a, s) : launch_backward_t<float>(a, s);
}

}  // namespace kda
