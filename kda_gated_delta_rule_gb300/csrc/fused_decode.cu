// Fused decode front/back-end: the short causal convolution, the KDA step and the gated output norm of one
// decode token in a single launch (d = 128), one CTA per (request, head).
//
// Source: "SGLang and Miles: day-0 support for Kimi K3", section "kernels" (the fused Conv + KDA + Onorm
// decode kernel; the bs = 1 decode step is launch- and latency-bound, so the module is one launch);
// "Kimi K3: Architecture and SGLang Day-0 Support", KDA math box (the step itself; the log-decay held above
// g_min = -5 by a scaled sigmoid; the output gate a full-rank projection of the input).  The pages give no
// formula for the convolution or the norm; this kernel takes the plain reading: a width-4 depthwise causal
// convolution with SiLU on each of the projected q, k, v (the last three inputs carried per slot), L2
// normalisation of q and k, g = -5 sigmoid(a), beta = sigmoid(b), and an RMS norm over the head's outputs
// with a per-channel weight, times sigmoid of the output-gate projection z.
//
// HBM per (request, head): the 64 KB state read and written once, the 4.5 KB of carried inputs read and
// written once, the token's projections and the output.  Convolution and norm weights are shared by all
// requests (L2-resident).
#include "launch.h"
#include "wstep.cuh"

namespace kda {
namespace {

constexpr int FD = 128;                 // dk = dv
constexpr int FW = 4;                   // convolution taps
constexpr int FNT = WCfg<FD>::NT;       // 256 threads: 8 warps of 16 value columns
constexpr float F_GMIN = -5.f;
constexpr float F_L2EPS = 1e-6f;

__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + __expf(-x)); }

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(FNT, 2) fused_decode_kernel(FusedDecodeArgs a) {
  __shared__ WTok<FD> tok;
  __shared__ float red[3][FNT / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / a.H, h = blockIdx.x % a.H;
  const int slot = a.slot_ids[b];
  if (slot < 0 || slot >= a.num_slots) {
    if (tid == 0) flag_status(a.status, KDA_DEV_SLOT_OOB);
    return;
  }
  float* Sg = a.pool + ((size_t)slot * a.H + h) * FD * FD;
  const size_t row = (size_t)b * a.H + h;
  float* cst = a.conv_state + ((size_t)slot * a.H + h) * 3 * (FW - 1) * FD;  // [3 streams][W-1 taps][d]
  const int c = tid & (FD - 1);
  // the front end's operands are loaded before the state, so they do not queue behind it: threads 0-127
  // take streams q and k of channel c, threads 128-255 stream v and the decay logit
  const int s0 = tid < FD ? 0 : 2, ns = tid < FD ? 2 : 1;
  float4 w[2];
  float xw[2][4];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    if (u < ns) {
      const int s = s0 + u;
      w[u] = *reinterpret_cast<const float4*>(a.conv_w + (((size_t)s * a.H + h) * FD + c) * FW);
      const float* st = cst + s * (FW - 1) * FD + c;
      xw[u][0] = st[0], xw[u][1] = st[FD], xw[u][2] = st[2 * FD];
      const void* xin = s == 0 ? a.xq : s == 1 ? a.xk : a.xv;
      xw[u][3] = to_f32(static_cast<const Tin*>(xin)[row * FD + c]);
    }
  }
  const float alog = tid < FD ? 0.f : a.a[row * FD + c];
  const int col = wstep_out_col(warp, lane);  // the output column this lane holds after the step
  const float zg = sigm(to_f32(static_cast<const Tin*>(a.z)[row * FD + col])) * a.norm_w[col];
  float2 S[WRows<FD>::P][4];
  wload<FD>(S, Sg, warp, lane);
  // window (3 carried inputs, x_t) against the taps, then SiLU; the carried inputs advance by one token
  // (each (stream, channel) belongs to one thread)
  float y[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    if (u < ns) {
      float* st = cst + (s0 + u) * (FW - 1) * FD + c;
      st[0] = xw[u][1];
      st[FD] = xw[u][2];
      st[2 * FD] = xw[u][3];
      const float v = fmaf(w[u].w, xw[u][3], fmaf(w[u].z, xw[u][2], fmaf(w[u].y, xw[u][1], w[u].x * xw[u][0])));
      y[u] = v * sigm(v);
    }
  }
  float qv = 0.f, kv = 0.f;
  if (tid < FD) {
    qv = y[0];
    kv = y[1];
  } else {
    tok.v[c] = y[0];
    tok.a[wperm(c, FD)] = __expf(F_GMIN * sigm(alog));
  }
  float sq = qv * qv, sk = kv * kv;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sq += __shfl_xor_sync(0xffffffffu, sq, o);
    sk += __shfl_xor_sync(0xffffffffu, sk, o);
  }
  if (lane == 0) red[0][warp] = sq, red[1][warp] = sk;
  if (tid == 0) tok.beta = sigm(a.b[row]);
  __syncthreads();
  if (tid < FD) {
    const float nq = (red[0][0] + red[0][1]) + (red[0][2] + red[0][3]);
    const float nk = (red[1][0] + red[1][1]) + (red[1][2] + red[1][3]);
    tok.q[wperm(c, FD)] = qv / sqrtf(nq + F_L2EPS);
    tok.k[wperm(c, FD)] = kv / sqrtf(nk + F_L2EPS);
  }
  __syncthreads();
  const float o = wstep<FD, true>(S, tok, warp, lane);
  wstore<FD>(S, Sg, warp, lane);
  // output norm over the head's 128 columns; a column's value sits in the lanes with bit 2 clear
  const bool holder = ((lane >> 2) & 1) == 0;
  float so = holder ? o * o : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) so += __shfl_xor_sync(0xffffffffu, so, off);
  if (lane == 0) red[2][warp] = so;
  __syncthreads();
  if (holder) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < FNT / 32; ++w) tot += red[2][w];
    const float inv = 1.f / sqrtf(tot * (1.f / FD) + a.eps);
    static_cast<Tout*>(a.out)[row * FD + col] = from_f32<Tout>(o * inv * zg);
  }
  if (tid == 0) add_work(a.status, 1);
}

template <typename Tin, typename Tout>
cudaError_t launch_t(const FusedDecodeArgs& a, cudaStream_t s) {
  fused_decode_kernel<Tin, Tout><<<a.B * a.H, FNT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused_decode(const FusedDecodeArgs& a, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  if (a.in_bf16) return a.out_bf16 ? launch_t<bf16, bf16>(a, s) : launch_t<bf16, float>(a, s);
  return a.out_bf16 ? launch_t<float, bf16>(a, s) : launch_t<float, float>(a, s);
}

}  // namespace kda
