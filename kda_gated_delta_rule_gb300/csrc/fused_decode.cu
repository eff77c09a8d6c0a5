// Fused decode front/back-end: the short causal convolution, the KDA step and the gated output norm of one
// decode token in a single launch (d = 128), one (request, head) unit at a time per CTA.
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
#include "device.h"
#include "launch.h"
#include "tc_ptx.cuh"
#include "wstep.cuh"

namespace kda {
namespace {

constexpr int FD = 128;                 // dk = dv
constexpr int FW = 4;                   // convolution taps
constexpr int FNT = WCfg<FD>::NT;       // 256 threads: 8 warps of 16 value columns
constexpr float F_GMIN = -5.f;
constexpr float F_L2EPS = 1e-6f;

__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + __expf(-x)); }

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// One unit's front-end operands as staged in shared memory: the convolution taps of its head, the token's
// three projections, decay logits, output-gate logits and write-strength logit.
template <typename Tin>
struct __align__(16) FrontBuf {
  float w[3][FD][FW];
  alignas(16) Tin x[3][FD];
  alignas(16) float a[FD];
  alignas(16) Tin z[FD];
  float b;
};

constexpr uint32_t F_STATE_BYTES = FD * FD * 4;
constexpr uint32_t F_CONV_BYTES = 3 * (FW - 1) * FD * 4;  // one (slot, head)'s carried inputs

template <typename Tin>
struct FusedStreamSmem {
  static constexpr size_t STAGE = 0;
  static constexpr size_t CONV = STAGE + F_STATE_BYTES;  // [2] carried inputs, bulk-copied with the state
  static constexpr size_t FRONT = CONV + 2 * F_CONV_BYTES;
  static constexpr size_t TOK = FRONT + 2 * sizeof(FrontBuf<Tin>);
  static constexpr size_t RED = TOK + sizeof(WTok<FD>);
  static constexpr size_t BAR = RED + 3 * (FNT / 32) * 4;
  static constexpr size_t BYTES = BAR + 16;
  static_assert(CONV % 16 == 0 && FRONT % 16 == 0 && TOK % 16 == 0 && BAR % 8 == 0, "shared layout");
};

// Two persistent CTAs per SM walk the (request, head) units with stride gridDim.x.  The next unit's state
// and carried inputs arrive by bulk copy (one mbarrier) and its front-end operands by cp.async while the
// current unit runs the convolution, the step, the state store and the norm, so every SM keeps its next
// state load in flight.  The step is the decode kernel's wstep.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(FNT, 2) fused_decode_stream_kernel(FusedDecodeArgs a, int units) {
  using L = FusedStreamSmem<Tin>;
  extern __shared__ __align__(128) uint8_t smem[];
  const float* stage = reinterpret_cast<const float*>(smem + L::STAGE);
  float* conv = reinterpret_cast<float*>(smem + L::CONV);
  FrontBuf<Tin>* front = reinterpret_cast<FrontBuf<Tin>*>(smem + L::FRONT);
  WTok<FD>& tok = *reinterpret_cast<WTok<FD>*>(smem + L::TOK);
  float(*red)[FNT / 32] = reinterpret_cast<float(*)[FNT / 32]>(smem + L::RED);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H;
  const int c = tid & (FD - 1);
  const int s0 = tid < FD ? 0 : 2, ns = tid < FD ? 2 : 1;  // threads 0-127: streams q, k; 128-255: v
  const int col = wstep_out_col(warp, lane);
  const float nw = a.norm_w[col];
  auto next_unit = [&](int u) {
    for (; u < units; u += (int)gridDim.x) {
      const int slot = a.slot_ids[u / H];
      if (slot >= 0 && slot < a.num_slots) break;
      if (tid == 0) flag_status(a.status, KDA_DEV_SLOT_OOB);
    }
    return u;
  };
  // requests unit u's state and carried inputs (thread 0, bulk) and its front-end operands into buffer buf
  auto prefetch = [&](int u, int buf) {
    const int h = u % H;
    const size_t sh = (size_t)a.slot_ids[u / H] * H + h;
    if (tid == 0) {
      tc::bar_arrive_expect_tx(bar, F_STATE_BYTES + F_CONV_BYTES);
      tc::bulk_g2s(smem + L::STAGE, a.pool + sh * FD * FD, F_STATE_BYTES, bar);
      tc::bulk_g2s(conv + buf * (F_CONV_BYTES / 4), a.conv_state + sh * 3 * (FW - 1) * FD, F_CONV_BYTES, bar);
    }
    FrontBuf<Tin>& f = front[buf];
    constexpr int CX = FD * (int)sizeof(Tin) / 16;  // 16-byte chunks of a projection row
    constexpr int NW = 3 * FD, NX = 3 * CX, NA = FD * 4 / 16;
    for (int e = tid; e < NW + NX + NA + CX; e += FNT) {
      if (e < NW) {
        const int st = e / FD, ch = e % FD;
        cp_async16(&f.w[st][ch][0], a.conv_w + (((size_t)st * H + h) * FD + ch) * FW);
      } else if (e < NW + NX) {
        const int st = (e - NW) / CX, r = (e - NW) % CX;
        const void* xin = st == 0 ? a.xq : st == 1 ? a.xk : a.xv;
        cp_async16(reinterpret_cast<uint8_t*>(f.x[st]) + 16 * r,
                   static_cast<const uint8_t*>(xin) + (size_t)u * FD * sizeof(Tin) + 16 * r);
      } else if (e < NW + NX + NA) {
        const int r = e - NW - NX;
        cp_async16(reinterpret_cast<uint8_t*>(f.a) + 16 * r,
                   reinterpret_cast<const uint8_t*>(a.a + (size_t)u * FD) + 16 * r);
      } else {
        const int r = e - NW - NX - NA;
        cp_async16(reinterpret_cast<uint8_t*>(f.z) + 16 * r,
                   static_cast<const uint8_t*>(a.z) + (size_t)u * FD * sizeof(Tin) + 16 * r);
      }
    }
    if (tid == FNT - 1) cp_async4(&f.b, a.b + u);
  };
  if (tid == 0) {
    tc::bar_init(bar, 1);
    tc::bar_fence_init();
  }
  __syncthreads();
  int u = next_unit((int)blockIdx.x);
  if (u < units) prefetch(u, 0);
  bool ok = true;
  float2 S[WRows<FD>::P][4];
#pragma unroll 1
  for (int it = 0; u < units; ++it) {
    const int buf = it & 1;
    const bool landed = tc::bar_wait(bar, (uint32_t)it & 1u);
    cp_async_wait_all();
    ok = __syncthreads_and(landed) != 0;
    if (!ok) break;
    const FrontBuf<Tin>& f = front[buf];
    const float* cs = conv + buf * (F_CONV_BYTES / 4);  // [3 streams][W-1 taps][d]
    float4 w[2];
    float xw[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (j < ns) {
        const int s = s0 + j;
        w[j] = *reinterpret_cast<const float4*>(&f.w[s][c][0]);
        const float* st = cs + s * (FW - 1) * FD + c;
        xw[j][0] = st[0], xw[j][1] = st[FD], xw[j][2] = st[2 * FD];
        xw[j][3] = to_f32(f.x[s][c]);
      }
    }
    const float alog = tid < FD ? 0.f : f.a[c];
    const float zg = sigm(to_f32(f.z[col])) * nw;
    const float bl = f.b;
    wload_shared<FD>(S, stage, warp, lane);
    __syncthreads();  // the stage, the carried inputs and the operands of buffer buf have been read
    const int un = next_unit(u + (int)gridDim.x);
    if (un < units) prefetch(un, buf ^ 1);
    const size_t row = (size_t)u;
    const size_t sh = (size_t)a.slot_ids[u / H] * H + u % H;
    float* cst = a.conv_state + sh * 3 * (FW - 1) * FD;
    float y[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (j < ns) {
        float* st = cst + (s0 + j) * (FW - 1) * FD + c;
        st[0] = xw[j][1];
        st[FD] = xw[j][2];
        st[2 * FD] = xw[j][3];
        const float v = fmaf(w[j].w, xw[j][3], fmaf(w[j].z, xw[j][2], fmaf(w[j].y, xw[j][1], w[j].x * xw[j][0])));
        y[j] = v * sigm(v);
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
    if (tid == 0) tok.beta = sigm(bl);
    __syncthreads();
    if (tid < FD) {
      const float nq = (red[0][0] + red[0][1]) + (red[0][2] + red[0][3]);
      const float nk = (red[1][0] + red[1][1]) + (red[1][2] + red[1][3]);
      tok.q[wperm(c, FD)] = qv / sqrtf(nq + F_L2EPS);
      tok.k[wperm(c, FD)] = kv / sqrtf(nk + F_L2EPS);
    }
    __syncthreads();
    const float o = wstep<FD, true>(S, tok, warp, lane);
    wstore<FD>(S, a.pool + sh * FD * FD, warp, lane);
    const bool holder = ((lane >> 2) & 1) == 0;
    float so = holder ? o * o : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) so += __shfl_xor_sync(0xffffffffu, so, off);
    if (lane == 0) red[2][warp] = so;
    __syncthreads();
    if (holder) {
      float tot = 0.f;
#pragma unroll
      for (int w8 = 0; w8 < FNT / 32; ++w8) tot += red[2][w8];
      const float inv = 1.f / sqrtf(tot * (1.f / FD) + a.eps);
      static_cast<Tout*>(a.out)[row * FD + col] = from_f32<Tout>(o * inv * zg);
    }
    if (tid == 0) add_work(a.status, 1);
    u = un;
  }
  if (!ok) {  // the state copy did not land in time: report it and give the copy one more bounded wait
    if (tid == 0) flag_status(a.status, KDA_DEV_TIMEOUT);
    tc::bar_wait(bar, 0u);
    tc::bar_wait(bar, 1u);
  }
}

template <typename Tin, typename Tout>
cudaError_t launch_t(const FusedDecodeArgs& a, cudaStream_t s) {
  using L = FusedStreamSmem<Tin>;
  cudaError_t e = cudaFuncSetAttribute(fused_decode_stream_kernel<Tin, Tout>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
  if (e != cudaSuccess) return e;
  const int units = a.B * a.H, sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = units < 2 * sms ? units : 2 * sms;
  fused_decode_stream_kernel<Tin, Tout><<<grid, FNT, L::BYTES, s>>>(a, units);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused_decode(const FusedDecodeArgs& a, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  if (a.in_bf16) return a.out_bf16 ? launch_t<bf16, bf16>(a, s) : launch_t<bf16, float>(a, s);
  return a.out_bf16 ? launch_t<float, bf16>(a, s) : launch_t<float, float>(a, s);
}

}  // namespace kda
