// Speculative verify on the tensor cores: the W-token draft window of one (request, head) as one chunk.
//
// Sources: "SGLang and Miles: day-0 support for Kimi K3", section "ReplaySSM: raw-input replay for KDA
// state" (verify reads the committed checkpoint, never writes it, and stores each step's raw inputs);
// the KDA update of "Kimi K3: Architecture and SGLang Day-0 Support", KDA math box, unrolled over the
// window.  With the in-window cumulative log-decay G_t = g_1 + ... + g_t (per key channel),
//   A_ts = beta_t sum_j k_t[j] k_s[j] exp(G_t[j] - G_s[j])   (s < t),
//   P_ts =        sum_j q_t[j] k_s[j] exp(G_t[j] - G_s[j])   (s <= t),
// the window's deltas solve (I + A) U = diag(beta) (V - (K o e^G) S0) and the outputs are
// O = (Q o e^G) S0 + P U.  Substituting U, with R = P (I + A)^-1 diag(beta):
//   O = Qh S0 + Oh,   Qh = Q o e^G - R (K o e^G),   Oh = R V.
// So verify is one product of the committed state with the W rows of Qh plus small fp32 work on the
// window, instead of W dependent rank-1 passes over the state.  The product runs on the tensor cores:
// S0^T is the A operand in tensor memory (lane c = value column c, K = key channel), split into bf16
// hi + lo; the B operand in shared memory stacks the bf16 hi parts of Qh's rows over their lo parts, so
// two products (S0 hi and S0 lo against the stacked rows) give all four hi/lo terms in fp32, summed per
// token in the epilogue.
//
// Decay factors: while every |G_t| <= 80 the pair factor exp(G_t - G_s) is the product of the per-token
// factors exp(G_t) and exp(-G_s), both finite in fp32, so the Gram entries are plain dot products of
// K o e^G (or Q o e^G) with K o e^-G.  A window whose decay leaves that range forms every pair factor as
// exp(G_t - G_s) directly, which never exceeds 1 for s <= t.
//
// Schedule: one persistent CTA per SM walks (request, head) items.  Warps 0-7 ("math") receive each
// window's raw inputs one item ahead (TMA tensor-map loads of k, q, v, g; cp.async for beta), write the
// raw-input record straight from those buffers (TMA tensor-map stores, issued as soon as they land) and
// compute Qh (into a double-buffered B tile) and Oh.  Warps 8-15 ("state") receive each committed state by a 64 KB bulk copy into a
// shared-memory ring (two items ahead when the window fits 8 tokens), split it into tensor memory, and one
// thread issues the product into one of two accumulators; the output epilogue of item n runs after the
// split of item n + 1.  The groups hand over through mbarriers with bounded waits.
#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"
#include "device.h"
#include "tmap.h"

namespace kda {
namespace {

constexpr int D = 128;
constexpr int MT = 256;  // math threads, warps 0-7
constexpr int ST = 256;  // state threads, warps 8-15
constexpr int NT = MT + ST;
constexpr int BAR_MATH = 1, BAR_STATE = 2, BAR_TEAM = 3;  // named barriers (BAR_TEAM + team: two-team math)
constexpr float G_SPAN = 80.f;              // |G| bound of the factored decay path
constexpr uint32_t STATE_BYTES = D * D * 4;

// tensor memory: two buffers of [S0^T hi (64 columns of bf16 pairs) | lo | two accumulators of 2*WP fp32
// columns: S0 hi and S0 lo against the stacked Qh rows, issued by two threads]
constexpr uint32_t TMEM_COLS = 512, BUF_COLS = 256, COL_AHI = 0, COL_ALO = 64, COL_ACC = 128, COL_ACC2 = 192;

template <int WP>
struct Raw {  // one window's raw inputs (cp.async targets); rows at or past W are stale
  alignas(16) bf16 k[WP][D];
  alignas(16) bf16 q[WP][D];
  alignas(16) bf16 v[WP][D];
  alignas(16) float g[WP][D];
  alignas(16) float beta[WP];  // zeroed past W before use
};

template <int WP>
struct Work {
  alignas(16) float G[WP][D];   // cumulative log-decay
  alignas(16) float Kp[WP][D];  // K o e^G   (zero past W)
  alignas(16) float Qp[WP][D];  // Q o e^G   (zero past W)
  alignas(16) float Y[WP][D];   // K o e^-G  (zero past W)
  alignas(16) float A[WP][WP];  // beta_t (k_t . k_s e^{G_t - G_s}), s < t
  alignas(16) float P[WP][WP];  // q_t . k_s e^{G_t - G_s}, s <= t
};

struct VMaps {  // [B*W][H][128] token rows, box = one head x W rows: inputs, then the record's k, v, g
  CUtensorMap q, k, v, g, rk, rv, rg;
};

template <int WP>
struct PLayout {
  static constexpr int STAGES = WP <= 8 ? 2 : 1;  // committed states in flight
  // W <= 8: two math teams of four warps take alternate items (each with two raw-input buffers and its own
  // work area); W > 8: one team of eight warps (shared memory holds no second set)
  static constexpr int TEAMS = WP <= 8 ? 2 : 1;
  // B operand: rows 0..WP-1 = bf16 hi of Qh, rows WP..2WP-1 = bf16 lo, x 128 key channels: two 64-channel
  // K-blocks, 8-row groups 1024 bytes apart
  static constexpr uint32_t B_ROWS = 2 * WP, B_BLOCK = B_ROWS * 128, B_TILE = 2 * B_BLOCK;
  static constexpr uint32_t BT = STAGES * STATE_BYTES;
  static constexpr uint32_t OH = BT + 2 * B_TILE;
  // Oh buffers: four with two math teams (item n uses n % 4, so a team's item waits for the epilogue of
  // the item four back, not two back, which the state warps reach one item late), two with one team
  static constexpr int OHB = TEAMS == 2 ? 4 : 2;
  static constexpr uint32_t RAW_BYTES = (uint32_t)((sizeof(Raw<WP>) + 127) / 128 * 128);
  static constexpr uint32_t RAW = OH + OHB * WP * D * 4;
  static constexpr uint32_t WORK = RAW + 2 * TEAMS * RAW_BYTES;
  static constexpr uint32_t WORK_BYTES = (uint32_t)((sizeof(Work<WP>) + 127) / 128 * 128);
  static constexpr uint32_t BARS = WORK + TEAMS * WORK_BYTES;
  static constexpr uint32_t BYTES = BARS + 128 + 1024;  // + slack for the 1024-byte alignment
  static_assert(BYTES <= 232448, "shared memory");
  static_assert(sizeof(Raw<WP>::k) % 16 == 0, "TMA destinations stay 16-byte aligned");
};

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}

// Butterfly reduce-scatter over the warp: on entry every lane holds partial sums x[0..N) of N values; on
// exit x[0 .. max(N/32, 1)) hold the full sums of values base, base + 1, ... (lanes that differ only in the
// bits of the trailing all-reduce stages hold the same values).
template <int N, int M>
__device__ __forceinline__ void reduce_scatter(float (&x)[N], int lane, int& base) {
  if constexpr (M > 0) {
    if constexpr (N >= 2) {
      constexpr int HN = N / 2;
      const bool up = (lane & M) != 0;
      float y[HN];
#pragma unroll
      for (int i = 0; i < HN; ++i) {
        const float keep = up ? x[HN + i] : x[i], send = up ? x[i] : x[HN + i];
        y[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
      }
      if (up) base += HN;
      reduce_scatter<HN, M / 2>(y, lane, base);
#pragma unroll
      for (int i = 0; i < HN; ++i) x[i] = y[i];
    } else {
      x[0] += __shfl_xor_sync(0xffffffffu, x[0], M);
      reduce_scatter<N, M / 2>(x, lane, base);
    }
  }
}

// Row t of A and P, computed by one warp: lane l covers channels 4l .. 4l+3.
template <int WP, bool FACTORED>
__device__ __forceinline__ void gram_row(const Raw<WP>& r, Work<WP>& w, int t, int W, int lane) {
  float x[2 * WP];
  const int j = 4 * lane;
  if (FACTORED) {
    const float4 kt = *reinterpret_cast<const float4*>(&w.Kp[t][j]);
    const float4 qt = *reinterpret_cast<const float4*>(&w.Qp[t][j]);
#pragma unroll
    for (int u = 0; u < WP; ++u) {
      const float4 y = *reinterpret_cast<const float4*>(&w.Y[u][j]);
      x[u] = fmaf(kt.x, y.x, fmaf(kt.y, y.y, fmaf(kt.z, y.z, kt.w * y.w)));
      x[WP + u] = fmaf(qt.x, y.x, fmaf(qt.y, y.y, fmaf(qt.z, y.z, qt.w * y.w)));
    }
  } else {
    // pairwise factors; rows past the window stay zero
    const bool row_in = t < W;
    const float4 gt = *reinterpret_cast<const float4*>(&w.G[t][j]);
    float kt[4], qt[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      kt[i] = row_in ? __bfloat162float(r.k[t][j + i]) : 0.f;
      qt[i] = row_in ? __bfloat162float(r.q[t][j + i]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < WP; ++u) {
      float a = 0.f, p = 0.f;
      if (row_in && u <= t) {
        const float4 gu = *reinterpret_cast<const float4*>(&w.G[u][j]);
        const float e[4] = {__expf(gt.x - gu.x), __expf(gt.y - gu.y), __expf(gt.z - gu.z), __expf(gt.w - gu.w)};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float ks = __bfloat162float(r.k[u][j + i]) * e[i];
          a = fmaf(kt[i], ks, a);
          p = fmaf(qt[i], ks, p);
        }
      }
      x[u] = a;
      x[WP + u] = p;
    }
  }
  int base = 0;
  reduce_scatter<2 * WP, 16>(x, lane, base);
  constexpr int PER = 2 * WP >= 32 ? 2 * WP / 32 : 1;
  constexpr int DUP = 2 * WP >= 32 ? 1 : 32 / (2 * WP);  // lanes holding the same values
  if ((lane & (DUP - 1)) == 0) {
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int idx = base + i;
      if (idx < WP) w.A[t][idx] = idx < t ? r.beta[t] * x[i] : 0.f;
      else w.P[t][idx - WP] = idx - WP <= t ? x[i] : 0.f;
    }
  }
}

// Item i = (request b, head h).  Its slot id is loaded by the callers one iteration ahead of use, so the
// dependent load never sits on a hand-off.
struct Item {
  int b, h;
  size_t row0;  // row of window token t: row0 + t * H
};

__device__ __forceinline__ Item item_at(int i, int W, int H) {
  Item it;
  it.b = i / H;
  it.h = i % H;
  it.row0 = (size_t)it.b * W * H + it.h;
  return it;
}

template <int WP, typename Tout>
__global__ void __launch_bounds__(NT, 1) verify_tc_kernel(const __grid_constant__ VMaps maps,
                                                          const float* __restrict__ beta, int B, int W, int H,
                                                          const float* __restrict__ pool, int num_slots,
                                                          const int32_t* __restrict__ slot_ids, Tout* __restrict__ out,
                                                          ReplayPtrs rec, int32_t* status) {
  using L = PLayout<WP>;
  constexpr int STAGES = L::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Work<WP>& wk = *reinterpret_cast<Work<WP>*>(sm + L::WORK);
  uint64_t* full_s = reinterpret_cast<uint64_t*>(sm + L::BARS);  // state copy landed      [2]
  uint64_t* full_w = full_s + 2;                                  // Qh / Oh written         [2]
  uint64_t* empty_w = full_s + 4;                                 // Oh consumed             [4]
  uint64_t* mma_bar = full_s + 8;                                 // product complete        [2]
  uint64_t* full_r = full_s + 10;                                 // raw inputs landed       [2 * TEAMS]
  constexpr int OHM = L::OHB - 1;                                 // Oh buffer of item n: n & OHM
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BARS + 112);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int items = B * H;
  const int cnt = (int)blockIdx.x < items ? (items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  auto item_index = [&](int n) { return (int)blockIdx.x + n * (int)gridDim.x; };
  auto raw_of = [&](int n) -> Raw<WP>& { return *reinterpret_cast<Raw<WP>*>(sm + L::RAW + (n & 1) * L::RAW_BYTES); };

  // setup: barriers, tensor memory, beta past the window
  constexpr int TEAMS = L::TEAMS;
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) tc::bar_init(&empty_w[i], ST);
    for (int i = 0; i < 2; ++i) {
      tc::bar_init(&full_s[i], 1);
      tc::bar_init(&full_w[i], MT / TEAMS);  // every thread of the team that computed the item
      tc::bar_init(&mma_bar[i], 4);  // one commit per issuing thread
    }
    for (int i = 0; i < 2 * TEAMS; ++i) tc::bar_init(&full_r[i], 1 + W);  // TMA issuer + a cp.async per beta
    tc::bar_fence_init();
  }
  if (warp == 8) tc::tmem_alloc(tslot, TMEM_COLS);
  if (tid < 2 * TEAMS * WP && (tid % WP) >= W)
    reinterpret_cast<Raw<WP>*>(sm + L::RAW + (tid / WP) * L::RAW_BYTES)->beta[tid % WP] = 0.f;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = *tslot;

  if (TEAMS == 2 && warp < 8) {
    // ------------------------------------------------------------------ math warps, two teams
    // team t (warps 4t .. 4t+3) takes items n = t, t + 2, ...; its m-th item uses raw buffer 2t + m%2 and
    // full_r barrier 2t + m%2 (parity (m/2)%2), its work area, and the B tile / Oh buffer n%2 = t
    const int team = warp >> 2, ttid = tid & 127, tw = warp & 3, c = ttid;
    const int bar_team = BAR_TEAM + team;
    Work<WP>& wt = *reinterpret_cast<Work<WP>*>(sm + L::WORK + team * L::WORK_BYTES);
    auto raw_t = [&](int m) -> Raw<WP>& {
      return *reinterpret_cast<Raw<WP>*>(sm + L::RAW + (2 * team + (m & 1)) * L::RAW_BYTES);
    };
    auto fetch = [&](int m) {  // the team's m-th item
      const Item it = item_at(item_index(2 * m + team), W, H);
      Raw<WP>& r = raw_t(m);
      uint64_t* fb = &full_r[2 * team + (m & 1)];
      if (ttid == 0) {
        tc::bulk_wait_read1();  // the record stores of the team's item m-2 have read this buffer
        tc::bar_arrive_expect_tx(fb, (uint32_t)W * (3 * D * 2 + D * 4));
        const int y = it.h, z = it.b * W;
        tc::tma_load_3d(r.k, &maps.k, 0, y, z, fb);
        tc::tma_load_3d(r.q, &maps.q, 0, y, z, fb);
        tc::tma_load_3d(r.v, &maps.v, 0, y, z, fb);
        tc::tma_load_3d(r.g, &maps.g, 0, y, z, fb);
      }
      if (ttid >= 32 && ttid < 32 + W) {
        const int t = ttid - 32;
        cp_async4(&r.beta[t], beta + it.row0 + (size_t)t * H);
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(fb)) : "memory");
      }
    };
    if (team < cnt) fetch(0);
    for (int m = 0; 2 * m + team < cnt; ++m) {
      const int n = 2 * m + team;
      const Item it = item_at(item_index(n), W, H);
      const int slot = slot_ids[item_index(n) / H];
      const bool ok = slot >= 0 && slot < num_slots;
      Raw<WP>& r = raw_t(m);
      if (!tc::bar_wait(&full_r[2 * team + (m & 1)], (m >> 1) & 1) && ttid == 0) flag_status(status, KDA_DEV_TIMEOUT);
      if (ttid == 0) {  // the raw-input record: the exact stored bits the fold consumes
        if (ok) {
          tc::tma_store_3d(&maps.rk, 0, it.h, it.b * W, r.k);
          tc::tma_store_3d(&maps.rv, 0, it.h, it.b * W, r.v);
          tc::tma_store_3d(&maps.rg, 0, it.h, it.b * W, r.g);
        }
        tc::bulk_commit();  // one group per item (empty when skipped)
      }
      tc::named_bar(bar_team, 128);  // the team is done with its previous item (and its buffers)
      if (n + 2 < cnt) fetch(m + 1);
      if (!ok && ttid == 0) flag_status(status, KDA_DEV_SLOT_OOB);

      // 1. per channel c: G, K o e^G, Q o e^G, Y = K o e^-G; is the factored path valid?
      bool out_of_span = false;
      {
        float gv[WP], kv[WP], qv[WP];
#pragma unroll
        for (int t = 0; t < WP; ++t) {
          const bool in = t < W;
          gv[t] = in ? r.g[t][c] : 0.f;
          kv[t] = in ? __bfloat162float(r.k[t][c]) : 0.f;
          qv[t] = in ? __bfloat162float(r.q[t][c]) : 0.f;
        }
        float run = 0.f;
#pragma unroll
        for (int t = 0; t < WP; ++t) {
          run = __fadd_rn(run, gv[t]);
          gv[t] = run;
        }
#pragma unroll
        for (int t = 0; t < WP; ++t) {
          const float ep = __expf(gv[t]);
          wt.Kp[t][c] = kv[t] * ep;
          wt.Qp[t][c] = qv[t] * ep;
          wt.G[t][c] = gv[t];
          wt.Y[t][c] = kv[t] * __expf(-gv[t]);
          out_of_span |= !(fabsf(gv[t]) <= G_SPAN);
        }
      }
      const bool pairwise = tc::named_bar_or(bar_team, 128, out_of_span);

      // 2. A and P, rows tw and 7 - tw per warp of the team
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int t = rr ? 7 - tw : tw;
        if (pairwise) gram_row<WP, false>(r, wt, t, W, lane);
        else gram_row<WP, true>(r, wt, t, W, lane);
      }
      tc::named_bar(bar_team, 128);

      // 3. per channel, both paths: x = (I + A)^-1 diag(beta) y by forward substitution, then P x, for y = K o e^G
      //    (Qh = Q o e^G - P x, into B tile n%2) and y = V (Oh = P x, into its buffer)
      // B tile n % 2 was read by item n-2's product; Oh buffer n % 4 by item n-4's epilogue
      if (n >= 2 && !tc::bar_wait(&mma_bar[n & 1], ((n >> 1) + 1) & 1) && ttid == 0)
        flag_status(status, KDA_DEV_TIMEOUT);
      if (n >= 4 && !tc::bar_wait(&empty_w[n & OHM], ((n >> 2) + 1) & 1) && ttid == 0)
        flag_status(status, KDA_DEV_TIMEOUT);
      {
        float xk[WP], xv[WP], rk[WP], rv[WP];
#pragma unroll
        for (int t = 0; t < WP; ++t) {
          const float bt = r.beta[t];
          float ak = bt * wt.Kp[t][c], av = bt * (t < W ? __bfloat162float(r.v[t][c]) : 0.f);
#pragma unroll
          for (int u = 0; u < t; ++u) {
            const float a = wt.A[t][u];
            ak = fmaf(-a, xk[u], ak);
            av = fmaf(-a, xv[u], av);
          }
          xk[t] = ak;
          xv[t] = av;
          rk[t] = wt.Qp[t][c];
          rv[t] = 0.f;
        }
#pragma unroll
        for (int t = 0; t < WP; ++t)
#pragma unroll
          for (int u = 0; u <= t; ++u) {
            const float pp = wt.P[t][u];
            rk[t] = fmaf(-pp, xk[u], rk[t]);
            rv[t] = fmaf(pp, xv[u], rv[t]);
          }
        uint8_t* bt = sm + L::BT + (n & 1) * L::B_TILE + (uint32_t)(c >> 6) * L::B_BLOCK;
        float* oh = reinterpret_cast<float*>(sm + L::OH) + (n & OHM) * WP * D;
#pragma unroll
        for (int t = 0; t < WP; ++t) {
          const bf16 hh = __float2bfloat16_rn(rk[t]);
          const bf16 ll = __float2bfloat16_rn(rk[t] - __bfloat162float(hh));
          *reinterpret_cast<bf16*>(bt + tc::sw128(t, c & 63)) = hh;
          *reinterpret_cast<bf16*>(bt + tc::sw128(WP + t, c & 63)) = ll;
          oh[t * D + c] = rv[t];
        }
        tc::fence_proxy_async();
      }
      tc::bar_arrive(&full_w[n & 1]);

      // 4. the record's beta (k, v and g went out by tensor stores)
      if (ok && ttid < W) rec.beta[it.row0 + (size_t)ttid * H] = r.beta[ttid];
    }
    if (ttid == 0) tc::bulk_wait_all();  // the record stores are complete before the CTA exits
  } else if (warp < 8) {
    // ------------------------------------------------------------------ math warps, one team
    const int mtid = tid, half = mtid >> 7, c = mtid & (D - 1);
    // raw inputs of item n into buffer n%2: four tensor-map loads (one thread) and W beta words
    auto fetch = [&](int n) {
      const Item it = item_at(item_index(n), W, H);
      Raw<WP>& r = raw_of(n);
      uint64_t* fb = &full_r[n & 1];
      if (mtid == 0) {
        tc::bulk_wait_read1();  // the record stores of item n-1 have read this buffer
        tc::bar_arrive_expect_tx(fb, (uint32_t)W * (3 * D * 2 + D * 4));
        const int y = it.h, z = it.b * W;
        tc::tma_load_3d(r.k, &maps.k, 0, y, z, fb);
        tc::tma_load_3d(r.q, &maps.q, 0, y, z, fb);
        tc::tma_load_3d(r.v, &maps.v, 0, y, z, fb);
        tc::tma_load_3d(r.g, &maps.g, 0, y, z, fb);
      }
      if (mtid >= 32 && mtid < 32 + W) {
        const int t = mtid - 32;
        cp_async4(&r.beta[t], beta + it.row0 + (size_t)t * H);
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(fb)) : "memory");
      }
    };
    int slot_next = cnt > 0 ? slot_ids[item_index(0) / H] : 0;
    if (cnt > 0) fetch(0);
    for (int n = 0; n < cnt; ++n) {
      const Item it = item_at(item_index(n), W, H);
      const int slot = slot_next;
      if (n + 1 < cnt) slot_next = slot_ids[item_index(n + 1) / H];
      const bool ok = slot >= 0 && slot < num_slots;
      Raw<WP>& r = raw_of(n);
      if (!tc::bar_wait(&full_r[n & 1], (n >> 1) & 1) && mtid == 0) flag_status(status, KDA_DEV_TIMEOUT);
      if (mtid == 0) {  // the raw-input record: the exact stored bits the fold consumes
        if (ok) {
          tc::tma_store_3d(&maps.rk, 0, it.h, it.b * W, r.k);
          tc::tma_store_3d(&maps.rv, 0, it.h, it.b * W, r.v);
          tc::tma_store_3d(&maps.rg, 0, it.h, it.b * W, r.g);
        }
        tc::bulk_commit();  // one group per item (empty when skipped): "all but the latest" is item n-1's
      }
      tc::named_bar(BAR_MATH, MT);  // every math thread is done with item n-1 (and its buffers)
      if (n + 1 < cnt) fetch(n + 1);
      if (!ok && mtid == 0) flag_status(status, KDA_DEV_SLOT_OOB);

      // 1. per channel c: G and Y (half 1), K o e^G and Q o e^G (half 0); is the factored path valid?
      // (every shared-memory load of a phase is issued before its first store: the compiler cannot tell
      //  the raw, work and operand buffers apart)
      bool out_of_span = false;
      {
        float gv[WP], kv[WP], qv[WP];
#pragma unroll
        for (int t = 0; t < WP; ++t) {
          const bool in = t < W;
          gv[t] = in ? r.g[t][c] : 0.f;
          kv[t] = in ? __bfloat162float(r.k[t][c]) : 0.f;
          qv[t] = in && half == 0 ? __bfloat162float(r.q[t][c]) : 0.f;
        }
        float run = 0.f;
#pragma unroll
        for (int t = 0; t < WP; ++t) {
          run = __fadd_rn(run, gv[t]);
          gv[t] = run;
        }
        if (half == 0) {
#pragma unroll
          for (int t = 0; t < WP; ++t) {
            const float ep = __expf(gv[t]);
            wk.Kp[t][c] = kv[t] * ep;
            wk.Qp[t][c] = qv[t] * ep;
          }
        } else {
#pragma unroll
          for (int t = 0; t < WP; ++t) {
            wk.G[t][c] = gv[t];
            wk.Y[t][c] = kv[t] * __expf(-gv[t]);
            out_of_span |= !(fabsf(gv[t]) <= G_SPAN);
          }
        }
      }
      const bool pairwise = tc::named_bar_or(BAR_MATH, MT, out_of_span);

      // 2. A and P, one row per warp (two rows, balanced, when WP = 16)
#pragma unroll
      for (int rr = 0; rr < WP / 8; ++rr) {
        const int t = (rr & 1) ? 8 * rr + 7 - warp : 8 * rr + warp;
        if (pairwise) gram_row<WP, false>(r, wk, t, W, lane);
        else gram_row<WP, true>(r, wk, t, W, lane);
      }
      tc::named_bar(BAR_MATH, MT);

      // 3. per channel: x = (I + A)^-1 diag(beta) y by forward substitution, then P x, with y = K o e^G for
      //    key channel c (half 0: Qh = Q o e^G - P x, into B tile n%2) or y = V for value column c (half 1:
      //    Oh = P x, into its buffer)
      if (n >= 2 && !tc::bar_wait(&empty_w[n & 1], ((n >> 1) + 1) & 1) && mtid == 0)
        flag_status(status, KDA_DEV_TIMEOUT);
      {
        float x[WP], res[WP];
#pragma unroll
        for (int t = 0; t < WP; ++t) {
          const float y = half == 0 ? wk.Kp[t][c] : (t < W ? __bfloat162float(r.v[t][c]) : 0.f);
          res[t] = half == 0 ? wk.Qp[t][c] : 0.f;
          float a = r.beta[t] * y;
#pragma unroll
          for (int u = 0; u < t; ++u) a = fmaf(-wk.A[t][u], x[u], a);
          x[t] = a;
        }
        const float sgn = half == 0 ? -1.f : 1.f;  // Qh = Q o e^G - P x,  Oh = P x
#pragma unroll
        for (int t = 0; t < WP; ++t)
#pragma unroll
          for (int u = 0; u <= t; ++u) res[t] = fmaf(sgn * wk.P[t][u], x[u], res[t]);
        if (half == 0) {
          uint8_t* bt = sm + L::BT + (n & 1) * L::B_TILE + (uint32_t)(c >> 6) * L::B_BLOCK;
#pragma unroll
          for (int t = 0; t < WP; ++t) {
            const bf16 hh = __float2bfloat16_rn(res[t]);
            const bf16 ll = __float2bfloat16_rn(res[t] - __bfloat162float(hh));
            *reinterpret_cast<bf16*>(bt + tc::sw128(t, c & 63)) = hh;
            *reinterpret_cast<bf16*>(bt + tc::sw128(WP + t, c & 63)) = ll;
          }
          tc::fence_proxy_async();
        } else {
          float* oh = reinterpret_cast<float*>(sm + L::OH) + (n & 1) * WP * D;
#pragma unroll
          for (int t = 0; t < WP; ++t) oh[t * D + c] = res[t];
        }
      }
      tc::bar_arrive(&full_w[n & 1]);

      // 4. the record's beta (k, v and g went out by tensor stores)
      if (ok && mtid < W) rec.beta[it.row0 + (size_t)mtid * H] = r.beta[mtid];
    }
    if (mtid == 0) tc::bulk_wait_all();  // the record stores are complete before the CTA exits
  } else {
    // ------------------------------------------------------------------ state warps
    const int sidx = tid - MT, half = sidx >> 7, c = sidx & (D - 1);
    const uint32_t tlane = (uint32_t)((warp & 3) * 32) << 16;  // this warp's 32 tensor-memory lanes
    auto issue_state = [&](int n, int slot) {
      const Item it = item_at(item_index(n), W, H);
      uint64_t* fb = &full_s[n % STAGES];
      if (slot >= 0 && slot < num_slots) {
        tc::bar_arrive_expect_tx(fb, STATE_BYTES);
        tc::bulk_g2s(sm + (n % STAGES) * STATE_BYTES, pool + ((size_t)slot * H + it.h) * D * D, STATE_BYTES, fb);
      } else {
        tc::bar_arrive(fb);
      }
    };
    auto epilogue = [&](int m, bool ok) {
      const Item it = item_at(item_index(m), W, H);
      const bool done = __all_sync(0xffffffffu, tc::bar_wait(&mma_bar[m & 1], (m >> 1) & 1));
      if (!done && lane == 0) flag_status(status, KDA_DEV_TIMEOUT);
      tc::fence_after_sync();
      // accumulator column t = S0 hi (first accumulator) or S0 lo (second) against Qh hi of token t, column
      // WP + t against its lo part
      // (four accumulators: S0 hi / lo x the two halves of the K range, 32 columns apart)
      float d[2 * WP];
#pragma unroll
      for (int q = 0; q < 2 * WP; q += 16) {
        tc::tmem_ld16(tm + tlane + (m & 1) * BUF_COLS + COL_ACC + q, d + q);
#pragma unroll
        for (int a = 1; a < 4; ++a) {  // the other three partial products, in a fixed order
          float d2[16];
          tc::tmem_ld16(tm + tlane + (m & 1) * BUF_COLS + ((a & 1) ? COL_ACC2 : COL_ACC) + 32 * (a >> 1) + q, d2);
#pragma unroll
          for (int e = 0; e < 16; ++e) d[q + e] += d2[e];
        }
      }
      const float* oh = reinterpret_cast<const float*>(sm + L::OH) + (m & OHM) * WP * D;
      if (ok && done) {
        constexpr int TH = WP / 2;
#pragma unroll
        for (int tt = 0; tt < TH; ++tt) {
          const int t = TH * half + tt;
          const float dt = half ? d[TH + tt] + d[WP + TH + tt] : d[tt] + d[WP + tt];
          if (t < W) out[(it.row0 + (size_t)t * H) * D + c] = from_f32<Tout>(dt + oh[t * D + c]);
        }
        if (sidx == 0) add_work(status, W);
      }
      tc::fence_before_sync();
      tc::bar_arrive(&empty_w[m & OHM]);
    };
    if (sidx == 0)
      for (int n = 0; n < STAGES && n < cnt; ++n) issue_state(n, slot_ids[item_index(n) / H]);
    bool ok_prev = false;
    for (int n = 0; n < cnt; ++n) {
      // slot ids loaded here are consumed after this item's split: its epilogue's and a later copy's
      const int slot_n = slot_ids[item_index(n) / H];
      const int slot_ahead = sidx == 0 && n + STAGES < cnt ? slot_ids[item_index(n + STAGES) / H] : 0;
      // S0^T of item n into tensor-memory buffer n%2: lane c, column 32*half + i holds key rows
      // 64*half + 2i (low half) and 2i + 1 (high half)
      if (!__all_sync(0xffffffffu, tc::bar_wait(&full_s[n % STAGES], (n / STAGES) & 1)) && lane == 0)
        flag_status(status, KDA_DEV_TIMEOUT);
      const float* st = reinterpret_cast<const float*>(sm + (n % STAGES) * STATE_BYTES) + (size_t)64 * half * D + c;
      const uint32_t tb = tm + tlane + (n & 1) * BUF_COLS;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 x = make_float2(st[(32 * part + 2 * e) * D], st[(32 * part + 2 * e + 1) * D]);
          const __nv_bfloat162 hh = __float22bfloat162_rn(x);
          const float2 hf = __bfloat1622float2(hh);
          const __nv_bfloat162 ll = __float22bfloat162_rn(make_float2(x.x - hf.x, x.y - hf.y));
          hi[e] = *reinterpret_cast<const uint32_t*>(&hh);
          lo[e] = *reinterpret_cast<const uint32_t*>(&ll);
        }
        tc::tmem_st16(tb + COL_AHI + 32 * half + 16 * part, hi);
        tc::tmem_st16(tb + COL_ALO + 32 * half + 16 * part, lo);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::named_bar(BAR_STATE, ST);  // stage n%STAGES read; tensor-memory buffer n%2 written
      if (sidx == 0 && n + STAGES < cnt) issue_state(n + STAGES, slot_ahead);
      if (n >= 1) epilogue(n - 1, ok_prev);  // frees item n-1's Qh / Oh buffers before waiting on item n's
      ok_prev = slot_n >= 0 && slot_n < num_slots;
      if (sidx < 128 && (sidx & 31) == 0) {
        if (!tc::bar_wait(&full_w[n & 1], (n >> 1) & 1)) flag_status(status, KDA_DEV_TIMEOUT);
        tc::fence_after_sync();
        // D = S0^T [Qh hi; Qh lo]^T (128 value columns x 2WP), 8 K-steps, from four threads side by side:
        // thread 0 of warp 8 + 2 kh + part issues S0 hi (part 0) or lo (part 1) over K-steps 4 kh .. 4 kh + 3
        // into an accumulator of its own (a chain of dependent MMAs advances ~90 cycles a step, so four
        // 4-deep chains finish well before two 8-deep ones).  A descriptor of base + off equals the base
        // descriptor + off/16 (the start-address field).
        const int part = (sidx >> 5) & 1, kh = sidx >> 6;
        const uint64_t bdesc = tc::sdesc(tc::smem_u32(sm + L::BT + (n & 1) * L::B_TILE));
        const uint32_t buf = tm + (n & 1) * BUF_COLS;
        constexpr uint32_t idesc = tc::idesc_bf16(128, L::B_ROWS);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int ks = 4 * kh + kk;
          tc::mma_ts(buf + (part ? COL_ACC2 : COL_ACC) + 32u * kh, buf + (part ? COL_ALO : COL_AHI) + 8 * ks,
                     bdesc + (((ks >> 2) * L::B_BLOCK + (ks & 3) * 32u) >> 4), idesc, kk != 0);
        }
        tc::commit(&mma_bar[n & 1]);
      }
    }
    if (cnt > 0) epilogue(cnt - 1, ok_prev);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 8) tc::tmem_dealloc(tm, TMEM_COLS);
}

template <int WP, typename Tout>
cudaError_t launch_wp(const VerifyArgs& a, cudaStream_t st) {
  using L = PLayout<WP>;
  cudaError_t e = cudaFuncSetAttribute(verify_tc_kernel<WP, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L::BYTES);
  if (e != cudaSuccess) return e;
  const int items = a.B * a.H, sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const long long rows = (long long)a.B * a.W;
  if (rows > 0x7fffffff) return cudaErrorInvalidValue;  // TMA coordinates are 32-bit
  VMaps maps;
  if (!encode_token_map(&maps.q, a.q, false, rows, a.H, a.W) || !encode_token_map(&maps.k, a.k, false, rows, a.H, a.W) ||
      !encode_token_map(&maps.v, a.v, false, rows, a.H, a.W) || !encode_token_map(&maps.g, a.g, true, rows, a.H, a.W) ||
      !encode_token_map(&maps.rk, a.rec.k, false, rows, a.H, a.W) ||
      !encode_token_map(&maps.rv, a.rec.v, false, rows, a.H, a.W) ||
      !encode_token_map(&maps.rg, a.rec.g, true, rows, a.H, a.W))
    return cudaErrorNotSupported;
  const int grid = items < sms ? items : sms;
  verify_tc_kernel<WP, Tout><<<grid, NT, L::BYTES, st>>>(maps, a.beta, a.B, a.W, a.H, a.pool, a.num_slots, a.slot_ids,
                                                         static_cast<Tout*>(a.out), a.rec, a.status);
  return cudaGetLastError();
}

}  // namespace

bool verify_tc_supported(const VerifyArgs& a) {
  return a.in_bf16 && a.d == D && a.W >= 1 && a.W <= 16 && a.snapshot_out == nullptr;
}

cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t st) {
  if (a.W <= 8) return a.out_bf16 ? launch_wp<8, bf16>(a, st) : launch_wp<8, float>(a, st);
  return a.out_bf16 ? launch_wp<16, bf16>(a, st) : launch_wp<16, float>(a, st);
}

}  // namespace kda
