// CF-BI prefill, chunk-parallel: the same row-level contract as the token-sequential prefill and the decode
// (cfbi.cu), with the work that does not depend on the recurrent state taken off the sequential path.
//
// Source: "Kimi K3.1 inference zero mismatch" (LLMNews), section 6.1 (CF-BI): a position's output depends
// only on the entry state of its chunk and the rows before it in that chunk, and prefill computes the
// rows in bulk where decode computes one.  The row arithmetic is the KDA update of "Kimi K3: Architecture
// and SGLang Day-0 Support" (KDA math box) unrolled over the open chunk (see cfbi.cu).
//
// Two kernels:
//  * rows (one CTA per (chunk, sequence, head), all chunks at once): G, A_t, P_t, T_t, R_t, and the
//    state-free parts of each output, qh_t = q_t o e^{G_t} - sum_u R_tu k_u o e^{G_u} and oh_t = sum_u R_tu v_u.
//    Only the rows of T depend on one another, and lane v of one warp walks column v of T down the chunk,
//    which reads only its own column of the rows above.
//  * state (one CTA per (8 value columns, sequence, head), the chunks in order): o_t = S_c^T qh_t + oh_t for
//    the chunk's tokens, then, if the chunk is complete, S_{c+1} = Diag(e^{G_15}) S_c + (K o e^{G_15 - G})^T U
//    with U = T diag(beta) (V - (K o e^G) S_c).  Every value column of S evolves on its own, so the columns
//    are split over CTAs.
// Each output element and each state element is formed by the same round-to-nearest operations in the same
// order as in cfbi.cu (the per-row steps, the read-out and the fold), so the bits match the token-sequential
// prefill and the decode whatever the split between them.
//
// Workspace (kda_cfbi_prefill_chunked_workspace_size), laid out so that the state pass fetches a chunk's
// operands as a few contiguous bulk copies: qh per head and token ([H][T][2][68] fp32, each key half padded
// to 68 floats), oh per head, 8-column group and token ([H][16][T][8]), a record per chunk ([T/16 + 2N + 2][H]
// records; chunk k of sequence i at index floor(s0_i / 16) + 2i + k, which keeps the sequences' ranges
// apart) holding the chunk's rows and, for a complete chunk, the fold's state-free factors k_u o e^{G_u}
// (padded like qh), k_u o e^{G_15 - G_u}, e^{G_15}, the rows' A | beta | T tails and their values by column
// group, and each (sequence, head)'s row count at entry ([N][H] int32).
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
constexpr int CG = 8;             // value columns per state CTA
constexpr int TAIL = RF - R_A;    // A_t | beta | T_t | padding: 36 floats from R_A
constexpr int PAD = RF - R_T - CH;  // padding floats after T_t
constexpr int HP = 68;               // a key half padded (conflict-free 16-byte loads of both halves)
constexpr int QP = 2 * HP;           // a padded key row
constexpr int NG = D / CG;           // value column groups
// a chunk's record in the workspace: rows [16][RF] | kp [16][QP] | kh [16][128] | eg [128] | tail [16][TAIL] |
// v [NG][16][CG]
constexpr int REC_KP = CH * RF, REC_KH = REC_KP + CH * QP, REC_EG = REC_KH + CH * D, REC_TL = REC_EG + D,
              REC_VG = REC_TL + CH * TAIL, REC_FLOATS = REC_VG + CH * D;
static_assert(REC_KP % 4 == 0 && REC_KH % 4 == 0 && REC_EG % 4 == 0 && REC_TL % 4 == 0 && REC_VG % 4 == 0 &&
                  REC_FLOATS % 4 == 0,
              "record pieces are 16-byte aligned");
__device__ __forceinline__ size_t qh_at(int64_t T, int h, int64_t t) { return ((size_t)h * T + t) * QP; }
__device__ __forceinline__ size_t oh_at(int64_t T, int h, int g, int64_t t) { return (((size_t)h * NG + g) * T + t) * CG; }
static_assert(R_A % 4 == 0 && TAIL % 4 == 0, "row tail copies in 16-byte pieces");

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// A sequence as one (sequence, head) walker sees it: its tokens [s0, s0 + len), its row count L before the
// call, its slot; false (and nothing to do) when the sequence, slot or count is out of range.  The rows
// kernel reads L from `counts` and records it in the workspace; the state kernel, whose CTAs of one
// (sequence, head) must agree while one of them rewrites `counts`, reads the record.
struct SeqView {
  int64_t s0;
  int len, L, slot, nch;
};
__device__ __forceinline__ bool seq_view(const int32_t* cu, int64_t T, int max_seqlen, int i, int h, int H,
                                         const int32_t* slot_ids, int num_slots, int L, SeqView& sv,
                                         int32_t* status, bool flag) {
  const int64_t s0 = cu[i], s1 = cu[i + 1];
  if (s0 < 0 || s1 < s0 || s1 > T || s1 - s0 > (int64_t)max_seqlen) {
    if (flag) flag_status(status, KDA_DEV_SEQ_OOB);
    return false;
  }
  const int slot = slot_ids[i];
  if (slot < 0 || slot >= num_slots) {
    if (flag) flag_status(status, KDA_DEV_SLOT_OOB);
    return false;
  }
  if (L < 0 || L >= CH) {
    if (flag) flag_status(status, KDA_DEV_SLOT_OOB);
    return false;
  }
  sv.s0 = s0;
  sv.len = (int)(s1 - s0);
  sv.L = L;
  sv.slot = slot;
  sv.nch = (L + sv.len + CH - 1) / CH;
  return true;
}

// chunk k of the walk: rows r_lo .. r_hi are new (row r is token s0 + 16 k + r - L)
__device__ __forceinline__ int chunk_lo(const SeqView& s, int k) { return k == 0 ? s.L : 0; }
__device__ __forceinline__ int chunk_hi(const SeqView& s, int k) {
  const int last = s.L + s.len - 1 - CH * k;
  return last < CH - 1 ? last : CH - 1;
}
__device__ __forceinline__ size_t rows_index(const SeqView& s, int i, int k) { return (size_t)(s.s0 / CH) + 2 * (size_t)i + k; }

struct RowsSmem {
  alignas(16) float rows[CH][RF];
  alignas(16) float q[CH][D];
  alignas(16) float ke[CH][D];  // k_u o e^{G_u}
  float p[CH][CH];              // P_t[u]
  float r[CH][CH];              // R_t[u]
};

template <typename Tin>
__global__ void __launch_bounds__(NT) cfbi_rows_kernel(CfbiArgs a, CfbiWorkspace w) {
  extern __shared__ float4 smem4[];
  RowsSmem& s = *reinterpret_cast<RowsSmem*>(smem4);
  const int k = blockIdx.x, i = blockIdx.y, h = blockIdx.z, H = a.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  SeqView sv;
  int L = -1;
  {
    const int slot = a.slot_ids[i];
    if (slot >= 0 && slot < a.num_slots) L = a.counts[(size_t)slot * H + h];
  }
  if (k == 0 && tid == 0) w.count[(size_t)i * H + h] = L;
  if (!seq_view(a.cu, a.T, a.max_seqlen, i, h, H, a.slot_ids, a.num_slots, L, sv, a.status, false)) return;
  if (k >= sv.nch) return;
  const int lo = chunk_lo(sv, k), hi = chunk_hi(sv, k);
  const size_t sh = (size_t)sv.slot * H + h;
  if (k == 0) {  // the rows the chunk already holds
    const float* cg = a.cache + sh * CH * RF;
    for (int e = tid; e < lo * RF / 4; e += NT) cp_async16(reinterpret_cast<float4*>(&s.rows[0][0]) + e, reinterpret_cast<const float4*>(cg) + e);
  }
  const Tin* q = static_cast<const Tin*>(a.q);
  const Tin* kk = static_cast<const Tin*>(a.k);
  const Tin* v = static_cast<const Tin*>(a.v);
  const int64_t t0 = sv.s0 + (int64_t)CH * k - sv.L;  // token of row 0 (row r: t0 + r)
  for (int e = tid; e < (hi - lo + 1) * D; e += NT) {
    const int r = lo + e / D, j = e % D;
    const size_t x = ((size_t)(t0 + r) * H + h) * D + j;
    s.rows[r][R_K + j] = to_f32(kk[x]);
    s.rows[r][R_V + j] = to_f32(v[x]);
    s.rows[r][R_G + j] = a.g[x];
    s.q[r][j] = to_f32(q[x]);
  }
  if (tid >= lo && tid <= hi) s.rows[tid][R_BETA] = a.beta[(size_t)(t0 + tid) * H + h];
  cp_async_wait_all();
  __syncthreads();
  // 1. G_t = G_{t-1} + g_t down the chunk; the slots of a new row no step writes are zeroed
  if (tid < D) {
    for (int r = lo; r <= hi; ++r) s.rows[r][R_G + tid] = __fadd_rn(r > 0 ? s.rows[r - 1][R_G + tid] : 0.f, s.rows[r][R_G + tid]);
  } else {
    for (int e = tid - D; e < (hi - lo + 1) * (CH + PAD); e += NT - D) {
      const int r = lo + e / (CH + PAD), x = e % (CH + PAD);  // A_t[u >= t] and the padding
      if (x < CH) {
        if (x >= r) s.rows[r][R_A + x] = 0.f;
      } else {
        s.rows[r][R_T + CH + x - CH] = 0.f;
      }
    }
  }
  __syncthreads();
  // 2. A_t[u] (u < t) and P_t[u] (u <= t) for every new row t: one warp per pair, lane l channels 4l .. 4l+3
  //    in order, then the fixed xor butterfly (the decode's step 2)
  {
    const int npairs = (hi + 1) * (hi + 2) / 2 - lo * (lo + 1) / 2;
    for (int pi = warp; pi < npairs; pi += NT / 32) {
      int t = lo, rem = pi;
      while (rem > t) {
        rem -= t + 1;
        ++t;
      }
      const int u = rem;
      const float* rt = s.rows[t];
      const float* ru = s.rows[u];
      const float4 kt = *reinterpret_cast<const float4*>(rt + R_K + 4 * lane);
      const float4 gt = *reinterpret_cast<const float4*>(rt + R_G + 4 * lane);
      const float4 qt = *reinterpret_cast<const float4*>(&s.q[t][4 * lane]);
      const float4 ku = *reinterpret_cast<const float4*>(ru + R_K + 4 * lane);
      const float4 gu = *reinterpret_cast<const float4*>(ru + R_G + 4 * lane);
      const float kc[4] = {ku.x, ku.y, ku.z, ku.w}, gc[4] = {gu.x, gu.y, gu.z, gu.w};
      const float ktc[4] = {kt.x, kt.y, kt.z, kt.w}, gtc[4] = {gt.x, gt.y, gt.z, gt.w};
      const float qc[4] = {qt.x, qt.y, qt.z, qt.w};
      float av = 0.f, pv = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float x = __fmul_rn(kc[c], __expf(__fsub_rn(gtc[c], gc[c])));
        av = __fmaf_rn(ktc[c], x, av);
        pv = __fmaf_rn(qc[c], x, pv);
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {
        av = __fadd_rn(av, __shfl_xor_sync(0xffffffffu, av, m));
        pv = __fadd_rn(pv, __shfl_xor_sync(0xffffffffu, pv, m));
      }
      if (lane == 0) {
        if (u < t) s.rows[t][R_A + u] = __fmul_rn(s.rows[t][R_BETA], av);
        s.p[t][u] = pv;
      }
    }
  }
  __syncthreads();
  // 3. rows of T: lane v walks column v down the chunk (it reads only its own column of the rows above)
  if (warp == 0 && lane < CH) {
    const int vv = lane;
    for (int t = lo; t <= hi; ++t) {
      float acc = vv == t ? 1.f : 0.f;
#pragma unroll
      for (int u = 0; u < CH - 1; ++u)
        if (u >= vv && u < t) acc = __fmaf_rn(-s.rows[t][R_A + u], s.rows[u][R_T + vv], acc);
      s.rows[t][R_T + vv] = acc;
    }
  }
  // k_u o e^{G_u} for the rows 0 .. hi (the same product the decode forms inside its step 4)
  for (int e = tid; e < (hi + 1) * D; e += NT) {
    const int u = e / D, j = e % D;
    s.ke[u][j] = __fmul_rn(s.rows[u][R_K + j], __expf(s.rows[u][R_G + j]));
  }
  __syncthreads();
  // R_t = (P_t T) diag(beta) for every new row (lane v of the decode's step 3, one thread per (t, v))
  {
    const int t = lo + tid / CH, vv = tid % CH;
    if (t <= hi) {
      float acc = 0.f;
#pragma unroll
      for (int x = 0; x < CH; ++x)
        if (x >= vv && x <= t) acc = __fmaf_rn(s.p[t][x], s.rows[x][R_T + vv], acc);
      s.r[t][vv] = vv <= t ? __fmul_rn(acc, s.rows[vv][R_BETA]) : 0.f;
    }
  }
  __syncthreads();
  // 4. qh (key channel j) and oh (value column c) of every new row, to the workspace
  for (int e = tid; e < (hi - lo + 1) * 2 * D; e += NT) {
    const int t = lo + e / (2 * D), x = e % (2 * D);
    if (x < D) {
      const int j = x;
      float acc = __fmul_rn(s.q[t][j], __expf(s.rows[t][R_G + j]));
#pragma unroll
      for (int u = 0; u < CH; ++u)
        if (u <= t) acc = __fmaf_rn(-s.r[t][u], s.ke[u][j], acc);
      w.qh[qh_at(a.T, h, t0 + t) + (j >> 6) * HP + (j & 63)] = acc;
    } else {
      const int c = x - D;
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < CH; ++u)
        if (u <= t) acc = __fmaf_rn(s.r[t][u], s.rows[u][R_V + c], acc);
      w.oh[oh_at(a.T, h, c / CG, t0 + t) + c % CG] = acc;
    }
  }
  // the chunk's record: rows 0 .. hi, and for a complete chunk the fold's state-free factors (the same
  // products the fold forms: kp = k_u o e^{G_u}, kh = k_u o e^{G_15 - G_u}, eg = e^{G_15})
  float* dst = w.rows + (rows_index(sv, i, k) * H + h) * REC_FLOATS;
  for (int e = tid; e < (hi + 1) * RF / 4; e += NT)
    reinterpret_cast<float4*>(dst)[e] = reinterpret_cast<const float4*>(&s.rows[0][0])[e];
  if (hi == CH - 1) {
    for (int e = tid; e < CH * D; e += NT) {
      const int u = e / D, j = e % D;
      dst[REC_KP + u * QP + (j >> 6) * HP + (j & 63)] = s.ke[u][j];
      dst[REC_KH + e] = __fmul_rn(s.rows[u][R_K + j], __expf(__fsub_rn(s.rows[CH - 1][R_G + j], s.rows[u][R_G + j])));
      dst[REC_VG + ((j / CG) * CH + u) * CG + j % CG] = s.rows[u][R_V + j];
    }
    if (tid < D) dst[REC_EG + tid] = __expf(s.rows[CH - 1][R_G + tid]);
    for (int e = tid; e < CH * TAIL; e += NT) dst[REC_TL + e] = s.rows[e / TAIL][R_A + e % TAIL];
  }
}

// One chunk's operands of the state pass, for this CTA's CG value columns.  qh and kp keep each row's two
// key halves 68 floats apart (conflict-free 16-byte loads of both halves); the fold's operands (kp, kh, eg,
// tail, v) are fetched only for a complete chunk.
struct StateBuf {
  alignas(16) float qh[CH][2][HP];
  alignas(16) float kp[CH][2][HP];
  alignas(16) float kh[CH][D];
  alignas(16) float eg[D];
  alignas(16) float tail[CH][TAIL];  // A_t | beta | T_t | padding
  alignas(16) float oh[CH][CG];
  alignas(16) float v[CH][CG];
};
constexpr int SH = 64 * CG + 8;  // floats between the state's two key halves (conflict-free float2 loads)
constexpr int NBUF = 3;          // chunks in flight: the current one and two ahead
struct StateSmem {
  alignas(16) float S[2 * SH];   // the state's key rows of this CTA's columns: [half][64][CG]
  float ws[2][CH][CG];
  alignas(16) float y[CH][CG];
  alignas(16) float U[CH][CG];
  StateBuf buf[NBUF];
  uint64_t bar[NBUF];            // a buffer's bulk copies have landed
};
__device__ __forceinline__ float& s_at(float* S, int j, int c) { return S[(j >> 6) * SH + (j & 63) * CG + c]; }

// 2 x 2 of the 64-term chains out[r][c] = sum_e a[r][half][e] S[half][e][c] (e in order), for rows r0, r0 + 1
// and columns c0, c0 + 1 of one key half: the read-out (a = qh) and (K o e^G) S_c (a = kp) of the fold.
__device__ __forceinline__ void chains2x2(const float (*a)[2][HP], const float* S, int r0, int c0, int half,
                                          float (&acc)[2][2]) {
  const float* s = S + half * SH + c0;
  const float* a0 = a[r0][half];
  const float* a1 = a[r0 + 1][half];
  acc[0][0] = acc[0][1] = acc[1][0] = acc[1][1] = 0.f;
  // blocks of 8 key rows; the next block's operands are loaded while the current block's products run
  float4 x[2][4];
  float2 sv[2][8];
  auto load = [&](int blk, int b) {
    x[b][0] = *reinterpret_cast<const float4*>(a0 + 8 * blk);
    x[b][1] = *reinterpret_cast<const float4*>(a0 + 8 * blk + 4);
    x[b][2] = *reinterpret_cast<const float4*>(a1 + 8 * blk);
    x[b][3] = *reinterpret_cast<const float4*>(a1 + 8 * blk + 4);
#pragma unroll
    for (int q = 0; q < 8; ++q) sv[b][q] = *reinterpret_cast<const float2*>(s + (8 * blk + q) * CG);
  };
  load(0, 0);
#pragma unroll
  for (int blk = 0; blk < 8; ++blk) {
    const int b = blk & 1;
    if (blk + 1 < 8) load(blk + 1, b ^ 1);
    const float r0v[8] = {x[b][0].x, x[b][0].y, x[b][0].z, x[b][0].w, x[b][1].x, x[b][1].y, x[b][1].z, x[b][1].w};
    const float r1v[8] = {x[b][2].x, x[b][2].y, x[b][2].z, x[b][2].w, x[b][3].x, x[b][3].y, x[b][3].z, x[b][3].w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      acc[0][0] = __fmaf_rn(r0v[q], sv[b][q].x, acc[0][0]);
      acc[0][1] = __fmaf_rn(r0v[q], sv[b][q].y, acc[0][1]);
      acc[1][0] = __fmaf_rn(r1v[q], sv[b][q].x, acc[1][0]);
      acc[1][1] = __fmaf_rn(r1v[q], sv[b][q].y, acc[1][1]);
    }
  }
}

template <typename Tout>
__global__ void __launch_bounds__(NT) cfbi_state_kernel(CfbiArgs a, CfbiWorkspace w) {
  extern __shared__ float4 smem4[];
  StateSmem& s = *reinterpret_cast<StateSmem*>(smem4);
  const int grp = blockIdx.x, i = blockIdx.y, h = blockIdx.z, H = a.H, c0 = grp * CG;
  const int tid = threadIdx.x;
  SeqView sv;
  if (!seq_view(a.cu, a.T, a.max_seqlen, i, h, H, a.slot_ids, a.num_slots, w.count[(size_t)i * H + h], sv, a.status,
                grp == 0 && tid == 0))
    return;
  const size_t sh = (size_t)sv.slot * H + h;
  float* Sg = a.pool + sh * D * D;
  const int64_t tbase = sv.s0 - sv.L;  // token of row 0 of chunk 0
  // chunk k's operands into buffer b: bulk copies issued by thread 128 on the buffer's mbarrier (the fold's
  // operands only when the chunk is complete)
  auto fetch = [&](int k, int b) {
    StateBuf& f = s.buf[b];
    const int lo = chunk_lo(sv, k), hi = chunk_hi(sv, k), n = hi - lo + 1;
    const int64_t t0 = tbase + (int64_t)CH * k;
    const bool full = hi == CH - 1;
    const uint32_t bytes = (n > 0 ? (uint32_t)n * (QP + CG) * 4 : 0u) +
                           (full ? (uint32_t)(CH * QP + CH * D + D + CH * TAIL + CH * CG) * 4 : 0u);
    tc::bar_arrive_expect_tx(&s.bar[b], bytes);
    if (n > 0) {
      tc::bulk_g2s(&f.qh[lo][0][0], w.qh + qh_at(a.T, h, t0 + lo), (uint32_t)n * QP * 4, &s.bar[b]);
      tc::bulk_g2s(&f.oh[lo][0], w.oh + oh_at(a.T, h, grp, t0 + lo), (uint32_t)n * CG * 4, &s.bar[b]);
    }
    if (full) {
      const float* rec = w.rows + (rows_index(sv, i, k) * H + h) * REC_FLOATS;
      tc::bulk_g2s(&f.kp[0][0][0], rec + REC_KP, CH * QP * 4, &s.bar[b]);
      tc::bulk_g2s(&f.kh[0][0], rec + REC_KH, CH * D * 4, &s.bar[b]);
      tc::bulk_g2s(&f.eg[0], rec + REC_EG, D * 4, &s.bar[b]);
      tc::bulk_g2s(&f.tail[0][0], rec + REC_TL, CH * TAIL * 4, &s.bar[b]);
      tc::bulk_g2s(&f.v[0][0], rec + REC_VG + grp * CH * CG, CH * CG * 4, &s.bar[b]);
    }
  };
  if (tid == 0) {
    for (int b = 0; b < NBUF; ++b) tc::bar_init(&s.bar[b], 1);
    tc::bar_fence_init();
  }
  __syncthreads();
  if (tid >= 128) {  // this CTA's columns of the state (rows 32 bytes apart)
    for (int e = tid - 128; e < D * CG / 4; e += NT - 128) {
      const int j = e / (CG / 4), x = e % (CG / 4);
      cp_async16(&s_at(s.S, j, 4 * x), Sg + (size_t)j * D + c0 + 4 * x);
    }
  }
  if (tid == 128) {
    if (sv.nch > 0) fetch(0, 0);
    if (sv.nch > 1) fetch(1, 1);
  }
  Tout* out = static_cast<Tout*>(a.out);
  bool ok = true;
  int k = 0;
  for (; k < sv.nch; ++k) {
    const int b = k % NBUF;
    cp_async_wait_all();
    ok = __syncthreads_and(tc::bar_wait(&s.bar[b], (uint32_t)(k / NBUF) & 1u)) != 0;
    if (!ok) break;  // chunk k's operands did not land in time
    // chunk k - 1 is done with buffer (k + 2) % 3
    if (tid == 128 && k + 2 < sv.nch) fetch(k + 2, (k + 2) % NBUF);
    const StateBuf& f = s.buf[b];
    const int lo = chunk_lo(sv, k), hi = chunk_hi(sv, k);
    const bool folds = hi == CH - 1;
    const int64_t t0 = tbase + (int64_t)CH * k;
    // threads 0-63: the read-out, 2 tokens x 2 columns of one key half each; threads 64-127: (K o e^G) S_c,
    // 2 rows u x 2 columns; the halves of one output in adjacent lanes
    if (tid < 128) {
      const int x = tid & 63, half = x & 1, cp = (x >> 1) & 3, rp = x >> 3;
      float acc[2][2];
      if (tid < 64) {
        if (2 * rp + 1 >= lo && 2 * rp <= hi) chains2x2(f.qh, s.S, 2 * rp, 2 * cp, half, acc);
        else acc[0][0] = acc[0][1] = acc[1][0] = acc[1][1] = 0.f;
      } else if (folds) {
        chains2x2(f.kp, s.S, 2 * rp, 2 * cp, half, acc);
      } else {
        acc[0][0] = acc[0][1] = acc[1][0] = acc[1][1] = 0.f;
      }
      float oth[2][2];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int c = 0; c < 2; ++c) oth[r][c] = __shfl_xor_sync(0xffffffffu, acc[r][c], 1);
      if (tid < 64) {
        if (half == 0) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int t = 2 * rp + r;
            if (t >= lo && t <= hi) {
#pragma unroll
              for (int c = 0; c < 2; ++c)
                out[((size_t)(t0 + t) * H + h) * D + c0 + 2 * cp + c] =
                    from_f32<Tout>(__fadd_rn(__fadd_rn(acc[r][c], oth[r][c]), f.oh[t][2 * cp + c]));
            }
          }
        }
      } else if (folds) {
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int c = 0; c < 2; ++c) s.ws[half][2 * rp + r][2 * cp + c] = acc[r][c];
      }
    }
    if (!folds) continue;  // the chunk stays open: no fold
    __syncthreads();
    if (tid < CH * CG) {  // y = diag(beta) (V - (K o e^G) S_c)
      const int ww = tid / CG, cl = tid % CG;
      s.y[ww][cl] = __fmul_rn(f.tail[ww][R_BETA - R_A], __fsub_rn(f.v[ww][cl], __fadd_rn(s.ws[0][ww][cl], s.ws[1][ww][cl])));
    }
    __syncthreads();
    if (tid < CH * CG) {  // U = T y
      const int u = tid / CG, cl = tid % CG;
      float acc = 0.f;
#pragma unroll
      for (int x = 0; x < CH; ++x)
        if (x <= u) acc = __fmaf_rn(f.tail[u][R_T - R_A + x], s.y[x][cl], acc);
      s.U[u][cl] = acc;
    }
    __syncthreads();
    // S_{c+1}[j][c] = e^{G_15[j]} S_c[j][c] + sum_u k_u[j] e^{G_15[j] - G_u[j]} U[u][c]: thread (j, 4 columns)
    {
      const int j = tid >> 1, cq = 4 * (tid & 1);
      float* sp = &s_at(s.S, j, cq);
      const float e15 = f.eg[j];
      float x[4] = {__fmul_rn(e15, sp[0]), __fmul_rn(e15, sp[1]), __fmul_rn(e15, sp[2]), __fmul_rn(e15, sp[3])};
#pragma unroll
      for (int u = 0; u < CH; ++u) {
        const float kv = f.kh[u][j];
        const float4 uu = *reinterpret_cast<const float4*>(&s.U[u][cq]);
        x[0] = __fmaf_rn(kv, uu.x, x[0]);
        x[1] = __fmaf_rn(kv, uu.y, x[1]);
        x[2] = __fmaf_rn(kv, uu.z, x[2]);
        x[3] = __fmaf_rn(kv, uu.w, x[3]);
      }
      sp[0] = x[0], sp[1] = x[1], sp[2] = x[2], sp[3] = x[3];
    }
  }
  cp_async_wait_all();  // (a walk with no chunk has waited for nothing yet)
  if (!ok) {  // report the timeout, give the copies in flight one more bounded wait each, leave the state
    if (tid == 0) flag_status(a.status, KDA_DEV_TIMEOUT);
    if (tid == 128)
      for (int c = k; c < sv.nch && c < k + 2; ++c) tc::bar_wait(&s.bar[c % NBUF], (uint32_t)(c / NBUF) & 1u);
    return;
  }
  __syncthreads();
  for (int e = tid; e < D * CG / 4; e += NT) {
    const int j = e / (CG / 4), x = e % (CG / 4);
    *reinterpret_cast<float4*>(Sg + (size_t)j * D + c0 + 4 * x) = *reinterpret_cast<const float4*>(&s_at(s.S, j, 4 * x));
  }
  if (grp != 0) return;
  // the open chunk's rows and position (one CTA per (sequence, head))
  const int last = sv.nch - 1, hi = sv.len > 0 ? chunk_hi(sv, last) : sv.L - 1;
  if (sv.len > 0 && hi < CH - 1) {
    const float* rs = w.rows + (rows_index(sv, i, last) * H + h) * REC_FLOATS;
    float* cg = a.cache + sh * CH * RF;
    for (int e = tid; e < (hi + 1) * RF / 4; e += NT)
      reinterpret_cast<float4*>(cg)[e] = reinterpret_cast<const float4*>(rs)[e];
  }
  if (tid == 0) {
    a.counts[sh] = (sv.L + sv.len) % CH;
    add_work(a.status, sv.len);
  }
}

template <typename Tin, typename Tout>
cudaError_t launch_t(const CfbiArgs& a, const CfbiWorkspace& w, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(cfbi_rows_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(RowsSmem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(cfbi_state_kernel<Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sizeof(StateSmem));
  if (e != cudaSuccess) return e;
  const int cmax = (a.max_seqlen + 2 * CH - 2) / CH;  // chunks of the longest sequence from any start position
  if (cmax > 0) {
    cfbi_rows_kernel<Tin><<<dim3(cmax, a.N, a.H), NT, sizeof(RowsSmem), st>>>(a, w);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  cfbi_state_kernel<Tout><<<dim3(D / CG, a.N, a.H), NT, sizeof(StateSmem), st>>>(a, w);
  return cudaGetLastError();
}

}  // namespace

size_t cfbi_chunked_records(int64_t T, int N) { return (size_t)(T / CH) + 2 * (size_t)N + 2; }
size_t cfbi_chunked_qh_row_floats() { return QP; }
size_t cfbi_chunked_record_bytes() { return (size_t)REC_FLOATS * 4; }

cudaError_t launch_cfbi_prefill_chunked(const CfbiArgs& a, const CfbiWorkspace& w, cudaStream_t st) {
  if (a.in_bf16) return a.out_bf16 ? launch_t<bf16, bf16>(a, w, st) : launch_t<bf16, float>(a, w, st);
  return a.out_bf16 ? launch_t<float, bf16>(a, w, st) : launch_t<float, float>(a, w, st);
}

}  // namespace kda
