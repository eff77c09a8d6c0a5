// Token-sequential prefill on CUDA cores, and the three phases of the segmented (KCP) prefill.
//
// Sources:
// * the per-token update: "Kimi K3: Architecture and SGLang Day-0 Support", KDA math box;
// * snapshots into a ping-pong extra buffer at chunk boundaries: "SGLang and Miles: day-0 support for
//   Kimi K3", "three state movements on the forward stream";
// * segment fragments and their composition: "Kimi K3 training and serving infra" (marsggbo blog),
//   section 4.1 (S_t = M_t S_{t-1} + b_t with M_t = (I - beta k k^T) Diag(alpha)) and section 4.2
//   (per segment: the cumulative transition M and the zero-input state S~; S_in2 = M1 S_in1 + S~1;
//   a prefix scan recovers every entry state, after which the outputs are computed).
//
// Segment fragments use column independence of the update: column c of S evolves with column c of v
// only.  Running the recurrence on the augmented state Z = [S | X] with Z_0 = [0 | I] and values [v | 0]
// gives X_L = M_L ... M_1 = M and S_L = S~ in one pass over the segment.
//
// Each CTA owns a D x DVT column tile of one (sequence or segment, head) and walks its tokens in order;
// the next token's inputs are fetched into registers while the current token is processed.
#include "launch.h"
#include "step.cuh"

namespace kda {

template <int D>
struct SeqCfg;
template <>
struct SeqCfg<128> {
  static constexpr int DVT = 32, NT = 256;
};
template <>
struct SeqCfg<64> {
  static constexpr int DVT = 32, NT = 128;
};
template <>
struct SeqCfg<32> {
  static constexpr int DVT = 32, NT = 64;
};
template <>
struct SeqCfg<16> {
  static constexpr int DVT = 16, NT = 32;
};

enum { MODE_PLAIN = 0, MODE_FRAG = 1, MODE_SEGOUT = 2 };

template <typename T>
__device__ __forceinline__ float ldx(const void* p, size_t i) {
  return to_f32(static_cast<const T*>(p)[i]);
}

template <int D, typename Tin, typename Tout, int MODE>
__global__ void __launch_bounds__(SeqCfg<D>::NT) prefill_seq_kernel(const PrefillArgs a) {
  constexpr int DVT = SeqCfg<D>::DVT, NT = SeqCfg<D>::NT;
  using TL = Tile<D, DVT, NT>;
  constexpr int WIDTH = (MODE == MODE_FRAG) ? 2 * D : D;
  constexpr int NTILES = WIDTH / DVT;
  constexpr bool WANT_O = MODE != MODE_FRAG;
  __shared__ TokenSmem<D, DVT> tok[2];
  __shared__ StepSmem<D, DVT, NT> sm;
  const int tid = threadIdx.x;
  const int tile = blockIdx.x % NTILES, h = blockIdx.x / NTILES;
  const int p = blockIdx.y;
  const int i = blockIdx.z;
  const int col0 = tile * DVT;
  const bool xcols = (MODE == MODE_FRAG) && col0 >= D;

  const int64_t s0 = a.cu[i], s1 = a.cu[i + 1];
  if (s0 < 0 || s1 < s0 || s1 > a.T || s1 - s0 > (int64_t)a.max_seqlen) {
    if (tid == 0) flag_status(a.status, KDA_DEV_SEQ_OOB);
    return;
  }
  int64_t t0 = s0, t1 = s1;
  if (MODE != MODE_PLAIN) {
    t0 = s0 + (int64_t)p * a.seg_len;
    t1 = t0 + a.seg_len < s1 ? t0 + a.seg_len : s1;
    if (MODE == MODE_FRAG) {
      // the last segment's fragment is never used on one GPU (also: segments past the end)
      if (t0 >= s1 || (t1 >= s1 && !a.frag_all)) return;
    } else if (t0 >= s1 && !(p == 0 && s1 == s0)) {
      return;  // past the end; an empty sequence keeps segment 0 to write its final state
    }
  }
  const bool writes_pool = (MODE == MODE_PLAIN) || (MODE == MODE_SEGOUT && t1 == s1);
  const bool reads_pool = (MODE == MODE_PLAIN) && !a.init_zero;
  int slot = 0;
  if (writes_pool || reads_pool) {
    slot = a.slot_ids[i];
    if (slot < 0 || slot >= a.num_slots) {
      if (tid == 0) flag_status(a.status, KDA_DEV_SLOT_OOB);
      return;
    }
  }
  const size_t head_elems = (size_t)D * D;

  float S[TL::ROWS][4];
  if (MODE == MODE_PLAIN) {
    if (a.init_zero)
      zero_tile<D, DVT, NT>(S);
    else
      load_tile<D, DVT, NT>(S, a.pool + ((size_t)slot * a.H + h) * head_elems, D, col0, tid);
  } else if (MODE == MODE_FRAG) {
    const int lane = tid % TL::LANES, rg = tid / TL::LANES;
#pragma unroll
    for (int r = 0; r < TL::ROWS; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) S[r][c] = (xcols && rg * TL::ROWS + r == col0 - D + 4 * lane + c) ? 1.f : 0.f;
  } else {
    load_tile<D, DVT, NT>(S, a.entry + (((size_t)i * a.P + p) * a.H + h) * head_elems, D, col0, tid);
  }

  float rk = 0.f, rq = 0.f, rgv = 0.f, rv = 0.f, rb = 0.f;
  auto fetch = [&](int64_t t) {
    const size_t base = ((size_t)t * a.H + h) * D;
    if (tid < D) {
      rk = ldx<Tin>(a.k, base + tid);
      if (WANT_O) rq = ldx<Tin>(a.q, base + tid);
      rgv = a.g[base + tid];
    }
    if (tid < DVT) rv = xcols ? 0.f : ldx<Tin>(a.v, base + col0 + tid);
    if (tid == 0) rb = a.beta[(size_t)t * a.H + h];
  };
  if (t0 < t1) fetch(t0);
  for (int64_t t = t0; t < t1; ++t) {
    TokenSmem<D, DVT>& tk = tok[(t - t0) & 1];
    if (tid < D) {
      tk.k[tid] = rk;
      tk.q[tid] = rq;
      tk.a[tid] = expf(rgv);
    }
    if (tid < DVT) tk.v[tid] = rv;
    if (tid == 0) tk.beta = rb;
    if (t + 1 < t1) fetch(t + 1);
    __syncthreads();
    const float o = step<D, DVT, NT, WANT_O>(S, tk, sm, tid);
    if (WANT_O) {
      if (tid < DVT) static_cast<Tout*>(a.out)[((size_t)t * a.H + h) * D + col0 + tid] = from_f32<Tout>(o);
      if (a.extra_pool && a.snap_every_tokens > 0) {
        // Snapshot m goes to ping-pong entry (m - 1) & 1.  Only the last two snapshots of a sequence
        // survive the call (an earlier one is overwritten by the snapshot two intervals later), so only
        // those are written: same final extra-pool contents, fewer bytes, and no two concurrent segments
        // ever write the same entry.
        const int64_t pos = t - s0 + 1;
        const int64_t n_snap = (s1 - s0) / a.snap_every_tokens;
        if (pos % a.snap_every_tokens == 0 && pos / a.snap_every_tokens + 1 >= n_snap) {
          const int64_t m = pos / a.snap_every_tokens;
          const int es = a.extra_slots[2 * (size_t)i + ((m - 1) & 1)];
          if (es >= 0 && es < a.num_extra)
            store_tile<D, DVT, NT>(S, a.extra_pool + ((size_t)es * a.H + h) * head_elems, D, col0, tid);
          else if (tid == 0)
            flag_status(a.status, KDA_DEV_SLOT_OOB);
        }
      }
    }
  }
  if (MODE == MODE_FRAG) {
    store_tile<D, DVT, NT>(S, a.frag + (((size_t)i * a.P + p) * a.H + h) * head_elems * 2, 2 * D, col0, tid);
  } else if (writes_pool) {
    store_tile<D, DVT, NT>(S, a.pool + ((size_t)slot * a.H + h) * head_elems, D, col0, tid);
  }
  if (tid == 0 && tile == 0) add_work(a.status, (int32_t)(t1 - t0));
}

// Fragment scan: for each (sequence, head, column tile of the state), sequentially over segments,
// entry_{p+1} = M_p entry_p + S~_p, with entry_0 the initial state.
//
// Only the running entry tile is on the dependent path: M_p and this tile's columns of S~_p do not depend
// on earlier steps, so the next segment's are copied into the other half of a double buffer (cp.async)
// while the current product runs.  Thread (kq, rgp, cgp) holds rows rgp + RGS r (r = 0..3) and columns
// 4 cgp..4 cgp + 3 over the kq-th of KS slices of the contraction; slices 1.. leave partial sums in shared
// memory for slice 0 to add in slice order.  With rows D + 4 floats apart the eight rows a warp reads fall
// in eight bank groups.
template <int D>
struct ScanCfg {
  static constexpr int CT = 16;  // state columns per CTA (D / 16 CTAs per head)
  static constexpr int KS = D >= 64 ? 4 : 1;  // contraction slices: more warps to cover shared-load latency
  static constexpr int RGS = D / 4, CGS = CT / 4, NTS = RGS * CGS, NT = NTS * KS;
  static constexpr int MS = D + 4;  // row stride of the staged M (16-byte aligned rows)
  static constexpr size_t M_FLOATS = (size_t)D * MS, B_FLOATS = (size_t)D * CT;
  // two staged (M, S~ tile) pairs, the running entry tile, the partial sums of slices 1..KS-1
  static constexpr size_t SMEM = sizeof(float) * (2 * (M_FLOATS + B_FLOATS) + B_FLOATS + (KS - 1) * B_FLOATS);
};

__device__ __forceinline__ void scan_cp16(float* dst, const float* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void scan_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void scan_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int D>
__global__ void __launch_bounds__(ScanCfg<D>::NT) seg_scan_kernel(const PrefillArgs a) {
  using C = ScanCfg<D>;
  constexpr int CT = C::CT, MS = C::MS;
  extern __shared__ __align__(16) float smem[];
  float* const Sin = smem + 2 * (C::M_FLOATS + C::B_FLOATS);  // [D][CT]
  const int tid = threadIdx.x;
  const int ct = blockIdx.x % (D / CT), h = blockIdx.x / (D / CT), i = blockIdx.y;
  const size_t head_elems = (size_t)D * D;
  int nseg;
  const float* init = nullptr;  // this head's initial state (null: zero)
  if (a.scan_nseg > 0) {        // fragments gathered from several GPUs: the count and initial state are given
    nseg = a.scan_nseg;
    if (a.scan_s0) init = a.scan_s0 + (size_t)h * head_elems;
  } else {
    const int64_t s0 = a.cu[i], s1 = a.cu[i + 1];
    if (s0 < 0 || s1 < s0 || s1 > a.T || s1 - s0 > (int64_t)a.max_seqlen) {
      if (tid == 0) flag_status(a.status, KDA_DEV_SEQ_OOB);
      return;
    }
    nseg = (int)((s1 - s0 + a.seg_len - 1) / a.seg_len);
    if (a.scan_init) {
      init = a.scan_init + ((size_t)i * a.H + h) * head_elems;
    } else if (!a.init_zero) {
      const int slot = a.slot_ids[i];
      if (slot < 0 || slot >= a.num_slots) {
        if (tid == 0) flag_status(a.status, KDA_DEV_SLOT_OOB);
        return;
      }
      init = a.pool + ((size_t)slot * a.H + h) * head_elems;
    }
  }
  const int c0 = ct * CT;
  float* entry_i = a.entry + (size_t)i * a.P * a.H * head_elems;
  // segment p's M (columns D..2D-1 of its fragment [D][2D]) and S~ columns c0..c0+CT-1 into buffer p & 1
  auto stage = [&](int p) {
    const float* fr = a.frag + (((size_t)i * a.P + p) * a.H + h) * head_elems * 2;
    float* Mb = smem + (p & 1) * (C::M_FLOATS + C::B_FLOATS);
    float* Bb = Mb + C::M_FLOATS;
#pragma unroll 4
    for (int e = tid; e < D * (D / 4); e += C::NT) {
      const int r = e / (D / 4), l4 = e % (D / 4);
      scan_cp16(Mb + r * MS + 4 * l4, fr + (size_t)r * 2 * D + D + 4 * l4);
    }
    for (int e = tid; e < D * (CT / 4); e += C::NT) {
      const int r = e / (CT / 4), q4 = e % (CT / 4);
      scan_cp16(Bb + r * CT + 4 * q4, fr + (size_t)r * 2 * D + c0 + 4 * q4);
    }
    scan_commit();
  };
  if (nseg > 1) stage(0);
  for (int e = tid; e < D * CT; e += C::NT) {
    const int r = e / CT, c = e % CT;
    const float x = init ? init[(size_t)r * D + c0 + c] : 0.f;
    Sin[r * CT + c] = x;
    entry_i[(size_t)h * head_elems + (size_t)r * D + c0 + c] = x;
  }
  float* const Part = Sin + C::B_FLOATS;  // [KS - 1][D][CT]
  const int kq = tid / C::NTS, rgp = (tid % C::NTS) / C::CGS, cgp = tid % C::CGS;
  constexpr int LK = D / C::KS;
  for (int p = 0; p + 1 < nseg; ++p) {
    if (p + 2 < nseg) {
      stage(p + 1);  // buffer (p + 1) & 1 was last read in step p - 1, before its closing barrier
      scan_wait<1>();
    } else {
      scan_wait<0>();
    }
    __syncthreads();  // staged buffer p & 1 and the entry tile visible to all threads
    const float* Mb = smem + (p & 1) * (C::M_FLOATS + C::B_FLOATS);
    const float* Bb = Mb + C::M_FLOATS;
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float4 x = kq == 0 ? *reinterpret_cast<const float4*>(Bb + (rgp + C::RGS * r) * CT + 4 * cgp)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
      acc[r][0] = x.x;
      acc[r][1] = x.y;
      acc[r][2] = x.z;
      acc[r][3] = x.w;
    }
#pragma unroll 4
    for (int l = kq * LK; l < (kq + 1) * LK; ++l) {
      const float4 s4 = *reinterpret_cast<const float4*>(&Sin[l * CT + 4 * cgp]);
      const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float m = Mb[(rgp + C::RGS * r) * MS + l];
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = __fmaf_rn(m, sv[c], acc[r][c]);
      }
    }
    if (kq > 0) {
#pragma unroll
      for (int r = 0; r < 4; ++r)
        *reinterpret_cast<float4*>(Part + (kq - 1) * C::B_FLOATS + (rgp + C::RGS * r) * CT + 4 * cgp) =
            make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    }
    __syncthreads();  // all reads of the entry tile and of buffer p & 1 done; partial sums visible
    if (kq > 0) continue;
    float* dst = entry_i + ((size_t)(p + 1) * a.H + h) * head_elems;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = rgp + C::RGS * r;
#pragma unroll
      for (int k = 1; k < C::KS; ++k) {
        const float4 y = *reinterpret_cast<const float4*>(Part + (k - 1) * C::B_FLOATS + row * CT + 4 * cgp);
        acc[r][0] = __fadd_rn(acc[r][0], y.x);
        acc[r][1] = __fadd_rn(acc[r][1], y.y);
        acc[r][2] = __fadd_rn(acc[r][2], y.z);
        acc[r][3] = __fadd_rn(acc[r][3], y.w);
      }
      const float4 x = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
      *reinterpret_cast<float4*>(&Sin[row * CT + 4 * cgp]) = x;
      *reinterpret_cast<float4*>(dst + (size_t)row * D + c0 + 4 * cgp) = x;
    }
  }
}

// ---------------------------------------------------------------- launchers

template <int D, typename Tin, typename Tout, int MODE>
static cudaError_t launch_seq_t(const PrefillArgs& a, cudaStream_t s) {
  constexpr int WIDTH = (MODE == MODE_FRAG) ? 2 * D : D;
  constexpr int NTILES = WIDTH / SeqCfg<D>::DVT;
  dim3 grid(NTILES * a.H, MODE == MODE_PLAIN ? 1 : a.P, a.N);
  prefill_seq_kernel<D, Tin, Tout, MODE><<<grid, SeqCfg<D>::NT, 0, s>>>(a);
  return cudaGetLastError();
}

template <int MODE, typename Tin, typename Tout>
static cudaError_t seq_d(const PrefillArgs& a, cudaStream_t s) {
  switch (a.d) {
    case 16: return launch_seq_t<16, Tin, Tout, MODE>(a, s);
    case 32: return launch_seq_t<32, Tin, Tout, MODE>(a, s);
    case 64: return launch_seq_t<64, Tin, Tout, MODE>(a, s);
    case 128: return launch_seq_t<128, Tin, Tout, MODE>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int MODE>
static cudaError_t seq_dispatch(const PrefillArgs& a, cudaStream_t s) {
  if (a.in_bf16) return a.out_bf16 ? seq_d<MODE, bf16, bf16>(a, s) : seq_d<MODE, bf16, float>(a, s);
  return a.out_bf16 ? seq_d<MODE, float, bf16>(a, s) : seq_d<MODE, float, float>(a, s);
}

cudaError_t launch_prefill_seq(const PrefillArgs& a, cudaStream_t s) { return seq_dispatch<MODE_PLAIN>(a, s); }

cudaError_t launch_seg_fragments(const PrefillArgs& a, cudaStream_t s) {
  // fragments never write outputs: instantiate with a single output type
  if (a.in_bf16) {
    switch (a.d) {
      case 16: return launch_seq_t<16, bf16, float, MODE_FRAG>(a, s);
      case 32: return launch_seq_t<32, bf16, float, MODE_FRAG>(a, s);
      case 64: return launch_seq_t<64, bf16, float, MODE_FRAG>(a, s);
      case 128: return launch_seq_t<128, bf16, float, MODE_FRAG>(a, s);
    }
  } else {
    switch (a.d) {
      case 16: return launch_seq_t<16, float, float, MODE_FRAG>(a, s);
      case 32: return launch_seq_t<32, float, float, MODE_FRAG>(a, s);
      case 64: return launch_seq_t<64, float, float, MODE_FRAG>(a, s);
      case 128: return launch_seq_t<128, float, float, MODE_FRAG>(a, s);
    }
  }
  return cudaErrorInvalidValue;
}

template <int D>
static cudaError_t launch_scan_t(const PrefillArgs& a, cudaStream_t s) {
  using C = ScanCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(seg_scan_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((D / C::CT) * a.H, a.N);
  seg_scan_kernel<D><<<grid, C::NT, C::SMEM, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_seg_scan(const PrefillArgs& a, cudaStream_t s) {
  switch (a.d) {
    case 16: return launch_scan_t<16>(a, s);
    case 32: return launch_scan_t<32>(a, s);
    case 64: return launch_scan_t<64>(a, s);
    case 128: return launch_seg_scan_tc(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_seg_outputs(const PrefillArgs& a, cudaStream_t s) { return seq_dispatch<MODE_SEGOUT>(a, s); }

}  // namespace kda
