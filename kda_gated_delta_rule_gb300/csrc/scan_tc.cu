// Fragment scan on the tensor cores (dk = dv = 128): for each (sequence, head, 16-column tile of the state),
// sequentially over segments, entry_{p+1} = M_p entry_p + S~_p, with entry_0 the initial state.
//
// Source: "Kimi K3 training and serving infra" (marsggbo blog), section 4.2 (the fragments (M, S~) of
// consecutive segments compose as S_in2 = M1 S_in1 + S~1; a prefix scan over them gives every segment's
// entry state, after which the outputs are computed).
//
// One step is the product of M_p [128 x 128] and the running entry tile [128 x 16]: a tcgen05 MMA with
// M = 128 (rows i of the state), N = 16 (the tile's columns), K = 128, both operands split into bf16
// hi + lo and multiplied as hi*hi + hi*lo + lo*hi into an fp32 accumulator in tensor memory.  Only the
// entry tile is on the dependent path: M_{p+1} is fetched and split while step p runs.  M is the A operand
// in tensor memory, so each MMA reads only the small B tile from shared memory.
//   warps 0-7 (two threads per tensor-memory lane = row i, 8 columns each): the accumulator + S~_p ->
//             entry_{p+1} (global) and the B operand of the next step (the tile transposed, K-major); lane 0
//             of warps 0-2 issues one of the three split products each, into an accumulator of its own
//             (summed in the epilogue);
//   warps 8-23: M_{p+1}'s rows -> a shared staging buffer (coalesced cp.async, issued a step ahead) ->
//             four threads per row i split its 128 values and store them (bf16 pairs, hi then lo) into the
//             half of a tensor-memory double buffer that step p does not read.
#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace kda {
namespace {

constexpr int SD = 128;      // dk = dv
constexpr int SCT = 16;      // state columns per CTA
constexpr int SCAN_EPI = 256;                 // epilogue threads (warps 0-7): two per row of the tile
constexpr int EC = SCT / (SCAN_EPI / 128);    // tile columns per epilogue thread
constexpr int N_STAGE = 512;                  // staging threads (warps 8-23): four per row of M
constexpr int SK = 128 / (N_STAGE / 128);     // values of a row of M per staging thread
constexpr int SCAN_NT = SCAN_EPI + N_STAGE;
constexpr uint32_t SC_B = 0;            // B operand: hi (two 2 KB K-blocks of 16 rows), then lo at + 4 KB
constexpr uint32_t SC_STAGE = 8192;     // two buffers of M rows, fp32, 528 bytes apart (conflict-free row reads)
constexpr uint32_t SC_ROW = 528;
constexpr uint32_t SC_STAGE_BYTES = 128 * SC_ROW;
constexpr uint32_t SC_BAR = SC_STAGE + 2 * SC_STAGE_BYTES;  // the MMA completion barrier
constexpr uint32_t SC_SLOT = SC_BAR + 8;
constexpr uint32_t SC_BYTES = SC_BAR + 16 + 1024;
// tensor memory columns (512 allocated): the accumulator, then two A operands of 128 columns each
// (M_p row i in lane i: 64 columns of bf16 pairs hi, then 64 lo)
constexpr uint32_t COL_D = 0;  // three partial products of 16 columns each
constexpr uint32_t COL_A = 128;
constexpr int BAR_STAGE = 1;  // named barrier of the staging warps

__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
// tensor memory -> registers, 8 columns of this warp's 32 lanes, without waiting
__device__ __forceinline__ void tmem_ld8_async(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

__device__ __forceinline__ uint8_t* align_1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}


__global__ void __launch_bounds__(SCAN_NT, 1) seg_scan_tc_kernel(const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align_1k(smem_raw);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + SC_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SC_SLOT);
  const int tid = threadIdx.x, warp = tid >> 5;
  tc::pdl_wait();  // the previous kernel in the stream (the fragments) is done
  tc::pdl_launch_dependents();
  const int ct = blockIdx.x % (SD / SCT), h = blockIdx.x / (SD / SCT), i = blockIdx.y;
  const size_t head_elems = (size_t)SD * SD;
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
        if (!a.zero_bad_slot) return;
      } else {
        init = a.pool + ((size_t)slot * a.H + h) * head_elems;
      }
    }
  }
  const int c0 = ct * SCT;
  uint32_t tm = 0;  // tensor memory base (allocated below)
  float* entry_i = a.entry + (size_t)i * a.P * a.H * head_elems;
  auto frag_of = [&](int p) { return a.frag + (((size_t)i * a.P + p) * a.H + h) * head_elems * 2; };  // [D][2D]
  // epilogue thread: row erow of the tile, columns ce .. ce + EC - 1 (of the tile)
  const int erow = tid & 127, ce = EC * ((tid >> 7) & 1);
  // epilogue: this thread's part of a row of a tile -> entry p (global)
  auto store_entry = [&](int p, int row, const float* x) {
    float4* dst =
        reinterpret_cast<float4*>(entry_i + ((size_t)p * a.H + h) * head_elems + (size_t)row * SD + c0 + ce);
#pragma unroll
    for (int q = 0; q < EC / 4; ++q) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
  };
  // epilogue: row `row` of the entry tile is column k = row of the B operand (rows n = tile columns).  Lanes
  // 2m and 2m + 1 hold rows k, k + 1 of the same columns: one shuffle per column pairs them, so every store
  // is a 32-bit word (k even, k + 1): the even lane writes the first EC/2 columns, the odd lane the rest.
  auto store_b = [&](int row, const float* x) {
    uint8_t* bh = sm + SC_B + (row >> 6) * 2048;
    const bool odd = row & 1;
    const int k = row & 62;
#pragma unroll
    for (int j = 0; j < EC / 2; ++j) {
      const float mine = odd ? x[EC / 2 + j] : x[j];
      const float other = __shfl_xor_sync(0xffffffffu, odd ? x[j] : x[EC / 2 + j], 1);
      uint32_t hi, lo;
      tc::split_pair(odd ? other : mine, odd ? mine : other, hi, lo);  // (row k, row k + 1)
      const uint32_t o = tc::sw128(ce + (odd ? EC / 2 : 0) + j, k);
      *reinterpret_cast<uint32_t*>(bh + o) = hi;
      *reinterpret_cast<uint32_t*>(bh + 4096 + o) = lo;
    }
  };
  // epilogue: this tile's columns of S~_p, row `row`
  auto load_stilde = [&](int p, int row, float* x) {
    const float4* src = reinterpret_cast<const float4*>(frag_of(p) + (size_t)row * 2 * SD + c0 + ce);
#pragma unroll
    for (int q = 0; q < EC / 4; ++q) {
      const float4 v = src[q];
      x[4 * q] = v.x, x[4 * q + 1] = v.y, x[4 * q + 2] = v.z, x[4 * q + 3] = v.w;
    }
  };
  // staging thread: row srow = stid % 128 of M, values SK sq .. SK sq + SK - 1 of it
  const int stid = tid - SCAN_EPI, srow = stid & 127, sq = stid >> 7;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  // M_p (columns D..2D-1 of its fragment) into the staging buffer: consecutive threads, consecutive 16 bytes
  auto fetch = [&](int p) {
    const float* fr = frag_of(p) + SD;
#pragma unroll 4
    for (int e = stid; e < SD * (SD / 4); e += N_STAGE) {
      const int r = e >> 5, l4 = e & 31;
      cp16(sm + SC_STAGE + (uint32_t)(p & 1) * SC_STAGE_BYTES + r * SC_ROW + l4 * 16, fr + (size_t)r * 2 * SD + 4 * l4);
    }
    cp_commit();
  };
  // the staged M_p -> A operand p & 1; then the staging buffer is free for M_{p+1} (fetched if `next`)
  // (M_{p+1}, if `next`, goes into the other staging buffer first: it has a whole step to land)
  auto stage = [&](int p, bool next) {
    if (next) {
      tc::named_bar(BAR_STAGE, N_STAGE);  // buffer (p + 1) & 1 was last read in stage p - 1
      fetch(p + 1);
      cp_wait_one();
    } else {
      cp_wait_all();
    }
    tc::named_bar(BAR_STAGE, N_STAGE);  // M_p landed, every thread's copies
    const float4* src =
        reinterpret_cast<const float4*>(sm + SC_STAGE + (uint32_t)(p & 1) * SC_STAGE_BYTES + srow * SC_ROW + 4 * SK * sq);
    float4 x[SK / 4];
#pragma unroll
    for (int q = 0; q < SK / 4; ++q) x[q] = src[q];
    uint32_t hi[SK / 2], lo[SK / 2];
#pragma unroll
    for (int q = 0; q < SK / 4; ++q) {
      tc::split_pair(x[q].x, x[q].y, hi[2 * q], lo[2 * q]);
      tc::split_pair(x[q].z, x[q].w, hi[2 * q + 1], lo[2 * q + 1]);
    }
    static_assert(SK == 32, "one 16-column store of hi and of lo per staging thread");
    const uint32_t col = COL_A + (uint32_t)(p & 1) * 128u + (uint32_t)(SK / 2) * (uint32_t)sq;
    tc::tmem_st16(tm + lane_base + col, hi);
    tc::tmem_st16(tm + lane_base + col + 64, lo);
    tc::tmem_wait_st();
  };

  // entry_0 = the initial state; with a single segment nothing else is needed
  float sv[EC];  // epilogue: this thread's part of its row of S~_p
  if (tid < SCAN_EPI) {
    float x[EC];
#pragma unroll
    for (int q = 0; q < EC / 4; ++q) {
      const float4 v = init ? *reinterpret_cast<const float4*>(init + (size_t)erow * SD + c0 + ce + 4 * q)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      x[4 * q] = v.x, x[4 * q + 1] = v.y, x[4 * q + 2] = v.z, x[4 * q + 3] = v.w;
    }
    store_entry(0, erow, x);
    if (nseg > 1) {
      store_b(erow, x);
      load_stilde(0, erow, sv);
    }
  }
  if (nseg <= 1) return;

  if (warp == 0) tc::tmem_alloc(tslot, 512);
  if (tid == 0) {
    tc::bar_init(mbar, 3);
    tc::bar_fence_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  tm = *tslot;
  if (tid >= SCAN_EPI) {
    fetch(0);
    stage(0, nseg > 2);
  }
  tc::fence_proxy_async();  // the B operand writes (epilogue), visible to the tensor core
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t base = tc::smem_u32(sm);
  constexpr uint32_t IDESC = tc::idesc_bf16(128, SCT);
  bool ok = true;
#pragma unroll 1
  for (int p = 0; p + 1 < nseg; ++p) {
    if (tid < 96 && (tid & 31) == 0) {  // M_p entry_p: (hi, hi), (hi, lo), (lo, hi), one issuer and accumulator each
      tc::fence_after_sync();
      const int part = tid >> 5;
      const uint32_t xa = tm + COL_A + (uint32_t)(p & 1) * 128u + (part == 2 ? 64u : 0u);
      const uint32_t xb = base + SC_B + (part == 1 ? 4096u : 0u);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        tc::mma_ts(tm + COL_D + 16u * part, xa + 8u * ks,
                   tc::sdesc(xb + (uint32_t)(ks >> 2) * 2048u + (uint32_t)(ks & 3) * 32u), IDESC, ks != 0);
      tc::commit(mbar);
    }
    if (tid < SCAN_EPI) {
      ok = __all_sync(0xffffffffu, tc::bar_wait(mbar, (uint32_t)p & 1u));
      tc::fence_after_sync();
      if (ok) {
        static_assert(EC == 8, "one 8-column load per partial product");
        uint32_t r0[EC], r1[EC], r2[EC];
        tmem_ld8_async(tm + lane_base + COL_D + ce, r0);
        tmem_ld8_async(tm + lane_base + COL_D + 16 + ce, r1);
        tmem_ld8_async(tm + lane_base + COL_D + 32 + ce, r2);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        tc::fence_before_sync();  // this thread's last tensor-memory access of the step
        float d[EC];
#pragma unroll
        for (int c = 0; c < EC; ++c)
          d[c] = __fadd_rn(__fadd_rn(__fadd_rn(__uint_as_float(r0[c]), __uint_as_float(r1[c])), __uint_as_float(r2[c])),
                           sv[c]);
        if (p + 2 < nseg) store_b(erow, d);
        tc::fence_proxy_async();  // the B operand, visible to the tensor core (before the global traffic)
        store_entry(p + 1, erow, d);
        if (p + 2 < nseg) load_stilde(p + 1, erow, sv);
      }
    } else if (p + 2 < nseg) {  // M_{p+1} into the A operand that step p does not read
      tc::fence_after_sync();
      stage(p + 1, p + 3 < nseg);
      tc::fence_before_sync();
    }
    // (tensor-core fences only where a thread orders its own tensor-memory work against the barrier: they
    // wait for the thread's global accesses in flight, so the epilogue takes them before its global traffic)
    ok = __syncthreads_and(ok);
    if (!ok) break;
  }
  if (tid >= SCAN_EPI) cp_wait_all();  // no copy into this CTA's shared memory outlives it
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tm, 512);
  if (!ok && tid == 0) flag_status(a.status, KDA_DEV_TIMEOUT);
}

}  // namespace

cudaError_t launch_seg_scan_tc(const PrefillArgs& a, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(seg_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SC_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid((SD / SCT) * a.H, a.N);
  return launch_pdl(seg_scan_tc_kernel, grid, dim3(SCAN_NT), SC_BYTES, s, a);
}

}  // namespace kda
