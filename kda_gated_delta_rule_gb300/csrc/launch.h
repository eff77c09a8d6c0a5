// Internal launch interface between the C ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

// Raw-input record of a draft window (see kda_replay_bytes in include/kda.h).
struct ReplayPtrs {
  void* k;      // [B][W][H][dk] in dtype
  void* v;      // [B][W][H][dv] in dtype
  float* g;     // [B][W][H][dk]
  float* beta;  // [B][W][H]
};

struct DecodeArgs {
  const void *q, *k, *v;
  const float *g, *beta;
  int B, H, d;
  bool in_bf16, out_bf16;
  float* pool;
  int num_slots;
  const int32_t* slot_ids;
  void* out;
  int32_t* status;
};

struct VerifyArgs {
  const void *q, *k, *v;
  const float *g, *beta;
  int B, W, H, d;
  bool in_bf16, out_bf16;
  const float* pool;
  int num_slots;
  const int32_t* slot_ids;
  void* out;
  ReplayPtrs rec;
  float* snapshot_out;
  int32_t* status;
};

struct FoldArgs {
  float* pool;
  int num_slots;
  const int32_t* slot_ids;
  int B, W, H, d;
  bool in_bf16;
  ReplayPtrs rec;
  const int32_t* accepted;
  int32_t* status;
};

struct CopyArgs {
  const float* src;
  int src_num_slots;
  const int32_t* src_slots;
  float* dst;
  int dst_num_slots;
  const int32_t* dst_slots;
  int n;
  int64_t state_elems;
  int32_t* status;
};

// Prefill over packed sequences; also drives the three phases of the segmented (KCP) path.
struct PrefillArgs {
  const void *q, *k, *v;
  const float *g, *beta;
  bool in_bf16, out_bf16;
  int64_t T;
  int H, d, N;
  const int32_t* cu;
  int max_seqlen;
  float* pool;
  int num_slots;
  const int32_t* slot_ids;
  bool init_zero;
  void* out;
  float* extra_pool;
  int num_extra;
  const int32_t* extra_slots;
  int snap_every_tokens;  // 0 = no snapshots
  int32_t* status;
  // segmented path
  int seg_len;  // tokens per segment (multiple of 64)
  int P;        // segments per sequence = ceil(max_seqlen / seg_len)
  float* frag;  // [N][P][H][d][2d]
  float* entry; // [N][P][H][d][d]
  // tensor-core path: per (chunk, head) operand records written by the prep kernel
  uint8_t* records;
  // sequence split across GPUs (KCP between ranks): fragments also for the last segment of each sequence;
  // a scan over scan_nseg given fragments (N = 1, no cu_seqlens) from scan_s0 [H][d][d] (null: zero)
  bool frag_all;
  int scan_nseg;
  const float* scan_s0;
  // test hook (kda_set_test_fault): the prep kernel issues no input copies and waits for them with a short
  // poll limit, so its first wait gives up and the kernel reports KDA_DEV_TIMEOUT; 0 in normal calls
  int test_stall_inputs;
  // the backward's forward pass (launch_tc_chain_states): every chunk's entry state and U into the
  // backward's per-(chunk, head) records (bw_rec_floats floats each, indexed like the backward's: chunk
  // starting at token t0 of sequence i -> (t0 / 64 + i) * H + h), at float offsets bw_off_h / bw_off_u
  float* bw_ws;
  int bw_rec_floats, bw_off_h, bw_off_u;
  bool no_work_count;  // the chain adds nothing to the work counter (a pass inside another call)
  bool zero_bad_slot;  // the scan starts a sequence whose slot id is out of range from zero (flagged)
  // the scan starts sequence i from scan_init + i * H * d * d (per head: + h * d * d) instead of the pool
  // (null: not used)
  const float* scan_init;
  // the backward's reverse pass (launch_tc_rev_frag / launch_tc_rev_pass): upstream gradients dL/do
  // [T][H][d] bf16, dL/dS_T [N][H][d][d] (null: zero) and dL/dS_0 out [N][H][d][d] (null: not written);
  // every chunk's exit gradient dS' and dU go to the backward's records at float offsets bw_off_ds /
  // bw_off_du
  const void* d_out;
  const float* d_final;
  float* d_init;
  int bw_off_ds, bw_off_du;
};

// Batch-invariant (CF-BI) prefill and decode (d = 128).
struct CfbiArgs {
  const void *q, *k, *v;
  const float *g, *beta;
  int B;                // decode: requests
  int N;                // prefill: sequences
  int64_t T;            // prefill: packed tokens
  int max_seqlen;       // prefill
  const int32_t* cu;    // prefill: cu_seqlens[N + 1]
  int H;
  bool in_bf16, out_bf16;
  float* pool;
  float* cache;
  int32_t* counts;
  int num_slots;
  const int32_t* slot_ids;
  void* out;
  int32_t* status;
};

// Workspace of the chunk-parallel CF-BI prefill (layout in cfbi_chunked.cu).
struct CfbiWorkspace {
  float* qh;       // [H][T][cfbi_chunked_qh_row_floats()]
  float* oh;       // [H][T][128] (by 8-column group)
  float* rows;     // [cfbi_chunked_records(T, N)][H] records of cfbi_chunked_record_bytes()
  int32_t* count;  // [N][H]
};
size_t cfbi_chunked_records(int64_t T, int N);
size_t cfbi_chunked_record_bytes();
size_t cfbi_chunked_qh_row_floats();
cudaError_t launch_cfbi_prefill_chunked(const CfbiArgs& a, const CfbiWorkspace& w, cudaStream_t s);

// Chunked backward (d = 128): gradients of sum <d_out, o> + <d_final, S_T> through a packed prefill.
struct BackwardArgs {
  const void *q, *k, *v;
  const float *g, *beta;
  bool in_bf16;
  int64_t T;
  int H, N;
  const int32_t* cu;
  int max_seqlen;
  const float* pool;
  int num_slots;
  const int32_t* slot_ids;
  bool init_zero;
  const void* d_out;     // [T][H][128] in dtype
  const float* d_final;  // [N][H][128][128] or null
  float *dq, *dk, *dv, *dg, *dbeta;
  float* d_init;         // [N][H][128][128] or null
  float* ws;             // backward_ws_bytes(T, N, H)
  int32_t* status;
  // set by the launcher on the tensor-core forward pass: per (sequence, head), nonzero when a 16-token block
  // of some chunk spans more decay than the block references allow (g below the pages' floor); the
  // CUDA-core chain then recomputes that (sequence, head)'s entry states and U
  int32_t* steep;
};

size_t backward_ws_bytes(int64_t T, int N, int H);

// Fused decode: short convolution + KDA step + gated output norm (d = 128).
struct FusedDecodeArgs {
  const void *xq, *xk, *xv;  // [B][H][128] pre-convolution projections
  const float* a;            // [B][H][128] decay logits
  const float* b;            // [B][H] write-strength logits
  const void* z;             // [B][H][128] output-gate logits
  bool in_bf16, out_bf16;
  int B, H;
  float* pool;
  int num_slots;
  const int32_t* slot_ids;
  float* conv_state;         // [num_slots][H][3][3][128]
  const float* conv_w;       // [3][H][128][4]
  const float* norm_w;       // [128]
  float eps;
  void* out;
  int32_t* status;
};

cudaError_t launch_fused_decode(const FusedDecodeArgs& a, cudaStream_t s);
cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s);

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s);
// Tensor-core verify (bf16 inputs, d = 128, W <= 16, no per-token snapshots).
bool verify_tc_supported(const VerifyArgs& a);
cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t s);
cudaError_t launch_fold(const FoldArgs& a, cudaStream_t s);
cudaError_t launch_cfbi_prefill(const CfbiArgs& a, cudaStream_t s);
cudaError_t launch_cfbi_decode(const CfbiArgs& a, cudaStream_t s);
cudaError_t launch_state_copy(const CopyArgs& a, cudaStream_t s);

// Sequential (token-by-token, CUDA-core) prefill; mode 0 = whole sequences.
cudaError_t launch_prefill_seq(const PrefillArgs& a, cudaStream_t s);
// Segmented path phases.
cudaError_t launch_seg_fragments(const PrefillArgs& a, cudaStream_t s);
cudaError_t launch_seg_scan(const PrefillArgs& a, cudaStream_t s);
// the same scan on the tensor cores (d = 128)
cudaError_t launch_seg_scan_tc(const PrefillArgs& a, cudaStream_t s);
cudaError_t launch_seg_outputs(const PrefillArgs& a, cudaStream_t s);

// Tensor-core chunked path (bf16 inputs, d = 128).
bool tc_supported(const PrefillArgs& a);
size_t tc_record_bytes(int64_t T, int N, int H);
cudaError_t launch_tc_prep(const PrefillArgs& a, uint8_t* records, cudaStream_t s);
cudaError_t launch_tc_chain_plain(const PrefillArgs& a, const uint8_t* records, cudaStream_t s);
cudaError_t launch_tc_chain_frag(const PrefillArgs& a, const uint8_t* records, cudaStream_t s);
// the backward's forward pass: like the segment outputs, but every chunk's entry state and U go to the
// backward's records (a.bw_*) instead of outputs, and the pool is not written
cudaError_t launch_tc_chain_states(const PrefillArgs& a, const uint8_t* records, cudaStream_t s);
cudaError_t launch_tc_chain_segout(const PrefillArgs& a, const uint8_t* records, cudaStream_t s);
// the backward's reverse pass over the same records: per-segment affine maps of the state gradient (stored
// in reverse segment order, for launch_seg_scan from d_final via scan_init), then every segment from its
// exit gradient, writing each chunk's dS' and dU (a.bw_*) and dL/dS_0
cudaError_t launch_tc_rev_frag(const PrefillArgs& a, const uint8_t* records, cudaStream_t s);
cudaError_t launch_tc_rev_pass(const PrefillArgs& a, const uint8_t* records, cudaStream_t s);

// Launches `kernel` so that it may be scheduled while the previous kernel in the stream finishes
// (programmatic dependent launch).  The kernel must call griddepcontrol.wait before it touches global
// memory, and trigger its own dependents only after that.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace kda
