// C ABI of the KDA library: host-side validation, workspace sizing and dispatch to the kernels.
// The declarations, argument meaning, layouts and error behaviour are documented in include/kda.h.
#include <stdint.h>

#include "../../include/kda.h"
#include "debug_checks.h"
#include "launch.h"

namespace {

constexpr int kVersion = 1 * 10000 + 0 * 100 + 0;

int g_test_fault = KDA_TEST_FAULT_NONE;  // kda_set_test_fault

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dtype_ok(kda_dtype t) { return t == KDA_DTYPE_F32 || t == KDA_DTYPE_BF16; }
bool head_ok(int dk, int dv) { return dk == dv && (dk == 16 || dk == 32 || dk == 64 || dk == 128); }
size_t esize(kda_dtype t) { return t == KDA_DTYPE_BF16 ? 2 : 4; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

kda_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

struct ReplayLayout {
  size_t off_k, off_v, off_g, off_beta, total;
};

ReplayLayout replay_layout(int B, int W, int H, int dk, int dv, kda_dtype t) {
  const size_t rows = (size_t)B * W * H;
  ReplayLayout L;
  L.off_k = 0;
  L.off_v = L.off_k + align256(rows * dk * esize(t));
  L.off_g = L.off_v + align256(rows * dv * esize(t));
  L.off_beta = L.off_g + align256(rows * dk * 4);
  L.total = L.off_beta + align256(rows * 4);
  return L;
}

kda::ReplayPtrs replay_ptrs(void* base, const ReplayLayout& L) {
  char* b = static_cast<char*>(base);
  return kda::ReplayPtrs{b + L.off_k, b + L.off_v, reinterpret_cast<float*>(b + L.off_g),
                         reinterpret_cast<float*>(b + L.off_beta)};
}

// Validates the parts of a prefill call shared by the plain and segmented paths.
kda_status check_prefill(const kda_prefill_args* a) {
  if (!a) return KDA_ERR_INVALID_ARG;
  if (!dtype_ok(a->in_dtype) || !dtype_ok(a->out_dtype)) return KDA_ERR_INVALID_ARG;
  if (a->H <= 0 || a->N < 0 || a->T < 0 || a->max_seqlen < 0 || a->num_slots < 0) return KDA_ERR_INVALID_ARG;
  if (!head_ok(a->dk, a->dv)) return KDA_ERR_UNSUPPORTED;
  if (a->N > 65535) return KDA_ERR_INVALID_ARG;
  if (!a->cu_seqlens || !a->pool || !a->slot_ids) return KDA_ERR_INVALID_ARG;
  if (!aligned16(a->pool) || !aligned16(a->cu_seqlens) || !aligned16(a->slot_ids)) return KDA_ERR_INVALID_ARG;
  if (a->T > 0) {
    if (!a->q || !a->k || !a->v || !a->g || !a->beta || !a->out) return KDA_ERR_INVALID_ARG;
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->g) || !aligned16(a->beta) ||
        !aligned16(a->out))
      return KDA_ERR_INVALID_ARG;
  }
  if (a->extra_pool) {
    if (a->snapshot_every_chunks < 0 || a->num_extra_slots < 0 || !a->extra_slot_ids) return KDA_ERR_INVALID_ARG;
    if (!aligned16(a->extra_pool)) return KDA_ERR_INVALID_ARG;
    if ((int64_t)a->snapshot_every_chunks * 64 > 0x7fffffff) return KDA_ERR_INVALID_ARG;
  }
  return KDA_OK;
}

kda::PrefillArgs to_internal(const kda_prefill_args* a) {
  kda::PrefillArgs p{};
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.g = a->g;
  p.beta = a->beta;
  p.in_bf16 = a->in_dtype == KDA_DTYPE_BF16;
  p.out_bf16 = a->out_dtype == KDA_DTYPE_BF16;
  p.T = a->T;
  p.H = a->H;
  p.d = a->dk;
  p.N = a->N;
  p.cu = a->cu_seqlens;
  p.max_seqlen = a->max_seqlen;
  p.pool = a->pool;
  p.num_slots = a->num_slots;
  p.slot_ids = a->slot_ids;
  p.init_zero = a->init_zero != 0;
  p.out = a->out;
  p.extra_pool = (a->extra_pool && a->snapshot_every_chunks > 0) ? a->extra_pool : nullptr;
  p.num_extra = a->num_extra_slots;
  p.extra_slots = a->extra_slot_ids;
  p.snap_every_tokens = p.extra_pool ? a->snapshot_every_chunks * 64 : 0;
  p.status = a->dev_status;
  return p;
}

// The tensor-core chunked path serves bf16 inputs at dk = dv = 128; everything else runs the
// token-sequential CUDA-core path.
bool use_tc(const kda_prefill_args* a) { return a->in_dtype == KDA_DTYPE_BF16 && a->dk == 128 && a->dv == 128; }

size_t align1024(size_t x) { return (x + 1023) & ~size_t(1023); }

// Per (chunk, head) operand records of the tensor-core path (0 for the CUDA-core path).
size_t record_bytes(const kda_prefill_args* a) {
  return use_tc(a) ? align1024(kda::tc_record_bytes(a->T, a->N, a->H)) : 0;
}

struct SegLayout {
  int P;
  size_t rec_bytes, frag_bytes, entry_bytes, total;
};

// Segmented workspace: [records][frag][entry].
SegLayout seg_layout(const kda_prefill_args* a, int32_t seg_len) {
  SegLayout L{};
  L.P = a->max_seqlen > 0 ? (int)((a->max_seqlen + (int64_t)seg_len - 1) / seg_len) : 1;
  const size_t heads = (size_t)a->N * L.P * a->H;
  L.rec_bytes = record_bytes(a);
  L.frag_bytes = align256(heads * a->dk * (size_t)(a->dv + a->dk) * 4);
  L.entry_bytes = align256(heads * a->dk * (size_t)a->dv * 4);
  L.total = L.rec_bytes + L.frag_bytes + L.entry_bytes;
  return L;
}

kda_status seg_prepare(const kda_prefill_args* a, int32_t seg_len, kda::PrefillArgs* p) {
  kda_status st = check_prefill(a);
  if (st != KDA_OK) return st;
  if (seg_len <= 0 || seg_len % 64 != 0) return KDA_ERR_INVALID_ARG;
  const SegLayout L = seg_layout(a, seg_len);
  if (L.P > 65535) return KDA_ERR_INVALID_ARG;
  if (!a->workspace || a->workspace_bytes < L.total) return KDA_ERR_WORKSPACE;
  if (!aligned16(a->workspace)) return KDA_ERR_INVALID_ARG;
  *p = to_internal(a);
  p->seg_len = seg_len;
  p->P = L.P;
  char* w = static_cast<char*>(a->workspace);
  p->records = L.rec_bytes ? reinterpret_cast<uint8_t*>(w) : nullptr;
  p->frag = reinterpret_cast<float*>(w + L.rec_bytes);
  p->entry = reinterpret_cast<float*>(w + L.rec_bytes + L.frag_bytes);
  return KDA_OK;
}

cudaError_t run_fragments(const kda::PrefillArgs& p, cudaStream_t s) {
  return p.records ? kda::launch_tc_chain_frag(p, p.records, s) : kda::launch_seg_fragments(p, s);
}

// Validates a varlen call's workspace for the tensor-core path and fills p.records (nullptr if none needed).
kda_status varlen_prepare(const kda_prefill_args* a, kda::PrefillArgs* p) {
  kda_status st = check_prefill(a);
  if (st != KDA_OK) return st;
  *p = to_internal(a);
  const size_t need = record_bytes(a);
  if (need == 0) return KDA_OK;
  if (!a->workspace || a->workspace_bytes < need) return KDA_ERR_WORKSPACE;
  if (!aligned16(a->workspace)) return KDA_ERR_INVALID_ARG;
  p->records = static_cast<uint8_t*>(a->workspace);
  return KDA_OK;
}

// Debug mode: sequences own distinct slots, snapshots go to distinct extra slots, and (one pool for both)
// no snapshot lands in a slot a sequence reads or writes.
kda_status prefill_debug_check(const kda_prefill_args* a, cudaStream_t s) {
  kda_status st = kda::debug_check_slots(a->slot_ids, a->N, nullptr, 0, s);
  if (st != KDA_OK || !a->extra_pool || a->snapshot_every_chunks <= 0) return st;
  st = kda::debug_check_slots(a->extra_slot_ids, 2 * a->N, nullptr, 0, s);
  if (st != KDA_OK || a->extra_pool != a->pool) return st;
  return kda::debug_check_slots(a->slot_ids, a->N, a->extra_slot_ids, 2 * a->N, s);
}

cudaError_t run_outputs(const kda::PrefillArgs& p, cudaStream_t s) {
  return p.records ? kda::launch_tc_chain_segout(p, p.records, s) : kda::launch_seg_outputs(p, s);
}

}  // namespace

extern "C" {

const char* kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
  }
  return "KDA_ERR_UNKNOWN";
}

int kda_version(void) { return kVersion; }

kda_status kda_set_test_fault(int fault) {
  if (fault != KDA_TEST_FAULT_NONE && fault != KDA_TEST_FAULT_STALL_RECORD_INPUTS) return KDA_ERR_INVALID_ARG;
  g_test_fault = fault;
  return KDA_OK;
}

size_t kda_state_bytes_per_head(int dk, int dv) { return (dk > 0 && dv > 0) ? (size_t)dk * dv * 4 : 0; }

kda_status kda_state_copy(const float* src_pool, int32_t src_num_slots, const int32_t* src_slots, float* dst_pool,
                          int32_t dst_num_slots, const int32_t* dst_slots, int32_t n, int64_t state_elems,
                          int32_t* dev_status, kda_stream_t stream) {
  if (n < 0 || state_elems <= 0 || state_elems % 4 != 0 || src_num_slots < 0 || dst_num_slots < 0)
    return KDA_ERR_INVALID_ARG;
  if (n == 0) return KDA_OK;
  if (!src_pool || !dst_pool || !src_slots || !dst_slots) return KDA_ERR_INVALID_ARG;
  if (!aligned16(src_pool) || !aligned16(dst_pool) || !aligned16(src_slots) || !aligned16(dst_slots))
    return KDA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // debug mode: destinations distinct; within one pool, no destination is also a source
  kda_status dbg = kda::debug_check_slots(dst_slots, n, src_pool == dst_pool ? src_slots : nullptr, n, s);
  if (dbg != KDA_OK) return dbg;
  kda::CopyArgs c{src_pool, src_num_slots, src_slots, dst_pool, dst_num_slots, dst_slots, n, state_elems, dev_status};
  return from_cuda(kda::launch_state_copy(c, s));
}

kda_status kda_decode_step(const void* q, const void* k, const void* v, const float* g, const float* beta, int B,
                           int H, int dk, int dv, kda_dtype in_dtype, float* pool, int32_t num_slots,
                           const int32_t* slot_ids, void* out, kda_dtype out_dtype, int32_t* dev_status,
                           kda_stream_t stream) {
  if (B < 0 || H <= 0 || num_slots < 0 || !dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return KDA_ERR_INVALID_ARG;
  if (!head_ok(dk, dv)) return KDA_ERR_UNSUPPORTED;
  if (B == 0) return KDA_OK;
  if ((int64_t)B * H > 0x7fffffff) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, g, beta, pool, slot_ids, out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  kda_status dbg = kda::debug_check_slots(slot_ids, B, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
  if (dbg != KDA_OK) return dbg;
  kda::DecodeArgs a{q,    k,         v,        g,   beta,      B, H, dk, in_dtype == KDA_DTYPE_BF16,
                    out_dtype == KDA_DTYPE_BF16, pool, num_slots, slot_ids, out, dev_status};
  return from_cuda(kda::launch_decode(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t kda_replay_bytes(int B, int W, int H, int dk, int dv, kda_dtype in_dtype) {
  if (B < 0 || W < 0 || H <= 0 || dk <= 0 || dv <= 0 || !dtype_ok(in_dtype)) return 0;
  return replay_layout(B, W, H, dk, dv, in_dtype).total;
}

kda_status kda_verify(const void* q, const void* k, const void* v, const float* g, const float* beta, int B, int W,
                      int H, int dk, int dv, kda_dtype in_dtype, const float* pool, int32_t num_slots,
                      const int32_t* slot_ids, void* out, kda_dtype out_dtype, void* replay, size_t replay_bytes,
                      float* snapshot_out, int32_t* dev_status, kda_stream_t stream) {
  if (B < 0 || W < 0 || H <= 0 || num_slots < 0 || !dtype_ok(in_dtype) || !dtype_ok(out_dtype))
    return KDA_ERR_INVALID_ARG;
  if (!head_ok(dk, dv)) return KDA_ERR_UNSUPPORTED;
  if (B == 0 || W == 0) return KDA_OK;
  if ((int64_t)B * H > 0x7fffffff) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, g, beta, pool, slot_ids, out, replay};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  if (snapshot_out && !aligned16(snapshot_out)) return KDA_ERR_INVALID_ARG;
  const ReplayLayout L = replay_layout(B, W, H, dk, dv, in_dtype);
  if (replay_bytes < L.total) return KDA_ERR_WORKSPACE;
  kda::VerifyArgs a{q,         k,        v,   g,   beta,   B, W, H, dk, in_dtype == KDA_DTYPE_BF16,
                    out_dtype == KDA_DTYPE_BF16, pool, num_slots, slot_ids, out, replay_ptrs(replay, L),
                    snapshot_out, dev_status};
  return from_cuda(kda::launch_verify(a, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_verify_replay(float* pool, int32_t num_slots, const int32_t* slot_ids, int B, int W, int H, int dk,
                             int dv, kda_dtype in_dtype, const void* replay, size_t replay_bytes,
                             const int32_t* accepted_len, int32_t* dev_status, kda_stream_t stream) {
  if (B < 0 || W < 0 || H <= 0 || num_slots < 0 || !dtype_ok(in_dtype)) return KDA_ERR_INVALID_ARG;
  if (!head_ok(dk, dv)) return KDA_ERR_UNSUPPORTED;
  if (B == 0) return KDA_OK;
  if ((int64_t)B * H > 0x7fffffff) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {pool, slot_ids, replay, accepted_len};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  const ReplayLayout L = replay_layout(B, W, H, dk, dv, in_dtype);
  if (replay_bytes < L.total) return KDA_ERR_WORKSPACE;
  kda_status dbg = kda::debug_check_slots(slot_ids, B, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
  if (dbg != KDA_OK) return dbg;
  kda::FoldArgs a{pool, num_slots, slot_ids, B, W, H, dk, in_dtype == KDA_DTYPE_BF16,
                  replay_ptrs(const_cast<void*>(replay), L), accepted_len, dev_status};
  return from_cuda(kda::launch_fold(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t kda_prefill_args_bytes(void) { return sizeof(kda_prefill_args); }

size_t kda_prefill_workspace_size(const kda_prefill_args* a) {
  if (!a || a->N < 0 || a->H <= 0 || a->T < 0) return 0;
  return record_bytes(a);
}

kda_status kda_prefill_varlen(const kda_prefill_args* a, kda_stream_t stream) {
  kda::PrefillArgs p;
  kda_status st = varlen_prepare(a, &p);
  if (st != KDA_OK || a->N == 0) return st;
  st = prefill_debug_check(a, reinterpret_cast<cudaStream_t>(stream));
  if (st != KDA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!p.records) return from_cuda(kda::launch_prefill_seq(p, s));
  cudaError_t e = kda::launch_tc_prep(p, p.records, s);
  if (e == cudaSuccess) e = kda::launch_tc_chain_plain(p, p.records, s);
  return from_cuda(e);
}

kda_status kda_prefill_records(const kda_prefill_args* a, kda_stream_t stream) {
  kda::PrefillArgs p;
  kda_status st = varlen_prepare(a, &p);
  if (st != KDA_OK || a->N == 0 || !p.records) return st;
  p.test_stall_inputs = g_test_fault == KDA_TEST_FAULT_STALL_RECORD_INPUTS;
  return from_cuda(kda::launch_tc_prep(p, p.records, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_prefill_chain(const kda_prefill_args* a, kda_stream_t stream) {
  kda::PrefillArgs p;
  kda_status st = varlen_prepare(a, &p);
  if (st != KDA_OK || a->N == 0) return st;
  if (!p.records) return KDA_ERR_UNSUPPORTED;
  return from_cuda(kda::launch_tc_chain_plain(p, p.records, reinterpret_cast<cudaStream_t>(stream)));
}

size_t kda_segmented_workspace_size(const kda_prefill_args* a, int32_t segment_len) {
  if (!a || segment_len <= 0 || segment_len % 64 != 0 || a->N < 0 || a->H <= 0 || a->dk <= 0 || a->dv <= 0)
    return 0;
  return seg_layout(a, segment_len).total;
}

kda_status kda_segment_fragments(const kda_prefill_args* a, int32_t segment_len, kda_stream_t stream) {
  kda::PrefillArgs p;
  kda_status st = seg_prepare(a, segment_len, &p);
  if (st != KDA_OK || a->N == 0) return st;
  return from_cuda(run_fragments(p, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_fragment_scan(const kda_prefill_args* a, int32_t segment_len, kda_stream_t stream) {
  kda::PrefillArgs p;
  kda_status st = seg_prepare(a, segment_len, &p);
  if (st != KDA_OK || a->N == 0) return st;
  return from_cuda(kda::launch_seg_scan(p, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_segment_outputs(const kda_prefill_args* a, int32_t segment_len, kda_stream_t stream) {
  kda::PrefillArgs p;
  kda_status st = seg_prepare(a, segment_len, &p);
  if (st != KDA_OK || a->N == 0) return st;
  return from_cuda(run_outputs(p, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_prefill_segmented(const kda_prefill_args* a, int32_t segment_len, kda_stream_t stream) {
  kda::PrefillArgs p;
  kda_status st = seg_prepare(a, segment_len, &p);
  if (st != KDA_OK || a->N == 0) return st;
  st = prefill_debug_check(a, reinterpret_cast<cudaStream_t>(stream));
  if (st != KDA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = p.records ? kda::launch_tc_prep(p, p.records, s) : cudaSuccess;
  if (e == cudaSuccess) e = run_fragments(p, s);
  if (e == cudaSuccess) e = kda::launch_seg_scan(p, s);
  if (e == cudaSuccess) e = run_outputs(p, s);
  return from_cuda(e);
}

size_t kda_cfbi_cache_bytes_per_head(int dk, int dv) {
  return (dk == 128 && dv == 128) ? (size_t)KDA_CFBI_CHUNK * KDA_CFBI_ROW_FLOATS * 4 : 0;
}

kda_status kda_cfbi_prefill(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            const int32_t* cu_seqlens, int32_t N, int64_t T, int32_t max_seqlen, int H, int dk,
                            int dv, kda_dtype in_dtype, float* pool, float* cache, int32_t* counts,
                            int32_t num_slots, const int32_t* slot_ids, void* out, kda_dtype out_dtype,
                            int32_t* dev_status, kda_stream_t stream) {
  if (N < 0 || T < 0 || max_seqlen < 0 || H <= 0 || num_slots < 0 || !dtype_ok(in_dtype) || !dtype_ok(out_dtype))
    return KDA_ERR_INVALID_ARG;
  if (dk != 128 || dv != 128) return KDA_ERR_UNSUPPORTED;
  if (N == 0) return KDA_OK;
  if (N > 65535 || H > 65535) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {cu_seqlens, pool, cache, counts, slot_ids};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  if (T > 0) {
    const void* tp[] = {q, k, v, g, beta, out};
    for (const void* p : tp)
      if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  }
  kda_status dbg = kda::debug_check_slots(slot_ids, N, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
  if (dbg != KDA_OK) return dbg;
  kda::CfbiArgs a{q,   k,    v,     g,     beta,  0,         N,        T,     max_seqlen,
                  cu_seqlens, H, in_dtype == KDA_DTYPE_BF16, out_dtype == KDA_DTYPE_BF16, pool, cache, counts,
                  num_slots,   slot_ids,  out,   dev_status};
  return from_cuda(kda::launch_cfbi_prefill(a, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
struct CfbiChunkedLayout {
  size_t qh, oh, rows, count, total;
};
CfbiChunkedLayout cfbi_chunked_layout(int64_t T, int32_t N, int H) {
  CfbiChunkedLayout L{};
  L.qh = 0;
  L.oh = align256((size_t)T * H * kda::cfbi_chunked_qh_row_floats() * 4);
  L.rows = L.oh + align256((size_t)T * H * 128 * 4);
  L.count = L.rows + align256(kda::cfbi_chunked_records(T, N) * H * kda::cfbi_chunked_record_bytes());
  L.total = L.count + align256((size_t)N * H * 4);
  return L;
}
}  // namespace

size_t kda_cfbi_prefill_chunked_workspace_size(int64_t T, int32_t N, int H, int dk, int dv) {
  if (T < 0 || N < 0 || H <= 0 || dk != 128 || dv != 128) return 0;
  return cfbi_chunked_layout(T, N, H).total;
}

kda_status kda_cfbi_prefill_chunked(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                    const int32_t* cu_seqlens, int32_t N, int64_t T, int32_t max_seqlen, int H,
                                    int dk, int dv, kda_dtype in_dtype, float* pool, float* cache, int32_t* counts,
                                    int32_t num_slots, const int32_t* slot_ids, void* out, kda_dtype out_dtype,
                                    void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                    kda_stream_t stream) {
  if (N < 0 || T < 0 || max_seqlen < 0 || H <= 0 || num_slots < 0 || !dtype_ok(in_dtype) || !dtype_ok(out_dtype))
    return KDA_ERR_INVALID_ARG;
  if (dk != 128 || dv != 128) return KDA_ERR_UNSUPPORTED;
  if (N == 0) return KDA_OK;
  if (N > 65535 || H > 65535 || max_seqlen > 65535 * KDA_CFBI_CHUNK - 2 * KDA_CFBI_CHUNK)
    return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {cu_seqlens, pool, cache, counts, slot_ids, workspace};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  if (T > 0) {
    const void* tp[] = {q, k, v, g, beta, out};
    for (const void* p : tp)
      if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  }
  const CfbiChunkedLayout L = cfbi_chunked_layout(T, N, H);
  if (workspace_bytes < L.total) return KDA_ERR_WORKSPACE;
  kda_status dbg = kda::debug_check_slots(slot_ids, N, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
  if (dbg != KDA_OK) return dbg;
  kda::CfbiArgs a{q,   k,    v,     g,     beta,  0,         N,        T,     max_seqlen,
                  cu_seqlens, H, in_dtype == KDA_DTYPE_BF16, out_dtype == KDA_DTYPE_BF16, pool, cache, counts,
                  num_slots,   slot_ids,  out,   dev_status};
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  kda::CfbiWorkspace w{reinterpret_cast<float*>(ws + L.qh), reinterpret_cast<float*>(ws + L.oh),
                       reinterpret_cast<float*>(ws + L.rows), reinterpret_cast<int32_t*>(ws + L.count)};
  return from_cuda(kda::launch_cfbi_prefill_chunked(a, w, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_cfbi_decode(const void* q, const void* k, const void* v, const float* g, const float* beta, int B,
                           int H, int dk, int dv, kda_dtype in_dtype, float* pool, float* cache, int32_t* counts,
                           int32_t num_slots, const int32_t* slot_ids, void* out, kda_dtype out_dtype,
                           int32_t* dev_status, kda_stream_t stream) {
  if (B < 0 || H <= 0 || num_slots < 0 || !dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return KDA_ERR_INVALID_ARG;
  if (dk != 128 || dv != 128) return KDA_ERR_UNSUPPORTED;
  if (B == 0) return KDA_OK;
  if ((int64_t)B * H > 0x7fffffff) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, g, beta, pool, cache, counts, slot_ids, out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  kda_status dbg = kda::debug_check_slots(slot_ids, B, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
  if (dbg != KDA_OK) return dbg;
  kda::CfbiArgs a{q,       k,        v,    g,        beta, B,         0,  0,         0,
                  nullptr, H, in_dtype == KDA_DTYPE_BF16, out_dtype == KDA_DTYPE_BF16, pool, cache, counts,
                  num_slots, slot_ids, out,  dev_status};
  return from_cuda(kda::launch_cfbi_decode(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

extern "C" {

size_t kda_backward_args_bytes(void) { return sizeof(kda_backward_args); }

size_t kda_backward_workspace_size(const kda_backward_args* a) {
  if (!a || a->T < 0 || a->N < 0 || a->H <= 0) return 0;
  return kda::backward_ws_bytes(a->T, a->N, a->H);
}

kda_status kda_prefill_backward(const kda_backward_args* a, kda_stream_t stream) {
  if (!a) return KDA_ERR_INVALID_ARG;
  if (!dtype_ok(a->in_dtype)) return KDA_ERR_INVALID_ARG;
  if (a->H <= 0 || a->N < 0 || a->T < 0 || a->max_seqlen < 0 || a->num_slots < 0 || a->N > 65535 || a->H > 32767)
    return KDA_ERR_INVALID_ARG;
  if (a->dk != 128 || a->dv != 128) return KDA_ERR_UNSUPPORTED;
  if (!a->cu_seqlens || !aligned16(a->cu_seqlens)) return KDA_ERR_INVALID_ARG;
  if (!a->init_zero && (!a->pool || !a->slot_ids || !aligned16(a->pool) || !aligned16(a->slot_ids)))
    return KDA_ERR_INVALID_ARG;
  const void* dense[] = {a->q, a->k, a->v, a->g, a->beta, a->d_out, a->dq, a->dk_out, a->dv_out, a->dg, a->dbeta};
  if (a->T > 0)
    for (const void* p : dense)
      if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  if ((a->d_final && !aligned16(a->d_final)) || (a->d_init && !aligned16(a->d_init))) return KDA_ERR_INVALID_ARG;
  if (a->N == 0) return KDA_OK;
  const size_t need = kda::backward_ws_bytes(a->T, a->N, a->H);
  if (a->workspace_bytes < need || !a->workspace || (reinterpret_cast<uintptr_t>(a->workspace) & 255u))
    return KDA_ERR_WORKSPACE;
  kda::BackwardArgs b{};
  b.q = a->q;
  b.k = a->k;
  b.v = a->v;
  b.g = a->g;
  b.beta = a->beta;
  b.in_bf16 = a->in_dtype == KDA_DTYPE_BF16;
  b.T = a->T;
  b.H = a->H;
  b.N = a->N;
  b.cu = a->cu_seqlens;
  b.max_seqlen = a->max_seqlen;
  b.pool = a->pool;
  b.num_slots = a->num_slots;
  b.slot_ids = a->slot_ids;
  b.init_zero = a->init_zero != 0;
  b.d_out = a->d_out;
  b.d_final = a->d_final;
  b.dq = a->dq;
  b.dk = a->dk_out;
  b.dv = a->dv_out;
  b.dg = a->dg;
  b.dbeta = a->dbeta;
  b.d_init = a->d_init;
  b.ws = static_cast<float*>(a->workspace);
  b.status = a->dev_status;
  return from_cuda(kda::launch_backward(b, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

extern "C" {

size_t kda_fused_decode_args_bytes(void) { return sizeof(kda_fused_decode_args); }

kda_status kda_fused_decode(const kda_fused_decode_args* a, kda_stream_t stream) {
  if (!a) return KDA_ERR_INVALID_ARG;
  if (!dtype_ok(a->in_dtype) || !dtype_ok(a->out_dtype)) return KDA_ERR_INVALID_ARG;
  if (a->B < 0 || a->H <= 0 || a->num_slots < 0 || !(a->norm_eps >= 0.f)) return KDA_ERR_INVALID_ARG;
  if ((int64_t)a->B * a->H > 0x7fffffff) return KDA_ERR_INVALID_ARG;
  if (a->dk != 128 || a->dv != 128) return KDA_ERR_UNSUPPORTED;
  if (a->B == 0) return KDA_OK;
  const void* ptrs[] = {a->xq, a->xk, a->xv, a->a, a->b, a->z, a->pool, a->slot_ids, a->conv_state, a->conv_w,
                        a->norm_w, a->out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  kda_status dbg = kda::debug_check_slots(a->slot_ids, a->B, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
  if (dbg != KDA_OK) return dbg;
  kda::FusedDecodeArgs f{};
  f.xq = a->xq;
  f.xk = a->xk;
  f.xv = a->xv;
  f.a = a->a;
  f.b = a->b;
  f.z = a->z;
  f.in_bf16 = a->in_dtype == KDA_DTYPE_BF16;
  f.out_bf16 = a->out_dtype == KDA_DTYPE_BF16;
  f.B = a->B;
  f.H = a->H;
  f.pool = a->pool;
  f.num_slots = a->num_slots;
  f.slot_ids = a->slot_ids;
  f.conv_state = a->conv_state;
  f.conv_w = a->conv_w;
  f.norm_w = a->norm_w;
  f.eps = a->norm_eps;
  f.out = a->out;
  f.status = a->dev_status;
  return from_cuda(kda::launch_fused_decode(f, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

extern "C" {

kda_status kda_kcp_fragments(const kda_prefill_args* a, int32_t segment_len, float* frag_out, kda_stream_t stream) {
  kda::PrefillArgs p;
  kda_status st = seg_prepare(a, segment_len, &p);
  if (st != KDA_OK || a->N == 0) return st;
  if (!frag_out || !aligned16(frag_out)) return KDA_ERR_INVALID_ARG;
  p.frag = frag_out;
  p.frag_all = true;
  return from_cuda(run_fragments(p, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_kcp_scan(const float* frags, int32_t P, int H, int dk, int dv, const float* s0, float* entries,
                        int32_t* dev_status, kda_stream_t stream) {
  if (P <= 0 || P > 65535 || H <= 0 || H > 65535) return KDA_ERR_INVALID_ARG;
  if (!head_ok(dk, dv)) return KDA_ERR_UNSUPPORTED;
  if (!frags || !entries || !aligned16(frags) || !aligned16(entries) || (s0 && !aligned16(s0)))
    return KDA_ERR_INVALID_ARG;
  kda::PrefillArgs p{};
  p.H = H;
  p.d = dk;
  p.N = 1;
  p.P = P;
  p.seg_len = 1;
  p.frag = const_cast<float*>(frags);
  p.entry = entries;
  p.scan_nseg = P;
  p.scan_s0 = s0;
  p.status = dev_status;
  return from_cuda(kda::launch_seg_scan(p, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_kcp_outputs(const kda_prefill_args* a, int32_t segment_len, const float* entries,
                           kda_stream_t stream) {
  kda::PrefillArgs p;
  kda_status st = seg_prepare(a, segment_len, &p);
  if (st != KDA_OK || a->N == 0) return st;
  if (!entries || !aligned16(entries)) return KDA_ERR_INVALID_ARG;
  p.entry = const_cast<float*>(entries);
  return from_cuda(run_outputs(p, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
