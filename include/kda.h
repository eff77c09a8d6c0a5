/*
 * kda.h -- C ABI of the KDA (Kimi Delta Attention) hot path on one NVIDIA GB300 (sm_103a).
 *
 * The recurrence (per sequence and head; S is dk x dv fp32, row j of S belongs to key channel j):
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,   o_t = S_t^T q_t
 * with alpha_t = exp(g_t) a per-channel decay (g is passed as the log-decay) and beta_t a scalar.
 * Source: "Kimi K3: Architecture and SGLang Day-0 Support" (AI-Infra-Visualized lesson), section
 * "attention mechanism explained: KDA", math box (full update; gate, read along the key, delta write);
 * section "linear attention" for the read-out o = S^T q after the write.  No 1/sqrt(dk) scale is applied.
 *
 * Conventions shared by every call
 * --------------------------------
 * * Every pointer argument is a DEVICE pointer owned by the caller unless stated otherwise.  The library
 *   never allocates, frees or retains memory; it keeps no state between calls.
 * * Every call is asynchronous: it validates its host-visible arguments, enqueues its kernels on `stream`
 *   (a cudaStream_t; NULL is the legacy default stream) and returns.  Stream order is the only ordering:
 *   a copy-on-write restore, a forward pass and a snapshot enqueued on one stream happen in that order.
 * * Return value: KDA_OK, or an error code; on an error nothing was enqueued, except KDA_ERR_CUDA, which
 *   reports a launch failure (the error of cudaGetLastError()).
 * * State pools are fp32, laid out [num_slots][H][dk][dv] row-major; a slot is H*dk*dv*4 bytes.
 * * Token-major inputs: q, k [T][H][dk]; v [T][H][dv] (fp32 or bf16, `in_dtype`); g [T][H][dk] fp32
 *   (log-decay, <= 0; the pages bound it below by -5); beta [T][H] fp32 in (0, 1).
 * * Outputs o [T][H][dv] in `out_dtype` (fp32 or bf16, round to nearest even).
 * * Supported head sizes: dk == dv in {16, 32, 64, 128}.  Anything else returns KDA_ERR_UNSUPPORTED.
 * * Alignment: every array base must be 16-byte aligned (KDA_ERR_INVALID_ARG otherwise).
 * * dev_status (optional, may be NULL): int32[2] in device memory.  Kernels OR error flags
 *   (KDA_DEV_*) into dev_status[0] and add the number of (token x head) state updates they performed
 *   to dev_status[1] (wrapping 32-bit counter; a test that sees 0 work knows it tested nothing).
 *   A slot id or accepted length out of range sets its flag; that unit is skipped without touching memory.
 * * Slot ids within one call must be distinct; a source and a destination slot of one copy must not be
 *   the same memory.  By default violations are not detected and give undefined results; with the debug
 *   checks on (kda_set_debug_checks below) the calls that take slot ids check this on the host first.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kda_stream_t; /* == cudaStream_t */

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative or inconsistent size */
  KDA_ERR_UNSUPPORTED = 2, /* head size or dtype combination not built */
  KDA_ERR_WORKSPACE = 3,   /* workspace or record buffer too small */
  KDA_ERR_CUDA = 4         /* a kernel launch failed */
} kda_status;

typedef enum { KDA_DTYPE_F32 = 0, KDA_DTYPE_BF16 = 1 } kda_dtype;

/* dev_status[0] flags */
#define KDA_DEV_SLOT_OOB 1   /* a slot id outside [0, num_slots) */
#define KDA_DEV_SEQ_OOB 2    /* cu_seqlens not non-decreasing within [0, T], or a sequence longer than max_seqlen */
#define KDA_DEV_TIMEOUT 4    /* a bounded wait inside a kernel gave up */
#define KDA_DEV_ACCEPT_OOB 8 /* an accepted length outside [0, W] */

/* Human-readable name of a status code (static storage). */
const char* kda_status_string(kda_status s);

/* Library version, major*10000 + minor*100 + patch. */
int kda_version(void);

/* Bytes of one head's state: dk*dv*4 (64 KB at dk = dv = 128, the figure the ReplaySSM section of
 * "SGLang and Miles: day-0 support for Kimi K3" gives per request, layer and head). */
size_t kda_state_bytes_per_head(int dk, int dv);

/*
 * kda_set_test_fault -- a test hook for the kernels' bounded waits (failure detection without a GPU fault).
 * KDA_TEST_FAULT_STALL_RECORD_INPUTS makes later kda_prefill_records calls launch the prep kernel with its
 * input copies left out: no copy is issued, so its first wait for the inputs finds nothing to wait for,
 * gives up after a short bounded poll, and every CTA flags KDA_DEV_TIMEOUT in dev_status and returns (its
 * tensor memory freed, nothing in flight).  The records are then not written; nothing else is touched.
 * KDA_TEST_FAULT_NONE (the initial value) restores normal calls.  Process-wide, not thread-safe; for tests.
 * Returns KDA_ERR_INVALID_ARG for an unknown value.
 */
#define KDA_TEST_FAULT_NONE 0
#define KDA_TEST_FAULT_STALL_RECORD_INPUTS 1
kda_status kda_set_test_fault(int fault);

/*
 * Debug checks of the slot-id contract.  Source: "SGLang and Miles: day-0 support for Kimi K3", three
 * state movements on the forward stream (each request owns its slot; a snapshot's target slot is never the
 * slot it copies).
 * kda_check_slot_ids -- HOST arrays: KDA_OK when the n ids are distinct and (other_ids not NULL) none of them
 *   is among the n_other other_ids; KDA_ERR_INVALID_ARG otherwise or for a negative count.  Range is not
 *   checked here (out-of-range ids are flagged on the device, KDA_DEV_SLOT_OOB).
 * kda_set_debug_checks(on) / kda_debug_checks() -- switch / read the debug mode (process-wide; initially on
 *   when the environment variable KDA_DEBUG_CHECKS is set to a value other than 0).  In debug mode the calls
 *   that take slot ids (kda_state_copy, kda_decode_step, kda_verify_replay, kda_prefill_varlen,
 *   kda_prefill_segmented, kda_cfbi_prefill, kda_cfbi_decode, kda_fused_decode) copy their ids to the host
 *   on their stream, wait for the copy (so the call is no longer asynchronous and cannot be captured in a
 *   CUDA graph), and return KDA_ERR_INVALID_ARG with nothing enqueued when:
 *     - two ids of the call are equal (kda_state_copy: two destination ids; a source may feed several);
 *     - kda_state_copy with src_pool == dst_pool: a destination id is also a source id;
 *     - a prefill with snapshots: two extra_slot_ids are equal, or (extra_pool == pool) an extra slot is
 *       also one of the sequences' slots.
 *   A failed copy or wait returns KDA_ERR_CUDA.
 */
kda_status kda_check_slot_ids(const int32_t* ids, int32_t n, const int32_t* other_ids, int32_t n_other);
void kda_set_debug_checks(int on);
int kda_debug_checks(void);

/*
 * kda_state_copy -- copy whole slot states: dst_pool[dst_slots[i]] = src_pool[src_slots[i]], i < n.
 * Source: "SGLang and Miles: day-0 support for Kimi K3", section "hybrid KDA memory management",
 * "three state movements on the forward stream": the copy-on-write restore (checkpoint -> working slot)
 * and the snapshot (working slot -> extra buffer) are kernels on the serial forward stream, so stream
 * order gives the happens-before.  Donating a slot moves no bytes and needs no call.
 *   src_pool [src_num_slots][state_elems], dst_pool [dst_num_slots][state_elems], fp32;
 *   state_elems = H*dk*dv (a multiple of 4);  src_slots, dst_slots: int32[n] device arrays.
 * Byte-exact.  An out-of-range slot id sets KDA_DEV_SLOT_OOB and that pair is skipped.
 */
kda_status kda_state_copy(const float* src_pool, int32_t src_num_slots, const int32_t* src_slots, float* dst_pool,
                          int32_t dst_num_slots, const int32_t* dst_slots, int32_t n, int64_t state_elems,
                          int32_t* dev_status, kda_stream_t stream);

/*
 * kda_decode_step -- one token per request, state updated in place in the pool.
 * Source: the KDA math box of "Kimi K3: Architecture and SGLang Day-0 Support" (gate-then-delta form:
 * S~ = Diag(alpha) S, r_old = S~^T k, S = S~ + beta k (v - r_old)^T) and the fused decode kernel named in
 * "SGLang and Miles: day-0 support for Kimi K3", section "kernels".
 *   q, k, g [B][H][dk]; v [B][H][dv]; beta [B][H]; out [B][H][dv];
 *   pool [num_slots][H][dk][dv] (read and written once per (request, head)); slot_ids int32[B].
 * The output is computed as o = S~^T q + (q . k) u with u = beta (v - r_old), which equals S_t^T q.
 * Decode, verify and replay run one shared per-token routine, so n decode steps and a replay of n
 * window tokens give bit-identical states.
 */
kda_status kda_decode_step(const void* q, const void* k, const void* v, const float* g, const float* beta, int B,
                           int H, int dk, int dv, kda_dtype in_dtype, float* pool, int32_t num_slots,
                           const int32_t* slot_ids, void* out, kda_dtype out_dtype, int32_t* dev_status,
                           kda_stream_t stream);

/*
 * kda_replay_bytes -- size of the raw-input record buffer for a W-token draft window.
 * Layout (each sub-array starts at a 256-byte aligned offset, in this order):
 *   k    [B][W][H][dk]  in_dtype      v    [B][W][H][dv]  in_dtype
 *   g    [B][W][H][dk]  fp32          beta [B][W][H]      fp32
 * i.e. the step inputs S_i = (v_i, k_i, gk_i, beta_i) of the ReplaySSM section (q is not needed to
 * advance the state): 1028 bytes per token and head at d = 128 with bf16 k and v.
 */
size_t kda_replay_bytes(int B, int W, int H, int dk, int dv, kda_dtype in_dtype);

/*
 * kda_verify -- speculative verify of a W-token draft window from the committed states.
 * Source: "SGLang and Miles: day-0 support for Kimi K3", section "ReplaySSM: raw-input replay for KDA
 * state": the verify kernel reads the committed checkpoint but never writes it, and stores each step's
 * raw inputs; rejected drafts are never replayed.
 *   q, k, g [B][W][H][dk]; v [B][W][H][dv]; beta [B][W][H]; out [B][W][H][dv];
 *   pool is read only; replay: record buffer of replay_bytes >= kda_replay_bytes(B, W, H, dk, dv, in_dtype);
 *   snapshot_out: NULL, or fp32 [B][W][H][dk][dv] receiving the state after every window token (the
 *   snapshot-every-draft-step baseline the section replaces; for tests and comparisons).
 */
kda_status kda_verify(const void* q, const void* k, const void* v, const float* g, const float* beta, int B, int W,
                      int H, int dk, int dv, kda_dtype in_dtype, const float* pool, int32_t num_slots,
                      const int32_t* slot_ids, void* out, kda_dtype out_dtype, void* replay, size_t replay_bytes,
                      float* snapshot_out, int32_t* dev_status, kda_stream_t stream);

/*
 * kda_verify_replay -- commit the accepted prefix of each window (the fold).
 * Source: same ReplaySSM section: one fold kernel over all heads replays only the accepted prefix from
 * the checkpoint, in place, consuming the gate values the verify kernel stored, so the rebuilt state is
 * bit-identical to the recurrence baseline.
 *   pool [num_slots][H][dk][dv], slot_ids int32[B] (the same slots verify read);
 *   replay: the record buffer written by kda_verify with the same B, W, H, dk, dv, in_dtype;
 *   accepted_len int32[B] device, each in [0, W]: tokens 1..n of the window are committed; n = 0 leaves
 *   the slot untouched (no read, no write).  A value outside [0, W] sets KDA_DEV_ACCEPT_OOB, skipped.
 */
kda_status kda_verify_replay(float* pool, int32_t num_slots, const int32_t* slot_ids, int B, int W, int H, int dk,
                             int dv, kda_dtype in_dtype, const void* replay, size_t replay_bytes,
                             const int32_t* accepted_len, int32_t* dev_status, kda_stream_t stream);

/* Arguments of a packed variable-length prefill. */
typedef struct {
  const void* q;          /* [T][H][dk] in_dtype */
  const void* k;          /* [T][H][dk] in_dtype */
  const void* v;          /* [T][H][dv] in_dtype */
  const float* g;         /* [T][H][dk] log-decay */
  const float* beta;      /* [T][H] */
  kda_dtype in_dtype;
  int64_t T;              /* total packed tokens (host) */
  int H, dk, dv;
  int N;                  /* number of sequences (host) */
  const int32_t* cu_seqlens; /* int32[N+1] device: sequence i is tokens [cu[i], cu[i+1]) */
  int32_t max_seqlen;     /* host: an upper bound on every sequence length (work sizing) */
  float* pool;            /* [num_slots][H][dk][dv]: initial states read from, final states written to */
  int32_t num_slots;
  const int32_t* slot_ids; /* int32[N] device */
  int init_zero;          /* nonzero: start every sequence from a zero state instead of pool[slot] */
  void* out;              /* [T][H][dv] out_dtype */
  kda_dtype out_dtype;
  float* extra_pool;      /* optional snapshot pool [num_extra_slots][H][dk][dv], or NULL */
  int32_t num_extra_slots;
  const int32_t* extra_slot_ids; /* int32[N][2] device: the ping-pong pair of each sequence */
  int32_t snapshot_every_chunks; /* 0: no snapshots; else a snapshot every this many 64-token chunks */
  void* workspace;        /* scratch device memory, >= the matching *_workspace_size() bytes, or NULL if 0 */
  size_t workspace_bytes;
  int32_t* dev_status;    /* optional int32[2] */
} kda_prefill_args;

/* sizeof(kda_prefill_args), so a binding can check its mirror of the struct. */
size_t kda_prefill_args_bytes(void);

/*
 * Workspace of kda_prefill_varlen.  bf16 inputs with dk = dv = 128 run the chunked tensor-core path, which
 * needs (ceil(T/64) + N) * H * 148480 bytes (16-byte aligned) for the per-chunk operand records; every
 * other combination runs the token-sequential path and needs none (0).
 */

/*
 * kda_prefill_varlen -- chunked prefill over packed sequences.
 * Source: the recurrence above; chunked computation with keys rescaled by the reciprocal cumulative decay,
 * made safe for dense tensor-core tiles by the log-decay floor g >= -5 ("Kimi K3: Architecture and SGLang
 * Day-0 Support", KDA math box); per-chunk snapshots into a ping-pong extra buffer ("SGLang and Miles:
 * day-0 support for Kimi K3", "three state movements on the forward stream").
 * Sequence i starts from pool[slot_ids[i]] (or zero) and its final state is written to pool[slot_ids[i]].
 * Snapshots (when extra_pool != NULL and snapshot_every_chunks > 0): after every p = 64 * m *
 * snapshot_every_chunks tokens of sequence i (p <= its length, counted from the sequence start), the
 * state is written to extra_pool[extra_slot_ids[2*i + ((m - 1) & 1)]]; the latest snapshot is in entry
 * ((n_snap - 1) & 1).  Sequences shorter than one interval leave their extra slots untouched.  Only the final
 * contents of the extra pool are defined: snapshots that a later snapshot of the same call overwrites (all but
 * the last two of a sequence) are not written.
 */
kda_status kda_prefill_varlen(const kda_prefill_args* a, kda_stream_t stream);
size_t kda_prefill_workspace_size(const kda_prefill_args* a);  /* see above; KDA_ERR_WORKSPACE if too small */

/*
 * The two phases of kda_prefill_varlen on the tensor-core path, exported so callers (and the benchmark)
 * can time or schedule them separately.  kda_prefill_records writes the per-chunk operand records into
 * a->workspace (all chunks of all sequences in parallel; a no-op returning KDA_OK where no records are
 * needed); kda_prefill_chain then carries the state through the chunks of each sequence from those
 * records (KDA_ERR_UNSUPPORTED where the token-sequential path applies).
 */
kda_status kda_prefill_records(const kda_prefill_args* a, kda_stream_t stream);
kda_status kda_prefill_chain(const kda_prefill_args* a, kda_stream_t stream);

/*
 * kda_prefill_segmented -- the same result as kda_prefill_varlen, computed by splitting every sequence into
 * segments of segment_len tokens (a multiple of 64) that run in parallel.
 * Source: "Kimi K3 training and serving infra" (marsggbo blog), section 4.2 "KCP: pass fixed-size
 * transition information": each segment computes its cumulative transition M and the state S~ it produces
 * from a zero input state; the true entry state of the next segment is S_in2 = M1 S_in1 + S~1; a prefix scan
 * over the segments recovers every entry state, and the outputs are then computed from them.  Here all
 * segments live on one GPU.  Three phases on `stream`: fragments, scan, outputs.
 * Needs workspace_bytes >= kda_segmented_workspace_size(a, segment_len).  Snapshots are supported.
 */
kda_status kda_prefill_segmented(const kda_prefill_args* a, int32_t segment_len, kda_stream_t stream);
size_t kda_segmented_workspace_size(const kda_prefill_args* a, int32_t segment_len);

/*
 * Phases of kda_prefill_segmented, exported for tests and timing.  Workspace layout, in this order:
 *   records                       the per-chunk operand records of the tensor-core path, as for
 *                                 kda_prefill_varlen (absent, 0 bytes, on the token-sequential path)
 *   frag  [N][P][H][dk][dv + dk]  fp32, per segment: columns 0..dv-1 hold S~ (zero input state),
 *                                 columns dv..dv+dk-1 hold M (cumulative transition)
 *   entry [N][P][H][dk][dv]       fp32, entry state of every segment (segment 0: the initial state)
 * with P = ceil(max_seqlen / segment_len) and frag, entry starting on 256-byte boundaries after the
 * records.  kda_prefill_segmented = kda_prefill_records, kda_segment_fragments, kda_fragment_scan,
 * kda_segment_outputs: the fragments and outputs phases read the records (tensor-core path),
 * kda_segment_fragments writes frag, kda_fragment_scan writes entry from frag and the initial states, and
 * kda_segment_outputs reads entry.
 */
kda_status kda_segment_fragments(const kda_prefill_args* a, int32_t segment_len, kda_stream_t stream);
kda_status kda_fragment_scan(const kda_prefill_args* a, int32_t segment_len, kda_stream_t stream);
/* Third phase: outputs, snapshots and final states of every segment from the entry states in the workspace. */
kda_status kda_segment_outputs(const kda_prefill_args* a, int32_t segment_len, kda_stream_t stream);

/*
 * kda_prefill_segmented_noalloc -- kda_prefill_segmented for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a deployment convenience of this library.
 * Some callers cannot pass a workspace: a plugin inside an inference server that owns all device memory
 * through its own pool and offers plugins no allocation hook, or a serving loop that must not call
 * cudaMalloc after start-up.  This call takes the whole workspace of kda_prefill_segmented (on the
 * tensor-core path: the per-chunk operand records, 145 KiB per 64-token chunk and head and most of the
 * total, then the segment fragments and the entry states, as kda_segmented_workspace_size counts them)
 * from a fixed 32 MiB array inside the library instead; a->workspace and a->workspace_bytes are ignored.
 * It launches the same kernels as kda_prefill_segmented (records, fragments, scan, outputs).  Everything
 * else (arguments, results, errors) is as for kda_prefill_segmented.
 *   * A problem whose scratch (kda_segmented_workspace_size) exceeds 32 MiB returns KDA_ERR_WORKSPACE.
 *     Example: one 1024-token sequence, H = 4, d = 128 (bf16), segment_len = 256 needs about 13 MiB.
 *   * The array occupies 32 MiB of device memory on every GPU that loads this code, until the process
 *     exits.
 *   * The first call on a device looks up the array's device address (with that device current); make
 *     that first call before any stream capture.
 *   * All calls share the array and it keeps the last call's contents (no clearing is needed: every
 *     byte read is first written by the same call).  Calls whose kernels overlap on the GPU race on it.
 */
kda_status kda_prefill_segmented_noalloc(const kda_prefill_args* a, int32_t segment_len, kda_stream_t stream);

/*
 * CF-BI: one row-level computation contract for prefill and decode (batch-invariant outputs).
 * Source: "Kimi K3.1 inference zero mismatch" (LLMNews), section 6.1: prefill and decode follow one
 * row-level contract -- a position's output depends on the entry state of its chunk and the rows before it
 * in that chunk, prefill computes the rows in bulk and decode the new row, in the same operation order; the
 * open chunk's row cache and position are kept besides the recurrent state; 16-token chunks, an fp32 row
 * cache per head.  Row t of a chunk with entry state S_c (G the in-chunk cumulative log-decay):
 *   A_tu = beta_t sum_j k_t k_u e^{G_t - G_u} (u < t),  P_tu = sum_j q_t k_u e^{G_t - G_u} (u <= t),
 *   R_t = row t of P (I + A)^-1 diag(beta),
 *   o_t = S_c^T (q_t o e^{G_t} - sum_u R_tu k_u o e^{G_u}) + sum_u R_tu v_u,
 * and a full chunk advances S_c with U = (I + A)^-1 diag(beta) (V - (K o e^G) S_c):
 *   S_{c+1} = Diag(e^{G_15}) S_c + (K o e^{G_15 - G})^T U.
 * The same device routines run in both calls, in fp32 with round-to-nearest operations in a fixed order,
 * so a token's output and the state are bit-identical whether it was prefilled or decoded, whatever the
 * batch and wherever a sequence is split between prefill and decode.  Values agree with the recurrence
 * above (kda_decode_step) to rounding, not bit for bit.
 *
 * Per (slot, head) state: S_c in `pool` ([num_slots][H][128][128] fp32, the usual layout), the open chunk's
 * rows in `cache` ([num_slots][H][KDA_CFBI_CHUNK][KDA_CFBI_ROW_FLOATS] fp32: k[128] | v[128] | G[128] |
 * A_t[16] (beta folded in) | beta | T_t[16] (row t of (I + A)^-1) | padding; A_t[u >= t], T_t[v > t] and the
 * padding are written as zeros, so the cached bytes depend on the chunk's tokens alone) and their number in
 * `counts` ([num_slots][H] int32, 0..15).
 * A fresh sequence starts from S_0 in its pool slot with counts = 0 (cache contents then unused).
 * dk = dv = 128 only (KDA_ERR_UNSUPPORTED otherwise).  A count outside [0, 16) sets KDA_DEV_SLOT_OOB and that
 * unit is skipped.
 */
#define KDA_CFBI_CHUNK 16
#define KDA_CFBI_ROW_FLOATS 420

/* Bytes of one head's row cache: KDA_CFBI_CHUNK * KDA_CFBI_ROW_FLOATS * 4 at dk = dv = 128, else 0. */
size_t kda_cfbi_cache_bytes_per_head(int dk, int dv);

/*
 * kda_cfbi_prefill -- packed sequences through the CF-BI contract; sequence i continues from the state of
 * slot_ids[i] (pool, cache, counts) and leaves its state there.  One CTA per (sequence, head) walks the
 * tokens in order.  q, k [T][H][128], v [T][H][128] (in_dtype), g [T][H][128], beta [T][H] fp32,
 * cu_seqlens int32[N + 1] (device), out [T][H][128] (out_dtype).
 */
kda_status kda_cfbi_prefill(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            const int32_t* cu_seqlens, int32_t N, int64_t T, int32_t max_seqlen, int H, int dk,
                            int dv, kda_dtype in_dtype, float* pool, float* cache, int32_t* counts,
                            int32_t num_slots, const int32_t* slot_ids, void* out, kda_dtype out_dtype,
                            int32_t* dev_status, kda_stream_t stream);

/*
 * kda_cfbi_prefill_chunked -- kda_cfbi_prefill's operation (same arguments, same results bit for bit:
 * outputs, states, row caches and counts), with the chunks of every sequence worked on in parallel.
 * Source: "Kimi K3.1 inference zero mismatch" (LLMNews), section 6.1: a position's output depends only on
 * its chunk's entry state and the rows before it in the chunk, so the rows of all chunks (and the parts of
 * each output that do not involve the state) are formed at once, one CTA per (chunk, sequence, head); the
 * state then walks the chunks in order, one CTA per (8 value columns, sequence, head), each value column of
 * the state evolving on its own.  Every element is formed by the same fp32 round-to-nearest operations in
 * the same order as in kda_cfbi_prefill / kda_cfbi_decode.
 * workspace: device memory of at least kda_cfbi_prefill_chunked_workspace_size(T, N, H, dk, dv) bytes,
 * 16-byte aligned, owned by the caller, contents ignored on entry and meaningless after; smaller: returns
 * KDA_ERR_WORKSPACE without launching.  max_seqlen bounds the sequence lengths (KDA_DEV_SEQ_OOB for a longer
 * one, as for kda_cfbi_prefill) and sizes the grid; at most 65535 * 16 - 32.
 */
size_t kda_cfbi_prefill_chunked_workspace_size(int64_t T, int32_t N, int H, int dk, int dv);
kda_status kda_cfbi_prefill_chunked(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                    const int32_t* cu_seqlens, int32_t N, int64_t T, int32_t max_seqlen, int H,
                                    int dk, int dv, kda_dtype in_dtype, float* pool, float* cache, int32_t* counts,
                                    int32_t num_slots, const int32_t* slot_ids, void* out, kda_dtype out_dtype,
                                    void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                    kda_stream_t stream);

/*
 * kda_cfbi_decode -- one token per request through the CF-BI contract.  q, k, v [B][H][128] (in_dtype),
 * g [B][H][128], beta [B][H] fp32, out [B][H][128] (out_dtype).  Reads the entry state; writes it only when
 * the token completes a chunk (then counts returns to 0).
 */
kda_status kda_cfbi_decode(const void* q, const void* k, const void* v, const float* g, const float* beta, int B,
                           int H, int dk, int dv, kda_dtype in_dtype, float* pool, float* cache, int32_t* counts,
                           int32_t num_slots, const int32_t* slot_ids, void* out, kda_dtype out_dtype,
                           int32_t* dev_status, kda_stream_t stream);

/*
 * Backward (vector-Jacobian product) of a packed prefill.
 * Source: the recurrence above ("Kimi K3: Architecture and SGLang Day-0 Support", KDA math box), whose
 * gradient the training side needs ("Kimi K3 training and serving infra" (marsggbo blog), section 7).
 * For the loss L = sum_t <d_out_t, o_t> + sum_i <d_final_i, S_T(i)>, where o and S_T(i) are the outputs and
 * final states kda_prefill_varlen computes from the same inputs, it returns dL/dq, dL/dk, dL/dv, dL/dg,
 * dL/dbeta and dL/dS_0.  The forward is recomputed inside the call (nothing is saved between the two);
 * the chunk algebra it differentiates is the one of kda_prefill_varlen.  With bf16 inputs the chunk-to-chunk
 * chains (the entry states and U forward, the state gradient dS' and dU in reverse) run on the tensor cores
 * in segments (split-bf16 products, fp32 accumulation) and the state products dO S^T, dU S^T, U dS'^T and
 * dO U^T likewise; the chunk-parallel rest is fp32 on the CUDA cores (fp32 inputs: all but the state
 * products).  Pair decays e^(G_t - G_s) are taken through the chunk's last token while the chunk's decay
 * span stays within e^80, else at 16-token references, and a block that would exceed e^80 takes them one
 * by one (its (sequence, head) then runs the CUDA-core chains); g >= -5 keeps every block within range.
 */
typedef struct {
  const void* q;             /* [T][H][dk] in_dtype */
  const void* k;             /* [T][H][dk] in_dtype */
  const void* v;             /* [T][H][dv] in_dtype */
  const float* g;            /* [T][H][dk] log-decay, <= 0 */
  const float* beta;         /* [T][H] */
  kda_dtype in_dtype;        /* also the dtype of d_out */
  int64_t T;                 /* total packed tokens (host) */
  int H, dk, dv;             /* dk = dv = 128 (KDA_ERR_UNSUPPORTED otherwise) */
  int N;                     /* sequences (host), <= 65535 */
  const int32_t* cu_seqlens; /* int32[N+1] device */
  int32_t max_seqlen;        /* host: an upper bound on every sequence length */
  const float* pool;         /* [num_slots][H][dk][dv]: initial states (read only), unless init_zero */
  int32_t num_slots;
  const int32_t* slot_ids;   /* int32[N] device, unless init_zero */
  int init_zero;             /* nonzero: every sequence starts from a zero state (pool, slot_ids unused) */
  const void* d_out;         /* [T][H][dv] in_dtype: dL/do */
  const float* d_final;      /* [N][H][dk][dv] fp32 dL/dS_T, or NULL for zero */
  float* dq;                 /* [T][H][dk] fp32 outputs */
  float* dk_out;             /* [T][H][dk] */
  float* dv_out;             /* [T][H][dv] */
  float* dg;                 /* [T][H][dk] */
  float* dbeta;              /* [T][H] */
  float* d_init;             /* [N][H][dk][dv] fp32 dL/dS_0, or NULL (not written) */
  void* workspace;           /* >= kda_backward_workspace_size(a) bytes of device scratch, 256-byte aligned */
  size_t workspace_bytes;
  int32_t* dev_status;       /* optional int32[2] */
} kda_backward_args;

/* sizeof(kda_backward_args), so a binding can check its mirror of the struct. */
size_t kda_backward_args_bytes(void);

/* Workspace of kda_prefill_backward, with n = (ceil(T/64) + N) * H chunk records: n * 574720 bytes of fp32
 * intermediates, then the tensor-core passes' scratch: n * 148480 bytes of operand records and
 * N * P * H * 196608 bytes of segment maps and entry states (P = max(1, 152 / H) segments per sequence), then
 * N * H int32 flags; the first two parts are rounded up to 1024 bytes, the last to 256. */
size_t kda_backward_workspace_size(const kda_backward_args* a);

/*
 * kda_prefill_backward -- enqueue the backward.  Every output element of a token of a listed sequence is
 * written; dq, dk, dg are written for all dk channels.  A slot id out of range sets KDA_DEV_SLOT_OOB and
 * that sequence is differentiated from a zero initial state; malformed cu_seqlens set KDA_DEV_SEQ_OOB and
 * that sequence's outputs are not written.  The work counter counts (token x head) pairs.
 */
kda_status kda_prefill_backward(const kda_backward_args* a, kda_stream_t stream);

/*
 * Fused decode front/back-end: one decode token through the short causal convolution, the KDA step and the
 * gated output norm in one launch.
 * Source: "SGLang and Miles: day-0 support for Kimi K3", section "kernels" (the fused Conv + KDA + Onorm
 * decode kernel); "Kimi K3: Architecture and SGLang Day-0 Support", KDA math box (the log-decay kept above
 * g_min = -5 by a scaled sigmoid; an input-dependent full-rank output gate).  The pages give no formula for
 * the convolution or the norm; this library's reading, per request b and head:
 *   q, k, v = SiLU(conv(x_q)), SiLU(conv(x_k)), SiLU(conv(x_v)), conv(x)_c = sum_tau w[c][tau] x_{t-3+tau, c}
 *             (the three previous inputs x_{t-3..t-1} of each stream come from conv_state, which then
 *             advances by one token);
 *   q <- q / sqrt(|q|^2 + 1e-6),  k <- k / sqrt(|k|^2 + 1e-6);  g = -5 sigmoid(a);  beta = sigmoid(b);
 *   o = the KDA step from pool[slot] (as kda_decode_step; pool updated in place);
 *   out = o / sqrt(mean_c o_c^2 + norm_eps) * norm_w * sigmoid(z).
 */
typedef struct {
  const void* xq;         /* [B][H][128] in_dtype: projected query, before the convolution */
  const void* xk;         /* [B][H][128] in_dtype */
  const void* xv;         /* [B][H][128] in_dtype */
  const float* a;         /* [B][H][128] decay logits */
  const float* b;         /* [B][H] write-strength logits */
  const void* z;          /* [B][H][128] in_dtype: output-gate logits */
  kda_dtype in_dtype;
  int B, H, dk, dv;       /* dk = dv = 128 (KDA_ERR_UNSUPPORTED otherwise) */
  float* pool;            /* [num_slots][H][128][128] */
  int32_t num_slots;
  const int32_t* slot_ids; /* int32[B] device */
  float* conv_state;      /* [num_slots][H][3][3][128] fp32: per stream (q, k, v) the 3 previous inputs,
                             oldest first; read and advanced in place */
  const float* conv_w;    /* [3][H][128][4] fp32 taps; tap 3 multiplies the current input */
  const float* norm_w;    /* [128] fp32 */
  float norm_eps;
  void* out;              /* [B][H][128] out_dtype */
  kda_dtype out_dtype;
  int32_t* dev_status;    /* optional int32[2]; the work counter counts (request x head) units */
} kda_fused_decode_args;

/* sizeof(kda_fused_decode_args), so a binding can check its mirror of the struct. */
size_t kda_fused_decode_args_bytes(void);

/* kda_fused_decode -- enqueue the fused decode; an out-of-range slot id sets KDA_DEV_SLOT_OOB and that
 * request is skipped (no state, carried input or output touched). */
kda_status kda_fused_decode(const kda_fused_decode_args* a, kda_stream_t stream);

/*
 * KCP across GPUs: one sequence split into contiguous shards held by W GPUs (ranks), rank r holding the
 * tokens after those of ranks 0..r-1.
 * Source: "Kimi K3 training and serving infra" (marsggbo blog), section 4.2 "KCP: pass fixed-size
 * transition information": each rank computes its shard's cumulative transition M and the state S~ it
 * produces from a zero input state; one all-gather of these fixed-size fragments (2 x 64 KB per head at
 * d = 128) and a local prefix scan give every rank its exact entry state; each rank then computes its
 * outputs.  The exchange itself is the caller's (e.g. torch.distributed); these calls are the per-rank
 * compute around it.  Per rank (kda_prefill_args describing the rank's shard as N sequences, normally one):
 *   1. kda_prefill_records (tensor-core path), then kda_kcp_fragments: the fragment of every segment of
 *      every sequence, the last included, into frag_out [N][P][H][dk][dv + dk] (S~ | M), P as for
 *      kda_prefill_segmented (one segment when segment_len >= the shard length);
 *   2. all-gather the fragments of all ranks (rank order);
 *   3. kda_kcp_scan over the gathered fragments: entries[0] = s0, entries[p+1] = M_p entries[p] + S~_p;
 *   4. kda_kcp_outputs: outputs and final states from the rank's entry states (entries [N][P][H][dk][dv]),
 *      reusing the records of step 1 (same workspace); the final state goes to pool[slot_ids[i]].
 */
kda_status kda_kcp_fragments(const kda_prefill_args* a, int32_t segment_len, float* frag_out, kda_stream_t stream);
/* frags [P][H][dk][dv + dk] fp32; s0 [H][dk][dv] fp32 or NULL (zero); entries [P][H][dk][dv] fp32. */
kda_status kda_kcp_scan(const float* frags, int32_t P, int H, int dk, int dv, const float* s0, float* entries,
                        int32_t* dev_status, kda_stream_t stream);
kda_status kda_kcp_outputs(const kda_prefill_args* a, int32_t segment_len, const float* entries,
                           kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
