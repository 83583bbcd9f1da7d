/*
 * attn.h - C ABI of libattn.so: exact softmax attention computed blockwise over
 * KV tiles and chunks, with the running (m, l, O) triplet merged by online
 * softmax, on one NVIDIA GB300 (sm_103a).
 *
 * Sources, by page title and section:
 *   [PREFILL]  "kernbench2 _gqa_prefill_long.py" - gqa_prefill_long_kernel:
 *              step 0 partial (scores = Q.K^T, m = rowmax, exp(scores - m),
 *              l = rowsum, O = exp_scores . V), ring steps 1..C-1 (KV block
 *              rotation and the online-softmax merge), final normalise O / l.
 *   [DECODE]   "kernbench2 _attention_mesh_mlo.py" - one-shot local partial of
 *              a sequence-sharded KV, the (m, l, o) merge, final O := o / l.
 *   [BOUNDS]   "[pallas] Support dependent Tile.end bounds in Pallas" - inner KV
 *              loop over [kv_begin, min(kv_end, tile_q.end)), trip count
 *              cdiv(active_end - begin, block_k), tail mask, flattened jagged
 *              worklists, jagged KV end seq_offsets[seq_idx + 1].
 *
 * Conventions for every call
 *   Layouts are token-major and dense (no strides):
 *     Q, O            [B, S_q, h_q, D]      K, V  [B, S_kv, h_kv, D]
 *     LSE, m, l       [B, h_q, S_q]  fp32   unnormalised O  [B, S_q, h_q, D] fp32
 *     jagged Q/K/V/O  [total_tokens, H, D]  jagged LSE      [H, total_tokens]
 *   Query head h reads KV head h / (h_q / h_kv) (contiguous groups).
 *   Scores are s = scale * q.k; LSE = ln sum_j exp(s_j) (natural log).
 *   Causal masking: key j is visible to query i iff pos(j) <= pos(i), with
 *   query and key positions in one index space (top-left alignment).
 *   A row that sees no key yields O = 0 and LSE = -inf; its partial triplet is
 *   the merge identity (m, l, O) = (-inf, 0, 0).
 *   Inputs are fp16 or bf16 (all of Q, K, V the same); accumulation is fp32;
 *   P is rounded to the input type before P.V; outputs O are rounded to the
 *   input type (nearest even).
 *
 *   Ownership: the caller owns every buffer and the stream; the library never
 *   allocates device memory.  Scratch space comes from the caller through a
 *   `workspace` argument sized by the matching *_workspace_bytes() helper.
 *   Every call is asynchronous on `stream` (0 = legacy default stream).
 *   Device pointers must be 16-byte aligned (LSE, m, l: 4-byte aligned).
 *
 *   Errors: every call returns an attn_status_t and never aborts.  Invalid
 *   arguments are rejected on the host before any launch.  Conditions only the
 *   device can see (a barrier wait that gave up, malformed seq_offsets) are
 *   recorded in a per-library device status word and reported, then cleared,
 *   by attn_last_device_status().
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* attn_stream_t; /* same object as cudaStream_t */

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad alignment, h_q % h_kv != 0, ... */
  ATTN_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels implement (e.g. D) */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, tensor map) */
  ATTN_ERR_TIMEOUT = 4,     /* a device-side wait gave up (reported by attn_last_device_status) */
  ATTN_ERR_DEVICE_INPUT = 5, /* device-side input check failed, e.g. non-monotone seq_offsets */
  ATTN_ERR_BOUNDS = 6        /* checked build: a kernel's index or tile coordinate left its extent */
} attn_status_t;

typedef enum { ATTN_FP16 = 0, ATTN_BF16 = 1 } attn_dtype_t;

/* Tile sizes of the prefill kernels: BLOCK_M query rows x BLOCK_N keys. */
#define ATTN_BLOCK_M 128
#define ATTN_BLOCK_N 128

/*
 * attn_prefill - causal or full prefill attention with a ring-order chunk walk.
 *   [PREFILL] (Algorithm paragraph of the kernel docstring; P6b ring rotation)
 *   [BOUNDS]  (dependent inner-loop end, trip count, tail mask)
 *
 * The KV sequence is cut into num_chunks chunks of ceil(S_kv / num_chunks) keys.
 * Each Q tile of ATTN_BLOCK_M rows visits the chunks in ring order (c0 + t) mod C,
 * starting at the chunk c0 = min(C-1, q_tile_start / chunk_len) that holds its
 * first position; the running (m, l, O) carries across chunks (the page's merge).
 * With causal = 1 a chunk whose first key lies after the tile's last query is
 * skipped, and inside a chunk only cdiv(min(chunk_end, q_tile_end) - chunk_start,
 * ATTN_BLOCK_N) KV tiles are visited (fully masked tiles are pruned, not masked).
 *
 *   q [B,S_q,h_q,D], k/v [B,S_kv,h_kv,D], o [B,S_q,h_q,D] (input dtype),
 *   lse [B,h_q,S_q] fp32 or NULL.  D in {64, 128, 256}.  num_chunks >= 1.
 *   S_q = 0 or B = 0 is a no-op; S_kv = 0 writes O = 0 and LSE = -inf.
 */
attn_status_t attn_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_q,
                           int S_kv, int h_q, int h_kv, int D, attn_dtype_t dtype, float scale, int causal,
                           int num_chunks, attn_stream_t stream);

/*
 * attn_prefill_window - causal prefill with a sliding window.
 *   [BOUNDS] ("Scalar minimum": the dependent lower bound max(kv_begin,
 *            tile_q.begin - window) deferred there to sliding-window support)
 *
 * As attn_prefill with causal = 1, except that key j is visible to query i only
 * if i - window <= j <= i: each query sees its own key and the `window` keys
 * before it.  Inside every chunk the walk starts at the first tile of the chunk's
 * ATTN_BLOCK_N grid that holds a key the Q tile's first row can see; tiles at the
 * window's lower edge are masked per row.  window >= S_kv is plain causal
 * attention.  window < 0 is ATTN_ERR_INVALID_ARG; other arguments as attn_prefill.
 */
attn_status_t attn_prefill_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_q,
                                  int S_kv, int h_q, int h_kv, int D, attn_dtype_t dtype, float scale, int window,
                                  int num_chunks, attn_stream_t stream);

/*
 * attn_partial - the partial triplet of one KV range (one ring step's partial).
 *   [PREFILL] (step 0 partial / per-step partial on the rotated KV block)
 *
 * Keys k[:, kv_begin:kv_end] sit at positions kv_begin..kv_end-1 (k's own index
 * space); query i sits at position q_pos0 + i.  Writes, per query row,
 *   m = max_j s_ij, l = sum_j exp(s_ij - m), o_unnorm = sum_j exp(s_ij - m) v_j
 * over the visible keys of the range (the identity (-inf, 0, 0) if none).
 *   m, l [B,h_q,S_q] fp32; o_unnorm [B,S_q,h_q,D] fp32.
 *   0 <= kv_begin <= kv_end <= S_kv.  To fill stacked partials [C, ...] pass
 *   pointers offset by c * (one partial's element count).
 */
attn_status_t attn_partial(const void* q, const void* k, const void* v, float* m, float* l, float* o_unnorm,
                           int B, int S_q, int S_kv, int h_q, int h_kv, int D, attn_dtype_t dtype, float scale,
                           int causal, int q_pos0, int kv_begin, int kv_end, attn_stream_t stream);

/*
 * attn_merge - fold C partial triplets per row and normalise.
 *   [PREFILL] (online-softmax merge into the running (m, l, O); final normalise)
 *   [DECODE]  (merge-from-W / merge-from-E; final normalize O := o / l)
 *
 * Per row: M = max_c m_c; l = sum_c l_c exp(m_c - M); O = sum_c o_c exp(m_c - M) / l;
 * LSE = M + ln l.  Partials with m_c = -inf contribute nothing; a row whose
 * partials are all empty gives O = 0, LSE = -inf.
 *   m, l [C,B,H,S_q] fp32; o_unnorm [C,B,S_q,H,D] fp32;
 *   out [B,S_q,H,D] in out_dtype; lse [B,H,S_q] fp32 or NULL.  D in {64,128,256}.
 */
attn_status_t attn_merge(const float* m, const float* l, const float* o_unnorm, int C, int B, int S_q, int H,
                         int D, void* out, attn_dtype_t out_dtype, float* lse, attn_stream_t stream);

/*
 * attn_jagged - variable-length causal (or full) self-attention over packed
 * sequences.
 *   [BOUNDS] (jagged KV end seq_offsets[seq_idx + 1]; flattened worklists with
 *            compute_end = min(source_end, compact_end) driving the trip count)
 *
 * Sequence b spans tokens [seq_offsets[b], seq_offsets[b+1]) and attends only to
 * itself.  Q tiles start at the sequence start.  A device kernel first builds the
 * flattened worklist from the device-resident seq_offsets into `workspace`: one
 * item per (sequence, Q tile) and one unit per sequence (its items, which are
 * contiguous).  The attention kernel then runs, for D = 64/128, one persistent
 * CTA per SM over (unit, head) pairs, a sequence's Q tiles back to back so its
 * K/V is re-read from L2 ("Grouping": successive Q items reuse the resident K/V
 * range); for D = 256 one CTA pair per (item, head).  No host synchronisation.
 * Workspace: int item count, int unit count, 8 bytes pad, the int4 items, then
 * the int2 units {first item, item count}; beyond 1024 sequences the builder
 * also keeps a table of per-CTA counts after the units.
 *   q/k/v/o [total_tokens,H,D]; lse [H,total_tokens] fp32 or NULL;
 *   seq_offsets int32 [num_seqs+1], device memory, non-decreasing, from 0 to at
 *   most total_tokens, every length <= max_seqlen (violations are reported as
 *   ATTN_ERR_DEVICE_INPUT by attn_last_device_status and their tokens are not
 *   written).  workspace >= attn_jagged_workspace_bytes(num_seqs, total_tokens,
 *   max_seqlen) bytes, 16-byte aligned.
 */
attn_status_t attn_jagged(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int32_t* seq_offsets, int num_seqs, int total_tokens, int max_seqlen, int H, int D,
                          attn_dtype_t dtype, float scale, int causal, void* workspace, size_t workspace_bytes,
                          attn_stream_t stream);
size_t attn_jagged_workspace_bytes(int num_seqs, int total_tokens, int max_seqlen);

/*
 * attn_decode_splitkv - one query per sequence against a long KV, split-KV.
 *   [DECODE] (KV sequence-sharded and read in place; one-shot local partial per
 *            shard; triplets merged; final normalize)
 *
 * The KV sequence is cut into num_splits chunks of ceil(S_kv / num_splits) keys
 * (trailing chunks may be empty: identity triplets).  One kernel computes a
 * partial (m, l, o) per (batch, query head, chunk) into `workspace`; the last CTA
 * to finish among the num_splits of a (batch, KV head) merges that group's
 * partials (as attn_merge) into o and lse in the same kernel.  Workspace layout:
 *   m [num_splits,B,h_q] fp32, l [num_splits,B,h_q] fp32 (16-byte aligned),
 *   o [num_splits,B,h_q,D] fp32, then B*h_q int32 counters (the call zeroes the
 *   first B*h_kv on `stream` before its kernel; size them with
 *   attn_decode_workspace_bytes).
 *   q [B,h_q,D]; k/v [B,S_kv,h_kv,D]; o [B,h_q,D]; lse [B,h_q] fp32 or NULL.
 *   D in {64,128,256}; h_q / h_kv <= 16.
 */
attn_status_t attn_decode_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                  int S_kv, int h_q, int h_kv, int D, attn_dtype_t dtype, float scale,
                                  int num_splits, void* workspace, size_t workspace_bytes, attn_stream_t stream);
size_t attn_decode_workspace_bytes(int B, int h_q, int D, int num_splits);

/*
 * attn_decode_splitkv_noalloc - attn_decode_splitkv without a workspace argument,
 * for callers that cannot allocate device memory: a program whose device memory is
 * owned by a host framework that gives it only its inputs and outputs, or a
 * latency-critical loop that must not call cudaMalloc/cudaFree (they can
 * synchronise the device) nor risk running out of memory mid-run.  No counterpart
 * on the pages: it only changes where the scratch lives.
 *
 * The partial triplets go to a fixed array of ATTN_NOALLOC_SCRATCH_BYTES in device
 * memory that is part of the library (present on every GPU that loads it, until
 * the process exits).  Nothing is allocated or freed.  Same arguments, layouts and
 * results as attn_decode_splitkv.  Returns ATTN_ERR_UNSUPPORTED when the partials,
 * attn_decode_workspace_bytes(B, h_q, D, num_splits), exceed the array.
 * The first call on a device looks up the array's device address (with that device
 * current) and keeps it for the device's current context; a later context on the
 * device (after a device reset) gets a fresh lookup on its first call.  Make the
 * first call on a device, and the first after a reset, before any stream capture.
 * All calls share the
 * array and it keeps the last call's contents (every entry a call reads is written
 * or zeroed by that call first); calls whose kernels overlap on the GPU race on it.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
attn_status_t attn_decode_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                          int S_kv, int h_q, int h_kv, int D, attn_dtype_t dtype, float scale,
                                          int num_splits, attn_stream_t stream);

/*
 * attn_last_device_status - synchronise `stream`, then return and clear the
 * device-side status (ATTN_ERR_TIMEOUT, ATTN_ERR_DEVICE_INPUT, ATTN_ERR_BOUNDS,
 * in that order of precedence) raised by any kernel of the library since the
 * previous call; ATTN_OK if none.
 */
attn_status_t attn_last_device_status(attn_stream_t stream);

/*
 * Checked builds.  The same sources compiled with ATTN_CHECKED=1 give
 * libattn_checked.so, a debug variant of this library: before every global
 * store, every TMA tile load and every read of a worklist entry its kernels
 * test the index or coordinate against the extent of its buffer (a tile's row
 * start may lie up to two tiles past the last row: such boxes read zeros, which
 * is how tail and empty tiles load).  A failed test records ATTN_ERR_BOUNDS in
 * the device status and the access is skipped (a tile load takes tile 0
 * instead), so the context stays usable.  No counterpart on the pages: it guards
 * the library's own indexing (the failure class of DMA copies started out of
 * step with their waits, which the ring-attention review thread warns about).
 *
 * attn_build_checked - 1 in the checked variant, 0 otherwise.
 * attn_selftest_bounds - checked variant only (else ATTN_ERR_UNSUPPORTED, no
 *   launch): one thread stores to index 1 of the one-element int buffer `buf`
 *   (device memory, 4-byte aligned, owned by the caller) through the store
 *   check, which records ATTN_ERR_BOUNDS and skips the store (buf is unchanged).
 *   Read the result with attn_last_device_status().
 */
int attn_build_checked(void);
attn_status_t attn_selftest_bounds(int* buf, attn_stream_t stream);

/*
 * attn_selftest_wait_timeout - failure-detection self-test.  Launches one thread
 * that waits on a shared-memory barrier nothing ever completes, through the same
 * bounded wait every kernel of the library uses, limited to timeout_ns
 * (1 ms .. 10 s).  The wait gives up, records ATTN_ERR_TIMEOUT in the device
 * status and the kernel returns normally, leaving the context usable; the
 * caller reads the status with attn_last_device_status().  Has no counterpart
 * on the pages: it tests this library's own wait discipline.
 */
attn_status_t attn_selftest_wait_timeout(uint64_t timeout_ns, attn_stream_t stream);

/*
 * attn_probe_mma_cycles - tensor-pipe rate probe.  One CTA issues groups x 8
 * back-to-back tcgen05.mma kind::f16 M=128 N=128 K=16 MMAs from one thread (bf16
 * operands in shared memory, fp32 accumulator in TMEM) and writes to cycles[0]
 * the SM clock cycles from the first issue to the completion of the last, and to
 * cycles[1] 0, or 1 if the bounded wait for that completion gave up.  cycles:
 * device memory, 2 x uint64, 8-byte aligned, owned by the caller.  groups in
 * [1, 1 << 20]; otherwise ATTN_ERR_INVALID_ARG.  128*128*16*2 / (cycles[0] /
 * (8 * groups)) is the per-SM dense bf16 rate that the nominal roofline
 * denominator is built from.  Has no counterpart on the pages.
 */
attn_status_t attn_probe_mma_cycles(unsigned long long* cycles, int groups, attn_stream_t stream);

/* Static description of a status code; never NULL. */
const char* attn_status_string(attn_status_t status);

/*
 * attn_tile_walk - host-side enumeration of the KV tiles one Q tile visits, by
 * the same scheduling code the kernels run (for tests and tooling).
 *   [BOUNDS] (dependent end, trip count); [PREFILL] (ring order, P6b)
 *
 * Q rows [q_lo, q_hi) at positions q_pos0 + i; keys [kv_lo, kv_hi) at positions
 * kv_pos0 + j, cut into num_chunks ring chunks; window >= 0 (causal only) applies
 * attn_prefill_window's sliding window, window = -1 none.  Writes up to max_tiles entries
 * (chunk, tile_start, mask_end) in visiting order, where mask_end is the first
 * key index that the tile's tail mask excludes, and stores the full count in
 * *n_tiles.  When the chunk length is a multiple of block_n, the ring visits
 * the tiles of the single-chunk walk in that walk's order rotated to the Q
 * tile's own chunk, and the entries come from that rotated walk (the one the
 * head-dim 64/128 kernels run), mask_end cut to the tile's chunk.  Returns
 * ATTN_ERR_INVALID_ARG on bad sizes or null pointers.
 */
attn_status_t attn_tile_walk(int q_lo, int q_hi, int kv_lo, int kv_hi, int block_n, int causal, int num_chunks,
                             int q_pos0, int kv_pos0, int window, int* chunk, int* tile_start, int* mask_end,
                             int max_tiles, int* n_tiles);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
