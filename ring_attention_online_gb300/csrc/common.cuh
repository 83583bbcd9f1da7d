// Shared host/device declarations of the library's kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/attn.h"

namespace attn {

// Device status word bits (one word per translation unit that launches
// kernels; attn_last_device_status() collects and clears all of them).
enum : unsigned int {
  kStatusTimeout = 1u,       // some bounded wait gave up
  kStatusDeviceInput = 2u,   // malformed device-side input (seq_offsets)
  kStatusBounds = 4u,        // checked builds: an index or tile coordinate out of its extent (access skipped)
  kStatusSiteShift = 8u,     // bits 8..23: which wait gave up (diagnostics)
};

// A bounded wait gives up after this long; each step of a kernel waits for
// microseconds, so only a broken pipeline ever reaches it.
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s

// kModeWindow is dense prefill with a causal sliding window (a separate
// instantiation, so the other modes carry none of its checks)
enum PrefillMode : int { kModeDense = 0, kModePartial = 1, kModeJagged = 2, kModeWindow = 3 };

struct PrefillParams {
  // outputs
  void* o;         // dense / jagged: normalised O in the input dtype
  float* lse;      // nullable
  float* m_out;    // partial: m [B,h_q,S_q]
  float* l_out;    // partial: l [B,h_q,S_q]
  float* o_part;   // partial: unnormalised O fp32 [B,S_q,h_q,D]
  // sizes (jagged: B = 1, S_q = S_kv = total_tokens, h_q = h_kv = H)
  int B, S_q, S_kv, h_q, h_kv, group;
  int causal, num_chunks;
  int pair_heads;  // paired kernel: the two Q sub-tiles are heads (h, h+1) at one Q tile (else Q tiles 2t, 2t+1)
  // paired kernel (persistent), dense / partial: n_items = n_qt * n_y * B work
  // items over n_qt Q tiles (128 rows with pair_heads, else 256) and n_y head
  // pairs (pair_heads) or heads
  int n_items, n_qt, n_y;
  int q_pos0, kv_pos0, kv_lo, kv_hi;  // dense / partial key range and positions
  int window;                         // kModeWindow: query q sees keys q - window .. q
  float scale_log2;                   // softmax scale * log2(e)
  // jagged worklist: item count, unit count; items {seq_begin, seq_len, tile_start,
  // tile_extent}; units {first item, item count}, one per sequence
  const int* work_count;
  const int4* work_items;
  const int2* work_units;
  unsigned int* status;
};

// Host-side launchers (one translation unit per head dimension).
attn_status_t launch_prefill_d64(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                 const CUtensorMap& mv, int mode, bool bf16, dim3 grid, cudaStream_t s);
attn_status_t launch_prefill_d128(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                  const CUtensorMap& mv, int mode, bool bf16, dim3 grid, cudaStream_t s);
attn_status_t launch_prefill_d256(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                  const CUtensorMap& mv, int mode, bool bf16, dim3 grid, cudaStream_t s);
unsigned int prefill_d64_take_status(cudaStream_t s);
unsigned int prefill_d128_take_status(cudaStream_t s);
unsigned int prefill_d256_take_status(cudaStream_t s);

// Merge of stacked partial triplets (also the second decode kernel).
attn_status_t launch_merge(const float* m, const float* l, const float* o, int C, int B, int S_q, int H, int D,
                           void* out, bool out_bf16, float* lse, cudaStream_t s);

// Jagged worklist builder; beyond 1024 sequences it uses `scratch`
// (worklist_scratch_bytes(num_seqs) bytes of device memory, 8-byte aligned).
constexpr int kWorklistBuckets = 64;  // tile-count buckets of the ordered worklist
attn_status_t launch_worklist(const int32_t* seq_offsets, int num_seqs, int total_tokens, int max_seqlen,
                              int block_m, int* count_and_items, int max_items, int2* scratch, cudaStream_t s);
size_t worklist_scratch_bytes(int num_seqs);
unsigned int worklist_take_status(cudaStream_t s);
attn_status_t launch_selftest_timeout(uint64_t timeout_ns, cudaStream_t s);
attn_status_t launch_selftest_bounds(int* buf, cudaStream_t s);
attn_status_t launch_probe_mma(unsigned long long* out, int groups, cudaStream_t s);

// Split-KV decode partials; with `counters` (B * h_kv zeroed ints) the last
// CTA of each (batch, KV head) also merges the partials into `out` and `lse`.
attn_status_t launch_decode_partial(const void* q, const CUtensorMap& mk, const CUtensorMap& mv, float* m, float* l,
                                    float* o, int B, int S_kv, int h_q, int h_kv, int D, bool bf16, float scale_log2,
                                    int num_splits, int* counters, void* out, float* lse, cudaStream_t s);
unsigned int decode_take_status(cudaStream_t s);
unsigned int merge_take_status(cudaStream_t s);

}  // namespace attn
