// C ABI of libattn.so: argument validation, tensor-map encoding and launches.
// Every public function checks its arguments on the host and returns a status
// before anything reaches the device; nothing here allocates device memory.
#include <math.h>
#include <mutex>

#include "checked.cuh"
#include "common.cuh"
#include "schedule.cuh"

namespace attn {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 4-D map over a dense [B, S, H, D] tensor of 16-bit elements, read as boxes
// of `box_rows` tokens x 64 columns (128 bytes, 128-byte swizzle) of one head.
bool make_map(CUtensorMap* map, const void* ptr, bool bf16, int D, int H, long long S, int B, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(S > 0 ? S : 1), (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)(S > 0 ? S : 1) * H * D * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
             const_cast<void*>(ptr), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool head_dim_ok(int D) { return D == 64 || D == 128 || D == 256; }
bool dtype_ok(attn_dtype_t d) { return d == ATTN_FP16 || d == ATTN_BF16; }
bool scale_ok(float s) { return isfinite(s) && s > 0.f; }
constexpr float kLog2e = 1.4426950408889634f;

// Head dims 64 and 128 run two 128-row Q sub-tiles per CTA (query heads h, h+1 of
// one KV group when the group size is even, else Q tiles 2t, 2t+1 of one head);
// head dim 256 runs the same pairing over the two CTAs of a cluster (two of its
// O tiles do not fit in one CTA's TMEM), each CTA one 128-row Q tile.  Either
// way a jagged item is 256 rows.
bool paired(int D) { return D <= 128; }
int jagged_block(int) { return 2 * ATTN_BLOCK_M; }
// Keys of a K tile each CTA of a head-dim-256 pair loads (the pair splits the
// tile's keys between its CTAs).
int k_box_rows(int D) { return paired(D) ? ATTN_BLOCK_N : ATTN_BLOCK_N / 2; }

// Streaming multiprocessors of the current device (the persistent grid size).
int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

// Persistent grid: one CTA per SM, or fewer when there are fewer items.
dim3 persistent_grid(long long items) {
  const long long g = items < sm_count() ? items : sm_count();
  return dim3((unsigned)(g > 0 ? g : 1));
}

// Persistent grid of CTA pairs: one pair per two SMs, or fewer when there are
// fewer units.
dim3 persistent_pair_grid(long long units) {
  const long long pairs = sm_count() / 2 > 0 ? sm_count() / 2 : 1;
  const long long g = units < pairs ? units : pairs;
  return dim3((unsigned)(2 * (g > 0 ? g : 1)));
}

// Fills the work-item decomposition of the paired kernel and its grid (one
// item per CTA); the head-dim-256 kernel runs one CTA pair per two SMs over
// units of up to two 256-row pair items of one (batch, head or head pair).  False when the item count does not fit a
// 32-bit item index.
bool dense_grid(PrefillParams& p, int D, dim3* grid) {
  if (!paired(D)) {
    // CTA pairs, persistent over units of up to two pair items (see prefill_cta2_kernel.cuh)
    const long long units = cta2_units(p.B, p.S_q, p.h_q, p.pair_heads);
    const long long pairs = sm_count() / 2 > 0 ? sm_count() / 2 : 1;
    if (2 * ((units + pairs - 1) / pairs) > 0x7fffffffLL) return false;
    *grid = persistent_pair_grid(units);
    return true;
  }
  const int rows = p.pair_heads ? ATTN_BLOCK_M : 2 * ATTN_BLOCK_M;
  p.n_qt = (p.S_q + rows - 1) / rows;
  p.n_y = p.pair_heads ? p.h_q / 2 : p.h_q;
  const long long items = (long long)p.n_qt * p.n_y * p.B;
  if (items > 0x7fffffffLL) return false;
  p.n_items = (int)items;
  *grid = dim3((unsigned)items);  // one item per CTA: see prefill_pair_kernel.cuh
  return true;
}

attn_status_t launch_prefill(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                             const CUtensorMap& mv, int mode, bool bf16, int D, dim3 grid, cudaStream_t s) {
  switch (D) {
    case 64: return launch_prefill_d64(p, mq, mk, mv, mode, bf16, grid, s);
    case 128: return launch_prefill_d128(p, mq, mk, mv, mode, bf16, grid, s);
    case 256: return launch_prefill_d256(p, mq, mk, mv, mode, bf16, grid, s);
  }
  return ATTN_ERR_UNSUPPORTED;
}

// Shared checks of the dense prefill-shaped calls.
attn_status_t check_dense(const void* q, const void* k, const void* v, int B, int S_q, int S_kv, int h_q, int h_kv,
                          int D, attn_dtype_t dtype, float scale, int causal) {
  if (!q || !k || !v) return ATTN_ERR_INVALID_ARG;
  if (B < 0 || S_q < 0 || S_kv < 0 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!dtype_ok(dtype) || !scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16)) return ATTN_ERR_INVALID_ARG;
  if (!head_dim_ok(D)) return ATTN_ERR_UNSUPPORTED;
  if ((long long)S_q > 0x7fffff80LL || (long long)S_kv > 0x7fffff80LL) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B > 65535 || (long long)h_q > 65535) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

size_t jagged_max_items(int num_seqs, int total_tokens, int block_m = ATTN_BLOCK_M) {
  // sum_b ceil(L_b / block_m) <= (T + num_seqs * (block_m - 1)) / block_m
  return ((size_t)total_tokens + (size_t)num_seqs * (block_m - 1)) / block_m;
}

// attn_prefill and attn_prefill_window: window < 0 is none.
attn_status_t prefill_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_q,
                           int S_kv, int h_q, int h_kv, int D, attn_dtype_t dtype, float scale, int causal,
                           int window, int num_chunks, attn_stream_t stream) {
  attn_status_t st = check_dense(q, k, v, B, S_q, S_kv, h_q, h_kv, D, dtype, scale, causal);
  if (st != ATTN_OK) return st;
  if (!o || !aligned(o, 16) || (lse && !aligned(lse, 4)) || num_chunks < 1) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || S_q == 0) return ATTN_OK;
  const bool bf16 = dtype == ATTN_BF16;
  PrefillParams p{};
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.S_q = S_q;
  p.S_kv = S_kv;
  p.h_q = h_q;
  p.h_kv = h_kv;
  p.group = h_q / h_kv;
  p.causal = causal;
  p.num_chunks = num_chunks;
  p.q_pos0 = 0;
  p.kv_pos0 = 0;
  p.kv_lo = 0;
  p.kv_hi = S_kv;
  p.scale_log2 = scale * kLog2e;
  p.pair_heads = (p.group % 2) == 0;
  p.window = window;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, bf16, D, h_q, S_q, B, ATTN_BLOCK_M) || !make_map(&mk, k, bf16, D, h_kv, S_kv, B, k_box_rows(D)) ||
      !make_map(&mv, v, bf16, D, h_kv, S_kv, B, ATTN_BLOCK_N))
    return ATTN_ERR_CUDA;
  dim3 grid;
  if (!dense_grid(p, D, &grid)) return ATTN_ERR_UNSUPPORTED;
  // the paired kernel's window launches are persistent over its items
  if (paired(D) && window >= 0) grid = persistent_grid(p.n_items);
  return launch_prefill(p, mq, mk, mv, window >= 0 ? kModeWindow : kModeDense, bf16, D, grid,
                        reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

attn_status_t attn_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_q,
                           int S_kv, int h_q, int h_kv, int D, attn_dtype_t dtype, float scale, int causal,
                           int num_chunks, attn_stream_t stream) {
  return prefill_impl(q, k, v, o, lse, B, S_q, S_kv, h_q, h_kv, D, dtype, scale, causal, -1, num_chunks, stream);
}

attn_status_t attn_prefill_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_q,
                                  int S_kv, int h_q, int h_kv, int D, attn_dtype_t dtype, float scale, int window,
                                  int num_chunks, attn_stream_t stream) {
  if (window < 0) return ATTN_ERR_INVALID_ARG;
  return prefill_impl(q, k, v, o, lse, B, S_q, S_kv, h_q, h_kv, D, dtype, scale, 1, window, num_chunks, stream);
}

attn_status_t attn_partial(const void* q, const void* k, const void* v, float* m, float* l, float* o_unnorm,
                           int B, int S_q, int S_kv, int h_q, int h_kv, int D, attn_dtype_t dtype, float scale,
                           int causal, int q_pos0, int kv_begin, int kv_end, attn_stream_t stream) {
  attn_status_t st = check_dense(q, k, v, B, S_q, S_kv, h_q, h_kv, D, dtype, scale, causal);
  if (st != ATTN_OK) return st;
  if (!m || !l || !o_unnorm || !aligned(m, 4) || !aligned(l, 4) || !aligned(o_unnorm, 16)) return ATTN_ERR_INVALID_ARG;
  if (kv_begin < 0 || kv_end < kv_begin || kv_end > S_kv) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || S_q == 0) return ATTN_OK;
  const bool bf16 = dtype == ATTN_BF16;
  PrefillParams p{};
  p.m_out = m;
  p.l_out = l;
  p.o_part = o_unnorm;
  p.B = B;
  p.S_q = S_q;
  p.S_kv = S_kv;
  p.h_q = h_q;
  p.h_kv = h_kv;
  p.group = h_q / h_kv;
  p.causal = causal;
  p.num_chunks = 1;
  p.q_pos0 = q_pos0;
  p.kv_pos0 = 0;
  p.kv_lo = kv_begin;
  p.kv_hi = kv_end;
  p.scale_log2 = scale * kLog2e;
  p.pair_heads = (p.group % 2) == 0;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, bf16, D, h_q, S_q, B, ATTN_BLOCK_M) || !make_map(&mk, k, bf16, D, h_kv, S_kv, B, k_box_rows(D)) ||
      !make_map(&mv, v, bf16, D, h_kv, S_kv, B, ATTN_BLOCK_N))
    return ATTN_ERR_CUDA;
  dim3 grid;
  if (!dense_grid(p, D, &grid)) return ATTN_ERR_UNSUPPORTED;
  return launch_prefill(p, mq, mk, mv, kModePartial, bf16, D, grid, reinterpret_cast<cudaStream_t>(stream));
}

attn_status_t attn_merge(const float* m, const float* l, const float* o_unnorm, int C, int B, int S_q, int H, int D,
                         void* out, attn_dtype_t out_dtype, float* lse, attn_stream_t stream) {
  if (!m || !l || !o_unnorm || !out) return ATTN_ERR_INVALID_ARG;
  if (C < 1 || B < 0 || S_q < 0 || H < 1) return ATTN_ERR_INVALID_ARG;
  if (!dtype_ok(out_dtype)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(m, 4) || !aligned(l, 4) || !aligned(o_unnorm, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4)))
    return ATTN_ERR_INVALID_ARG;
  if (!head_dim_ok(D)) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || S_q == 0) return ATTN_OK;
  return launch_merge(m, l, o_unnorm, C, B, S_q, H, D, out, out_dtype == ATTN_BF16, lse,
                      reinterpret_cast<cudaStream_t>(stream));
}

size_t attn_jagged_workspace_bytes(int num_seqs, int total_tokens, int max_seqlen) {
  (void)max_seqlen;
  if (num_seqs < 0 || total_tokens < 0) return 0;
  // counts, items (sized for 128-row Q tiles, the larger count), one unit per
  // sequence, then the builder's per-CTA table (beyond 1024 sequences)
  return 16 + 16 * jagged_max_items(num_seqs, total_tokens) + (((size_t)num_seqs * 8 + 15) & ~size_t(15)) +
         worklist_scratch_bytes(num_seqs);
}

attn_status_t attn_jagged(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int32_t* seq_offsets, int num_seqs, int total_tokens, int max_seqlen, int H, int D,
                          attn_dtype_t dtype, float scale, int causal, void* workspace, size_t workspace_bytes,
                          attn_stream_t stream) {
  attn_status_t st = check_dense(q, k, v, 1, total_tokens, total_tokens, H, H, D, dtype, scale, causal);
  if (st != ATTN_OK) return st;
  if (!o || !seq_offsets || !aligned(o, 16) || (lse && !aligned(lse, 4)) || !aligned(seq_offsets, 4))
    return ATTN_ERR_INVALID_ARG;
  if (num_seqs < 0 || max_seqlen < 0) return ATTN_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_tokens == 0) return ATTN_OK;
  if (!workspace || !aligned(workspace, 16) || workspace_bytes < attn_jagged_workspace_bytes(num_seqs, total_tokens, max_seqlen))
    return ATTN_ERR_INVALID_ARG;
  const int block = jagged_block(D);
  const size_t max_items = jagged_max_items(num_seqs, total_tokens, block);
  if (max_items > 0x7fffffffULL || H > 65535) return ATTN_ERR_UNSUPPORTED;
  if (paired(D) && (unsigned long long)num_seqs * H > 0x7fffffffULL) return ATTN_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* wl = static_cast<int*>(workspace);
  // the builder's table follows this launch's units (its item count is at most
  // the one the workspace size allows for)
  int2* wl_scratch = reinterpret_cast<int2*>(reinterpret_cast<char*>(workspace) + 16 + 16 * max_items +
                                             (((size_t)num_seqs * 8 + 15) & ~size_t(15)));
  st = launch_worklist(seq_offsets, num_seqs, total_tokens, max_seqlen, block, wl, (int)max_items, wl_scratch, s);
  if (st != ATTN_OK) return st;
  const bool bf16 = dtype == ATTN_BF16;
  PrefillParams p{};
  p.o = o;
  p.lse = lse;
  p.B = 1;
  p.S_q = total_tokens;
  p.S_kv = total_tokens;
  p.h_q = H;
  p.h_kv = H;
  p.group = 1;
  p.causal = causal;
  p.num_chunks = 1;
  p.scale_log2 = scale * kLog2e;
  p.work_count = wl;
  p.work_items = reinterpret_cast<const int4*>(wl + 4);
  p.work_units = reinterpret_cast<const int2*>(wl + 4 + 4 * max_items);
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, bf16, D, H, total_tokens, 1, ATTN_BLOCK_M) ||
      !make_map(&mk, k, bf16, D, H, total_tokens, 1, k_box_rows(D)) ||
      !make_map(&mv, v, bf16, D, H, total_tokens, 1, ATTN_BLOCK_N))
    return ATTN_ERR_CUDA;
  // paired kernel: persistent over (sequence, head) units; CTA pairs: one pair per (item, head)
  if (!paired(D) && 2 * max_items > 0x7fffffffULL) return ATTN_ERR_UNSUPPORTED;
  const dim3 grid = paired(D) ? persistent_grid((long long)num_seqs * H) : dim3((unsigned)(2 * max_items), H, 1);
  return launch_prefill(p, mq, mk, mv, kModeJagged, bf16, D, grid, s);
}

size_t attn_decode_workspace_bytes(int B, int h_q, int D, int num_splits) {
  if (B < 0 || h_q < 0 || D < 0 || num_splits < 0) return 0;
  const size_t rows = (size_t)num_splits * B * h_q;
  const size_t ml = (rows * 2 * sizeof(float) + 15) & ~size_t(15);
  const size_t counters = ((size_t)B * h_q * sizeof(int) + 15) & ~size_t(15);  // B * h_kv <= B * h_q used
  return ml + rows * D * sizeof(float) + counters;
}

attn_status_t attn_decode_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                  int S_kv, int h_q, int h_kv, int D, attn_dtype_t dtype, float scale,
                                  int num_splits, void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  attn_status_t st = check_dense(q, k, v, B, 1, S_kv, h_q, h_kv, D, dtype, scale, 0);
  if (st != ATTN_OK) return st;
  if (!o || !aligned(o, 16) || (lse && !aligned(lse, 4)) || num_splits < 1) return ATTN_ERR_INVALID_ARG;
  if (h_q / h_kv > 16) return ATTN_ERR_UNSUPPORTED;
  if (B == 0) return ATTN_OK;
  if (num_splits > 65535 || h_kv > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 16) || workspace_bytes < attn_decode_workspace_bytes(B, h_q, D, num_splits))
    return ATTN_ERR_INVALID_ARG;
  const bool bf16 = dtype == ATTN_BF16;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t rows = (size_t)num_splits * B * h_q;
  float* wm = static_cast<float*>(workspace);
  float* wl = wm + rows;
  float* wo = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((rows * 2 * sizeof(float) + 15) & ~size_t(15)));
  int* counters = reinterpret_cast<int*>(wo + rows * D);
  CUtensorMap mk, mv;
  if (!make_map(&mk, k, bf16, D, h_kv, S_kv, B, 64) || !make_map(&mv, v, bf16, D, h_kv, S_kv, B, 64))
    return ATTN_ERR_CUDA;
  // the fused merge counts the chunks of each (batch, KV head) from zero
  if (cudaMemsetAsync(counters, 0, (size_t)B * h_kv * sizeof(int), s) != cudaSuccess) return ATTN_ERR_CUDA;
  return launch_decode_partial(q, mk, mv, wm, wl, wo, B, S_kv, h_q, h_kv, D, bf16, scale * kLog2e, num_splits,
                               counters, o, lse, s);
}

attn_status_t attn_last_device_status(attn_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const unsigned int v = prefill_d64_take_status(s) | prefill_d128_take_status(s) | prefill_d256_take_status(s) |
                         worklist_take_status(s) | decode_take_status(s) | merge_take_status(s);
  if (v & kStatusTimeout) return ATTN_ERR_TIMEOUT;
  if (v & kStatusDeviceInput) return ATTN_ERR_DEVICE_INPUT;
  if (v & kStatusBounds) return ATTN_ERR_BOUNDS;
  return ATTN_OK;
}

attn_status_t attn_probe_mma_cycles(unsigned long long* cycles, int groups, attn_stream_t stream) {
  if (!cycles || !aligned(cycles, 8) || groups < 1 || groups > (1 << 20)) return ATTN_ERR_INVALID_ARG;
  return launch_probe_mma(cycles, groups, reinterpret_cast<cudaStream_t>(stream));
}

int attn_build_checked(void) { return ATTN_CHECKED ? 1 : 0; }

attn_status_t attn_selftest_bounds(int* buf, attn_stream_t stream) {
  if (!buf || !aligned(buf, 4)) return ATTN_ERR_INVALID_ARG;
  if (!ATTN_CHECKED) return ATTN_ERR_UNSUPPORTED;
  return launch_selftest_bounds(buf, reinterpret_cast<cudaStream_t>(stream));
}

attn_status_t attn_selftest_wait_timeout(uint64_t timeout_ns, attn_stream_t stream) {
  if (timeout_ns < 1000000ull || timeout_ns > 10000000000ull) return ATTN_ERR_INVALID_ARG;
  return launch_selftest_timeout(timeout_ns, reinterpret_cast<cudaStream_t>(stream));
}

const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA call failed";
    case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
    case ATTN_ERR_DEVICE_INPUT: return "device-side input check failed";
    case ATTN_ERR_BOUNDS: return "device-side bounds check failed (checked build)";
  }
  return "unknown status";
}

attn_status_t attn_tile_walk(int q_lo, int q_hi, int kv_lo, int kv_hi, int block_n, int causal, int num_chunks,
                             int q_pos0, int kv_pos0, int window, int* chunk, int* tile_start, int* mask_end,
                             int max_tiles, int* n_tiles) {
  if (!n_tiles || block_n < 1 || num_chunks < 1 || q_hi < q_lo || kv_hi < kv_lo || max_tiles < 0 ||
      (max_tiles > 0 && (!chunk || !tile_start || !mask_end)) || (causal != 0 && causal != 1) || window < -1 ||
      (window >= 0 && !causal))
    return ATTN_ERR_INVALID_ARG;
  TileWalk w;
  w.init(q_lo, q_hi, kv_lo, kv_hi, q_pos0, kv_pos0, causal, num_chunks, block_n, window);
  if (ring_walk_is_rotation(kv_lo, kv_hi, num_chunks, block_n)) {
    // the paired kernel walks such rings as a rotated single-chunk walk; report
    // that walk, with each tile's chunk and the chunk's own tail limit
    TileWalk w1;
    w1.init(q_lo, q_hi, kv_lo, kv_hi, q_pos0, kv_pos0, causal, 1, block_n, window);
    LinearWalk lw;
    lw.init(w1, ring_first_key(q_lo, kv_lo, kv_hi, q_pos0, kv_pos0, num_chunks), block_n);
    const int len = kv_hi - kv_lo;
    const int chunk_len = (len + num_chunks - 1) / num_chunks;
    for (int i = 0; i < lw.n && i < max_tiles; ++i) {
      int st, me;
      lw.next(st, me, block_n);
      const int c = (st - kv_lo) / chunk_len;
      const long long chunk_hi = (long long)kv_lo + (long long)(c + 1) * chunk_len;
      chunk[i] = c;
      tile_start[i] = st;
      mask_end[i] = (int)(me < chunk_hi ? me : chunk_hi);
    }
    *n_tiles = lw.n;
    return ATTN_OK;
  }
  const int total = w.count();
  int i = 0, c, st, me;
  while (i < max_tiles && w.next(c, st, me)) {
    chunk[i] = c;
    tile_start[i] = st;
    mask_end[i] = me;
    ++i;
  }
  *n_tiles = total;
  return ATTN_OK;
}

}  // extern "C"
