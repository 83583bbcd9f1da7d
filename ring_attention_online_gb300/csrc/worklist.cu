// Flattened jagged worklist, built on the device from device-resident
// seq_offsets (no host synchronisation).
//
// "[pallas] Support dependent Tile.end bounds in Pallas" ("Flattened
// worklists"): a work item carries the resident source range
// (range_start, range_len) and the compact Q tile (tile_start, tile_extent);
// its compute end is min(source_end, compact_end).  The review thread on the
// same page fixes the jagged KV end as seq_offsets[seq_idx + 1].
//
// Item = int4 {range_start, range_len, tile_start, tile_extent}, one per
// (sequence, Q tile of block_m rows).  Order: sequences with more Q tiles
// first (so long causal work starts early), sequences in index order within a
// tile count, and inside a sequence its tiles from first to last: each tile
// re-reads from L2 the K/V the earlier tiles of the sequence brought in and
// fetches the next tiles of it (measured 1.8 % faster in the paired kernel than
// last to first, where the first, longest walk took the whole range from HBM at
// once).  When ceil(max_seqlen / block_m) > 64 the count buckets are skipped and
// sequences stay in index order.
//
// Units ("Grouping" on the same page: successive Q work items of one sequence
// reuse its resident K/V range): one int2 {first_item, n_items} per sequence
// with at least one tile, in the same order; a persistent kernel takes a unit
// and one head at a time, so the sequence's tiles run back to back on one SM
// and its K/V is re-read from L2 rather than HBM.
//
// Output buffer: int item count at word 0, int unit count at word 1, items
// from byte 16 (max_items of them), then the units.
//
// Up to 1024 sequences one CTA builds the list.  Beyond that two kernels share
// the work, so the cost no longer grows with the sequence count: a count kernel
// (one thread per sequence) sums each CTA's items and units per tile-count
// bucket into a small table (int2 per CTA and bucket, after the units), and a
// write kernel gives each CTA its positions from that table.  Both produce the
// same list in the same order.
//
// All sequences of a bucket have the same tile count, so a sequence's first
// item is its bucket's first position plus its rank among the bucket's earlier
// sequences times that count: one pass over the sequences (ranks within a warp
// by matching buckets, then a sum over the warps before it per bucket) places
// every bucket at once.  Without buckets (sequence order, tile counts that
// differ) a block-wide scan of the tile counts places them.
#include "checked.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace attn {

static __device__ unsigned int g_worklist_status;

// Sequence b's tile count (0 for an invalid or empty sequence) and start.
__device__ __forceinline__ int seq_tiles(const int32_t* __restrict__ offs, int b, int num_seqs, int total_tokens,
                                         int max_seqlen, int block_m, int& begin, int& len, bool& bad) {
  begin = 0;
  len = 0;
  bad = false;
  if (b >= num_seqs) return 0;
  begin = offs[b];
  const int end = offs[b + 1];
  len = end - begin;
  if (begin < 0 || end > total_tokens || len < 0 || len > max_seqlen) {
    bad = true;
    len = 0;
  }
  return (len + block_m - 1) / block_m;
}

// One thread per sequence of a CTA's 1024 (nt its tile count, 0 if empty):
// writes its items and its unit in bucketed order.  base[k] / ubase[k]: the
// position of the CTA's first item / unit of bucket k (bucket k holds the
// sequences of nmax - k tiles).  Every thread of the CTA calls it.
__device__ void write_bucketed(int nt, int begin, int len, int nmax, int block_m, const int* base, const int* ubase,
                               int (*s_wcnt)[kWorklistBuckets], int4* __restrict__ items, int max_items,
                               int2* __restrict__ units, int num_seqs) {
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int w = tid >> 5;
  const int nb = nmax;
  for (int i = tid; i < 32 * kWorklistBuckets; i += blockDim.x) s_wcnt[i / kWorklistBuckets][i % kWorklistBuckets] = 0;
  __syncthreads();
  const int k = nt > 0 ? nmax - nt : -1;  // 0 .. nmax - 1: more tiles first
  const unsigned peers = __match_any_sync(0xffffffffu, k);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));  // earlier lanes of the bucket
  if (k >= 0 && rank_w == 0) s_wcnt[w][k] = __popc(peers);
  __syncthreads();
  // per bucket, the sequences of the warps before each warp
  if (tid < nb) {
    int run = 0;
    for (int v = 0; v < 32; ++v) {
      const int c = s_wcnt[v][tid];
      s_wcnt[v][tid] = run;
      run += c;
    }
  }
  __syncthreads();
  if (k >= 0) {
    const int r = s_wcnt[w][k] + rank_w;  // rank among the CTA's sequences of bucket k
    const long long first = (long long)base[k] + (long long)r * nt;
    for (int t = 0; t < nt; ++t) {
      const long long pos = first + t;
      if (pos < max_items) items[pos] = make_int4(begin, len, begin + t * block_m, min(block_m, len - t * block_m));
    }
    if (check_index((long long)ubase[k] + r, num_seqs, &g_worklist_status))  // < num_seqs by construction
      units[ubase[k] + r] = make_int2((int)min(first, (long long)0x7fffffff), nt);
  }
}

// One CTA, num_seqs <= 1024 (the launcher's choice): the tile-count buckets'
// sizes in shared memory, then the one-pass write; without buckets, one
// block-wide scan of the tile counts in sequence order.
__global__ void __launch_bounds__(1024) worklist_kernel(const int32_t* __restrict__ offs, int num_seqs,
                                                        int total_tokens, int max_seqlen, int block_m,
                                                        int* __restrict__ out, int max_items) {
  int4* items = reinterpret_cast<int4*>(out + 4);
  int2* units = reinterpret_cast<int2*>(out + 4 + 4 * (size_t)max_items);
  __shared__ int s_wcnt[32][kWorklistBuckets];
  __shared__ int s_items[kWorklistBuckets], s_units[kWorklistBuckets], s_base[kWorklistBuckets],
      s_ubase[kWorklistBuckets];
  __shared__ long long warp_sums[32];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int w = tid >> 5;
  const int nmax = (max_seqlen + block_m - 1) / block_m;
  const bool bucketed = nmax <= kWorklistBuckets;
  if (tid < kWorklistBuckets) {
    s_items[tid] = 0;
    s_units[tid] = 0;
  }
  if (tid == 0) s_bad = num_seqs > (int)blockDim.x;  // never, by the launcher's choice
  __syncthreads();
  int begin, len;
  bool bad;
  const int nt = seq_tiles(offs, tid, num_seqs, total_tokens, max_seqlen, block_m, begin, len, bad);
  if (bad) s_bad = 1;
  if (bucketed) {
    if (nt > 0) {
      atomicAdd(&s_items[nmax - nt], nt);
      atomicAdd(&s_units[nmax - nt], 1);
    }
    __syncthreads();
    if (tid == 0) {
      long long ib = 0, ub = 0;
      for (int k = 0; k < nmax; ++k) {
        s_base[k] = (int)min(ib, (long long)0x7fffffff);
        s_ubase[k] = (int)ub;
        ib += s_items[k];
        ub += s_units[k];
      }
      out[0] = ib < max_items ? (int)ib : max_items;
      out[1] = (int)ub;  // consumers skip unit items at or beyond out[0]
      if (s_bad || ib > max_items) atomicOr(&g_worklist_status, kStatusDeviceInput);
    }
    __syncthreads();
    write_bucketed(nt, begin, len, nmax, block_m, s_base, s_ubase, s_wcnt, items, max_items, units, num_seqs);
    return;
  }
  // block-wide exclusive scan of (tiles << 32) | units, both counts < 2^31
  const long long v = ((long long)nt << 32) | (nt > 0 ? 1 : 0);
  long long x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  if (w == 0) {
    long long y = warp_sums[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const long long z = __shfl_up_sync(0xffffffffu, y, d);
      if (lane >= d) y += z;
    }
    warp_sums[lane] = y;
  }
  __syncthreads();
  const long long ex = x - v + (w > 0 ? warp_sums[w - 1] : 0);
  const long long excl = ex >> 32;
  const int uexcl = (int)(ex & 0xffffffffLL);
  if (nt > 0) {
    for (int t = 0; t < nt; ++t) {
      const long long pos = excl + t;
      if (pos < max_items) items[pos] = make_int4(begin, len, begin + t * block_m, min(block_m, len - t * block_m));
    }
    if (check_index((long long)uexcl, num_seqs, &g_worklist_status))  // < num_seqs by construction
      units[uexcl] = make_int2((int)min(excl, (long long)0x7fffffff), nt);
  }
  if (tid == 0) {
    const long long total = warp_sums[31] >> 32;
    out[0] = total < max_items ? (int)total : max_items;
    out[1] = (int)(warp_sums[31] & 0xffffffffLL);
    if (s_bad || total > max_items) atomicOr(&g_worklist_status, kStatusDeviceInput);
  }
}

// Count kernel: CTA c sums, for each tile-count bucket, the items and units of
// its sequences [1024 c, 1024 c + 1024) into counts[c * kWorklistBuckets + bucket].
__global__ void __launch_bounds__(1024) worklist_count_kernel(const int32_t* __restrict__ offs, int num_seqs,
                                                              int total_tokens, int max_seqlen, int block_m,
                                                              int2* __restrict__ counts) {
  __shared__ int s_items[kWorklistBuckets], s_units[kWorklistBuckets];
  const int tid = threadIdx.x;
  const int nmax = (max_seqlen + block_m - 1) / block_m;
  const bool bucketed = nmax <= kWorklistBuckets;
  if (tid < kWorklistBuckets) {
    s_items[tid] = 0;
    s_units[tid] = 0;
  }
  __syncthreads();
  int begin, len;
  bool bad;
  const int nt = seq_tiles(offs, blockIdx.x * 1024 + tid, num_seqs, total_tokens, max_seqlen, block_m, begin, len, bad);
  if (bad) atomicOr(&g_worklist_status, kStatusDeviceInput);
  if (nt > 0) {
    const int bucket = bucketed ? nmax - nt : 0;  // 0 .. nmax - 1: more tiles first
    atomicAdd(&s_items[bucket], nt);
    atomicAdd(&s_units[bucket], 1);
  }
  __syncthreads();
  if (tid < kWorklistBuckets) counts[(size_t)blockIdx.x * kWorklistBuckets + tid] = make_int2(s_items[tid], s_units[tid]);
}

// Write kernel: CTA c writes the items and units of its sequences.  Bucket k's
// items start after every item of the buckets before it (all CTAs) and those
// of bucket k in CTAs before c; within the CTA the one-pass bucketed write, or
// without buckets a block scan in sequence order.
__global__ void __launch_bounds__(1024) worklist_write_kernel(const int32_t* __restrict__ offs, int num_seqs,
                                                              int total_tokens, int max_seqlen, int block_m,
                                                              const int2* __restrict__ counts, int n_cta,
                                                              int* __restrict__ out, int max_items) {
  int4* items = reinterpret_cast<int4*>(out + 4);
  int2* units = reinterpret_cast<int2*>(out + 4 + 4 * (size_t)max_items);
  __shared__ long long warp_sums[32];
  __shared__ int s_base[kWorklistBuckets], s_ubase[kWorklistBuckets], s_mine[kWorklistBuckets];
  __shared__ long long s_col[kWorklistBuckets], s_ucol[kWorklistBuckets];  // bucket totals, all CTAs
  __shared__ int s_wcnt[32][kWorklistBuckets];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int w = tid >> 5;
  const int nmax = (max_seqlen + block_m - 1) / block_m;
  const bool bucketed = nmax <= kWorklistBuckets;
  const int nb = bucketed ? nmax : 1;
  // thread k < nb: bucket k's totals over all CTAs and over the CTAs before this one
  long long before = 0, ubefore = 0;
  if (tid < nb) {
    long long col = 0, ucol = 0;
    for (int c = 0; c < n_cta; ++c) {
      const int2 e = counts[(size_t)c * kWorklistBuckets + tid];
      col += e.x;
      ucol += e.y;
      if (c < (int)blockIdx.x) {
        before += e.x;
        ubefore += e.y;
      }
    }
    s_col[tid] = col;
    s_ucol[tid] = ucol;
    s_mine[tid] = counts[(size_t)blockIdx.x * kWorklistBuckets + tid].y;
  }
  __syncthreads();
  if (tid < nb) {
    long long ib = before, ub = ubefore;
    for (int k = 0; k < tid; ++k) {
      ib += s_col[k];
      ub += s_ucol[k];
    }
    s_base[tid] = (int)min(ib, (long long)0x7fffffff);
    s_ubase[tid] = (int)min(ub, (long long)0x7fffffff);
  }
  if (blockIdx.x == 0 && tid == 0) {
    long long total = 0, utotal = 0;
    for (int k = 0; k < nb; ++k) {
      total += s_col[k];
      utotal += s_ucol[k];
    }
    out[0] = total < max_items ? (int)total : max_items;
    out[1] = (int)utotal;  // consumers skip unit items at or beyond out[0]
    if (total > max_items) atomicOr(&g_worklist_status, kStatusDeviceInput);
  }
  __syncthreads();
  int begin, len;
  bool bad;
  const int nt = seq_tiles(offs, blockIdx.x * 1024 + tid, num_seqs, total_tokens, max_seqlen, block_m, begin, len, bad);
  if (bucketed) {
    write_bucketed(nt, begin, len, nmax, block_m, s_base, s_ubase, s_wcnt, items, max_items, units, num_seqs);
    return;
  }
  if (s_mine[0] == 0) return;  // no sequence with tiles here (the same for every thread of the CTA)
  // block-wide exclusive scan of (tiles << 32) | units, both counts < 2^31
  const long long v = ((long long)nt << 32) | (nt > 0 ? 1 : 0);
  long long x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  if (w == 0) {
    long long y = warp_sums[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const long long z = __shfl_up_sync(0xffffffffu, y, d);
      if (lane >= d) y += z;
    }
    warp_sums[lane] = y;
  }
  __syncthreads();
  const long long ex = x - v + (w > 0 ? warp_sums[w - 1] : 0);
  const long long first = (long long)s_base[0] + (ex >> 32);
  const int uexcl = (int)(ex & 0xffffffffLL);
  if (nt > 0) {
    for (int t = 0; t < nt; ++t) {
      const long long pos = first + t;
      if (pos < max_items) items[pos] = make_int4(begin, len, begin + t * block_m, min(block_m, len - t * block_m));
    }
    if (check_index((long long)s_ubase[0] + uexcl, num_seqs, &g_worklist_status))  // < num_seqs by construction
      units[s_ubase[0] + uexcl] = make_int2((int)min(first, (long long)0x7fffffff), nt);
  }
}

size_t worklist_scratch_bytes(int num_seqs) {
  const size_t n_cta = ((size_t)(num_seqs > 0 ? num_seqs : 0) + 1023) / 1024;
  return n_cta * kWorklistBuckets * sizeof(int2);
}

attn_status_t launch_worklist(const int32_t* seq_offsets, int num_seqs, int total_tokens, int max_seqlen, int block_m,
                              int* count_and_items, int max_items, int2* scratch, cudaStream_t s) {
  if (num_seqs <= 1024) {
    worklist_kernel<<<1, 1024, 0, s>>>(seq_offsets, num_seqs, total_tokens, max_seqlen, block_m, count_and_items,
                                       max_items);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  const int n_cta = (num_seqs + 1023) / 1024;
  worklist_count_kernel<<<n_cta, 1024, 0, s>>>(seq_offsets, num_seqs, total_tokens, max_seqlen, block_m, scratch);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  worklist_write_kernel<<<n_cta, 1024, 0, s>>>(seq_offsets, num_seqs, total_tokens, max_seqlen, block_m, scratch, n_cta,
                                               count_and_items, max_items);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// One thread waits, bounded, on a barrier that nothing completes.
__global__ void selftest_timeout_kernel(uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  abort_flag = 0;
  mbar_init(&bar, 1);
  fence_barrier_init();
  mbar_wait_bounded(&bar, 0, &abort_flag, &g_worklist_status, kStatusTimeout | (0xA0u << kStatusSiteShift),
                    timeout_ns);
}

// Index 1 of a one-element buffer, through the checked build's store check: a
// checked build reports it (kStatusBounds) and skips the store; without checks
// the store goes to index 0, in range either way.
__global__ void selftest_bounds_kernel(int* buf) {
  if (check_index(1, 1, &g_worklist_status)) buf[0] = 1;
}

attn_status_t launch_selftest_bounds(int* buf, cudaStream_t s) {
  selftest_bounds_kernel<<<1, 1, 0, s>>>(buf);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t launch_selftest_timeout(uint64_t timeout_ns, cudaStream_t s) {
  selftest_timeout_kernel<<<1, 1, 0, s>>>(timeout_ns);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

unsigned int worklist_take_status(cudaStream_t s) {
  if (cudaStreamSynchronize(s) != cudaSuccess) return kStatusTimeout;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_worklist_status, sizeof(v)) != cudaSuccess) return kStatusTimeout;
  if (v != 0) {
    const unsigned int zero = 0;
    cudaMemcpyToSymbol(g_worklist_status, &zero, sizeof(zero));
  }
  return v;
}

}  // namespace attn
