// Checked builds (compiled with ATTN_CHECKED=1, the library libattn_checked.so):
// the kernels compare every global store index, every TMA tile coordinate and
// every worklist index with the extent of its buffer before the access.  A
// violation ORs kStatusBounds into the translation unit's device status word and
// skips the access (no trap, no fault), so attn_last_device_status() reports
// ATTN_ERR_BOUNDS and the context stays usable.  In ordinary builds every check
// is the constant true and compiles to nothing.
#pragma once

#include "common.cuh"

#ifndef ATTN_CHECKED
#define ATTN_CHECKED 0
#endif

namespace attn {

// i in [0, n).
__device__ __forceinline__ bool check_index(long long i, long long n, unsigned int* status) {
#if ATTN_CHECKED
  if (i < 0 || i >= n) {
    atomicOr(status, kStatusBounds);
    return false;
  }
#else
  (void)i;
  (void)n;
  (void)status;
#endif
  return true;
}

// The coordinates of a 4-D tile load over a [batch, rows, heads, cols] tensor
// of 16-bit elements, read as boxes of 64 columns: the column start must be a
// multiple of 64 inside [0, cols) (a 128-byte, hence 16-byte aligned, start),
// head and batch inside their extents, and the row start inside [0, rows +
// row_slack): boxes that lie partly or wholly past the last row read zeros,
// which is how tail tiles and empty tiles load, but never further out than
// `row_slack` rows.
__device__ __forceinline__ bool check_tile(int c0, int c1, int c2, int c3, int cols, int heads, long long rows,
                                           int batch, int row_slack, unsigned int* status) {
#if ATTN_CHECKED
  const bool ok = c0 >= 0 && c0 < cols && (c0 & 63) == 0 && c1 >= 0 && c1 < heads && c2 >= 0 &&
                  (long long)c2 < rows + row_slack && c3 >= 0 && c3 < batch;
  if (!ok) atomicOr(status, kStatusBounds);
  return ok;
#else
  (void)c0;
  (void)c1;
  (void)c2;
  (void)c3;
  (void)cols;
  (void)heads;
  (void)rows;
  (void)batch;
  (void)row_slack;
  (void)status;
  return true;
#endif
}

}  // namespace attn
