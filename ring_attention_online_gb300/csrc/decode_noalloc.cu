// Split-KV decode for callers that cannot allocate device memory.
//
// attn_decode_splitkv needs a caller-provided workspace for the per-chunk
// partial triplets.  Some callers have no way to provide one: a host program
// whose memory is owned by a framework that hands plugins only their input and
// output buffers, or a latency-critical loop that must never call cudaMalloc /
// cudaFree (both can synchronise the whole device) and must not risk an
// out-of-memory failure in the middle of a run.  For them this file keeps the
// scratch in a fixed-size array in device memory that is part of the library
// image: it exists on every GPU that loads the library, from load until the
// process exits, and no call here allocates or frees anything.
//
// The array is shared by every call on a device and keeps whatever the last
// call wrote.  Nothing needs to start at zero: each call zeroes its merge
// counters and writes every (chunk, batch, head) triplet before reading it.
// Two calls whose kernels overlap on the GPU (e.g. on two streams) race on the
// array.
#include <mutex>

#include "common.cuh"
#include "context_cache.h"

namespace attn {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
ContextAddressCache<kMaxDevices> g_scratch_addr;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Driver entry points for naming the current context (looked up once).
bool ctx_functions(CtxGetCurrentFn* get_current, CtxGetIdFn* get_id) {
  static CtxGetCurrentFn cur = nullptr;
  static CtxGetIdFn id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      id = reinterpret_cast<CtxGetIdFn>(p);
  });
  *get_current = cur;
  *get_id = id;
  return cur != nullptr && id != nullptr;
}

// Process-unique id of the calling thread's current context; false if there is none.
bool current_context_id(unsigned long long* out) {
  CtxGetCurrentFn get_current;
  CtxGetIdFn get_id;
  if (!ctx_functions(&get_current, &get_id)) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, out) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current device's current context.
// The host-side symbol g_decode_scratch is only a stand-in, not a device
// address.  The address is looked up with cudaGetSymbolAddress the first time
// a device is used under a context and kept for that context; a new context
// on the device (after a device reset) gets a fresh lookup, because the
// module, and the array with it, may then sit at another address.
attn_status_t scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  unsigned long long ctx_id = 0;
  if (current_context_id(&ctx_id)) {
    if (void* p = g_scratch_addr.get(dev, ctx_id)) {
      *out = p;
      return ATTN_OK;
    }
  }
  // the lookup also creates the device's primary context if the thread has none yet
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
  if (!current_context_id(&ctx_id)) return ATTN_ERR_CUDA;
  g_scratch_addr.put(dev, ctx_id, p);
  *out = p;
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" attn_status_t attn_decode_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                                     int B, int S_kv, int h_q, int h_kv, int D, attn_dtype_t dtype,
                                                     float scale, int num_splits, attn_stream_t stream) {
  if (B < 0 || h_q < 1 || num_splits < 1) return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_decode_workspace_bytes(B, h_q, D, num_splits);
  if (need > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;  // partials do not fit the fixed scratch
  void* scratch = nullptr;
  const attn_status_t st = attn::scratch_on_current_device(&scratch);
  if (st != ATTN_OK) return st;
  return attn_decode_splitkv(q, k, v, o, lse, B, S_kv, h_q, h_kv, D, dtype, scale, num_splits, scratch,
                             ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
