// Host-only: one device address per device, remembered together with the CUDA
// context it belongs to.
//
// The address of a `__device__` variable is a property of the module loaded in
// one context.  A device reset (cudaDeviceReset, or another library ending the
// primary context) creates a new context in which the module, and the variable,
// may sit elsewhere.  A context is named here by its process-unique id
// (cuCtxGetId), never by its handle: a later context can reuse the handle value
// of one that was destroyed, but never its id.  An entry recorded under one
// context id is not returned for any other.
#pragma once

#include <mutex>

namespace attn {

template <int kMaxDevices>
class ContextAddressCache {
 public:
  // The address recorded for `dev` under context `ctx_id`, or nullptr when the
  // device has none or recorded it under another context.
  void* get(int dev, unsigned long long ctx_id) const {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu_);
    return (valid_[dev] && ctx_[dev] == ctx_id) ? addr_[dev] : nullptr;
  }

  // Records `addr` for `dev` under context `ctx_id`, replacing what was there.
  bool put(int dev, unsigned long long ctx_id, void* addr) {
    if (dev < 0 || dev >= kMaxDevices || addr == nullptr) return false;
    std::lock_guard<std::mutex> lock(mu_);
    ctx_[dev] = ctx_id;
    addr_[dev] = addr;
    valid_[dev] = true;
    return true;
  }

 private:
  mutable std::mutex mu_;
  unsigned long long ctx_[kMaxDevices] = {};
  void* addr_[kMaxDevices] = {};
  bool valid_[kMaxDevices] = {};
};

}  // namespace attn
