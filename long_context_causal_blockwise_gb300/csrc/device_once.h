// Host-side "once per device context" set-up flags.
//
// Settings such as a kernel's dynamic shared-memory limit
// (cudaFuncSetAttribute) belong to one device's context: a process that drives
// two GPUs must apply them on each, and a context torn down by
// cudaDeviceReset and created again has lost them. DeviceOnce keeps, per
// device ordinal, the id of the context in which the set-up last succeeded;
// run(dev, ctx_id, f) calls f unless that id equals ctx_id. Context ids are
// unique within a process and never 0; ctx_id 0 (no id known) runs f every
// time. A failed set-up is not remembered, so the next call retries it.
// Plain C++ (no CUDA), so that its logic can be checked on a machine without
// a GPU with made-up device ordinals and context ids.
#pragma once

#include <atomic>
#include <mutex>

namespace lcb {

constexpr int kMaxDeviceOrdinals = 64;

class DeviceOnce {
 public:
  // Returns f()'s status when it runs, 0 when the set-up is already done in
  // context ctx_id of device `dev`, and `bad_device` for an ordinal outside
  // [0, kMaxDeviceOrdinals).
  template <class F>
  int run(int dev, unsigned long long ctx_id, F&& f, int bad_device) {
    if (dev < 0 || dev >= kMaxDeviceOrdinals) return bad_device;
    if (ctx_id == 0) return f();
    if (key_[dev].load(std::memory_order_acquire) == ctx_id) return 0;
    std::lock_guard<std::mutex> lk(mu_);
    if (key_[dev].load(std::memory_order_relaxed) == ctx_id) return 0;
    const int rc = f();
    if (rc == 0) key_[dev].store(ctx_id, std::memory_order_release);
    return rc;
  }

  // True if the set-up succeeded in context ctx_id of device `dev`.
  bool done(int dev, unsigned long long ctx_id) const {
    return dev >= 0 && dev < kMaxDeviceOrdinals && ctx_id != 0 &&
           key_[dev].load(std::memory_order_acquire) == ctx_id;
  }

 private:
  std::mutex mu_;
  std::atomic<unsigned long long> key_[kMaxDeviceOrdinals] = {};
};

}  // namespace lcb
