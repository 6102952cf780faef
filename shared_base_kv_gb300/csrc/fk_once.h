// One-time set-up of a kernel (shared-memory opt-in, register check) per
// device: cudaFuncSetAttribute acts on the current device only, so every
// device a process drives needs its own.  Not part of the C ABI.
#pragma once
#include <cuda_runtime.h>

#include <mutex>

#include "fk_internal.h"

namespace fk {

class PerDeviceOnce {
 public:
  // Runs setup() (returning a cudaError_t as int) on the first call from
  // each device until it succeeds; 0 afterwards.
  template <class F>
  int run(F&& setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev]) return 0;
    const int r = setup();
    if (r == 0) done_[dev] = true;
    return r;
  }

 private:
  std::mutex mu_;
  bool done_[kMaxDevices] = {};
};

}  // namespace fk
