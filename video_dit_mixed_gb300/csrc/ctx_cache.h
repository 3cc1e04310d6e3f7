// Per-context caches for host-side set-up that belongs to a CUDA context:
// kernel attributes, SM counts, occupancy, symbol addresses.  A value is
// computed once per (device, context) and recomputed when the current context
// of that device changes (another device, or the same device after
// cudaDeviceReset).  Lookups are serialised by a mutex, so concurrent host
// threads never race on the cache.
#pragma once

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

namespace sixbit {

// Identity of the calling thread's current CUDA context (cuCtxGetId), or 0
// when no context is current yet (a value cached under 0 is recomputed once
// the context exists).
uint64_t current_context_id();

constexpr int kMaxCachedDevices = 64;

template <typename T>
class ContextCache {
 public:
  // *out = the cached value for the current context, computing it with
  // make(T*) -> cudaError_t on first use (an error is returned, not cached).
  template <typename Make>
  cudaError_t get(T* out, Make make) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxCachedDevices) return make(out);
    const uint64_t id = current_context_id();
    std::lock_guard<std::mutex> lock(mu_);
    if (!valid_[dev] || ctx_[dev] != id || id == 0) {
      T v{};
      e = make(&v);
      if (e != cudaSuccess) return e;
      val_[dev] = v;
      ctx_[dev] = id;
      valid_[dev] = true;
    }
    *out = val_[dev];
    return cudaSuccess;
  }

 private:
  std::mutex mu_;
  bool valid_[kMaxCachedDevices] = {};
  uint64_t ctx_[kMaxCachedDevices] = {};
  T val_[kMaxCachedDevices] = {};
};

// Sets the dynamic shared-memory limit of the kernel KERNEL once per context
// (one cache per kernel: the template is instantiated per function pointer).
template <auto KERNEL>
cudaError_t set_smem_once(int bytes) {
  static ContextCache<int> done;
  int v = 0;
  return done.get(&v, [&](int* o) {
    *o = 1;
    return cudaFuncSetAttribute(KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  });
}

// Number of SMs of the current device (cached per context).
int sm_count();

}  // namespace sixbit
