// Allocation-free variant of sixbit_block_stats.
//
// Who needs it: callers that cannot call cudaMalloc -- code that runs where
// the allocator is off limits (inside a custom memory pool that owns all
// device memory, in a plugin host that forbids allocation after start-up, or
// in a process whose allocations must all be accounted up front).  The
// regular entry point takes the reduction scratch from the caller; this one
// keeps it in a fixed array in the library's own device memory instead.
//
// The scratch lives in one file-scope __device__ array of
// kNoallocScratchBytes (about 256 KB), which every GPU that loads the library
// holds until the process exits.  Host code may not use the array's name as a
// device address (on the host it names a shadow variable), so the device
// address is looked up with cudaGetSymbolAddress, with the device current,
// once per device and CUDA context (again after a cudaDeviceReset, which can
// move the array).  The library does that lookup at its first call of any
// entry point on each device: under CUDA's lazy module loading that lookup is
// when the driver creates the array, so a caller whose memory pool will own
// all device memory makes one library call first (or runs with
// CUDA_MODULE_LOADING=EAGER).  That first call should also come before any
// stream capture.  Every call shares the one array: calls that overlap on the
// GPU (different streams, or different host threads without ordering) race on
// it and corrupt each other's results.
#include <cstdint>

#include "common.cuh"
#include "ctx_cache.h"
#include "internal.h"

namespace sixbit {

// Counter (16 bytes) + one 64-byte partial record per CTA.
constexpr int64_t kNoallocMaxCtas = 4096;
constexpr size_t kNoallocScratchBytes = 16 + static_cast<size_t>(kNoallocMaxCtas) * 64;
constexpr int64_t kNoallocMaxElems = kNoallocMaxCtas * kFixedElemsPerCta;  // 268,435,456

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch in the current context.
sixbit_status noalloc_scratch(void** out) {
  static ContextCache<void*> cache;
  const cudaError_t e = cache.get(out, [](void** p) {
    *p = nullptr;
    const cudaError_t r = cudaGetSymbolAddress(p, g_noalloc_scratch);
    return (r == cudaSuccess && *p != nullptr) ? cudaSuccess : cudaErrorInvalidSymbol;
  });
  return e == cudaSuccess ? SIXBIT_OK : SIXBIT_ECUDA;
}

}  // namespace sixbit

using namespace sixbit;

extern "C" int64_t sixbit_block_stats_noalloc_max_elems(void) { return kNoallocMaxElems; }

extern "C" sixbit_status sixbit_block_stats_noalloc(const uint16_t* x_in, const uint16_t* x_out,
                                                    uint16_t* delta_cache, int64_t n, const int32_t* mode_dev,
                                                    sixbit_stats* stats_dev, int32_t* err_dev, void* stream) {
  (void)err_dev;  // the statistics kernel has no device-side error path
  if (x_in == nullptr || x_out == nullptr || delta_cache == nullptr || stats_dev == nullptr) return SIXBIT_EINVAL;
  if (n <= 0 || n % 8 != 0 || n > kNoallocMaxElems) return SIXBIT_ESHAPE;
  if ((reinterpret_cast<uintptr_t>(x_in) | reinterpret_cast<uintptr_t>(x_out) |
       reinterpret_cast<uintptr_t>(delta_cache)) & 15u)
    return SIXBIT_EALIGN;
  sixbit_status s = check_device();
  if (s != SIXBIT_OK) return s;
  void* scratch = nullptr;
  s = noalloc_scratch(&scratch);
  if (s != SIXBIT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the completion counter must start at zero (the kernel also leaves it zero)
  if (cudaMemsetAsync(scratch, 0, 16, st) != cudaSuccess) return SIXBIT_ECUDA;
  return launch_block_stats_fixed_grid(x_in, x_out, delta_cache, n, mode_dev, stats_dev, scratch, st) == cudaSuccess
             ? SIXBIT_OK
             : SIXBIT_ECUDA;
}
