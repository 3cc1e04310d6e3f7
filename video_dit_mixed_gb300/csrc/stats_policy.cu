// Block statistics, temporal-delta-cache update / skip, and the per-block
// decision kernel.
//
// Method: "6Bit-Diffusion" technical summary sections 2.A (Gamma_{t-1}, the
// relative input-output difference of a block), 2.B (Temporal Delta Cache:
// skip when Delta_{t-1} and Delta_{t-2} agree; error-guided refresh) and 2.C
// (PDR: outliers force an FP16/BF16 recompute before a delta is cached);
// popular summary sections 2-3 (error accumulator; max/mean outlier ratio;
// INT8 for every layer after a skip).
//
// The reductions are one pass over HBM with 16-byte loads.  Sums of squares
// and products of bf16 values are exact in FP32 per term; each thread keeps
// them as an unevaluated pair (s, c) updated with Knuth's TwoSum, so a
// thread's partial carries about 48 bits; partials are combined in float64 in
// a fixed order (warp shuffle tree, then CTA, then a last-CTA pass over the
// per-CTA partials in scratch), so results are run-to-run deterministic.
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace sixbit {

constexpr int kStThreads = 256;
constexpr int kStMaxBlocks = 1216;  // 152 SMs x 8
constexpr int kNumSums = 8;

struct TwoF {
  float s, c;
};

__device__ __forceinline__ void two_add(TwoF& a, float x) {
  const float s = __fadd_rn(a.s, x);
  const float bp = __fsub_rn(s, a.s);
  const float err = __fadd_rn(__fsub_rn(a.s, __fsub_rn(s, bp)), __fsub_rn(x, bp));
  a.s = s;
  a.c = __fadd_rn(a.c, err);
}

__device__ __forceinline__ double to_d(const TwoF& a) { return static_cast<double>(a.s) + static_cast<double>(a.c); }

__device__ __forceinline__ uint4 ld16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void unpack8(const uint4& r, float (&v)[8]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&p);
}

struct Scratch {
  unsigned int* counter;
  double* partial;  // [gridDim.x][kNumSums]
};

__device__ __forceinline__ Scratch scratch_view(void* p) {
  Scratch s;
  s.counter = reinterpret_cast<unsigned int*>(p);
  s.partial = reinterpret_cast<double*>(reinterpret_cast<char*>(p) + 16);
  return s;
}

// Reduces per-thread float64 values v[0..NS) (index NS-? as max where is_max)
// across the grid in a fixed order.  Returns true in exactly one thread of the
// last CTA to finish, with the totals in `tot`.
template <int NS>
__device__ bool grid_reduce(double (&v)[NS], const bool (&is_max)[NS], Scratch sc, double (&tot)[NS]) {
  __shared__ double red[kStThreads / 32][NS];
  __shared__ bool last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    double x = v[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double y = __shfl_xor_sync(0xffffffffu, x, o);
      x = is_max[k] ? fmax(x, y) : x + y;
    }
    if (lane == 0) red[warp][k] = x;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      double x = red[0][k];
      for (int w = 1; w < kStThreads / 32; ++w) x = is_max[k] ? fmax(x, red[w][k]) : x + red[w][k];
      sc.partial[static_cast<size_t>(blockIdx.x) * kNumSums + k] = x;
    }
    __threadfence();
    const unsigned int done = atomicAdd(sc.counter, 1u);
    last = (done == gridDim.x - 1);
  }
  __syncthreads();
  if (!last) return false;
  __threadfence();
  // last CTA: thread t folds partials t, t+256, ... then the same tree
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    double x = is_max[k] ? 0.0 : 0.0;
    for (unsigned int b = threadIdx.x; b < gridDim.x; b += kStThreads) {
      const double y = *reinterpret_cast<volatile double*>(&sc.partial[static_cast<size_t>(b) * kNumSums + k]);
      x = is_max[k] ? fmax(x, y) : x + y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double y = __shfl_xor_sync(0xffffffffu, x, o);
      x = is_max[k] ? fmax(x, y) : x + y;
    }
    if (lane == 0) red[warp][k] = x;
  }
  __syncthreads();
  if (threadIdx.x != 0) return false;
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    double x = red[0][k];
    for (int w = 1; w < kStThreads / 32; ++w) x = is_max[k] ? fmax(x, red[w][k]) : x + red[w][k];
    tot[k] = x;
  }
  *sc.counter = 0;  // leave the scratch ready for the next call
  return true;
}

__device__ __forceinline__ bool mode_is_not(const int32_t* mode_dev, int want) {
  return mode_dev != nullptr && SIXBIT_MODE_OF(*mode_dev) != want;
}

__device__ __forceinline__ bool mode_is(const int32_t* mode_dev, int want) {
  return mode_dev != nullptr && SIXBIT_MODE_OF(*mode_dev) == want;
}

// out[0..3] = {max |x|, sum |x|, count, sum x^2}
__global__ void __launch_bounds__(kStThreads) tensor_stats_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                                  double* out, void* scratch) {
  const int64_t n8 = n >> 3;
  float mx = 0.f;
  TwoF sa{0.f, 0.f}, sq{0.f, 0.f};
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kStThreads) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * kStThreads) {
    float v[8];
    unpack8(ld16(x + 8 * i), v);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float a = fabsf(v[j]);
      mx = fmaxf(mx, a);
      two_add(sa, a);
      two_add(sq, __fmul_rn(v[j], v[j]));
    }
  }
  double v[3] = {static_cast<double>(mx), to_d(sa), to_d(sq)};
  const bool is_max[3] = {true, false, false};
  double tot[3];
  if (grid_reduce<3>(v, is_max, scratch_view(scratch), tot)) {
    out[0] = tot[0];
    out[1] = tot[1];
    out[2] = static_cast<double>(n);
    out[3] = tot[2];
  }
}

__global__ void __launch_bounds__(kStThreads) block_stats_kernel(const uint16_t* __restrict__ x_in,
                                                                 const uint16_t* __restrict__ x_out,
                                                                 uint16_t* delta, int64_t n, const int32_t* mode_dev,
                                                                 sixbit_stats* stats, void* scratch) {
  if (mode_is(mode_dev, SIXBIT_MODE_SKIP)) return;
  const int64_t n8 = n >> 3;
  float mx = 0.f;
  TwoF d2{0.f, 0.f}, xi2{0.f, 0.f}, ddp{0.f, 0.f}, dp2{0.f, 0.f}, sa{0.f, 0.f};
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kStThreads) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * kStThreads) {
    float a[8], b[8], p[8], d[8];
    unpack8(ld16(x_in + 8 * i), a);
    unpack8(ld16(x_out + 8 * i), b);
    unpack8(*reinterpret_cast<const uint4*>(delta + 8 * i), p);
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      w[j] = pack2(__fsub_rn(b[2 * j], a[2 * j]), __fsub_rn(b[2 * j + 1], a[2 * j + 1]));
      d[2 * j] = __uint_as_float(w[j] << 16);
      d[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
    *reinterpret_cast<uint4*>(delta + 8 * i) = make_uint4(w[0], w[1], w[2], w[3]);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      two_add(d2, __fmul_rn(d[j], d[j]));
      two_add(xi2, __fmul_rn(a[j], a[j]));
      two_add(ddp, __fmul_rn(d[j], p[j]));
      two_add(dp2, __fmul_rn(p[j], p[j]));
      const float ab = fabsf(b[j]);
      mx = fmaxf(mx, ab);
      two_add(sa, ab);
    }
  }
  double v[6] = {to_d(d2), to_d(xi2), to_d(ddp), to_d(dp2), static_cast<double>(mx), to_d(sa)};
  const bool is_max[6] = {false, false, false, false, true, false};
  double tot[6];
  if (grid_reduce<6>(v, is_max, scratch_view(scratch), tot)) {
    stats->sum_d2 = tot[0];
    stats->sum_xin2 = tot[1];
    stats->sum_ddp = tot[2];
    stats->sum_dp2 = tot[3];
    stats->max_abs_out = tot[4];
    stats->sum_abs_out = tot[5];
    stats->count = static_cast<double>(n);
  }
}

__global__ void __launch_bounds__(kStThreads) skip_apply_kernel(const uint16_t* __restrict__ x_in,
                                                                const uint16_t* __restrict__ delta,
                                                                uint16_t* x_out, int64_t n, const int32_t* mode_dev,
                                                                sixbit_stats* stats, void* scratch) {
  if (mode_is_not(mode_dev, SIXBIT_MODE_SKIP)) return;
  const int64_t n8 = n >> 3;
  float mx = 0.f;
  TwoF sa{0.f, 0.f};
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kStThreads) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * kStThreads) {
    float a[8], d[8];
    unpack8(ld16(x_in + 8 * i), a);
    unpack8(ld16(delta + 8 * i), d);
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      w[j] = pack2(__fadd_rn(a[2 * j], d[2 * j]), __fadd_rn(a[2 * j + 1], d[2 * j + 1]));
      const float o0 = fabsf(__uint_as_float(w[j] << 16)), o1 = fabsf(__uint_as_float(w[j] & 0xFFFF0000u));
      mx = fmaxf(mx, fmaxf(o0, o1));
      two_add(sa, o0);
      two_add(sa, o1);
    }
    *reinterpret_cast<uint4*>(x_out + 8 * i) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  double v[2] = {static_cast<double>(mx), to_d(sa)};
  const bool is_max[2] = {true, false};
  double tot[2];
  if (grid_reduce<2>(v, is_max, scratch_view(scratch), tot)) {
    stats->max_abs_out = tot[0];
    stats->sum_abs_out = tot[1];
    stats->count = static_cast<double>(n);
  }
}

// ------------------------------------------------------------------ policy --

__device__ __forceinline__ bool near_thr(double v, double thr, double rel) { return fabs(v - thr) <= rel * fabs(thr); }

__global__ void policy_kernel(sixbit_policy_cfg cfg, sixbit_policy_state* st, const sixbit_stats* last,
                              const double* in_stats, int32_t* mode_out) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  sixbit_policy_state s = *st;
  // fold the statistics of the previous computed step
  if (s.pending) {
    const sixbit_stats L = *last;
    s.gamma = (L.sum_xin2 == 0.0) ? __longlong_as_double(0x7FF0000000000000ll)
                                  : __dsqrt_rn(L.sum_d2) / __dsqrt_rn(L.sum_xin2);
    s.have_gamma = 1;
    if (s.n_computed >= 1) {
      double c;
      if (L.sum_d2 == 0.0 && L.sum_dp2 == 0.0) c = 1.0;
      else if (L.sum_d2 == 0.0 || L.sum_dp2 == 0.0) c = 0.0;
      else c = L.sum_ddp / __dsqrt_rn(L.sum_d2 * L.sum_dp2);
      s.cos = c;
    }
    s.n_computed += 1;
    s.acc = 0.0;
    s.skipped_last = 0;
    s.pending = 0;
  }
  const double mx = in_stats[0], sabs = in_stats[1], cnt = in_stats[2];
  const double ratio = (sabs == 0.0) ? 0.0 : mx / (sabs / cnt);
  int word = 0;
  bool near = false, refresh = false;
  bool decided = false;
  if (s.n_computed >= 2) {
    near |= near_thr(s.cos, cfg.cos_thr, cfg.near_rel);
    if (s.cos >= cfg.cos_thr) {
      const double pred = s.acc + (1.0 - s.cos);
      near |= near_thr(pred, cfg.err_cap, cfg.near_rel);
      if (pred <= cfg.err_cap) {
        s.acc = pred;
        s.skipped_last = 1;
        word = SIXBIT_MODE_SKIP;
        s.n_skip += 1;
        decided = true;
      } else {
        refresh = true;
      }
    }
  }
  if (!decided) {
    near |= near_thr(ratio, cfg.pdr_ratio, cfg.near_rel);
    if (ratio > cfg.pdr_ratio || (refresh && cfg.refresh_bf16)) {
      word = SIXBIT_MODE_BF16 | (ratio > cfg.pdr_ratio ? SIXBIT_FLAG_PDR : 0);
      if (ratio > cfg.pdr_ratio) s.n_pdr += 1;
      s.n_bf16 += 1;
    } else if (s.skipped_last || !s.have_gamma) {
      word = SIXBIT_MODE_INT8 | (s.skipped_last ? SIXBIT_FLAG_POSTSKIP : 0);
      s.n_int8 += 1;
    } else {
      near |= near_thr(s.gamma, cfg.gamma_thr, cfg.near_rel);
      if (s.gamma >= cfg.gamma_thr) {
        word = SIXBIT_MODE_INT8;
        s.n_int8 += 1;
      } else {
        word = SIXBIT_MODE_NVFP4;
        s.n_nvfp4 += 1;
      }
    }
    if (refresh) {
      word |= SIXBIT_FLAG_REFRESH;
      s.n_refresh += 1;
    }
    s.pending = 1;
  }
  if (near) {
    word |= SIXBIT_FLAG_NEAR;
    s.n_near += 1;
  }
  s.last_word = word;
  s.steps += 1;
  *st = s;
  *mode_out = word;
}

// ------------------------------------------------------------ host launch --

static int stats_grid(int64_t n) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 152;
  }
  const int64_t per = static_cast<int64_t>(kStThreads) * 8 * 4;  // >= 4 iterations per thread
  int64_t want = (n + per - 1) / per;
  const int64_t cap = static_cast<int64_t>(sms) * 8 < kStMaxBlocks ? static_cast<int64_t>(sms) * 8 : kStMaxBlocks;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return static_cast<int>(want);
}

size_t stats_scratch_bytes(int64_t) { return 16 + static_cast<size_t>(kStMaxBlocks) * kNumSums * sizeof(double); }

cudaError_t launch_tensor_stats(const uint16_t* x, int64_t n, double* out, void* scratch, cudaStream_t st) {
  tensor_stats_kernel<<<stats_grid(n), kStThreads, 0, st>>>(x, n, out, scratch);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_block_stats(const uint16_t* x_in, const uint16_t* x_out, uint16_t* delta, int64_t n,
                               const int32_t* mode_dev, sixbit_stats* stats, void* scratch, cudaStream_t st) {
  block_stats_kernel<<<stats_grid(n), kStThreads, 0, st>>>(x_in, x_out, delta, n, mode_dev, stats, scratch);
  note_launch();
  return cudaGetLastError();
}

// Same kernel with a fixed amount of work per CTA (kFixedElemsPerCta), so the
// grid -- and with it the per-CTA partials in scratch -- grows with n.  Used
// by the allocation-free entry point, whose scratch has a fixed capacity.
cudaError_t launch_block_stats_fixed_grid(const uint16_t* x_in, const uint16_t* x_out, uint16_t* delta, int64_t n,
                                          const int32_t* mode_dev, sixbit_stats* stats, void* scratch,
                                          cudaStream_t st) {
  const int64_t grid = (n + kFixedElemsPerCta - 1) / kFixedElemsPerCta;
  block_stats_kernel<<<static_cast<unsigned int>(grid), kStThreads, 0, st>>>(x_in, x_out, delta, n, mode_dev, stats,
                                                                             scratch);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_skip_apply(const uint16_t* x_in, const uint16_t* delta, uint16_t* x_out, int64_t n,
                              const int32_t* mode_dev, sixbit_stats* stats, void* scratch, cudaStream_t st) {
  skip_apply_kernel<<<stats_grid(n), kStThreads, 0, st>>>(x_in, delta, x_out, n, mode_dev, stats, scratch);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_policy(const sixbit_policy_cfg& cfg, sixbit_policy_state* st_dev, const sixbit_stats* last,
                          const double* in_stats, int32_t* mode_out, cudaStream_t st) {
  policy_kernel<<<1, 32, 0, st>>>(cfg, st_dev, last, in_stats, mode_out);
  note_launch();
  return cudaGetLastError();
}

}  // namespace sixbit
