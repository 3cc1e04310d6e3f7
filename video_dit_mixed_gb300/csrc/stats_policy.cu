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
// and products of bf16 values are exact in FP32 per term.  The three sums
// behind the delta cosine (whose threshold sits near 1) are kept per thread
// as an unevaluated pair (s, c) updated with Knuth's TwoSum (about 48 bits);
// the sums for Gamma and the outlier ratio use Kahan compensation.  Partials
// are combined as float-float pairs in a fixed order (warp shuffle tree, then
// CTA, then a last-CTA pass over the per-CTA partials in scratch) and widened
// to float64 once at the end, so results are run-to-run deterministic.
#include <cstdint>

#include "common.cuh"
#include "ctx_cache.h"
#include "internal.h"
#include "stats_common.cuh"

namespace sixbit {

constexpr int kStThreads = 256;
constexpr int kStMaxBlocks = 1216;  // 152 SMs x 8
constexpr int kNumSums = 8;


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
  FF* partial;  // [gridDim.x][kNumSums]
};

__device__ __forceinline__ Scratch scratch_view(void* p) {
  Scratch s;
  s.counter = reinterpret_cast<unsigned int*>(p);
  s.partial = reinterpret_cast<FF*>(reinterpret_cast<char*>(p) + 16);
  return s;
}


// Combines the warps' values through shared memory; the CTA's result ends up
// in warp 0.
template <int NS>
__device__ __forceinline__ void cta_reduce(FF (&v)[NS], const bool (&is_max)[NS], FF (*red)[NS]) {
  constexpr int kWarps = kStThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_reduce<NS>(v, is_max);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < NS; ++k) red[warp][k] = v[k];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < NS; ++k) v[k] = lane < kWarps ? red[lane][k] : FF{0.f, 0.f};
    warp_reduce<NS, kWarps>(v, is_max);
  }
}

// Reduces per-thread values v[0..NS) (maxima where is_max, sums otherwise)
// across the grid in a fixed order: warp tree, CTA, then the last CTA to finish
// folds the per-CTA partials in scratch.  Returns true in exactly one thread
// (W0: in every lane of warp 0 of the last CTA), with the totals in `tot`.
// All values are non-negative except sums of products, whose error stays
// relative to the sum of magnitudes.
template <int NS, bool W0 = false>
__device__ bool grid_reduce(FF (&v)[NS], const bool (&is_max)[NS], Scratch sc, double (&tot)[NS]) {
  __shared__ FF red[kStThreads / 32][NS];
  __shared__ bool last;
  cta_reduce<NS>(v, is_max, red);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < NS; ++k) sc.partial[static_cast<size_t>(blockIdx.x) * kNumSums + k] = v[k];
    __threadfence();
    const unsigned int done = atomicAdd(sc.counter, 1u);
    last = (done == gridDim.x - 1);
  }
  __syncthreads();
  if (!last) return false;
  __threadfence();
  // last CTA: thread t folds partials t, t + 256, ... then the same trees
#pragma unroll
  for (int k = 0; k < NS; ++k) v[k] = FF{0.f, 0.f};
  for (unsigned int b = threadIdx.x; b < gridDim.x; b += kStThreads) {
    const float2* row = reinterpret_cast<const float2*>(sc.partial + static_cast<size_t>(b) * kNumSums);
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      const float2 r = __ldcg(row + k);  // L2: written by other CTAs
      const FF y{r.x, r.y};
      v[k] = is_max[k] ? ff_max(v[k], y) : ff_add(v[k], y);
    }
  }
  __syncthreads();  // red is reused
  cta_reduce<NS>(v, is_max, red);
  if constexpr (W0) {
    if (threadIdx.x >= 32) return false;
#pragma unroll
    for (int k = 0; k < NS; ++k)  // lane 0 holds the result
      tot[k] = static_cast<double>(__shfl_sync(0xffffffffu, v[k].hi, 0)) +
               static_cast<double>(__shfl_sync(0xffffffffu, v[k].lo, 0));
    if (threadIdx.x == 0) *sc.counter = 0;  // leave the scratch ready for the next call
    return true;
  } else {
    if (threadIdx.x != 0) return false;
#pragma unroll
    for (int k = 0; k < NS; ++k) tot[k] = static_cast<double>(v[k].hi) + static_cast<double>(v[k].lo);
    *sc.counter = 0;  // leave the scratch ready for the next call
    return true;
  }
}

__device__ __forceinline__ bool mode_is_not(const int32_t* mode_dev, int want) {
  return mode_dev != nullptr && SIXBIT_MODE_OF(*mode_dev) != want;
}

__device__ __forceinline__ bool mode_is(const int32_t* mode_dev, int want) {
  return mode_dev != nullptr && SIXBIT_MODE_OF(*mode_dev) == want;
}

// Each thread walks vectors of 8 elements (four packed pairs) with a grid
// stride, several vectors per iteration (their loads issued before any is
// used).


__device__ __forceinline__ void tensor_stats_vec(const uint4& r, float& mx, Kahan2& sa, Kahan2& sq) {
  uint64_t v[4];
  unpack4x2(r, v);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    mx = f2_max_abs(v[j], mx);
    kahan_add2(sa, f2_abs(v[j]));
    kahan_add2(sq, f2_mul(v[j], v[j]));
  }
}

// Grid-wide {max |x|, sum |x|, sum x^2} of x[0..n); true in one thread of
// the last CTA (W0: in its warp 0), with the totals in tot.
template <bool W0 = false>
__device__ bool tensor_stats_body(const uint16_t* __restrict__ x, int64_t n, void* scratch, double (&tot)[3]) {
  const int64_t n8 = n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kStThreads;
  float mx = 0.f;
  Kahan2 sa{0, 0}, sq{0, 0};
  // four vectors a thread per iteration, all four loads issued before any is
  // used (few registers are live here, so more bytes can be in flight)
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kStThreads) + threadIdx.x; i < n8; i += 4 * stride) {
    uint4 r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) r[u] = i + u * stride < n8 ? ld16(x + 8 * (i + u * stride)) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 4; ++u) tensor_stats_vec(r[u], mx, sa, sq);   // zeros add nothing
  }
  FF v[3] = {FF{mx, 0.f}, to_ff(sa), to_ff(sq)};
  const bool is_max[3] = {true, false, false};
  return grid_reduce<3, W0>(v, is_max, scratch_view(scratch), tot);
}

// out[0..3] = {max |x|, sum |x|, count, sum x^2}
__global__ void __launch_bounds__(kStThreads) tensor_stats_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                                  double* out, void* scratch) {
  double tot[3];
  if (tensor_stats_body(x, n, scratch, tot)) {
    out[0] = tot[0];
    out[1] = tot[1];
    out[2] = static_cast<double>(n);
    out[3] = tot[2];
  }
}


// One pass over x_in, x_out, Delta_prev: writes Delta_new over Delta_prev and
// reduces {sum Delta^2, sum x_in^2, sum Delta*Delta_prev, sum Delta_prev^2,
// max |x_out|, sum |x_out|}; true in one thread of the last CTA (W0: in its
// warp 0).
template <bool W0 = false>
__device__ bool block_stats_body(const uint16_t* __restrict__ x_in, const uint16_t* __restrict__ x_out,
                                 uint16_t* delta, int64_t n, void* scratch, double (&tot)[6]) {
  const int64_t n8 = n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kStThreads;
  float mx = 0.f;
  TwoF2 d2{0, 0}, ddp{0, 0}, dp2{0, 0};
  Kahan2 xi2{0, 0}, sa{0, 0};
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kStThreads) + threadIdx.x; i < n8; i += 2 * stride) {
    const int64_t i1 = i + stride;
    const bool two = i1 < n8;
    const uint4 a0 = ld16(x_in + 8 * i), b0 = ld16(x_out + 8 * i);
    const uint4 p0 = *reinterpret_cast<const uint4*>(delta + 8 * i);
    uint4 a1 = make_uint4(0, 0, 0, 0), b1 = a1, p1 = a1;
    if (two) {
      a1 = ld16(x_in + 8 * i1);
      b1 = ld16(x_out + 8 * i1);
      p1 = *reinterpret_cast<const uint4*>(delta + 8 * i1);
    }
    *reinterpret_cast<uint4*>(delta + 8 * i) = block_stats_vec(a0, b0, p0, d2, xi2, ddp, dp2, mx, sa);
    const uint4 w1 = block_stats_vec(a1, b1, p1, d2, xi2, ddp, dp2, mx, sa);  // zeros add nothing
    if (two) *reinterpret_cast<uint4*>(delta + 8 * i1) = w1;
  }
  FF v[6] = {to_ff(d2), to_ff(xi2), to_ff(ddp), to_ff(dp2), FF{mx, 0.f}, to_ff(sa)};
  const bool is_max[6] = {false, false, false, false, true, false};
  return grid_reduce<6, W0>(v, is_max, scratch_view(scratch), tot);
}

__device__ __forceinline__ void write_block_stats(sixbit_stats* stats, const double (&tot)[6], int64_t n) {
  stats->sum_d2 = tot[0];
  stats->sum_xin2 = tot[1];
  stats->sum_ddp = tot[2];
  stats->sum_dp2 = tot[3];
  stats->max_abs_out = tot[4];
  stats->sum_abs_out = tot[5];
  stats->count = static_cast<double>(n);
}

__global__ void __launch_bounds__(kStThreads) block_stats_kernel(const uint16_t* __restrict__ x_in,
                                                                 const uint16_t* __restrict__ x_out,
                                                                 uint16_t* delta, int64_t n, const int32_t* mode_dev,
                                                                 sixbit_stats* stats, void* scratch) {
  if (mode_is(mode_dev, SIXBIT_MODE_SKIP)) return;
  double tot[6];
  if (block_stats_body(x_in, x_out, delta, n, scratch, tot)) write_block_stats(stats, tot, n);
}

__device__ __forceinline__ uint4 skip_vec(const uint4& ra, const uint4& rd, float& mx, Kahan2& sa) {
  uint64_t a[4], d[4];
  unpack4x2(ra, a);
  unpack4x2(rd, d);
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    w[j] = f2_to_bf16x2(f2_add(a[j], d[j]));      // x_out = bf16(x_in + Delta)
    const uint64_t o = f2_from_bf16x2(w[j]);
    mx = f2_max_abs(o, mx);
    kahan_add2(sa, f2_abs(o));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(kStThreads) skip_apply_kernel(const uint16_t* __restrict__ x_in,
                                                                const uint16_t* __restrict__ delta,
                                                                uint16_t* x_out, int64_t n, const int32_t* mode_dev,
                                                                sixbit_stats* stats, void* scratch) {
  if (mode_is_not(mode_dev, SIXBIT_MODE_SKIP)) return;
  const int64_t n8 = n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kStThreads;
  float mx = 0.f;
  Kahan2 sa{0, 0};
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kStThreads) + threadIdx.x; i < n8; i += 2 * stride) {
    const int64_t i1 = i + stride;
    const bool two = i1 < n8;
    const uint4 a0 = ld16(x_in + 8 * i), d0 = ld16(delta + 8 * i);
    uint4 a1 = make_uint4(0, 0, 0, 0), d1 = a1;
    if (two) {
      a1 = ld16(x_in + 8 * i1);
      d1 = ld16(delta + 8 * i1);
    }
    *reinterpret_cast<uint4*>(x_out + 8 * i) = skip_vec(a0, d0, mx, sa);
    const uint4 w1 = skip_vec(a1, d1, mx, sa);  // zeros add nothing
    if (two) *reinterpret_cast<uint4*>(x_out + 8 * i1) = w1;
  }
  FF v[2] = {FF{mx, 0.f}, to_ff(sa)};
  const bool is_max[2] = {true, false};
  double tot[2];
  if (grid_reduce<2>(v, is_max, scratch_view(scratch), tot)) {
    stats->max_abs_out = tot[0];
    stats->sum_abs_out = tot[1];
    stats->count = static_cast<double>(n);
  }
}

// ------------------------------------------------- MXFP8 Delta cache --
//
// The cache can hold each Delta in MXFP8 (OCP Microscaling, E4M3 elements):
// blocks of 32 consecutive elements share an E8M0 scale 2^X with
// X = floor(log2 amax) - 8 (clamped to >= -127; a zero block takes -127), and
// element k is E4M3(Delta_k / 2^X), round to nearest even, saturating at 448.
// Codes: [n] bytes, element k in byte k; scales: [n / 32] E8M0 bytes (X + 127).
// The fresh bf16 Delta feeds the statistics as it is and is then encoded; the
// previous Delta enters the statistics (and a skip) dequantized, which is
// exact in FP32 (4 significant bits times 2^X, X >= -127).
//
// In the grid-stride loops a thread's vector index i has i % 4 == lane % 4
// (the CTA size and the stride are multiples of 4), so lanes 4g .. 4g+3 hold
// one 32-element block: its maximum is two xor-shuffles among those lanes,
// and with n % 32 == 0 every branch is uniform over the four.

// 2^(c - 127) for an E8M0 code (c = 0: 2^-127, a subnormal; c = 255: NaN)
__device__ __forceinline__ float e8m0_value(uint32_t c) {
  return __uint_as_float(c == 0 ? 0x00400000u : (c == 255 ? 0x7FC00000u : c << 23));
}

// E8M0 code of a block whose largest magnitude is amax >= 0: the biased FP32
// exponent of amax minus 8, or 0 (X = -127) for amax below 2^-118.
__device__ __forceinline__ uint32_t mx_scale_code(float amax) {
  const int e = static_cast<int>(__float_as_uint(amax) >> 23);
  return static_cast<uint32_t>(e > 8 ? e - 8 : 0);
}

__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(static_cast<uint16_t>(h)));
  return f;
}

// eight E4M3 codes (element k in byte k) times 2^X -> four FP32 pairs (exact)
__device__ __forceinline__ void mx_unpack8(const uint2& c, float scale, uint64_t (&p)[4]) {
  const uint64_t s2 = f2_pack(scale, scale);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w = j < 2 ? c.x : c.y;
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(w >> (16 * (j & 1)))));
    p[j] = f2_mul(f2_pack(f16_bits_to_f32(h2 & 0xFFFFu), f16_bits_to_f32(h2 >> 16)), s2);
  }
}

// four FP32 pairs times 2^-X -> eight E4M3 codes (RN, satfinite)
__device__ __forceinline__ uint2 mx_pack8(const uint64_t (&d)[4], uint32_t code) {
  const float inv = __uint_as_float((254u - code) << 23);  // 2^-X, X in [-127, 119]: a normal float
  const uint64_t i2 = f2_pack(inv, inv);
  uint32_t h[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t q = f2_mul(d[j], i2);  // exact unless it underflows, which rounds to zero in E4M3 anyway
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(f2_hi(q)), "f"(f2_lo(q)));
    h[j] = r;
  }
  return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

__device__ __forceinline__ uint2 ld8(const void* p) {
  uint2 v;
  asm volatile("ld.global.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld8_nc(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_u8_nc(const uint8_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// One vector of the MXFP8 block-statistics pass (vector i of the caller's
// loop, whose four-lane group is `gmask`): statistics as block_stats_vec with
// the previous Delta (codes pc; scale byte ps, read by the group leader)
// dequantized, then the new Delta encoded over it.  The leader read the old
// scale before it writes the new one, so read and write are one thread's.
__device__ __forceinline__ void block_stats_mx_vec(const uint4& ra, const uint4& rb, const uint2& pc, uint32_t ps,
                                                   uint8_t* codes, uint8_t* scales, int64_t i, unsigned gmask,
                                                   int leader, TwoF2& d2, Kahan2& xi2, TwoF2& ddp, TwoF2& dp2,
                                                   float& mx, Kahan2& sa) {
  ps = __shfl_sync(gmask, ps, leader);
  uint64_t a[4], b[4], p[4], d[4];
  unpack4x2(ra, a);
  unpack4x2(rb, b);
  mx_unpack8(pc, e8m0_value(ps), p);
  float dmax = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    d[j] = f2_from_bf16x2(f2_to_bf16x2(f2_sub(b[j], a[j])));  // Delta = bf16(x_out - x_in)
    two_add2(d2, f2_mul(d[j], d[j]));
    two_add2(ddp, f2_mul(d[j], p[j]));
    two_add2(dp2, f2_mul(p[j], p[j]));
    kahan_add2(xi2, f2_mul(a[j], a[j]));
    mx = f2_max_abs(b[j], mx);
    kahan_add2(sa, f2_abs(b[j]));
    dmax = f2_max_abs(d[j], dmax);
  }
  dmax = fmaxf(dmax, __shfl_xor_sync(gmask, dmax, 1));
  dmax = fmaxf(dmax, __shfl_xor_sync(gmask, dmax, 2));
  const uint32_t code = mx_scale_code(dmax);
  *reinterpret_cast<uint2*>(codes + 8 * i) = mx_pack8(d, code);
  if ((threadIdx.x & 3) == 0) scales[i >> 2] = static_cast<uint8_t>(code);
}

__device__ __forceinline__ uint32_t ld_u8(const uint8_t* p) {
  uint16_t v;
  asm volatile("ld.global.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// block_stats_body with the Delta cache in MXFP8 (n % 32 == 0).  Both
// vectors' loads (activations, codes, the leader's scale bytes) are issued
// before either is used.
template <bool W0 = false>
__device__ bool block_stats_mx_body(const uint16_t* __restrict__ x_in, const uint16_t* __restrict__ x_out,
                                    uint8_t* codes, uint8_t* scales, int64_t n, void* scratch, double (&tot)[6]) {
  const int64_t n8 = n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kStThreads;
  const int lane = threadIdx.x & 31, leader = lane & ~3;
  const unsigned gmask = 0xFu << leader;
  const bool lead = (lane & 3) == 0;
  float mx = 0.f;
  TwoF2 d2{0, 0}, ddp{0, 0}, dp2{0, 0};
  Kahan2 xi2{0, 0}, sa{0, 0};
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kStThreads) + threadIdx.x; i < n8; i += 2 * stride) {
    const int64_t i1 = i + stride;
    const bool two = i1 < n8;  // uniform over the four lanes of a block
    const uint4 a0 = ld16(x_in + 8 * i), b0 = ld16(x_out + 8 * i);
    const uint2 c0 = ld8(codes + 8 * i);
    const uint32_t s0 = lead ? ld_u8(scales + (i >> 2)) : 0u;
    uint4 a1 = make_uint4(0, 0, 0, 0), b1 = a1;
    uint2 c1 = make_uint2(0, 0);
    uint32_t s1 = 0;
    if (two) {
      a1 = ld16(x_in + 8 * i1);
      b1 = ld16(x_out + 8 * i1);
      c1 = ld8(codes + 8 * i1);
      if (lead) s1 = ld_u8(scales + (i1 >> 2));
    }
    block_stats_mx_vec(a0, b0, c0, s0, codes, scales, i, gmask, leader, d2, xi2, ddp, dp2, mx, sa);
    if (two) block_stats_mx_vec(a1, b1, c1, s1, codes, scales, i1, gmask, leader, d2, xi2, ddp, dp2, mx, sa);
  }
  FF v[6] = {to_ff(d2), to_ff(xi2), to_ff(ddp), to_ff(dp2), FF{mx, 0.f}, to_ff(sa)};
  const bool is_max[6] = {false, false, false, false, true, false};
  return grid_reduce<6, W0>(v, is_max, scratch_view(scratch), tot);
}

__global__ void __launch_bounds__(kStThreads) block_stats_mx_kernel(const uint16_t* __restrict__ x_in,
                                                                    const uint16_t* __restrict__ x_out,
                                                                    uint8_t* codes, uint8_t* scales, int64_t n,
                                                                    const int32_t* mode_dev, sixbit_stats* stats,
                                                                    void* scratch) {
  if (mode_is(mode_dev, SIXBIT_MODE_SKIP)) return;
  double tot[6];
  if (block_stats_mx_body(x_in, x_out, codes, scales, n, scratch, tot)) write_block_stats(stats, tot, n);
}

// v += dequantized Delta (vector i of a cache with `codes` / `scales`), rounded to bf16 per element
__device__ __forceinline__ void mx_skip_add(uint64_t (&v)[4], const uint2& c, uint32_t sc) {
  uint64_t d[4];
  mx_unpack8(c, e8m0_value(sc), d);
#pragma unroll
  for (int q = 0; q < 4; ++q) v[q] = f2_from_bf16x2(f2_to_bf16x2(f2_add(v[q], d[q])));
}

__global__ void __launch_bounds__(kStThreads) skip_apply_mx_kernel(const uint16_t* __restrict__ x_in,
                                                                   const uint8_t* __restrict__ codes,
                                                                   const uint8_t* __restrict__ scales,
                                                                   uint16_t* x_out, int64_t n, const int32_t* mode_dev,
                                                                   sixbit_stats* stats, void* scratch) {
  if (mode_is_not(mode_dev, SIXBIT_MODE_SKIP)) return;
  const int64_t n8 = n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kStThreads;
  float mx = 0.f;
  Kahan2 sa{0, 0};
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kStThreads) + threadIdx.x; i < n8; i += stride) {
    uint64_t v[4];
    unpack4x2(ld16(x_in + 8 * i), v);
    mx_skip_add(v, ld8_nc(codes + 8 * i), ld_u8_nc(scales + (i >> 2)));
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      w[q] = f2_to_bf16x2(v[q]);  // exact: v holds bf16 values
      mx = f2_max_abs(v[q], mx);
      kahan_add2(sa, f2_abs(v[q]));
    }
    *reinterpret_cast<uint4*>(x_out + 8 * i) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  FF v[2] = {FF{mx, 0.f}, to_ff(sa)};
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

// One decision of the per-block policy: folds the previous compute's
// statistics into `s` if it is pending, decides, and updates `s`.  Returns
// the decision word.  A pure function of (cfg, s, *last, in_stats), shared by
// the policy kernel and by the skip-run look-ahead below.
__device__ int policy_decide(const sixbit_policy_cfg& cfg, sixbit_policy_state& s, const sixbit_stats* last,
                             const double* in_stats) {
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
  // A statistic that is not a number (a corrupted or overflowed sum) fails
  // its threshold test toward the safer path: a NaN cosine never skips, a
  // NaN Gamma picks INT8, a NaN input ratio picks BF16; each such decision
  // is counted (n_nonfinite).
  int word = 0;
  bool near = false, refresh = false, nonfinite = false;
  bool decided = false;
  if (s.n_computed >= 2) {
    nonfinite |= isnan(s.cos);
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
    // the input's max/mean ratio only matters when the block computes (two
    // float64 divisions, slow on this GPU, are not spent on a skip)
    const double mx = in_stats[0], sabs = in_stats[1], cnt = in_stats[2];
    const double ratio = (sabs == 0.0) ? 0.0 : mx / (sabs / cnt);
    const bool pdr = !(ratio <= cfg.pdr_ratio);  // ratio > pdr_ratio, or not a number
    nonfinite |= isnan(ratio);
    near |= near_thr(ratio, cfg.pdr_ratio, cfg.near_rel);
    if (pdr || (refresh && cfg.refresh_bf16)) {
      word = SIXBIT_MODE_BF16 | (pdr ? SIXBIT_FLAG_PDR : 0);
      if (pdr) s.n_pdr += 1;
      s.n_bf16 += 1;
    } else if (s.skipped_last || !s.have_gamma) {
      word = SIXBIT_MODE_INT8 | (s.skipped_last ? SIXBIT_FLAG_POSTSKIP : 0);
      s.n_int8 += 1;
    } else {
      near |= near_thr(s.gamma, cfg.gamma_thr, cfg.near_rel);
      nonfinite |= isnan(s.gamma);
      if (!(s.gamma < cfg.gamma_thr)) {  // Gamma >= gamma_thr, or not a number
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
  if (nonfinite) s.n_nonfinite += 1;
  if (near) {
    word |= SIXBIT_FLAG_NEAR;
    s.n_near += 1;
  }
  s.last_word = word;
  s.steps += 1;
  return word;
}

__global__ void policy_kernel(sixbit_policy_cfg cfg, sixbit_policy_state* st, const sixbit_stats* last,
                              const double* in_stats, int32_t* mode_out) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  sixbit_policy_state s = *st;
  const int word = policy_decide(cfg, s, last, in_stats);
  *st = s;
  *mode_out = word;
}

// ----------------------------------------------- the DiT step protocol --
//
// Per step, block l's decision needs the statistics of its input, which the
// last kernel before it produces; so every decision is taken at the tail of
// that kernel, by warp 0 of the CTA that holds the totals:
//   dit_begin_kernel     statistics of x0, then the decision of block 0;
//   dit_block_end_kernel block statistics + Delta update of a computed block
//                        l, then the decision of block l+1;
//   dit_skip_run_kernel  the skip of the run of blocks l .. l+k-1 that block
//                        l starts, then the decision of block l+k.
// A skip decision depends only on the block's own state (cos, acc, number of
// computes) and the statistics of its last compute, never on its input, so
// when block l skips, the run of blocks that will skip after it is already
// fixed: decide_block finds it (the warp's lanes evaluate the following
// blocks in parallel), decides those blocks as well (recording their states
// and mode words; they launch nothing) and records k in run_len[l].  The
// run's output x_{l+k-1} = bf16(... bf16(bf16(x_{l-1} + D_l) + D_{l+1}) ... +
// D_{l+k-1}) is written in one pass (the same roundings as k separate skips;
// the intermediate activations are never read, so they are not written),
// with its {max, sum |x|, count} into stats[l+k-1].  Each decision also sets
// the block's graph condition when a handle array is given: a compute mode
// to its body (0, 1, 2), a run start to 3, a block inside a run to none (4).
// The protocol's kernels cap registers at 64 (launch bounds; 80 for the
// MXFP8-cache block end, which keeps both vectors' loads in flight): the
// decisions run in one warp at the tail and may spill; the streaming body
// may not.
__device__ __forceinline__ const double* block_in_stats(const sixbit_dit_blocks& B, int l) {
  return l == 0 ? B.in_stats0 : &B.stats[l - 1].max_abs_out;  // {max, sum |x|, count}
}

constexpr int kDitBranches = 4;

__device__ __forceinline__ void set_branch(const sixbit_dit_blocks& B, int l, int branch) {
  if (B.conds != nullptr)
    cudaGraphSetConditional(static_cast<cudaGraphConditionalHandle>(B.conds[l]),
                            (branch >= 0 && branch < kDitBranches) ? static_cast<unsigned int>(branch)
                                                                   : static_cast<unsigned int>(kDitBranches));
}

// Decides block l (all 32 lanes of one warp call it; lane 0 decides).  When
// block l starts a run, the blocks after it are evaluated 32 at a time, one
// per lane -- a skip depends only on the block's own state and statistics,
// so the evaluations are independent -- and the run is the leading skips
// (__ballot_sync): only those blocks are recorded (state, mode word, no
// body), exactly the ones a walk that stops at the first non-skip records;
// the first non-skip is decided later, from the run's output statistics.
// Block l's thresholds: its own entry of B.block_cfg (per-depth thresholds), or the step's cfg.
__device__ __forceinline__ sixbit_policy_cfg cfg_of(const sixbit_policy_cfg& cfg, const sixbit_dit_blocks& B, int l) {
  return B.block_cfg != nullptr ? B.block_cfg[l] : cfg;
}

__device__ void decide_block(const sixbit_policy_cfg& cfg, const sixbit_dit_blocks& B, int l) {
  const int lane = threadIdx.x & 31;
  int word = 0;
  if (lane == 0) {
    sixbit_policy_state s = B.states[l];
    word = policy_decide(cfg_of(cfg, B, l), s, &B.stats[l], block_in_stats(B, l));
    B.states[l] = s;
    B.modes[l] = word;
    if (SIXBIT_MODE_OF(word) != SIXBIT_MODE_SKIP) set_branch(B, l, SIXBIT_MODE_OF(word) - SIXBIT_MODE_NVFP4);
  }
  word = __shfl_sync(0xffffffffu, word, 0);
  if (SIXBIT_MODE_OF(word) != SIXBIT_MODE_SKIP) return;  // compute modes: branches 0, 1, 2
  int k = 1;
  for (int base = l + 1; base < B.L; base += 32) {
    const int j = base + lane;
    sixbit_policy_state sj{};
    int wj = 0;
    bool skip = false;
    if (j < B.L) {
      sj = B.states[j];
      const sixbit_stats tj = B.stats[j];
      wj = policy_decide(cfg_of(cfg, B, j), sj, &tj, &B.stats[j - 1].max_abs_out);  // input: block j-1's output
      skip = SIXBIT_MODE_OF(wj) == SIXBIT_MODE_SKIP;
    }
    const unsigned sk = __ballot_sync(0xffffffffu, skip);
    const int lead = sk == 0xffffffffu ? 32 : __ffs(~sk) - 1;  // leading skips (lanes past L vote no)
    if (lane < lead) {
      B.states[j] = sj;
      B.modes[j] = wj;
      set_branch(B, j, kDitBranches);  // applied by the run: no body
    }
    k += lead;
    if (lead < 32) break;
  }
  if (lane == 0) {
    B.run_len[l] = static_cast<uint32_t>(k);
    set_branch(B, l, 3);
  }
}

// (selects, not an index into the parameter array: that would copy B to local memory)
__device__ __forceinline__ const uint16_t* block_input(const sixbit_dit_blocks& B, int l) {
  return l == 0 ? B.x0 : (((l - 1) & 1) ? B.buf[1] : B.buf[0]);
}
__device__ __forceinline__ uint16_t* block_output(const sixbit_dit_blocks& B, int l) {
  return (l & 1) ? B.buf[1] : B.buf[0];
}

__global__ void __launch_bounds__(kStThreads, 4) dit_begin_kernel(sixbit_policy_cfg cfg, sixbit_dit_blocks B,
                                                               void* scratch, int32_t* err) {
  double tot[3];
  if (tensor_stats_body<true>(B.x0, B.n, scratch, tot)) {  // warp 0 of the last CTA
    if (threadIdx.x == 0) {
      B.in_stats0[0] = tot[0];
      B.in_stats0[1] = tot[1];
      B.in_stats0[2] = static_cast<double>(B.n);
      B.in_stats0[3] = tot[2];
    }
    __syncwarp();
    decide_block(cfg, B, 0);
  }
}

template <bool MX>
__global__ void __launch_bounds__(kStThreads, MX ? 3 : 4) dit_block_end_kernel(sixbit_policy_cfg cfg, sixbit_dit_blocks B, int l,
                                                                   void* scratch, int32_t* err) {
  if (SIXBIT_MODE_OF(B.modes[l]) == SIXBIT_MODE_SKIP) return;  // uniform: a skipped block has no end
  double tot[6];
  bool last;
  if constexpr (MX)
    last = block_stats_mx_body<true>(block_input(B, l), block_output(B, l),
                                     static_cast<uint8_t*>(B.deltas) + static_cast<size_t>(l) * B.n,
                                     B.delta_scales + static_cast<size_t>(l) * (B.n >> 5), B.n, scratch, tot);
  else
    last = block_stats_body<true>(block_input(B, l), block_output(B, l),
                                  static_cast<uint16_t*>(B.deltas) + static_cast<size_t>(l) * B.n, B.n, scratch, tot);
  if (last) {  // warp 0 of the last CTA
    if (threadIdx.x == 0) write_block_stats(&B.stats[l], tot, B.n);
    __syncwarp();
    if (l + 1 < B.L) decide_block(cfg, B, l + 1);
  }
}

// Folds the partial rows a GEMM epilogue wrote for a block's statistics
// (count, then rows of kBsSums float-float values; internal.h) in a fixed
// order: thread t takes rows t, t + 256, ..., then the CTA tree.  One CTA;
// true in warp 0, with the totals in tot.
__device__ bool fold_bs_parts(const void* parts, double (&tot)[kBsSums]) {
  __shared__ FF red[kStThreads / 32][kBsSums];
  const bool is_max[kBsSums] = {false, false, false, false, true, false};
  FF v[kBsSums];
#pragma unroll
  for (int k = 0; k < kBsSums; ++k) v[k] = FF{0.f, 0.f};
  const uint32_t rows = *static_cast<const uint32_t*>(parts);
  const FF* base = reinterpret_cast<const FF*>(static_cast<const char*>(parts) + 16);
  uint32_t r = threadIdx.x;
  for (; r + 3 * kStThreads < rows; r += 4 * kStThreads) {  // four rows' loads in flight
    FF y[4][kBsSums];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int k = 0; k < kBsSums; ++k) y[u][k] = base[static_cast<size_t>(r + u * kStThreads) * kBsSums + k];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int k = 0; k < kBsSums; ++k) v[k] = is_max[k] ? ff_max(v[k], y[u][k]) : ff_add(v[k], y[u][k]);
  }
  for (; r < rows; r += kStThreads) {
#pragma unroll
    for (int k = 0; k < kBsSums; ++k) {
      const FF y = base[static_cast<size_t>(r) * kBsSums + k];
      v[k] = is_max[k] ? ff_max(v[k], y) : ff_add(v[k], y);
    }
  }
  cta_reduce<kBsSums>(v, is_max, red);
  if (threadIdx.x >= 32) return false;
#pragma unroll
  for (int k = 0; k < kBsSums; ++k)
    tot[k] = static_cast<double>(__shfl_sync(0xffffffffu, v[k].hi, 0)) +
             static_cast<double>(__shfl_sync(0xffffffffu, v[k].lo, 0));
  return true;
}

__global__ void __launch_bounds__(kStThreads) block_stats_parts_kernel(const void* parts, int64_t n,
                                                                       sixbit_stats* stats) {
  double tot[kBsSums];
  if (fold_bs_parts(parts, tot) && threadIdx.x == 0) write_block_stats(stats, tot, n);
}

// dit_block_end_kernel for a block whose down projection produced the
// statistics and Delta in its epilogue: the fold, stats[l], block l+1's
// decision.
__global__ void __launch_bounds__(kStThreads) dit_block_end_parts_kernel(sixbit_policy_cfg cfg, sixbit_dit_blocks B,
                                                                         int l, const void* parts) {
  if (SIXBIT_MODE_OF(B.modes[l]) == SIXBIT_MODE_SKIP) return;  // uniform: a skipped block has no end
  double tot[kBsSums];
  if (!fold_bs_parts(parts, tot)) return;  // warp 0 continues
  if (threadIdx.x == 0) write_block_stats(&B.stats[l], tot, B.n);
  __syncwarp();
  if (l + 1 < B.L) decide_block(cfg, B, l + 1);
}

// v = bf16(v + Delta_j) for the k cached deltas of a run, in order (bf16 cache:
// vector i of each [n] slice; eight / four / one loads in flight)
__device__ __forceinline__ void skip_run_bf16(uint64_t (&v)[4], const uint16_t* dp, int64_t n, int k) {
  int j = 0;
  for (; j + 8 <= k; j += 8) {
    uint4 r[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) r[u] = ld16(dp + static_cast<size_t>(j + u) * n);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      uint64_t d[4];
      unpack4x2(r[u], d);
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = f2_from_bf16x2(f2_to_bf16x2(f2_add(v[q], d[q])));
    }
  }
  if (j + 4 <= k) {
    uint4 r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) r[u] = ld16(dp + static_cast<size_t>(j + u) * n);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint64_t d[4];
      unpack4x2(r[u], d);
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = f2_from_bf16x2(f2_to_bf16x2(f2_add(v[q], d[q])));
    }
    j += 4;
  }
  for (; j < k; ++j) {
    uint64_t d[4];
    unpack4x2(ld16(dp + static_cast<size_t>(j) * n), d);
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = f2_from_bf16x2(f2_to_bf16x2(f2_add(v[q], d[q])));
  }
}

// The same with an MXFP8 cache: cp = codes of vector i in block l's slice
// (slices n bytes apart), sp = its scale byte (slices n / 32 bytes apart);
// eight / four / one deltas in flight
__device__ __forceinline__ void skip_run_mx(uint64_t (&v)[4], const uint8_t* cp, const uint8_t* sp, int64_t n,
                                            int k) {
  const int64_t ns = n >> 5;
  int j = 0;
  for (; j + 8 <= k; j += 8) {
    uint2 c[8];
    uint32_t sc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      c[u] = ld8_nc(cp + static_cast<size_t>(j + u) * n);
      sc[u] = ld_u8_nc(sp + static_cast<size_t>(j + u) * ns);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) mx_skip_add(v, c[u], sc[u]);
  }
  if (j + 4 <= k) {
    uint2 c[4];
    uint32_t sc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      c[u] = ld8_nc(cp + static_cast<size_t>(j + u) * n);
      sc[u] = ld_u8_nc(sp + static_cast<size_t>(j + u) * ns);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) mx_skip_add(v, c[u], sc[u]);
    j += 4;
  }
  for (; j < k; ++j)
    mx_skip_add(v, ld8_nc(cp + static_cast<size_t>(j) * n), ld_u8_nc(sp + static_cast<size_t>(j) * ns));
}

template <bool MX>
__global__ void __launch_bounds__(kStThreads, 4) dit_skip_run_kernel(sixbit_policy_cfg cfg, sixbit_dit_blocks B, int l,
                                                                  void* scratch, int32_t* err) {
  const int k = static_cast<int>(B.run_len[l]);
  if (k == 0) return;  // uniform across the grid: block l starts no run
  const uint16_t* __restrict__ x_in = block_input(B, l);
  uint16_t* x_out = block_output(B, l + k - 1);
  const int64_t n8 = B.n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kStThreads;
  float mx = 0.f;
  Kahan2 sa{0, 0};
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kStThreads) + threadIdx.x; i < n8; i += stride) {
    uint64_t v[4];
    unpack4x2(ld16(x_in + 8 * i), v);
    if constexpr (MX)
      skip_run_mx(v, static_cast<const uint8_t*>(B.deltas) + static_cast<size_t>(l) * B.n + 8 * i,
                  B.delta_scales + static_cast<size_t>(l) * (B.n >> 5) + (i >> 2), B.n, k);
    else
      skip_run_bf16(v, static_cast<const uint16_t*>(B.deltas) + static_cast<size_t>(l) * B.n + 8 * i, B.n, k);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      w[q] = f2_to_bf16x2(v[q]);  // exact: v holds bf16 values
      mx = f2_max_abs(v[q], mx);
      kahan_add2(sa, f2_abs(v[q]));
    }
    *reinterpret_cast<uint4*>(x_out + 8 * i) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  FF v[2] = {FF{mx, 0.f}, to_ff(sa)};
  const bool is_max[2] = {true, false};
  double tot[2];
  if (grid_reduce<2, true>(v, is_max, scratch_view(scratch), tot)) {  // warp 0 of the last CTA
    if (threadIdx.x == 0) {
      sixbit_stats* o = &B.stats[l + k - 1];
      o->max_abs_out = tot[0];
      o->sum_abs_out = tot[1];
      o->count = static_cast<double>(B.n);
      B.run_len[l] = 0;  // every CTA has read it
    }
    __syncwarp();
    if (l + k < B.L) decide_block(cfg, B, l + k);
  }
}

// ------------------------------------------------------------ host launch --

// One wave: as many CTAs as fit on the GPU at once (occupancy of `kernel`),
// fewer for small n (at least 4 vectors per thread), never more than the
// scratch holds.
template <auto KERNEL>
static int stats_grid(int64_t n) {
  static ContextCache<int> cache;  // per kernel and context
  int resident = 0;
  if (cache.get(&resident, [](int* o) {
        int per_sm = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, KERNEL, kStThreads, 0);
        *o = sm_count() * (per_sm > 0 ? per_sm : 4);
        if (*o > kStMaxBlocks) *o = kStMaxBlocks;
        return cudaSuccess;
      }) != cudaSuccess)
    resident = kStMaxBlocks;
  const int64_t per = static_cast<int64_t>(kStThreads) * 8 * 4;
  int64_t want = (n + per - 1) / per;
  if (want > resident) want = resident;
  if (want < 1) want = 1;
  return static_cast<int>(want);
}

size_t stats_scratch_bytes(int64_t) { return 16 + static_cast<size_t>(kStMaxBlocks) * kNumSums * sizeof(FF); }
size_t bs_parts_bytes() { return 16 + static_cast<size_t>(sm_count()) * kBsSums * sizeof(FF); }

cudaError_t launch_block_stats_parts(const void* parts, int64_t n, sixbit_stats* stats, cudaStream_t st) {
  block_stats_parts_kernel<<<1, kStThreads, 0, st>>>(parts, n, stats);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_dit_block_end_parts(const sixbit_policy_cfg& cfg, const sixbit_dit_blocks& B, int l,
                                       const void* parts, cudaStream_t st) {
  dit_block_end_parts_kernel<<<1, kStThreads, 0, st>>>(cfg, B, l, parts);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_tensor_stats(const uint16_t* x, int64_t n, double* out, void* scratch, cudaStream_t st) {
  tensor_stats_kernel<<<stats_grid<tensor_stats_kernel>(n), kStThreads, 0, st>>>(x, n, out, scratch);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_block_stats(const uint16_t* x_in, const uint16_t* x_out, uint16_t* delta, int64_t n,
                               const int32_t* mode_dev, sixbit_stats* stats, void* scratch, cudaStream_t st) {
  block_stats_kernel<<<stats_grid<block_stats_kernel>(n), kStThreads, 0, st>>>(x_in, x_out, delta, n, mode_dev, stats, scratch);
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
  skip_apply_kernel<<<stats_grid<skip_apply_kernel>(n), kStThreads, 0, st>>>(x_in, delta, x_out, n, mode_dev, stats, scratch);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_dit_begin(const sixbit_policy_cfg& cfg, const sixbit_dit_blocks& B, void* scratch, int32_t* err,
                             cudaStream_t st) {
  dit_begin_kernel<<<stats_grid<dit_begin_kernel>(B.n), kStThreads, 0, st>>>(cfg, B, scratch, err);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_dit_block_end(const sixbit_policy_cfg& cfg, const sixbit_dit_blocks& B, int l, void* scratch,
                                 int32_t* err, cudaStream_t st) {
  if (B.delta_format == SIXBIT_DELTA_MXFP8)
    dit_block_end_kernel<true><<<stats_grid<dit_block_end_kernel<true>>(B.n), kStThreads, 0, st>>>(cfg, B, l, scratch,
                                                                                                  err);
  else
    dit_block_end_kernel<false><<<stats_grid<dit_block_end_kernel<false>>(B.n), kStThreads, 0, st>>>(cfg, B, l,
                                                                                                    scratch, err);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_dit_skip_run(const sixbit_policy_cfg& cfg, const sixbit_dit_blocks& B, int l, void* scratch,
                                int32_t* err, cudaStream_t st) {
  if (B.delta_format == SIXBIT_DELTA_MXFP8)
    dit_skip_run_kernel<true><<<stats_grid<dit_skip_run_kernel<true>>(B.n), kStThreads, 0, st>>>(cfg, B, l, scratch,
                                                                                                err);
  else
    dit_skip_run_kernel<false><<<stats_grid<dit_skip_run_kernel<false>>(B.n), kStThreads, 0, st>>>(cfg, B, l, scratch,
                                                                                                  err);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_block_stats_mx(const uint16_t* x_in, const uint16_t* x_out, uint8_t* codes, uint8_t* scales,
                                  int64_t n, const int32_t* mode_dev, sixbit_stats* stats, void* scratch,
                                  cudaStream_t st) {
  block_stats_mx_kernel<<<stats_grid<block_stats_mx_kernel>(n), kStThreads, 0, st>>>(x_in, x_out, codes, scales, n,
                                                                                      mode_dev, stats, scratch);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_skip_apply_mx(const uint16_t* x_in, const uint8_t* codes, const uint8_t* scales, uint16_t* x_out,
                                 int64_t n, const int32_t* mode_dev, sixbit_stats* stats, void* scratch,
                                 cudaStream_t st) {
  skip_apply_mx_kernel<<<stats_grid<skip_apply_mx_kernel>(n), kStThreads, 0, st>>>(x_in, codes, scales, x_out, n,
                                                                                    mode_dev, stats, scratch);
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
