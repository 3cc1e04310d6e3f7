// Per-thread statistics accumulators and their float-float reduction, shared
// by the statistics kernels (stats_policy.cu) and the GEMM epilogues that
// produce a block's statistics while they write its output.
//
// Method: "6Bit-Diffusion" technical summary section 2.A-2.B (the block's
// relative difference Gamma, the Temporal Delta Cache's Delta and its cosine
// with the previous Delta) and popular summary section 3 (the max/mean
// outlier ratio of the block output).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace sixbit {

// Per-thread accumulators on packed FP32 pairs (two independent lanes per
// instruction, lane-wise identical rounding); a thread accumulates even and
// odd elements in the two lanes.  TwoF2 keeps an unevaluated sum s + c with
// Knuth's TwoSum (about 48 bits); Kahan2 keeps s - c with Kahan compensation
// (error about 2u|S| for a thread's partial, enough for the outlier ratio and
// Gamma, whose bands are relative 1e-6).
struct TwoF2 {
  uint64_t s, c;
};

__device__ __forceinline__ void two_add2(TwoF2& a, uint64_t x) {
  const uint64_t s = f2_add(a.s, x);
  const uint64_t bp = f2_sub(s, a.s);
  const uint64_t err = f2_add(f2_sub(a.s, f2_sub(s, bp)), f2_sub(x, bp));
  a.s = s;
  a.c = f2_add(a.c, err);
}

struct Kahan2 {
  uint64_t s, c;
};

__device__ __forceinline__ void kahan_add2(Kahan2& k, uint64_t x) {
  const uint64_t y = f2_sub(x, k.c);
  const uint64_t t = f2_add(k.s, y);
  k.c = f2_sub(f2_sub(t, k.s), y);
  k.s = t;
}

// Float-float value hi + lo (|lo| <= ulp(hi)/2 after ff_add).  ff_add is the
// double-float addition of Dekker / Bailey: TwoSum of the high parts, then the
// low parts folded in and renormalised; its error is a few 2^-44 of |a| + |b|.
// Combining partials this way keeps GB300's slow FP64 pipe off the reduction.
struct FF {
  float hi, lo;
};

__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float bp = __fsub_rn(s, a.hi);
  const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bp)), __fsub_rn(b.hi, bp));
  const float lo = __fadd_rn(__fadd_rn(a.lo, b.lo), e);
  const float hi = __fadd_rn(s, lo);
  return FF{hi, __fsub_rn(lo, __fsub_rn(hi, s))};
}

__device__ __forceinline__ FF ff_max(FF a, FF b) { return FF{fmaxf(a.hi, b.hi), 0.f}; }

__device__ __forceinline__ FF to_ff(const TwoF2& a) {
  return ff_add(FF{f2_lo(a.s), f2_lo(a.c)}, FF{f2_hi(a.s), f2_hi(a.c)});
}

__device__ __forceinline__ FF to_ff(const Kahan2& k) {
  return ff_add(FF{f2_lo(k.s), -f2_lo(k.c)}, FF{f2_hi(k.s), -f2_hi(k.c)});
}

__device__ __forceinline__ FF ff_shfl_xor(FF a, int o) {
  return FF{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}

__device__ __forceinline__ float f2_max_abs(uint64_t v, float m) {
  return fmaxf(m, fmaxf(fabsf(f2_lo(v)), fabsf(f2_hi(v))));
}

// Combines v[k] over a warp (xor-shuffle tree; sums with ff_add, maxima with
// ff_max), leaving the result in every lane.
template <int NS, int W = 32>
__device__ __forceinline__ void warp_reduce(FF (&v)[NS], const bool (&is_max)[NS]) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) {
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      const FF y = ff_shfl_xor(v[k], o);
      v[k] = is_max[k] ? ff_max(v[k], y) : ff_add(v[k], y);
    }
  }
}

__device__ __forceinline__ void unpack4x2(const uint4& r, uint64_t (&v)[4]) {
  v[0] = f2_from_bf16x2(r.x);
  v[1] = f2_from_bf16x2(r.y);
  v[2] = f2_from_bf16x2(r.z);
  v[3] = f2_from_bf16x2(r.w);
}

// One vector of 8 elements of a computed block: returns Delta =
// bf16(x_out - x_in) (packed) and accumulates sum Delta^2,
// sum x_in^2, sum Delta * Delta_prev, sum Delta_prev^2, max |x_out| and
// sum |x_out| (ra = x_in, rb = x_out, rp = Delta_prev, bf16).
__device__ __forceinline__ uint4 block_stats_vec(const uint4& ra, const uint4& rb, const uint4& rp, TwoF2& d2,
                                                 Kahan2& xi2, TwoF2& ddp, TwoF2& dp2, float& mx, Kahan2& sa) {
  uint64_t a[4], b[4], p[4];
  unpack4x2(ra, a);
  unpack4x2(rb, b);
  unpack4x2(rp, p);
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    w[j] = f2_to_bf16x2(f2_sub(b[j], a[j]));      // Delta = bf16(x_out - x_in)
    const uint64_t d = f2_from_bf16x2(w[j]);
    two_add2(d2, f2_mul(d, d));
    two_add2(ddp, f2_mul(d, p[j]));
    two_add2(dp2, f2_mul(p[j], p[j]));
    kahan_add2(xi2, f2_mul(a[j], a[j]));
    mx = f2_max_abs(b[j], mx);
    kahan_add2(sa, f2_abs(b[j]));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace sixbit
