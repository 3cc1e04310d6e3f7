// Online block-Hadamard rotation fused with dynamic NVFP4 / INT8 quantization
// of activations, and the offline rotation + 4-bit packing of weights.
//
// Method: "6Bit-Diffusion" technical summary section 2.A (DMPQ: NVFP4 for
// stable blocks, INT8 for volatile ones; online block Hadamard transform
// against outliers) and section 4 (custom CUDA kernels fuse the
// quantization with the block Hadamard transform).
//
// Work layout: one warp per row.  A row is walked in chunks of 256 elements;
// lane l holds elements [8l, 8l+8) of the chunk, loaded with one 16-byte
// non-coherent load.  A Hadamard block of b elements therefore lives in b/8
// consecutive lanes: strides 1, 2, 4 of the butterfly are done in registers,
// strides 8 .. b/2 with shfl.xor across lanes, in ascending order, each step
// one IEEE FP32 add or subtract, then one exact multiply by 2^-log4(b).  The
// 16-element NVFP4 groups are lane pairs; the 128-element INT4 weight groups
// are 16-lane halves.
#include <cstdint>

#include "common.cuh"
#include "ctx_cache.h"
#include "internal.h"

namespace sixbit {

constexpr int kHqWarps = 8;  // warps per CTA

__device__ __forceinline__ size_t sf_offset(int r, int kb, int K) {
  return static_cast<size_t>(r >> 7) * static_cast<size_t>(128 * (K >> 4)) + static_cast<size_t>(kb >> 2) * 512 +
         static_cast<size_t>((r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3));
}

__device__ __forceinline__ uint4 ld_nc_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& r, float (&v)[8]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Fixed-order FP32 butterfly over a Hadamard block of B elements spread over
// B/8 lanes (8 per lane), followed by the exact 1/sqrt(B) scaling.
template <int B>
__device__ __forceinline__ void fwht8(float (&v)[8], int lane) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], c = v[i + h];
        v[i] = __fadd_rn(a, c);
        v[i + h] = __fsub_rn(a, c);
      }
    }
  }
#pragma unroll
  for (int h = 8; h < B; h <<= 1) {
    const int m = h >> 3;
    // lower lane: v + o; upper lane: o - v.  fma(+-1, v, o) is that one sum
    // with a single rounding, i.e. the same IEEE add or subtract.
    const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
      v[i] = __fmaf_rn(sgn, v[i], o);
    }
  }
  constexpr float s = B == 16 ? 0.25f : (B == 64 ? 0.125f : 0.0625f);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], s);
}

// Correctly rounded y / d from a correctly rounded reciprocal rd = RN(1/d):
// q = RN(y*rd), then one FMA correction q + rd*(y - d*q) (Markstein's
// theorem: with rd within half an ulp of 1/d and q within one ulp of y/d, the
// corrected quotient is RN(y/d) barring overflow and underflow).  Callers use
// it only when d and rd are normal numbers and fall back to the IEEE
// division otherwise.
__device__ __forceinline__ float div_by_recip(float y, float d, float rd) {
  const float q = __fmul_rn(y, rd);
  const float res = __fmaf_rn(-d, q, y);
  return __fmaf_rn(res, rd, q);
}

// True when d is in the range where div_by_recip is exact (also excludes 0).
__device__ __forceinline__ bool recip_ok(float d) {
  const float a = fabsf(d);
  return a >= 0x1p-100f && a <= 0x1p+100f;
}

__device__ __forceinline__ uint32_t f32_to_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(c)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Eight FP32 values -> eight E2M1 codes, element 0 in the low nibble.
__device__ __forceinline__ uint32_t f32x8_to_e2m1(const float (&q)[8]) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return out;
}

__device__ __forceinline__ bool mode_skips(const int32_t* mode_dev, int want) {
  return mode_dev != nullptr && SIXBIT_MODE_OF(*mode_dev) != want;
}

__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

// Loads up to 4 chunks of a bf16 row (chunks c0..c0+3) into registers.
__device__ __forceinline__ void load_chunks_bf16(const uint16_t* row, int K, int c0, int nch, int lane,
                                                 uint4 (&raw)[4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int col = (c0 + u) * 256 + lane * 8;
    raw[u] = make_uint4(0, 0, 0, 0);
    if (c0 + u < nch && col < K) raw[u] = ld_nc_16(row + col);
  }
}

// ------------------------------------------------ pass 1: tensor amax |y| --

template <int B>
__global__ void __launch_bounds__(kHqWarps * 32) hq_amax_kernel(const uint16_t* __restrict__ X, int M, int K,
                                                                const int32_t* mode_dev, float* amax_out) {
  if (mode_skips(mode_dev, SIXBIT_MODE_NVFP4)) return;
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kHqWarps + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kHqWarps;
  const int nch = (K + 255) >> 8;
  float m = 0.f;
  for (int r = warp; r < M; r += nwarps) {
    const uint16_t* row = X + static_cast<size_t>(r) * K;
    for (int c0 = 0; c0 < nch; c0 += 4) {
      uint4 raw[4];
      load_chunks_bf16(row, K, c0, nch, lane, raw);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c0 + u >= nch) break;
        float v[8];
        bf16x8_to_f32(raw[u], v);
        fwht8<B>(v, lane);
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
      }
    }
  }
  m = warp_max(m);
  __shared__ float red[kHqWarps];
  if (lane == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = red[0];
    for (int i = 1; i < kHqWarps; ++i) b = fmaxf(b, red[i]);
    atomicMax(reinterpret_cast<unsigned int*>(amax_out), __float_as_uint(b));  // b >= 0
  }
}

// ----------------------------------------------------- NVFP4 quantization --

// One 256-element chunk of NVFP4 quantization for lane `lane` of row r.
template <int B>
__device__ __forceinline__ void nvfp4_chunk(float (&v)[8], int r, int col, bool row_ok, int K, int lane, float s_t,
                                            uint8_t* codes, uint8_t* scales, float* rotated) {
  const bool active = row_ok && col < K;
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(v[i]));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
  const float sb = __fdiv_rn(__fdiv_rn(am, 6.0f), s_t);
  const uint32_t e = f32_to_e4m3(sb);
  const float S = __fmul_rn(e4m3_to_f32(e), s_t);
  float q[8];
  if (recip_ok(S)) {
    const float rS = __frcp_rn(S);
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = div_by_recip(v[i], S, rS);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = (S != 0.f) ? __fdiv_rn(v[i], S) : 0.f;
  }
  const uint32_t packed = f32x8_to_e2m1(q);
  if (active) {
    *reinterpret_cast<uint32_t*>(codes + static_cast<size_t>(r) * (K >> 1) + (col >> 1)) = packed;
    if (rotated != nullptr) {
      float4* dst = reinterpret_cast<float4*>(rotated + static_cast<size_t>(r) * K + col);
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
  if ((lane & 1) == 0 && col < K) scales[sf_offset(r, col >> 4, K)] = row_ok ? static_cast<uint8_t>(e) : 0;
}

// Rows [0, M) are quantized; rows [M, round_up(M,128)) get zero scales so the
// GEMM never multiplies by an undefined scale.
template <int B>
__global__ void __launch_bounds__(kHqWarps * 32) hq_nvfp4_kernel(const uint16_t* __restrict__ X, int M, int K,
                                                                 const int32_t* mode_dev, const float* amax_src,
                                                                 uint8_t* codes, uint8_t* scales, float* tscale_out,
                                                                 float* rotated) {
  if (mode_skips(mode_dev, SIXBIT_MODE_NVFP4)) return;
  const float amax = *amax_src;
  const float s_t = amax == 0.f ? 1.0f : __fdiv_rn(amax, 2688.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *tscale_out = s_t;
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kHqWarps + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kHqWarps;
  const int nch = (K + 255) >> 8;
  const int mpad = (M + 127) & ~127;
  for (int r = warp; r < mpad; r += nwarps) {
    const bool row_ok = r < M;
    const uint16_t* row = X + static_cast<size_t>(row_ok ? r : 0) * K;
    for (int c0 = 0; c0 < nch; c0 += 4) {
      uint4 raw[4];
      if (row_ok) {
        load_chunks_bf16(row, K, c0, nch, lane, raw);
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) raw[u] = make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c0 + u >= nch) break;
        float v[8];
        bf16x8_to_f32(raw[u], v);
        fwht8<B>(v, lane);
        nvfp4_chunk<B>(v, r, (c0 + u) * 256 + lane * 8, row_ok, K, lane, s_t, codes, scales, rotated);
      }
    }
  }
}

// ------------------------------------------------------ INT8 quantization --

// Quantizes and stores one lane's 8 rotated values of row r at column col:
// q = clamp(RN(y / s), -127, 127); the int8 codes and (optional) the rotated
// values.  Rounding to an integer is
// done by adding 1.5 * 2^23: for |d| <= 127 the sum lies in [2^23, 2^24),
// where the float spacing is 1, so the IEEE add rounds d to the nearest
// integer with ties to even (rint) and the low mantissa bits hold q in two's
// complement.  Clamping before rounding equals clamping after it (rounding
// is monotone and +-127 are integers).  When s == 0 (all |y| rounded away)
// the reciprocal is taken as 0, which gives q = 0.
constexpr float kRound = 12582912.0f;  // 1.5 * 2^23

// Writes one lane's 8 codes from t = the rounding sums (0x4B400000 + q): the
// low byte of each is q in two's complement.
__device__ __forceinline__ void int8_write8(const uint32_t (&t)[8], size_t off, int8_t* codes) {
  const uint32_t lo = __byte_perm(__byte_perm(t[0], t[1], 0x0040), __byte_perm(t[2], t[3], 0x0040), 0x5410);
  const uint32_t hi = __byte_perm(__byte_perm(t[4], t[5], 0x0040), __byte_perm(t[6], t[7], 0x0040), 0x5410);
  *reinterpret_cast<uint2*>(codes + off) = make_uint2(lo, hi);
}

__device__ __forceinline__ void int8_chunk_store(const float (&v)[8], int r, int col, int K, float s, bool fast,
                                                 float rs, int8_t* codes, float* rotated) {
  uint32_t t[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // With s = RN(amax / 127) normal, |RN(y / s)| <= 127 (1 + 2^-24): the clamp
    // cannot bind, and is only applied on the IEEE-division path (s subnormal
    // or huge, where s carries less precision).  (A NaN y gives an unspecified
    // code on the fast path.)
    const float d = fast ? div_by_recip(v[i], s, rs) : fminf(fmaxf(__fdiv_rn(v[i], s), -127.f), 127.f);
    t[i] = __float_as_uint(__fadd_rn(d, kRound));  // 0x4B400000 + q
  }
  const size_t off = static_cast<size_t>(r) * K + col;
  int8_write8(t, off, codes);
  if (rotated != nullptr) {
    float4* dst = reinterpret_cast<float4*>(rotated + off);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

// Two passes per row (row amax, then the row again from cache); serves any K.
template <int B>
__global__ void __launch_bounds__(kHqWarps * 32) hq_int8_kernel(const uint16_t* __restrict__ X, int M, int K,
                                                                const int32_t* mode_dev, int8_t* codes,
                                                                float* row_scale, float* rotated) {
  if (mode_skips(mode_dev, SIXBIT_MODE_INT8)) return;
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kHqWarps + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kHqWarps;
  const int nch = (K + 255) >> 8;
  for (int r = warp; r < M; r += nwarps) {
    const uint16_t* row = X + static_cast<size_t>(r) * K;
    // pass 1: row amax of the rotated values
    float m = 0.f;
    for (int c0 = 0; c0 < nch; c0 += 4) {
      uint4 raw[4];
      load_chunks_bf16(row, K, c0, nch, lane, raw);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c0 + u >= nch) break;
        float v[8];
        bf16x8_to_f32(raw[u], v);
        fwht8<B>(v, lane);
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
      }
    }
    m = warp_max(m);
    const float s = __fdiv_rn(m, 127.0f);
    const bool fast = recip_ok(s) || s == 0.f;
    const float rs = s != 0.f ? __frcp_rn(s) : 0.f;
    if (lane == 0) row_scale[r] = s;
    // pass 2: the row again (from cache), rotate, quantize
    for (int c0 = 0; c0 < nch; c0 += 4) {
      uint4 raw[4];
      load_chunks_bf16(row, K, c0, nch, lane, raw);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c0 + u >= nch) break;
        float v[8];
        bf16x8_to_f32(raw[u], v);
        fwht8<B>(v, lane);
        const int col = (c0 + u) * 256 + lane * 8;
        if (col < K) int8_chunk_store(v, r, col, K, s, fast, rs, codes, rotated);
      }
    }
  }
}

// One pass: a CTA of 16 warps takes 16 / R rows, R = 2^lr warps per row, and
// each warp holds up to four 256-element chunks of its row (chunks t, t + R,
// t + 2R, t + 3R for warp t of the row's team) in registers, so X is read
// once.  The row amax is combined across the team through shared memory.
// Serves rows of up to 16 * 4 * 256 elements, with the results of
// hq_int8_kernel (same butterfly, same per-element division).
//
// Chunks are processed in pairs on packed FP32 pairs: element i of chunk 2p
// in the low lane, element i of chunk 2p + 1 in the high lane.  Both lanes
// take the same butterfly position, so every stage and every step of the
// division is one f32x2 instruction for two elements, each lane rounded
// exactly as the scalar operation.  The exact 1/sqrt(b) scaling is folded
// into the divisor: y / s = v / (s sqrt(b)) with both scalings exact, so
// RN(y / s) is unchanged (when y = v / sqrt(b) is an inexact subnormal,
// |y / s| < 2^-26 on this path and both round to q = 0).
constexpr int kHqRowWarps = 16;
constexpr int kHqRowChunks = 4;

template <int B>
__device__ __forceinline__ void fwht8x2(uint64_t (&v)[8], int lane) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if ((i & h) == 0) {
        const uint64_t a = v[i], c = v[i + h];
        v[i] = f2_add(a, c);
        v[i + h] = f2_sub(a, c);
      }
    }
  }
#pragma unroll
  for (int h = 8; h < B; h <<= 1) {
    const int m = h >> 3;
    const float sgn = (lane & m) ? -1.0f : 1.0f;  // lower lane: v + o; upper lane: o - v (one rounding)
    const uint64_t sg2 = f2_pack(sgn, sgn);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, static_cast<unsigned long long>(v[i]), m);
      v[i] = f2_fma(sg2, v[i], o);
    }
  }
}

template <int B>
__global__ void __launch_bounds__(kHqRowWarps * 32, 2) hq_int8_rows_kernel(const uint16_t* __restrict__ X, int M,
                                                                        int K, int lr, const int32_t* mode_dev,
                                                                        int8_t* codes, float* row_scale,
                                                                        float* rotated) {
  if (mode_skips(mode_dev, SIXBIT_MODE_INT8)) return;
  constexpr float kScale = B == 16 ? 0.25f : (B == 64 ? 0.125f : 0.0625f);  // 1/sqrt(B), exact
  __shared__ float red[kHqRowWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = 1 << lr;
  const int team = warp >> lr, t = warp & (R - 1);
  const int r = blockIdx.x * (kHqRowWarps >> lr) + team;
  const bool row_ok = r < M;
  const int nch = (K + 255) >> 8;
  const uint16_t* row = X + static_cast<size_t>(row_ok ? r : 0) * K;
  uint4 raw[kHqRowChunks];
#pragma unroll
  for (int u = 0; u < kHqRowChunks; ++u) {
    const int c = t + u * R;
    const int col = c * 256 + lane * 8;
    raw[u] = make_uint4(0, 0, 0, 0);
    if (row_ok && c < nch && col < K) raw[u] = ld_nc_16(row + col);
  }
  uint64_t v[kHqRowChunks / 2][8];  // unscaled rotated values of chunk pairs (2p, 2p + 1)
  float m = 0.f;
#pragma unroll
  for (int p = 0; p < kHqRowChunks / 2; ++p) {
    float a[8], b[8];
    bf16x8_to_f32(raw[2 * p], a);
    bf16x8_to_f32(raw[2 * p + 1], b);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[p][i] = f2_pack(a[i], b[i]);
    if (t + 2 * p * R < nch) fwht8x2<B>(v[p], lane);  // warp-uniform; an absent chunk holds zeros
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fmaxf(fabsf(f2_lo(v[p][i])), fabsf(f2_hi(v[p][i]))));
  }
  m = warp_max(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[team << lr];
  for (int i = 1; i < R; ++i) m = fmaxf(m, red[(team << lr) + i]);
  if (!row_ok) return;
  // max |y| = RN(max |v| / sqrt(B)): rounding is monotone, so this is the
  // maximum of the rounded rotated values.
  const float s = __fdiv_rn(__fmul_rn(m, kScale), 127.0f);
  const bool fast = recip_ok(s) || s == 0.f;
  const float rs = s != 0.f ? __frcp_rn(s) : 0.f;
  const uint64_t rs2 = f2_pack(rs * kScale, rs * kScale);  // RN(1 / (s sqrt(B))), exact; s sqrt(B) = s / kScale
  const uint64_t kr2 = f2_pack(kRound, kRound);
  if (t == 0 && lane == 0) row_scale[r] = s;
  const uint64_t ns2 = f2_pack(-(s / kScale), -(s / kScale));
#pragma unroll
  for (int p = 0; p < kHqRowChunks / 2; ++p) {
    // the rounding sums 1.5 * 2^23 + q (low byte: q); the row-uniform branch
    // keeps the IEEE-division fallback out of the fast loop.
    if (rotated != nullptr) {  // the rotated values y = v / sqrt(B) (FP32, test output)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = t + (2 * p + h) * R;
        const int col = c * 256 + lane * 8;
        if (c >= nch || col >= K) continue;
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(h ? f2_hi(v[p][i]) : f2_lo(v[p][i]), kScale);
        float4* dst = reinterpret_cast<float4*>(rotated + static_cast<size_t>(r) * K + col);
        dst[0] = make_float4(y[0], y[1], y[2], y[3]);
        dst[1] = make_float4(y[4], y[5], y[6], y[7]);
      }
    }
    uint64_t oi[8];
    if (fast) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // div_by_recip on both lanes
        const uint64_t q = f2_mul(v[p][i], rs2);
        const uint64_t d = f2_fma(f2_fma(ns2, q, v[p][i]), rs2, q);
        oi[i] = f2_add(d, kr2);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float dl = fminf(fmaxf(__fdiv_rn(__fmul_rn(f2_lo(v[p][i]), kScale), s), -127.f), 127.f);
        const float dh = fminf(fmaxf(__fdiv_rn(__fmul_rn(f2_hi(v[p][i]), kScale), s), -127.f), 127.f);
        oi[i] = f2_add(f2_pack(dl, dh), kr2);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = t + (2 * p + h) * R;
      const int col = c * 256 + lane * 8;
      if (c >= nch || col >= K) continue;
      uint32_t tt[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) tt[i] = static_cast<uint32_t>(h ? (oi[i] >> 32) : oi[i]);
      int8_write8(tt, static_cast<size_t>(r) * K + col, codes);
    }
  }
}

// b = 64 with 32 consecutive elements per lane (half a Hadamard block, the
// other half in the neighbouring lane): a warp covers 1024 consecutive
// elements of its row, a team of R = 2^lr warps the row (K <= 16384).  The
// lane's elements i and i + 16 share an f32x2 register, so the stages of
// stride 1, 2, 4, 8 are one f32x2 instruction for two butterflies, stride 16
// pairs the two lanes of a register, and only stride 32 crosses lanes (one
// 64-bit shuffle per pair: a third of the cross-lane traffic of the
// 8-elements-per-lane form above, whose stages 8, 16, 32 all cross lanes).
// Same stage order, same roundings, same division: bit-identical results.
// Persistent CTAs of W warps (W * 1024 >= K), MINB per SM, each walking
// groups of W / R rows; every thread loads its part of the next group
// before it works on the current one, so an SM keeps the loads of a whole
// group per thread in flight while it computes.  (With one load phase per
// row, HBM idled while the row was computed: long-scoreboard stalls led and
// DRAM was ~49% busy at 17776 x 7680; prefetched, 101.0 -> 94.9 us there and
// 31.4 -> 29.3 us at 17776 x 1920, four CTAs an SM; three, 96.9 us.)  Each
// lane writes its 32 codes as two 16-byte stores, half the store
// instructions of four 8-byte ones: 94.9 -> 90.8 us at 17776 x 7680.
template <int W, int MINB>
__global__ void __launch_bounds__(W * 32, MINB) hq_int8_half_kernel(const uint16_t* __restrict__ X, int M, int K,
                                                                  int lr, const int32_t* mode_dev, int8_t* codes,
                                                                  float* row_scale, float* rotated) {
  if (mode_skips(mode_dev, SIXBIT_MODE_INT8)) return;
  constexpr float kScale = 0.125f;  // 1/sqrt(64), exact
  __shared__ float red[2][W];       // the team's warp maxima, two groups apart
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = 1 << lr;
  const int team = warp >> lr, t = warp & (R - 1);
  const int rows_per_cta = W >> lr;
  const int ngroups = (M + rows_per_cta - 1) / rows_per_cta;
  const int col = t * 1024 + lane * 32;  // K % 64 == 0: a block's two halves are both in range or both out
  auto load = [&](int g, uint4 (&raw)[4]) {
    const int r = g * rows_per_cta + team;
    const bool have = g < ngroups && r < M && col < K;
    const uint16_t* src = X + static_cast<size_t>(have ? r : 0) * K + (have ? col : 0);
#pragma unroll
    for (int c = 0; c < 4; ++c) raw[c] = have ? ld_nc_16(src + 8 * c) : make_uint4(0, 0, 0, 0);
  };
  uint4 raw[4];
  load(blockIdx.x, raw);
  int par = 0;
  for (int g = blockIdx.x; g < ngroups; g += gridDim.x, par ^= 1) {
    uint4 nxt[4];
    load(g + gridDim.x, nxt);  // in flight while this group is computed
    const int r = g * rows_per_cta + team;
    const bool have = r < M && col < K;
    uint64_t P[16];  // P[i] = (element i, element i + 16) of the lane's 32
    {
      float e0[8], e1[8], e2[8], e3[8];
      bf16x8_to_f32(raw[0], e0);
      bf16x8_to_f32(raw[1], e1);
      bf16x8_to_f32(raw[2], e2);
      bf16x8_to_f32(raw[3], e3);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        P[i] = f2_pack(e0[i], e2[i]);
        P[8 + i] = f2_pack(e1[i], e3[i]);
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) raw[c] = nxt[c];
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if ((i & h) == 0) {
          const uint64_t a = P[i], c = P[i + h];
          P[i] = f2_add(a, c);
          P[i + h] = f2_sub(a, c);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {  // stride 16: the two lanes of each register
      const float a = f2_lo(P[i]), c = f2_hi(P[i]);
      P[i] = f2_pack(__fadd_rn(a, c), __fsub_rn(a, c));
    }
    {  // stride 32: the neighbouring lane holds the block's other half
      const float sgn = (lane & 1) ? -1.0f : 1.0f;  // lower half: v + o; upper half: o - v (one rounding)
      const uint64_t sg2 = f2_pack(sgn, sgn);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, static_cast<unsigned long long>(P[i]), 1);
        P[i] = f2_fma(sg2, P[i], o);
      }
    }
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fmaxf(fabsf(f2_lo(P[i])), fabsf(f2_hi(P[i]))));
    m = warp_max(m);
    // one barrier a group: red[par] is rewritten two groups later, after
    // every warp has passed the next group's barrier (and so read it)
    if (lane == 0) red[par][warp] = m;
    __syncthreads();
    m = red[par][team << lr];
    for (int i = 1; i < R; ++i) m = fmaxf(m, red[par][(team << lr) + i]);
    if (!have) continue;
    const float s = __fdiv_rn(__fmul_rn(m, kScale), 127.0f);
    const bool fast = recip_ok(s) || s == 0.f;
    const float rs = s != 0.f ? __frcp_rn(s) : 0.f;
    if (t == 0 && lane == 0) row_scale[r] = s;
    const size_t off = static_cast<size_t>(r) * K + col;
    if (rotated != nullptr) {  // the rotated values y = v / 8 (FP32, test output)
      float4* dst = reinterpret_cast<float4*>(rotated + off);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        dst[i] = make_float4(__fmul_rn(f2_lo(P[4 * i]), kScale), __fmul_rn(f2_lo(P[4 * i + 1]), kScale),
                             __fmul_rn(f2_lo(P[4 * i + 2]), kScale), __fmul_rn(f2_lo(P[4 * i + 3]), kScale));
        dst[4 + i] = make_float4(__fmul_rn(f2_hi(P[4 * i]), kScale), __fmul_rn(f2_hi(P[4 * i + 1]), kScale),
                                 __fmul_rn(f2_hi(P[4 * i + 2]), kScale), __fmul_rn(f2_hi(P[4 * i + 3]), kScale));
      }
    }
    const uint64_t kr2 = f2_pack(kRound, kRound);
    uint64_t oi[16];
    if (fast) {
      const uint64_t rs2 = f2_pack(rs * kScale, rs * kScale);  // RN(1 / (8 s)), exact
      const uint64_t ns2 = f2_pack(-(s / kScale), -(s / kScale));
#pragma unroll
      for (int i = 0; i < 16; ++i) {  // div_by_recip on both lanes
        const uint64_t q = f2_mul(P[i], rs2);
        const uint64_t d = f2_fma(f2_fma(ns2, q, P[i]), rs2, q);
        oi[i] = f2_add(d, kr2);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float dl = fminf(fmaxf(__fdiv_rn(__fmul_rn(f2_lo(P[i]), kScale), s), -127.f), 127.f);
        const float dh = fminf(fmaxf(__fdiv_rn(__fmul_rn(f2_hi(P[i]), kScale), s), -127.f), 127.f);
        oi[i] = f2_add(f2_pack(dl, dh), kr2);
      }
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {  // elements 0..15 from the low lanes, 16..31 from the high lanes
      uint32_t w[4];                  // one 16-byte store each
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t tt[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) tt[i] = static_cast<uint32_t>(hh ? (oi[4 * j + i] >> 32) : oi[4 * j + i]);
        w[j] = __byte_perm(__byte_perm(tt[0], tt[1], 0x0040), __byte_perm(tt[2], tt[3], 0x0040), 0x5410);
      }
      *reinterpret_cast<uint4*>(codes + off + 16 * hh) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// ----------------------------------- thread-per-block NVFP4 forms (b = 16) --
//
// For b <= 64 one thread holds a whole Hadamard block (b contiguous elements
// of a row, b/8 16-byte loads) and runs every butterfly stage in registers
// (b = 64 stages its blocks through shared memory first: see below):
// no shuffles (which otherwise occupy the load/store pipe) and fewer
// instructions per element.  Same stage order (ascending strides, each an
// IEEE add or subtract), same exact 1/sqrt(b) scaling and same per-16-group
// NVFP4 and per-row INT8 arithmetic as the warp-per-row kernels above, so
// the results are bit-identical.  Consecutive threads take consecutive
// blocks of a row, so a warp's loads cover a contiguous 32*2b bytes.  (The
// same layout for INT8, with the row amax combined in shared memory, was
// slower than the row-team kernel: one 480-thread CTA per SM.)

template <int B>
__device__ __forceinline__ void load_block_bf16(const uint16_t* p, float (&v)[B]) {
#pragma unroll
  for (int c = 0; c < B / 8; ++c) {
    float t[8];
    bf16x8_to_f32(ld_nc_16(p + 8 * c), t);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[8 * c + i] = t[i];
  }
}

template <int B>
__device__ __forceinline__ void fwht_block(float (&v)[B]) {
#pragma unroll
  for (int h = 1; h < B; h <<= 1) {
#pragma unroll
    for (int i = 0; i < B; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], c = v[i + h];
        v[i] = __fadd_rn(a, c);
        v[i + h] = __fsub_rn(a, c);
      }
    }
  }
  constexpr float s = B == 16 ? 0.25f : 0.125f;
#pragma unroll
  for (int i = 0; i < B; ++i) v[i] = __fmul_rn(v[i], s);
}

template <int B>
__global__ void __launch_bounds__(256) hq_amax_tpb_kernel(const uint16_t* __restrict__ X, int M, int K,
                                                          const int32_t* mode_dev, float* amax_out) {
  if (mode_skips(mode_dev, SIXBIT_MODE_NVFP4)) return;
  const int per_row = K / B;
  const int64_t nblk = static_cast<int64_t>(M) * per_row;
  float m = 0.f;
  for (int64_t t = blockIdx.x * 256ll + threadIdx.x; t < nblk; t += static_cast<int64_t>(gridDim.x) * 256) {
    float v[B];
    load_block_bf16<B>(X + t * B, v);
    fwht_block<B>(v);
#pragma unroll
    for (int i = 0; i < B; ++i) m = fmaxf(m, fabsf(v[i]));
  }
  m = warp_max(m);
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = red[0];
    for (int i = 1; i < 8; ++i) b = fmaxf(b, red[i]);
    atomicMax(reinterpret_cast<unsigned int*>(amax_out), __float_as_uint(b));  // b >= 0
  }
}

// Rows [M, round_up(M,128)) get zero scales (no codes), as in hq_nvfp4_kernel.
template <int B>
__global__ void __launch_bounds__(256) hq_nvfp4_tpb_kernel(const uint16_t* __restrict__ X, int M, int K,
                                                           const int32_t* mode_dev, const float* amax_src,
                                                           uint8_t* codes, uint8_t* scales, float* tscale_out,
                                                           float* rotated) {
  if (mode_skips(mode_dev, SIXBIT_MODE_NVFP4)) return;
  const float amax = *amax_src;
  const float s_t = amax == 0.f ? 1.0f : __fdiv_rn(amax, 2688.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *tscale_out = s_t;
  const int per_row = K / B;
  const int mpad = (M + 127) & ~127;
  const int64_t nblk = static_cast<int64_t>(mpad) * per_row;
  for (int64_t t = blockIdx.x * 256ll + threadIdx.x; t < nblk; t += static_cast<int64_t>(gridDim.x) * 256) {
    const int r = static_cast<int>(t / per_row);
    const int col = static_cast<int>(t - static_cast<int64_t>(r) * per_row) * B;
    if (r >= M) {  // pad row: zero scales
#pragma unroll
      for (int g = 0; g < B / 16; ++g) scales[sf_offset(r, (col >> 4) + g, K)] = 0;
      continue;
    }
    float v[B];
    load_block_bf16<B>(X + static_cast<size_t>(r) * K + col, v);
    fwht_block<B>(v);
    uint32_t packed[B / 8];
    uint32_t sc = 0;
#pragma unroll
    for (int g = 0; g < B / 16; ++g) {
      float am = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(v[16 * g + i]));
      const float sb = __fdiv_rn(__fdiv_rn(am, 6.0f), s_t);
      const uint32_t e = f32_to_e4m3(sb);
      const float S = __fmul_rn(e4m3_to_f32(e), s_t);
      float q[16];
      if (recip_ok(S)) {
        const float rS = __frcp_rn(S);
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i] = div_by_recip(v[16 * g + i], S, rS);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i] = (S != 0.f) ? __fdiv_rn(v[16 * g + i], S) : 0.f;
      }
      float q0[8], q1[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        q0[i] = q[i];
        q1[i] = q[8 + i];
      }
      packed[2 * g] = f32x8_to_e2m1(q0);
      packed[2 * g + 1] = f32x8_to_e2m1(q1);
      sc |= e << (8 * g);
    }
    uint8_t* cp = codes + static_cast<size_t>(r) * (K >> 1) + (col >> 1);
    if constexpr (B == 64) {
      reinterpret_cast<uint4*>(cp)[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      reinterpret_cast<uint4*>(cp)[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
      *reinterpret_cast<uint32_t*>(scales + sf_offset(r, col >> 4, K)) = sc;  // 4 consecutive groups
    } else {
      *reinterpret_cast<uint2*>(cp) = make_uint2(packed[0], packed[1]);
      scales[sf_offset(r, col >> 4, K)] = static_cast<uint8_t>(sc);
    }
    if (rotated != nullptr) {
      float4* dst = reinterpret_cast<float4*>(rotated + static_cast<size_t>(r) * K + col);
#pragma unroll
      for (int i = 0; i < B / 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
}

// ------------------------------------------- shared-memory-staged b = 64 forms --
//
// The thread-per-block kernels above load each thread's 128-byte block
// directly, so one 16-byte warp load touches 32 lines (32 L1 wavefronts) and
// the load/store pipe, not HBM, bounds them.  Here each warp stages its next
// 32 consecutive blocks (4 KB, contiguous: K % 64 == 0) with coalesced
// 16-byte cp.async copies, three tiles ahead, into its own shared-memory
// ring; chunk q of block r lands at chunk q ^ (r & 7) of the block's 128-byte
// row, so both the copies and each thread's eight 16-byte reads of its own
// block are conflict-free.  The arithmetic is that of the thread-per-block
// kernels (same stage order, same per-group divisions), so the results are
// bit-identical.  Warps need no synchronization beyond their own lanes.
constexpr int kStgWarps = 8;
constexpr int kStgDepth = 3;
constexpr int kStgTileBytes = 32 * 128;
constexpr int kStgSmem = kStgWarps * kStgDepth * kStgTileBytes;  // 96 KB

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Copies tile `tile` (blocks 32 tile .. 32 tile + 31 of X, zero past nblk)
// into the warp's slot at `slot` (shared address), one commit group.
__device__ __forceinline__ void stage_tile(const uint16_t* X, int64_t nblk, int64_t tile, uint32_t slot, int lane) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int off = c * 512 + lane * 16;  // byte offset within the tile
    const int r = off >> 7, q = (off >> 4) & 7;
    const int64_t blk = tile * 32 + r;
    const bool v = blk < nblk;
    cp_async16_zfill(slot + r * 128 + ((q ^ (r & 7)) << 4),
                     v ? reinterpret_cast<const uint8_t*>(X) + tile * kStgTileBytes + off : reinterpret_cast<const uint8_t*>(X), v);
  }
  cp_async_commit();
}

// This lane's block (row `lane` of the slot) as 64 floats.
__device__ __forceinline__ void read_staged_block(const uint8_t* slot, int lane, float (&v)[64]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 raw = *reinterpret_cast<const uint4*>(slot + lane * 128 + ((c ^ (lane & 7)) << 4));
    float t[8];
    bf16x8_to_f32(raw, t);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[8 * c + i] = t[i];
  }
}

// AMAX: max |rotated X| into amax_out (atomicMax of a non-negative float's
// bits).  Otherwise: the NVFP4 codes and scales with s_t from *amax_src, as
// the thread-per-block kernel computes them, including zero scales for the
// pad rows.
template <bool AMAX>
__global__ void __launch_bounds__(kStgWarps * 32, 2) hq_nvfp4_staged_kernel(
    const uint16_t* __restrict__ X, int M, int K, const int32_t* mode_dev, const float* amax_src, float* amax_out,
    uint8_t* codes, uint8_t* scales, float* tscale_out, float* rotated) {
  if (mode_skips(mode_dev, SIXBIT_MODE_NVFP4)) return;
  extern __shared__ __align__(1024) uint8_t stg_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per_row = K / 64;
  const int64_t nblk = static_cast<int64_t>(M) * per_row;
  const int64_t ntiles = (nblk + 31) / 32;
  const int64_t G = static_cast<int64_t>(gridDim.x) * kStgWarps;  // warps in the grid
  const int64_t w0 = static_cast<int64_t>(blockIdx.x) * kStgWarps + warp;
  uint8_t* ring = stg_smem + warp * (kStgDepth * kStgTileBytes);
  const uint32_t ring_s = smem_u32(ring);
  float s_t = 1.0f;
  if constexpr (!AMAX) {
    const float amax = *amax_src;
    s_t = amax == 0.f ? 1.0f : __fdiv_rn(amax, 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *tscale_out = s_t;
  }
  float m = 0.f;
#pragma unroll
  for (int d = 0; d < kStgDepth; ++d) stage_tile(X, nblk, w0 + d * G, ring_s + d * kStgTileBytes, lane);
  int it = 0;
  for (int64_t tile = w0; tile < ntiles; tile += G, ++it) {
    const int slot = it % kStgDepth;
    cp_async_wait<kStgDepth - 1>();  // this lane's copies of this tile have landed
    __syncwarp();                    // and every other lane's
    float v[64];
    read_staged_block(ring + slot * kStgTileBytes, lane, v);
    __syncwarp();                    // the slot is free again
    stage_tile(X, nblk, tile + kStgDepth * G, ring_s + slot * kStgTileBytes, lane);
    const int64_t t = tile * 32 + lane;
    if (t >= nblk) continue;
    // P[i] = (v[i], v[32 + i]): the block's two halves side by side.  Stages
    // of stride 1 .. 16 pair equal positions of both halves, so each is one
    // f32x2 add or subtract per two butterflies; the stride-32 stage pairs
    // the two lanes of a register.  Every lane rounds as the scalar
    // fwht_block<64> does, in the same order.
    uint64_t P[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) P[i] = f2_pack(v[i], v[32 + i]);
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if ((i & h) == 0) {
          const uint64_t a = P[i], c = P[i + h];
          P[i] = f2_add(a, c);
          P[i + h] = f2_sub(a, c);
        }
      }
    }
    const uint64_t eighth = f2_pack(0.125f, 0.125f);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float a = f2_lo(P[i]), c = f2_hi(P[i]);
      P[i] = f2_mul(f2_pack(__fadd_rn(a, c), __fsub_rn(a, c)), eighth);
    }
    if constexpr (AMAX) {
#pragma unroll
      for (int i = 0; i < 32; ++i) m = fmaxf(m, fmaxf(fabsf(f2_lo(P[i])), fabsf(f2_hi(P[i]))));
    } else {
      const int r = static_cast<int>(t / per_row);
      const int col = static_cast<int>(t - static_cast<int64_t>(r) * per_row) * 64;
      // 16-element groups: g = 0, 1 in the low lanes of P[0..15], P[16..31];
      // g = 2, 3 in the high lanes of the same registers.
      float S[4];
      uint32_t sc = 0;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float am = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t y = P[16 * (g & 1) + i];
          am = fmaxf(am, fabsf(g < 2 ? f2_lo(y) : f2_hi(y)));
        }
        const float sb = __fdiv_rn(__fdiv_rn(am, 6.0f), s_t);
        const uint32_t e = f32_to_e4m3(sb);
        S[g] = __fmul_rn(e4m3_to_f32(e), s_t);
        sc |= e << (8 * g);
      }
      uint32_t packed[8];
#pragma unroll
      for (int hg = 0; hg < 2; ++hg) {  // registers P[16 hg ..]: groups hg (low lanes) and hg + 2 (high lanes)
        const float Sl = S[hg], Sh = S[hg + 2];
        uint64_t q[16];
        if (recip_ok(Sl) && recip_ok(Sh)) {  // div_by_recip on both lanes
          const uint64_t R2 = f2_pack(__frcp_rn(Sl), __frcp_rn(Sh));
          const uint64_t N2 = f2_pack(-Sl, -Sh);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t y = P[16 * hg + i];
            const uint64_t q0 = f2_mul(y, R2);
            q[i] = f2_fma(f2_fma(N2, q0, y), R2, q0);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t y = P[16 * hg + i];
            float ql, qh;
            if (recip_ok(Sl)) ql = div_by_recip(f2_lo(y), Sl, __frcp_rn(Sl));
            else ql = (Sl != 0.f) ? __fdiv_rn(f2_lo(y), Sl) : 0.f;
            if (recip_ok(Sh)) qh = div_by_recip(f2_hi(y), Sh, __frcp_rn(Sh));
            else qh = (Sh != 0.f) ? __fdiv_rn(f2_hi(y), Sh) : 0.f;
            q[i] = f2_pack(ql, qh);
          }
        }
        float a0[8], a1[8], b0[8], b1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          a0[i] = f2_lo(q[i]);
          a1[i] = f2_lo(q[8 + i]);
          b0[i] = f2_hi(q[i]);
          b1[i] = f2_hi(q[8 + i]);
        }
        packed[2 * hg] = f32x8_to_e2m1(a0);
        packed[2 * hg + 1] = f32x8_to_e2m1(a1);
        packed[2 * (hg + 2)] = f32x8_to_e2m1(b0);
        packed[2 * (hg + 2) + 1] = f32x8_to_e2m1(b1);
      }
      uint8_t* cp = codes + static_cast<size_t>(r) * (K >> 1) + (col >> 1);
      reinterpret_cast<uint4*>(cp)[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      reinterpret_cast<uint4*>(cp)[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
      *reinterpret_cast<uint32_t*>(scales + sf_offset(r, col >> 4, K)) = sc;  // 4 consecutive groups
      if (rotated != nullptr) {
        float4* dst = reinterpret_cast<float4*>(rotated + static_cast<size_t>(r) * K + col);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          dst[i] = make_float4(f2_lo(P[4 * i]), f2_lo(P[4 * i + 1]), f2_lo(P[4 * i + 2]), f2_lo(P[4 * i + 3]));
          dst[8 + i] = make_float4(f2_hi(P[4 * i]), f2_hi(P[4 * i + 1]), f2_hi(P[4 * i + 2]), f2_hi(P[4 * i + 3]));
        }
      }
    }
  }
  cp_async_wait<0>();  // no copy outlives the kernel
  if constexpr (AMAX) {
    m = warp_max(m);
    __shared__ float red[kStgWarps];
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float b = red[0];
      for (int i = 1; i < kStgWarps; ++i) b = fmaxf(b, red[i]);
      atomicMax(reinterpret_cast<unsigned int*>(amax_out), __float_as_uint(b));  // b >= 0
    }
  } else {
    // rows [M, round_up(M, 128)): zero scales (one 32-bit word per 64 columns)
    const int mpad = (M + 127) & ~127;
    const int64_t npad = static_cast<int64_t>(mpad - M) * per_row;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < npad;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const int r = M + static_cast<int>(i / per_row);
      const int col = static_cast<int>(i % per_row) * 64;
      *reinterpret_cast<uint32_t*>(scales + sf_offset(r, col >> 4, K)) = 0u;
    }
  }
}

template <bool AMAX>
static cudaError_t launch_staged(const uint16_t* X, int M, int K, const int32_t* mode_dev, const float* amax_src,
                                 float* amax_out, const sixbit_qact* o, cudaStream_t st) {
  const cudaError_t ae = set_smem_once<hq_nvfp4_staged_kernel<AMAX>>(kStgSmem);
  if (ae != cudaSuccess) return ae;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t ntiles = (static_cast<int64_t>(M) * (K / 64) + 31) / 32;
  const int64_t want = (ntiles + kStgWarps - 1) / kStgWarps;
  const int grid = static_cast<int>(want < 2 * sms ? (want < 1 ? 1 : want) : 2 * sms);
  hq_nvfp4_staged_kernel<AMAX><<<grid, kStgWarps * 32, kStgSmem, st>>>(
      X, M, K, mode_dev, amax_src, amax_out, AMAX ? nullptr : o->fp4_codes, AMAX ? nullptr : o->fp4_scales,
      AMAX ? nullptr : o->tensor_scale, AMAX ? nullptr : o->rotated);
  note_launch();
  return cudaGetLastError();
}

// --------------------------------------------------------- weight packing --

__device__ __forceinline__ void load8_f32(const float* p, float (&v)[8]) {
  const uint4 a = ld_nc_16(p), b = ld_nc_16(p + 4);
  v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
  v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y); v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}

template <int B>
__global__ void __launch_bounds__(kHqWarps * 32) pack_amax_kernel(const float* __restrict__ W, int N, int K,
                                                                  float* amax_out) {
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kHqWarps + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kHqWarps;
  const int nch = (K + 255) >> 8;
  float m = 0.f;
  for (int r = warp; r < N; r += nwarps) {
    for (int c = 0; c < nch; ++c) {
      const int col = c * 256 + lane * 8;
      float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (col < K) load8_f32(W + static_cast<size_t>(r) * K + col, v);
      fwht8<B>(v, lane);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    }
  }
  m = warp_max(m);
  if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(amax_out), __float_as_uint(m));
}

template <int B>
__global__ void __launch_bounds__(kHqWarps * 32) pack_quant_kernel(const float* __restrict__ W, int N, int K,
                                                                   const float* amax_src, sixbit_weights out) {
  const float amax = *amax_src;
  const float s_t = amax == 0.f ? 1.0f : __fdiv_rn(amax, 2688.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *out.fp4_tensor_scale = s_t;
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kHqWarps + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kHqWarps;
  const int nch = (K + 255) >> 8;
  const int npad = (N + 127) & ~127;
  for (int r = warp; r < npad; r += nwarps) {
    const bool row_ok = r < N;
    for (int c = 0; c < nch; ++c) {
      const int col = c * 256 + lane * 8;
      const bool active = row_ok && col < K;
      float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (active) {
        load8_f32(W + static_cast<size_t>(r) * K + col, v);
        uint32_t bw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
          bw[i] = *reinterpret_cast<const uint32_t*>(&p);
        }
        *reinterpret_cast<uint4*>(out.bf16_w + static_cast<size_t>(r) * K + col) = make_uint4(bw[0], bw[1], bw[2], bw[3]);
      }
      fwht8<B>(v, lane);
      nvfp4_chunk<B>(v, r, col, row_ok, K, lane, s_t, out.fp4_codes, out.fp4_scales, nullptr);
      // INT4, groups of 128 = 16 lanes
      float am = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(v[i]));
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      const float s = __fdiv_rn(am, 7.0f);
      if (active) {
        uint32_t nib = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float q = 0.f;
          if (s != 0.f) q = fminf(fmaxf(rintf(__fdiv_rn(v[i], s)), -7.f), 7.f);
          nib |= (static_cast<uint32_t>(static_cast<int>(q)) & 0xFu) << (4 * i);
        }
        *reinterpret_cast<uint32_t*>(out.i4_codes + static_cast<size_t>(r) * (K >> 1) + (col >> 1)) = nib;
        if ((lane & 15) == 0) out.i4_scales[static_cast<size_t>(col >> 7) * N + r] = s;
      }
    }
  }
}

// ----------------------------------------------------------- host launch --

static int hq_grid(int rows) {
  const int sms = sm_count();
  const int want = (rows + kHqWarps - 1) / kHqWarps;
  const int cap = sms * 8;
  return want < cap ? (want > 0 ? want : 1) : cap;
}

#define SIXBIT_DISPATCH_B(b, KERNEL, ...)                                              \
  do {                                                                                 \
    if ((b) == 16) KERNEL<16><<<grid, kHqWarps * 32, 0, st>>>(__VA_ARGS__);            \
    else if ((b) == 64) KERNEL<64><<<grid, kHqWarps * 32, 0, st>>>(__VA_ARGS__);       \
    else KERNEL<256><<<grid, kHqWarps * 32, 0, st>>>(__VA_ARGS__);                     \
    note_launch();                                                                     \
  } while (0)

// Grid of the thread-per-block kernels: one thread per Hadamard block, at
// most 16 CTAs of 256 per SM (the rest is walked with a grid stride).
static int tpb_grid(int64_t nblk) {
  const int sms = sm_count();
  const int64_t want = (nblk + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 16;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

cudaError_t launch_hq_amax(const uint16_t* X, int M, int K, int b, const int32_t* mode_dev, float* amax_out,
                           cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  if (b == 64) return launch_staged<true>(X, M, K, mode_dev, nullptr, amax_out, nullptr, st);
  if (b == 16) {
    const int grid = tpb_grid(static_cast<int64_t>(M) * (K / b));
    hq_amax_tpb_kernel<16><<<grid, 256, 0, st>>>(X, M, K, mode_dev, amax_out);
    note_launch();
    return cudaGetLastError();
  }
  const int grid = hq_grid(M);
  SIXBIT_DISPATCH_B(b, hq_amax_kernel, X, M, K, mode_dev, amax_out);
  return cudaGetLastError();
}

cudaError_t launch_hq_nvfp4(const uint16_t* X, int M, int K, int b, const int32_t* mode_dev, const float* amax_src,
                            const sixbit_qact* o, cudaStream_t st) {
  // b = 64 stores its four group scales as one 32-bit word
  if (b == 64 && (reinterpret_cast<uintptr_t>(o->fp4_scales) & 3u) == 0)
    return launch_staged<false>(X, M, K, mode_dev, amax_src, nullptr, o, st);
  if (b == 16) {
    const int grid = tpb_grid(static_cast<int64_t>((M + 127) & ~127) * (K / b));
    hq_nvfp4_tpb_kernel<16><<<grid, 256, 0, st>>>(X, M, K, mode_dev, amax_src, o->fp4_codes, o->fp4_scales,
                                                  o->tensor_scale, o->rotated);
    note_launch();
    return cudaGetLastError();
  }
  const int grid = hq_grid((M + 127) & ~127);
  SIXBIT_DISPATCH_B(b, hq_nvfp4_kernel, X, M, K, mode_dev, amax_src, o->fp4_codes, o->fp4_scales, o->tensor_scale,
                    o->rotated);
  return cudaGetLastError();
}

cudaError_t launch_hq_int8(const uint16_t* X, int M, int K, int b, const int32_t* mode_dev, const sixbit_qact* o,
                           cudaStream_t st) {
  if (b == 64 && K <= kHqRowWarps * 1024) {  // half a block per lane: one warp per 1024 elements of a row
    int lr = 0;
    while ((1024 << lr) < K) ++lr;
    const int sms = sm_count();
    if (lr <= 3) {  // rows up to 8192 elements: 8-warp CTAs, four per SM (62 registers a thread)
      const int groups = (M + (8 >> lr) - 1) / (8 >> lr);
      const int grid = groups < 4 * sms ? groups : 4 * sms;
      hq_int8_half_kernel<8, 4><<<grid, 8 * 32, 0, st>>>(X, M, K, lr, mode_dev, o->i8_codes, o->row_scale,
                                                         o->rotated);
    } else {
      const int groups = (M + (kHqRowWarps >> lr) - 1) / (kHqRowWarps >> lr);
      const int grid = groups < sms ? groups : sms;
      hq_int8_half_kernel<kHqRowWarps, 1><<<grid, kHqRowWarps * 32, 0, st>>>(X, M, K, lr, mode_dev, o->i8_codes,
                                                                           o->row_scale, o->rotated);
    }
    note_launch();
    return cudaGetLastError();
  }
  const int nch = (K + 255) / 256;
  int lr = 0;
  while ((kHqRowChunks << lr) < nch && lr < 5) ++lr;
  if ((kHqRowChunks << lr) >= nch && (1 << lr) <= kHqRowWarps) {
    const int rows_per_cta = kHqRowWarps >> lr;
    const int grid = (M + rows_per_cta - 1) / rows_per_cta;
    if (b == 16)
      hq_int8_rows_kernel<16><<<grid, kHqRowWarps * 32, 0, st>>>(X, M, K, lr, mode_dev, o->i8_codes, o->row_scale,
                                                                 o->rotated);
    else if (b == 64)
      hq_int8_rows_kernel<64><<<grid, kHqRowWarps * 32, 0, st>>>(X, M, K, lr, mode_dev, o->i8_codes, o->row_scale,
                                                                 o->rotated);
    else
      hq_int8_rows_kernel<256><<<grid, kHqRowWarps * 32, 0, st>>>(X, M, K, lr, mode_dev, o->i8_codes, o->row_scale,
                                                                  o->rotated);
    note_launch();
    return cudaGetLastError();
  }
  const int grid = hq_grid(M);
  SIXBIT_DISPATCH_B(b, hq_int8_kernel, X, M, K, mode_dev, o->i8_codes, o->row_scale, o->rotated);
  return cudaGetLastError();
}

cudaError_t launch_pack_weights(const float* W, int N, int K, int b, const sixbit_weights* o, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(o->fp4_amax, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  int grid = hq_grid(N);
  SIXBIT_DISPATCH_B(b, pack_amax_kernel, W, N, K, o->fp4_amax);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  grid = hq_grid((N + 127) & ~127);
  SIXBIT_DISPATCH_B(b, pack_quant_kernel, W, N, K, o->fp4_amax, *o);
  return cudaGetLastError();
}

}  // namespace sixbit
