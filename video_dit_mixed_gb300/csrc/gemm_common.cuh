// Device helpers shared by the GEMM kernels: register reallocation, the
// exact-erf GELU of the up projection, cp.async, accumulator hand-back, and
// the bf16 epilogue (GELU or residual, direct or TMA-staged stores).
#pragma once

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace sixbit {

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
// GELU(v) = v Phi(v) with Phi(v) = (1 + erf(v / sqrt 2)) / 2.  erfc(z), z = |v| / sqrt 2,
// is taken as t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2), t = 1 / (1 + p z)
// (Abramowitz & Stegun, Handbook of Mathematical Functions, formula 7.1.26: the
// erf it gives is within 1.5e-7 of the exact one), then 1 + erf = 2 - erfc for
// v >= 0 and erfc(|z|) for v < 0, so the negative tail keeps its relative
// accuracy.  Branch-free; its GELU differs from the exact-erf one by at most
// a few 1e-7 |v|, inside the FP32 epilogue's error budget.
__device__ __forceinline__ float gelu_erf(float v) {
  const float z = fabsf(v) * 0.7071067811865475244f;
  const float t = __fdividef(1.0f, fmaf(0.3275911f, z, 1.0f));
  float q = fmaf(t, 1.061405429f, -1.453152027f);
  q = fmaf(t, q, 1.421413741f);
  q = fmaf(t, q, -0.284496736f);
  q = fmaf(t, q, 0.254829592f);
  const float c = t * q * __expf(-z * z);  // erfc(z)
  const float w = v >= 0.f ? 2.0f - c : c;  // 1 + erf(v / sqrt 2)
  return 0.5f * v * w;
}

// 16-byte global -> shared copy without a register round trip (zero-fill when
// !valid; src must still be a valid address).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// Waits until at most N of this thread's most recent cp.async groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_newest() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Hands an accumulator buffer back to the MMA warp: one arrival per warp,
// after every lane's tensor-memory loads have completed.
__device__ __forceinline__ void release_acc(uint64_t* bar, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// Applies the epilogue (GELU, or the residual add) to 32 consecutive columns
// [n, n+32) of row `row` < M.
__device__ __forceinline__ void epilogue_apply32(const GemmParams& p, int row, int n, float (&v)[32]) {
  const size_t base = static_cast<size_t>(row) * p.N + n;
  if (p.epilogue == SIXBIT_EPI_GELU) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = gelu_erf(v[j]);
  } else if (p.epilogue == SIXBIT_EPI_RESIDUAL) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (n + 8 * q + 8 <= p.N) {
        const uint4 r = *reinterpret_cast<const uint4*>(p.residual + base + 8 * q);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[8 * q + 2 * i] = __fadd_rn(v[8 * q + 2 * i], __uint_as_float(w[i] << 16));
          v[8 * q + 2 * i + 1] = __fadd_rn(v[8 * q + 2 * i + 1], __uint_as_float(w[i] & 0xFFFF0000u));
        }
      }
    }
  }
}

// Applies the epilogue to 32 consecutive columns [n, n+32) of one row and
// stores them (bf16 or fp32) directly.
__device__ __forceinline__ void epilogue_store32(const GemmParams& p, int row, int n, float (&v)[32]) {
  if (row >= p.M) return;
  const size_t base = static_cast<size_t>(row) * p.N + n;
  epilogue_apply32(p, row, n, v);
  if (p.Yf != nullptr) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (n + 4 * q + 4 <= p.N)
        *reinterpret_cast<float4*>(p.Yf + base + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&b);
        v[8 * q + 2 * i] = __uint_as_float(w[i] << 16);            // the stored value (read by rot_amax)
        v[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
      if (n + 8 * q + 8 <= p.N) *reinterpret_cast<uint4*>(p.Y + base + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Writes row r's 32 values as bf16 (round to nearest even) into a 32-row box
// of 64-byte rows, 16-byte chunk q of row r at chunk q ^ ((r >> 1) & 3): the
// TMA 64-byte swizzle (box 512-byte aligned), which also spreads a warp's
// 16-byte writes over all banks.
__device__ __forceinline__ void stage_bf16x32(uint8_t* box, int r, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(box + r * 64 + ((q ^ ((r >> 1) & 3)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace sixbit
