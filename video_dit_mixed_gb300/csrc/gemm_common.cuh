// Device helpers shared by the GEMM kernels: register reallocation, the
// erf GELU of the up projection, cp.async, accumulator hand-back, and
// the bf16 epilogue (GELU or residual, direct or TMA-staged stores).
#pragma once

#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "stats_common.cuh"

namespace sixbit {

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
// GELU(v) = v Phi(v) = 0.5 v (1 + erf(x)), x = v / sqrt 2, for two elements at
// once (packed f32x2 arithmetic).  erf(x) = x Q(s) on |x| <= 3.9, where
// Q(s) ~ erf(x) / x is the degree-15 Chebyshev interpolant of that even
// function in s = 2 x^2 / 3.9^2 - 1, written as monomial coefficients in s
// (all below 1 in magnitude) and evaluated by Horner in s; x is first clamped
// to +-3.9 (erf(3.9) = 1 - 3.5e-8), in one instruction (min.xorsign.abs keeps
// x's sign).  In FP32 with FMAs the erf is within 1.9e-7 of the exact one for
// every x and the GELU within 1.3e-7 |v|.  No reciprocal or exponential: the
// special-function unit, a quarter-rate pipe, paced the epilogue with the
// two an element of Abramowitz & Stegun's formula 7.1.26.  The coefficients
// are printed by gelu_coeffs.py (beside this file).
__host__ __device__ constexpr float gelu_q(int i) {  // coefficient c_i of Q
  constexpr float c[16] = {
      0x1.7349360000000p-2f,  // c_0
      -0x1.72b5ec0000000p-3f,  // c_1
      0x1.13d9060000000p-3f,  // c_2
      -0x1.c0a6ce0000000p-4f,  // c_3
      0x1.735e940000000p-4f,  // c_4
      -0x1.2e36520000000p-4f,  // c_5
      0x1.da8d980000000p-5f,  // c_6
      -0x1.5f5f0c0000000p-5f,  // c_7
      0x1.dc399a0000000p-6f,  // c_8
      -0x1.3b50de0000000p-6f,  // c_9
      0x1.c06c100000000p-7f,  // c_10
      -0x1.eeb2900000000p-8f,  // c_11
      0x1.df33080000000p-10f,  // c_12
      -0x1.2e7bc00000000p-10f,  // c_13
      0x1.fdde5c0000000p-10f,  // c_14
      -0x1.ac851a0000000p-11f,  // c_15
  };
  return c[i];
}
constexpr float kGeluS = 0x1.0d4be80000000p-3f;  // 2 / 3.9^2, rounded
__device__ __forceinline__ float clamp_erf_arg(float x) {  // sign(x) min(|x|, 3.9)
  float d;
  asm("min.xorsign.abs.f32 %0, %1, %2;" : "=f"(d) : "f"(x), "f"(3.9f));
  return d;
}
__device__ __forceinline__ uint64_t gelu_pair(uint64_t v) {
  const uint64_t x = f2_mul(v, f2_pack(0.7071067811865475244f, 0.7071067811865475244f));
  const uint64_t xc = f2_pack(clamp_erf_arg(f2_lo(x)), clamp_erf_arg(f2_hi(x)));
  const uint64_t s = f2_fma(f2_mul(xc, xc), f2_pack(kGeluS, kGeluS), f2_pack(-1.0f, -1.0f));
  uint64_t q = f2_pack(gelu_q(15), gelu_q(15));
#pragma unroll
  for (int i = 14; i >= 0; --i) q = f2_fma(q, s, f2_pack(gelu_q(i), gelu_q(i)));
  const uint64_t h = f2_mul(v, f2_pack(0.5f, 0.5f));
  return f2_fma(h, f2_mul(xc, q), h);  // h (1 + erf)
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
    for (int j = 0; j < 32; j += 2) {
      const uint64_t g = gelu_pair(f2_pack(v[j], v[j + 1]));
      v[j] = f2_lo(g);
      v[j + 1] = f2_hi(g);
    }
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

// ------------------------------------ block statistics from the epilogue --
// With p.bs_delta set, the residual epilogue of a block's down projection also
// does that block's statistics pass (technical summary sections 2.A-2.B,
// popular summary section 3; the separate pass is block_stats_body in
// stats_policy.cu): per 8 output elements x_out = bf16(Y) as stored, x_in =
// the residual, Delta_prev read from bs_delta and Delta = bf16(x_out - x_in)
// written over it, and the six sums accumulated per thread by the same
// block_stats_vec.  When a thread is done, each epilogue warp reduces its
// sums (shuffle tree) into one partial row at a fixed index; the row count
// goes to the first word.  A separate kernel folds the rows in a fixed
// order, so the totals are run-to-run deterministic.
struct BsAcc {
  TwoF2 d2, ddp, dp2;
  Kahan2 xi2, sa;
  float mx;
};
__device__ __forceinline__ BsAcc bs_zero() { return BsAcc{{0, 0}, {0, 0}, {0, 0}, {0, 0}, {0, 0}, 0.f}; }

// Columns [n, n + 32) of row `row` < M; v holds their fp32 outputs (residual
// added); the bf16 rounding of Y is redone here (round to nearest even).
__device__ __forceinline__ void bs_chunk32(const GemmParams& p, int row, int n, const float (&v)[32], BsAcc& a) {
  const size_t base = static_cast<size_t>(row) * p.N + n;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (n + 8 * q + 8 <= p.N) {
      const uint4 ra = *reinterpret_cast<const uint4*>(p.residual + base + 8 * q);
      const uint4 rp = *reinterpret_cast<const uint4*>(p.bs_delta + base + 8 * q);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&b);
      }
      *reinterpret_cast<uint4*>(p.bs_delta + base + 8 * q) =
          block_stats_vec(ra, make_uint4(w[0], w[1], w[2], w[3]), rp, a.d2, a.xi2, a.ddp, a.dp2, a.mx, a.sa);
    }
  }
}

// The RESIDUAL epilogue and bs_chunk32 in one: per half of the chunk, the
// residual and Delta_prev vectors are loaded together (one memory round trip
// for both), the residual added to v (as epilogue_apply32 does), and the
// statistics taken.
__device__ __forceinline__ void residual_bs_chunk32(const GemmParams& p, int row, int n, float (&v)[32], BsAcc& a) {
  const size_t base = static_cast<size_t>(row) * p.N + n;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint4 ra[2], rp[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int q = 2 * h + u;
      if (n + 8 * q + 8 <= p.N) {
        ra[u] = *reinterpret_cast<const uint4*>(p.residual + base + 8 * q);
        rp[u] = *reinterpret_cast<const uint4*>(p.bs_delta + base + 8 * q);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int q = 2 * h + u;
      if (n + 8 * q + 8 <= p.N) {
        const uint32_t x[4] = {ra[u].x, ra[u].y, ra[u].z, ra[u].w};
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[8 * q + 2 * i] = __fadd_rn(v[8 * q + 2 * i], __uint_as_float(x[i] << 16));
          v[8 * q + 2 * i + 1] = __fadd_rn(v[8 * q + 2 * i + 1], __uint_as_float(x[i] & 0xFFFF0000u));
          const __nv_bfloat162 b = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
          w[i] = *reinterpret_cast<const uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(p.bs_delta + base + 8 * q) =
            block_stats_vec(ra[u], make_uint4(w[0], w[1], w[2], w[3]), rp[u], a.d2, a.xi2, a.ddp, a.dp2, a.mx, a.sa);
      }
    }
  }
}

// L2 prefetch of the residual and Delta_prev of columns [n, n + ncols) of
// row `row` (ncols * 2 bytes, one line per 128 bytes and the last one);
// ncols >= 1.
__device__ __forceinline__ void bs_prefetch(const GemmParams& p, int row, int n, int ncols) {
  const size_t base = static_cast<size_t>(row) * p.N + n;
  for (int c = 0; c < ncols; c += 64) {
    prefetch_l2(p.residual + base + c);
    prefetch_l2(p.bs_delta + base + c);
  }
  prefetch_l2(p.residual + base + ncols - 1);
  prefetch_l2(p.bs_delta + base + ncols - 1);
}

// The same for the residual alone (the plain RESIDUAL epilogue).
__device__ __forceinline__ void residual_prefetch(const GemmParams& p, int row, int n, int ncols) {
  const size_t base = static_cast<size_t>(row) * p.N + n;
  for (int c = 0; c < ncols; c += 64) prefetch_l2(p.residual + base + c);
  prefetch_l2(p.residual + base + ncols - 1);
}

// The epilogue's nw warps (warp index ew, all lanes) end the statistics:
// each reduces its threads' sums (shuffle tree), the CTA's rows meet in
// shared memory behind a named barrier over those warps only (id 1), and
// warp 0 folds them in a fixed order into the CTA's partial row (row
// blockIdx.x); CTA 0 also writes the row count.
__device__ __forceinline__ void bs_flush(const GemmParams& p, const BsAcc& a, int ew, int nw, int lane) {
  __shared__ FF bs_red[kBsMaxWarps][kBsSums];
  FF v[kBsSums] = {to_ff(a.d2), to_ff(a.xi2), to_ff(a.ddp), to_ff(a.dp2), FF{a.mx, 0.f}, to_ff(a.sa)};
  const bool is_max[kBsSums] = {false, false, false, false, true, false};
  warp_reduce<kBsSums>(v, is_max);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < kBsSums; ++k) bs_red[ew][k] = v[k];
  }
  asm volatile("bar.sync 1, %0;" ::"r"(nw * 32) : "memory");
  if (ew != 0) return;
#pragma unroll
  for (int k = 0; k < kBsSums; ++k) v[k] = lane < nw ? bs_red[lane][k] : FF{0.f, 0.f};
  warp_reduce<kBsSums, kBsMaxWarps>(v, is_max);
  if (lane == 0) {
    FF* row = reinterpret_cast<FF*>(static_cast<char*>(p.bs_parts) + 16) + static_cast<size_t>(blockIdx.x) * kBsSums;
#pragma unroll
    for (int k = 0; k < kBsSums; ++k) row[k] = v[k];
    if (blockIdx.x == 0) *static_cast<uint32_t*>(p.bs_parts) = gridDim.x;
  }
}

}  // namespace sixbit
