// Quantized GEMMs on the fifth-generation tensor cores (tcgen05) of sm_103a.
//
// Method: "6Bit-Diffusion" technical summary sections 2.A and 4 (NVFP4 or
// INT8 activations against 4-bit weights: W4A4 / W4A8) and 2.C (PDR's
// FP16/BF16 recompute); popular summary section 4 (custom CUDA kernels).
//
// One CTA computes one 128 x 128 output tile with three warp roles:
//   warp 0      TMA producer: A/B tiles (128-byte swizzle) and, for NVFP4,
//               the 2 KB scale-factor chunks, into a ring of shared-memory
//               stages guarded by full/empty mbarriers;
//   warp 1      allocates tensor memory; one lane issues tcgen05.mma (and,
//               for NVFP4, tcgen05.cp of the scale factors into tensor
//               memory) and tcgen05.commit to release stages;
//   warps 2..5  epilogue: tcgen05.ld of the FP32 accumulators (warp w reads
//               lanes 32*(w%4)..+31 = tile rows), scaling, GELU or residual,
//               bf16 (or fp32) stores.
// Kinds:
//   NVFP4  kind::mxf4nvf4.block_scale.scale_vec::4X, E2M1 x E2M1 with one
//          E4M3 scale per 16 elements, 256 K-elements (128 bytes) per stage.
//   BF16   kind::f16 with bf16 operands, 64 K-elements per stage.  Used for
//          the PDR path and, with "grouped" accumulation, for W4A8: INT8
//          activation codes and INT4 weight codes are small integers, exact
//          in bf16, every product and every 128-term group sum (|.| < 2^17)
//          is an integer exactly representable in FP32, so each group's FP32
//          accumulator holds the exact integer sum.  Groups alternate
//          between two accumulator buffers in tensor memory; the epilogue
//          folds s_w[g][n] * acc_g into registers while the next group runs.
// Every mbarrier wait is bounded (2 s); on expiry the kernel records
// SIXBIT_ETIMEOUT in the error word, drains its in-flight copies and tensor
// core work with bounded waits, frees tensor memory and returns.
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace sixbit {

constexpr int kBM = 128;
constexpr int kBN = 128;

enum { KIND_BF16 = 0, KIND_NVF4 = 1 };

template <int KIND>
struct GemmCfg;
template <>
struct GemmCfg<KIND_BF16> {
  static constexpr int kStages = 6;
  static constexpr int kKStage = 64;      // K elements per stage
  static constexpr int kKCoord = 64;      // TMA x coordinate step per stage
  static constexpr int kMmaPerStage = 4;  // K = 16 per MMA
  static constexpr int kSfBytes = 0;
  static constexpr uint32_t kIdesc = idesc_bf16(kBM, kBN);
};
template <>
struct GemmCfg<KIND_NVF4> {
  static constexpr int kStages = 5;
  static constexpr int kKStage = 256;
  static constexpr int kKCoord = 128;     // bytes of packed E2M1
  static constexpr int kMmaPerStage = 4;  // K = 64 per MMA
  static constexpr int kSfBytes = 2048;   // 128 rows x 16 scales
  static constexpr uint32_t kIdesc = idesc_nvf4(kBM, kBN);
};

constexpr int kTileBytes = kBM * 128;  // one 128 x 128-byte operand tile

template <int KIND>
__host__ __device__ constexpr int stage_bytes() {
  return 2 * kTileBytes + 2 * GemmCfg<KIND>::kSfBytes;
}
template <int KIND>
__host__ __device__ constexpr int gemm_smem_bytes() {
  return GemmCfg<KIND>::kStages * stage_bytes<KIND>() + 1024 /*align*/ + 256 /*barriers*/;
}



__device__ __forceinline__ float gelu_erf(float v) {
  return 0.5f * v * (1.0f + erff(v * 0.7071067811865475244f));
}

// Applies the epilogue to 32 consecutive columns [n, n+32) of one row and
// stores them (bf16 or fp32).
__device__ __forceinline__ void epilogue_store32(const GemmParams& p, int row, int n, float (&v)[32]) {
  if (row >= p.M) return;
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
  if (p.Yf != nullptr) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (n + 4 * q + 4 <= p.N)
        *reinterpret_cast<float4*>(p.Yf + base + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (n + 8 * q + 8 <= p.N) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162 b = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
          w[i] = *reinterpret_cast<const uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(p.Y + base + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

// Stages of the shared-memory ring; the grouped (W4A8) kernel gives one stage
// up for its staged group scales (up to K = 16768).
template <int KIND, bool GROUPED>
__host__ __device__ constexpr int gemm_stages() {
  return GROUPED ? 5 : GemmCfg<KIND>::kStages;
}

template <bool GROUPED>
struct EpiCfg {
  static constexpr int kWarps = GROUPED ? 8 : 4;    // epilogue warps
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kCols = kBN / (kWarps / 4);  // accumulator columns per epilogue thread
};

template <bool GROUPED>
constexpr int gemm_threads() {
  return 64 + EpiCfg<GROUPED>::kThreads;
}

// Persistent kernel: each CTA walks output tiles t = blockIdx.x, +gridDim.x,
// ... (row tiles fastest, so the CTAs in flight share the same weight tiles).
// Two accumulator buffers in tensor memory let the epilogue of one tile (or
// K group) overlap the MMAs of the next.
template <int KIND, bool GROUPED, bool DBG>
__global__ void __launch_bounds__(gemm_threads<GROUPED>(), 1)
    qgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const GemmParams p) {
  using C = GemmCfg<KIND>;
  using E = EpiCfg<GROUPED>;
  constexpr int S = gemm_stages<KIND, GROUPED>();
  constexpr uint32_t kCols = (KIND == KIND_NVF4) ? 512 : 256;
  constexpr uint32_t kSfCol = 2 * kBN;  // NVFP4 scale factors live after the two accumulators
  if (p.mode_dev != nullptr && SIXBIT_MODE_OF(*p.mode_dev) != p.want_mode) return;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* tiles = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * stage_bytes<KIND>());
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* accf = bars + 2 * S;      // [2] accumulator buffer ready
  uint64_t* acce = bars + 2 * S + 2;  // [2] accumulator buffer drained
  uint64_t* drain = bars + 2 * S + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* sw_full = bars + 2 * S + 6;   // GROUPED: a tile's group scales are staged
  uint64_t* sw_empty = bars + 2 * S + 7;  // GROUPED: ... and no longer read
  float* sw_smem = reinterpret_cast<float*>(bars + 2 * S + 8);  // GROUPED: [K/128][128] group scales of a tile

  auto A_tile = [&](int s) { return tiles + s * stage_bytes<KIND>(); };
  auto B_tile = [&](int s) { return tiles + s * stage_bytes<KIND>() + kTileBytes; };
  auto SFA = [&](int s) { return tiles + s * stage_bytes<KIND>() + 2 * kTileBytes; };
  auto SFB = [&](int s) { return tiles + s * stage_bytes<KIND>() + 2 * kTileBytes + C::kSfBytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + kBM - 1) / kBM;
  const int tiles_n = (p.N + kBN - 1) / kBN;
  const int ntiles = tiles_m * tiles_n;
  // NVFP4 stages hold 256 K-elements; a K that is an odd multiple of 128
  // leaves a half stage at the end (TMA zero-fills its missing columns; only
  // its valid scale chunks are copied and only its valid MMAs issued).
  const int nk = (p.K + C::kKStage - 1) / C::kKStage;
  const int groups = p.K / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&accf[0], 1);
    mbar_init(&accf[1], 1);
    mbar_init(&acce[0], E::kThreads);
    mbar_init(&acce[1], E::kThreads);
    mbar_init(drain, 1);
    mbar_init(sw_full, E::kThreads);
    mbar_init(sw_empty, E::kThreads);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer --
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const int m_tile = t % tiles_m, n_tile = t / tiles_m;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (it >= S && !mbar_wait(&empty[s], ph ^ 1, abort_flag)) {
            set_error(p.err, SIXBIT_ETIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          const int kvalid = min(C::kKStage, p.K - kb * C::kKStage);
          const uint32_t sf_bytes = C::kSfBytes == 0 ? 0u : static_cast<uint32_t>(kvalid / 64) * 512u;
          mbar_expect_tx(&full[s], 2 * kTileBytes + 2 * sf_bytes);
          tma_load_2d(A_tile(s), &tmA, &full[s], kb * C::kKCoord, m_tile * kBM);
          tma_load_2d(B_tile(s), &tmB, &full[s], kb * C::kKCoord, n_tile * kBN);
          if constexpr (KIND == KIND_NVF4) {
            const size_t row_bytes = static_cast<size_t>(128) * (p.K >> 4);
            bulk_load(SFA(s), p.sfa + m_tile * row_bytes + static_cast<size_t>(kb) * 2048, sf_bytes, &full[s]);
            bulk_load(SFB(s), p.sfb + n_tile * row_bytes + static_cast<size_t>(kb) * 2048, sf_bytes, &full[s]);
          }
        }
      }
      // every copy this CTA started lands before it can exit
      for (uint32_t j = (it > S ? it - S : 0); j < it; ++j) (void)mbar_wait(&full[j % S], (j / S) & 1, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------- MMA issuer --
      uint32_t it = 0;   // stage counter
      uint32_t ac = 0;   // accumulator-buffer use counter (tiles, or K groups when GROUPED)
      bool ok = true;
      constexpr int spg = 128 / C::kKStage > 0 ? 128 / C::kKStage : 1;  // stages per K group (bf16 kinds)
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        for (int kb = 0; kb < nk && ok; ++kb, ++it) {
          const bool acc_start = GROUPED ? (kb % spg) == 0 : kb == 0;
          const uint32_t buf = ac & 1;
          if (acc_start && ac >= 2 && !mbar_wait(&acce[buf], ((ac >> 1) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const int s = it % S;
          if (!mbar_wait(&full[s], (it / S) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(A_tile(s));
          const uint32_t b_base = smem_u32(B_tile(s));
          const uint32_t d_tmem = tmem + buf * kBN;
          if constexpr (KIND == KIND_NVF4) {
            const int nmma = min(C::kKStage, p.K - kb * C::kKStage) / 64;
#pragma unroll
            for (int k = 0; k < C::kMmaPerStage; ++k) {
              if (k < nmma) {
                tmem_cp_32x128b_warpx4(tmem + kSfCol + 4 * k, sdesc_sf(smem_u32(SFA(s)) + 512 * k));
                tmem_cp_32x128b_warpx4(tmem + kSfCol + 16 + 4 * k, sdesc_sf(smem_u32(SFB(s)) + 512 * k));
              }
            }
#pragma unroll
            for (int k = 0; k < C::kMmaPerStage; ++k)
              if (k < nmma)
                mma_nvf4(d_tmem, sdesc_sw128(a_base + 32 * k), sdesc_sw128(b_base + 32 * k), C::kIdesc,
                         tmem + kSfCol + 4 * k, tmem + kSfCol + 16 + 4 * k, (acc_start && k == 0) ? 0u : 1u);
          } else {
#pragma unroll
            for (int k = 0; k < C::kMmaPerStage; ++k)
              mma_bf16(d_tmem, sdesc_sw128(a_base + 32 * k), sdesc_sw128(b_base + 32 * k), C::kIdesc,
                       (acc_start && k == 0) ? 0u : 1u);
          }
          tc_commit(&empty[s]);
          const bool acc_end = GROUPED ? (kb % spg) == spg - 1 : kb == nk - 1;
          if (acc_end) {
            tc_commit(&accf[buf]);
            ++ac;
          }
        }
      }
      if (!ok) {
        set_error(p.err, SIXBIT_ETIMEOUT);
        *abort_flag = 1;
      }
      tc_commit(drain);  // all tensor-core work issued here completes before exit
      (void)mbar_wait(drain, 0, nullptr);
    }
  } else {
    // -------------------------------------------------------- epilogue --
    const int ew = warp - 2;              // 0 .. kWarps-1
    const int q = warp & 3;               // tensor-memory lane quarter this warp may read
    const int col0 = (ew >> 2) * E::kCols;  // first accumulator column of this thread
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q) << 16);
    uint32_t ac = 0;
    uint32_t lt = 0;  // local tile counter
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++lt) {
      const int m_tile = t % tiles_m, n_tile = t / tiles_m;
      const int row = m_tile * kBM + 32 * q + lane;
      const int n0 = n_tile * kBN;
      if constexpr (GROUPED) {
        // the tile's group scales s_w[g][n0 .. n0+127] into shared memory, once
        // every epilogue thread is done with the previous tile's (bounded waits)
        if (lt >= 1 && !mbar_wait(sw_empty, (lt - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        for (int i = threadIdx.x - 64; i < groups * kBN; i += E::kThreads) {
          const int g = i / kBN, c = i % kBN;
          sw_smem[i] = (n0 + c < p.N) ? __ldg(p.grp_scale + static_cast<size_t>(g) * p.N + n0 + c) : 0.f;
        }
        mbar_arrive(sw_full);
        if (!mbar_wait(sw_full, lt & 1, abort_flag)) {
          ok = false;
          break;
        }
        float sum[E::kCols];
#pragma unroll
        for (int j = 0; j < E::kCols; ++j) sum[j] = 0.f;
        for (int g = 0; g < groups; ++g, ++ac) {
          const uint32_t buf = ac & 1;
          if (!mbar_wait(&accf[buf], (ac >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float4* sw4 = reinterpret_cast<const float4*>(sw_smem + g * kBN + col0);
#pragma unroll
          for (int c = 0; c < E::kCols / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_addr + buf * kBN + col0 + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 s4 = sw4[c * 8 + j4];
              const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int j = c * 32 + j4 * 4 + u;
                sum[j] = fmaf(sv[u], __uint_as_float(r[j4 * 4 + u]), sum[j]);
              }
            }
            if constexpr (DBG) {
              if (row < p.M) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const int n = n0 + col0 + c * 32 + j;
                  if (n < p.N)
                    p.acc_dbg[(static_cast<size_t>(g) * p.M + row) * p.N + n] = __float2int_rn(__uint_as_float(r[j]));
                }
              }
            }
          }
          tc_fence_before();
          mbar_arrive(&acce[buf]);
        }
        if (!ok) break;
        mbar_arrive(sw_empty);
        const float sm = (row < p.M) ? p.row_scale[row] : 0.f;
#pragma unroll
        for (int c = 0; c < E::kCols / 32; ++c) {
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(sum[c * 32 + j], sm);
          if (n0 + col0 + c * 32 < p.N) epilogue_store32(p, row, n0 + col0 + c * 32, v);
        }
      } else {
        const uint32_t buf = ac & 1;
        if (!mbar_wait(&accf[buf], (ac >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float alpha = 1.0f;
        if constexpr (KIND == KIND_NVF4) alpha = __fmul_rn(*p.s_a, *p.s_b);
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(lane_addr + buf * kBN + c * 32, r);
          tmem_ld_wait();
          if (c == kBN / 32 - 1) {  // buffer fully read: hand it back to the MMA warp
            tc_fence_before();
            mbar_arrive(&acce[buf]);
          }
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(__uint_as_float(r[j]), alpha);
          if (n0 + c * 32 < p.N) epilogue_store32(p, row, n0 + c * 32, v);
        }
        ++ac;
      }
    }
    if (!ok) {
      set_error(p.err, SIXBIT_ETIMEOUT);
      *abort_flag = 1;
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ------------------------------------------------------------ host launch --

static int num_sms() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  return sms;
}

template <int KIND, bool GROUPED, bool DBG>
static cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, cudaStream_t st) {
  static int attr_done = 0;
  const int smem = gemm_stages<KIND, GROUPED>() * stage_bytes<KIND>() + 1024 + 256 +
                   (GROUPED ? (p.K / 128) * kBN * 4 : 0);
  if (smem > attr_done) {
    cudaError_t e = cudaFuncSetAttribute(qgemm_kernel<KIND, GROUPED, DBG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_done = smem;
  }
  const int ntiles = ((p.M + kBM - 1) / kBM) * ((p.N + kBN - 1) / kBN);
  const int grid = ntiles < num_sms() ? ntiles : num_sms();
  qgemm_kernel<KIND, GROUPED, DBG><<<grid, gemm_threads<GROUPED>(), smem, st>>>(a, b, p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_qgemm_nvf4(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, cudaStream_t st) {
  return launch_one<KIND_NVF4, false, false>(a, b, p, st);
}
cudaError_t launch_qgemm_bf16(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, cudaStream_t st) {
  return launch_one<KIND_BF16, false, false>(a, b, p, st);
}
cudaError_t launch_qgemm_int8(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, cudaStream_t st) {
  if (p.acc_dbg != nullptr) return launch_one<KIND_BF16, true, true>(a, b, p, st);
  return launch_one<KIND_BF16, true, false>(a, b, p, st);
}

}  // namespace sixbit
