// Quantized GEMMs on the fifth-generation tensor cores (tcgen05) of sm_103a:
// the NVFP4 (W4A4) kind and the BF16 kind.  The W4A8 kind, whose integer
// operands need their own pipeline, is in qgemm_w4a8.cu.
//
// Method: "6Bit-Diffusion" technical summary sections 2.A and 4 (NVFP4
// activations against 4-bit weights: W4A4) and 2.C (PDR's FP16/BF16
// recompute); popular summary section 4 (custom CUDA kernels).
//
// A persistent CTA per SM walks 128 x 256 output tiles with three warp roles:
//   warp 0      TMA producer: A/B tiles (128-byte swizzle) and, for NVFP4,
//               the scale-factor chunks, into a ring of shared-memory stages
//               guarded by full/empty mbarriers;
//   warp 1      allocates tensor memory; one lane issues tcgen05.mma and
//               tcgen05.commit to release stages and accumulators;
//   epilogue    16 warps from warp 2: tcgen05.ld of the FP32 accumulators
//               (warp w reads lanes 32*(w%4)..+31 = tile rows, a 64-column
//               part), scaling, GELU or residual, bf16 TMA stores (or direct
//               stores: NVFP4, FP32 output);
//   last warp   (NVFP4) tcgen05.cp of each stage's scale factors into its
//               own tensor-memory slot.
// Kinds:
//   NVFP4  kind::mxf4nvf4.block_scale.scale_vec::4X, E2M1 x E2M1 with one
//          E4M3 scale per 16 elements, 256 K-elements (128 bytes) per stage;
//          a 128 x 256 tile is one N = 256 MMA per K step.  One
//          accumulator buffer (256 columns) plus the scale factors fill
//          tensor memory; the epilogue drains the accumulator to registers
//          and releases it before its stores, so they overlap the next tile.
//   BF16   kind::f16 with bf16 operands, N = 256 MMAs, 64 K-elements per
//          stage, two accumulator buffers (the epilogue of tile t overlaps
//          the MMAs of tile t + 1).
// Every mbarrier wait is bounded (2 s); on expiry the kernel records
// SIXBIT_ETIMEOUT in the error word, drains its in-flight copies and tensor
// core work with bounded waits, frees tensor memory and returns.
#include <cstdint>

#include "common.cuh"
#include "ctx_cache.h"
#include "gemm_common.cuh"
#include "internal.h"

namespace sixbit {

constexpr int kBM = 128;
constexpr int kBN = 256;        // output tile columns
// 16 epilogue warps, four per tensor-memory lane quarter (64 columns each),
// spread the GELU / residual / store work of a tile over 512 threads (whose
// registers fit the 96-per-thread budget of 576-608 threads).
constexpr int kEpiWarps = 16;
constexpr int kEpiCols = kBN / (kEpiWarps / 4);  // accumulator columns per thread
constexpr int kEpiWarp0 = 2;                     // first epilogue warp
static_assert(kEpiWarps <= kBsMaxWarps, "block statistics: one partial per epilogue warp");

enum { KIND_BF16 = 0, KIND_NVF4 = 1 };

// NVFP4 adds a warp that copies the scale factors into tensor memory: each
// tcgen05.cp costs its issuing thread about 64 cycles and an NVFP4 MMA of a
// stage's K step about 130, so twelve copies per four MMAs on the MMA thread
// would pace the main loop.  (Splitting the copies over two warps was slower.)
template <int KIND>
__host__ __device__ constexpr int gemm_threads() {
  return 64 + kEpiWarps * 32 + (KIND == KIND_NVF4 ? 32 : 0);
}

template <int KIND>
struct GemmCfg;
template <>
struct GemmCfg<KIND_BF16> {
  static constexpr int kStages = 4;
  static constexpr int kKStage = 64;      // K elements per stage
  static constexpr int kKCoord = 64;      // TMA x coordinate step per stage
  static constexpr int kMmaPerStage = 4;  // K = 16 per MMA
  static constexpr int kSfaBytes = 0;
  static constexpr int kSfbBytes = 0;
  static constexpr uint32_t kIdesc = idesc_bf16(kBM, kBN);
};
template <>
struct GemmCfg<KIND_NVF4> {
  static constexpr int kStages = 4;
  static constexpr int kKStage = 256;
  static constexpr int kKCoord = 128;     // bytes of packed E2M1
  static constexpr int kMmaPerStage = 4;  // K = 64 per MMA
  static constexpr int kSfaBytes = 2048;  // 128 rows x 16 scales
  static constexpr int kSfbBytes = 4096;  // 256 rows x 16 scales (two 128-row chunks)
  static constexpr uint32_t kIdesc = idesc_nvf4(kBM, 128);
};

constexpr int kATileBytes = kBM * 128;  // 128 rows x 128 bytes
constexpr int kBTileBytes = kBN * 128;  // 256 rows x 128 bytes

template <int KIND>
__host__ __device__ constexpr int stage_bytes() {
  return kATileBytes + kBTileBytes + GemmCfg<KIND>::kSfaBytes + GemmCfg<KIND>::kSfbBytes;
}

// The BF16 kind stages each epilogue warp's 32 x 32 bf16 output chunk in
// shared memory (64-byte rows, 64-byte TMA swizzle) and writes it with one
// TMA store: a warp's direct stores would touch 32 rows, 16 bytes each
// (310 vs 329 us at 17776 x 7680 x 1920).  NVFP4 has no shared memory left
// and stores directly.
template <int KIND>
__host__ __device__ constexpr bool tma_y() {
  return KIND != KIND_NVF4;
}
constexpr int kBoxBytes = 32 * 64;
template <int KIND>
__host__ __device__ constexpr int staging_bytes() {
  return tma_y<KIND>() ? kEpiWarps * kBoxBytes : 0;
}

// Layout: [stages | output staging | barriers (256 B)].
template <int KIND>
__host__ __device__ constexpr int gemm_smem_bytes() {
  return GemmCfg<KIND>::kStages * stage_bytes<KIND>() + staging_bytes<KIND>() + 1024 /*align*/ + 256 /*barriers*/;
}
static_assert(gemm_smem_bytes<KIND_BF16>() <= 227 * 1024 && gemm_smem_bytes<KIND_NVF4>() <= 227 * 1024,
              "shared memory per CTA");

// max |y| over a thread's 64 output columns after the block Hadamard rotation
// y = x . blockdiag(H_b / sqrt b), b in {16, 64}: the same FP32 butterfly
// (ascending strides, exact power-of-two scale last) as the quantizer, so
// the maximum over all threads equals its amax pass over the stored Y.
template <int B>
__device__ __forceinline__ float rot_amax64(float (&v)[2][32]) {
#pragma unroll
  for (int h = 1; h < 32 && h < B; h <<= 1) {
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if ((i & h) == 0) {
          const float a = v[c][i], b = v[c][i + h];
          v[c][i] = __fadd_rn(a, b);
          v[c][i + h] = __fsub_rn(a, b);
        }
  }
  constexpr float s = B == 16 ? 0.25f : 0.125f;
  float m = 0.f;
  if constexpr (B == 64) {  // the last stage pairs the two halves
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      m = fmaxf(m, fabsf(__fmul_rn(__fadd_rn(v[0][i], v[1][i]), s)));
      m = fmaxf(m, fabsf(__fmul_rn(__fsub_rn(v[0][i], v[1][i]), s)));
    }
  } else {
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(__fmul_rn(v[c][i], s)));
  }
  return m;
}

// Persistent kernel: each CTA walks output tiles t = blockIdx.x, +gridDim.x,
// ...; p.n_fastest picks whether row or column tiles vary fastest along t.
// BS: the residual epilogue also produces the block's statistics and Delta
// (p.bs_delta, p.bs_parts; gemm_common.cuh).
template <int KIND, bool BS>
__global__ void __launch_bounds__(gemm_threads<KIND>(), 1)
    qgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmY, const GemmParams p) {
  using C = GemmCfg<KIND>;
  constexpr int S = C::kStages;
  constexpr bool kNvf4 = KIND == KIND_NVF4;
  constexpr uint32_t kCols = 512;
  // NVFP4: the scale factors of stage s live in TMEM columns 256 + 64 s:
  // SFA in [0, 16), SFB in [16, 48) of that slot; one slot per stage, so the
  // copies for later stages never overwrite scales earlier MMAs still read.
  constexpr uint32_t kSfSlot0 = 256, kSfSlotCols = 64, kSfbOff = 16;
  static_assert(!kNvf4 || kSfSlot0 + S * kSfSlotCols <= 512, "scale-factor slots exceed tensor memory");
  constexpr uint32_t kBufs = kNvf4 ? 1 : 2;  // accumulator buffers of kBN columns
  if (p.mode_dev != nullptr && SIXBIT_MODE_OF(*p.mode_dev) != p.want_mode) return;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* tiles = smem;
  uint8_t* staging = smem + S * stage_bytes<KIND>();  // [kEpiWarps] output boxes (BF16 kind)
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + staging_bytes<KIND>());
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* accf = bars + 2 * S;                    // [kBufs] accumulator buffer ready
  uint64_t* acce = bars + 2 * S + 2;                // [kBufs] accumulator buffer drained
  uint64_t* drain = bars + 2 * S + 4;
  uint64_t* sf_full = drain + 1;                    // NVFP4: [S] the stage's scale factors are in tensor memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_full + S);
  static_assert((3 * S + 5) * 8 + 8 <= 256, "barrier area");
  static_assert(kBufs <= 2 && kBufs * kBN + (kNvf4 ? S * 64 : 0) <= kCols, "tensor memory");
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  auto A_tile = [&](int s) { return tiles + s * stage_bytes<KIND>(); };
  auto B_tile = [&](int s) { return tiles + s * stage_bytes<KIND>() + kATileBytes; };
  auto SFA = [&](int s) { return tiles + s * stage_bytes<KIND>() + kATileBytes + kBTileBytes; };
  auto SFB = [&](int s) { return tiles + s * stage_bytes<KIND>() + kATileBytes + kBTileBytes + C::kSfaBytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + kBM - 1) / kBM;
  const int tiles_n = (p.N + kBN - 1) / kBN;
  const int ntiles = tiles_m * tiles_n;
  auto tile_of = [&](int t, int& m_tile, int& n_tile) {
    if (p.n_fastest) {
      n_tile = t % tiles_n;
      m_tile = t / tiles_n;
    } else {
      m_tile = t % tiles_m;
      n_tile = t / tiles_m;
    }
  };
  // NVFP4 stages hold 256 K-elements; a K that is an odd multiple of 128
  // leaves a half stage at the end (TMA zero-fills its missing columns; only
  // its valid scale chunks are copied and only its valid MMAs issued).
  const int nk = (p.K + C::kKStage - 1) / C::kKStage;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (uint32_t b = 0; b < kBufs; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], kEpiWarps);
    }
    mbar_init(drain, 1);
    if constexpr (kNvf4)
      for (int s = 0; s < S; ++s) mbar_init(&sf_full[s], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (tma_y<KIND>() && p.y_tma) prefetch_tmap(&tmY);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < kEpiWarp0) {
    if (warp == 0) {
      if (lane == 0) {
        // ------------------------------------------------------ producer --
        uint32_t it = 0;
        bool ok = true;
        const size_t sf_rows_bytes = static_cast<size_t>(128) * (p.K >> 4);  // one 128-row scale tile
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
          int m_tile, n_tile;
          tile_of(t, m_tile, n_tile);
          const int nj = (n_tile * kBN + 128 < p.N) ? 2 : 1;  // 128-row halves of B that exist
          for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = it % S;
            const uint32_t ph = (it / S) & 1;
            if (it >= S && !mbar_wait(&empty[s], ph ^ 1, abort_flag, p.wait_ns)) {
              set_error(p.err, SIXBIT_ETIMEOUT);
              *abort_flag = 1;
              ok = false;
              break;
            }
            if (p.withhold_first && it == 0) continue;  // failure-path test: stage 0 never lands
            const int kvalid = min(C::kKStage, p.K - kb * C::kKStage);
            const uint32_t sf_bytes = kNvf4 ? static_cast<uint32_t>(kvalid / 64) * 512u : 0u;
            mbar_expect_tx(&full[s], kATileBytes + kBTileBytes + sf_bytes * (1 + (kNvf4 ? nj : 0)));
            tma_load_2d(A_tile(s), &tmA, &full[s], kb * C::kKCoord, m_tile * kBM);
            tma_load_2d(B_tile(s), &tmB, &full[s], kb * C::kKCoord, n_tile * kBN);
            if constexpr (kNvf4) {
              bulk_load(SFA(s), p.sfa + m_tile * sf_rows_bytes + static_cast<size_t>(kb) * 2048, sf_bytes, &full[s]);
              for (int j = 0; j < nj; ++j)
                bulk_load(SFB(s) + 2048 * j, p.sfb + (2 * n_tile + j) * sf_rows_bytes + static_cast<size_t>(kb) * 2048,
                          sf_bytes, &full[s]);
            }
          }
        }
        // every copy this CTA started lands before it can exit
        for (uint32_t j = (it > S ? it - S : 0); j < it; ++j) (void)mbar_wait(&full[j % S], (j / S) & 1, nullptr, p.wait_ns);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---------------------------------------------------- MMA issuer --
        uint32_t it = 0;  // stage counter
        uint32_t ac = 0;  // accumulator-buffer use counter (tiles)
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
          int m_tile, n_tile;
          tile_of(t, m_tile, n_tile);
          (void)m_tile;
          const int nj = (n_tile * kBN + 128 < p.N) ? 2 : 1;
          for (int kb = 0; kb < nk && ok; ++kb, ++it) {
            const bool acc_start = kb == 0;
            const uint32_t buf = ac % kBufs;
            // the buffer's previous contents must have been drained by the epilogue
            if (acc_start && ac >= kBufs && !mbar_wait(&acce[buf], ((ac / kBufs) - 1) & 1, abort_flag, p.wait_ns)) {
              ok = false;
              break;
            }
            const int s = it % S;
            if (!mbar_wait(&full[s], (it / S) & 1, abort_flag, p.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(A_tile(s));
            const uint32_t b_base = smem_u32(B_tile(s));
            const uint32_t d_tmem = tmem + buf * kBN;
            if constexpr (kNvf4) {
              const int nmma = min(C::kKStage, p.K - kb * C::kKStage) / 64;
              const uint32_t sfa_col = tmem + kSfSlot0 + kSfSlotCols * s;
              const uint32_t sfb_col = sfa_col + kSfbOff;
              if (!mbar_wait(&sf_full[s], (it / S) & 1, abort_flag, p.wait_ns)) {  // copied by the scale-factor warp
                ok = false;
                break;
              }
              tc_fence_after();
              // one N = 256 MMA (B scale chunks for rows 0-127 and 128-255 in
              // consecutive 4-column groups), or N = 128 when only half the tile exists
              const uint32_t idesc = nj == 2 ? idesc_nvf4(kBM, 256) : C::kIdesc;
  #pragma unroll
              for (int k = 0; k < C::kMmaPerStage; ++k) {
                if (k < nmma)
                  mma_nvf4(d_tmem, sdesc_sw128(a_base + 32 * k), sdesc_sw128(b_base + 32 * k), idesc,
                           sfa_col + 4 * k, sfb_col + 8 * k, (acc_start && k == 0) ? 0u : 1u);
              }
            } else {
  #pragma unroll
              for (int k = 0; k < C::kMmaPerStage; ++k)
                mma_bf16(d_tmem, sdesc_sw128(a_base + 32 * k), sdesc_sw128(b_base + 32 * k), C::kIdesc,
                         (acc_start && k == 0) ? 0u : 1u);
            }
            tc_commit(&empty[s]);
            const bool acc_end = kb == nk - 1;
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
        (void)mbar_wait(drain, 0, nullptr, p.wait_ns);
      }
    }
  } else if (warp < kEpiWarp0 + kEpiWarps) {
    // -------------------------------------------------------- epilogue --
    const int ew = warp - kEpiWarp0;              // 0 .. kEpiWarps-1
    const int q = warp & 3;                       // tensor-memory lane quarter this warp may read
    const int col0 = (ew >> 2) * kEpiCols;        // first accumulator column of this thread
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q) << 16) + col0;
    uint8_t* my_box = staging + ew * kBoxBytes;   // BF16 kind: this warp's output box
    BsAcc bs = bs_zero();
    // Epilogue + store of columns [n, n + 32) of this lane's row (n < N, warp-uniform).
    auto store32 = [&](int row, int n, float (&v)[32]) {
      if constexpr (tma_y<KIND>()) {
        if (p.y_tma) {
          if (row < p.M) {
            if constexpr (BS)
              residual_bs_chunk32(p, row, n, v, bs);
            else
              epilogue_apply32(p, row, n, v);
          }
          if (lane == 0) bulk_wait_read0();  // the previous box has been read out
          __syncwarp();
          stage_bf16x32(my_box, lane, v);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {  // rows >= M and columns >= N of the box are not written
            tma_store_2d(&tmY, my_box, n, row - lane);
            bulk_commit();
          }
          return;
        }
      }
      epilogue_store32(p, row, n, v);  // leaves the stored bf16 values in v
      if constexpr (BS)
        if (row < p.M) bs_chunk32(p, row, n, v, bs);
    };
    uint32_t ac = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      int m_tile, n_tile;
      tile_of(t, m_tile, n_tile);
      const int row = m_tile * kBM + 32 * q + lane;
      const int nb = n_tile * kBN + col0;         // first output column of this thread
      if (nb >= p.N) {                            // nothing of this part exists (ragged N)
        const uint32_t buf = ac % kBufs;
        if (!mbar_wait(&accf[buf], (ac / kBufs) & 1, abort_flag, p.wait_ns)) { ok = false; break; }
        release_acc(&acce[buf], lane);
        ++ac;
        continue;
      }
      {
        const uint32_t buf = ac % kBufs;
        if (!mbar_wait(&accf[buf], (ac / kBufs) & 1, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float alpha = 1.0f;
        if constexpr (kNvf4) alpha = __fmul_rn(*p.s_a, *p.s_b);
        if constexpr (kNvf4 && BS) {
          // the block statistics need the registers: one 32-column chunk at a
          // time, the accumulator released after the last load
#pragma unroll 1
          for (int c = 0; c < kEpiCols / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_addr + c * 32, r);
            tmem_ld_wait(r);
            if (c == kEpiCols / 32 - 1) release_acc(&acce[buf], lane);
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(__uint_as_float(r[j]), alpha);
            if (nb + c * 32 < p.N) {
              epilogue_store32(p, row, nb + c * 32, v);  // leaves the stored bf16 values in v
              if (row < p.M) bs_chunk32(p, row, nb + c * 32, v, bs);
            }
          }
        } else if constexpr (kNvf4) {
          // single accumulator: drain all of this thread's columns, release, then store
          uint32_t r[kEpiCols / 32][32];
#pragma unroll
          for (int c = 0; c < kEpiCols / 32; ++c) tmem_ld32(lane_addr + c * 32, r[c]);
#pragma unroll
          for (int c = 0; c < kEpiCols / 32; ++c) tmem_ld_wait(r[c]);
          release_acc(&acce[buf], lane);
          float v[kEpiCols / 32][32];
#pragma unroll
          for (int c = 0; c < kEpiCols / 32; ++c) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[c][j] = __fmul_rn(__uint_as_float(r[c][j]), alpha);
            if (nb + c * 32 < p.N) epilogue_store32(p, row, nb + c * 32, v[c]);
          }
          if constexpr (kEpiCols == 64 && !BS) {  // (an up projection's epilogue; BS is a down projection's)
            if (p.rot_amax != nullptr) {  // the next quantizer's amax pass, on the stored values
              float m = 0.f;
              if (row < p.M && nb < p.N) m = p.had_block == 16 ? rot_amax64<16>(v) : rot_amax64<64>(v);
              m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
              m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
              m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
              m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
              m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
              if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(p.rot_amax), __float_as_uint(m));  // m >= 0
            }
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < kEpiCols / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_addr + buf * kBN + c * 32, r);
            tmem_ld_wait(r);
            if (c == kEpiCols / 32 - 1) release_acc(&acce[buf], lane);  // buffer fully read
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(__uint_as_float(r[j]), alpha);
            if (nb + c * 32 < p.N) store32(row, nb + c * 32, v);
          }
        }
        ++ac;
      }
    }
    if constexpr (BS) bs_flush(p, bs, ew, kEpiWarps, lane);
    if (!ok) {
      set_error(p.err, SIXBIT_ETIMEOUT);
      *abort_flag = 1;
    }
    if (tma_y<KIND>() && lane == 0) bulk_wait0();  // every output box has been written
    __syncwarp();
    tc_fence_before();
  } else if constexpr (kNvf4) {
    if (lane == 0) {
      // ------------------------------------- scale factors -> tensor memory --
      // Stage s's scales go to slot s once the MMAs that read the slot in the
      // previous round are done (empty[s]) and the stage has landed (full[s]).
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        int m_tile, n_tile;
        tile_of(t, m_tile, n_tile);
        (void)m_tile;
        const int nj = (n_tile * kBN + 128 < p.N) ? 2 : 1;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % S;
          if ((it >= S && !mbar_wait(&empty[s], ((it / S) - 1) & 1, abort_flag, p.wait_ns)) ||
              !mbar_wait(&full[s], (it / S) & 1, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nmma = min(C::kKStage, p.K - kb * C::kKStage) / 64;
          const uint32_t sfa_col = tmem + kSfSlot0 + kSfSlotCols * s;
          const uint32_t sfb_col = sfa_col + kSfbOff;
#pragma unroll
          for (int k = 0; k < C::kMmaPerStage; ++k) {
            if (k < nmma) {
              tmem_cp_32x128b_warpx4(sfa_col + 4 * k, sdesc_sf(smem_u32(SFA(s)) + 512 * k));
              for (int j = 0; j < nj; ++j)
                tmem_cp_32x128b_warpx4(sfb_col + 8 * k + 4 * j, sdesc_sf(smem_u32(SFB(s)) + 2048 * j + 512 * k));
            }
          }
          tc_commit(&sf_full[s]);
        }
      }
      if (!ok) {
        set_error(p.err, SIXBIT_ETIMEOUT);
        *abort_flag = 1;
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ------------------------------------------------------------ host launch --

template <int KIND, bool BS>
static cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& y, const GemmParams& p,
                              cudaStream_t st) {
  constexpr int smem = gemm_smem_bytes<KIND>();
  const cudaError_t e = set_smem_once<qgemm_kernel<KIND, BS>>(smem);
  if (e != cudaSuccess) return e;
  const int ntiles = ((p.M + kBM - 1) / kBM) * ((p.N + kBN - 1) / kBN);
  const int sms = sm_count();
  const int grid = ntiles < sms ? ntiles : sms;
  qgemm_kernel<KIND, BS><<<grid, gemm_threads<KIND>(), smem, st>>>(a, b, y, p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_qgemm_nvf4(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, cudaStream_t st) {
  GemmParams q = p;
  q.y_tma = 0;
  return q.bs_delta != nullptr ? launch_one<KIND_NVF4, true>(a, b, a /*unused*/, q, st)
                                : launch_one<KIND_NVF4, false>(a, b, a /*unused*/, q, st);
}
cudaError_t launch_qgemm_bf16(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& y, const GemmParams& p,
                              cudaStream_t st) {
  return p.bs_delta != nullptr ? launch_one<KIND_BF16, true>(a, b, y, p, st)
                                : launch_one<KIND_BF16, false>(a, b, y, p, st);
}

}  // namespace sixbit
