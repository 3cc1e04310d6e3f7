// W4A8 GEMM from the quantized operands, on the tcgen05 tensor cores of sm_103a.
//
// Method: "6Bit-Diffusion" technical summary sections 2.A and 4 (a volatile
// block runs INT8 activations against the 4-bit weights: W4A8); popular
// summary section 4 (custom CUDA kernels).
//
//   A  INT8 activation codes, s8 [M, K], symmetric per token, row scales s_m [M]
//   W  INT4 weight codes [N, K/2] (two's-complement nibbles, even k in the low
//      nibble), group scales s_w [K/128][N]
//   Y[m, n] = s_m[m] * sum_g s_w[g][n] * acc_g[m, n],
//   acc_g[m, n] = sum_{k in group g} qa[m, k] * qw[n, k]   (exact integers)
//
// GB300 has no integer MMA on its tensor cores (kind::i8 is not available on
// sm_103a), so the integers run through kind::f16 with fp16 operands: every
// code is exact in fp16, every product (|.| <= 889) and every 128-term group
// sum (|.| < 2^17) is an integer exactly representable in FP32, so the FP32
// accumulator of a group holds the exact integer sum, and the group's scale is
// applied afterwards.
//
// Operand expansion.  The weights are expanded once per call (w4_expand_kernel:
// INT4 -> fp16 into a caller-provided workspace of N*K*2 bytes, which stays in
// L2 for the GEMM that follows).  The activation codes are read by the GEMM
// itself (TMA, one byte per element) and expanded on chip by two converter
// warps: with u = q ^ 0x80, the fp16 bit pattern 0x64:u is 1024 + u =
// 1152 + q, and one fp16 subtraction of 1152 leaves q exactly.  (Expanding the
// 256-row weight tile on chip as well would repeat that work for every one of
// the ceil(M/128) output-row tiles and needs about 2.5 bytes of load/store
// traffic per element, beyond what the SM's shared-memory port has left next
// to the tensor core's own operand traffic.)
//
// A persistent CTA per SM walks 128 x 256 output tiles through a ring of four
// 64-K stages (fp16 A tile 16 KB, fp16 W tile 32 KB).  The s8 codes of a
// stage land in the upper half of its A tile; each converter warp reads its
// rows' codes into registers before it writes their fp16 rows over the region
// (warp 1, whose rows overwrite every row's codes, starts after warp 0 holds
// its own).
// Warps:
//   0       TMA producer: the s8 A tile and the fp16 W tile of each stage
//   1       allocates tensor memory; one lane issues tcgen05.mma and commits
//   2, 3    converters: s8 -> fp16 A operand, rows 64 c .. 64 c + 63 of a stage
//   4 - 11  fold + epilogue
// Warpgroup 0 lowers itself to 72 registers with setmaxnreg and the fold
// warpgroups raise themselves to 216 (4 x 72 + 8 x 216 = 12 x 168, and per SM
// sub-partition 72 + 2 x 216 = 3 x 168): a converter's 8 chunks of codes, and
// a fold thread's 128 running sums with a 32-column accumulator load, fit
// without spills.
//
// Tensor memory holds two 256-column accumulators; K groups alternate between
// them and the fold warps add s_w[g][n] * acc_g into registers while the next
// group accumulates.  The MMA thread waits on one barrier per stage (the
// weight tile's copy completes on the barrier the converters arrive on: an
// mbarrier phase needs its arrivals and its transaction bytes) and commits
// once per stage; a group's completion is the commit after its second stage.
// Every mbarrier wait is bounded (2 s); on expiry the kernel records
// SIXBIT_ETIMEOUT, raises an abort flag for the other roles, waits (bounded)
// for its copies and tensor-core work in flight, frees tensor memory and
// returns.
#include <cstdint>

#include "common.cuh"
#include "ctx_cache.h"
#include "gemm_common.cuh"
#include "internal.h"

namespace sixbit {
namespace w4a8 {

constexpr int kBM = 128, kBN = 256, kHalf = 128;
constexpr int kStages = 4;
constexpr int kKStage = 64;                          // K elements per stage
constexpr int kATile = kBM * kKStage * 2;            // fp16 A operand, 16 KB (128-byte swizzle)
constexpr int kBTile = kBN * kKStage * 2;            // fp16 W operand, 32 KB
constexpr int kS8Tile = kBM * kKStage;               // s8 A codes, 8 KB (row-major, 64-byte rows)
constexpr int kS8Off = kATile - kS8Tile;             // ... landing in the A tile's upper half
constexpr int kStageBytes = kATile + kBTile;
constexpr int kFoldWarps = 8, kWarp0 = 4, kThreads = 384;
constexpr int kCols = 64;                            // columns of each half a fold thread folds
constexpr int kSums = 2 * kCols;                     // running sums per fold thread
constexpr int kSwRing = 4;                           // groups of scales in flight per fold warp
constexpr int kBoxBytes = 32 * 64;                   // one 32 x 32 bf16 output box
constexpr int kRegsLaunch = 168, kRegsLow = 72, kRegsHigh = 216;
static_assert(4 * kRegsLow + 8 * kRegsHigh <= 12 * kRegsLaunch && kRegsLow + 2 * kRegsHigh <= 3 * kRegsLaunch,
              "the register split must fit in what the CTA is launched with");
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(kBN >> 3) << 17) |
                            (static_cast<uint32_t>(kBM >> 4) << 24);  // f16 x f16 -> f32, M 128, N 256, K-major

// [stages | output boxes | barriers (256 B) | per-warp rings of group scales]
constexpr int kSmemBytes = kStages * kStageBytes + kFoldWarps * kBoxBytes + 1024 + 256 +
                           kSwRing * kFoldWarps * kSums * 4;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

// fp16 pair (1152 + a, 1152 + b) -> (a, b): exact (both sides integers below 2048)
__device__ __forceinline__ uint32_t hsub1152(uint32_t x) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(0x64806480u));
  return d;
}

// 16 s8 codes -> 16 fp16 values (two 16-byte chunks, element order kept).
__device__ __forceinline__ void s8x16_to_f16(const uint4& in, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {in.x ^ 0x80808080u, in.y ^ 0x80808080u, in.z ^ 0x80808080u, in.w ^ 0x80808080u};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = hsub1152(__byte_perm(w[i], 0x64646464u, 0x4140));      // bytes 0, 1 -> 0x64:b0, 0x64:b1
    o[2 * i + 1] = hsub1152(__byte_perm(w[i], 0x64646464u, 0x4342));  // bytes 2, 3
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

template <bool DBG>
__global__ void __launch_bounds__(kThreads, 1)
    w4a8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmY, const GemmParams p) {
  if (p.mode_dev != nullptr && SIXBIT_MODE_OF(*p.mode_dev) != SIXBIT_MODE_INT8) return;
  constexpr int S = kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* boxes = smem + S * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(boxes + kFoldWarps * kBoxBytes);
  uint64_t* s8_full = bars + S;     // [S] s8 A tile landed
  // [S] the stage is ready: the W tile's bytes landed (the producer's
  // expect-tx arrival) and both converter warps wrote the fp16 A tile
  uint64_t* op_full = bars + 2 * S;
  uint64_t* empty = bars + 3 * S;   // [S] the stage's MMAs are done
  uint64_t* read0 = bars + 4 * S;   // [S] converter warp 0 holds its s8 codes
  uint64_t* afree = bars + 5 * S;   // [2] accumulator read back (eight fold warps)
  uint64_t* drain = afree + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert((5 * kStages + 3) * 8 + 8 <= 256, "barrier area");
  float* sw_smem = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 256);

  auto A_op = [&](int s) { return smem + s * kStageBytes; };
  auto W_op = [&](int s) { return smem + s * kStageBytes + kATile; };
  auto A_s8 = [&](int s) { return smem + s * kStageBytes + kS8Off; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_m = (p.M + kBM - 1) / kBM, tiles_n = (p.N + kBN - 1) / kBN;
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
  const int nk = p.K / kKStage;  // K % 128 == 0
  const int groups = p.K / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&s8_full[s], 1);
      mbar_init(&op_full[s], 3);
      mbar_init(&empty[s], 1);
      mbar_init(&read0[s], 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&afree[b], kFoldWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmY);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < kWarp0) {
    setmaxnreg_dec<kRegsLow>();  // the whole warpgroup, one instruction
    if (warp == 0) {
      if (lane == 0) {
        // ---------------------------------------------------------- producer --
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
          int m_tile, n_tile;
          tile_of(t, m_tile, n_tile);
          for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = it % S;
            if (it >= S && !mbar_wait(&empty[s], ((it / S) - 1) & 1, abort_flag, p.wait_ns)) {
              ok = false;
              break;
            }
            if (p.withhold_first && it == 0) continue;  // failure-path test: stage 0 never lands
            mbar_expect_tx(&op_full[s], kBTile);
            tma_load_2d(W_op(s), &tmW, &op_full[s], kb * kKStage, n_tile * kBN);
            mbar_expect_tx(&s8_full[s], kS8Tile);
            tma_load_2d(A_s8(s), &tmA, &s8_full[s], kb * kKStage, m_tile * kBM);
          }
        }
        if (!ok) {
          set_error(p.err, SIXBIT_ETIMEOUT);
          *abort_flag = 1;
        }
        // every copy this CTA started lands before it can exit
        for (uint32_t j = (it > S ? it - S : 0); j < it; ++j) {
          (void)mbar_wait(&op_full[j % S], (j / S) & 1, nullptr, p.wait_ns);
          (void)mbar_wait(&s8_full[j % S], (j / S) & 1, nullptr, p.wait_ns);
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // -------------------------------------------------------- MMA issuer --
        // Stage counter it and K-group counter gi run across tiles; group gi
        // is stages 2 gi and 2 gi + 1 and accumulates into buffer gi & 1.
        uint32_t it = 0, gi = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
          for (int g = 0; g < groups && ok; ++g, ++gi) {
            if (gi >= 2 && !mbar_wait(&afree[gi & 1], ((gi >> 1) - 1) & 1, abort_flag, p.wait_ns)) {
              ok = false;
              break;
            }
            const uint32_t d_tmem = tmem + (gi & 1) * kBN;
            for (int ss = 0; ss < 2; ++ss, ++it) {
              const int s = it % S;
              if (!mbar_wait(&op_full[s], (it / S) & 1, abort_flag, p.wait_ns)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a_base = smem_u32(A_op(s)), b_base = smem_u32(W_op(s));
#pragma unroll
              for (int k = 0; k < kKStage / 16; ++k)
                mma_bf16(d_tmem, sdesc_sw128(a_base + 32 * k), sdesc_sw128(b_base + 32 * k), kIdesc,
                         (ss == 0 && k == 0) ? 0u : 1u);
              tc_commit(&empty[s]);  // frees the stage; after a group's second stage, also its completion
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
    } else {
      // ------------------------------------------------------------ converters --
      // Warp c converts rows 64 c .. 64 c + 63.  Each lane first loads its 8
      // chunks (rows 64 c + 8 i + lane / 4, 16 bytes at column 16 (lane % 4):
      // every load of the warp reads 512 contiguous bytes); then each chunk
      // becomes two fp16 chunks of the 128-byte-swizzled operand (16-byte
      // chunk j of row r at j ^ (r & 7)).  The fp16 rows 0 .. 63 lie below the
      // s8 codes, but rows 64 .. 127 overwrite the codes of every row, so warp
      // 1 starts only once warp 0 holds its codes (read0, a bounded wait);
      // nothing but warp 1 itself overwrites warp 1's codes.
      const int c = warp - 2;
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % S;
          if (!mbar_wait(&s8_full[s], (it / S) & 1, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          if (c == 1 && !mbar_wait(&read0[s], (it / S) & 1, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          const uint8_t* src = A_s8(s);
          uint8_t* dst = A_op(s);
          const int j = lane & 3;
          uint4 in[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) in[i] = *reinterpret_cast<const uint4*>(src + (64 * c + 8 * i + (lane >> 2)) * 64 + j * 16);
          __syncwarp();
          if (c == 0 && lane == 0) mbar_arrive(&read0[s]);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 64 * c + 8 * i + (lane >> 2);
            uint4 lo, hi;
            s8x16_to_f16(in[i], lo, hi);
            *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * j) ^ (r & 7)) << 4)) = lo;
            *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * j + 1) ^ (r & 7)) << 4)) = hi;
          }
          fence_proxy_async_smem();  // the tensor core reads these through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive(&op_full[s]);
        }
      }
      if (!ok && lane == 0) {
        set_error(p.err, SIXBIT_ETIMEOUT);
        *abort_flag = 1;
      }
    }
  } else {
    setmaxnreg_inc<kRegsHigh>();  // each fold warpgroup, one instruction
    // -------------------------------------------------------- fold + epilogue --
    const int ew = warp - kWarp0;          // 0 .. 7
    const int q = warp & 3;                // tensor-memory lane quarter this warp may read
    const int cs = (ew >> 2) * kCols;      // first column of this thread within each half
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q) << 16) + cs;
    float* my_sw = sw_smem + ew * kSwRing * kSums;  // [slot][half][64]
    uint8_t* my_box = boxes + ew * kBoxBytes;
    uint32_t gi = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      int m_tile, n_tile;
      tile_of(t, m_tile, n_tile);
      const int row = m_tile * kBM + 32 * q + lane;
      const int n0 = n_tile * kBN + cs;    // output column of sum[0]; sum[64 + j] is column n0 + 128 + j
      float sum[kSums];
#pragma unroll
      for (int j = 0; j < kSums; ++j) sum[j] = 0.f;
      // s_w[g][n0 .. n0 + 64) and s_w[g][n0 + 128 .. + 64): lanes 0-15 copy the
      // first, 16-31 the second, 16 bytes each; group g goes to slot g % kSwRing.
      auto fetch_sw = [&](int g) {
        const int n = n0 + (lane >> 4) * kHalf + 4 * (lane & 15);
        const bool v = g < groups && n < p.N;
        cp_async16(smem_u32(my_sw + (g % kSwRing) * kSums + 4 * lane),
                   v ? p.grp_scale + static_cast<size_t>(g) * p.N + n : p.grp_scale, v);
      };
#pragma unroll
      for (int g = 0; g < kSwRing - 1; ++g) fetch_sw(g);
      for (int g = 0; g < groups; ++g, ++gi) {
        __syncwarp();                          // every lane is done with slot (g - 1) % kSwRing
        fetch_sw(g + kSwRing - 1);             // ... which now receives group g + kSwRing - 1
        cp_async_wait_newest<kSwRing - 1>();   // this lane's copy of group g has landed
        __syncwarp();                          // and every other lane's
        const float4* sw4 = reinterpret_cast<const float4*>(my_sw + (g % kSwRing) * kSums);
        // group gi is complete when the commit after its second stage (stage
        // counter 2 gi + 1) arrives on that stage's barrier; that barrier cannot
        // run a phase past this wait, since its next phase needs group gi + 2,
        // which needs this accumulator back
        const uint32_t last = 2 * gi + 1;
        if (!mbar_wait(&empty[last % S], (last / S) & 1, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc_addr = lane_addr + (gi & 1) * kBN;
#pragma unroll
        for (int c = 0; c < 4; ++c) {            // 32-column loads: columns cs + 32 (c & 1) of half c >> 1
          const int h = c >> 1, hc = c & 1;
          uint32_t r[32];
          tmem_ld32(acc_addr + h * kHalf + 32 * hc, r);
          tmem_ld_wait(r);
          if (c == 3) release_acc(&afree[gi & 1], lane);  // the accumulator is free once read back
          if (DBG && row < p.M) {
            for (int j = 0; j < 32; ++j) {
              const int n = n0 + h * kHalf + 32 * hc + j;
              if (n < p.N) p.acc_dbg[(static_cast<size_t>(g) * p.M + row) * p.N + n] = __float2int_rn(__uint_as_float(r[j]));
            }
          }
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 s4 = sw4[h * (kCols / 4) + hc * 8 + j4];
            float* sm = sum + h * kCols + 32 * hc + 4 * j4;
            sm[0] = fmaf(s4.x, __uint_as_float(r[4 * j4]), sm[0]);
            sm[1] = fmaf(s4.y, __uint_as_float(r[4 * j4 + 1]), sm[1]);
            sm[2] = fmaf(s4.z, __uint_as_float(r[4 * j4 + 2]), sm[2]);
            sm[3] = fmaf(s4.w, __uint_as_float(r[4 * j4 + 3]), sm[3]);
          }
        }
        if (!ok) break;
      }
      cp_async_wait_all();  // no scale copy outlives the tile
      __syncwarp();
      if (!ok) break;
      const float sm = (row < p.M) ? p.row_scale[row] : 0.f;
#pragma unroll
      for (int c = 0; c < kSums / 32; ++c) {
        const int n = n0 + (c >> 1) * kHalf + (c & 1) * 32;  // warp-uniform
        if (n >= p.N) continue;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(sum[c * 32 + j], sm);
        if (p.Yf != nullptr) {
          epilogue_store32(p, row, n, v);
          continue;
        }
        if (row < p.M) epilogue_apply32(p, row, n, v);
        if (lane == 0) bulk_wait_read0();  // the previous box has been read out
        __syncwarp();
        stage_bf16x32(my_box, lane, v);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {  // rows >= M and columns >= N of the box are not written
          tma_store_2d(&tmY, my_box, n, row - lane);
          bulk_commit();
        }
      }
    }
    if (!ok) {
      set_error(p.err, SIXBIT_ETIMEOUT);
      *abort_flag = 1;
    }
    if (lane == 0) bulk_wait0();  // every output box has been written
    __syncwarp();
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// INT4 codes [N, K/2] -> fp16 [N, K] (exact); one thread per 16 code bytes.
__global__ void __launch_bounds__(256) w4_expand_kernel(const uint8_t* __restrict__ codes, int64_t nbytes,
                                                        uint16_t* __restrict__ out, const int32_t* mode_dev) {
  if (mode_dev != nullptr && SIXBIT_MODE_OF(*mode_dev) != SIXBIT_MODE_INT8) return;
  const int64_t n16 = nbytes >> 4;
  for (int64_t i = blockIdx.x * 256ll + threadIdx.x; i < n16; i += static_cast<int64_t>(gridDim.x) * 256) {
    const uint4 in = *reinterpret_cast<const uint4*>(codes + 16 * i);
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t o[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t byte = (w[j] >> (8 * b)) & 0xFFu;
        // nibble x -> fp16 0x64:(x ^ 8) = 1024 + (v + 8), v the signed value; minus 1032 -> v
        const uint32_t pair = (((byte & 0xFu) ^ 8u) | ((((byte >> 4) & 0xFu) ^ 8u) << 16)) | 0x64006400u;
        uint32_t d;
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(pair), "r"(0x64086408u));
        o[4 * j + b] = d;
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(out + 32 * i);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    dst[2] = make_uint4(o[8], o[9], o[10], o[11]);
    dst[3] = make_uint4(o[12], o[13], o[14], o[15]);
  }
}

}  // namespace w4a8

size_t w4a8_workspace_bytes(int N, int K) { return static_cast<size_t>(N) * static_cast<size_t>(K) * 2; }

cudaError_t launch_w4_expand(const uint8_t* codes, int N, int K, uint16_t* ws, const int32_t* mode_dev,
                             cudaStream_t st) {
  const int64_t nbytes = static_cast<int64_t>(N) * (K / 2);
  const int64_t want = ((nbytes >> 4) + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  const int grid = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
  w4a8::w4_expand_kernel<<<grid, 256, 0, st>>>(codes, nbytes, ws, mode_dev);
  note_launch();
  return cudaGetLastError();
}

template <bool DBG>
static cudaError_t launch_w4a8(const CUtensorMap& a_s8, const CUtensorMap& w_f16, const CUtensorMap& y,
                               const GemmParams& p, cudaStream_t st) {
  using namespace w4a8;
  cudaError_t e = set_smem_once<w4a8_kernel<DBG>>(kSmemBytes);
  if (e != cudaSuccess) return e;
  static ContextCache<int> regs_cache;
  int regs = 0;
  e = regs_cache.get(&regs, [](int* o) {
    cudaFuncAttributes fa;
    const cudaError_t r = cudaFuncGetAttributes(&fa, w4a8_kernel<DBG>);
    *o = fa.numRegs;
    return r;
  });
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits until the block's own registers cover the increase:
  // launch only with the register count the split was sized for.
  if (regs < kRegsLaunch || 4 * kRegsLow + 8 * kRegsHigh > 12 * regs) return cudaErrorInvalidConfiguration;
  const int ntiles = ((p.M + kBM - 1) / kBM) * ((p.N + kBN - 1) / kBN);
  const int sms = sm_count();
  const int grid = ntiles < sms ? ntiles : sms;
  w4a8_kernel<DBG><<<grid, kThreads, kSmemBytes, st>>>(a_s8, w_f16, y, p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_qgemm_w4a8(const CUtensorMap& a_s8, const CUtensorMap& w_f16, const CUtensorMap& y,
                              const GemmParams& p, cudaStream_t st) {
  return p.acc_dbg != nullptr ? launch_w4a8<true>(a_s8, w_f16, y, p, st) : launch_w4a8<false>(a_s8, w_f16, y, p, st);
}

}  // namespace sixbit
