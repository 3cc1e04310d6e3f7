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
// Operands.  The weights are expanded once per call (w4_expand_kernel: INT4
// -> fp16 into a caller-provided workspace of N*K*2 bytes, which stays in L2
// for the GEMM that follows) and reach the tensor core from shared memory
// (TMA, 128-byte swizzle).  The activation codes are read by the GEMM itself,
// one byte per element, and the A operand is held in tensor memory: four
// converter warps, one per 32-lane quarter, turn each thread's row of a
// stage's codes into 128 fp16 values (with u = q ^ 0x80, the fp16 bit pattern
// 0x64:u is 1152 + q, and one fp16 subtraction of 1152 leaves q exactly) and
// store them into the row's tensor-memory lane (column j holds k = 2j, 2j+1),
// from where the MMA reads A.  So shared memory carries only the weight tiles
// (their copies in, the tensor core's reads out), the codes (16 KB a stage)
// and the group scales; with the A operand in shared memory its writes and
// the tensor core's reads of it made the shared-memory port, not the tensor
// core, the limit.
//
// A persistent CTA per SM walks 128 x 192 output tiles in 128-K stages (one
// scale group each) through three rings: fp16 W tiles (three slots of 48 KB in
// shared memory, TMA, two 64-K halves a stage), s8 codes (three slots of
// 16 KB in shared memory, TMA with the 128-byte swizzle: chunk c of row r at
// chunk c ^ (r & 7), so a thread's reads of its own row are conflict-free)
// and fp16 A tiles (two slots of 64 columns in tensor memory).  A group's
// MMAs wait for its W slot (bytes landed), its A slot (four converter warps
// done) and its accumulator (eight fold warps done with group g - 2), and
// free the A slot and the W slot with one commit each; the W-slot commit is
// also the group's completion for the fold warps.  (Copying the codes per
// lane with cp.async instead cost the converter warps ~300 cycles a stage in
// issue stalls, measured.)
// Warps:
//   0       TMA producer: the fp16 W tile of each stage
//   1, 3    MMA issuers: one lane of warp 1 issues the even groups, one lane
//           of warp 3 the odd ones (tcgen05.mma issue blocks at the tensor
//           core's rate, so a single issuer's barrier waits and commits left
//           the tensor core idle ~45% of each group, measured with a clock64
//           trace; with two, each one's waits overlap the other's MMAs).
//           Warp 1 also allocates tensor memory.
//   2       TMA producer: the s8 code tile of each stage
//   4 - 7   converters: warp 4 + q converts rows 32 q .. 32 q + 31
//   8 - 15  fold + epilogue: warp 8 + e reads lanes 32 (e & 3) .. + 31 and
//           columns 96 (e >> 2) .. + 95 of each accumulator
// The CTA launches with 128 registers a thread; setmaxnreg gives warpgroup 0
// 40, the converters 80 and the fold warpgroups 192 (4 x 40 + 4 x 80 + 8 x 192
// = 2016 <= 16 x 128, and per SM sub-partition 40 + 80 + 2 x 192 = 504 <= 512):
// a fold thread's 96 running sums with three 16-column accumulator loads in
// flight fit.
//
// Tensor memory: two 192-column accumulators (columns 0 .. 191 and
// 256 .. 447; K groups alternate between them and the fold warps add
// s_w[g][n] * acc_g into registers while the next group accumulates) and the
// two 64-column A slots beside them (192 and 448).  Every mbarrier wait is
// bounded (2 s); on expiry the kernel records SIXBIT_ETIMEOUT, raises an abort
// flag for the other roles, waits (bounded) for its copies and tensor-core
// work in flight, frees tensor memory and returns.
#include <cstdint>

#include "common.cuh"
#include "ctx_cache.h"
#include "gemm_common.cuh"
#include "internal.h"

namespace sixbit {
namespace w4a8 {

constexpr int kBM = 128, kBN = 192;
constexpr int kKStage = 128;                         // K elements per stage: one scale group
constexpr int kStages = 3;                           // W ring (shared memory)
constexpr int kS8Stages = 3;                         // code ring (shared memory)
constexpr int kAStages = 2;                          // A ring (tensor memory)
constexpr int kBHalf = kBN * 64 * 2;                 // fp16 W tile of 64 K (128-byte rows, 128-byte swizzle), 24 KB
constexpr int kBTile = 2 * kBHalf;                   // a stage's two halves, 48 KB
constexpr int kS8Slot = kBM * kKStage;               // s8 codes of a stage, 16 KB (128-byte rows, 128-byte swizzle)
constexpr int kAccStride = 256;                      // tensor-memory columns between the two accumulators
constexpr int kAColsPerStage = kKStage / 2;          // fp16 pairs of a row's stage
// A slot a: the 64 columns after accumulator a (192 .. 255 and 448 .. 511)
__host__ __device__ constexpr int a_slot_col(int a) { return a * kAccStride + kBN; }
static_assert(kAStages == 2 && kBN + kAColsPerStage <= kAccStride && a_slot_col(1) + kAColsPerStage <= 512,
              "tensor memory columns");
constexpr int kConvWarp0 = 4, kFoldWarp0 = 8, kFoldWarps = 8, kThreads = 512;
constexpr int kCols = kBN / 2;                       // columns (and running sums) per fold thread
constexpr int kSwRing = 4;                           // groups of scales in flight per fold warp
constexpr int kSwLanes = kCols / 4;                  // lanes copying a group's scales (16 bytes each)
constexpr int kBoxBytes = 32 * 64;                   // one 32 x 32 bf16 output box
constexpr int kWarpArea = 2048;                      // a fold warp's scale ring, or its output box
static_assert(kSwRing * kCols * 4 <= kWarpArea && kBoxBytes <= kWarpArea, "fold warp area");
static_assert(kFoldWarps <= kBsMaxWarps, "block statistics: one partial per fold warp");
constexpr int kRegsLaunch = 128, kRegsLow = 40, kRegsConv = 80, kRegsHigh = 192;
static_assert(4 * kRegsLow + 4 * kRegsConv + 8 * kRegsHigh <= 16 * kRegsLaunch &&
                  kRegsLow + kRegsConv + 2 * kRegsHigh <= 4 * kRegsLaunch,
              "the register split must fit in what the CTA is launched with");
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(kBN >> 3) << 17) |
                            (static_cast<uint32_t>(kBM >> 4) << 24);  // f16 x f16 -> f32, M 128, N 192, K-major

// [W ring | code ring | fold warp areas | barriers].  A fold warp's
// output box is its scale ring: the ring is idle from the end of a tile's
// last group until the next tile's first scale copies, which wait for the
// box's last store to have been read out.
constexpr int kBarBytes = 512;
constexpr int kSmemBytes = kStages * kBTile + kS8Stages * kS8Slot + kFoldWarps * kWarpArea + 1024 + kBarBytes;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

// D[tmem] (+)= A[tmem] * B[smem]^T, fp16 inputs, fp32 accumulate (kind::f16).
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Each thread of the warp writes 32 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// fp16 pair (1152 + a, 1152 + b) -> (a, b): exact (both sides integers below 2048)
__device__ __forceinline__ uint32_t hsub1152(uint32_t x) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(0x64806480u));
  return d;
}

// 16 s8 codes -> 8 fp16 pairs (element order kept: pair i holds codes 2i, 2i + 1).
__device__ __forceinline__ void s8x16_to_f16x8(const uint4& in, uint32_t* o) {
  const uint32_t w[4] = {in.x ^ 0x80808080u, in.y ^ 0x80808080u, in.z ^ 0x80808080u, in.w ^ 0x80808080u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = hsub1152(__byte_perm(w[i], 0x64646464u, 0x4140));      // bytes 0, 1 -> 0x64:b0, 0x64:b1
    o[2 * i + 1] = hsub1152(__byte_perm(w[i], 0x64646464u, 0x4342));  // bytes 2, 3
  }
}

// DBG: write the exact group sums to p.acc_dbg.  BS: the residual epilogue
// also produces the block's statistics and Delta (p.bs_delta, p.bs_parts).
template <bool DBG, bool BS>
__global__ void __launch_bounds__(kThreads, 1)
    w4a8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmY, const GemmParams p) {
  if (p.mode_dev != nullptr && SIXBIT_MODE_OF(*p.mode_dev) != SIXBIT_MODE_INT8) return;
  constexpr int S = kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* s8_ring = smem + S * kBTile;
  uint8_t* fold_area = s8_ring + kS8Stages * kS8Slot;
  uint64_t* bars = reinterpret_cast<uint64_t*>(fold_area + kFoldWarps * kWarpArea);
  uint64_t* w_full = bars;                    // [S] W tile landed (the producer's expect-tx arrival + bytes)
  uint64_t* w_empty = bars + S;               // [S] the stage's MMAs are done with the W slot
  uint64_t* a_full = bars + 2 * S;            // [kAStages] the four converter warps stored the A tile
  uint64_t* a_empty = a_full + kAStages;      // [kAStages] the stage's MMAs are done with the A slot
  uint64_t* c_full = a_empty + kAStages;      // [kS8Stages] code tile landed
  uint64_t* c_empty = c_full + kS8Stages;     // [kS8Stages] the four converter warps read the code tile
  uint64_t* afree = c_empty + kS8Stages;      // [2] accumulator read back (eight fold warps)
  uint64_t* drain = afree + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert((2 * kStages + 2 * kAStages + 2 * kS8Stages + 3) * 8 + 8 <= kBarBytes, "barrier area");

  auto W_op = [&](int s) { return smem + s * kBTile; };

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
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], 1);
    }
    for (int a = 0; a < kAStages; ++a) {
      mbar_init(&a_full[a], 4);
      mbar_init(&a_empty[a], 1);
    }
    for (int c = 0; c < kS8Stages; ++c) {
      mbar_init(&c_full[c], 1);
      mbar_init(&c_empty[c], 4);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&afree[b], kFoldWarps);
    mbar_init(drain, 2);
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

  if (warp < kConvWarp0) {
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
            if (it >= S && !mbar_wait(&w_empty[s], ((it / S) - 1) & 1, abort_flag, p.wait_ns)) {
              ok = false;
              break;
            }
            if (p.withhold_first && it == 0) continue;  // failure-path test: stage 0 never lands
            mbar_expect_tx(&w_full[s], kBTile);
            tma_load_2d(W_op(s), &tmW, &w_full[s], kb * kKStage, n_tile * kBN);
            tma_load_2d(W_op(s) + kBHalf, &tmW, &w_full[s], kb * kKStage + 64, n_tile * kBN);
          }
        }
        if (!ok) {
          set_error(p.err, SIXBIT_ETIMEOUT);
          *abort_flag = 1;
        }
        // every copy this warp started lands before it can exit
        for (uint32_t j = (it > S ? it - S : 0); j < it; ++j)
          (void)mbar_wait(&w_full[j % S], (j / S) & 1, nullptr, p.wait_ns);
      }
    } else if (warp == 1 || warp == 3) {
      if (lane == 0) {
        // ------------------------------------------------------- MMA issuers --
        // Group counter gi runs across tiles; group gi accumulates into
        // buffer gi & 1, reads A slot gi & 1 and W slot gi % S.  Warp 1's
        // lane issues the even groups, warp 3's the odd ones, each waiting
        // for its own group's operands and accumulator: tcgen05.mma issue
        // blocks at the tensor core's rate, so one issuer's waits and
        // commits leave the tensor core idle, while with two each one's
        // waits overlap the other's MMAs.  A commit tracks only its own
        // thread's MMAs, which is the group's.
        const uint32_t par = warp == 1 ? 0u : 1u;
        uint32_t gi = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
          for (int g = 0; g < groups; ++g, ++gi) {
            if ((gi & 1) != par) continue;
            const int a = static_cast<int>(par), s = static_cast<int>(gi % S);
            if ((gi >= 2 && !mbar_wait(&afree[a], ((gi >> 1) - 1) & 1, abort_flag, p.wait_ns)) ||
                !mbar_wait(&w_full[s], (gi / S) & 1, abort_flag, p.wait_ns) ||
                !mbar_wait(&a_full[a], (gi >> 1) & 1, abort_flag, p.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + par * kAccStride;
            const uint32_t a_tmem = tmem + a_slot_col(a), b_base = smem_u32(W_op(s));
#pragma unroll
            for (int k = 0; k < kKStage / 16; ++k)  // k < 4 from the first 64-K half of the W tile, then the second
              mma_f16_tmem_a(d_tmem, a_tmem + 8 * k, sdesc_sw128(b_base + (k >> 2) * kBHalf + 32 * (k & 3)), kIdesc,
                             k == 0 ? 0u : 1u);
            tc_commit(&a_empty[a]);
            tc_commit(&w_empty[s]);  // frees the W slot; also the group's completion
          }
        }
        if (!ok) {
          set_error(p.err, SIXBIT_ETIMEOUT);
          *abort_flag = 1;
        }
        tc_commit(drain);  // all tensor-core work issued here completes before exit (count 2: both issuers)
        (void)mbar_wait(drain, 0, nullptr, p.wait_ns);
      }
    } else if (warp == 2) {
      if (lane == 0) {
        // ----------------------------------------------------- code producer --
        uint32_t j = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
          int m_tile, n_tile;
          tile_of(t, m_tile, n_tile);
          for (int kb = 0; kb < nk; ++kb, ++j) {
            const int c = j % kS8Stages;
            if (j >= kS8Stages && !mbar_wait(&c_empty[c], ((j / kS8Stages) - 1) & 1, abort_flag, p.wait_ns)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&c_full[c], kS8Slot);
            tma_load_2d(s8_ring + c * kS8Slot, &tmA, &c_full[c], kb * kKStage, m_tile * kBM);
          }
        }
        if (!ok) {
          set_error(p.err, SIXBIT_ETIMEOUT);
          *abort_flag = 1;
        }
        // every copy this warp started lands before it can exit
        for (uint32_t jj = (j > kS8Stages ? j - kS8Stages : 0); jj < j; ++jj)
          (void)mbar_wait(&c_full[jj % kS8Stages], (jj / kS8Stages) & 1, nullptr, p.wait_ns);
      }
    }
  } else if (warp < kFoldWarp0) {
    setmaxnreg_dec<kRegsConv>();
    // ------------------------------------------------------------ converters --
    // Warp 4 + q converts rows 32 q .. 32 q + 31 of every stage; thread
    // `lane` converts row 32 q + lane, the row of its tensor-memory lane.
    // Per stage: wait for the code tile, read the row's eight chunks, release
    // the slot, wait for the A slot, convert and store 64 columns (two halves
    // of 32, through one set of registers), arrive.  The
    // release comes after every lane's reads have returned (each lane's value
    // of `zero` needs them) and each lane's proxy fence: the refill is an
    // async-proxy write after these generic-proxy reads, and without the
    // fence such refills overwrote codes still being read (measured: wrong
    // group sums in every stage whose slot was refilled).
    const int q = warp & 3;
    const int myrow = 32 * q + lane;
    const uint32_t rd_off = static_cast<uint32_t>(myrow * 128);
    const int swz = myrow & 7;  // 128-byte swizzle: chunk c of row r at chunk c ^ (r & 7)
    uint32_t it = 0;
    int r_slot = 0;  // code ring slot of stage it
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int a = it % kAStages;
        if (!mbar_wait(&c_full[r_slot], (it / kS8Stages) & 1, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        const uint8_t* row = s8_ring + r_slot * kS8Slot + rd_off;
        uint4 in[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) in[c] = *reinterpret_cast<const uint4*>(row + ((c ^ swz) << 4));
        uint32_t zero;
        asm volatile("and.b32 %0, %1, 0;"
                     : "=r"(zero)
                     : "r"(in[0].x ^ in[1].x ^ in[2].x ^ in[3].x ^ in[4].x ^ in[5].x ^ in[6].x ^ in[7].x));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c_empty[r_slot]);
        r_slot = r_slot + 1 == kS8Stages ? 0 : r_slot + 1;
        if (it >= kAStages && !mbar_wait(&a_empty[a], ((it / kAStages) - 1) & 1, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acol = tmem + (static_cast<uint32_t>(32 * q) << 16) + a_slot_col(a);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) s8x16_to_f16x8(in[4 * h + c], v + 8 * c);
          tmem_st32(acol + 32 * h, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[a]);
      }
    }
    if (!ok && lane == 0) {
      set_error(p.err, SIXBIT_ETIMEOUT);
      *abort_flag = 1;
    }
  } else {
    setmaxnreg_inc<kRegsHigh>();  // each fold warpgroup, one instruction
    // -------------------------------------------------------- fold + epilogue --
    const int ew = warp - kFoldWarp0;      // 0 .. 7
    const int q = warp & 3;                // tensor-memory lane quarter this warp may read
    const int cs = (ew >> 2) * kCols;      // first column of this thread within the tile
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q) << 16) + cs;
    float* my_sw = reinterpret_cast<float*>(fold_area + ew * kWarpArea);  // [slot][96]
    uint8_t* my_box = fold_area + ew * kWarpArea;                          // the same bytes
    uint32_t gi = 0;
    bool ok = true;
    BsAcc bs = bs_zero();
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      int m_tile, n_tile;
      tile_of(t, m_tile, n_tile);
      const int row = m_tile * kBM + 32 * q + lane;
      const int n0 = n_tile * kBN + cs;    // output column of sum[0]
      // The epilogue's residual rows to L2 while the tile's groups run: from
      // HBM its loads kept the epilogue waiting ~1.5 us a 32-column chunk
      // (clock64 trace: ~9600 cycles for a tile's residual epilogue, against
      // the ~2700 the MMAs can run ahead), 465 -> 458 us at 17776 x 1920 x
      // 7680.  (The same prefetch issued inside the group loop cost more
      // than it saved.)
      if constexpr (!BS)
        if (p.epilogue == SIXBIT_EPI_RESIDUAL && row < p.M && n0 < p.N)
          residual_prefetch(p, row, n0, min(kCols, p.N - n0));
      float sum[kCols];
#pragma unroll
      for (int j = 0; j < kCols; ++j) sum[j] = 0.f;
      // s_w[g][n0 .. n0 + 96): lanes 0 .. 23 copy 16 bytes each; group g goes
      // to slot g % kSwRing.
      auto fetch_sw = [&](int g) {
        if (lane < kSwLanes) {
          const int n = n0 + 4 * lane;
          const bool v = g < groups && n < p.N;
          cp_async16(smem_u32(my_sw + (g % kSwRing) * kCols + 4 * lane),
                     v ? p.grp_scale + static_cast<size_t>(g) * p.N + n : p.grp_scale, v);
        }
      };
      if (lane == 0) bulk_wait_read0();  // the ring doubled as the last tile's output box
      __syncwarp();
#pragma unroll
      for (int g = 0; g < kSwRing - 1; ++g) fetch_sw(g);
      for (int g = 0; g < groups; ++g, ++gi) {
        __syncwarp();                          // every lane is done with slot (g - 1) % kSwRing
        fetch_sw(g + kSwRing - 1);             // ... which now receives group g + kSwRing - 1
        cp_async_wait_newest<kSwRing - 1>();   // this lane's copy of group g has landed
        __syncwarp();                          // and every other lane's
        const float4* sw4 = reinterpret_cast<const float4*>(my_sw + (g % kSwRing) * kCols);
        if constexpr (BS)  // the epilogue's residual and Delta_prev, to L2 a few groups ahead
          if (g == (groups > 4 ? groups - 4 : 0) && row < p.M && n0 < p.N) bs_prefetch(p, row, n0, min(kCols, p.N - n0));
        // group gi is complete when its commit arrives on its stage's W-slot
        // barrier; that barrier cannot run a phase past this wait, since its
        // next phase is group gi + 3, which needs buffer (gi + 1) & 1 back
        if (!mbar_wait(&w_empty[gi % S], (gi / S) & 1, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc_addr = lane_addr + (gi & 1) * kAccStride;
        // Six 16-column chunks, three loads in flight: chunks 0-2 are loaded
        // together, and chunk c + 3 is loaded as soon as chunk c is folded,
        // so the buffer goes back to the MMA thread two load latencies after
        // the group completes (the MMA of group gi + 2 waits for it) instead
        // of one per chunk.
        auto fold16 = [&](int c, const uint32_t (&r)[16]) {
          if (DBG && row < p.M) {
            for (int j = 0; j < 16; ++j) {
              const int n = n0 + 16 * c + j;
              if (n < p.N) p.acc_dbg[(static_cast<size_t>(g) * p.M + row) * p.N + n] = __float2int_rn(__uint_as_float(r[j]));
            }
          }
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const float4 s4 = sw4[c * 4 + j4];
            float* sm = sum + 16 * c + 4 * j4;
            sm[0] = fmaf(s4.x, __uint_as_float(r[4 * j4]), sm[0]);
            sm[1] = fmaf(s4.y, __uint_as_float(r[4 * j4 + 1]), sm[1]);
            sm[2] = fmaf(s4.z, __uint_as_float(r[4 * j4 + 2]), sm[2]);
            sm[3] = fmaf(s4.w, __uint_as_float(r[4 * j4 + 3]), sm[3]);
          }
        };
        static_assert(kCols == 96, "six 16-column chunks");
        uint32_t r0[16], r1[16], r2[16];
        tmem_ld16(acc_addr, r0);
        tmem_ld16(acc_addr + 16, r1);
        tmem_ld16(acc_addr + 32, r2);
        tmem_ld_wait(r0);
        tmem_ld_wait(r1);   // (no load outstanding: ties the registers to the wait)
        tmem_ld_wait(r2);
        fold16(0, r0);
        tmem_ld16(acc_addr + 48, r0);
        fold16(1, r1);
        tmem_ld16(acc_addr + 64, r1);
        fold16(2, r2);
        tmem_ld16(acc_addr + 80, r2);
        tmem_ld_wait(r0);
        tmem_ld_wait(r1);
        tmem_ld_wait(r2);
        release_acc(&afree[gi & 1], lane);  // the accumulator is free once read back
        fold16(3, r0);
        fold16(4, r1);
        fold16(5, r2);
        if (!ok) break;
      }
      cp_async_wait_all();  // no scale copy outlives the tile
      __syncwarp();
      if (!ok) break;
      const float sm = (row < p.M) ? p.row_scale[row] : 0.f;
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c) {
        const int n = n0 + 32 * c;  // warp-uniform
        if (n >= p.N) continue;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(sum[c * 32 + j], sm);
        if (p.Yf != nullptr) {
          epilogue_store32(p, row, n, v);
          continue;
        }
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
      }
    }
    if constexpr (BS) bs_flush(p, bs, ew, kFoldWarps, lane);
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

// INT4 codes [N, K/2] -> fp16 [N, K] (exact).  A warp converts 512 code
// bytes an iteration: lane t takes the 4-byte words t, t + 32, t + 64 and
// t + 96 of the chunk (each load instruction reads 128 contiguous bytes) and
// writes each word's 8 fp16 values as one 16-byte store (each store
// instruction writes 512 contiguous bytes); nbytes % 4 == 0.
__device__ __forceinline__ uint4 w4_word_to_f16x8(uint32_t w) {
  uint32_t o[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t byte = (w >> (8 * b)) & 0xFFu;
    // nibble x -> fp16 0x64:(x ^ 8) = 1024 + (v + 8), v the signed value; minus 1032 -> v
    const uint32_t pair = (((byte & 0xFu) ^ 8u) | ((((byte >> 4) & 0xFu) ^ 8u) << 16)) | 0x64006400u;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[b]) : "r"(pair), "r"(0x64086408u));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(256) w4_expand_kernel(const uint8_t* __restrict__ codes, int64_t nbytes,
                                                        uint16_t* __restrict__ out, const int32_t* mode_dev) {
  if (mode_dev != nullptr && SIXBIT_MODE_OF(*mode_dev) != SIXBIT_MODE_INT8) return;
  const int64_t nwords = nbytes >> 2;
  const uint32_t* in = reinterpret_cast<const uint32_t*>(codes);
  uint4* dst = reinterpret_cast<uint4*>(out);
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t c = (blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5)) * 128; c < nwords;
       c += warps * 128) {
    uint32_t w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t k = c + 32 * u + lane;
      w[u] = k < nwords ? __ldg(in + k) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t k = c + 32 * u + lane;
      if (k < nwords) dst[k] = w4_word_to_f16x8(w[u]);
    }
  }
}

}  // namespace w4a8

size_t w4a8_workspace_bytes(int N, int K) { return static_cast<size_t>(N) * static_cast<size_t>(K) * 2; }

cudaError_t launch_w4_expand(const uint8_t* codes, int N, int K, uint16_t* ws, const int32_t* mode_dev,
                             cudaStream_t st) {
  const int64_t nbytes = static_cast<int64_t>(N) * (K / 2);  // K % 128 == 0: a multiple of 64
  const int64_t want = ((nbytes >> 2) + 1023) / 1024;       // 8 warps x 128 words a CTA iteration
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  const int grid = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
  w4a8::w4_expand_kernel<<<grid, 256, 0, st>>>(codes, nbytes, ws, mode_dev);
  note_launch();
  return cudaGetLastError();
}

template <bool DBG, bool BS>
static cudaError_t launch_w4a8(const CUtensorMap& a_s8, const CUtensorMap& w_f16, const CUtensorMap& y,
                               const GemmParams& p, cudaStream_t st) {
  using namespace w4a8;
  cudaError_t e = set_smem_once<w4a8_kernel<DBG, BS>>(kSmemBytes);
  if (e != cudaSuccess) return e;
  static ContextCache<int> regs_cache;
  int regs = 0;
  e = regs_cache.get(&regs, [](int* o) {
    cudaFuncAttributes fa;
    const cudaError_t r = cudaFuncGetAttributes(&fa, w4a8_kernel<DBG, BS>);
    *o = fa.numRegs;
    return r;
  });
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits until the block's own registers cover the increase:
  // launch only with the register count the split was sized for.
  if (regs < kRegsLaunch || 4 * (kRegsLow + kRegsConv) + 8 * kRegsHigh > 16 * regs) return cudaErrorInvalidConfiguration;
  const int ntiles = ((p.M + kBM - 1) / kBM) * ((p.N + kBN - 1) / kBN);
  const int sms = sm_count();
  const int grid = ntiles < sms ? ntiles : sms;
  w4a8_kernel<DBG, BS><<<grid, kThreads, kSmemBytes, st>>>(a_s8, w_f16, y, p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_qgemm_w4a8(const CUtensorMap& a_s8, const CUtensorMap& w_f16, const CUtensorMap& y,
                              const GemmParams& p, cudaStream_t st) {
  if (p.acc_dbg != nullptr) return launch_w4a8<true, false>(a_s8, w_f16, y, p, st);
  return p.bs_delta != nullptr ? launch_w4a8<false, true>(a_s8, w_f16, y, p, st)
                               : launch_w4a8<false, false>(a_s8, w_f16, y, p, st);
}

}  // namespace sixbit
