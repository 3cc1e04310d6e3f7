/*
 * libsixbit -- C ABI of the dynamically quantized linear layer of a video
 * diffusion transformer ("6Bit-Diffusion: Inference-Time Mixed-Precision
 * Quantization for Video Diffusion Models"), for one NVIDIA GB300 (sm_103a).
 *
 * Conventions for every call:
 *  - Tensor pointers are DEVICE pointers, allocated and owned by the caller.
 *    The library never allocates or frees device memory.
 *  - bf16 tensors are passed as uint16_t bit patterns, row-major, densely
 *    packed (row stride = number of columns).
 *  - Every call enqueues its kernels on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and returns without waiting for them.
 *  - Argument errors are detected on the host before anything is enqueued
 *    and returned as a sixbit_status; nothing is launched in that case.
 *  - Device-side errors (a bounded wait that ran out, an out-of-range
 *    index caught by a check) are recorded in the caller-supplied device word
 *    `err_dev` (may be NULL to ignore them) as a SIXBIT_E* code; the first
 *    error wins.  sixbit_check() synchronizes the stream and decodes it.
 *  - "mode" arguments: when `mode_dev` is non-NULL the device word it points
 *    to (written by sixbit_policy_step) selects the mode at run time and a
 *    kernel whose mode does not match returns at once; when it is NULL the
 *    host value `mode` is used.
 */
#ifndef SIXBIT_H
#define SIXBIT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int sixbit_status;
enum {
  SIXBIT_OK = 0,
  SIXBIT_EINVAL = 1,       /* NULL pointer or bad enum value */
  SIXBIT_ESHAPE = 2,       /* a size violates the documented constraints */
  SIXBIT_EALIGN = 3,       /* a pointer is not 16-byte aligned */
  SIXBIT_EUNSUPPORTED = 4, /* no GPU of compute capability 10.3 */
  SIXBIT_ECUDA = 5,        /* a CUDA runtime call failed */
  SIXBIT_ETIMEOUT = 6,     /* a device-side bounded wait ran out */
  SIXBIT_EDEVICE = 7       /* a device-side check failed */
};

/* Per-block precision decision (low byte of the mode word) and flags. */
enum {
  SIXBIT_MODE_NVFP4 = 1, /* stable block: NVFP4 activations, W4A4 GEMM */
  SIXBIT_MODE_INT8 = 2,  /* volatile block: INT8 activations, W4A8 GEMM */
  SIXBIT_MODE_BF16 = 3,  /* PDR: full-precision recompute */
  SIXBIT_MODE_SKIP = 4   /* TDC: output = input + cached delta */
};
#define SIXBIT_MODE_OF(w) ((w)&0xFF)
enum {
  SIXBIT_FLAG_REFRESH = 1 << 8,   /* error accumulator forced a compute */
  SIXBIT_FLAG_PDR = 1 << 9,       /* outlier ratio forced BF16 */
  SIXBIT_FLAG_POSTSKIP = 1 << 10, /* INT8 because the previous step skipped */
  SIXBIT_FLAG_NEAR = 1 << 11      /* a deciding statistic was within near_rel of its threshold */
};

enum { SIXBIT_EPI_NONE = 0, SIXBIT_EPI_GELU = 1, SIXBIT_EPI_RESIDUAL = 2 };

/*
 * Quantized activations (output of sixbit_hadamard_quant, A operand of
 * sixbit_qgemm).  M tokens x K channels.  Fields of the mode not produced may
 * be NULL.
 *
 * NVFP4 (technical summary section 2.A; popular summary section 1):
 *   fp4_codes    [M, K/2] bytes, two E2M1 codes per byte, even k in the low nibble
 *   fp4_scales   E4M3 block scales, one per 16 elements, in the tiled layout
 *                of sixbit_fp4_scale_offset(); sixbit_fp4_scale_bytes(M, K) bytes
 *   tensor_amax  [1] float: max |y| of the rotated tensor (written by the call
 *                unless an amax is supplied)
 *   tensor_scale [1] float: s_t = amax / 2688 (1 when amax == 0)
 * INT8 (technical summary section 2.A):
 *   i8_codes     [M, K] int8, symmetric, per token, in [-127, 127] (the A
 *                operand of the W4A8 GEMM)
 *   row_scale    [M] float: s_m = row amax / 127
 * Debug:
 *   rotated      [M, K] float, the rotated FP32 activations (optional)
 */
typedef struct {
  uint8_t* fp4_codes;
  uint8_t* fp4_scales;
  float* tensor_amax;
  float* tensor_scale;
  int8_t* i8_codes;
  float* row_scale;
  float* rotated;
} sixbit_qact;

/*
 * Packed weights of one linear layer, W [N, K] (output channels x input
 * channels), produced by sixbit_pack_weights.  The 4-bit forms are of the
 * rotated weight W' = W . blockdiag(H_b / sqrt(b)); the bf16 form is unrotated.
 *   fp4_codes        [N, K/2], fp4_scales (tiled, sixbit_fp4_scale_bytes(N, K)),
 *   fp4_amax [1], fp4_tensor_scale [1]           -- NVFP4, static tensor scale
 *   i4_codes         [N, K/2] two's-complement nibbles in [-7, 7], even k low
 *   i4_scales        [K/128, N] float (group-major): s[g][n] = amax / 7
 *   bf16_w           [N, K] bf16(W)
 * (about 3.1 bytes per weight: 0.5625 NVFP4, 0.53 INT4 with scales, 2 bf16).
 */
typedef struct {
  uint8_t* fp4_codes;
  uint8_t* fp4_scales;
  float* fp4_amax;
  float* fp4_tensor_scale;
  uint8_t* i4_codes;
  float* i4_scales;
  uint16_t* bf16_w;
} sixbit_weights;

/*
 * Statistics of one computed block step (sixbit_block_stats) -- float64 sums
 * over the whole [T, H] block tensor, Delta = bf16(x_out - x_in):
 * sum_d2 = sum Delta^2, sum_xin2 = sum x_in^2, sum_ddp = sum Delta*Delta_prev,
 * sum_dp2 = sum Delta_prev^2, then the block OUTPUT's max |x|, sum |x| and
 * element count, which are the next block's input statistics.  The three
 * output fields are laid out like sixbit_tensor_stats' first three, so
 * &stats->max_abs_out can be passed as a policy `in_stats`.
 */
typedef struct {
  double sum_d2;
  double sum_xin2;
  double sum_ddp;
  double sum_dp2;
  double max_abs_out;
  double sum_abs_out;
  double count;
  double reserved;
} sixbit_stats;

/* Policy thresholds (technical summary sections 2.A-2.C; popular summary sections 1-3). */
typedef struct {
  double gamma_thr;   /* Gamma >= gamma_thr (or NaN) -> INT8, else NVFP4 */
  double cos_thr;     /* cos(Delta_{t-1}, Delta_{t-2}) >= cos_thr may skip */
  double err_cap;     /* accumulated 1 - cos above err_cap forces a refresh */
  double pdr_ratio;   /* input max/mean above pdr_ratio (or NaN) forces BF16 */
  double near_rel;    /* relative band around thresholds reported as "near" */
  int32_t refresh_bf16; /* 1: every forced refresh runs BF16 */
  int32_t reserved;
} sixbit_policy_cfg;

/* Per-block policy state; zero-initialise before the first step. */
typedef struct {
  int32_t n_computed;
  int32_t skipped_last;
  int32_t have_gamma;
  int32_t pending;      /* the last decision computed; fold its stats next step */
  double gamma;
  double cos;
  double acc;
  int32_t last_word;
  int32_t steps;
  int32_t n_skip, n_refresh, n_pdr, n_near, n_nvfp4, n_int8, n_bf16;
  int32_t n_nonfinite;  /* decisions taken on a statistic that was not a number
                           (a NaN cosine never skips, a NaN Gamma picks INT8,
                           a NaN input ratio picks BF16) */
} sixbit_policy_state;

/* ---- sizes and layouts ------------------------------------------------- */

/* Bytes of a tiled E4M3 scale array for `rows` x K elements (K % 64 == 0):
 * rows rounded up to 128, times K/16. */
size_t sixbit_fp4_scale_bytes(int rows, int K);
/* Byte offset of the scale of row r, 16-element block kb in the tiled layout:
 * (r/128)*(128*K/16) + (kb/4)*512 + (r%32)*16 + ((r/32)%4)*4 + kb%4.  Each
 * 512-byte chunk holds 128 rows x 4 blocks, the unit the GEMM's scale copy
 * into tensor memory consumes. */
size_t sixbit_fp4_scale_offset(int r, int kb, int K);
/* Scratch bytes sixbit_tensor_stats / sixbit_block_stats / sixbit_skip_apply
 * need for `n` elements (per-CTA partial sums and a completion counter). */
size_t sixbit_stats_scratch_bytes(int64_t n);

/* ---- the hot path ------------------------------------------------------ */

/*
 * Offline weight preparation (technical summary section 4: 4-bit weights,
 * W4A6/W4A8).  W: [N, K] float32.  had_block b in {16, 64, 256}, K % 128 == 0,
 * K % b == 0.  Rotates W with the same FP32 butterfly as the activations, then
 * quantizes W' to NVFP4 (two-level, static tensor scale) and to INT4
 * (symmetric, groups of 128 along K), and rounds W to bf16.  Every field of
 * `out` must be non-NULL.
 */
sixbit_status sixbit_pack_weights(const float* W, int N, int K, int had_block,
                                  const sixbit_weights* out, int32_t* err_dev, void* stream);

/*
 * Online block-Hadamard rotation fused with dynamic quantization (technical
 * summary section 2.A; popular summary section 1): y = x . blockdiag(H_b/sqrt b)
 * by a fixed-order FP32 butterfly, then NVFP4 (mode 1) or INT8 (mode 2).
 * X: [M, K] bf16; K % 128 == 0; b in {16, 64, 256}.  In NVFP4 mode the tensor
 * amax is taken from `tamax_in` (a device float, e.g. from the producer of X)
 * or, when it is NULL, computed by a first pass into out->tensor_amax.  Other
 * modes (BF16, SKIP) enqueue nothing when mode_dev is NULL and return at once
 * on the device otherwise.
 */
sixbit_status sixbit_hadamard_quant(const uint16_t* X, int M, int K, int had_block, int mode,
                                    const int32_t* mode_dev, const float* tamax_in,
                                    const sixbit_qact* out, int32_t* err_dev, void* stream);

/*
 * Quantized GEMM with fused epilogue (technical summary sections 2.A, 2.C, 4):
 *   NVFP4: Y = s_tx * s_tw * sum_k (E2M1*E4M3)_x (E2M1*E4M3)_w   (A = qact, W fp4)
 *   INT8 : Y = s_m * sum_g s_w[g] * acc_g, acc_g exact integer sums over
 *          128-wide K groups (A = qact i8_codes / row_scale, W i4_codes /
 *          i4_scales)
 *   BF16 : Y = X_bf16 . bf16(W)^T  (A = X_bf16 unrotated, W bf16_w)
 * then epilogue NONE, GELU (exact erf) or RESIDUAL (+ residual [M, N] bf16),
 * rounded to bf16 into Y [M, N] -- or, when Y_f32 is non-NULL, written as
 * float32 without the bf16 rounding (Y may then be NULL).  Accumulation is on
 * the tensor cores in FP32 (tcgen05, accumulators in tensor memory).
 * Constraints: K % 128 == 0, N % 16 == 0, M >= 1.  acc_dbg (INT8 only,
 * optional): receives the exact group accumulators as int32 [K/128][M][N].
 * workspace: device memory of sixbit_qgemm_workspace_bytes(N, K) bytes,
 * 16-byte aligned, required whenever the INT8 kind may run (mode INT8, or
 * mode_dev non-NULL), else may be NULL: the INT8 call expands the INT4
 * weights into it (as fp16) before its GEMM reads them; its contents are
 * scratch and are not preserved.
 */
sixbit_status sixbit_qgemm(const sixbit_qact* A, const uint16_t* X_bf16, const sixbit_weights* W,
                           int M, int N, int K, int mode, const int32_t* mode_dev, int epilogue,
                           const uint16_t* residual, uint16_t* Y, float* Y_f32, int32_t* acc_dbg,
                           void* workspace, int32_t* err_dev, void* stream);

/* Bytes of the workspace sixbit_qgemm's INT8 kind needs for an [N, K] weight. */
size_t sixbit_qgemm_workspace_bytes(int N, int K);

/*
 * The NVFP4 sixbit_qgemm (bf16 output Y) whose epilogue also takes the first
 * pass of the NVFP4 quantization of Y (technical summary section 4: the
 * quantization fused with the kernels around it): *amax_out = max |y| over
 * y = bf16(Y) . blockdiag(H_b / sqrt b), by the quantizer's own butterfly, so
 * it equals the amax pass of sixbit_hadamard_quant(Y, b, NVFP4) and can be
 * passed to it as tamax_in.  had_block in {16, 64}; N % 128 == 0; amax_out a
 * device float (zeroed by the call).  With mode_dev, the kernel runs (and
 * amax_out is written) only when the mode word is NVFP4.
 */
sixbit_status sixbit_qgemm_rotamax(const sixbit_qact* A, const sixbit_weights* W, int M, int N, int K,
                                   const int32_t* mode_dev, int epilogue, const uint16_t* residual, uint16_t* Y,
                                   int had_block, float* amax_out, int32_t* err_dev, void* stream);

/*
 * sixbit_qgemm with the RESIDUAL epilogue (Y = bf16(A.W^T + residual), bf16
 * Y required) whose epilogue also does the block statistics pass of
 * sixbit_block_stats for x_in = residual and x_out = Y (technical summary
 * sections 2.A-2.B; popular summary sections 3-4: the statistics fused into
 * the kernel that produces the block output): delta_cache [M*N] bf16 holds
 * Delta_prev on entry and Delta = bf16(f32(x_out) - f32(x_in)) on return,
 * exactly as sixbit_block_stats writes it, and the sums go as partial rows
 * to parts (device memory of sixbit_blockstats_parts_bytes() bytes, 16-byte
 * aligned; written whole by the call, no initial contents needed), to be
 * folded by sixbit_block_stats_parts or sixbit_dit_block_end_parts.  The
 * partial rows are a fixed function of the launch, so the folded sums are
 * run-to-run deterministic; they equal sixbit_block_stats's up to the order
 * of the float-float additions (about 1e-7 relative, Kahan sums; 1e-12,
 * TwoSum sums), while Delta and Y are bit-identical.  Other arguments,
 * constraints and mode gating as for sixbit_qgemm.
 */
sixbit_status sixbit_qgemm_blockstats(const sixbit_qact* A, const uint16_t* X_bf16, const sixbit_weights* W, int M,
                                      int N, int K, int mode, const int32_t* mode_dev, const uint16_t* residual,
                                      uint16_t* Y, uint16_t* delta_cache, void* parts, void* workspace,
                                      int32_t* err_dev, void* stream);

/* Bytes of sixbit_qgemm_blockstats's parts buffer on the current device (0 on error). */
size_t sixbit_blockstats_parts_bytes(void);

/*
 * Folds the partial rows of a sixbit_qgemm_blockstats call into stats_dev
 * (the sums of sixbit_stats, count = n = M*N).  One CTA on `stream`, which
 * must order it after the GEMM.
 */
sixbit_status sixbit_block_stats_parts(const void* parts, int64_t n, sixbit_stats* stats_dev, int32_t* err_dev,
                                       void* stream);

/*
 * Block statistics and delta cache update for a computed block step
 * (technical summary sections 2.A-2.C; popular summary sections 1-3):
 * Delta = bf16(f32(x_out) - f32(x_in)) overwrites delta_cache (which holds
 * Delta_prev on entry; zero it before the first step), and stats_dev receives
 * the sums of sixbit_stats.  n = T*H elements, n % 8 == 0.  With mode_dev
 * non-NULL and the mode SKIP, nothing is done.  scratch: device memory of
 * sixbit_stats_scratch_bytes(n) bytes whose completion counter is zero on
 * entry (zero it once; every call leaves it zero again).
 */
sixbit_status sixbit_block_stats(const uint16_t* x_in, const uint16_t* x_out, uint16_t* delta_cache,
                                 int64_t n, const int32_t* mode_dev, sixbit_stats* stats_dev,
                                 void* scratch, int32_t* err_dev, void* stream);

/*
 * Per-block decision for this step (technical summary sections 2.A-2.C;
 * popular summary sections 1-3), one device thread.  If the previous decision
 * computed, its statistics (last_stats_dev) are folded first: Gamma =
 * sqrt(sum_d2)/sqrt(sum_xin2), cos = sum_ddp/sqrt(sum_d2*sum_dp2).  Then:
 * skip if at least two computes happened, cos >= cos_thr and
 * acc + (1 - cos) <= err_cap (acc += 1 - cos); else compute in BF16 if the
 * input ratio max/mean > pdr_ratio, INT8 after a skip or before any Gamma,
 * else INT8 if Gamma >= gamma_thr, else NVFP4.  in_stats_dev points to
 * {max |x_in|, sum |x_in|, count} (float64).  The decision word goes to
 * mode_dev[0].  cfg is a HOST pointer.
 */
sixbit_status sixbit_policy_step(const sixbit_policy_cfg* cfg, sixbit_policy_state* state_dev,
                                 const sixbit_stats* last_stats_dev, const double* in_stats_dev,
                                 int32_t* mode_dev, int32_t* err_dev, void* stream);

/*
 * The per-block device state of a stack of L residual blocks evaluated in
 * order, block l reading x_{l-1} (x_{-1} = x0) and writing x_l into
 * buf[l % 2].  All pointers are DEVICE pointers owned by the caller.
 *   states [L], stats [L], modes [L]  as for sixbit_policy_step, one per block
 *   run_len [L] uint32, zero before the first step (the library leaves
 *               it zero between steps)
 *   in_stats0   [4] float64, written by sixbit_dit_begin: {max |x0|,
 *               sum |x0|, count, sum x0^2}
 *   x0 [n], buf[0], buf[1] [n] bf16
 *   deltas      the Delta cache, one slice of n elements per block, in
 *               delta_format: SIXBIT_DELTA_BF16, [L][n] bf16; or
 *               SIXBIT_DELTA_MXFP8, [L][n] E4M3 codes with delta_scales
 *               [L][n / 32] E8M0 codes (see sixbit_block_stats_mxfp8)
 *   delta_scales NULL for a bf16 cache
 *   conds       NULL, or [L] conditional handles (sixbit_graph_cond_create)
 *               of the per-block switches of a captured graph
 *   block_cfg   NULL, or [L] per-block thresholds (DEVICE memory): block l
 *               decides with block_cfg[l] instead of the call's cfg.  The
 *               popular summary (section 5) finds that blocks at different
 *               depths differ in temporal stability; per-depth thresholds
 *               are the configuration that finding calls for.
 * n % 8 == 0 (n % 32 == 0 for MXFP8); 16-byte aligned tensors.
 */
typedef struct {
  sixbit_policy_state* states;
  sixbit_stats* stats;
  int32_t* modes;
  double* in_stats0;
  const uint16_t* x0;
  uint16_t* buf[2];
  void* deltas;
  uint8_t* delta_scales;
  uint32_t* run_len;
  const uint64_t* conds;
  const sixbit_policy_cfg* block_cfg;
  int64_t n;
  int32_t L;
  int32_t delta_format;
} sixbit_dit_blocks;

/*
 * One denoising step of the stack (technical summary sections 2.A-2.C;
 * popular summary sections 1-3), with every per-block decision taken on the
 * device at the tail of the kernel that produces the statistics it needs:
 *   sixbit_dit_begin      statistics of x0, then block 0's decision;
 *   sixbit_dit_block_end  for a block l that computed (its mode word is not
 *                         SKIP): sixbit_block_stats of x_{l-1}, x_l and
 *                         Delta_l into stats[l], then block l+1's decision;
 *                         nothing for a skipped block;
 *   sixbit_dit_skip_run   for a block l that starts a run of k skipping
 *                         blocks: their TDC skips in one pass,
 *                         x_{l+k-1} = bf16(...bf16(x_{l-1} + Delta_l)... +
 *                         Delta_{l+k-1}) into buf[(l+k-1) % 2] with its
 *                         {max |x|, sum |x|, count} into stats[l+k-1], then
 *                         the decision of block l+k; nothing otherwise.
 * A decision is sixbit_policy_step's (input statistics from stats[l-1], or
 * in_stats0 for l = 0; the word to modes[l]).  A skip depends only on the
 * block's own state, never on its input, so when block l skips, the blocks
 * l+1 .. l+k-1 that will also skip are known: block l's decision takes
 * theirs too (they launch nothing) and records k in run_len[l].  Results
 * are bit-identical to one policy step + one skip
 * (or the block's compute + block statistics) per block; the skipped
 * intermediate activations are not written.  With conds, each decision also
 * sets conds[l]: 0, 1, 2 for NVFP4, INT8, BF16 (the compute bodies, each
 * ending with sixbit_dit_block_end), 3 for a run start (sixbit_dit_skip_run)
 * and 4 (no body) for the other blocks of a run.  Eager use: after sixbit_dit_begin,
 * per block the mode-gated compute calls, sixbit_dit_block_end and
 * sixbit_dit_skip_run (each a no-op when it does not apply).  scratch as for
 * sixbit_block_stats.  cfg is a HOST pointer.  err_dev is reserved (no
 * device-side error is possible).
 */
sixbit_status sixbit_dit_begin(const sixbit_policy_cfg* cfg, const sixbit_dit_blocks* blocks, void* scratch,
                               int32_t* err_dev, void* stream);
sixbit_status sixbit_dit_block_end(const sixbit_policy_cfg* cfg, const sixbit_dit_blocks* blocks, int l,
                                   void* scratch, int32_t* err_dev, void* stream);
sixbit_status sixbit_dit_skip_run(const sixbit_policy_cfg* cfg, const sixbit_dit_blocks* blocks, int l,
                                  void* scratch, int32_t* err_dev, void* stream);

/*
 * sixbit_dit_block_end for a block l whose down projection ran as
 * sixbit_qgemm_blockstats (residual = x_{l-1}, Y = x_l, delta_cache =
 * Delta_l's slot of blocks->deltas) with these parts: folds them into
 * stats[l], then block l+1's decision; nothing for a skipped block.  Bf16
 * Delta cache only (delta_format SIXBIT_DELTA_BF16).
 */
sixbit_status sixbit_dit_block_end_parts(const sixbit_policy_cfg* cfg, const sixbit_dit_blocks* blocks, int l,
                                         const void* parts, int32_t* err_dev, void* stream);

/*
 * Storage format of the Delta cache.  The method only says the cache may be
 * kept in a low precision to save memory (popular summary, section 7);
 * MXFP8 is the OCP Microscaling format with E4M3 elements: blocks of 32
 * consecutive elements share an E8M0 scale 2^X, X = floor(log2 max|Delta|)
 * - 8 clamped to [-127, 127] (-127 for an all-zero block), stored as the byte
 * X + 127; element k is E4M3(Delta_k / 2^X), round to nearest even,
 * saturating at 448, stored in byte k.  About 1.03 bytes per element instead
 * of 2.
 */
enum { SIXBIT_DELTA_BF16 = 0, SIXBIT_DELTA_MXFP8 = 1 };

/*
 * sixbit_block_stats with the Delta cache in MXFP8: the fresh
 * Delta = bf16(f32(x_out) - f32(x_in)) enters the sums as it is; the
 * previous one, read from (delta_codes [n], delta_scales [n / 32]),
 * dequantized (exact in FP32); then the fresh Delta is encoded over it.  A
 * zeroed cache holds Delta = 0.  n % 32 == 0; delta_codes 16-byte aligned.
 */
sixbit_status sixbit_block_stats_mxfp8(const uint16_t* x_in, const uint16_t* x_out, uint8_t* delta_codes,
                                       uint8_t* delta_scales, int64_t n, const int32_t* mode_dev,
                                       sixbit_stats* stats_dev, void* scratch, int32_t* err_dev, void* stream);

/* sixbit_skip_apply with an MXFP8 Delta cache: x_out = bf16(f32(x_in) +
 * dequantized Delta).  n % 32 == 0; delta_codes 16-byte aligned. */
sixbit_status sixbit_skip_apply_mxfp8(const uint16_t* x_in, const uint8_t* delta_codes, const uint8_t* delta_scales,
                                      uint16_t* x_out, int64_t n, const int32_t* mode_dev, sixbit_stats* stats_dev,
                                      void* scratch, int32_t* err_dev, void* stream);

/* ---- companions of the hot path ---------------------------------------- */

/* Input statistics of a bf16 tensor (the first block's input): out_dev[0..3] =
 * {max |x|, sum |x|, count, sum x^2} in float64.  n % 8 == 0.  scratch as for
 * sixbit_block_stats. */
sixbit_status sixbit_tensor_stats(const uint16_t* x, int64_t n, double* out_dev, void* scratch,
                                  int32_t* err_dev, void* stream);

/* TDC skip (technical summary section 2.B): x_out = bf16(f32(x_in) + f32(Delta)),
 * and the output statistics into stats_dev->{max_abs_out, sum_abs_out, count}
 * (other fields untouched).  With mode_dev non-NULL, runs only when the mode
 * is SKIP.  n % 8 == 0.  scratch as for sixbit_block_stats. */
sixbit_status sixbit_skip_apply(const uint16_t* x_in, const uint16_t* delta_cache, uint16_t* x_out,
                                int64_t n, const int32_t* mode_dev, sixbit_stats* stats_dev,
                                void* scratch, int32_t* err_dev, void* stream);

/*
 * Allocation-free variant of sixbit_block_stats.  The paper has no
 * counterpart to this call; it exists for callers that cannot call
 * cudaMalloc (code running under an allocator that owns all device memory,
 * or in a host that forbids allocation after start-up) and so cannot provide
 * the scratch buffer sixbit_block_stats asks for.  Same inputs and outputs as
 * sixbit_block_stats; the delta cache, the maximum and the count are
 * bit-identical to it, while the sums are reduced over a different grid and
 * so in a different order: they agree to about 5e-7 relative (the
 * Kahan-summed sum_xin2 and sum_abs_out) and 1e-9 (the others), and a
 * policy decision can differ only for a statistic within the policy's 1e-6
 * near band of its threshold.  The reduction scratch is a fixed 256 KB array
 * inside the library, which every GPU that loads the library holds until
 * the process exits.  n must not exceed
 * sixbit_block_stats_noalloc_max_elems() (268,435,456 elements); larger n
 * returns SIXBIT_ESHAPE and launches nothing.  The call allocates no memory
 * itself.  The library looks up the array's device address at its first
 * call of any entry point on each device (and again after a device reset);
 * under CUDA's lazy module loading that is when the driver creates the
 * array, so make one library call before a memory pool claims all device
 * memory, or set CUDA_MODULE_LOADING=EAGER.  Make that first call before any
 * stream capture.  All calls share the one array: calls that overlap on the
 * GPU race and corrupt each other's results, so order them (one stream, or
 * events).  err_dev is unused (the kernel has no device-side error path) and
 * may be NULL.
 */
sixbit_status sixbit_block_stats_noalloc(const uint16_t* x_in, const uint16_t* x_out, uint16_t* delta_cache,
                                         int64_t n, const int32_t* mode_dev, sixbit_stats* stats_dev,
                                         int32_t* err_dev, void* stream);
/* Largest n sixbit_block_stats_noalloc accepts. */
int64_t sixbit_block_stats_noalloc_max_elems(void);

/* ---- device-decided branches in a captured CUDA graph ------------------- */

/*
 * The policy decides per block on the device (technical summary sections
 * 2.A-2.C), so a captured denoising step needs a branch the GPU resolves.
 * While `stream` is being captured into a CUDA graph, sixbit_graph_switch_begin
 * appends a one-thread selector kernel and a SWITCH conditional node with
 * `nbranches` bodies: when the graph runs, body i executes when the low byte
 * of *mode_dev equals first_mode + i, and no body executes otherwise.  Fill
 * each body with sixbit_graph_branch_begin (returns `body_stream`, a
 * caller-owned stream other than `stream`, now capturing into that body;
 * enqueue the body's work there) and sixbit_graph_branch_end, then close with
 * sixbit_graph_switch_end; capture of `stream` continues after the node.
 * nbranches <= 8.  The returned object is
 * owned by the library and freed by sixbit_graph_switch_end.  Errors:
 * SIXBIT_EINVAL when `stream` is not capturing or calls are out of order.
 */
typedef struct sixbit_switch sixbit_switch;
sixbit_status sixbit_graph_switch_begin(void* stream, void* body_stream, const int32_t* mode_dev, int first_mode,
                                        int nbranches, sixbit_switch** sw);
/*
 * The same SWITCH node without the selector kernel: the condition is set by
 * kernels captured before it (the sixbit_dit_* calls, through the blocks'
 * conds).  sixbit_graph_cond_create makes a handle in the graph `stream` is
 * capturing (its value defaults to "no body" at every graph launch);
 * sixbit_graph_switch_begin_cond appends the node.
 */
sixbit_status sixbit_graph_cond_create(void* stream, int nbranches, uint64_t* handle);
sixbit_status sixbit_graph_switch_begin_cond(void* stream, void* body_stream, uint64_t handle, int nbranches,
                                             sixbit_switch** sw);
sixbit_status sixbit_graph_branch_begin(sixbit_switch* sw, int branch, void** body_stream);
sixbit_status sixbit_graph_branch_end(sixbit_switch* sw);
sixbit_status sixbit_graph_switch_end(sixbit_switch* sw);

/*
 * Test setting for the GEMMs' failure path (every GEMM launched after the
 * call, process-wide).  Every wait in the GEMM kernels is bounded; this
 * lets a test make those waits run out on purpose, without faulting anything:
 * wait_limit_ns replaces the 2 s limit (0 restores it), and with
 * withhold_first_stage = 1 the producer of every CTA skips the copies of its
 * first pipeline stage, so the tensor-core thread's wait for it runs out.
 * The kernel then records SIXBIT_ETIMEOUT in err_dev, stops its other roles,
 * waits (bounded) for its copies and tensor-core work in flight, frees its
 * tensor memory and returns, leaving the context usable.  Returns
 * SIXBIT_EINVAL for withhold_first_stage outside {0, 1}.  Not for production
 * use: call it with (0, 0) afterwards.
 */
sixbit_status sixbit_debug_gemm_timeout(uint64_t wait_limit_ns, int32_t withhold_first_stage);

/* Synchronize `stream` and return the status recorded in err_dev (and clear it). */
sixbit_status sixbit_check(int32_t* err_dev, void* stream);

/* Human-readable name of a status code. */
const char* sixbit_status_str(sixbit_status s);

/* Number of kernels the library has launched since it was loaded. */
uint64_t sixbit_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SIXBIT_H */
