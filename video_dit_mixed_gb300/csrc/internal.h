// Internal interface between the C-ABI layer and the kernel translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sixbit.h"

namespace sixbit {

// SIXBIT_OK when the current device is a compute capability 10.3 GPU (checked
// once per context), else SIXBIT_EUNSUPPORTED.
sixbit_status check_device();
// Device address of the allocation-free entry point's scratch array in the
// current context (resolved once per context).
sixbit_status noalloc_scratch(void** out);

struct GemmParams {
  int M, N, K;
  const int32_t* mode_dev;
  int want_mode;
  int epilogue;
  const uint8_t* sfa;      // NVFP4 tiled scales of A
  const uint8_t* sfb;      // NVFP4 tiled scales of B
  const float* s_a;        // NVFP4 tensor scale of A
  const float* s_b;        // NVFP4 tensor scale of B
  const float* row_scale;  // INT8: s_m [M]
  const float* grp_scale;  // INT8: s_w [K/128][N]
  const uint16_t* residual;
  uint16_t* Y;
  float* Yf;
  int32_t* acc_dbg;
  int32_t* err;
  int n_fastest;           // tile order: 1 = output column tiles fastest, 0 = row tiles fastest
  float* rot_amax;         // NVFP4 epilogue: atomicMax of |bf16(Y) . blockdiag(H_b / sqrt b)| (or NULL)
  int had_block;           // b of rot_amax (16 or 64)
  int y_tma;               // bf16-operand kinds: bf16 Y is written by TMA stores through the Y tensor map
  uint64_t wait_ns;        // limit of every bounded wait (kWaitLimitNs unless a test shortens it)
  int withhold_first;      // test of the failure path: each CTA's producer skips its first stage
  uint16_t* bs_delta;      // residual epilogue: the block's Delta cache (Delta_prev in, Delta out), or NULL
  void* bs_parts;          // ... and its statistics, one partial row per epilogue warp (see gemm_common.cuh)
};

// Partial rows of a GEMM epilogue's block statistics: a uint32 row count at
// byte 0, then one row per CTA of kBsSums float-float values {hi, lo} from
// byte 16, in the order sum Delta^2, sum x_in^2, sum Delta Delta_prev,
// sum Delta_prev^2, max |x_out| (lo = 0), sum |x_out|.  At most sm_count
// rows; a CTA has at most kBsMaxWarps epilogue warps.
constexpr int kBsSums = 6;
constexpr int kBsMaxWarps = 16;
size_t bs_parts_bytes();
cudaError_t launch_block_stats_parts(const void* parts, int64_t n, sixbit_stats* stats, cudaStream_t st);
cudaError_t launch_dit_block_end_parts(const sixbit_policy_cfg& cfg, const sixbit_dit_blocks& B, int l,
                                       const void* parts, cudaStream_t st);

// Test setting of the GEMMs' failure path (sixbit_debug_gemm_timeout).
void gemm_debug_params(GemmParams& p);

cudaError_t launch_hq_amax(const uint16_t* X, int M, int K, int b, const int32_t* mode_dev, float* amax_out,
                           cudaStream_t st);
cudaError_t launch_hq_nvfp4(const uint16_t* X, int M, int K, int b, const int32_t* mode_dev, const float* amax_src,
                            const sixbit_qact* o, cudaStream_t st);
cudaError_t launch_hq_int8(const uint16_t* X, int M, int K, int b, const int32_t* mode_dev, const sixbit_qact* o,
                           cudaStream_t st);
cudaError_t launch_pack_weights(const float* W, int N, int K, int b, const sixbit_weights* o, cudaStream_t st);

size_t stats_scratch_bytes(int64_t n);
cudaError_t launch_tensor_stats(const uint16_t* x, int64_t n, double* out, void* scratch, cudaStream_t st);
cudaError_t launch_block_stats(const uint16_t* x_in, const uint16_t* x_out, uint16_t* delta, int64_t n,
                               const int32_t* mode_dev, sixbit_stats* stats, void* scratch, cudaStream_t st);
// Elements one CTA of the fixed-grid statistics launch covers.
constexpr int64_t kFixedElemsPerCta = 65536;
cudaError_t launch_block_stats_fixed_grid(const uint16_t* x_in, const uint16_t* x_out, uint16_t* delta, int64_t n,
                                          const int32_t* mode_dev, sixbit_stats* stats, void* scratch,
                                          cudaStream_t st);
cudaError_t launch_skip_apply(const uint16_t* x_in, const uint16_t* delta, uint16_t* x_out, int64_t n,
                              const int32_t* mode_dev, sixbit_stats* stats, void* scratch, cudaStream_t st);
cudaError_t launch_block_stats_mx(const uint16_t* x_in, const uint16_t* x_out, uint8_t* codes, uint8_t* scales,
                                  int64_t n, const int32_t* mode_dev, sixbit_stats* stats, void* scratch,
                                  cudaStream_t st);
cudaError_t launch_skip_apply_mx(const uint16_t* x_in, const uint8_t* codes, const uint8_t* scales, uint16_t* x_out,
                                 int64_t n, const int32_t* mode_dev, sixbit_stats* stats, void* scratch,
                                 cudaStream_t st);
cudaError_t launch_dit_begin(const sixbit_policy_cfg& cfg, const sixbit_dit_blocks& B, void* scratch, int32_t* err,
                             cudaStream_t st);
cudaError_t launch_dit_block_end(const sixbit_policy_cfg& cfg, const sixbit_dit_blocks& B, int l, void* scratch,
                                 int32_t* err, cudaStream_t st);
cudaError_t launch_dit_skip_run(const sixbit_policy_cfg& cfg, const sixbit_dit_blocks& B, int l, void* scratch,
                                int32_t* err, cudaStream_t st);
cudaError_t launch_policy(const sixbit_policy_cfg& cfg, sixbit_policy_state* st_dev, const sixbit_stats* last,
                          const double* in_stats, int32_t* mode_out, cudaStream_t st);

cudaError_t launch_qgemm_nvf4(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, cudaStream_t st);
// y: tensor map of the bf16 output (box 32 x 32, 64-byte swizzle), used when p.y_tma.
cudaError_t launch_qgemm_bf16(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& y, const GemmParams& p,
                              cudaStream_t st);
// W4A8: INT4 codes [N, K/2] -> fp16 [N, K] into ws (w4a8_workspace_bytes(N, K)),
// then the GEMM: a_s8 maps the s8 codes [M, K] (box 128 x 128, 128-byte
// swizzle), w_f16 the expanded weights (box 64 x 192, 128-byte swizzle), y the
// bf16 output.
size_t w4a8_workspace_bytes(int N, int K);
cudaError_t launch_w4_expand(const uint8_t* codes, int N, int K, uint16_t* ws, const int32_t* mode_dev,
                             cudaStream_t st);
cudaError_t launch_qgemm_w4a8(const CUtensorMap& a_s8, const CUtensorMap& w_f16, const CUtensorMap& y,
                              const GemmParams& p, cudaStream_t st);

}  // namespace sixbit
