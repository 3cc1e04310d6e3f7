// extern "C" entry points of libsixbit: argument validation, tensor-map
// construction for the GEMM's TMA loads, and kernel dispatch.  The library
// allocates no device memory.
#include <atomic>
#include <cstdint>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "ctx_cache.h"
#include "internal.h"

namespace sixbit {

uint64_t current_context_id() {
  struct Fns {
    PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    PFN_cuCtxGetId_v12000 get_id = nullptr;
  };
  static const Fns fns = [] {
    Fns f;
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    return f;
  }();
  if (fns.get_current == nullptr || fns.get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (fns.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (fns.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return static_cast<uint64_t>(id);
}

int sm_count() {
  static ContextCache<int> cache;
  int sms = 0;
  const cudaError_t e = cache.get(&sms, [](int* o) {
    int dev = 0;
    cudaError_t r = cudaGetDevice(&dev);
    if (r == cudaSuccess) r = cudaDeviceGetAttribute(o, cudaDevAttrMultiProcessorCount, dev);
    return (r == cudaSuccess && *o > 0) ? cudaSuccess : cudaErrorInvalidDevice;
  });
  return (e == cudaSuccess && sms > 0) ? sms : 148;
}

static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// sixbit_debug_gemm_timeout's setting (0: the normal 2 s limit, no withheld stage).
static std::atomic<uint64_t> g_dbg_wait_ns{0};
static std::atomic<int> g_dbg_withhold{0};
void gemm_debug_params(GemmParams& p) {
  const uint64_t w = g_dbg_wait_ns.load();
  p.wait_ns = w != 0 ? w : kWaitLimitNs;
  p.withhold_first = g_dbg_withhold.load();
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool valid_block(int b) { return b == 16 || b == 64 || b == 256; }

// Checks that the current device is a compute capability 10.3 GPU (once per
// context); the first successful check in a context also resolves the device
// address of the allocation-free entry point's scratch array, so its module
// is loaded at the library's first call on each device.
sixbit_status check_device() {
  static ContextCache<int> ok;
  int v = 0;
  const cudaError_t e = ok.get(&v, [](int* o) {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return cudaErrorInvalidDevice;
    if (major != 10 || minor != 3) return cudaErrorInvalidDevice;
    void* scratch = nullptr;
    (void)noalloc_scratch(&scratch);   // its own call reports a failure
    *o = 1;
    return cudaSuccess;
  });
  return e == cudaSuccess ? SIXBIT_OK : SIXBIT_EUNSUPPORTED;
}

static sixbit_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SIXBIT_OK : SIXBIT_ECUDA; }

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// 2-D row-major tensor [rows, cols] of `dtype`, box = 128 bytes of columns x
// `box_rows` rows, 128-byte swizzle, out-of-bounds rows read as zero.
static bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dtype, int elem_bytes, int rows, int cols,
                     int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem_bytes};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem_bytes), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dtype, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// int8 [rows, cols] for the W4A8 GEMM's activation codes: box 128 bytes of
// columns x 128 rows, 128-byte swizzle (16-byte chunk c of row r lands at
// chunk c ^ (r & 7), so each converter thread's reads of its own row are
// conflict-free), out-of-bounds rows read as zero.
static bool make_map_s8(CUtensorMap* m, const int8_t* base, int rows, int cols) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 output Y [rows, cols] for the GEMM epilogue's TMA stores: box 32
// columns (64 bytes) x 32 rows, 64-byte swizzle.
static bool make_store_map(CUtensorMap* m, const uint16_t* Y, int rows, int cols) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(Y), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace sixbit

using namespace sixbit;

extern "C" {

size_t sixbit_fp4_scale_bytes(int rows, int K) {
  if (rows < 0 || K < 0) return 0;
  return static_cast<size_t>((rows + 127) / 128) * 128 * static_cast<size_t>(K / 16);
}

size_t sixbit_fp4_scale_offset(int r, int kb, int K) {
  return static_cast<size_t>(r / 128) * (128 * static_cast<size_t>(K / 16)) + static_cast<size_t>(kb / 4) * 512 +
         static_cast<size_t>((r % 32) * 16 + ((r / 32) % 4) * 4 + (kb % 4));
}

size_t sixbit_stats_scratch_bytes(int64_t n) { return stats_scratch_bytes(n); }

size_t sixbit_qgemm_workspace_bytes(int N, int K) {
  if (N <= 0 || K <= 0) return 0;
  return w4a8_workspace_bytes(N, K);
}

uint64_t sixbit_launch_count(void) { return g_launches.load(); }

const char* sixbit_status_str(sixbit_status s) {
  switch (s) {
    case SIXBIT_OK: return "ok";
    case SIXBIT_EINVAL: return "invalid argument";
    case SIXBIT_ESHAPE: return "unsupported shape";
    case SIXBIT_EALIGN: return "pointer not 16-byte aligned";
    case SIXBIT_EUNSUPPORTED: return "no compute capability 10.3 device";
    case SIXBIT_ECUDA: return "CUDA runtime error";
    case SIXBIT_ETIMEOUT: return "device-side wait timed out";
    case SIXBIT_EDEVICE: return "device-side check failed";
    default: return "unknown status";
  }
}

sixbit_status sixbit_debug_gemm_timeout(uint64_t wait_limit_ns, int32_t withhold_first_stage) {
  if (withhold_first_stage != 0 && withhold_first_stage != 1) return SIXBIT_EINVAL;
  g_dbg_wait_ns.store(wait_limit_ns);
  g_dbg_withhold.store(withhold_first_stage);
  return SIXBIT_OK;
}

sixbit_status sixbit_check(int32_t* err_dev, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SIXBIT_ECUDA;
  if (err_dev == nullptr) return SIXBIT_OK;
  int32_t v = 0;
  if (cudaMemcpy(&v, err_dev, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SIXBIT_ECUDA;
  if (v != 0) {
    const int32_t z = 0;
    cudaMemcpy(err_dev, &z, sizeof(z), cudaMemcpyHostToDevice);
  }
  return v;
}

sixbit_status sixbit_pack_weights(const float* W, int N, int K, int had_block, const sixbit_weights* out,
                                  int32_t* err_dev, void* stream) {
  (void)err_dev;
  if (W == nullptr || out == nullptr || out->fp4_codes == nullptr || out->fp4_scales == nullptr ||
      out->fp4_amax == nullptr || out->fp4_tensor_scale == nullptr || out->i4_codes == nullptr ||
      out->i4_scales == nullptr || out->bf16_w == nullptr)
    return SIXBIT_EINVAL;
  if (N <= 0 || K <= 0 || K % 128 != 0 || !valid_block(had_block) || K % had_block != 0) return SIXBIT_ESHAPE;
  if (!aligned16(W) || !aligned16(out->fp4_codes) || !aligned16(out->i4_codes) || !aligned16(out->bf16_w))
    return SIXBIT_EALIGN;
  sixbit_status s = check_device();
  if (s != SIXBIT_OK) return s;
  return cuda_status(launch_pack_weights(W, N, K, had_block, out, static_cast<cudaStream_t>(stream)));
}

sixbit_status sixbit_hadamard_quant(const uint16_t* X, int M, int K, int had_block, int mode,
                                    const int32_t* mode_dev, const float* tamax_in, const sixbit_qact* out,
                                    int32_t* err_dev, void* stream) {
  (void)err_dev;
  if (X == nullptr || out == nullptr) return SIXBIT_EINVAL;
  if (M <= 0 || K <= 0 || K % 128 != 0 || !valid_block(had_block) || K % had_block != 0) return SIXBIT_ESHAPE;
  if (!aligned16(X) || (out->rotated && !aligned16(out->rotated))) return SIXBIT_EALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool want_fp4 = mode_dev != nullptr || mode == SIXBIT_MODE_NVFP4;
  const bool want_i8 = mode_dev != nullptr || mode == SIXBIT_MODE_INT8;
  if (mode_dev == nullptr && mode != SIXBIT_MODE_NVFP4 && mode != SIXBIT_MODE_INT8) {
    if (mode == SIXBIT_MODE_BF16 || mode == SIXBIT_MODE_SKIP) return SIXBIT_OK;
    return SIXBIT_EINVAL;
  }
  if (want_fp4 && (out->fp4_codes == nullptr || out->fp4_scales == nullptr || out->tensor_scale == nullptr ||
                   (tamax_in == nullptr && out->tensor_amax == nullptr)))
    return SIXBIT_EINVAL;
  if (want_i8 && (out->row_scale == nullptr || out->i8_codes == nullptr)) return SIXBIT_EINVAL;
  if (want_fp4 && !aligned16(out->fp4_codes)) return SIXBIT_EALIGN;
  if (want_i8 && !aligned16(out->i8_codes)) return SIXBIT_EALIGN;
  sixbit_status s = check_device();
  if (s != SIXBIT_OK) return s;
  if (want_fp4) {
    const float* amax = tamax_in;
    if (amax == nullptr) {
      cudaError_t e = launch_hq_amax(X, M, K, had_block, mode_dev, out->tensor_amax, st);
      if (e != cudaSuccess) return SIXBIT_ECUDA;
      amax = out->tensor_amax;
    }
    cudaError_t e = launch_hq_nvfp4(X, M, K, had_block, mode_dev, amax, out, st);
    if (e != cudaSuccess) return SIXBIT_ECUDA;
  }
  if (want_i8) {
    cudaError_t e = launch_hq_int8(X, M, K, had_block, mode_dev, out, st);
    if (e != cudaSuccess) return SIXBIT_ECUDA;
  }
  return SIXBIT_OK;
}

static sixbit_status qgemm_impl(const sixbit_qact* A, const uint16_t* X_bf16, const sixbit_weights* W, int M,
                                int N, int K, int mode, const int32_t* mode_dev, int epilogue,
                                const uint16_t* residual, uint16_t* Y, float* Y_f32, int32_t* acc_dbg,
                                void* workspace, int32_t* err_dev, void* stream, int had_block, float* rot_amax,
                                uint16_t* bs_delta = nullptr, void* bs_parts = nullptr) {
  if (W == nullptr || (Y == nullptr && Y_f32 == nullptr)) return SIXBIT_EINVAL;
  if (epilogue != SIXBIT_EPI_NONE && epilogue != SIXBIT_EPI_GELU && epilogue != SIXBIT_EPI_RESIDUAL)
    return SIXBIT_EINVAL;
  if (epilogue == SIXBIT_EPI_RESIDUAL && residual == nullptr) return SIXBIT_EINVAL;
  if (M <= 0 || N <= 0 || K <= 0 || K % 128 != 0 || N % 16 != 0) return SIXBIT_ESHAPE;
  if ((Y && !aligned16(Y)) || (Y_f32 && !aligned16(Y_f32)) || (residual && !aligned16(residual)))
    return SIXBIT_EALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool only_fp4 = rot_amax != nullptr;  // the rotated-amax epilogue exists for the NVFP4 kind only
  const bool run_fp4 = mode_dev != nullptr || mode == SIXBIT_MODE_NVFP4;
  const bool run_i8 = !only_fp4 && (mode_dev != nullptr || mode == SIXBIT_MODE_INT8);
  const bool run_bf = !only_fp4 && (mode_dev != nullptr || mode == SIXBIT_MODE_BF16);
  if (mode_dev == nullptr && !run_fp4 && !run_i8 && !run_bf) return mode == SIXBIT_MODE_SKIP ? SIXBIT_OK : SIXBIT_EINVAL;
  if ((run_fp4 || run_i8) && A == nullptr) return SIXBIT_EINVAL;
  if (run_fp4 && (A->fp4_codes == nullptr || A->fp4_scales == nullptr || A->tensor_scale == nullptr ||
                  W->fp4_codes == nullptr || W->fp4_scales == nullptr || W->fp4_tensor_scale == nullptr))
    return SIXBIT_EINVAL;
  if (run_i8 && (A->i8_codes == nullptr || A->row_scale == nullptr || W->i4_codes == nullptr ||
                 W->i4_scales == nullptr || workspace == nullptr))
    return SIXBIT_EINVAL;
  if (run_bf && (X_bf16 == nullptr || W->bf16_w == nullptr)) return SIXBIT_EINVAL;
  if ((run_fp4 && (!aligned16(A->fp4_codes) || !aligned16(A->fp4_scales) || !aligned16(W->fp4_codes) ||
                   !aligned16(W->fp4_scales))) ||
      (run_i8 && (!aligned16(A->i8_codes) || !aligned16(W->i4_codes) || !aligned16(workspace))) ||
      (run_bf && (!aligned16(X_bf16) || !aligned16(W->bf16_w))))
    return SIXBIT_EALIGN;
  sixbit_status s = check_device();
  if (s != SIXBIT_OK) return s;
  if (rot_amax != nullptr && cudaMemsetAsync(rot_amax, 0, sizeof(float), st) != cudaSuccess) return SIXBIT_ECUDA;

  GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.mode_dev = mode_dev;
  p.epilogue = epilogue;
  p.residual = residual;
  p.Y = Y;
  p.Yf = Y_f32;
  p.err = err_dev;
  // Walk the shorter output dimension fastest: the CTAs in flight then share
  // tiles of the larger operand, which streams from HBM once, while the
  // smaller one is re-read from L2 (an A of 17776 x 7680 bf16 does not fit
  // in L2 and would be re-read from HBM once per column-tile pass).
  p.n_fastest = M > N ? 1 : 0;
  p.rot_amax = rot_amax;
  p.had_block = had_block;
  p.bs_delta = bs_delta;
  p.bs_parts = bs_parts;
  gemm_debug_params(p);
  // The bf16-operand kinds (BF16, W4A8) write a bf16 Y through TMA stores
  // (Y 16-byte aligned, N % 16 == 0 checked above); an FP32 Y is stored
  // directly.
  CUtensorMap my{};
  p.y_tma = (Y_f32 == nullptr && (run_bf || run_i8)) ? 1 : 0;
  if (p.y_tma && !make_store_map(&my, Y, M, N)) return SIXBIT_ECUDA;
  if (run_fp4) {
    CUtensorMap ma, mb;
    if (!make_map(&ma, A->fp4_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, M, K / 2, 128) ||
        !make_map(&mb, W->fp4_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, N, K / 2, 256))
      return SIXBIT_ECUDA;
    GemmParams q = p;
    q.want_mode = SIXBIT_MODE_NVFP4;
    q.sfa = A->fp4_scales;
    q.sfb = W->fp4_scales;
    q.s_a = A->tensor_scale;
    q.s_b = W->fp4_tensor_scale;
    if (launch_qgemm_nvf4(ma, mb, q, st) != cudaSuccess) return SIXBIT_ECUDA;
  }
  if (run_i8) {
    // the INT4 weights, expanded to fp16 once per call into the workspace
    uint16_t* wexp = static_cast<uint16_t*>(workspace);
    CUtensorMap ma, mb;
    if (!make_map_s8(&ma, A->i8_codes, M, K) ||
        !make_map(&mb, wexp, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, N, K, 192))
      return SIXBIT_ECUDA;
    if (launch_w4_expand(W->i4_codes, N, K, wexp, mode_dev, st) != cudaSuccess) return SIXBIT_ECUDA;
    GemmParams q = p;
    q.want_mode = SIXBIT_MODE_INT8;
    q.row_scale = A->row_scale;
    q.grp_scale = W->i4_scales;
    q.acc_dbg = acc_dbg;
    if (launch_qgemm_w4a8(ma, mb, my, q, st) != cudaSuccess) return SIXBIT_ECUDA;
  }
  if (run_bf) {
    CUtensorMap ma, mb;
    if (!make_map(&ma, X_bf16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, K, 128) ||
        !make_map(&mb, W->bf16_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, N, K, 256))
      return SIXBIT_ECUDA;
    GemmParams q = p;
    q.want_mode = SIXBIT_MODE_BF16;
    if (launch_qgemm_bf16(ma, mb, my, q, st) != cudaSuccess) return SIXBIT_ECUDA;
  }
  return SIXBIT_OK;
}

sixbit_status sixbit_qgemm(const sixbit_qact* A, const uint16_t* X_bf16, const sixbit_weights* W, int M, int N,
                           int K, int mode, const int32_t* mode_dev, int epilogue, const uint16_t* residual,
                           uint16_t* Y, float* Y_f32, int32_t* acc_dbg, void* workspace, int32_t* err_dev,
                           void* stream) {
  return qgemm_impl(A, X_bf16, W, M, N, K, mode, mode_dev, epilogue, residual, Y, Y_f32, acc_dbg, workspace, err_dev,
                    stream, 0, nullptr);
}

sixbit_status sixbit_qgemm_rotamax(const sixbit_qact* A, const sixbit_weights* W, int M, int N, int K,
                                   const int32_t* mode_dev, int epilogue, const uint16_t* residual, uint16_t* Y,
                                   int had_block, float* amax_out, int32_t* err_dev, void* stream) {
  if (Y == nullptr || amax_out == nullptr) return SIXBIT_EINVAL;
  if ((had_block != 16 && had_block != 64) || N % 128 != 0) return SIXBIT_ESHAPE;
  return qgemm_impl(A, nullptr, W, M, N, K, SIXBIT_MODE_NVFP4, mode_dev, epilogue, residual, Y, nullptr, nullptr,
                    nullptr, err_dev, stream, had_block, amax_out);
}

sixbit_status sixbit_qgemm_blockstats(const sixbit_qact* A, const uint16_t* X_bf16, const sixbit_weights* W, int M,
                                      int N, int K, int mode, const int32_t* mode_dev, const uint16_t* residual,
                                      uint16_t* Y, uint16_t* delta_cache, void* parts, void* workspace,
                                      int32_t* err_dev, void* stream) {
  if (residual == nullptr || Y == nullptr || delta_cache == nullptr || parts == nullptr) return SIXBIT_EINVAL;
  if (!aligned16(delta_cache) || !aligned16(parts)) return SIXBIT_EALIGN;
  return qgemm_impl(A, X_bf16, W, M, N, K, mode, mode_dev, SIXBIT_EPI_RESIDUAL, residual, Y, nullptr, nullptr,
                    workspace, err_dev, stream, 0, nullptr, delta_cache, parts);
}

size_t sixbit_blockstats_parts_bytes(void) {
  if (check_device() != SIXBIT_OK) return 0;
  return bs_parts_bytes();
}

sixbit_status sixbit_block_stats_parts(const void* parts, int64_t n, sixbit_stats* stats_dev, int32_t* err_dev,
                                       void* stream) {
  (void)err_dev;
  if (parts == nullptr || stats_dev == nullptr) return SIXBIT_EINVAL;
  if (n <= 0) return SIXBIT_ESHAPE;
  if (!aligned16(parts)) return SIXBIT_EALIGN;
  sixbit_status s = check_device();
  if (s != SIXBIT_OK) return s;
  return cuda_status(launch_block_stats_parts(parts, n, stats_dev, static_cast<cudaStream_t>(stream)));
}

sixbit_status sixbit_block_stats(const uint16_t* x_in, const uint16_t* x_out, uint16_t* delta_cache, int64_t n,
                                 const int32_t* mode_dev, sixbit_stats* stats_dev, void* scratch, int32_t* err_dev,
                                 void* stream) {
  (void)err_dev;
  if (x_in == nullptr || x_out == nullptr || delta_cache == nullptr || stats_dev == nullptr || scratch == nullptr)
    return SIXBIT_EINVAL;
  if (n <= 0 || n % 8 != 0) return SIXBIT_ESHAPE;
  if (!aligned16(x_in) || !aligned16(x_out) || !aligned16(delta_cache) || !aligned16(scratch)) return SIXBIT_EALIGN;
  sixbit_status s = check_device();
  if (s != SIXBIT_OK) return s;
  return cuda_status(
      launch_block_stats(x_in, x_out, delta_cache, n, mode_dev, stats_dev, scratch, static_cast<cudaStream_t>(stream)));
}

sixbit_status sixbit_tensor_stats(const uint16_t* x, int64_t n, double* out_dev, void* scratch, int32_t* err_dev,
                                  void* stream) {
  (void)err_dev;
  if (x == nullptr || out_dev == nullptr || scratch == nullptr) return SIXBIT_EINVAL;
  if (n <= 0 || n % 8 != 0) return SIXBIT_ESHAPE;
  if (!aligned16(x) || !aligned16(scratch)) return SIXBIT_EALIGN;
  sixbit_status s = check_device();
  if (s != SIXBIT_OK) return s;
  return cuda_status(launch_tensor_stats(x, n, out_dev, scratch, static_cast<cudaStream_t>(stream)));
}

sixbit_status sixbit_skip_apply(const uint16_t* x_in, const uint16_t* delta_cache, uint16_t* x_out, int64_t n,
                                const int32_t* mode_dev, sixbit_stats* stats_dev, void* scratch, int32_t* err_dev,
                                void* stream) {
  (void)err_dev;
  if (x_in == nullptr || delta_cache == nullptr || x_out == nullptr || stats_dev == nullptr || scratch == nullptr)
    return SIXBIT_EINVAL;
  if (n <= 0 || n % 8 != 0) return SIXBIT_ESHAPE;
  if (!aligned16(x_in) || !aligned16(x_out) || !aligned16(delta_cache) || !aligned16(scratch)) return SIXBIT_EALIGN;
  sixbit_status s = check_device();
  if (s != SIXBIT_OK) return s;
  return cuda_status(
      launch_skip_apply(x_in, delta_cache, x_out, n, mode_dev, stats_dev, scratch, static_cast<cudaStream_t>(stream)));
}

sixbit_status sixbit_block_stats_mxfp8(const uint16_t* x_in, const uint16_t* x_out, uint8_t* delta_codes,
                                       uint8_t* delta_scales, int64_t n, const int32_t* mode_dev,
                                       sixbit_stats* stats_dev, void* scratch, int32_t* err_dev, void* stream) {
  (void)err_dev;
  if (x_in == nullptr || x_out == nullptr || delta_codes == nullptr || delta_scales == nullptr ||
      stats_dev == nullptr || scratch == nullptr)
    return SIXBIT_EINVAL;
  if (n <= 0 || n % 32 != 0) return SIXBIT_ESHAPE;
  if (!aligned16(x_in) || !aligned16(x_out) || !aligned16(delta_codes) || !aligned16(scratch)) return SIXBIT_EALIGN;
  sixbit_status s = check_device();
  if (s != SIXBIT_OK) return s;
  return cuda_status(launch_block_stats_mx(x_in, x_out, delta_codes, delta_scales, n, mode_dev, stats_dev, scratch,
                                           static_cast<cudaStream_t>(stream)));
}

sixbit_status sixbit_skip_apply_mxfp8(const uint16_t* x_in, const uint8_t* delta_codes, const uint8_t* delta_scales,
                                      uint16_t* x_out, int64_t n, const int32_t* mode_dev, sixbit_stats* stats_dev,
                                      void* scratch, int32_t* err_dev, void* stream) {
  (void)err_dev;
  if (x_in == nullptr || delta_codes == nullptr || delta_scales == nullptr || x_out == nullptr ||
      stats_dev == nullptr || scratch == nullptr)
    return SIXBIT_EINVAL;
  if (n <= 0 || n % 32 != 0) return SIXBIT_ESHAPE;
  if (!aligned16(x_in) || !aligned16(x_out) || !aligned16(delta_codes) || !aligned16(scratch)) return SIXBIT_EALIGN;
  sixbit_status s = check_device();
  if (s != SIXBIT_OK) return s;
  return cuda_status(launch_skip_apply_mx(x_in, delta_codes, delta_scales, x_out, n, mode_dev, stats_dev, scratch,
                                          static_cast<cudaStream_t>(stream)));
}

sixbit_status sixbit_policy_step(const sixbit_policy_cfg* cfg, sixbit_policy_state* state_dev,
                                 const sixbit_stats* last_stats_dev, const double* in_stats_dev, int32_t* mode_dev,
                                 int32_t* err_dev, void* stream) {
  (void)err_dev;
  if (cfg == nullptr || state_dev == nullptr || last_stats_dev == nullptr || in_stats_dev == nullptr ||
      mode_dev == nullptr)
    return SIXBIT_EINVAL;
  sixbit_status s = check_device();
  if (s != SIXBIT_OK) return s;
  return cuda_status(
      launch_policy(*cfg, state_dev, last_stats_dev, in_stats_dev, mode_dev, static_cast<cudaStream_t>(stream)));
}

static sixbit_status check_blocks(const sixbit_policy_cfg* cfg, const sixbit_dit_blocks* blocks, int l,
                                  void* scratch) {
  if (cfg == nullptr || blocks == nullptr || scratch == nullptr) return SIXBIT_EINVAL;
  const sixbit_dit_blocks& B = *blocks;
  if (B.states == nullptr || B.stats == nullptr || B.modes == nullptr || B.run_len == nullptr ||
      B.in_stats0 == nullptr || B.x0 == nullptr || B.buf[0] == nullptr || B.buf[1] == nullptr ||
      B.deltas == nullptr)
    return SIXBIT_EINVAL;
  if (B.delta_format != SIXBIT_DELTA_BF16 && B.delta_format != SIXBIT_DELTA_MXFP8) return SIXBIT_EINVAL;
  if (B.delta_format == SIXBIT_DELTA_MXFP8 && B.delta_scales == nullptr) return SIXBIT_EINVAL;
  if (B.L <= 0 || l < 0 || l >= B.L || B.n <= 0 || B.n % 8 != 0) return SIXBIT_ESHAPE;
  if (B.delta_format == SIXBIT_DELTA_MXFP8 && B.n % 32 != 0) return SIXBIT_ESHAPE;
  if (!aligned16(B.x0) || !aligned16(B.buf[0]) || !aligned16(B.buf[1]) || !aligned16(B.deltas) ||
      !aligned16(scratch))
    return SIXBIT_EALIGN;
  return check_device();
}

sixbit_status sixbit_dit_begin(const sixbit_policy_cfg* cfg, const sixbit_dit_blocks* blocks, void* scratch,
                               int32_t* err_dev, void* stream) {
  const sixbit_status s = check_blocks(cfg, blocks, 0, scratch);
  if (s != SIXBIT_OK) return s;
  return cuda_status(launch_dit_begin(*cfg, *blocks, scratch, err_dev, static_cast<cudaStream_t>(stream)));
}

sixbit_status sixbit_dit_block_end(const sixbit_policy_cfg* cfg, const sixbit_dit_blocks* blocks, int l,
                                   void* scratch, int32_t* err_dev, void* stream) {
  const sixbit_status s = check_blocks(cfg, blocks, l, scratch);
  if (s != SIXBIT_OK) return s;
  return cuda_status(launch_dit_block_end(*cfg, *blocks, l, scratch, err_dev, static_cast<cudaStream_t>(stream)));
}

sixbit_status sixbit_dit_block_end_parts(const sixbit_policy_cfg* cfg, const sixbit_dit_blocks* blocks, int l,
                                         const void* parts, int32_t* err_dev, void* stream) {
  (void)err_dev;
  if (parts == nullptr || (blocks != nullptr && blocks->delta_format != SIXBIT_DELTA_BF16)) return SIXBIT_EINVAL;
  if (!aligned16(parts)) return SIXBIT_EALIGN;
  const sixbit_status s = check_blocks(cfg, blocks, l, const_cast<void*>(parts));
  if (s != SIXBIT_OK) return s;
  return cuda_status(launch_dit_block_end_parts(*cfg, *blocks, l, parts, static_cast<cudaStream_t>(stream)));
}

sixbit_status sixbit_dit_skip_run(const sixbit_policy_cfg* cfg, const sixbit_dit_blocks* blocks, int l,
                                  void* scratch, int32_t* err_dev, void* stream) {
  const sixbit_status s = check_blocks(cfg, blocks, l, scratch);
  if (s != SIXBIT_OK) return s;
  return cuda_status(launch_dit_skip_run(*cfg, *blocks, l, scratch, err_dev, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
