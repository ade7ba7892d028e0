// C ABI of libfgq.so (declared in include/fgq.h): argument checks, device
// checks, then one kernel launch per call on the caller's stream.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fgq.h"
#include "fgq_internal.h"

namespace fgq {

cudaError_t device_info(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool valid[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!valid[dev]) {
    DeviceInfo d{};
    d.device = dev;
    int smem = 0;
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return e;
    d.smem_optin = static_cast<size_t>(smem);
    cache[dev] = d;
    valid[dev] = true;
  }
  *out = cache[dev];
  return cudaSuccess;
}

}  // namespace fgq

namespace {

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// The kernels are built for sm_103a only.
fgq_status get_device(fgq::DeviceInfo* dev) {
  cudaError_t e = fgq::device_info(dev);
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) return FGQ_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return FGQ_ERR_CUDA;
  if (dev->cc_major != 10 || dev->cc_minor != 3) return FGQ_ERR_UNSUPPORTED;
  return FGQ_OK;
}

inline fgq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FGQ_OK : FGQ_ERR_CUDA; }

constexpr int64_t kMaxGroups = (int64_t{1} << 31) - 1;

}  // namespace

extern "C" {

fgq_status fgq_quant_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                               int64_t ldq, float* sx, int mode, void* stream) {
  if (M < 0 || K <= 0 || K % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (mode != FGQ_SCALE_FP32 && mode != FGQ_SCALE_UE8M0) return FGQ_ERR_INVALID_ARG;
  if (M == 0) return FGQ_OK;
  if (!x || !xq || !sx) return FGQ_ERR_INVALID_ARG;
  if (ldx < K || ldq < K || ldx % 8 != 0 || ldq % 16 != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(xq, 16) || !aligned(sx, 4)) return FGQ_ERR_INVALID_ARG;
  if (M > kMaxGroups / (K / 128)) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_quant_act_1x128(x, M, K, ldx, xq, ldq, sx, mode,
                                               static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_quant_act_128x1(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xqt,
                               float* sxt, int mode, void* stream) {
  if (M < 0 || K <= 0 || M % 128 != 0 || K % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (mode != FGQ_SCALE_FP32 && mode != FGQ_SCALE_UE8M0) return FGQ_ERR_INVALID_ARG;
  if (M == 0) return FGQ_OK;
  if (!x || !xqt || !sxt) return FGQ_ERR_INVALID_ARG;
  if (ldx < K || ldx % 8 != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(xqt, 16) || !aligned(sxt, 4)) return FGQ_ERR_INVALID_ARG;
  if ((M / 128) > kMaxGroups / (K / 128)) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_quant_act_128x1(x, M, K, ldx, xqt, sxt, mode,
                                               static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_quant_mxfp4_1x32(const void* x, int64_t R, int64_t K, int64_t ldx, uint8_t* xq,
                                uint8_t* sx, void* stream) {
  if (R < 0 || K <= 0 || K % 32 != 0) return FGQ_ERR_INVALID_ARG;
  if (R == 0) return FGQ_OK;
  if (!x || !xq || !sx) return FGQ_ERR_INVALID_ARG;
  if (ldx < K || ldx % 8 != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(xq, 4)) return FGQ_ERR_INVALID_ARG;
  if (R > kMaxGroups / (K / 32)) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_quant_mxfp4_1x32(x, R, K, ldx, xq, sx, false,
                                                static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_quant_mxfp4_1x32_tiled(const void* x, int64_t R, int64_t K, int64_t ldx,
                                      uint8_t* xq, uint8_t* s_tiles, void* stream) {
  if (R < 0 || K <= 0 || K % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (R == 0) return FGQ_OK;
  if (!x || !xq || !s_tiles) return FGQ_ERR_INVALID_ARG;
  if (ldx < K || ldx % 8 != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(xq, 4) || !aligned(s_tiles, 16)) return FGQ_ERR_INVALID_ARG;
  if (R > kMaxGroups / (K / 32)) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_quant_mxfp4_1x32(x, R, K, ldx, xq, s_tiles, true,
                                                static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_nvfp4_global_scale(const void* x, int64_t R, int64_t K, int64_t ldx, float* g,
                                  void* stream) {
  if (R < 0 || K <= 0 || K % 16 != 0) return FGQ_ERR_INVALID_ARG;
  if (!x || !g) return FGQ_ERR_INVALID_ARG;
  if (ldx < K || ldx % 8 != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(g, 4)) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_nvfp4_global_scale(x, R, K, ldx, g,
                                                  static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_quant_nvfp4_1x16(const void* x, int64_t R, int64_t K, int64_t ldx, const float* g,
                                uint8_t* xq, uint8_t* sx, void* stream) {
  if (R < 0 || K <= 0 || K % 16 != 0) return FGQ_ERR_INVALID_ARG;
  if (R == 0) return FGQ_OK;
  if (!x || !g || !xq || !sx) return FGQ_ERR_INVALID_ARG;
  if (ldx < K || ldx % 8 != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(g, 4) || !aligned(xq, 4)) return FGQ_ERR_INVALID_ARG;
  if (R > kMaxGroups / (K / 16)) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_quant_nvfp4_1x16(x, R, K, ldx, g, xq, sx, false,
                                                static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_quant_w_128x128(const void* w, int64_t K, int64_t N, int64_t ldw, uint8_t* wq,
                               float* sw, int mode, void* stream) {
  if (K <= 0 || N <= 0 || K % 128 != 0 || N % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (mode != FGQ_SCALE_FP32 && mode != FGQ_SCALE_UE8M0) return FGQ_ERR_INVALID_ARG;
  if (!w || !wq || !sw) return FGQ_ERR_INVALID_ARG;
  if (ldw < N || ldw % 8 != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(wq, 16) || !aligned(sw, 4)) return FGQ_ERR_INVALID_ARG;
  if ((K / 128) > kMaxGroups / (N / 128)) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_quant_w_128x128(w, K, N, ldw, wq, sw, mode,
                                               static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_quant_operands(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                              int64_t ldq, float* sx, const void* w, int64_t N, int64_t ldw,
                              uint8_t* wq, float* sw, int mode, void* stream) {
  // the checks of fgq_quant_act_1x128 and fgq_quant_w_128x128 together
  if (M < 0 || K <= 0 || K % 128 != 0 || N <= 0 || N % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (mode != FGQ_SCALE_FP32 && mode != FGQ_SCALE_UE8M0) return FGQ_ERR_INVALID_ARG;
  if (!w || !wq || !sw) return FGQ_ERR_INVALID_ARG;
  if (ldw < N || ldw % 8 != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(wq, 16) || !aligned(sw, 4)) return FGQ_ERR_INVALID_ARG;
  if ((K / 128) > kMaxGroups / (N / 128)) return FGQ_ERR_INVALID_ARG;
  if (M > 0) {
    if (!x || !xq || !sx) return FGQ_ERR_INVALID_ARG;
    if (ldx < K || ldq < K || ldx % 8 != 0 || ldq % 16 != 0) return FGQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(xq, 16) || !aligned(sx, 4)) return FGQ_ERR_INVALID_ARG;
    if (M > kMaxGroups / (K / 128)) return FGQ_ERR_INVALID_ARG;
  }
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_quant_operands(x, M, K, ldx, xq, ldq, sx, w, N, ldw, wq, sw, mode,
                                              static_cast<cudaStream_t>(stream), dev));
}

namespace {

// Checks shared by the GEMM entry points (M == 0 returns OK before pointer checks).
fgq_status check_gemm_args(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                           const void* C, int64_t ldc, int64_t M, int64_t N, int64_t K, int out,
                           int mode) {
  if (M < 0 || N <= 0 || K <= 0 || K % 128 != 0 || N % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (out != FGQ_OUT_F32 && out != FGQ_OUT_BF16) return FGQ_ERR_INVALID_ARG;
  if (mode != FGQ_SCALE_FP32 && mode != FGQ_SCALE_UE8M0) return FGQ_ERR_INVALID_ARG;
  // int32 tile coordinates inside the kernels
  if (M >= (int64_t{1} << 31) || N >= (int64_t{1} << 31) || K >= (int64_t{1} << 31))
    return FGQ_ERR_INVALID_ARG;
  if (M == 0) return FGQ_OK;
  if (!A || !sA || !B || !sB || !C) return FGQ_ERR_INVALID_ARG;
  const int64_t vec = (out == FGQ_OUT_F32) ? 4 : 8;  // elements per 16-byte store
  if (ldc < N || ldc % vec != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(sA, 4) || !aligned(sB, 4))
    return FGQ_ERR_INVALID_ARG;
  return FGQ_OK;
}

// fgq_gemm_fp8_blockscaled_ex sends M up to kLowMDirect to the
// swapped-operand kernel (measured faster there; at larger M the main
// kernel's epilogue is cheaper); the split-K entry point uses it up to kLowM.
constexpr int64_t kLowMDirect = 32;
constexpr int64_t kLowM = 256;

}  // namespace

fgq_status fgq_gemm_fp8_blockscaled_ex(const uint8_t* A, const float* sA, const uint8_t* B,
                                       const float* sB, void* C, int64_t ldc, int64_t M,
                                       int64_t N, int64_t K, int out, int mode, void* stream) {
  fgq_status st = check_gemm_args(A, sA, B, sB, C, ldc, M, N, K, out, mode);
  if (st != FGQ_OK || M == 0) return st;
  fgq::DeviceInfo dev;
  st = get_device(&dev);
  if (st != FGQ_OK) return st;
  const int bf16 = out == FGQ_OUT_BF16 ? 1 : 0;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M <= kLowMDirect)
    return from_cuda(
        fgq::launch_gemm_lowm(A, sA, B, sB, C, ldc, M, N, K, bf16, false, nullptr, s, dev));
  // power-of-two scales: applied by the tensor core, no promotion step
  if (mode == FGQ_SCALE_UE8M0)
    return from_cuda(fgq::launch_gemm_mx(A, sA, B, sB, C, ldc, M, N, K, bf16, s, dev));
  return from_cuda(fgq::launch_gemm_fp8_blockscaled(A, sA, B, sB, C, ldc, M, N, K, bf16, mode, s, dev));
}

fgq_status fgq_gemm_fp8_blockscaled_fused_act(const void* A, int64_t lda, const uint8_t* B,
                                              const float* sB, void* C, int64_t ldc, int64_t M,
                                              int64_t N, int64_t K, int out, int mode,
                                              void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || K % 128 != 0 || N % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (out != FGQ_OUT_F32 && out != FGQ_OUT_BF16) return FGQ_ERR_INVALID_ARG;
  if (mode != FGQ_SCALE_FP32 && mode != FGQ_SCALE_UE8M0) return FGQ_ERR_INVALID_ARG;
  if (N >= (int64_t{1} << 31) || K >= (int64_t{1} << 31)) return FGQ_ERR_INVALID_ARG;
  if (M == 0) return FGQ_OK;
  if (!fgq::lowm_fused_fits(M, K)) return FGQ_ERR_INVALID_ARG;  // M <= 32 and A fits on chip
  if (!A || !B || !sB || !C) return FGQ_ERR_INVALID_ARG;
  const int64_t vec = (out == FGQ_OUT_F32) ? 4 : 8;
  if (lda < K || lda % 8 != 0 || ldc < N || ldc % vec != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(sB, 4))
    return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_gemm_lowm_fused(A, lda, B, sB, C, ldc, M, N, K,
                                               out == FGQ_OUT_BF16 ? 1 : 0, mode,
                                               static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_quant_nvfp4_1x16_tiled(const void* x, int64_t R, int64_t K, int64_t ldx,
                                      const float* g, uint8_t* xq, uint8_t* s_tiles, void* stream) {
  if (R < 0 || K <= 0 || K % 64 != 0) return FGQ_ERR_INVALID_ARG;
  if (R == 0) return FGQ_OK;
  if (!x || !g || !xq || !s_tiles) return FGQ_ERR_INVALID_ARG;
  if (ldx < K || ldx % 8 != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(g, 4) || !aligned(xq, 4) || !aligned(s_tiles, 16))
    return FGQ_ERR_INVALID_ARG;
  if (R > kMaxGroups / (K / 16)) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_quant_nvfp4_1x16(x, R, K, ldx, g, xq, s_tiles, true,
                                                static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_fp4_scale_tiles_bytes(int64_t R, int64_t F, size_t* bytes) {
  if (!bytes || R < 0 || F <= 0 || F % 4 != 0) return FGQ_ERR_INVALID_ARG;
  if (R >= (int64_t{1} << 31) || F >= (int64_t{1} << 31)) return FGQ_ERR_INVALID_ARG;
  *bytes = static_cast<size_t>((R + 127) / 128) * 128u * static_cast<size_t>(F);
  return FGQ_OK;
}

fgq_status fgq_fp4_scales_to_tiles(const uint8_t* s, int64_t R, int64_t F, uint8_t* tiles,
                                   void* stream) {
  if (R < 0 || F <= 0 || F % 4 != 0) return FGQ_ERR_INVALID_ARG;
  if (R >= (int64_t{1} << 31) || F >= (int64_t{1} << 31)) return FGQ_ERR_INVALID_ARG;
  if (R == 0) return FGQ_OK;
  if (!s || !tiles || !aligned(s, 4) || !aligned(tiles, 4)) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_fp4_scales_to_tiles(s, R, F, tiles, static_cast<cudaStream_t>(stream),
                                                   dev));
}

fgq_status fgq_gemm_mxfp4(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                          const uint8_t* sB, void* C, int64_t ldc, int64_t M, int64_t N,
                          int64_t K, int out, void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || K % 128 != 0 || N % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (out != FGQ_OUT_F32 && out != FGQ_OUT_BF16) return FGQ_ERR_INVALID_ARG;
  if (M >= (int64_t{1} << 31) || N >= (int64_t{1} << 31) || K >= (int64_t{1} << 31))
    return FGQ_ERR_INVALID_ARG;
  if (M == 0) return FGQ_OK;
  if (!A || !sA || !B || !sB || !C) return FGQ_ERR_INVALID_ARG;
  const int64_t vec = (out == FGQ_OUT_F32) ? 4 : 8;
  if (ldc < N || ldc % vec != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(sA, 4) || !aligned(sB, 4))
    return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_gemm_mxf4(A, sA, B, sB, C, ldc, M, N, K, out == FGQ_OUT_BF16 ? 1 : 0,
                                         static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_gemm_nvfp4(const uint8_t* A, const uint8_t* sA, const float* gA,
                          const uint8_t* B, const uint8_t* sB, const float* gB, void* C,
                          int64_t ldc, int64_t M, int64_t N, int64_t K, int out, void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || K % 128 != 0 || N % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (out != FGQ_OUT_F32 && out != FGQ_OUT_BF16) return FGQ_ERR_INVALID_ARG;
  if (M >= (int64_t{1} << 31) || N >= (int64_t{1} << 31) || K >= (int64_t{1} << 31))
    return FGQ_ERR_INVALID_ARG;
  if (M == 0) return FGQ_OK;
  if (!A || !sA || !gA || !B || !sB || !gB || !C) return FGQ_ERR_INVALID_ARG;
  const int64_t vec = (out == FGQ_OUT_F32) ? 4 : 8;
  if (ldc < N || ldc % vec != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(sA, 4) ||
      !aligned(sB, 4) || !aligned(gA, 4) || !aligned(gB, 4))
    return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_gemm_nvf4(A, sA, gA, B, sB, gB, C, ldc, M, N, K,
                                         out == FGQ_OUT_BF16 ? 1 : 0,
                                         static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_gemm_mxfp4_tiled(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                                const uint8_t* sB, void* C, int64_t ldc, int64_t M, int64_t N,
                                int64_t K, int out, void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || K % 128 != 0 || N % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (out != FGQ_OUT_F32 && out != FGQ_OUT_BF16) return FGQ_ERR_INVALID_ARG;
  if (M >= (int64_t{1} << 31) || N >= (int64_t{1} << 31) || K >= (int64_t{1} << 31))
    return FGQ_ERR_INVALID_ARG;
  if (M == 0) return FGQ_OK;
  if (!A || !sA || !B || !sB || !C) return FGQ_ERR_INVALID_ARG;
  const int64_t vec = (out == FGQ_OUT_F32) ? 4 : 8;
  if (ldc < N || ldc % vec != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(sA, 16) ||
      !aligned(sB, 16))
    return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_gemm_mxf4_tiled(A, sA, B, sB, C, ldc, M, N, K,
                                               out == FGQ_OUT_BF16 ? 1 : 0,
                                               static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_gemm_nvfp4_tiled(const uint8_t* A, const uint8_t* sA, const float* gA,
                                const uint8_t* B, const uint8_t* sB, const float* gB, void* C,
                                int64_t ldc, int64_t M, int64_t N, int64_t K, int out,
                                void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || K % 128 != 0 || N % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (out != FGQ_OUT_F32 && out != FGQ_OUT_BF16) return FGQ_ERR_INVALID_ARG;
  if (M >= (int64_t{1} << 31) || N >= (int64_t{1} << 31) || K >= (int64_t{1} << 31))
    return FGQ_ERR_INVALID_ARG;
  if (M == 0) return FGQ_OK;
  if (!A || !sA || !gA || !B || !sB || !gB || !C) return FGQ_ERR_INVALID_ARG;
  const int64_t vec = (out == FGQ_OUT_F32) ? 4 : 8;
  if (ldc < N || ldc % vec != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(sA, 16) ||
      !aligned(sB, 16) || !aligned(gA, 4) || !aligned(gB, 4))
    return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_gemm_nvf4_tiled(A, sA, gA, B, sB, gB, C, ldc, M, N, K,
                                               out == FGQ_OUT_BF16 ? 1 : 0,
                                               static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_quant_operands_ue8m0_tiles(const void* x, int64_t M, int64_t K, int64_t ldx,
                                          uint8_t* xq, int64_t ldq, uint8_t* sA_tiles,
                                          const void* w, int64_t N, int64_t ldw, uint8_t* wq,
                                          uint8_t* sB_tiles, void* stream) {
  // the checks of fgq_quant_operands, with the code tiles in place of the
  // fp32 scale arrays
  if (M < 0 || K <= 0 || K % 128 != 0 || N <= 0 || N % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (!w || !wq || !sB_tiles) return FGQ_ERR_INVALID_ARG;
  if (ldw < N || ldw % 8 != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(wq, 16)) return FGQ_ERR_INVALID_ARG;
  if ((K / 128) > kMaxGroups / (N / 128)) return FGQ_ERR_INVALID_ARG;
  if (M > 0) {
    if (!x || !xq || !sA_tiles) return FGQ_ERR_INVALID_ARG;
    if (ldx < K || ldq < K || ldx % 8 != 0 || ldq % 16 != 0) return FGQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(xq, 16)) return FGQ_ERR_INVALID_ARG;
    if (M > kMaxGroups / (K / 128)) return FGQ_ERR_INVALID_ARG;
  }
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_quant_operands(x, M, K, ldx, xq, ldq,
                                              reinterpret_cast<float*>(sA_tiles), w, N, ldw, wq,
                                              reinterpret_cast<float*>(sB_tiles), FGQ_SCALE_UE8M0,
                                              static_cast<cudaStream_t>(stream), dev, true));
}

fgq_status fgq_ue8m0_scale_tiles_bytes(int64_t R, int64_t K, size_t* bytes) {
  if (!bytes || R < 0 || K <= 0 || K % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (R >= (int64_t{1} << 31) || K >= (int64_t{1} << 31)) return FGQ_ERR_INVALID_ARG;
  *bytes = static_cast<size_t>((R + 127) / 128) * static_cast<size_t>((K / 128 + 3) / 4) * 512u;
  return FGQ_OK;
}

fgq_status fgq_ue8m0_scale_tiles_act(const float* sA, int64_t M, int64_t K, uint8_t* tiles,
                                     void* stream) {
  if (M < 0 || K <= 0 || K % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (M >= (int64_t{1} << 31) || K >= (int64_t{1} << 31)) return FGQ_ERR_INVALID_ARG;
  if (M == 0) return FGQ_OK;
  if (!sA || !tiles || !aligned(sA, 4) || !aligned(tiles, 16)) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_ue8m0_scale_tiles(sA, M, K, 0, false, tiles,
                                                 static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_ue8m0_scale_tiles_weight(const float* sB, int64_t K, int64_t N, uint8_t* tiles,
                                        void* stream) {
  if (K <= 0 || N <= 0 || K % 128 != 0 || N % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (N >= (int64_t{1} << 31) || K >= (int64_t{1} << 31)) return FGQ_ERR_INVALID_ARG;
  if (!sB || !tiles || !aligned(sB, 4) || !aligned(tiles, 16)) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_ue8m0_scale_tiles(sB, N, K, N, true, tiles,
                                                 static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_gemm_fp8_ue8m0_tiled(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                                    const uint8_t* sB, void* C, int64_t ldc, int64_t M, int64_t N,
                                    int64_t K, int out, void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || K % 128 != 0 || N % 128 != 0) return FGQ_ERR_INVALID_ARG;
  if (out != FGQ_OUT_F32 && out != FGQ_OUT_BF16) return FGQ_ERR_INVALID_ARG;
  if (M >= (int64_t{1} << 31) || N >= (int64_t{1} << 31) || K >= (int64_t{1} << 31))
    return FGQ_ERR_INVALID_ARG;
  if (M == 0) return FGQ_OK;
  if (!A || !sA || !B || !sB || !C) return FGQ_ERR_INVALID_ARG;
  const int64_t vec = (out == FGQ_OUT_F32) ? 4 : 8;
  if (ldc < N || ldc % vec != 0) return FGQ_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(sA, 16) ||
      !aligned(sB, 16))
    return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_gemm_mx8_tiled(A, sA, B, sB, C, ldc, M, N, K,
                                              out == FGQ_OUT_BF16 ? 1 : 0,
                                              static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_gemm_splitk_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes) {
  if (!bytes || M < 0 || N <= 0 || K <= 0 || K % 128 != 0 || N % 128 != 0) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  *bytes = (M == 0 || M > kLowM) ? 0 : fgq::lowm_workspace_bytes(M, N, K, dev.sm_count);
  return FGQ_OK;
}

fgq_status fgq_gemm_fp8_blockscaled_splitk(const uint8_t* A, const float* sA, const uint8_t* B,
                                           const float* sB, void* C, int64_t ldc, int64_t M,
                                           int64_t N, int64_t K, int out, int mode,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  fgq_status st = check_gemm_args(A, sA, B, sB, C, ldc, M, N, K, out, mode);
  if (st != FGQ_OK || M == 0) return st;
  if (M > kLowM) return fgq_gemm_fp8_blockscaled_ex(A, sA, B, sB, C, ldc, M, N, K, out, mode, stream);
  fgq::DeviceInfo dev;
  st = get_device(&dev);
  if (st != FGQ_OK) return st;
  if (!workspace || !aligned(workspace, 16) ||
      workspace_bytes < fgq::lowm_workspace_bytes(M, N, K, dev.sm_count))
    return FGQ_ERR_INVALID_ARG;
  return from_cuda(fgq::launch_gemm_lowm(A, sA, B, sB, C, ldc, M, N, K, out == FGQ_OUT_BF16 ? 1 : 0,
                                         true, workspace, static_cast<cudaStream_t>(stream), dev));
}

fgq_status fgq_gemm_fp8_blockscaled(const uint8_t* A, const float* sA, const uint8_t* B,
                                    const float* sB, float* C, int64_t M, int64_t N, int64_t K,
                                    void* stream) {
  return fgq_gemm_fp8_blockscaled_ex(A, sA, B, sB, C, N, M, N, K, FGQ_OUT_F32, FGQ_SCALE_FP32,
                                     stream);
}

fgq_status fgq_gemm_fp8_blockscaled_splitk_noalloc(const uint8_t* A, const float* sA,
                                                   const uint8_t* B, const float* sB, void* C,
                                                   int64_t ldc, int64_t M, int64_t N, int64_t K,
                                                   int out, int mode, void* stream) {
  // Same checks and kernels as fgq_gemm_fp8_blockscaled_splitk, with the
  // library's fixed scratch array in place of a caller workspace.
  fgq_status st = check_gemm_args(A, sA, B, sB, C, ldc, M, N, K, out, mode);
  if (st != FGQ_OK || M == 0) return st;
  if (M > kLowM) return fgq_gemm_fp8_blockscaled_ex(A, sA, B, sB, C, ldc, M, N, K, out, mode, stream);
  fgq::DeviceInfo dev;
  st = get_device(&dev);
  if (st != FGQ_OK) return st;
  const size_t need = fgq::lowm_workspace_bytes(M, N, K, dev.sm_count);
  if (need > FGQ_NOALLOC_SCRATCH_BYTES) return FGQ_ERR_INVALID_ARG;  // beyond the fixed array
  void* scratch = nullptr;
  if (fgq::noalloc_scratch(dev, &scratch) != cudaSuccess) return FGQ_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t zero = fgq::lowm_workspace_zero_bytes(M, N, K, dev.sm_count);
  if (zero > 0) {
    // the stream-K counters and flags must start at zero; an earlier call
    // that gave up on a wait may have left them otherwise (they lie inside
    // `need`)
    if (cudaMemsetAsync(scratch, 0, zero, s) != cudaSuccess) return FGQ_ERR_CUDA;
  }
  return from_cuda(fgq::launch_gemm_lowm(A, sA, B, sB, C, ldc, M, N, K, out == FGQ_OUT_BF16 ? 1 : 0,
                                         true, scratch, s, dev));
}

const char* fgq_status_string(fgq_status status) {
  switch (status) {
    case FGQ_OK: return "ok";
    case FGQ_ERR_INVALID_ARG: return "invalid argument (null pointer, size, stride or alignment)";
    case FGQ_ERR_UNSUPPORTED: return "unsupported device (needs an sm_103 GPU)";
    case FGQ_ERR_CUDA: return "CUDA runtime error";
    case FGQ_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting (device error word set)";
  }
  return "unknown status";
}

fgq_status fgq_device_error(uint32_t* word, int clear) {
  if (!word) return FGQ_ERR_INVALID_ARG;
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return FGQ_ERR_CUDA;
  uint32_t w = 0;
  for (auto read : {fgq::read_device_error_gemm, fgq::read_device_error_lowm,
                    fgq::read_device_error_mx, fgq::read_device_error_mxf4}) {
    uint32_t u = 0;
    e = read(&u, clear != 0);
    if (e != cudaSuccess) return FGQ_ERR_CUDA;
    w |= u;
  }
  *word = w;
  return *word ? FGQ_ERR_DEVICE_TIMEOUT : FGQ_OK;
}

fgq_status fgq_selftest_wait_timeout(void* stream) {
  fgq::DeviceInfo dev;
  fgq_status st = get_device(&dev);
  if (st != FGQ_OK) return st;
  return from_cuda(fgq::launch_selftest_wait_timeout(static_cast<cudaStream_t>(stream)));
}

int fgq_version(void) { return 100; }

}  // extern "C"
