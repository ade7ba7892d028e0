// Internal declarations shared by the translation units of libfgq.so.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

// Bits of the device error word: which wait gave up.
#define FGQ_DEVERR_PRODUCER_EMPTY 0x1u  // TMA producer waiting for a free stage
#define FGQ_DEVERR_MMA_FULL 0x2u        // MMA issuer waiting for a loaded stage
#define FGQ_DEVERR_MMA_TMEM 0x4u        // MMA issuer waiting for a drained TMEM buffer
#define FGQ_DEVERR_EPI_TMEM 0x8u        // epilogue waiting for a finished partial
#define FGQ_DEVERR_DRAIN 0x10u          // unwinding: waiting for copies in flight

namespace fgq {

struct DeviceInfo {
  int device;
  int sm_count;
  int cc_major, cc_minor;
  size_t smem_optin;
};

// Cached per-device properties; returns cudaErrorNoDevice etc. on failure.
cudaError_t device_info(DeviceInfo* out);

cudaError_t launch_quant_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx,
                                   uint8_t* xq, int64_t ldq, float* sx, int mode,
                                   cudaStream_t stream, const DeviceInfo& dev);

cudaError_t launch_quant_w_128x128(const void* w, int64_t K, int64_t N, int64_t ldw,
                                   uint8_t* wq, float* sw, int mode, cudaStream_t stream,
                                   const DeviceInfo& dev);

cudaError_t launch_gemm_fp8_blockscaled(const uint8_t* A, const float* sA, const uint8_t* B,
                                        const float* sB, void* C, int64_t ldc, int64_t M,
                                        int64_t N, int64_t K, int out_bf16, int mode,
                                        cudaStream_t stream, const DeviceInfo& dev);

cudaError_t read_device_error(uint32_t* word, bool clear);

}  // namespace fgq
