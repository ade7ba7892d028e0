// Internal declarations shared by the translation units of libfgq.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

// Bits of the device error word: which wait gave up.
#define FGQ_DEVERR_PRODUCER_EMPTY 0x1u  // TMA producer waiting for a free stage
#define FGQ_DEVERR_MMA_FULL 0x2u        // MMA issuer waiting for a loaded stage
#define FGQ_DEVERR_MMA_TMEM 0x4u        // MMA issuer waiting for a drained TMEM buffer
#define FGQ_DEVERR_EPI_TMEM 0x8u        // epilogue waiting for a finished partial
#define FGQ_DEVERR_DRAIN 0x10u          // unwinding: waiting for copies in flight
#define FGQ_DEVERR_SF_SLOT 0x20u        // scale-factor writer waiting for a free TMEM slot
#define FGQ_DEVERR_MMA_SF 0x40u         // MMA issuer waiting for scale factors in TMEM
#define FGQ_DEVERR_SELFTEST 0x80u       // the self-test's wait on a barrier nothing completes
#define FGQ_DEVERR_SK_FLAG 0x100u       // stream-K fix-up waiting for another CTA's partial tile

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

cudaError_t launch_quant_act_128x1(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xqt,
                                   float* sxt, int mode, cudaStream_t stream,
                                   const DeviceInfo& dev);

// MXFP4 1x32 quantizer; with `tiled` the scales go out in the tiled FP4
// scale layout (K % 128 == 0) instead of row-major [R, K/32].
cudaError_t launch_quant_mxfp4_1x32(const void* x, int64_t R, int64_t K, int64_t ldx, uint8_t* xq,
                                    uint8_t* sx, bool tiled, cudaStream_t stream,
                                    const DeviceInfo& dev);

cudaError_t launch_quant_w_128x128(const void* w, int64_t K, int64_t N, int64_t ldw,
                                   uint8_t* wq, float* sw, int mode, cudaStream_t stream,
                                   const DeviceInfo& dev);

// Both operands of a GEMM in one launch: X [M, K] 1x128 and W [K, N]
// 128x128, the same codes and scales as the two launches above.
// (code_tiles: UE8M0 mode with the scales written as the UE8M0 code tiles
// of the tiled-scale FP8 GEMM, sx and sw then being the two tile buffers.)
cudaError_t launch_quant_operands(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                  int64_t ldq, float* sx, const void* w, int64_t N, int64_t ldw,
                                  uint8_t* wq, float* sw, int mode, cudaStream_t stream,
                                  const DeviceInfo& dev, bool code_tiles = false);

cudaError_t launch_gemm_fp8_blockscaled(const uint8_t* A, const float* sA, const uint8_t* B,
                                        const float* sB, void* C, int64_t ldc, int64_t M,
                                        int64_t N, int64_t K, int out_bf16, int mode,
                                        cudaStream_t stream, const DeviceInfo& dev);

// Power-of-two (UE8M0) scales folded into the tensor core: same arguments
// and result as launch_gemm_fp8_blockscaled for scales that are powers of
// two.
cudaError_t launch_gemm_mx(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                           void* C, int64_t ldc, int64_t M, int64_t N, int64_t K, int out_bf16,
                           cudaStream_t stream, const DeviceInfo& dev);

// Diagnostic: one warp waits, with the kernels' bounded wait, on a barrier
// that nothing completes; the wait gives up and records FGQ_DEVERR_SELFTEST.
cudaError_t launch_selftest_wait_timeout(cudaStream_t stream);

// MXFP4 GEMM: A codes [M, K/2], B codes [N, K/2] (E2M1 pairs), UE8M0 codes
// sA [M, K/32], sB [N, K/32]; K % 128 == 0, N % 128 == 0.
cudaError_t launch_gemm_mxf4(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                             const uint8_t* sB, void* C, int64_t ldc, int64_t M, int64_t N,
                             int64_t K, int out_bf16, cudaStream_t stream, const DeviceInfo& dev);
cudaError_t launch_gemm_nvf4(const uint8_t* A, const uint8_t* sA, const float* ga,
                             const uint8_t* B, const uint8_t* sB, const float* gb, void* C,
                             int64_t ldc, int64_t M, int64_t N, int64_t K, int out_bf16,
                             cudaStream_t stream, const DeviceInfo& dev);
// The same two GEMMs on block scales in the tiled FP4 scale layout, loaded
// by the tensor-map engine (16-byte aligned scale tiles).
cudaError_t launch_gemm_mxf4_tiled(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                                   const uint8_t* sB, void* C, int64_t ldc, int64_t M, int64_t N,
                                   int64_t K, int out_bf16, cudaStream_t stream,
                                   const DeviceInfo& dev);
cudaError_t launch_gemm_nvf4_tiled(const uint8_t* A, const uint8_t* sA, const float* ga,
                                   const uint8_t* B, const uint8_t* sB, const float* gb, void* C,
                                   int64_t ldc, int64_t M, int64_t N, int64_t K, int out_bf16,
                                   cudaStream_t stream, const DeviceInfo& dev);
// FP8 GEMM with power-of-two scales given as UE8M0 code tiles (the tiled
// FP4 scale layout with F = K/128 padded to a multiple of 4): activation
// codes per row, weight codes per column of the transposed weight.
cudaError_t launch_gemm_mx8_tiled(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                                  const uint8_t* sB, void* C, int64_t ldc, int64_t M, int64_t N,
                                  int64_t K, int out_bf16, cudaStream_t stream,
                                  const DeviceInfo& dev);
// Those code tiles from fp32 power-of-two scales: activation sA [R, K/128]
// (weight = false) or weight sB [K/128, N/128] for R = N rows (weight = true).
cudaError_t launch_ue8m0_scale_tiles(const float* s, int64_t R, int64_t K, int64_t N, bool weight,
                                     uint8_t* tiles, cudaStream_t stream, const DeviceInfo& dev);
// Row-major FP4 block scales [R, F] (F % 4 == 0) into the tiled layout.
cudaError_t launch_fp4_scales_to_tiles(const uint8_t* s, int64_t R, int64_t F, uint8_t* tiles,
                                       cudaStream_t stream, const DeviceInfo& dev);
cudaError_t launch_nvfp4_global_scale(const void* x, int64_t R, int64_t K, int64_t ldx, float* g,
                                      cudaStream_t stream, const DeviceInfo& dev);
// NVFP4 1x16 quantizer; with `tiled` the scales go out in the tiled FP4
// scale layout (K % 64 == 0) instead of row-major [R, K/16].
cudaError_t launch_quant_nvfp4_1x16(const void* x, int64_t R, int64_t K, int64_t ldx,
                                    const float* g, uint8_t* xq, uint8_t* sx, bool tiled,
                                    cudaStream_t stream, const DeviceInfo& dev);

// Each kernel translation unit keeps its own device error word; these read
// (and optionally clear) one unit's word.
cudaError_t read_device_error_gemm(uint32_t* word, bool clear);
cudaError_t read_device_error_lowm(uint32_t* word, bool clear);
cudaError_t read_device_error_mx(uint32_t* word, bool clear);
cudaError_t read_device_error_mxf4(uint32_t* word, bool clear);

// TMA descriptor of a K-major E4M3 operand [rows, K] with a 128 (K) x
// box_rows box, 128-byte swizzle, zero fill outside the tensor.
bool make_k_major_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows);

// TMA descriptor of FP4 scale tiles in the tiled layout: `tiles` 512-byte
// tiles, read box_tiles consecutive tiles at a time (no swizzle, zero fill
// past the end).
bool make_scale_tile_map(CUtensorMap* map, const void* base, int64_t tiles, int box_tiles);

// Low-M GEMM that quantizes bf16 A (1x128, scale mode `mode`) in the kernel
// and keeps all of it in shared memory: M <= 32 and K small enough for
// that (lowm_fused_fits); no split.
bool lowm_fused_fits(int64_t M, int64_t K);
cudaError_t launch_gemm_lowm_fused(const void* a16, int64_t lda, const uint8_t* B, const float* sB,
                                   void* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                   int out_bf16, int mode, cudaStream_t stream,
                                   const DeviceInfo& dev);

// Bytes of the fixed scratch array behind fgq_gemm_fp8_blockscaled_splitk_noalloc.
#ifndef FGQ_NOALLOC_SCRATCH_BYTES
#define FGQ_NOALLOC_SCRATCH_BYTES (16u << 20)
#endif

// Device address of that array on the current device (looked up on the
// first call for each device).
cudaError_t noalloc_scratch(const DeviceInfo& dev, void** ptr);

// Low-M GEMM (M <= 256).  With stream_k, the tiles left after the last
// whole wave are shared out by K chunks (stream-K) and the workspace holds
// the partial tiles: lowm_workspace_bytes of it, whose first
// lowm_workspace_zero_bytes must be zero before a call (every completed call
// leaves them zero).  Without, whole tiles only and no workspace.
size_t lowm_workspace_bytes(int64_t M, int64_t N, int64_t K, int sm_count);
size_t lowm_workspace_zero_bytes(int64_t M, int64_t N, int64_t K, int sm_count);
cudaError_t launch_gemm_lowm(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                             void* C, int64_t ldc, int64_t M, int64_t N, int64_t K, int out_bf16,
                             bool stream_k, void* workspace, cudaStream_t stream,
                             const DeviceInfo& dev);

}  // namespace fgq
