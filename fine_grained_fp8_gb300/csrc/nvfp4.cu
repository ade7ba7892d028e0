// NVFP4 quantization for sm_103a ("Fine-Grained FP8/FP4 Quantization",
// §NVFP4 Two-Level Scaling: a value is global_scale * block_scale * e2m1,
// with one E4M3 block scale per 16 consecutive elements of a row and one
// fp32 global scale per tensor; E2M1 values 0, 0.5, 1, 1.5, 2, 3, 4, 6).
//
// The page gives the dequantization only.  The encoder applies the FP8
// rule amax / 448 at both levels, with 6 the largest E2M1 value:
//   global   g = amax / 2688 over the whole tensor (2688 = 6 * 448), 1 for
//            an all-zero tensor;
//   block    s_b = E4M3(amax_b / (6 g)), round to nearest even, saturating;
//   element  q = E2M1(x / D), D = g * s_b (fp32), round to nearest even,
//            saturating at 6; a block whose D is 0 gets signed zeros.
// Every quotient is, or encodes exactly as, the IEEE fp32 quotient.
//
// Element quotients without a division: y = RN(x * RN(1/D)) has a relative
// error below 2^-23 + 2^-48, so it lies within 3 ulps of RN(x/D) (2 from
// the two roundings, 1/2 for RN(x/D) itself).  The bracket
// [RN(y (1 - 2^-20)), RN(y (1 + 2^-20))] reaches at least 7.5 ulps on each
// side of y, so it holds RN(x/D); E2M1 rounding is monotone, so when its
// two ends encode alike every value in it does, RN(x/D) included, and the
// code of y is the code of RN(x/D).  Otherwise (about 1 in 10^4 elements
// on ordinary data, every exact boundary value included) the lane's eight
// elements are recomputed with __fdiv_rn, as are blocks with a subnormal D.
// A host test replays this over every bf16 x against divisors that put
// quotients on and beside the E2M1 rounding boundaries.
//
// Two entry points: the global scale (a max reduction of |x| with one
// atomic per warp into the output word, then one thread turns it into g in
// place) and the block quantizer, which reads g from device memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "fgq_device.cuh"
#include "fgq_internal.h"
#include "fgq_quant.cuh"

namespace fgq {
namespace {

constexpr int kAmaxThreads = 256;

// Max of the bf16 magnitude bits (non-negative bf16 patterns order like
// their values) over 16-byte chunks of the rows; one atomicMax per warp.
template <bool DENSE>
__global__ void __launch_bounds__(kAmaxThreads)
    nvfp4_amax_kernel(const uint16_t* __restrict__ x, uint64_t chunks_per_row, uint64_t chunks,
                      int64_t ldx, unsigned int* __restrict__ out) {
  uint32_t m = 0;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kAmaxThreads;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * kAmaxThreads + threadIdx.x; i < chunks;
       i += stride) {
    const uint16_t* src;
    if (DENSE) {
      src = x + i * 8;
    } else {
      const uint64_t r = i / chunks_per_row, c = i - r * chunks_per_row;
      src = x + static_cast<int64_t>(r) * ldx + c * 8;
    }
    const uint32_t p = absmax_pairs(ld_stream_16(src));
    m = max(m, max(p & 0xFFFFu, p >> 16));
  }
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if ((threadIdx.x & 31u) == 0 && m != 0) atomicMax(out, m);
}

// g = amax / 2688 (1 for amax == 0), written over the magnitude bits.
__global__ void nvfp4_global_scale_kernel(float* g) {
  const uint32_t bits = *reinterpret_cast<const uint32_t*>(g);
  const float amax = __uint_as_float(bits << 16);
  *g = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
}

// E4M3 code of t >= 0: nearest, ties to even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_code(float t) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(h) : "f"(t));
  return h & 0xFFu;
}

// Value of a non-negative E4M3 code (0 .. 0x7E): m 2^-9 for exponent field
// 0, else (1 + m/8) 2^(e - 7).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = c >> 3, m = c & 7u;
  return e == 0 ? static_cast<float>(m) * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// One block of 16 per two lanes (8 elements, 16 bytes each), 16 blocks per
// warp per round, kNvRounds rounds of loads in flight.
constexpr int kNvThreads = 256;
constexpr int kNvRounds = 2;

// Byte of factor f of row r in the tiled FP4 scale layout (F factor bytes a
// row, F % 4 == 0): 512-byte tiles of 128 rows x 4 factor bytes, tile
// (r / 128, f / 4); in a tile, row r at 16 (r % 32) + 4 ((r % 128) / 32),
// the byte at + f % 4.
__device__ __forceinline__ uint64_t nv_tile_offset(uint32_t r, uint32_t f, uint32_t F) {
  return (static_cast<uint64_t>(r >> 7) * (F >> 2) + (f >> 2)) * 512u + (r & 31u) * 16u +
         ((r >> 5) & 3u) * 4u + (f & 3u);
}

template <bool DENSE, bool TILED>
__global__ void __launch_bounds__(kNvThreads)
    quant_nvfp4_1x16_kernel(const uint16_t* __restrict__ x, uint32_t kb, uint32_t blocks,
                            int64_t ldx, const float* __restrict__ gptr, uint8_t* __restrict__ xq,
                            uint8_t* __restrict__ sx) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t sub = lane >> 1, l2 = lane & 1u;
  const uint32_t warp = (blockIdx.x * kNvThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kNvThreads) >> 5;
  constexpr uint32_t kPerWarp = 16 * kNvRounds;
  const float g = __ldg(gptr);
  const float d6 = __fmul_rn(6.0f, g);
  // Tiled scales: the row and block index of `base`, advanced by the loop's
  // stride without a division per iteration.
  const uint32_t step = nwarps * kPerWarp;
  const uint32_t step_r = TILED ? step / kb : 0u, step_f = TILED ? step - step_r * kb : 0u;
  uint32_t r_base = TILED ? (warp * kPerWarp) / kb : 0u;
  uint32_t f_base = TILED ? warp * kPerWarp - r_base * kb : 0u;
  for (uint32_t base = warp * kPerWarp; base < blocks; base += step) {
    uint4 v[kNvRounds];
    uint32_t b[kNvRounds];
#pragma unroll
    for (int u = 0; u < kNvRounds; ++u) {
      b[u] = base + 16 * u + sub;
      v[u] = make_uint4(0, 0, 0, 0);
      if (b[u] < blocks) {
        const uint16_t* src;
        if (DENSE) {
          src = x + static_cast<uint64_t>(b[u]) * 16;
        } else {
          const uint32_t r = b[u] / kb, c = b[u] - r * kb;
          src = x + static_cast<int64_t>(r) * ldx + c * 16;
        }
        v[u] = ld_stream_16(src + 8 * l2);
      }
    }
#pragma unroll
    for (int u = 0; u < kNvRounds; ++u) {
      uint32_t mx = absmax_pairs(v[u]);
      mx = __vmaxu2(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      const float amax = __uint_as_float(max(mx & 0xFFFFu, mx >> 16) << 16);
      const uint32_t sc = e4m3_code(__fdiv_rn(amax, d6));
      const float d = __fmul_rn(g, e4m3_value(sc));
      if (b[u] < blocks) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t packed = 0;
        if (d == 0.0f) {
          // signed zeros: code 8 where the bf16 sign bit is set
#pragma unroll
          for (int p = 0; p < 4; ++p)
            packed |= (((w[p] >> 12) & 0x8u) | ((w[p] >> 24) & 0x80u)) << (8 * p);
        } else {
          float ylo[8], yhi[8];
          const float r = __frcp_rn(d);
          const float2 r2 = make_float2(r, r);
          const float2 lo2 = make_float2(1.0f - 0x1p-20f, 1.0f - 0x1p-20f);
          const float2 hi2 = make_float2(1.0f + 0x1p-20f, 1.0f + 0x1p-20f);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const float2 q = mul2(bf16x2_to_f32x2(w[p]), r2);
            const float2 ql = mul2(q, lo2), qh = mul2(q, hi2);
            ylo[2 * p] = ql.x;
            ylo[2 * p + 1] = ql.y;
            yhi[2 * p] = qh.x;
            yhi[2 * p + 1] = qh.y;
          }
          // the two ends of the bracket; equal codes are the code of y too
          packed = cvt_e2m1x8(ylo);
          if (!(d >= 0x1p-126f) || packed != cvt_e2m1x8(yhi)) {
            // rare: recompute the lane's eight quotients exactly
            float y[8];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const float2 f = bf16x2_to_f32x2(w[p]);
              y[2 * p] = __fdiv_rn(f.x, d);
              y[2 * p + 1] = __fdiv_rn(f.y, d);
            }
            packed = cvt_e2m1x8(y);
          }
        }
        // row-major [R, K/2]: block b covers bytes 8 b .. 8 b + 7
        *reinterpret_cast<uint32_t*>(xq + static_cast<uint64_t>(b[u]) * 8 + 4 * l2) = packed;
        if (!TILED && l2 == 0) sx[b[u]] = static_cast<uint8_t>(sc);
      }
      if (TILED) {
        // Four consecutive blocks (subs 4j .. 4j + 3) are one 4-byte cell of
        // one row (kb % 4 == 0 and the blocks start at a multiple of 4): the
        // cell's first lane gathers the codes and stores the cell whole.
        const uint32_t c1 = __shfl_down_sync(0xFFFFFFFFu, sc, 2);
        const uint32_t c2 = __shfl_down_sync(0xFFFFFFFFu, sc, 4);
        const uint32_t c3 = __shfl_down_sync(0xFFFFFFFFu, sc, 6);
        if ((lane & 7u) == 0 && b[u] < blocks) {
          uint32_t r = r_base, f = f_base + 16 * u + (lane >> 1);
          while (f >= kb) {  // at most 28 / kb + 1 times
            f -= kb;
            ++r;
          }
          *reinterpret_cast<uint32_t*>(sx + nv_tile_offset(r, f, kb)) =
              sc | (c1 << 8) | (c2 << 16) | (c3 << 24);
        }
      }
    }
    if (TILED) {
      r_base += step_r;
      f_base += step_f;
      if (f_base >= kb) {
        f_base -= kb;
        ++r_base;
      }
    }
  }
}

}  // namespace

cudaError_t launch_nvfp4_global_scale(const void* x, int64_t R, int64_t K, int64_t ldx, float* g,
                                      cudaStream_t stream, const DeviceInfo& dev) {
  cudaError_t e = cudaMemsetAsync(g, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const uint64_t per_row = static_cast<uint64_t>(K / 8);
  const uint64_t chunks = static_cast<uint64_t>(R) * per_row;
  if (chunks > 0) {
    const bool dense = ldx == K;
    auto k = dense ? nvfp4_amax_kernel<true> : nvfp4_amax_kernel<false>;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kAmaxThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const uint64_t needed = (chunks + kAmaxThreads - 1) / kAmaxThreads;
    uint64_t grid = static_cast<uint64_t>(dev.sm_count) * static_cast<uint64_t>(per_sm);
    if (grid > needed) grid = needed;
    k<<<static_cast<unsigned>(grid), kAmaxThreads, 0, stream>>>(
        static_cast<const uint16_t*>(x), per_row, chunks, ldx, reinterpret_cast<unsigned int*>(g));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  nvfp4_global_scale_kernel<<<1, 1, 0, stream>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_quant_nvfp4_1x16(const void* x, int64_t R, int64_t K, int64_t ldx,
                                    const float* g, uint8_t* xq, uint8_t* sx, bool tiled,
                                    cudaStream_t stream, const DeviceInfo& dev) {
  const uint32_t kb = static_cast<uint32_t>(K / 16);
  const uint32_t blocks = static_cast<uint32_t>(R * (K / 16));
  if (blocks == 0) return cudaSuccess;
  const bool dense = ldx == K;
  auto k = dense ? (tiled ? quant_nvfp4_1x16_kernel<true, true> : quant_nvfp4_1x16_kernel<true, false>)
                 : (tiled ? quant_nvfp4_1x16_kernel<false, true> : quant_nvfp4_1x16_kernel<false, false>);
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kNvThreads, 0);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const uint32_t per_block = (kNvThreads / 32) * 16 * kNvRounds;
  const uint32_t needed = (blocks + per_block - 1) / per_block;
  uint32_t grid = static_cast<uint32_t>(dev.sm_count) * static_cast<uint32_t>(per_sm);
  if (grid > needed) grid = needed;
  k<<<grid, kNvThreads, 0, stream>>>(static_cast<const uint16_t*>(x), kb, blocks, ldx, g, xq, sx);
  return cudaGetLastError();
}

// Row-major FP4 block scales [R, F] (F % 4 == 0) into the tiled layout:
// one 4-byte cell (four factor bytes of one row) per thread, read and
// written whole (a cell's four bytes stay together in the tiled layout).
__global__ void __launch_bounds__(256)
    fp4_scales_to_tiles_kernel(const uint32_t* __restrict__ s, uint32_t cells_per_row,
                               uint64_t cells, uint32_t* __restrict__ tiles) {
  for (uint64_t i = blockIdx.x * 256ull + threadIdx.x; i < cells; i += gridDim.x * 256ull) {
    const uint32_t r = static_cast<uint32_t>(i / cells_per_row);
    const uint32_t c = static_cast<uint32_t>(i - static_cast<uint64_t>(r) * cells_per_row);
    const uint64_t word = (static_cast<uint64_t>(r >> 7) * cells_per_row + c) * 128u +
                          (r & 31u) * 4u + ((r >> 5) & 3u);
    tiles[word] = __ldg(s + i);
  }
}

cudaError_t launch_fp4_scales_to_tiles(const uint8_t* s, int64_t R, int64_t F, uint8_t* tiles,
                                       cudaStream_t stream, const DeviceInfo& dev) {
  const uint64_t cells = static_cast<uint64_t>(R) * static_cast<uint64_t>(F / 4);
  if (cells == 0) return cudaSuccess;
  uint64_t grid = (cells + 255) / 256;
  const uint64_t cap = static_cast<uint64_t>(dev.sm_count) * 8;
  if (grid > cap) grid = cap;
  fp4_scales_to_tiles_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      reinterpret_cast<const uint32_t*>(s), static_cast<uint32_t>(F / 4), cells,
      reinterpret_cast<uint32_t*>(tiles));
  return cudaGetLastError();
}

}  // namespace fgq
