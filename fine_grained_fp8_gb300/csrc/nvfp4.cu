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
// Element quotients without a division: y = RN(x * r), r the hardware
// reciprocal approximation of D (at most 1 ulp from 1/D for 2^-126 <= D <=
// 2^125), has a relative error below 2^-22, so it lies within 4 ulps of
// RN(x/D).  The bracket [RN(y (1 - 2^-20)), RN(y (1 + 2^-20))] reaches at
// least 7.5 ulps on each side of y, so it holds RN(x/D); E2M1 rounding is
// monotone, so when its two ends encode alike every value in it does,
// RN(x/D) included, and the code of y is the code of RN(x/D).  Otherwise
// (about 1 in 10^4 elements on ordinary data, every exact boundary value
// included) those eight elements are recomputed with __fdiv_rn, as are
// blocks with D outside that range.  The block scale E4M3(RN(amax /
// d6)) takes the same route with t = RN(amax * RN(1/d6)).  A host test
// replays both over every bf16 x (amax) against divisors that put
// quotients on and beside the rounding boundaries, for every reciprocal
// within 1 ulp of the true one.
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
// Each thread has kAmaxLoads independent 16-byte loads in flight per round.
constexpr int kAmaxLoads = 4;

template <bool DENSE>
__device__ __forceinline__ const uint16_t* amax_chunk(const uint16_t* x, uint64_t i,
                                                      uint64_t chunks_per_row, int64_t ldx) {
  if (DENSE) return x + i * 8;
  const uint64_t r = i / chunks_per_row, c = i - r * chunks_per_row;
  return x + static_cast<int64_t>(r) * ldx + c * 8;
}

template <bool DENSE>
__global__ void __launch_bounds__(kAmaxThreads)
    nvfp4_amax_kernel(const uint16_t* __restrict__ x, uint64_t chunks_per_row, uint64_t chunks,
                      int64_t ldx, unsigned int* __restrict__ out) {
  uint32_t m = 0;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kAmaxThreads;
  uint64_t i = static_cast<uint64_t>(blockIdx.x) * kAmaxThreads + threadIdx.x;
  for (; i + (kAmaxLoads - 1) * stride < chunks; i += kAmaxLoads * stride) {
    uint4 v[kAmaxLoads];
#pragma unroll
    for (int u = 0; u < kAmaxLoads; ++u)
      v[u] = ld_stream_16(amax_chunk<DENSE>(x, i + u * stride, chunks_per_row, ldx));
#pragma unroll
    for (int u = 0; u < kAmaxLoads; ++u) {
      const uint32_t p = absmax_pairs(v[u]);
      m = max(m, max(p & 0xFFFFu, p >> 16));
    }
  }
  for (; i < chunks; i += stride) {
    const uint32_t p = absmax_pairs(ld_stream_16(amax_chunk<DENSE>(x, i, chunks_per_row, ldx)));
    m = max(m, max(p & 0xFFFFu, p >> 16));
  }
  // One atomic per CTA, and none where the word already holds as much: it
  // only grows, so a read that is stale is never larger than the truth.
  // (One atomic per warp on the one word: 45.7 us on the quantize-bandwidth
  // activations.)
  __shared__ uint32_t wmax[kAmaxThreads / 32];
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if ((threadIdx.x & 31u) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0;
#pragma unroll
    for (int w = 0; w < kAmaxThreads / 32; ++w) b = max(b, wmax[w]);
    if (b != 0 && b > *reinterpret_cast<volatile unsigned int*>(out)) atomicMax(out, b);
  }
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

// Value of a non-negative E4M3 code (0 .. 0x7E), through the exact
// E4M3 -> f16 conversion (every E4M3 value is an f16 value).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(c)));
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(static_cast<uint16_t>(h2 & 0xFFFFu)));
  return f;
}

// E4M3 codes of two non-negative floats (lo in byte 0, hi in byte 1).
__device__ __forceinline__ uint32_t e4m3_code2(float lo, float hi) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
  return h;
}

// The hardware reciprocal approximation (at most 1 ulp from 1/d for normal
// d and 1/d; subnormal results flush to zero).
__device__ __forceinline__ float rcp_approx(float d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
  return r;
}

// Block scale E4M3(RN(amax / d6)): from t = RN(amax * r6) (r6 = RN(1/d6))
// when the codes of t (1 -+ 2^-20) agree, else from the IEEE quotient.
__device__ __forceinline__ uint32_t nv_scale_code(float amax, float d6, float r6, bool fast) {
  if (fast) {
    const float t = amax * r6;
    const uint32_t c2 = e4m3_code2(t * (1.0f - 0x1p-20f), t * (1.0f + 0x1p-20f));
    if ((c2 & 0xFFu) == (c2 >> 8)) return c2 & 0xFFu;
  }
  return e4m3_code(__fdiv_rn(amax, d6));
}

// One block of 16 per thread (two 16-byte loads), 32 consecutive blocks per
// warp per round, kNvRounds rounds of loads in flight.  A thread holds its
// whole block, so the block's amax needs no shuffle and its scale code,
// divisor and reciprocal are formed once for 16 elements: 57.4 us on the
// quantize-bandwidth activations, against 68.9 us with two lanes a block.
constexpr int kNvThreads = 256;
constexpr int kNvRounds = 2;

// One block of 16 elements (v0: elements 0-7, v1: 8-15) under the global
// scale g (d6 = fl32(6 g), r6 = RN(1 / d6), fast6 = d6 in the reciprocal's
// range): the block's E4M3 scale code, and its 16 E2M1 codes as two words
// (elements 0-7 in out[0], 8-15 in out[1]).
__device__ __forceinline__ uint32_t nv_block(const uint4& v0, const uint4& v1, float g, float d6,
                                             float r6, bool fast6, uint32_t (&out)[2]) {
  const uint32_t mx = __vmaxu2(absmax_pairs(v0), absmax_pairs(v1));
  const float amax = __uint_as_float(max(mx & 0xFFFFu, mx >> 16) << 16);
  const uint32_t sc = nv_scale_code(amax, d6, r6, fast6);
  const float d = __fmul_rn(g, e4m3_value(sc));
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  if (d == 0.0f) {
    // signed zeros: code 8 where the bf16 sign bit is set
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      out[h] = 0;
#pragma unroll
      for (int p = 0; p < 4; ++p)
        out[h] |= (((w[4 * h + p] >> 12) & 0x8u) | ((w[4 * h + p] >> 24) & 0x80u)) << (8 * p);
    }
    return sc;
  }
  const float r = rcp_approx(d);
  const float2 r2 = make_float2(r, r);
  const float2 lo2 = make_float2(1.0f - 0x1p-20f, 1.0f - 0x1p-20f);
  const float2 hi2 = make_float2(1.0f + 0x1p-20f, 1.0f + 0x1p-20f);
  const bool in_range = d >= 0x1p-126f && d <= 0x1p125f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float ylo[8], yhi[8];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 q = mul2(bf16x2_to_f32x2(w[4 * h + p]), r2);
      const float2 ql = mul2(q, lo2), qh = mul2(q, hi2);
      ylo[2 * p] = ql.x;
      ylo[2 * p + 1] = ql.y;
      yhi[2 * p] = qh.x;
      yhi[2 * p + 1] = qh.y;
    }
    // the two ends of the bracket; equal codes are the code of y too
    uint32_t packed = cvt_e2m1x8(ylo);
    if (!in_range || packed != cvt_e2m1x8(yhi)) {
      // rare: recompute these eight quotients exactly
      float y[8];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float2 f = bf16x2_to_f32x2(w[4 * h + p]);
        y[2 * p] = __fdiv_rn(f.x, d);
        y[2 * p + 1] = __fdiv_rn(f.y, d);
      }
      packed = cvt_e2m1x8(y);
    }
    out[h] = packed;
  }
  return sc;
}

// Block b (row b / kb, block b % kb of the row) of x, as two 16-byte loads.
template <bool DENSE>
__device__ __forceinline__ void nv_load(const uint16_t* x, uint32_t b, uint32_t kb, int64_t ldx,
                                        uint4& v0, uint4& v1) {
  const uint16_t* src;
  if (DENSE) {
    src = x + static_cast<uint64_t>(b) * 16;
  } else {
    const uint32_t r = b / kb, c = b - r * kb;
    src = x + static_cast<int64_t>(r) * ldx + c * 16;
  }
  v0 = ld_stream_16(src);
  v1 = ld_stream_16(src + 8);
}

template <bool DENSE>
__global__ void __launch_bounds__(kNvThreads)
    quant_nvfp4_1x16_kernel(const uint16_t* __restrict__ x, uint32_t kb, uint32_t blocks,
                            int64_t ldx, const float* __restrict__ gptr, uint8_t* __restrict__ xq,
                            uint8_t* __restrict__ sx) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = (blockIdx.x * kNvThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kNvThreads) >> 5;
  constexpr uint32_t kPerWarp = 32 * kNvRounds;
  const float g = __ldg(gptr);
  const float d6 = __fmul_rn(6.0f, g);
  const bool fast6 = d6 >= 0x1p-125f && d6 <= 0x1p125f;
  const float r6 = __frcp_rn(d6);
  for (uint32_t base = warp * kPerWarp; base < blocks; base += nwarps * kPerWarp) {
    uint4 v[kNvRounds][2];
    uint32_t b[kNvRounds];
#pragma unroll
    for (int u = 0; u < kNvRounds; ++u) {
      b[u] = base + 32 * u + lane;
      v[u][0] = v[u][1] = make_uint4(0, 0, 0, 0);
      if (b[u] < blocks) nv_load<DENSE>(x, b[u], kb, ldx, v[u][0], v[u][1]);
    }
#pragma unroll
    for (int u = 0; u < kNvRounds; ++u) {
      uint32_t packed[2];
      const uint32_t sc = nv_block(v[u][0], v[u][1], g, d6, r6, fast6, packed);
      if (b[u] < blocks) {
        // row-major [R, K/2]: block b covers bytes 8 b .. 8 b + 7
        uint32_t* dst = reinterpret_cast<uint32_t*>(xq + static_cast<uint64_t>(b[u]) * 8);
        dst[0] = packed[0];
        dst[1] = packed[1];
        sx[b[u]] = static_cast<uint8_t>(sc);
      }
    }
  }
}

// The same quantizer with the scales in the tiled FP4 layout (512-byte tiles
// of 128 rows x 4 factor bytes; 16-byte tile row i holds the cells of rows
// 32 j + i, j = 0..3).  A warp's unit is 16-byte row i of eight neighbouring
// tiles: four rounds, round j quantizing 32 blocks (1 KB of x) of row
// 32 j + i, one a lane, with two rounds' loads in flight at a time (56
// registers; all four at once took 74 and measured 1.5% slower); lanes 0,
// 4, .., 28 then each gather tile row i of one cell (the scale codes of
// their own and the next three lanes' blocks) and store it whole.  Rows
// past R read as zeros and give padding codes.
__global__ void __launch_bounds__(kNvThreads)
    quant_nvfp4_1x16_tiled_kernel(const uint16_t* __restrict__ x, uint32_t R, uint32_t kb,
                                  int64_t ldx, const float* __restrict__ gptr,
                                  uint8_t* __restrict__ xq, uint8_t* __restrict__ st) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = (blockIdx.x * kNvThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kNvThreads) >> 5;
  const float g = __ldg(gptr);
  const float d6 = __fmul_rn(6.0f, g);
  const bool fast6 = d6 >= 0x1p-125f && d6 <= 0x1p125f;
  const float r6 = __frcp_rn(d6);
  const uint32_t cpr = kb >> 2;            // cells (tiles) per 128-row tile
  const uint32_t octs = (cpr + 7u) >> 3;   // groups of eight cells per 128-row tile
  const uint32_t units = ((R + 127u) >> 7) * octs * 32u;
  for (uint32_t unit = warp; unit < units; unit += nwarps) {
    const uint32_t i = unit & 31u, t = unit >> 5;
    const uint32_t rb = t / octs, co = t - rb * octs;
    const uint32_t blk = 32u * co + lane;  // this lane's block within the row
    const bool col_ok = blk < kb;          // the last cells of the eight may not exist
    uint32_t cell[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // rows 32 (2 h) + i and 32 (2 h + 1) + i
      uint4 v[2][2];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const uint32_t row = rb * 128u + 32u * (2 * h + jj) + i;
        v[jj][0] = v[jj][1] = make_uint4(0, 0, 0, 0);
        if (row < R && col_ok) {
          const uint16_t* src = x + static_cast<int64_t>(row) * ldx + blk * 16u;
          v[jj][0] = ld_stream_16(src);
          v[jj][1] = ld_stream_16(src + 8);
        }
      }
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const uint32_t row = rb * 128u + 32u * (2 * h + jj) + i;
        uint32_t packed[2];
        const uint32_t sc = nv_block(v[jj][0], v[jj][1], g, d6, r6, fast6, packed);
        if (row < R && col_ok) {
          uint32_t* dst = reinterpret_cast<uint32_t*>(xq + static_cast<uint64_t>(row) * (8u * kb) +
                                                      blk * 8u);
          dst[0] = packed[0];
          dst[1] = packed[1];
        }
        // lanes 4 q: the cell (blocks in lanes +0 .. +3)
        const uint32_t c1 = __shfl_down_sync(0xFFFFFFFFu, sc, 1);
        const uint32_t c2 = __shfl_down_sync(0xFFFFFFFFu, sc, 2);
        const uint32_t c3 = __shfl_down_sync(0xFFFFFFFFu, sc, 3);
        cell[2 * h + jj] = sc | (c1 << 8) | (c2 << 16) | (c3 << 24);
      }
    }
    if ((lane & 3u) == 0 && col_ok)
      *reinterpret_cast<uint4*>(st + (static_cast<uint64_t>(rb) * cpr + 8u * co + (lane >> 2)) * 512u +
                                16u * i) = make_uint4(cell[0], cell[1], cell[2], cell[3]);
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
  if (tiled) {
    // one warp per 16-byte row of eight neighbouring tiles (128 blocks)
    const uint32_t units = static_cast<uint32_t>((R + 127) / 128) * ((kb / 4 + 7) / 8) * 32u;
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, quant_nvfp4_1x16_tiled_kernel, kNvThreads, 0);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    const uint32_t per_block = kNvThreads / 32;
    const uint32_t needed = (units + per_block - 1) / per_block;
    uint32_t grid = static_cast<uint32_t>(dev.sm_count) * static_cast<uint32_t>(per_sm);
    if (grid > needed) grid = needed;
    quant_nvfp4_1x16_tiled_kernel<<<grid, kNvThreads, 0, stream>>>(
        static_cast<const uint16_t*>(x), static_cast<uint32_t>(R), kb, ldx, g, xq, sx);
    return cudaGetLastError();
  }
  const bool dense = ldx == K;
  auto k = dense ? quant_nvfp4_1x16_kernel<true> : quant_nvfp4_1x16_kernel<false>;
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kNvThreads, 0);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const uint32_t per_block = kNvThreads * kNvRounds;
  const uint32_t needed = (blocks + per_block - 1) / per_block;
  uint32_t grid = static_cast<uint32_t>(dev.sm_count) * static_cast<uint32_t>(per_sm);
  if (grid > needed) grid = needed;
  k<<<grid, kNvThreads, 0, stream>>>(static_cast<const uint16_t*>(x), kb, blocks, ldx, g, xq, sx);
  return cudaGetLastError();
}

// Row-major FP4 block scales [R, F] (F % 4 == 0) into the tiled layout.  A
// block takes one 128-row tile x 8 cells: it reads 32 contiguous bytes of
// each of the 128 rows, transposes through shared memory, and writes the 8
// tiles (4 KB, contiguous in the tiled layout) with whole-sector stores.
// Rows past R are written as zeros.
__global__ void __launch_bounds__(256)
    fp4_scales_to_tiles_kernel(const uint32_t* __restrict__ s, uint32_t R, uint32_t cpr,
                               uint32_t* __restrict__ tiles) {
  __shared__ uint32_t t[8 * 128];
  const uint32_t cgroups = (cpr + 7u) / 8u;
  const uint32_t rb = blockIdx.x / cgroups, c0 = (blockIdx.x - rb * cgroups) * 8u;
  const uint32_t ncell = cpr - c0 < 8u ? cpr - c0 : 8u;
  for (uint32_t k = threadIdx.x; k < 1024u; k += 256u) {
    const uint32_t rr = k >> 3, cell = k & 7u;  // row in the tile, cell
    const uint32_t r = rb * 128u + rr;
    uint32_t w = 0;
    if (cell < ncell && r < R) w = __ldg(s + static_cast<uint64_t>(r) * cpr + c0 + cell);
    t[cell * 128u + (rr & 31u) * 4u + (rr >> 5)] = w;
  }
  __syncthreads();
  uint32_t* out = tiles + (static_cast<uint64_t>(rb) * cpr + c0) * 128u;
  for (uint32_t k = threadIdx.x; k < ncell * 128u; k += 256u) out[k] = t[k];
}

cudaError_t launch_fp4_scales_to_tiles(const uint8_t* s, int64_t R, int64_t F, uint8_t* tiles,
                                       cudaStream_t stream, const DeviceInfo& dev) {
  (void)dev;
  const uint32_t cpr = static_cast<uint32_t>(F / 4);
  const uint64_t blocks = static_cast<uint64_t>((R + 127) / 128) * ((cpr + 7) / 8);
  if (blocks == 0) return cudaSuccess;
  fp4_scales_to_tiles_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      reinterpret_cast<const uint32_t*>(s), static_cast<uint32_t>(R), cpr,
      reinterpret_cast<uint32_t*>(tiles));
  return cudaGetLastError();
}

}  // namespace fgq
