// Fine-grained FP8 quantizers for sm_103a: 1x128 activation tiles and
// 128x128 weight blocks ("Fine-Grained FP8/FP4 Quantization",
// §Scaling Granularities; scale shapes from §DeepGEMM).
//
// Both are HBM-bound streaming kernels.  Per group: amax of |x| (exact: the
// magnitude order of non-NaN bf16 values is the order of their bit patterns
// with the sign cleared, so it is taken with 16-bit SIMD integer max),
// s = amax / 448 in fp32 (or its power-of-two ceiling), then each element is
// divided by s in IEEE fp32 and rounded to E4M3 by the hardware convert
// (round to nearest even, saturating to +-448).
#include <cuda_runtime.h>

#include <cstdint>

#include "fgq_device.cuh"
#include "fgq_internal.h"

namespace fgq {
namespace {

constexpr int kScaleFp32 = 0;
constexpr int kScaleUe8m0 = 1;

__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream_8(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_stream_16(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Max of |x| over 8 bf16 held in a uint4, as a pair of 16-bit magnitudes.
__device__ __forceinline__ uint32_t absmax_pairs(uint4 v) {
  const uint32_t m = 0x7FFF7FFFu;
  uint32_t a = __vmaxu2(v.x & m, v.y & m);
  uint32_t b = __vmaxu2(v.z & m, v.w & m);
  return __vmaxu2(a, b);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Dequantisation multiplier of a group from the bit pattern of its amax
// (a non-negative bf16 magnitude widened to fp32).
template <int MODE>
__device__ __forceinline__ float scale_from_amax(float amax) {
  if (amax == 0.0f) return 1.0f;
  float t = __fdiv_rn(amax, 448.0f);
  if (MODE == kScaleFp32) return t;
  // Smallest power of two >= t, exponent clamped at -127 (t < 2^120 always).
  uint32_t b = __float_as_uint(t);
  uint32_t e = b >> 23, man = b & 0x7FFFFFu;
  if (e == 0) return __uint_as_float(b <= 0x00400000u ? 0x00400000u : 0x00800000u);
  return __uint_as_float((man != 0 ? e + 1 : e) << 23);
}

// q = E4M3(x / s) for the 8 bf16 of v, packed little-endian into 8 bytes.
// fp32 mode divides (IEEE, round to nearest even).  In UE8M0 mode s = 2^e
// and inv = 2^-e exactly, so x * inv rounds exactly like x / s.
template <int MODE>
__device__ __forceinline__ uint2 encode8(uint4 v, float s, float inv) {
  float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = (MODE == kScaleFp32) ? __fdiv_rn(f[i], s) : __fmul_rn(f[i], inv);
  uint2 r;
  r.x = cvt_e4m3x2(f[0], f[1]) | (cvt_e4m3x2(f[2], f[3]) << 16);
  r.y = cvt_e4m3x2(f[4], f[5]) | (cvt_e4m3x2(f[6], f[7]) << 16);
  return r;
}

// ---- 1x128 activation quantizer ----------------------------------------------
//
// A half-warp owns one 128-element group: lane l of the half loads bytes
// [16 l, 16 l + 16) of the group's 256.  The two halves of a warp take
// adjacent groups, so each warp load covers 512 contiguous bytes of a dense
// row.  Each warp first issues UNROLL pairs of group loads, then reduces and
// encodes them, keeping 16 * UNROLL bytes per lane in flight.
constexpr int kActThreads = 256;
constexpr int kActUnroll = 4;

template <int MODE, bool DENSE>
__global__ void __launch_bounds__(kActThreads)
    quant_act_1x128_kernel(const uint16_t* __restrict__ x, uint32_t kc, uint32_t groups,
                           int64_t ldx, uint8_t* __restrict__ xq, int64_t ldq,
                           float* __restrict__ sx) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t half = lane >> 4, l16 = lane & 15u;
  const uint32_t warp = (blockIdx.x * kActThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kActThreads) >> 5;

  for (uint32_t base = warp * (2 * kActUnroll); base < groups;
       base += nwarps * (2 * kActUnroll)) {
    uint4 v[kActUnroll];
    uint32_t g[kActUnroll];
#pragma unroll
    for (int u = 0; u < kActUnroll; ++u) {
      g[u] = base + 2 * u + half;
      v[u] = make_uint4(0, 0, 0, 0);
      if (g[u] < groups) {
        const uint16_t* src;
        if (DENSE) {
          src = x + static_cast<uint64_t>(g[u]) * 128 + l16 * 8;
        } else {
          uint32_t m = g[u] / kc, c = g[u] - m * kc;
          src = x + static_cast<int64_t>(m) * ldx + c * 128 + l16 * 8;
        }
        v[u] = ld_stream_16(src);
      }
    }
#pragma unroll
    for (int u = 0; u < kActUnroll; ++u) {
      uint32_t mx = absmax_pairs(v[u]);
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mx = __vmaxu2(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
      uint32_t mag = max(mx & 0xFFFFu, mx >> 16);
      float amax = __uint_as_float(mag << 16);
      float s = scale_from_amax<MODE>(amax);
      float inv = (MODE == kScaleFp32) ? 0.0f : __fdiv_rn(1.0f, s);  // exact for 2^e
      if (g[u] < groups) {
        uint2 q = encode8<MODE>(v[u], s, inv);
        uint8_t* dst;
        if (DENSE) {
          dst = xq + static_cast<uint64_t>(g[u]) * 128 + l16 * 8;
        } else {
          uint32_t m = g[u] / kc, c = g[u] - m * kc;
          dst = xq + static_cast<int64_t>(m) * ldq + c * 128 + l16 * 8;
        }
        st_stream_8(dst, q);
        if (l16 == 0) sx[g[u]] = s;
      }
    }
  }
}

// ---- 128x128 weight quantizer ------------------------------------------------
//
// One CTA per 128x128 block of W [K, N].  Thread t loads the 16-byte column
// chunk c = t % 16 (columns 8c .. 8c+7) of the 8 consecutive rows
// 8 rg .. 8 rg + 7, rg = t / 16: each warp load covers two 256-byte row
// segments.  The block amax is reduced by warp shuffles and shared memory;
// the codes are written transposed (Wq is [N, K], K-major) through a 16 KB
// shared tile T[n][k] whose 8-byte k-chunks are XOR-swizzled by (n / 8) % 16
// so that both the transposing writes and the row reads avoid bank
// conflicts.
constexpr int kWThreads = 256;

template <int MODE>
__global__ void __launch_bounds__(kWThreads)
    quant_w_128x128_kernel(const uint16_t* __restrict__ w, int64_t K, int64_t N, int64_t ldw,
                           uint8_t* __restrict__ wq, float* __restrict__ sw) {
  __shared__ __align__(16) uint2 tile[128 * 16];  // [n][k-chunk of 8], swizzled
  __shared__ uint32_t warp_max[kWThreads / 32];

  const int nb_count = static_cast<int>(N / 128);
  const int nb = blockIdx.x % nb_count, kb = blockIdx.x / nb_count;
  const int64_t n0 = static_cast<int64_t>(nb) * 128, k0 = static_cast<int64_t>(kb) * 128;
  const int t = threadIdx.x, c = t & 15, rg = t >> 4;

  uint4 v[8];
  const uint16_t* src = w + (k0 + 8 * rg) * ldw + n0 + 8 * c;
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = ld_stream_16(src + i * ldw);

  uint32_t mx = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) mx = __vmaxu2(mx, absmax_pairs(v[i]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = __vmaxu2(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  if ((t & 31) == 0) warp_max[t >> 5] = max(mx & 0xFFFFu, mx >> 16);
  __syncthreads();
  uint32_t mag = 0;
#pragma unroll
  for (int i = 0; i < kWThreads / 32; ++i) mag = max(mag, warp_max[i]);
  const float amax = __uint_as_float(mag << 16);
  const float s = scale_from_amax<MODE>(amax);
  const float inv = (MODE == kScaleFp32) ? 0.0f : __fdiv_rn(1.0f, s);

  // Encode: for column j of the chunk, the 8 rows give 8 consecutive k codes.
  uint32_t codes[8][2];  // [row i][lo: cols 0-3, hi: cols 4-7]
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint2 q = encode8<MODE>(v[i], s, inv);
    codes[i][0] = q.x;
    codes[i][1] = q.y;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) lo |= ((codes[i][j >> 2] >> (8 * (j & 3))) & 0xFFu) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) hi |= ((codes[i + 4][j >> 2] >> (8 * (j & 3))) & 0xFFu) << (8 * i);
    const int n = 8 * c + j;
    tile[n * 16 + (rg ^ c)] = make_uint2(lo, hi);
  }
  if (t == 0) sw[static_cast<int64_t>(kb) * nb_count + nb] = s;
  __syncthreads();

  const uint4* tile16 = reinterpret_cast<const uint4*>(tile);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int idx = p * kWThreads + t;
    const int n = idx >> 3, q = idx & 7;
    const int sw_ = (n >> 3) & 15;
    uint4 val = tile16[n * 8 + q];
    if (sw_ & 1) val = make_uint4(val.z, val.w, val.x, val.y);
    uint8_t* dst = wq + (n0 + n) * K + k0 + 16 * (q ^ (sw_ >> 1));
    st_stream_16(dst, val);
  }
}

}  // namespace

cudaError_t launch_quant_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx,
                                   uint8_t* xq, int64_t ldq, float* sx, int mode,
                                   cudaStream_t stream, const DeviceInfo& dev) {
  const uint32_t kc = static_cast<uint32_t>(K / 128);
  const uint32_t groups = static_cast<uint32_t>(M * (K / 128));
  if (groups == 0) return cudaSuccess;
  const bool dense = (ldx == K) && (ldq == K);
  const uint32_t groups_per_block = (kActThreads / 32) * 2 * kActUnroll;
  const uint32_t needed = (groups + groups_per_block - 1) / groups_per_block;

  using Kern = void (*)(const uint16_t*, uint32_t, uint32_t, int64_t, uint8_t*, int64_t, float*);
  Kern k;
  if (mode == kScaleFp32)
    k = dense ? quant_act_1x128_kernel<kScaleFp32, true> : quant_act_1x128_kernel<kScaleFp32, false>;
  else
    k = dense ? quant_act_1x128_kernel<kScaleUe8m0, true> : quant_act_1x128_kernel<kScaleUe8m0, false>;
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kActThreads, 0);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  uint32_t grid = static_cast<uint32_t>(dev.sm_count) * static_cast<uint32_t>(per_sm);
  if (grid > needed) grid = needed;
  k<<<grid, kActThreads, 0, stream>>>(static_cast<const uint16_t*>(x), kc, groups, ldx, xq, ldq,
                                      sx);
  return cudaGetLastError();
}

cudaError_t launch_quant_w_128x128(const void* w, int64_t K, int64_t N, int64_t ldw,
                                   uint8_t* wq, float* sw, int mode, cudaStream_t stream,
                                   const DeviceInfo& dev) {
  (void)dev;
  const int64_t blocks = (K / 128) * (N / 128);
  if (blocks == 0) return cudaSuccess;
  if (mode == kScaleFp32)
    quant_w_128x128_kernel<kScaleFp32><<<static_cast<unsigned>(blocks), kWThreads, 0, stream>>>(
        static_cast<const uint16_t*>(w), K, N, ldw, wq, sw);
  else
    quant_w_128x128_kernel<kScaleUe8m0><<<static_cast<unsigned>(blocks), kWThreads, 0, stream>>>(
        static_cast<const uint16_t*>(w), K, N, ldw, wq, sw);
  return cudaGetLastError();
}

}  // namespace fgq
