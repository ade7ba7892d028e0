// Fine-grained FP8 quantizers for sm_103a: 1x128 activation tiles and
// 128x128 weight blocks ("Fine-Grained FP8/FP4 Quantization",
// §Scaling Granularities; scale shapes from §DeepGEMM).
//
// Both are HBM-bound streaming kernels.  Per group: amax of |x| (exact: the
// magnitude order of non-NaN bf16 values is the order of their bit patterns
// with the sign cleared, so it is taken with 16-bit SIMD integer max),
// s = amax / 448 in fp32 (or its power-of-two ceiling), then each element
// becomes E4M3(fl32(x / s)) through the hardware convert (round to nearest
// even, saturating to +-448).
//
// The quotient fl32(x / s) is formed without a per-element division:
//   r  = RN(1 / s)                      (once per group)
//   q0 = RN(x * r)
//   q1 = RN(q0 + r * RN(x - q0 * s))    (both steps fused multiply-adds)
// which is Markstein's correction of a reciprocal-based quotient (P.
// Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990).  For the operands these
// kernels can see -- x a bf16 value with |x| <= amax, s = RN(amax / 448)
// with amax a bf16 value and s >= 2^-100 -- E4M3(q1) equals E4M3(x / s)
// for every pair, signs aside (the residual step turns -0 into +0, so the
// sign bit of every code is taken from x).  This was checked exhaustively
// over all 1.07e9 such (amax, x) bf16 pairs against IEEE division, and the
// GPU tests compare every bf16 pattern against the oracle.  Groups with
// s < 2^-100 (amax below about 2^-91) take IEEE division instead.  In UE8M0
// mode s = 2^e and x * 2^-e is exact, so a single multiply is used.
#include <cuda_runtime.h>

#include <cstdint>

#include "fgq_device.cuh"
#include "fgq_internal.h"
#include "fgq_quant.cuh"

namespace fgq {
namespace {

// ---- 1x128 activation quantizer ----------------------------------------------
//
// Eight lanes own one 128-element (256-byte) group: lane l of the eight loads
// bytes [16 l, 16 l + 16) and [128 + 16 l, 128 + 16 l + 16), so each warp
// load instruction covers two full 128-byte lines of each of its four
// groups.  A warp first issues the loads of kActRounds rounds (4 groups
// each), then reduces and encodes them: 16 * 2 * kActRounds bytes per lane
// in flight.
constexpr int kActThreads = 256;
constexpr int kActRounds = 2;
constexpr int kActGroupsPerWarp = 4 * kActRounds;

// The groups of warp `warp` out of `nwarps` warps sharing the work.
// UE8M0 code of a power-of-two scale (its biased exponent field) at its
// place in the code tiles of the tiled-scale FP8 GEMM: row r, chunk c of
// F = kc chunks a row, cells of four chunks (F padded to a multiple of 4),
// 512-byte tiles of 128 rows: byte ((r / 128) * cpr + c / 4) * 512 +
// (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4, cpr = ceil(kc / 4).
__device__ __forceinline__ void store_code_tile(uint8_t* tiles, uint32_t r, uint32_t c,
                                                uint32_t cpr, float s) {
  tiles[(static_cast<uint64_t>(r >> 7) * cpr + (c >> 2)) * 512u + (r & 31u) * 16u +
        ((r >> 5) & 3u) * 4u + (c & 3u)] = static_cast<uint8_t>((__float_as_uint(s) >> 23) & 0xFFu);
}

// TILES (UE8M0 only): the scales go out as code tiles (sx is then the tile
// buffer, as bytes) instead of fp32 [M, K/128].
template <int MODE, bool DENSE, bool TILES = false>
__device__ __forceinline__ void act_groups(const uint16_t* __restrict__ x, uint32_t kc,
                                           uint32_t groups, int64_t ldx, uint8_t* __restrict__ xq,
                                           int64_t ldq, float* __restrict__ sx, uint32_t warp,
                                           uint32_t nwarps) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t sub = lane >> 3, l8 = lane & 7u;

  for (uint32_t base = warp * kActGroupsPerWarp; base < groups;
       base += nwarps * kActGroupsPerWarp) {
    uint4 v[kActRounds][2];
    uint32_t g[kActRounds];
#pragma unroll
    for (int u = 0; u < kActRounds; ++u) {
      g[u] = base + 4 * u + sub;
      v[u][0] = v[u][1] = make_uint4(0, 0, 0, 0);
      if (g[u] < groups) {
        const uint16_t* src;
        if (DENSE) {
          src = x + static_cast<uint64_t>(g[u]) * 128;
        } else {
          const uint32_t m = g[u] / kc, c = g[u] - m * kc;
          src = x + static_cast<int64_t>(m) * ldx + c * 128;
        }
        v[u][0] = ld_stream_16(src + 8 * l8);
        v[u][1] = ld_stream_16(src + 64 + 8 * l8);
      }
    }
#pragma unroll
    for (int u = 0; u < kActRounds; ++u) {
      uint32_t mx = __vmaxu2(absmax_pairs(v[u][0]), absmax_pairs(v[u][1]));
#pragma unroll
      for (int off = 4; off > 0; off >>= 1) mx = __vmaxu2(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
      const GroupScale gs = group_scale<MODE>(max(mx & 0xFFFFu, mx >> 16));
      if (g[u] < groups) {
        const uint2 q0 = encode8<MODE>(v[u][0], gs);
        const uint2 q1 = encode8<MODE>(v[u][1], gs);
        uint8_t* dst;
        if (DENSE) {
          dst = xq + static_cast<uint64_t>(g[u]) * 128;
        } else {
          const uint32_t m = g[u] / kc, c = g[u] - m * kc;
          dst = xq + static_cast<int64_t>(m) * ldq + c * 128;
        }
        st_stream_8(dst + 8 * l8, q0);
        st_stream_8(dst + 64 + 8 * l8, q1);
        if (l8 == 0) {
          if (TILES) {
            const uint32_t m = g[u] / kc;
            store_code_tile(reinterpret_cast<uint8_t*>(sx), m, g[u] - m * kc, (kc + 3) / 4, gs.s);
          } else {
            sx[g[u]] = gs.s;
          }
        }
      }
    }
  }
}

template <int MODE, bool DENSE>
__global__ void __launch_bounds__(kActThreads)
    quant_act_1x128_kernel(const uint16_t* __restrict__ x, uint32_t kc, uint32_t groups,
                           int64_t ldx, uint8_t* __restrict__ xq, int64_t ldq,
                           float* __restrict__ sx) {
  act_groups<MODE, DENSE>(x, kc, groups, ldx, xq, ldq, sx,
                          (blockIdx.x * kActThreads + threadIdx.x) >> 5,
                          (gridDim.x * kActThreads) >> 5);
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

// Transpose a 4x4 byte matrix held as four row words r0..r3 (byte b of r_i
// = element (i, b)) into column words c0..c3 (byte i of c_b = element (i, b)).
__device__ __forceinline__ void transpose4x4_bytes(uint32_t r0, uint32_t r1, uint32_t r2,
                                                   uint32_t r3, uint32_t& c0, uint32_t& c1,
                                                   uint32_t& c2, uint32_t& c3) {
  const uint32_t t0 = __byte_perm(r0, r1, 0x5140);  // r0.b0 r1.b0 r0.b1 r1.b1
  const uint32_t t1 = __byte_perm(r0, r1, 0x7362);  // r0.b2 r1.b2 r0.b3 r1.b3
  const uint32_t t2 = __byte_perm(r2, r3, 0x5140);
  const uint32_t t3 = __byte_perm(r2, r3, 0x7362);
  c0 = __byte_perm(t0, t2, 0x5410);
  c1 = __byte_perm(t0, t2, 0x7632);
  c2 = __byte_perm(t1, t3, 0x5410);
  c3 = __byte_perm(t1, t3, 0x7632);
}

// Four CTAs per SM (55 registers a thread, no spill): measured 28.8 us on a
// 7168 x 7168 weight, against 28.9-30.3 us with five (51 registers and a
// few bytes of spill) and 35 us with six.
// Block `block` of W (k-block major), by the CTA's kWThreads threads.
template <int MODE, bool TILES = false>
__device__ __forceinline__ void w_block(const uint16_t* __restrict__ w, int64_t K, int64_t N,
                                        int64_t ldw, uint8_t* __restrict__ wq,
                                        float* __restrict__ sw, uint32_t block) {
  __shared__ __align__(16) uint2 tile[128 * 16];  // [n][k-chunk of 8], swizzled
  __shared__ uint32_t warp_max[kWThreads / 32];

  const int nb_count = static_cast<int>(N / 128);
  const int nb = static_cast<int>(block % nb_count), kb = static_cast<int>(block / nb_count);
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
  const GroupScale gs = group_scale<MODE>(mag);

  // Encode: for column j of the chunk, the 8 rows give 8 consecutive k codes.
  // The block's exact-division test is taken once; the common copy has none.
  uint32_t codes[8][2];  // [row i][lo: cols 0-3, hi: cols 4-7]
  if (MODE == kScaleFp32 && gs.exact) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint2 q = encode8<MODE>(v[i], gs);
      codes[i][0] = q.x;
      codes[i][1] = q.y;
    }
  } else {
    GroupScale g2 = gs;
    g2.exact = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint2 q = encode8<MODE>(v[i], g2);
      codes[i][0] = q.x;
      codes[i][1] = q.y;
    }
  }
  // Column j of the 8x8 code block, as rows 0-3 (lo) and 4-7 (hi): four
  // 4x4 byte transposes, byte i of each result word = row i.
  uint32_t lo[8], hi[8];
  transpose4x4_bytes(codes[0][0], codes[1][0], codes[2][0], codes[3][0], lo[0], lo[1], lo[2], lo[3]);
  transpose4x4_bytes(codes[0][1], codes[1][1], codes[2][1], codes[3][1], lo[4], lo[5], lo[6], lo[7]);
  transpose4x4_bytes(codes[4][0], codes[5][0], codes[6][0], codes[7][0], hi[0], hi[1], hi[2], hi[3]);
  transpose4x4_bytes(codes[4][1], codes[5][1], codes[6][1], codes[7][1], hi[4], hi[5], hi[6], hi[7]);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int n = 8 * c + j;
    tile[n * 16 + (rg ^ c)] = make_uint2(lo[j], hi[j]);
  }
  if (TILES) {
    // the block's code for each of its 128 columns (rows of the transposed
    // weight's code tiles)
    if (t < 128)
      store_code_tile(reinterpret_cast<uint8_t*>(sw), static_cast<uint32_t>(n0) + t,
                      static_cast<uint32_t>(kb), static_cast<uint32_t>((K / 128 + 3) / 4), gs.s);
  } else if (t == 0) {
    sw[static_cast<int64_t>(kb) * nb_count + nb] = gs.s;
  }
  __syncthreads();

  const uint4* tile16 = reinterpret_cast<const uint4*>(tile);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int idx = p * kWThreads + t;
    const int n = idx >> 3, q = idx & 7;
    const int swz = (n >> 3) & 15;
    uint4 val = tile16[n * 8 + q];
    if (swz & 1) val = make_uint4(val.z, val.w, val.x, val.y);
    uint8_t* dst = wq + (n0 + n) * K + k0 + 16 * (q ^ (swz >> 1));
    st_stream_16(dst, val);
  }
}

template <int MODE>
__global__ void __launch_bounds__(kWThreads, 4)
    quant_w_128x128_kernel(const uint16_t* __restrict__ w, int64_t K, int64_t N, int64_t ldw,
                           uint8_t* __restrict__ wq, float* __restrict__ sw) {
  w_block<MODE>(w, K, N, ldw, wq, sw, blockIdx.x);
}

// Both operands of one GEMM in one launch: CTAs [0, w_blocks) quantize one
// 128x128 weight block each (as quant_w_128x128_kernel); the rest share the
// 1x128 activation groups (as quant_act_1x128_kernel, kActThreads / 32
// warps each).  The same arithmetic, so the same codes and scales as the
// two kernels; one launch saves the second kernel's fill and drain.
// (Four CTAs per SM: at five, the activation half spills.)
static_assert(kActThreads == kWThreads, "one block size for both halves");
template <int MODE, bool DENSE, bool TILES = false>
__global__ void __launch_bounds__(kWThreads, 4)
    quant_operands_kernel(const uint16_t* __restrict__ x, uint32_t kc, uint32_t groups,
                          int64_t ldx, uint8_t* __restrict__ xq, int64_t ldq,
                          float* __restrict__ sx, const uint16_t* __restrict__ w, int64_t K,
                          int64_t N, int64_t ldw, uint8_t* __restrict__ wq,
                          float* __restrict__ sw, uint32_t w_blocks) {
  // Launched with programmatic stream serialization: the previous kernel's
  // memory is visible after pdl_wait(); the next kernel (the GEMM) may then
  // start its set-up, and waits for this grid itself before touching memory.
  pdl_wait();
  pdl_launch_dependents();
  if (blockIdx.x < w_blocks) {
    w_block<MODE, TILES>(w, K, N, ldw, wq, sw, blockIdx.x);
    return;
  }
  const uint32_t act_ctas = gridDim.x - w_blocks;
  act_groups<MODE, DENSE, TILES>(x, kc, groups, ldx, xq, ldq, sx,
                          ((blockIdx.x - w_blocks) * kActThreads + threadIdx.x) >> 5,
                          act_ctas * (kActThreads / 32));
}

// ---- 128x1 (transposed) activation quantizer -----------------------------------
//
// Groups of 128 consecutive rows of one column of X [M, K], written in the
// layout a GEMM reducing over M takes for its A operand: XqT [K, M] codes
// and sXT [K, M/128] scales (the 1x128 quantization of X^T).  One CTA per
// 128x128 block; thread t loads the 8 columns 8c .. 8c+7 (c = t % 16) of
// rows 8 rg .. 8 rg + 7 (rg = t / 16), as the weight quantizer does.  Each
// column's amax is reduced over the 16 row groups (one shuffle, then a
// shared table over the 8 warps); each element is encoded with its
// column's scale; the codes go out transposed through the same swizzled
// shared tile as the weight quantizer's.

// Codes of 8 bf16 of v whose element j has the scale s_j of column j,
// given as ns[j] = -s_j (the residual's multiplier; kept negated so that no
// element pair pays for a negation) and r[j] = RN(1 / s_j).
template <int MODE>
__device__ __forceinline__ uint2 encode8_cols(uint4 v, const float (&ns)[8], const float (&r)[8],
                                              uint32_t exact_mask) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const float2 x = bf16x2_to_f32x2(w[p]);
    const float2 r2 = make_float2(r[2 * p], r[2 * p + 1]);
    float2 q;
    if (MODE == kScaleUe8m0) {
      q = mul2(x, r2);
    } else {
      const float2 q0 = mul2(x, r2);
      const float2 d = fma2(q0, make_float2(ns[2 * p], ns[2 * p + 1]), x);  // exact residual
      q = fma2(d, r2, q0);
      if (exact_mask & (1u << (2 * p))) q.x = __fdiv_rn(x.x, -ns[2 * p]);
      if (exact_mask & (2u << (2 * p))) q.y = __fdiv_rn(x.y, -ns[2 * p + 1]);
    }
    c[p] = cvt_e4m3x2(q.x, q.y);
  }
  const uint32_t s01 = __byte_perm(v.x, v.y, 0x7531) & 0x80808080u;
  const uint32_t s23 = __byte_perm(v.z, v.w, 0x7531) & 0x80808080u;
  uint2 out;
  out.x = __byte_perm(c[0], c[1], 0x5410) | s01;
  out.y = __byte_perm(c[2], c[3], 0x5410) | s23;
  return out;
}

template <int MODE>
__global__ void __launch_bounds__(kWThreads, 4)
    quant_act_128x1_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                           uint8_t* __restrict__ xqt, float* __restrict__ sxt) {
  __shared__ __align__(16) uint2 tile[128 * 16];     // [k][m-chunk of 8], swizzled
  __shared__ uint32_t colmax[kWThreads / 32][16][4];  // per warp: 16 chunks x 4 column pairs
  __shared__ __align__(16) float col_ns[128], col_r[128];  // each column's -scale, reciprocal

  const int kb_count = static_cast<int>(K / 128);
  const int mc = static_cast<int>(M / 128);
  const int kb = blockIdx.x % kb_count, mb = blockIdx.x / kb_count;
  const int64_t m0 = static_cast<int64_t>(mb) * 128, k0 = static_cast<int64_t>(kb) * 128;
  const int t = threadIdx.x, c = t & 15, rg = t >> 4, lane = t & 31, warp = t >> 5;

  uint4 v[8];
  const uint16_t* src = x + (m0 + 8 * rg) * ldx + k0 + 8 * c;
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = ld_stream_16(src + i * ldx);

  // column maxima (16-bit magnitude pairs: columns 2p, 2p+1 of the chunk)
  const uint32_t msk = 0x7FFF7FFFu;
  uint32_t cm[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    cm[0] = __vmaxu2(cm[0], v[i].x & msk);
    cm[1] = __vmaxu2(cm[1], v[i].y & msk);
    cm[2] = __vmaxu2(cm[2], v[i].z & msk);
    cm[3] = __vmaxu2(cm[3], v[i].w & msk);
  }
#pragma unroll
  for (int p = 0; p < 4; ++p) cm[p] = __vmaxu2(cm[p], __shfl_xor_sync(0xFFFFFFFFu, cm[p], 16));
  if (lane < 16) {
#pragma unroll
    for (int p = 0; p < 4; ++p) colmax[warp][lane][p] = cm[p];
  }
  __syncthreads();
  // one thread per column: its amax over the 8 warps, its scale
  if (t < 128) {
    const int cc = t >> 3, p = (t & 7) >> 1;
    uint32_t mx = 0;
#pragma unroll
    for (int w = 0; w < kWThreads / 32; ++w) mx = __vmaxu2(mx, colmax[w][cc][p]);
    const uint32_t mag = (t & 1) ? (mx >> 16) : (mx & 0xFFFFu);
    const GroupScale gs = group_scale<MODE>(mag);
    col_ns[t] = -gs.s;
    col_r[t] = gs.r2.x;
    sxt[(k0 + t) * mc + mb] = gs.s;
  }
  __syncthreads();

  float sc[8], rc[8];
  {
    const float4 s0 = reinterpret_cast<const float4*>(col_ns)[2 * c];
    const float4 s1 = reinterpret_cast<const float4*>(col_ns)[2 * c + 1];
    const float4 r0 = reinterpret_cast<const float4*>(col_r)[2 * c];
    const float4 r1 = reinterpret_cast<const float4*>(col_r)[2 * c + 1];
    sc[0] = s0.x; sc[1] = s0.y; sc[2] = s0.z; sc[3] = s0.w;
    sc[4] = s1.x; sc[5] = s1.y; sc[6] = s1.z; sc[7] = s1.w;
    rc[0] = r0.x; rc[1] = r0.y; rc[2] = r0.z; rc[3] = r0.w;
    rc[4] = r1.x; rc[5] = r1.y; rc[6] = r1.z; rc[7] = r1.w;
  }
  uint32_t exact_mask = 0;
  if (MODE == kScaleFp32) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (!(-sc[j] >= 0x1p-100f)) exact_mask |= 1u << j;  // the exact-division range (sc = -s)
  }

  // The exact-division test once for all eight rows: the common case runs
  // with no per-pair branch (74.4 -> 63.7 us on the quantize-bandwidth
  // activations, together with the negated scales).
  uint32_t codes[8][2];  // [row i][lo: cols 0-3, hi: cols 4-7]
  if (exact_mask != 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint2 q = encode8_cols<MODE>(v[i], sc, rc, exact_mask);
      codes[i][0] = q.x;
      codes[i][1] = q.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint2 q = encode8_cols<MODE>(v[i], sc, rc, 0u);
      codes[i][0] = q.x;
      codes[i][1] = q.y;
    }
  }
  uint32_t lo[8], hi[8];
  transpose4x4_bytes(codes[0][0], codes[1][0], codes[2][0], codes[3][0], lo[0], lo[1], lo[2], lo[3]);
  transpose4x4_bytes(codes[0][1], codes[1][1], codes[2][1], codes[3][1], lo[4], lo[5], lo[6], lo[7]);
  transpose4x4_bytes(codes[4][0], codes[5][0], codes[6][0], codes[7][0], hi[0], hi[1], hi[2], hi[3]);
  transpose4x4_bytes(codes[4][1], codes[5][1], codes[6][1], codes[7][1], hi[4], hi[5], hi[6], hi[7]);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int kk = 8 * c + j;
    tile[kk * 16 + (rg ^ c)] = make_uint2(lo[j], hi[j]);
  }
  __syncthreads();

  const uint4* tile16 = reinterpret_cast<const uint4*>(tile);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int idx = p * kWThreads + t;
    const int kk = idx >> 3, q = idx & 7;
    const int swz = (kk >> 3) & 15;
    uint4 val = tile16[kk * 8 + q];
    if (swz & 1) val = make_uint4(val.z, val.w, val.x, val.y);
    uint8_t* dst = xqt + (k0 + kk) * M + m0 + 16 * (q ^ (swz >> 1));
    st_stream_16(dst, val);
  }
}

// ---- MXFP4 1x32 quantizer --------------------------------------------------------
//
// E2M1 elements with one UE8M0 scale per 32 consecutive elements of a row
// ("Fine-Grained FP8/FP4 Quantization", §UE8M0 vs E4M3 Scale Formats, block
// size 32).  Scale 2^e = the smallest power of two >= amax / 6 (6 = largest
// E2M1 value), exponent clamped to [-127, 127], 1 for a zero group; each
// element is x * 2^-e (exact) converted to E2M1, round to nearest even.
// Four lanes own a group (8 elements, 16 bytes each); codes are packed two
// per byte, the even element in the low nibble.
constexpr int kMxThreads = 256;
constexpr int kMxRounds = 2;

// UE8M0 exponent field of the smallest power of two >= amax / 6 (field 0 =
// 2^-127, the clamp; 127 = 2^0 for a zero group).
__device__ __forceinline__ uint32_t mx_scale_code(uint32_t mag_bits) {
  const float amax = __uint_as_float(mag_bits << 16);
  if (amax == 0.0f) return 127u;
  const uint32_t b = __float_as_uint(__fdiv_rn(amax, 6.0f));
  const uint32_t e = b >> 23, man = b & 0x7FFFFFu;
  if (e == 0) return b <= 0x00400000u ? 0u : 1u;  // subnormal quotient: 2^-127 or 2^-126
  return man != 0 ? e + 1 : e;
}

// One group of 32 elements over four lanes (8 each, v): the group's UE8M0
// code (the same in the four lanes) and this lane's eight E2M1 codes.
__device__ __forceinline__ uint32_t mx_group(const uint4& v, uint32_t* packed) {
  uint32_t mx = absmax_pairs(v);
  mx = __vmaxu2(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
  mx = __vmaxu2(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
  const uint32_t code = mx_scale_code(max(mx & 0xFFFFu, mx >> 16));
  // 2^-e: exponent field 254 - code; code 0 (2^-127) gives 2^127
  const float inv = __uint_as_float((254u - code) << 23);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float y[8];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const float2 f = bf16x2_to_f32x2(w[p]);
    y[2 * p] = f.x * inv;
    y[2 * p + 1] = f.y * inv;
  }
  *packed = cvt_e2m1x8(y);
  return code;
}

template <bool DENSE>
__global__ void __launch_bounds__(kMxThreads)
    quant_mxfp4_1x32_kernel(const uint16_t* __restrict__ x, uint32_t kg, uint32_t groups,
                            int64_t ldx, uint8_t* __restrict__ xq, uint8_t* __restrict__ sx) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t sub = lane >> 2, l4 = lane & 3u;
  const uint32_t warp = (blockIdx.x * kMxThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kMxThreads) >> 5;
  constexpr uint32_t kPerWarp = 8 * kMxRounds;
  for (uint32_t base = warp * kPerWarp; base < groups; base += nwarps * kPerWarp) {
    uint4 v[kMxRounds];
    uint32_t g[kMxRounds];
#pragma unroll
    for (int u = 0; u < kMxRounds; ++u) {
      g[u] = base + 8 * u + sub;
      v[u] = make_uint4(0, 0, 0, 0);
      if (g[u] < groups) {
        const uint16_t* src;
        if (DENSE) {
          src = x + static_cast<uint64_t>(g[u]) * 32;
        } else {
          const uint32_t r = g[u] / kg, c = g[u] - r * kg;
          src = x + static_cast<int64_t>(r) * ldx + c * 32;
        }
        v[u] = ld_stream_16(src + 8 * l4);
      }
    }
#pragma unroll
    for (int u = 0; u < kMxRounds; ++u) {
      uint32_t packed;
      const uint32_t code = mx_group(v[u], &packed);
      if (g[u] < groups) {
        // row-major [R, K/2]: group g covers bytes 16 g .. 16 g + 15
        *reinterpret_cast<uint32_t*>(xq + static_cast<uint64_t>(g[u]) * 16 + 4 * l4) = packed;
        if (l4 == 0) sx[g[u]] = static_cast<uint8_t>(code);
      }
    }
  }
}

// One group of 32 elements held by one thread (v: four 16-byte chunks): the
// group's UE8M0 code, formed once, and its 32 E2M1 codes as four words.
__device__ __forceinline__ uint32_t mx_group32(const uint4 (&v)[4], uint32_t (&packed)[4]) {
  const uint32_t mx = __vmaxu2(__vmaxu2(absmax_pairs(v[0]), absmax_pairs(v[1])),
                               __vmaxu2(absmax_pairs(v[2]), absmax_pairs(v[3])));
  const uint32_t code = mx_scale_code(max(mx & 0xFFFFu, mx >> 16));
  // 2^-e: exponent field 254 - code; code 0 (2^-127) gives 2^127
  const float inv = __uint_as_float((254u - code) << 23);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
    float y[8];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 f = bf16x2_to_f32x2(w[p]);
      y[2 * p] = f.x * inv;
      y[2 * p + 1] = f.y * inv;
    }
    packed[q] = cvt_e2m1x8(y);
  }
  return code;
}

// The same quantizer with the scales in the tiled FP4 layout: 512-byte tiles
// of 128 rows x 4 factor bytes; tile (r / 128, f / 4) holds, in its 16-byte
// row i, the cells (4 factor bytes) of rows 32 j + i, j = 0..3 (the 32-row x
// 16-byte tile the FP4 GEMM copies into TMEM).  One thread per group of 32
// (64 contiguous bytes of x), so the group's amax takes no shuffle and its
// scale is formed once for 32 elements.  A warp's unit is 16-byte row i of
// eight neighbouring tiles: rows 32 j + i, j = 0..3, each 32 groups (2 KB of
// x), two rows' loads in flight at a time; lanes 0, 4, .., 28 then each hold
// tile row i of one cell (the codes of their own and the next three lanes'
// groups) and store it whole.  Rows past R read as zeros and give padding
// codes (127).  (Four lanes per group, as the row-major kernel: 59.4 us on
// the quantize-bandwidth activations.)
__global__ void __launch_bounds__(kMxThreads)
    quant_mxfp4_1x32_tiled_kernel(const uint16_t* __restrict__ x, uint32_t R, uint32_t kg,
                                  int64_t ldx, uint8_t* __restrict__ xq,
                                  uint8_t* __restrict__ st) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = (blockIdx.x * kMxThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kMxThreads) >> 5;
  const uint32_t cpr = kg >> 2;            // cells (tiles) per 128-row tile
  const uint32_t octs = (cpr + 7u) >> 3;   // groups of eight cells per 128-row tile
  const uint32_t units = ((R + 127u) >> 7) * octs * 32u;
  for (uint32_t unit = warp; unit < units; unit += nwarps) {
    const uint32_t i = unit & 31u, t = unit >> 5;
    const uint32_t rb = t / octs, co = t - rb * octs;
    const uint32_t grp = 32u * co + lane;  // this lane's group within the row
    const bool col_ok = grp < kg;          // the last cells of the eight may not exist
    uint32_t cell[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 v[2][4];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const uint32_t row = rb * 128u + 32u * (2 * h + jj) + i;
        const uint16_t* src = x + static_cast<int64_t>(row) * ldx + grp * 32u;
        const bool ok = row < R && col_ok;
#pragma unroll
        for (int q = 0; q < 4; ++q) v[jj][q] = ok ? ld_stream_16(src + 8 * q) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const uint32_t row = rb * 128u + 32u * (2 * h + jj) + i;
        uint32_t packed[4];
        const uint32_t code = mx_group32(v[jj], packed);
        if (row < R && col_ok) {
          uint32_t* dst = reinterpret_cast<uint32_t*>(xq + static_cast<uint64_t>(row) * (16u * kg) +
                                                      grp * 16u);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = packed[q];
        }
        // lanes 4 c: the cell (groups in lanes +0 .. +3)
        const uint32_t c1 = __shfl_down_sync(0xFFFFFFFFu, code, 1);
        const uint32_t c2 = __shfl_down_sync(0xFFFFFFFFu, code, 2);
        const uint32_t c3 = __shfl_down_sync(0xFFFFFFFFu, code, 3);
        cell[2 * h + jj] = code | (c1 << 8) | (c2 << 16) | (c3 << 24);
      }
    }
    if ((lane & 3u) == 0 && col_ok)
      *reinterpret_cast<uint4*>(st + (static_cast<uint64_t>(rb) * cpr + 8u * co + (lane >> 2)) * 512u +
                                16u * i) = make_uint4(cell[0], cell[1], cell[2], cell[3]);
  }
}

}  // namespace

cudaError_t launch_quant_mxfp4_1x32(const void* x, int64_t R, int64_t K, int64_t ldx, uint8_t* xq,
                                    uint8_t* sx, bool tiled, cudaStream_t stream,
                                    const DeviceInfo& dev) {
  const uint32_t kg = static_cast<uint32_t>(K / 32);
  const uint32_t groups = static_cast<uint32_t>(R * (K / 32));
  if (groups == 0) return cudaSuccess;
  if (tiled) {
    // one warp per 16-byte row of eight neighbouring tiles (128 groups)
    const uint32_t units = static_cast<uint32_t>((R + 127) / 128) * ((kg / 4 + 7) / 8) * 32u;
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, quant_mxfp4_1x32_tiled_kernel, kMxThreads, 0);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    const uint32_t needed = (units + kMxThreads / 32 - 1) / (kMxThreads / 32);
    uint32_t grid = static_cast<uint32_t>(dev.sm_count) * static_cast<uint32_t>(per_sm);
    if (grid > needed) grid = needed;
    quant_mxfp4_1x32_tiled_kernel<<<grid, kMxThreads, 0, stream>>>(
        static_cast<const uint16_t*>(x), static_cast<uint32_t>(R), kg, ldx, xq, sx);
    return cudaGetLastError();
  }
  const bool dense = ldx == K;
  auto k = dense ? quant_mxfp4_1x32_kernel<true> : quant_mxfp4_1x32_kernel<false>;
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kMxThreads, 0);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const uint32_t per_block = (kMxThreads / 32) * 8 * kMxRounds;
  const uint32_t needed = (groups + per_block - 1) / per_block;
  uint32_t grid = static_cast<uint32_t>(dev.sm_count) * static_cast<uint32_t>(per_sm);
  if (grid > needed) grid = needed;
  k<<<grid, kMxThreads, 0, stream>>>(static_cast<const uint16_t*>(x), kg, groups, ldx, xq, sx);
  return cudaGetLastError();
}

cudaError_t launch_quant_act_128x1(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xqt,
                                   float* sxt, int mode, cudaStream_t stream,
                                   const DeviceInfo& dev) {
  (void)dev;
  const int64_t blocks = (M / 128) * (K / 128);
  if (blocks == 0) return cudaSuccess;
  if (blocks >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
  if (mode == kScaleFp32)
    quant_act_128x1_kernel<kScaleFp32><<<static_cast<unsigned>(blocks), kWThreads, 0, stream>>>(
        static_cast<const uint16_t*>(x), M, K, ldx, xqt, sxt);
  else
    quant_act_128x1_kernel<kScaleUe8m0><<<static_cast<unsigned>(blocks), kWThreads, 0, stream>>>(
        static_cast<const uint16_t*>(x), M, K, ldx, xqt, sxt);
  return cudaGetLastError();
}

cudaError_t launch_quant_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx,
                                   uint8_t* xq, int64_t ldq, float* sx, int mode,
                                   cudaStream_t stream, const DeviceInfo& dev) {
  const uint32_t kc = static_cast<uint32_t>(K / 128);
  const uint32_t groups = static_cast<uint32_t>(M * (K / 128));
  if (groups == 0) return cudaSuccess;
  const bool dense = (ldx == K) && (ldq == K);
  const uint32_t groups_per_block = (kActThreads / 32) * kActGroupsPerWarp;
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

cudaError_t launch_quant_operands(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                  int64_t ldq, float* sx, const void* w, int64_t N, int64_t ldw,
                                  uint8_t* wq, float* sw, int mode, cudaStream_t stream,
                                  const DeviceInfo& dev, bool code_tiles) {
  const uint32_t kc = static_cast<uint32_t>(K / 128);
  const uint32_t groups = static_cast<uint32_t>(M * (K / 128));
  const int64_t w_blocks = (K / 128) * (N / 128);
  // activation CTAs: kRoundsPerWarp rounds of kActGroupsPerWarp groups per
  // warp, at least one CTA when there are groups, and at most one wave (four
  // per SM): they run after the weight blocks, so a second, partial wave of
  // them would be the kernel's tail (measured 45.7 against 47.4 us on the
  // large-prefill operands)
  constexpr uint32_t kRoundsPerWarp = 4;
  const uint32_t per_cta = (kActThreads / 32) * kActGroupsPerWarp * kRoundsPerWarp;
  uint32_t act_ctas = (groups + per_cta - 1) / per_cta;
  const uint32_t wave = 4u * static_cast<uint32_t>(dev.sm_count);
  if (act_ctas > wave) act_ctas = wave;
  const int64_t grid = w_blocks + act_ctas;
  if (grid == 0) return cudaSuccess;
  if (grid >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
  const bool dense = (ldx == K) && (ldq == K);
  using Kern = void (*)(const uint16_t*, uint32_t, uint32_t, int64_t, uint8_t*, int64_t, float*,
                        const uint16_t*, int64_t, int64_t, int64_t, uint8_t*, float*, uint32_t);
  Kern k;
  if (code_tiles)
    k = dense ? quant_operands_kernel<kScaleUe8m0, true, true>
              : quant_operands_kernel<kScaleUe8m0, false, true>;
  else if (mode == kScaleFp32)
    k = dense ? quant_operands_kernel<kScaleFp32, true> : quant_operands_kernel<kScaleFp32, false>;
  else
    k = dense ? quant_operands_kernel<kScaleUe8m0, true> : quant_operands_kernel<kScaleUe8m0, false>;
  return launch_pdl(k, dim3(static_cast<unsigned>(grid)), dim3(kWThreads), 0, stream,
                    static_cast<const uint16_t*>(x), kc, groups, ldx, xq, ldq, sx,
                    static_cast<const uint16_t*>(w), K, N, ldw, wq, sw,
                    static_cast<uint32_t>(w_blocks));
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
