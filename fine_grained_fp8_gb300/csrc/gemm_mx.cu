// Block-scaled FP8 GEMM with power-of-two (UE8M0) scales applied by the
// tensor core ("Fine-Grained FP8/FP4 Quantization", §Blackwell: Native Block
// Scaling, §UE8M0 vs E4M3 Scale Formats):
//
//   C[m,n] = sum_c sum_{k in chunk c} (Aq[m,k] sA[m,c]) (Bq[k,n] sB[c,n/128])
//
// When every scale is a power of two the scaling is exact, so it can move
// inside the MMA: tcgen05.mma kind::mxf8f6f4.block_scale multiplies each
// K = 32 slice of A's row m by 2^(a-127) and of B's column n by 2^(b-127),
// with the UE8M0 codes a, b read from TMEM.  A 1x128 activation scale is
// the same code for the four slices of its chunk, and a 128x128 weight
// scale the same code for the 128 columns of its block.  The accumulator
// then stays in TMEM for the whole K loop; nothing passes through registers
// until the tile is done (no promotion step).
//
// Design (persistent, 128 x BN tiles, static stride schedule, M fastest, as
// the fp32-scale kernel):
//   - warp 0: TMA producer: per stage one 128-wide K chunk of A (128 x 128
//     bytes) and B (BN x 128 bytes), 128-byte swizzled;
//   - warp 1: MMA issuer: four K = 32 MMAs per chunk into the tile's
//     accumulator, scale factors from one slot of a TMEM ring;
//   - warps 4-7: scale-factor writers: each ring slot holds the codes of
//     four consecutive chunks, chunk 4g + b in byte b of every cell (the
//     instruction descriptor selects the byte), written with tcgen05.st;
//   - warps 8-15: epilogue: after a tile's last MMA they read its
//     accumulator in 32-column loads, hand it back after the last load, and
//     convert and store.  BN = 128 tiles have two accumulators, so the next
//     tile's MMAs overlap the epilogue; a BN = 256 accumulator takes half of
//     TMEM and the scale-factor ring the rest, so the next tile starts once
//     the accumulator has been read.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fgq_device.cuh"
#include "fgq_internal.h"

namespace fgq {
namespace {

constexpr int BM = 128;
constexpr int BK = 128;
constexpr int kThreads = 512;  // warpgroup 0 control, 1 scale factors, 2-3 epilogue
constexpr int kEpiWarps = 8;
constexpr int kSlots = 4;              // scale-factor ring
constexpr int kChunksPerSlot = 4;      // one byte of each cell per chunk
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfaCol0 = 256;     // slot r: A factors at kSfaCol0 + 32 r (+ 0..3)
constexpr uint32_t kSfbCol0 = 384;     // slot r: B factors at kSfbCol0 + 32 r (+ 0..7)

template <int BN, int STAGES>
struct MxCfg {
  static constexpr int kNAcc = BN == 128 ? 2 : 1;  // accumulators in TMEM columns 0..255
  static constexpr int kABytes = BM * BK;
  static constexpr int kBBytes = BN * BK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kNumBars = 2 * STAGES + 2 * kSlots + 2 * kNAcc + 1;
  static constexpr int kStoreBytes = kEpiWarps * 2048;  // per-warp staging of C rows
  static constexpr size_t kSmemBytes =
      1024 + static_cast<size_t>(STAGES) * kStageBytes + kStoreBytes + kNumBars * 8 + 16;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kNAcc * BN <= static_cast<int>(kSfaCol0), "accumulators overlap the scale ring");
  static_assert(BN / 32 <= 8, "B factors of one slot take BN/32 <= 8 columns");
};

__device__ __forceinline__ bool mx_wait_drain(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > FGQ_WAIT_NS) {
      record_error(FGQ_DEVERR_DRAIN);
      return false;
    }
  }
  return true;
}

// UE8M0 code of a power-of-two fp32 scale 2^e, e in [-127, 127]: its biased
// exponent field (2^-127 is the subnormal 0x00400000, whose field is 0).
__device__ __forceinline__ uint32_t ue8m0_code(float s) { return (__float_as_uint(s) >> 23) & 0xFFu; }

template <int BN, int STAGES, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, const float* __restrict__ sA,
                   const float* __restrict__ sB, void* __restrict__ C, int64_t ldc, int M, int N,
                   int K) {
  using CF = MxCfg<BN, STAGES>;
  constexpr int NACC = CF::kNAcc;
  constexpr int HALF = BN / 2;    // columns per epilogue warp
  constexpr int NLD = HALF / 32;  // 32-column loads per warp and tile
  static_assert(NLD >= 2, "the load pipeline assumes at least two loads");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sm_a = smem;
  uint8_t* sm_b = smem + STAGES * CF::kABytes;
  uint8_t* sm_st = sm_b + STAGES * CF::kBBytes;  // C row staging, 2 KB per epilogue warp
  uint64_t* full = reinterpret_cast<uint64_t*>(sm_st + CF::kStoreBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* sf_full = empty + STAGES;
  uint64_t* sf_empty = sf_full + kSlots;
  uint64_t* acc_full = sf_empty + kSlots;
  uint64_t* acc_empty = acc_full + NACC;
  uint64_t* drain = acc_empty + NACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (M + BM - 1) / BM;
  const int n_tiles = N / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int kchunks = K / BK;
  const int nb = N / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int r = 0; r < kSlots; ++r) {
      mbar_init(&sf_full[r], 4);
      mbar_init(&sf_empty[r], 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above (barrier set-up, TMEM allocation) may overlap the
  // previous kernel in the stream; global memory is touched only after it
  // has completed.
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (elect_one_sync()) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int tm = tile % m_tiles, tn = tile / m_tiles;
        for (int kc = 0; kc < kchunks; ++kc, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, FGQ_DEVERR_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], CF::kStageBytes);
          tma_load_2d(sm_a + s * CF::kABytes, &tmap_a, &full[s], kc * BK, tm * BM);
          tma_load_2d(sm_b + s * CF::kBBytes, &tmap_b, &full[s], kc * BK, tn * BN);
        }
      }
      // No copy may still target this CTA's shared memory when it exits.
      const uint32_t first = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u;
      for (uint32_t j = first; j < it; ++j) mx_wait_drain(&full[j % STAGES], (j / STAGES) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (elect_one_sync()) {
      constexpr uint32_t idesc0 = idesc_mx_e4m3_ue8m0(BM, BN);
      const uint64_t dA0 = smem_desc_k_sw128(smem_u32(sm_a));
      const uint32_t a_lo0 = static_cast<uint32_t>(dA0), dhi = static_cast<uint32_t>(dA0 >> 32);
      const uint32_t b_lo0 = static_cast<uint32_t>(smem_desc_k_sw128(smem_u32(sm_b)));
      int ls = 0;
      uint32_t lph = 0, g_it = 0, t_it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++t_it) {
        const uint32_t buf = t_it % NACC, aph = (t_it / NACC) & 1u;
        if (!mbar_wait(&acc_empty[buf], aph ^ 1u, abort_flag, FGQ_DEVERR_MMA_TMEM)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * BN;
        uint32_t tsfa = 0, tsfb = 0, r = 0;
        for (int kc = 0; kc < kchunks; ++kc) {
          const uint32_t id = static_cast<uint32_t>(kc) & 3u;
          if (id == 0) {
            r = g_it % kSlots;
            if (!mbar_wait(&sf_full[r], (g_it / kSlots) & 1u, abort_flag, FGQ_DEVERR_MMA_SF)) {
              ok = false;
              break;
            }
            tsfa = tmem_base + kSfaCol0 + 32u * r;
            tsfb = tmem_base + kSfbCol0 + 32u * r;
          }
          if (!mbar_wait(&full[ls], lph, abort_flag, FGQ_DEVERR_MMA_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t idesc = idesc0 | (id << 29) | (id << 4);
          const uint32_t a_lo = a_lo0 + ls * (CF::kABytes >> 4);
          const uint32_t b_lo = b_lo0 + ls * (CF::kBBytes >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            umma_mxf8f6f4(d, make_desc(a_lo + kk * 2, dhi), make_desc(b_lo + kk * 2, dhi), idesc,
                          tsfa, tsfb, (kc > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty[ls]);
          if (id == kChunksPerSlot - 1 || kc == kchunks - 1) {
            umma_commit(&sf_empty[r]);
            ++g_it;
          }
          if (++ls == STAGES) {
            ls = 0;
            lph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&acc_full[buf]);
      }
      // Every MMA this thread issued must finish before TMEM is released.
      umma_commit(drain);
      mx_wait_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ---------------- scale-factor writers ----------------
    const int q = warp & 3;
    const uint32_t t_lane = static_cast<uint32_t>(32 * q) << 16;
    const int groups = (kchunks + kChunksPerSlot - 1) / kChunksPerSlot;
    uint32_t g_it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      const int tm = tile % m_tiles, tn = tile / m_tiles;
      const int row = tm * BM + 32 * q + lane;
      const bool row_ok = row < M;
      const float* sa_row = sA + static_cast<int64_t>(row_ok ? row : 0) * kchunks;
      const int nb0 = tn * (BN / 128);
      for (int g = 0; g < groups; ++g, ++g_it) {
        const uint32_t r = g_it % kSlots;
        // A's codes for this thread's row, B's for the tile's column blocks
        uint32_t wa = 0x7F7F7F7Fu, wb0 = 0x7F7F7F7Fu, wb1 = 0x7F7F7F7Fu;
#pragma unroll
        for (int b = 0; b < kChunksPerSlot; ++b) {
          const int c = g * kChunksPerSlot + b;
          if (c < kchunks) {
            const uint32_t sh = 8u * b;
            if (row_ok) wa = (wa & ~(0xFFu << sh)) | (ue8m0_code(__ldg(sa_row + c)) << sh);
            const float* sbc = sB + static_cast<int64_t>(c) * nb + nb0;
            wb0 = (wb0 & ~(0xFFu << sh)) | (ue8m0_code(__ldg(sbc)) << sh);
            if (BN == 256) wb1 = (wb1 & ~(0xFFu << sh)) | (ue8m0_code(__ldg(sbc + 1)) << sh);
          }
        }
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sf_empty[r], ((g_it / kSlots) & 1u) ^ 1u,
                                               abort_flag, FGQ_DEVERR_SF_SLOT))) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st_32x32b_x1(tmem_base + t_lane + kSfaCol0 + 32u * r + static_cast<uint32_t>(q), wa);
        if (BN == 256)
          tmem_st_32x32b_x8_aabb(tmem_base + t_lane + kSfbCol0 + 32u * r, wb0, wb1);
        else
          tmem_st_32x32b_x4(tmem_base + t_lane + kSfbCol0 + 32u * r, wb0);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_full[r]);
      }
    }
  } else if (warp >= 8) {
    // ---------------- epilogue ----------------
    const int ew = warp - 8;
    const int q = warp & 3;
    const int half = ew >> 2;
    const uint32_t t_lane = static_cast<uint32_t>(32 * q) << 16;
    uint32_t t_it = 0;
    uint8_t* stage = sm_st + ew * 2048;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++t_it) {
      const int tm = tile % m_tiles, tn = tile / m_tiles;
      const int row0 = tm * BM + 32 * q;  // the warp's first row
      const int col0 = tn * BN + half * HALF;
      const uint32_t buf = t_it % NACC, aph = (t_it / NACC) & 1u;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&acc_full[buf], aph, abort_flag, FGQ_DEVERR_EPI_TMEM)))
        break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + t_lane + buf * BN + half * HALF;
      uint32_t ra[32], rb[32];
      tmem_ld_32x32b_x32(taddr, ra);
      tmem_wait_ld_regs(ra);
#pragma unroll
      for (int j = 0; j < NLD; ++j) {
        if (j + 1 < NLD) {
          if (j % 2 == 0)
            tmem_ld_32x32b_x32(taddr + 32 * (j + 1), rb);
          else
            tmem_ld_32x32b_x32(taddr + 32 * (j + 1), ra);
        } else {
          // the whole accumulator is in registers: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
        // the warp's rows go out through its staging buffer (whole row
        // segments per store instruction)
        if (j % 2 == 0)
          warp_store32<OUT_BF16>(stage, ra, C, ldc, row0, col0 + 32 * j, M - row0);
        else
          warp_store32<OUT_BF16>(stage, rb, C, ldc, row0, col0 + 32 * j, M - row0);
        if (j + 1 < NLD) {
          if (j % 2 == 0)
            tmem_wait_ld_regs(rb);
          else
            tmem_wait_ld_regs(ra);
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int BN, int STAGES, bool OUT_BF16>
cudaError_t launch_mx_cfg(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                          void* C, int64_t ldc, int M, int N, int K, cudaStream_t stream,
                          const DeviceInfo& dev) {
  using CF = MxCfg<BN, STAGES>;
  auto kern = gemm_mx_kernel<BN, STAGES, OUT_BF16>;
  static bool attr_set[64] = {};
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev.device < 64 && !attr_set[dev.device]) {
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(CF::kSmemBytes));
      if (e != cudaSuccess) return e;
      attr_set[dev.device] = true;
    }
  }
  CUtensorMap ta, tb;
  if (!make_k_major_map(&ta, A, M, K, BM) || !make_k_major_map(&tb, B, N, K, BN))
    return cudaErrorInvalidValue;
  const int tiles = ((M + BM - 1) / BM) * (N / BN);
  const int grid = tiles < dev.sm_count ? tiles : dev.sm_count;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), CF::kSmemBytes, stream, ta, tb, sA, sB, C,
                    ldc, M, N, K);
}

}  // namespace

cudaError_t launch_gemm_mx(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                           void* C, int64_t ldc, int64_t M, int64_t N, int64_t K, int out_bf16,
                           cudaStream_t stream, const DeviceInfo& dev) {
  if (M == 0 || N == 0) return cudaSuccess;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  const int64_t tiles256 = ((M + BM - 1) / BM) * (N / 256);
  const bool wide = (N % 256 == 0) && tiles256 >= dev.sm_count;
  if (out_bf16) {
    return wide ? launch_mx_cfg<256, 4, true>(A, sA, B, sB, C, ldc, m, n, k, stream, dev)
                : launch_mx_cfg<128, 6, true>(A, sA, B, sB, C, ldc, m, n, k, stream, dev);
  }
  return wide ? launch_mx_cfg<256, 4, false>(A, sA, B, sB, C, ldc, m, n, k, stream, dev)
              : launch_mx_cfg<128, 6, false>(A, sA, B, sB, C, ldc, m, n, k, stream, dev);
}

// ---- UE8M0 codes in the tiled scale layout ------------------------------------
//
// For the tiled-scale FP8 GEMM (gemm_mxf4.cu, kind MXF8): the codes of a
// power-of-two scale matrix laid out as the FP4 scale tiles, F = K/128 codes
// a row padded to a multiple of 4 (padding codes 0).  Activation scales
// sA [M, K/128] give row m's codes; weight scales sB [K/128, N/128] give
// column n of the transposed weight the codes of its blocks, sB[c, n/128].
// One thread per output word (a cell: four codes of one row), consecutive
// threads writing consecutive words of a tile.
template <bool WEIGHT>
__global__ void __launch_bounds__(256)
    ue8m0_scale_tiles_kernel(const float* __restrict__ s, uint32_t R, uint32_t F, uint32_t cpr,
                             uint32_t nb, uint32_t words, uint32_t* __restrict__ tiles) {
  for (uint32_t w = blockIdx.x * 256u + threadIdx.x; w < words; w += gridDim.x * 256u) {
    const uint32_t tile = w >> 7, in = w & 127u;
    const uint32_t rt = tile / cpr, c = tile - rt * cpr;
    const uint32_t r = rt * 128u + 32u * (in & 3u) + (in >> 2);
    uint32_t cell = 0;
    if (r < R) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t f = 4u * c + b;
        if (f < F) {
          const float v = WEIGHT ? __ldg(s + static_cast<uint64_t>(f) * nb + r / 128u)
                                 : __ldg(s + static_cast<uint64_t>(r) * F + f);
          cell |= ue8m0_code(v) << (8 * b);
        }
      }
    }
    tiles[w] = cell;
  }
}

cudaError_t launch_ue8m0_scale_tiles(const float* s, int64_t R, int64_t K, int64_t N, bool weight,
                                     uint8_t* tiles, cudaStream_t stream, const DeviceInfo& dev) {
  const uint32_t F = static_cast<uint32_t>(K / 128), cpr = (F + 3) / 4;
  const uint64_t words = static_cast<uint64_t>((R + 127) / 128) * cpr * 128u;
  if (words == 0) return cudaSuccess;
  if (words >= (uint64_t{1} << 32)) return cudaErrorInvalidValue;  // 16 GB of tiles
  uint64_t grid = (words + 255) / 256;
  const uint64_t cap = static_cast<uint64_t>(dev.sm_count) * 8;
  if (grid > cap) grid = cap;
  auto k = weight ? ue8m0_scale_tiles_kernel<true> : ue8m0_scale_tiles_kernel<false>;
  k<<<static_cast<unsigned>(grid), 256, 0, stream>>>(s, static_cast<uint32_t>(R), F, cpr,
                                                      static_cast<uint32_t>(N / 128),
                                                      static_cast<uint32_t>(words),
                                                      reinterpret_cast<uint32_t*>(tiles));
  return cudaGetLastError();
}

cudaError_t read_device_error_mx(uint32_t* word, bool clear) {
  return read_unit_device_error(word, clear);
}

}  // namespace fgq
