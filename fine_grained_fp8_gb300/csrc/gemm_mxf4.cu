// FP4 GEMMs for sm_103a: E2M1 elements with block scales along K on both
// operands ("Fine-Grained FP8/FP4 Quantization", §UE8M0 vs E4M3 Scale
// Formats; §NVFP4 Two-Level Scaling; §When to Use: NVFP4 with E4M3 block
// scales for precision, MXFP4 with UE8M0 scales for native acceleration):
//
//   MXFP4  C[m,n] = sum_k e2m1(A[m,k]) 2^(sA[m,k/32]-127) e2m1(B[n,k]) 2^(sB[n,k/32]-127)
//   NVFP4  C[m,n] = gA gB sum_k e2m1(A[m,k]) e4m3(sA[m,k/16]) e2m1(B[n,k]) e4m3(sB[n,k/16])
//
// tcgen05.mma kind::mxf4 (scale_vec::2X, UE8M0) or kind::mxf4nvf4
// (scale_vec::4X, UE4M3) takes K = 64 packed E2M1 elements (32 bytes a
// row) and the block factors of that K range per row of A and per column
// of B, applied by the tensor core; the fp32 accumulator stays in TMEM for
// the whole K loop.  Measured factor layout (as for kind::mxf8f6f4 with
// scale_vec::1X): A's row m at lane m, column base + m/32; B's column n at
// lane 32 q + n%32, column base + n/32.  2X: the descriptor's factor id 0
// reads bytes 0-1 of the cell (the two 32-element blocks of one MMA), id 2
// bytes 2-3.  4X: byte b of the cell scales the MMA's b-th 16-element block.
//
// Two kernels:
//   - gemm_mxf4_kernel, for block scales stored row-major ([rows, K/32] or
//     [rows, K/16]): the same structure as the power-of-two FP8 kernel
//     (gemm_mx.cu), persistent CTAs on 128 x BN tiles, warp 0 TMA producer
//     (one 128-byte stage = 256 elements of K), warp 1 MMA issuer (factor
//     copies, four MMAs per stage), warps 4-7 gather the factors into
//     shared memory, warps 8-15 epilogue;
//   - gemm_fp4_tiled_kernel, for block scales stored as tiles the
//     tensor-map engine loads with the operands (no factor warps), on CTA
//     pairs once A has two row tiles.  It also serves the FP8 GEMM with
//     power-of-two scales given as UE8M0 code tiles (kind MXF8:
//     kind::mxf8f6f4.block_scale.scale_vec::1X, 128 elements a stage).
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
constexpr uint32_t kTmemCols = 512;

// The two FP4 formats.  MXFP4: one UE8M0 factor per 32 elements, MMA
// kind::mxf4 with scale_vec::2X (a 32-bit factor cell serves two K = 64
// MMAs, the descriptor's factor id picking bytes 0-1 or 2-3).  NVFP4: one
// E4M3 factor per 16 elements, kind::mxf4nvf4 with scale_vec::4X (one cell
// per MMA, byte b scaling its b-th 16-element block; measured), and an fp32
// per-tensor scale on each operand, applied in the epilogue.
//
// Scale-factor ring: a slot = one stage = 256 elements of K = four K = 64
// MMAs = kCells 32-bit cells per row of A and per column of B.  Cell w of A
// sits at the slot's A base + 4 w (+ 0..3 for the four row quarters), cell
// w of B at its B base + 8 w (+ 0..7 for the column groups); the factor
// addresses need only 4-column (A) and 8-column (B) alignment (measured).
// The writers stage the codes in chunks of 32 bytes per row, kChunkStages
// stages, in shared memory tiles the issuer copies into the slot with
// tcgen05.cp.32x128b.warpx4 (32 rows of 16 bytes, row i to lane 32 q + i of
// every lane quarter q, word j to column j; measured).  A tile of cell c
// holds, in row i, the cells of rows i, 32 + i, 64 + i, 96 + i of A (of
// columns 128 h + i + 32 j of B): A's row m lands at lane m, column
// base + m/32, and B's column n at lane 32 q + n%32, column base + n/32 —
// the layouts the MMA reads.
template <bool NV>
struct Fp4Fmt {
  static constexpr int kBlock = NV ? 16 : 32;      // elements per factor
  static constexpr int kCells = NV ? 4 : 2;        // factor cells per row per stage
  static constexpr int kSlots = NV ? 5 : 8;  // >= operand stages + kChunkStages - 1
  static constexpr uint32_t kSfaSlot = 4 * kCells, kSfbSlot = 8 * kCells;
  static constexpr uint32_t kSfaCol0 = 256;        // after the accumulators
  static constexpr uint32_t kSfbCol0 = kSfaCol0 + kSfaSlot * kSlots;
  static constexpr int kChunkStages = 8 / kCells;  // 32 bytes of codes per row
};

template <int BN, int STAGES, bool NV>
struct Mxf4Cfg {
  using F = Fp4Fmt<NV>;
  static constexpr int kNAcc = BN == 128 ? 2 : 1;  // accumulators in TMEM columns 0..255
  static constexpr int kABytes = BM * BK;
  static constexpr int kBBytes = BN * BK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kNumBars = 2 * STAGES + 4 + 2 * kNAcc + 1;
  // factor staging: two chunk buffers of 8 A tiles (one per cell of the
  // chunk) and 8 BN/128 B tiles; tiles 528 bytes apart (16-byte aligned, and
  // shifted by four banks so a warp's 4-byte writes to eight tiles at one
  // row and four words never share a bank)
  static constexpr int kSfTile = 528;
  static constexpr int kTilesB = 8 * (BN / 128);
  static constexpr int kSfBufBytes = (8 + kTilesB) * kSfTile;
  static constexpr int kStoreBytes = kEpiWarps * 1024;  // per-warp staging of C rows
  static constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(STAGES) * kStageBytes +
                                       2 * kSfBufBytes + kStoreBytes + kNumBars * 8 + 16;
  // At the first stage s of a chunk the issuer, past the full[] wait of
  // stage s (whose TMA waited for the MMAs of stage s - STAGES), copies the
  // factors of stages s .. s + kChunkStages - 1; the slot of stage s + j last
  // served stage s + j - kSlots <= s - STAGES, whose MMAs have completed.
  static_assert(F::kSlots >= STAGES + F::kChunkStages - 1, "factor ring too short");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kNAcc * BN <= static_cast<int>(F::kSfaCol0), "accumulators overlap the scale ring");
  static_assert(F::kSfbCol0 % 8 == 0 && F::kSfbCol0 + F::kSfbSlot * F::kSlots <= kTmemCols,
                "scale ring within TMEM");
  static_assert(BN / 32 <= 8, "B factors of one slot take BN/32 <= 8 columns");
};

__device__ __forceinline__ bool mxf4_wait_drain(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > FGQ_WAIT_NS) {
      record_error(FGQ_DEVERR_DRAIN);
      return false;
    }
  }
  return true;
}

// A and B E2M1 (type 1); factors UE8M0 (bit 23 set, MXFP4) or UE4M3 (bit 23
// clear, NVFP4); factor ids 0.
__host__ __device__ constexpr uint32_t idesc_fp4(int m, int n, bool nv) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (nv ? 0u : 1u << 23) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void umma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// tcgen05.cp of a 32-row x 16-byte shared-memory tile to TMEM columns
// taddr .. taddr + 3 of all four lane quarters, and the no-swizzle
// descriptor of such a tile (four 8-row core matrices 128 bytes apart).
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
__device__ __forceinline__ uint64_t sf_tile_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 32) |
         (uint64_t{1} << 46);
}

// 4-byte asynchronous copy global -> shared (cp.async), the group commit,
// the wait for all of this thread's groups, and the fence that orders this
// thread's shared-memory writes before later async-proxy (tensor core) reads.
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int BN, int STAGES, bool OUT_BF16, bool NV>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mxf4_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, const uint8_t* __restrict__ sA,
                   const uint8_t* __restrict__ sB, const float* __restrict__ ga,
                   const float* __restrict__ gb, void* __restrict__ C, int64_t ldc, int M, int N,
                   int K) {
  using CF = Mxf4Cfg<BN, STAGES, NV>;
  using F = Fp4Fmt<NV>;
  constexpr int kSlots = F::kSlots;
  constexpr uint32_t kSfaSlot = F::kSfaSlot, kSfbSlot = F::kSfbSlot;
  constexpr uint32_t kSfaCol0 = F::kSfaCol0, kSfbCol0 = F::kSfbCol0;
  constexpr int kCells = F::kCells, kCh = F::kChunkStages;
  constexpr int NACC = CF::kNAcc;
  constexpr int HALF = BN / 2;    // columns per epilogue warp
  constexpr int NLD = HALF / 32;  // 32-column loads per warp and tile
  static_assert(NLD >= 2, "the load pipeline assumes at least two loads");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sm_a = smem;
  uint8_t* sm_b = smem + STAGES * CF::kABytes;
  uint8_t* sf_stage = sm_b + STAGES * CF::kBBytes;  // two chunk buffers of factor tiles
  uint8_t* sm_st = sf_stage + 2 * CF::kSfBufBytes;   // C row staging, 1 KB per epilogue warp
  uint64_t* full = reinterpret_cast<uint64_t*>(sm_st + CF::kStoreBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* sf_full = empty + STAGES;
  uint64_t* sf_empty = sf_full + 2;
  uint64_t* acc_full = sf_empty + 2;
  uint64_t* acc_empty = acc_full + NACC;
  uint64_t* drain = acc_empty + NACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (M + BM - 1) / BM;
  const int n_tiles = N / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int kstages = (K + 255) / 256;  // 128-byte stages of 256 elements (the last may be half)
  const bool half_last = (K % 256) != 0;  // the last stage holds 128 elements of K
  const int kg = K / F::kBlock;         // factor codes per row of sA / sB

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sf_full[b], 4);   // one arrival per writer warp
      mbar_init(&sf_empty[b], 1);  // the issuer's commit after the chunk's MMAs
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
        for (int kc = 0; kc < kstages; ++kc, ++it) {
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
      for (uint32_t j = first; j < it; ++j) mxf4_wait_drain(&full[j % STAGES], (j / STAGES) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (elect_one_sync()) {
      constexpr uint32_t idesc0 = idesc_fp4(BM, BN, NV);
      constexpr uint32_t kId2 = (2u << 29) | (2u << 4);  // factor bytes 2-3 of A and B
      const uint64_t dA0 = smem_desc_k_sw128(smem_u32(sm_a));
      const uint32_t a_lo0 = static_cast<uint32_t>(dA0), dhi = static_cast<uint32_t>(dA0 >> 32);
      const uint32_t b_lo0 = static_cast<uint32_t>(smem_desc_k_sw128(smem_u32(sm_b)));
      const uint32_t sf0 = smem_u32(sf_stage);
      int ls = 0;
      uint32_t lph = 0, g_it = 0, t_it = 0, gch = 0;  // gch: factor chunks consumed
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++t_it) {
        const uint32_t buf = t_it % NACC, aph = (t_it / NACC) & 1u;
        if (!mbar_wait(&acc_empty[buf], aph ^ 1u, abort_flag, FGQ_DEVERR_MMA_TMEM)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * BN;
        for (int kc = 0; kc < kstages; ++kc, ++g_it) {
          const int st = kc % kCh;  // stage within the factor chunk
          if (!mbar_wait(&full[ls], lph, abort_flag, FGQ_DEVERR_MMA_FULL)) {
            ok = false;
            break;
          }
          // Factors into their slots, in order before the MMAs that read
          // them: cell w of A to columns 4 w .. 4 w + 3 of a slot's A part,
          // cell w of B columns 128 h .. 128 h + 127 to columns 8 w + 4 h ..
          // + 3 of its B part.  NVFP4 (two-stage chunks) copies a whole
          // chunk at its first stage and hands the buffer back at once;
          // MXFP4 copies stage by stage and hands it back after its last
          // stage's copies, before that stage's MMAs.
          constexpr bool kBulk = NV;
          const uint32_t cb = gch & 1u;
          const bool last = st == kCh - 1 || kc + 1 == kstages;
          if (st == 0 && !mbar_wait(&sf_full[cb], (gch >> 1) & 1u, abort_flag, FGQ_DEVERR_MMA_SF)) {
            ok = false;
            break;
          }
          if (!kBulk || st == 0) {
            tc_fence_after();
            const uint32_t tiles = sf0 + cb * CF::kSfBufBytes;
            const int j0 = kBulk ? 0 : st;
            const int j1 = kBulk ? (kstages - kc < kCh ? kstages - kc : kCh) : st + 1;
            for (int j = j0; j < j1; ++j) {
              const uint32_t rj = (g_it + (j - st)) % kSlots;
#pragma unroll
              for (int w = 0; w < kCells; ++w) {
                const int cc = j * kCells + w;
                tmem_cp_32x128b_x4(tmem_base + kSfaCol0 + kSfaSlot * rj + 4 * w,
                                   sf_tile_desc(tiles + cc * CF::kSfTile));
#pragma unroll
                for (int h = 0; h < BN / 128; ++h)
                  tmem_cp_32x128b_x4(tmem_base + kSfbCol0 + kSfbSlot * rj + 8 * w + 4 * h,
                                     sf_tile_desc(tiles + (8 + cc * (BN / 128) + h) * CF::kSfTile));
              }
            }
            if (kBulk || last) umma_commit(&sf_empty[cb]);
          }
          if (last) ++gch;
          tc_fence_after();
          const uint32_t a_lo = a_lo0 + ls * (CF::kABytes >> 4);
          const uint32_t b_lo = b_lo0 + ls * (CF::kBBytes >> 4);
          const uint32_t r = g_it % kSlots;
          const uint32_t sfa = tmem_base + kSfaCol0 + kSfaSlot * r;
          const uint32_t sfb = tmem_base + kSfbCol0 + kSfbSlot * r;
          // four K = 64 MMAs (32 bytes of each row apart); a final half
          // stage has two.  MXFP4: factor bytes 0-1 and 2-3 of cell 0, then
          // of cell 1.  NVFP4: cell kk for MMA kk.
          const bool full_stage = kc + 1 < kstages || !half_last;
          if constexpr (NV) {
            umma_nvf4(d, make_desc(a_lo, dhi), make_desc(b_lo, dhi), idesc0, sfa, sfb,
                      kc > 0 ? 1u : 0u);
            umma_nvf4(d, make_desc(a_lo + 2, dhi), make_desc(b_lo + 2, dhi), idesc0, sfa + 4,
                      sfb + 8, 1u);
            if (full_stage) {
              umma_nvf4(d, make_desc(a_lo + 4, dhi), make_desc(b_lo + 4, dhi), idesc0, sfa + 8,
                        sfb + 16, 1u);
              umma_nvf4(d, make_desc(a_lo + 6, dhi), make_desc(b_lo + 6, dhi), idesc0, sfa + 12,
                        sfb + 24, 1u);
            }
          } else {
            umma_mxf4(d, make_desc(a_lo, dhi), make_desc(b_lo, dhi), idesc0, sfa, sfb,
                      kc > 0 ? 1u : 0u);
            umma_mxf4(d, make_desc(a_lo + 2, dhi), make_desc(b_lo + 2, dhi), idesc0 | kId2, sfa,
                      sfb, 1u);
            if (full_stage) {
              umma_mxf4(d, make_desc(a_lo + 4, dhi), make_desc(b_lo + 4, dhi), idesc0, sfa + 4,
                        sfb + 8, 1u);
              umma_mxf4(d, make_desc(a_lo + 6, dhi), make_desc(b_lo + 6, dhi), idesc0 | kId2,
                        sfa + 4, sfb + 8, 1u);
            }
          }
          umma_commit(&empty[ls]);
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
      mxf4_wait_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ---------------- scale-factor writers ----------------
    // The factors of a tile's rows (columns) are one contiguous block of
    // BM (BN) rows of kg codes.  Per chunk (32 bytes of every row) the four
    // warps copy each 4-byte cell with cp.async straight into its place in
    // the chunk buffer's tiles: lane l takes cell l % 8 of the chunk and row
    // quarter l / 8, so a warp instruction reads whole 32-byte sectors of
    // four rows and writes 32 different banks.  Then wait for the copies,
    // fence them to the async proxy (the tensor core reads the tiles) and
    // arrive on the buffer's full barrier.  Codes past a row's end (the final
    // partial chunk) and rows past M are not copied: they feed only unused
    // factor bytes of a final half stage or accumulator rows never stored.
    const int wq = warp & 3;
    const int c8 = lane & 7, kq = lane >> 3;
    uint32_t gch = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      const int tm = tile % m_tiles, tn = tile / m_tiles;
      const uint8_t* a_blk = sA + static_cast<int64_t>(tm) * BM * kg;
      const uint8_t* b_blk = sB + static_cast<int64_t>(tn) * BN * kg;
      const int a_rows = M - tm * BM < BM ? M - tm * BM : BM;
      const int nchunks = (kstages + kCh - 1) / kCh;
      for (int c = 0; c < nchunks; ++c, ++gch) {
        const uint32_t cb = gch & 1u;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sf_empty[cb], ((gch >> 1) & 1u) ^ 1u, abort_flag,
                                               FGQ_DEVERR_SF_SLOT))) {
          ok = false;
          break;
        }
        uint8_t* tiles = sf_stage + cb * CF::kSfBufBytes;
        const int byte = 32 * c + 4 * c8;
        if (byte < kg) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {  // A rows m = r + 32 kq, r = wq + 4 i
            const int r = wq + 4 * i, m = r + 32 * kq;
            if (m < a_rows) cp_async4(tiles + c8 * CF::kSfTile + 16 * r + 4 * kq, a_blk + m * kg + byte);
          }
#pragma unroll
          for (int i = 0; i < BN / 16; ++i) {  // B columns n = 128 h + 32 kq + r
            const int r = wq + 4 * (i % 8), h = i / 8, n = 128 * h + 32 * kq + r;
            cp_async4(tiles + (8 + c8 * (BN / 128) + h) * CF::kSfTile + 16 * r + 4 * kq,
                      b_blk + n * kg + byte);
          }
        }
        cp_async_commit();
        cp_async_wait_all();
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_full[cb]);
      }
    }
  } else if (warp >= 8) {
    // ---------------- epilogue ----------------
    const int ew = warp - 8;
    const int q = warp & 3;
    const int half = ew >> 2;
    const uint32_t t_lane = static_cast<uint32_t>(32 * q) << 16;
    // NVFP4: C = gA gB * (the tensor core's sum over E2M1 x E4M3 products)
    float alpha = 1.0f;
    if constexpr (NV) alpha = __fmul_rn(__ldg(ga), __ldg(gb));
    auto scale32 = [&](uint32_t (&r)[32]) {
      if constexpr (NV) {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[i]), alpha));
      }
    };
    uint32_t t_it = 0;
    uint8_t* stage = sm_st + (warp - 8) * 1024;
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
        if (j % 2 == 0) {
          scale32(ra);
          warp_store32<OUT_BF16, 1024>(stage, ra, C, ldc, row0, col0 + 32 * j, M - row0);
        } else {
          scale32(rb);
          warp_store32<OUT_BF16, 1024>(stage, rb, C, ldc, row0, col0 + 32 * j, M - row0);
        }
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

// ---- block scales in the tiled layout ----------------------------------------
//
// The same two products with the block scales stored in the tiled FP4 scale
// layout: 512-byte tiles of 128 rows x 4 factor bytes, row r of a tile at
// byte 16 (r % 32) + 4 ((r % 128) / 32).  Each such tile is exactly the
// 32-row x 16-byte shared-memory tile tcgen05.cp.32x128b.warpx4 spreads
// over the four lane quarters, so the factors need no gathering: the
// producer loads a stage's factor tiles with the tensor-map engine next to
// its operand tiles (one `full` barrier for both), and the issuer copies
// them into a TMEM slot before the stage's MMAs.  There are no
// factor-writer warps.
//
// PAIR: 256 x BN tiles on clusters of two CTAs.  Each CTA holds 128 rows of
// A and BN/2 of the tile's BN columns of B, and the even CTA (leader)
// issues tcgen05.mma.cta_group::2 (M = 256), so each SM takes in A plus
// half of B per stage for the MMA work a single CTA needs A plus all of B
// for.  Each CTA loads the factor tiles of its own rows of A and of all BN
// columns of B (the MMA reads, in each CTA's TMEM, its own rows' A factors
// and every column's B factors); the leader's tcgen05.cp.cta_group::2
// copies each CTA's tiles into that CTA's TMEM.  Both CTAs' tensor-map
// copies complete on the leader's `full` barrier; the leader's commits
// arrive on the `empty` and `acc_full` barriers of both CTAs (multicast);
// both epilogues hand the accumulator back on the leader's `acc_empty`
// (the peer with a relaxed cluster arrive after tcgen05.wait::ld, when its
// reads have completed).
// The three block-scaled kinds on tiled scales: MXFP4 (E2M1, UE8M0 per 32
// elements), NVFP4 (E2M1, E4M3 per 16) and MXF8 (E4M3 operands, one UE8M0
// code per 128-element chunk of a row of A and per 128 x 128 block of the
// weight: the power-of-two scales of the FP8 GEMM, applied by
// kind::mxf8f6f4.block_scale.scale_vec::1X).  A stage is 128 bytes of
// every row: 256 elements of K for FP4, 128 for FP8.
constexpr int kMx4 = 0, kNv4 = 1, kMx8 = 2;

template <int KIND>
struct Fp4TiledFmt {
  // factor tiles per 128 rows per stage (MXF8: one tile serves four stages,
  // its bytes b = 0..3 the codes of chunks 4 g + b)
  static constexpr int kCells = KIND == kNv4 ? 4 : KIND == kMx4 ? 2 : 1;
  static constexpr int kSlots = KIND == kNv4 ? 5 : KIND == kMx4 ? 10 : 12;
  static constexpr uint32_t kSfaSlot = 4 * kCells, kSfbSlot = 8 * kCells;
  static constexpr uint32_t kSfaCol0 = 256;     // after the accumulators
  static constexpr uint32_t kSfbCol0 = kSfaCol0 + kSfaSlot * kSlots;
};

template <bool PAIR, int BN, int KIND>
struct TiledCfg {
  using F = Fp4TiledFmt<KIND>;
  static constexpr int kNAcc = BN == 128 ? 2 : 1;
  static constexpr int kABytes = BM * BK;                    // this CTA's 128 rows of A
  static constexpr int kBRows = PAIR ? BN / 2 : BN;          // this CTA's rows of B
  static constexpr int kBBytes = kBRows * BK;
  static constexpr int kSfABytes = F::kCells * 512;
  static constexpr int kSfBBytes = (BN / 128) * F::kCells * 512;
  static constexpr int kSfBytes = kSfABytes + kSfBBytes;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfBytes;
  static constexpr uint32_t kTxBytes = (PAIR ? 2 : 1) * kStageBytes;
  static constexpr int kStoreBytes = kEpiWarps * 1024;
  static constexpr int kFit = (232448 - 1024 - kStoreBytes - 256) / kStageBytes;
  static constexpr int STAGES = kFit < F::kSlots ? kFit : F::kSlots;
  static constexpr int kNumBars = 2 * STAGES + 2 * kNAcc + 1;
  static constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(STAGES) * kStageBytes +
                                       kStoreBytes + kNumBars * 8 + 16;
  // the slot of stage s last served stage s - kSlots <= s - STAGES, whose
  // MMAs completed before the copy into full[s]'s buffer was issued
  static_assert(F::kSlots >= STAGES && STAGES >= 3, "stages");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kNAcc * BN <= static_cast<int>(F::kSfaCol0), "accumulators overlap the scale ring");
  static_assert(F::kSfbCol0 % 8 == 0 && F::kSfbCol0 + F::kSfbSlot * F::kSlots <= kTmemCols,
                "scale ring within TMEM");
  static_assert(kBBytes % 1024 == 0 && kSfBytes % 512 == 0, "tile alignment");
};

__device__ __forceinline__ void umma_mxf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t sfa_tmem,
                                               uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_nvf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t sfa_tmem,
                                               uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// tcgen05.cp issued by the leader of a pair: each CTA's tile at this
// shared-memory offset into the same TMEM columns of that CTA.
__device__ __forceinline__ void tmem_cp_32x128b_x4_pair(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

__device__ __forceinline__ void umma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t sfa_tmem,
                                               uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

template <bool PAIR, int KIND>
__device__ __forceinline__ void fp4_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t sfa, uint32_t sfb, uint32_t acc) {
  if constexpr (PAIR) {
    if constexpr (KIND == kNv4)
      umma_nvf4_pair(d, a, b, idesc, sfa, sfb, acc);
    else if constexpr (KIND == kMx4)
      umma_mxf4_pair(d, a, b, idesc, sfa, sfb, acc);
    else
      umma_mxf8_pair(d, a, b, idesc, sfa, sfb, acc);
  } else {
    if constexpr (KIND == kNv4)
      umma_nvf4(d, a, b, idesc, sfa, sfb, acc);
    else if constexpr (KIND == kMx4)
      umma_mxf4(d, a, b, idesc, sfa, sfb, acc);
    else
      umma_mxf8f6f4(d, a, b, idesc, sfa, sfb, acc);
  }
}

template <bool PAIR, int BN, bool OUT_BF16, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp4_tiled_kernel(const __grid_constant__ CUtensorMap tmap_a,
                          const __grid_constant__ CUtensorMap tmap_b,
                          const __grid_constant__ CUtensorMap tmap_sa,
                          const __grid_constant__ CUtensorMap tmap_sb,
                          const float* __restrict__ ga, const float* __restrict__ gb,
                          void* __restrict__ C, int64_t ldc, int M, int N, int K) {
  using CF = TiledCfg<PAIR, BN, KIND>;
  using F = Fp4TiledFmt<KIND>;
  constexpr bool NV = KIND == kNv4, FP8 = KIND == kMx8;
  constexpr int STAGES = CF::STAGES;
  constexpr int kSlots = F::kSlots;
  constexpr int kCells = F::kCells;
  constexpr int NACC = CF::kNAcc;
  constexpr int G = PAIR ? 2 : 1;  // CTAs per tile
  constexpr int HALF = BN / 2;     // columns per epilogue warp
  constexpr int NLD = HALF / 32;   // 32-column loads per warp and tile
  constexpr uint16_t kMask = 0x3;
  static_assert(NLD >= 2, "the load pipeline assumes at least two loads");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sm_a = smem;
  uint8_t* sm_b = sm_a + STAGES * CF::kABytes;
  uint8_t* sm_sf = sm_b + STAGES * CF::kBBytes;  // per stage: A factor tiles, then B's
  uint8_t* sm_st = sm_sf + STAGES * CF::kSfBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm_st + CF::kStoreBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + NACC;
  uint64_t* drain = acc_empty + NACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = rank == 0;
  // tiles of G stacked 128-row tiles x BN columns, M fastest; a cluster (a
  // CTA) takes tiles first, first + stride, ...
  const int m_tiles = (M + BM - 1) / BM;
  const int m_units = (m_tiles + G - 1) / G;
  const int total = m_units * (N / BN);
  const int first = static_cast<int>(blockIdx.x) / G;
  const int stride = static_cast<int>(gridDim.x) / G;
  // stages of 128 bytes a row (FP4: 256 elements, the last may be half)
  const int kstages = FP8 ? K / 128 : (K + 255) / 256;
  const bool half_last = !FP8 && (K % 256) != 0;
  // factor tiles per 128 rows (one per 4 factor bytes; MXF8: one per four
  // 128-element chunks, the last padded)
  const int cpr = FP8 ? (K / 128 + 3) / 4 : K / (NV ? 64 : 128);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], G * kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_sa);
    tma_prefetch_desc(&tmap_sb);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();  // both CTAs' barriers and TMEM exist before either uses the other's
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------- TMA producer (operands and factor tiles) ----------------
    if (elect_one_sync()) {
      uint32_t it = 0;
      bool ok = true;
      const uint32_t bar0 = PAIR ? mapa_shared(&full[0], 0) : smem_u32(&full[0]);
      for (int u = first; u < total && ok; u += stride) {
        const int tm = (u % m_units) * G + rank, tn = u / m_units;
        const int b_row = tn * BN + rank * CF::kBRows;
        for (int kc = 0; kc < kstages; ++kc, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, FGQ_DEVERR_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[s], CF::kTxBytes);
          uint8_t* sf = sm_sf + s * CF::kSfBytes;
          // first factor tile of this stage within a row tile
          const int t0 = FP8 ? kc >> 2 : kc * kCells;
          if constexpr (PAIR) {
            const uint32_t bar = bar0 + s * 8;
            tma_load_2d_pair(sm_a + s * CF::kABytes, &tmap_a, bar, kc * BK, tm * BM);
            tma_load_2d_pair(sm_b + s * CF::kBBytes, &tmap_b, bar, kc * BK, b_row);
            tma_load_2d_pair(sf, &tmap_sa, bar, 0, tm * cpr + t0);
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tma_load_2d_pair(sf + CF::kSfABytes + h * kCells * 512, &tmap_sb, bar, 0,
                               (tn * (BN / 128) + h) * cpr + t0);
          } else {
            tma_load_2d(sm_a + s * CF::kABytes, &tmap_a, &full[s], kc * BK, tm * BM);
            tma_load_2d(sm_b + s * CF::kBBytes, &tmap_b, &full[s], kc * BK, b_row);
            tma_load_2d(sf, &tmap_sa, &full[s], 0, tm * cpr + t0);
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tma_load_2d(sf + CF::kSfABytes + h * kCells * 512, &tmap_sb, &full[s], 0,
                          (tn * (BN / 128) + h) * cpr + t0);
          }
        }
      }
      // Before leaving: every copy into this CTA's (the pair's) shared memory
      // has landed, and for a pair every commit addressed to this CTA's empty
      // barriers has arrived.
      const uint32_t lo = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u;
      for (uint32_t j = lo; j < it; ++j) {
        if (leader) mxf4_wait_drain(&full[j % STAGES], (j / STAGES) & 1u);
        if (PAIR) mxf4_wait_drain(&empty[j % STAGES], (j / STAGES) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1 && leader) {
    // ---------------- MMA issuer (the leader of a pair) ----------------
    if (elect_one_sync()) {
      constexpr uint32_t idesc0 = FP8 ? idesc_mx_e4m3_ue8m0(G * BM, BN) : idesc_fp4(G * BM, BN, NV);
      constexpr uint32_t kId2 = (2u << 29) | (2u << 4);  // factor bytes 2-3 of A and B
      const uint64_t dA0 = smem_desc_k_sw128(smem_u32(sm_a));
      const uint32_t a_lo0 = static_cast<uint32_t>(dA0), dhi = static_cast<uint32_t>(dA0 >> 32);
      const uint32_t b_lo0 = static_cast<uint32_t>(smem_desc_k_sw128(smem_u32(sm_b)));
      const uint32_t sf0 = smem_u32(sm_sf);
      int ls = 0;
      uint32_t lph = 0, g_it = 0, t_it = 0;
      bool ok = true;
      for (int u = first; u < total && ok; u += stride, ++t_it) {
        const uint32_t buf = t_it % NACC, aph = (t_it / NACC) & 1u;
        if (!mbar_wait(&acc_empty[buf], aph ^ 1u, abort_flag, FGQ_DEVERR_MMA_TMEM)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * BN;
        for (int kc = 0; kc < kstages; ++kc, ++g_it) {
          if (!mbar_wait(&full[ls], lph, abort_flag, FGQ_DEVERR_MMA_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t r = g_it % kSlots;
          const uint32_t sfa = tmem_base + F::kSfaCol0 + F::kSfaSlot * r;
          const uint32_t sfb = tmem_base + F::kSfbCol0 + F::kSfbSlot * r;
          // the stage's factor tiles into slot r: A tile w to columns 4 w ..
          // 4 w + 3, B tile w of columns 128 h .. 128 h + 127 to 8 w + 4 h ..
          // + 3 (in order before the MMAs that read them)
          const uint32_t sfs = sf0 + ls * CF::kSfBytes;
#pragma unroll
          for (int w = 0; w < kCells; ++w) {
            const uint64_t da = sf_tile_desc(sfs + w * 512);
            if constexpr (PAIR)
              tmem_cp_32x128b_x4_pair(sfa + 4 * w, da);
            else
              tmem_cp_32x128b_x4(sfa + 4 * w, da);
#pragma unroll
            for (int h = 0; h < BN / 128; ++h) {
              const uint64_t db = sf_tile_desc(sfs + CF::kSfABytes + (h * kCells + w) * 512);
              if constexpr (PAIR)
                tmem_cp_32x128b_x4_pair(sfb + 8 * w + 4 * h, db);
              else
                tmem_cp_32x128b_x4(sfb + 8 * w + 4 * h, db);
            }
          }
          const uint32_t a_lo = a_lo0 + ls * (CF::kABytes >> 4);
          const uint32_t b_lo = b_lo0 + ls * (CF::kBBytes >> 4);
          // four K = 64 MMAs (32 bytes of each row apart); a final half stage
          // has two.  MXFP4: factor bytes 0-1 and 2-3 of tile 0, then of
          // tile 1.  NVFP4: tile kk for MMA kk.
          const bool full_stage = kc + 1 < kstages || !half_last;
          if constexpr (FP8) {
            // four K = 32 MMAs, all reading byte kc % 4 of the slot's cells
            const uint32_t id = static_cast<uint32_t>(kc) & 3u;
            const uint32_t idesc = idesc0 | (id << 29) | (id << 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              fp4_mma<PAIR, KIND>(d, make_desc(a_lo + 2 * kk, dhi), make_desc(b_lo + 2 * kk, dhi),
                                  idesc, sfa, sfb, (kc > 0 || kk > 0) ? 1u : 0u);
          } else if constexpr (NV) {
            fp4_mma<PAIR, KIND>(d, make_desc(a_lo, dhi), make_desc(b_lo, dhi), idesc0, sfa, sfb,
                              kc > 0 ? 1u : 0u);
            fp4_mma<PAIR, KIND>(d, make_desc(a_lo + 2, dhi), make_desc(b_lo + 2, dhi), idesc0,
                              sfa + 4, sfb + 8, 1u);
            if (full_stage) {
              fp4_mma<PAIR, KIND>(d, make_desc(a_lo + 4, dhi), make_desc(b_lo + 4, dhi), idesc0,
                                sfa + 8, sfb + 16, 1u);
              fp4_mma<PAIR, KIND>(d, make_desc(a_lo + 6, dhi), make_desc(b_lo + 6, dhi), idesc0,
                                sfa + 12, sfb + 24, 1u);
            }
          } else {
            fp4_mma<PAIR, KIND>(d, make_desc(a_lo, dhi), make_desc(b_lo, dhi), idesc0, sfa, sfb,
                              kc > 0 ? 1u : 0u);
            fp4_mma<PAIR, KIND>(d, make_desc(a_lo + 2, dhi), make_desc(b_lo + 2, dhi),
                              idesc0 | kId2, sfa, sfb, 1u);
            if (full_stage) {
              fp4_mma<PAIR, KIND>(d, make_desc(a_lo + 4, dhi), make_desc(b_lo + 4, dhi), idesc0,
                                sfa + 4, sfb + 8, 1u);
              fp4_mma<PAIR, KIND>(d, make_desc(a_lo + 6, dhi), make_desc(b_lo + 6, dhi),
                                idesc0 | kId2, sfa + 4, sfb + 8, 1u);
            }
          }
          if constexpr (PAIR)
            umma_commit_pair(&empty[ls], kMask);
          else
            umma_commit(&empty[ls]);
          if (++ls == STAGES) {
            ls = 0;
            lph ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          umma_commit_pair(&acc_full[buf], kMask);
        else
          umma_commit(&acc_full[buf]);
      }
      // Every MMA this thread issued must finish before TMEM is released.
      if constexpr (PAIR)
        umma_commit_pair(drain, 0x1);
      else
        umma_commit(drain);
      mxf4_wait_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 8) {
    // ---------------- epilogue (each CTA its own 128 rows) ----------------
    const int ew = warp - 8;
    const int q = warp & 3;
    const int half = ew >> 2;
    const uint32_t t_lane = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t acc_empty0 = PAIR ? mapa_shared(&acc_empty[0], 0) : 0u;
    float alpha = 1.0f;
    if constexpr (NV) alpha = __fmul_rn(__ldg(ga), __ldg(gb));
    auto scale32 = [&](uint32_t (&r)[32]) {
      if constexpr (NV) {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[i]), alpha));
      }
    };
    uint32_t t_it = 0;
    uint8_t* stage = sm_st + ew * 1024;
    for (int u = first; u < total; u += stride, ++t_it) {
      const int tm = (u % m_units) * G + rank, tn = u / m_units;
      const int row0 = tm * BM + 32 * q;
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
          if (lane == 0) {
            if (PAIR && !leader)
              mbar_arrive_cluster_relaxed(acc_empty0 + buf * 8);
            else
              mbar_arrive_relaxed(&acc_empty[buf]);
          }
        }
        if (j % 2 == 0) {
          scale32(ra);
          warp_store32<OUT_BF16, 1024>(stage, ra, C, ldc, row0, col0 + 32 * j, M - row0);
        } else {
          scale32(rb);
          warp_store32<OUT_BF16, 1024>(stage, rb, C, ldc, row0, col0 + 32 * j, M - row0);
        }
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
  if constexpr (PAIR) {
    cluster_sync();  // neither CTA leaves while its peer may still reach its memory
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem_base, kTmemCols);
    }
  } else {
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem_base, kTmemCols);
    }
  }
}

template <int BN, int STAGES, bool OUT_BF16, bool NV>
cudaError_t launch_mxf4_cfg(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                          const float* ga, const float* gb, void* C, int64_t ldc, int M, int N,
                          int K, cudaStream_t stream, const DeviceInfo& dev) {
  using CF = Mxf4Cfg<BN, STAGES, NV>;
  auto kern = gemm_mxf4_kernel<BN, STAGES, OUT_BF16, NV>;
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
  // rows of K/2 bytes (two E2M1 per byte)
  if (!make_k_major_map(&ta, A, M, K / 2, BM) || !make_k_major_map(&tb, B, N, K / 2, BN))
    return cudaErrorInvalidValue;
  const int tiles = ((M + BM - 1) / BM) * (N / BN);
  const int grid = tiles < dev.sm_count ? tiles : dev.sm_count;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), CF::kSmemBytes, stream, ta, tb, sA, sB, ga,
                    gb, C, ldc, M, N, K);
}

// Tiled-scale kernel set-up, once per device and configuration: the shared
// memory attribute, and for pairs the clusters of two that fit at once (0
// when the pair kernel cannot run).
template <bool PAIR, int BN, bool OUT_BF16, int KIND>
cudaError_t tiled_setup(const DeviceInfo& dev, int* clusters) {
  using CF = TiledCfg<PAIR, BN, KIND>;
  auto kern = gemm_fp4_tiled_kernel<PAIR, BN, OUT_BF16, KIND>;
  static std::mutex mu;
  static int cached[64] = {};
  static bool ready[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev.device]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(CF::kSmemBytes));
    if (e != cudaSuccess) return e;
    int n = 1;
    if (PAIR) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * (dev.sm_count / 2));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = CF::kSmemBytes;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return e;
    }
    cached[dev.device] = n;
    ready[dev.device] = true;
  }
  *clusters = cached[dev.device];
  return cudaSuccess;
}

template <bool PAIR, int BN, bool OUT_BF16, int KIND>
cudaError_t launch_tiled_cfg(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                             const uint8_t* sB, const float* ga, const float* gb, void* C,
                             int64_t ldc, int M, int N, int K, int clusters, cudaStream_t stream,
                             const DeviceInfo& dev) {
  using CF = TiledCfg<PAIR, BN, KIND>;
  constexpr int G = PAIR ? 2 : 1;
  constexpr bool FP8 = KIND == kMx8;
  CUtensorMap ta, tb, tsa, tsb;
  // operand rows of K/2 bytes (two E2M1 per byte); factor tiles: one per
  // 128 rows and 4 factor bytes, K/128 (MXFP4) or K/64 (NVFP4) per row tile
  const int64_t cpr = FP8 ? (K / 128 + 3) / 4 : K / (KIND == kNv4 ? 64 : 128);
  const int64_t a_tiles = (M + BM - 1) / BM * cpr, b_tiles = N / 128 * cpr;
  const int64_t row_bytes = FP8 ? K : K / 2;
  if (!make_k_major_map(&ta, A, M, row_bytes, BM) ||
      !make_k_major_map(&tb, B, N, row_bytes, CF::kBRows) ||
      !make_scale_tile_map(&tsa, sA, a_tiles, Fp4TiledFmt<KIND>::kCells) ||
      !make_scale_tile_map(&tsb, sB, b_tiles, Fp4TiledFmt<KIND>::kCells))
    return cudaErrorInvalidValue;
  const int units = ((M + BM - 1) / BM + G - 1) / G * (N / BN);
  const int cap = PAIR ? clusters : dev.sm_count;
  const int grid = G * (units < cap ? units : cap);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na++].val.programmaticStreamSerializationAllowed = 1;
  if (PAIR) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na++].val.clusterDim.z = 1;
  }
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = CF::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_fp4_tiled_kernel<PAIR, BN, OUT_BF16, KIND>, ta, tb, tsa, tsb,
                            ga, gb, C, ldc, M, N, K);
}

// Configuration choice for tiled scales: CTA pairs once A has two row tiles,
// on 256-column tiles when there is at least one per cluster, else
// 128-column ones; a single CTA per 128 x 128 tile for one row tile.
template <bool OUT_BF16, int KIND>
cudaError_t launch_fp4_tiled(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                             const uint8_t* sB, const float* ga, const float* gb, void* C,
                             int64_t ldc, int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                             const DeviceInfo& dev) {
  if (M == 0 || N == 0) return cudaSuccess;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  const int64_t m_tiles = (M + BM - 1) / BM;
  if (m_tiles >= 2) {
    int c256 = 0, c128 = 0;
    cudaError_t e = tiled_setup<true, 256, OUT_BF16, KIND>(dev, &c256);
    if (e != cudaSuccess) return e;
    e = tiled_setup<true, 128, OUT_BF16, KIND>(dev, &c128);
    if (e != cudaSuccess) return e;
    const int64_t groups = (m_tiles + 1) / 2;
    if (N % 256 == 0 && c256 > 0 && groups * (N / 256) >= c256)
      return launch_tiled_cfg<true, 256, OUT_BF16, KIND>(A, sA, B, sB, ga, gb, C, ldc, m, n, k, c256,
                                                       stream, dev);
    if (c128 > 0)
      return launch_tiled_cfg<true, 128, OUT_BF16, KIND>(A, sA, B, sB, ga, gb, C, ldc, m, n, k, c128,
                                                       stream, dev);
  }
  int one = 0;
  const cudaError_t e = tiled_setup<false, 128, OUT_BF16, KIND>(dev, &one);
  if (e != cudaSuccess) return e;
  return launch_tiled_cfg<false, 128, OUT_BF16, KIND>(A, sA, B, sB, ga, gb, C, ldc, m, n, k, 0, stream,
                                                    dev);
}

template <bool NV>
cudaError_t launch_fp4(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                       const float* ga, const float* gb, void* C, int64_t ldc, int64_t M,
                       int64_t N, int64_t K, int out_bf16, cudaStream_t stream,
                       const DeviceInfo& dev) {
  if (M == 0 || N == 0) return cudaSuccess;
  // 128-column tiles: six operand stages, or fewer as the factor ring needs
  constexpr int kNarrow = Fp4Fmt<NV>::kSlots - Fp4Fmt<NV>::kChunkStages + 1 < 6
                              ? Fp4Fmt<NV>::kSlots - Fp4Fmt<NV>::kChunkStages + 1
                              : 6;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  const int64_t tiles256 = ((M + BM - 1) / BM) * (N / 256);
  const bool wide = (N % 256 == 0) && tiles256 >= dev.sm_count;
  if (out_bf16) {
    return wide ? launch_mxf4_cfg<256, 4, true, NV>(A, sA, B, sB, ga, gb, C, ldc, m, n, k, stream, dev)
                : launch_mxf4_cfg<128, kNarrow, true, NV>(A, sA, B, sB, ga, gb, C, ldc, m, n, k, stream, dev);
  }
  return wide ? launch_mxf4_cfg<256, 4, false, NV>(A, sA, B, sB, ga, gb, C, ldc, m, n, k, stream, dev)
              : launch_mxf4_cfg<128, kNarrow, false, NV>(A, sA, B, sB, ga, gb, C, ldc, m, n, k, stream, dev);
}

}  // namespace

cudaError_t launch_gemm_mxf4(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                             const uint8_t* sB, void* C, int64_t ldc, int64_t M, int64_t N,
                             int64_t K, int out_bf16, cudaStream_t stream, const DeviceInfo& dev) {
  return launch_fp4<false>(A, sA, B, sB, nullptr, nullptr, C, ldc, M, N, K, out_bf16, stream, dev);
}

cudaError_t launch_gemm_nvf4(const uint8_t* A, const uint8_t* sA, const float* ga,
                             const uint8_t* B, const uint8_t* sB, const float* gb, void* C,
                             int64_t ldc, int64_t M, int64_t N, int64_t K, int out_bf16,
                             cudaStream_t stream, const DeviceInfo& dev) {
  return launch_fp4<true>(A, sA, B, sB, ga, gb, C, ldc, M, N, K, out_bf16, stream, dev);
}

cudaError_t launch_gemm_mxf4_tiled(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                                   const uint8_t* sB, void* C, int64_t ldc, int64_t M, int64_t N,
                                   int64_t K, int out_bf16, cudaStream_t stream,
                                   const DeviceInfo& dev) {
  return out_bf16 ? launch_fp4_tiled<true, kMx4>(A, sA, B, sB, nullptr, nullptr, C, ldc, M, N, K,
                                                 stream, dev)
                  : launch_fp4_tiled<false, kMx4>(A, sA, B, sB, nullptr, nullptr, C, ldc, M, N, K,
                                                  stream, dev);
}

cudaError_t launch_gemm_nvf4_tiled(const uint8_t* A, const uint8_t* sA, const float* ga,
                                   const uint8_t* B, const uint8_t* sB, const float* gb, void* C,
                                   int64_t ldc, int64_t M, int64_t N, int64_t K, int out_bf16,
                                   cudaStream_t stream, const DeviceInfo& dev) {
  return out_bf16 ? launch_fp4_tiled<true, kNv4>(A, sA, B, sB, ga, gb, C, ldc, M, N, K, stream, dev)
                  : launch_fp4_tiled<false, kNv4>(A, sA, B, sB, ga, gb, C, ldc, M, N, K, stream, dev);
}

cudaError_t launch_gemm_mx8_tiled(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                                  const uint8_t* sB, void* C, int64_t ldc, int64_t M, int64_t N,
                                  int64_t K, int out_bf16, cudaStream_t stream,
                                  const DeviceInfo& dev) {
  return out_bf16 ? launch_fp4_tiled<true, kMx8>(A, sA, B, sB, nullptr, nullptr, C, ldc, M, N, K,
                                                 stream, dev)
                  : launch_fp4_tiled<false, kMx8>(A, sA, B, sB, nullptr, nullptr, C, ldc, M, N, K,
                                                  stream, dev);
}

cudaError_t read_device_error_mxf4(uint32_t* word, bool clear) {
  return read_unit_device_error(word, clear);
}

}  // namespace fgq
