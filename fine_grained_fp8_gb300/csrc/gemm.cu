// Block-scaled FP8 GEMM for sm_103a ("Fine-Grained FP8/FP4 Quantization",
// §DeepGEMM: Tile-wise and Block-wise Scaling):
//
//   C[m,n] = sum_c sA[m,c] * sB[c, n/128] * P_c[m,n],
//   P_c    = sum_{k in chunk c} Aq[m,k] * Bq[k,n]   (one 128-wide K chunk)
//
// Design (GB300-native; the page's Hopper promotion loop is prior art):
//   - Persistent CTAs, one per SM, walking output tiles of 128 x BN with a
//     static stride-gridDim schedule ("Persistent kernel (grid = SM count,
//     internal tile loop)", linear scheduler, M fastest).
//   - Warp 0: TMA producer.  Each stage holds one 128-wide K chunk of A
//     (128 x 128 bytes) and B (BN x 128 bytes), 128-byte swizzled.
//   - Warp 1: one thread issues 4 tcgen05.mma (K = 32 each) per chunk into
//     one of 512 / BN TMEM partial buffers (128 lanes x BN fp32 columns
//     each: two for BN = 256, four for BN = 128),
//     then commits to the stage's "empty" and the buffer's "full" barriers.
//   - Warps 4-11: epilogue.  Per chunk they read the partial from TMEM in
//     32-column loads (the next load in flight while the current one is
//     used), multiply by sA[m,c] * sB[c, n/128] and add it into fp32
//     accumulators held in registers with packed f32x2 FMAs (the promotion
//     step), hand the TMEM buffer back as soon as it is read, and after the
//     last chunk convert and store the tile.  The buffers let the tensor
//     core run chunks ahead while chunk c is promoted.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "fgq_device.cuh"
#include "fgq_internal.h"

namespace fgq {
namespace {

constexpr int BM = 128;
constexpr int BK = 128;  // one scale chunk per pipeline stage
// Warpgroup 0: warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM owner),
// warps 2-3 idle.  Warpgroups 1-2: eight epilogue warps, two per TMEM lane
// quadrant.  Registers are moved from warpgroup 0 to the epilogue with
// setmaxnreg: the launch gives every thread kLaunchRegs, warpgroup 0 drops
// to kCtlRegs and the epilogue rises to kEpiRegs.
constexpr int kCtlWarps = 4;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (kCtlWarps + kEpiWarps);
constexpr int kLaunchRegs = 168;  // 65536 / 384, rounded down to a multiple of 8
constexpr uint32_t kCtlRegs = 56;
constexpr uint32_t kEpiRegs = 224;
static_assert(128 * kCtlRegs + 256 * kEpiRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");

template <int BN, int STAGES>
struct Cfg {
  static constexpr int kABytes = BM * BK;
  static constexpr int kBBytes = BN * BK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kNBuf = 512 / BN;    // partial buffers: all 512 TMEM columns
  static constexpr int kTmemCols = kNBuf * BN;
  static constexpr int kBarBytes = (2 * STAGES + 2 * kNBuf) * 8 + 16;
  static constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(STAGES) * kStageBytes + kBarBytes;
  static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation must be a power of 2");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// Bounded wait used while unwinding; ignores the abort flag.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > FGQ_WAIT_NS) {
      record_error(FGQ_DEVERR_DRAIN);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// acc[j] += comb * partial[j] for the 32 columns held in r (16 packed pairs).
// (Called from fully unrolled loops, so j0 is a constant and acc stays in
// registers.)
template <int NACC>
__device__ __forceinline__ void promote32(uint64_t (&acc)[NACC], const uint32_t (&r)[32],
                                          uint64_t comb2, int j0) {
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j0 + j] = ffma2_acc(pack2(r[2 * j], r[2 * j + 1]), comb2, acc[j0 + j]);
}

template <int BN, int STAGES, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_blockscaled_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                const __grid_constant__ CUtensorMap tmap_b,
                                const float* __restrict__ sA, const float* __restrict__ sB,
                                void* __restrict__ C, int64_t ldc, int M, int N, int K,
                                int wide_stores) {
  using CF = Cfg<BN, STAGES>;
  constexpr uint32_t NBUF = CF::kNBuf;
  constexpr int HALF = BN / 2;     // columns per epilogue warp
  constexpr int NLD = HALF / 32;   // 32-column TMEM loads per chunk
  static_assert(NLD >= 2, "the load pipeline below assumes at least two loads per chunk");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sm_a = smem;
  uint8_t* sm_b = smem + STAGES * CF::kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm_b + STAGES * CF::kBBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + NBUF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + NBUF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (M + BM - 1) / BM;
  const int n_tiles = (N + BN - 1) / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int kchunks = K / BK;
  const int nb = N / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, CF::kTmemCols);
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

  if (warp < kCtlWarps) {
    setmaxnreg_dec<kCtlRegs>();
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
        for (uint32_t j = first; j < it; ++j) mbar_wait_drain(&full[j % STAGES], (j / STAGES) & 1u);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      if (elect_one_sync()) {
        constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
        // Lean issue loop (this thread shares its scheduler with two
        // FMA-heavy epilogue warps): the descriptor of an operand tile at
        // offset d from the stage base is the base descriptor with d >> 4
        // added to its low word (shared memory is below 256 KB, so the start
        // field never carries), and the stage index and phase advance
        // incrementally.
        const uint64_t dA0 = smem_desc_k_sw128(smem_u32(sm_a));
        const uint32_t a_lo0 = static_cast<uint32_t>(dA0), dhi = static_cast<uint32_t>(dA0 >> 32);
        const uint32_t b_lo0 = static_cast<uint32_t>(smem_desc_k_sw128(smem_u32(sm_b)));
        int ls = 0;
        uint32_t lph = 0;
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
          for (int kc = 0; kc < kchunks; ++kc, ++it) {
            const uint32_t buf = it % NBUF, tph = (it / NBUF) & 1u;
            if (!mbar_wait(&tempty[buf], tph ^ 1u, abort_flag, FGQ_DEVERR_MMA_TMEM) ||
                !mbar_wait(&full[ls], lph, abort_flag, FGQ_DEVERR_MMA_FULL)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem_base + buf * BN;
            const uint32_t a_lo = a_lo0 + ls * (CF::kABytes >> 4);
            const uint32_t b_lo = b_lo0 + ls * (CF::kBBytes >> 4);
#pragma unroll
            for (int kk = 0; kk < BK / 32; ++kk) {
              uint64_t da, db;
              asm("mov.b64 %0, {%1, %2};" : "=l"(da) : "r"(a_lo + kk * 2), "r"(dhi));
              asm("mov.b64 %0, {%1, %2};" : "=l"(db) : "r"(b_lo + kk * 2), "r"(dhi));
              umma_f8f6f4(d, da, db, idesc, kk > 0 ? 1u : 0u);
            }
            umma_commit(&empty[ls]);
            umma_commit(&tfull[buf]);
            if (++ls == STAGES) {
              ls = 0;
              lph ^= 1u;
            }
          }
        }
        // MMAs still in flight must finish before TMEM is released.
        if (it > 0) mbar_wait_drain(&tfull[(it - 1) % NBUF], ((it - 1) / NBUF) & 1u);
      }
      __syncwarp();
    }
  } else {
    // ---------------- epilogue: promotion + store ----------------
    setmaxnreg_inc<kEpiRegs>();
    const int ew = warp - kCtlWarps;
    const int quad = warp & 3;   // TMEM lanes this warp may access
    const int half = ew >> 2;    // which half of the tile's columns
    const int r_in_tile = quad * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      const int tm = tile % m_tiles, tn = tile / m_tiles;
      const int row = tm * BM + r_in_tile;
      const bool row_ok = row < M;
      const int col0 = tn * BN + half * HALF;
      const bool cols_ok = col0 < N;
      const int nblk = cols_ok ? col0 / 128 : nb - 1;
      const float* sa_row = sA + static_cast<int64_t>(row_ok ? row : 0) * kchunks;
      const float* sb_col = sB + nblk;

      uint64_t acc[HALF / 2];
#pragma unroll
      for (int j = 0; j < HALF / 2; ++j) acc[j] = 0ull;

      float sa_next = row_ok ? __ldg(sa_row) : 0.0f;
      float sb_next = __ldg(sb_col);
      for (int kc = 0; kc < kchunks; ++kc, ++it) {
        const uint32_t buf = it % NBUF, tph = (it / NBUF) & 1u;
        const float comb = sa_next * sb_next;
        if (kc + 1 < kchunks) {  // prefetch the next chunk's scales
          sa_next = row_ok ? __ldg(sa_row + kc + 1) : 0.0f;
          sb_next = __ldg(sb_col + static_cast<int64_t>(kc + 1) * nb);
        }
        const uint64_t comb2 = pack2(__float_as_uint(comb), __float_as_uint(comb));
        // warp-uniform outcome: the TMEM loads below are warp-collective
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tfull[buf], tph, abort_flag, FGQ_DEVERR_EPI_TMEM))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + t_lane + buf * BN + half * HALF;
        uint32_t ra[32], rb[32];
        tmem_ld_32x32b_x32(taddr, ra);
        tmem_wait_ld_regs(ra);
#pragma unroll
        for (int q = 0; q < NLD; ++q) {
          if (q + 1 < NLD) {
            if (q % 2 == 0)
              tmem_ld_32x32b_x32(taddr + 32 * (q + 1), rb);
            else
              tmem_ld_32x32b_x32(taddr + 32 * (q + 1), ra);
          } else {
            // every column of this buffer is in registers: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
          }
          if (q % 2 == 0)
            promote32(acc, ra, comb2, 16 * q);
          else
            promote32(acc, rb, comb2, 16 * q);
          if (q + 1 < NLD) {
            if (q % 2 == 0)
              tmem_wait_ld_regs(rb);
            else
              tmem_wait_ld_regs(ra);
          }
        }
      }
      if (!ok) break;
      // Store with 32-byte stores, one whole sector of the row per lane and
      // instruction.  (With 16-byte stores the C store took about 23 us of
      // the large-prefill GEMM: the next tile's MMAs waited for the TMEM
      // buffers while the epilogue stored.  Staging the rows through shared
      // memory for fully coalesced stores measured no better here: the
      // staging buffer takes 16 KB of the L1 the scale loads use.)
      // wide_stores: C and its row pitch are 32-byte aligned (the host
      // checks); otherwise 16-byte stores.
      if (row_ok && cols_ok && !wide_stores) {
        if (OUT_BF16) {
          uint16_t* crow = static_cast<uint16_t*>(C) + static_cast<int64_t>(row) * ldc + col0;
#pragma unroll
          for (int j = 0; j < HALF / 2; j += 4) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(acc[j])),
                              __uint_as_float(static_cast<uint32_t>(acc[j] >> 32)));
            v.y = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(acc[j + 1])),
                              __uint_as_float(static_cast<uint32_t>(acc[j + 1] >> 32)));
            v.z = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(acc[j + 2])),
                              __uint_as_float(static_cast<uint32_t>(acc[j + 2] >> 32)));
            v.w = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(acc[j + 3])),
                              __uint_as_float(static_cast<uint32_t>(acc[j + 3] >> 32)));
            *reinterpret_cast<uint4*>(crow + 2 * j) = v;
          }
        } else {
          float* crow = static_cast<float*>(C) + static_cast<int64_t>(row) * ldc + col0;
#pragma unroll
          for (int j = 0; j < HALF / 2; j += 2) {
            uint4 v = make_uint4(static_cast<uint32_t>(acc[j]), static_cast<uint32_t>(acc[j] >> 32),
                                 static_cast<uint32_t>(acc[j + 1]),
                                 static_cast<uint32_t>(acc[j + 1] >> 32));
            *reinterpret_cast<uint4*>(crow + 2 * j) = v;
          }
        }
      } else if (row_ok && cols_ok) {
        if (OUT_BF16) {
          uint16_t* crow = static_cast<uint16_t*>(C) + static_cast<int64_t>(row) * ldc + col0;
#pragma unroll
          for (int j = 0; j < HALF / 2; j += 8) {
            uint32_t w[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
              w[q] = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(acc[j + q])),
                                 __uint_as_float(static_cast<uint32_t>(acc[j + q] >> 32)));
            st_global_32B(crow + 2 * j, w);
          }
        } else {
          float* crow = static_cast<float*>(C) + static_cast<int64_t>(row) * ldc + col0;
#pragma unroll
          for (int j = 0; j < HALF / 2; j += 4) {
            const uint32_t w[8] = {
                static_cast<uint32_t>(acc[j]),         static_cast<uint32_t>(acc[j] >> 32),
                static_cast<uint32_t>(acc[j + 1]),     static_cast<uint32_t>(acc[j + 1] >> 32),
                static_cast<uint32_t>(acc[j + 2]),     static_cast<uint32_t>(acc[j + 2] >> 32),
                static_cast<uint32_t>(acc[j + 3]),     static_cast<uint32_t>(acc[j + 3] >> 32)};
            st_global_32B(crow + 2 * j, w);
          }
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, CF::kTmemCols);
  }
}

// ---- CTA pairs: 256 x 128 tiles, four partial buffers ------------------------------
//
// The single-CTA kernel above takes 48 KB of operands into shared memory per
// K chunk of a 128 x 256 tile, which is what bounds its tensor core (about
// 15 TB/s of L2-to-SM traffic over the GPU), and its epilogue has only two
// partial buffers of 256 columns.  Here two CTAs of a cluster share one
// tcgen05.mma.cta_group::2 of M = 256, N = 128: each CTA holds its own 128
// rows of A and half of B's 128 rows (24 KB per chunk, the same bytes per
// multiply-add as the 128 x 256 tile) and receives its 128 rows of the
// partial in its own TMEM.  A 128-column partial leaves room for four
// buffers, so the tensor core can run three chunks ahead of the promotion,
// and each epilogue warp reads its 64 columns of a chunk with both loads in
// flight and one wait.
//   - The even CTA (leader) issues the MMAs.  Both CTAs' TMA copies of a
//     stage complete on the leader's `full` barrier; the leader's commits
//     arrive on the `empty` and `tfull` barriers of both CTAs (multicast).
//   - Both CTAs' epilogues hand a drained buffer back on the leader's
//     `tempty` barrier (the peer with a cluster-scope release arrive).
constexpr int kPairBN = 128;   // output columns of a pair tile (the MMA's N)
constexpr int kPairStages = 8;
constexpr int kPairBufs = 4;   // TMEM partial buffers of kPairBN columns
constexpr uint16_t kPairMask = 0x3;
// Measured slower than the single-CTA kernel on the shapes tried (large
// prefill 204 against 155-162 us; skinny M = 256 27.5 against 21.7 us), so
// launch_gemm_fp8_blockscaled does not route to it.
constexpr bool kUsePairs = false;
// A 64-column accumulator needs fewer epilogue registers than the 128 of the
// single-CTA kernel; the control warps get the rest.
constexpr uint32_t kPairCtlRegs = 104;
constexpr uint32_t kPairEpiRegs = 200;
static_assert(128 * kPairCtlRegs + 256 * kPairEpiRegs <= kThreads * kLaunchRegs, "register split");

struct PairCfg {
  static constexpr int kABytes = BM * BK;                // this CTA's 128 rows of A
  static constexpr int kBBytes = (kPairBN / 2) * BK;     // this CTA's 64 rows of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTxBytes = 2 * kStageBytes;  // both CTAs' copies of a stage
  static constexpr int kTmemCols = kPairBufs * kPairBN;
  static constexpr int kBarBytes = (2 * kPairStages + 2 * kPairBufs) * 8 + 16;
  static constexpr size_t kSmemBytes =
      1024 + static_cast<size_t>(kPairStages) * kStageBytes + kBarBytes;
  static_assert(kTmemCols == 512, "TMEM allocation");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

template <bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b,
                         const float* __restrict__ sA, const float* __restrict__ sB,
                         void* __restrict__ C, int64_t ldc, int M, int N, int K) {
  using CF = PairCfg;
  constexpr int STAGES = kPairStages;
  constexpr int HALF = kPairBN / 2;  // columns per epilogue warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sm_a = smem;
  uint8_t* sm_b = smem + STAGES * CF::kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm_b + STAGES * CF::kBBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + kPairBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + kPairBufs);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  // Pair tiles (two stacked 128-row tiles x 128 columns), M fastest; the
  // cluster c takes tiles c, c + clusters, ...
  const int m_tiles = (M + BM - 1) / BM;
  const int m_groups = (m_tiles + 1) / 2;
  const int n_tiles = N / kPairBN;
  const int total = m_groups * n_tiles;
  const int first = static_cast<int>(blockIdx.x) / 2;
  const int stride = static_cast<int>(gridDim.x) / 2;
  const int kchunks = K / BK;
  const int nb = N / 128;

  if (threadIdx.x == 0) {
    // The leader's full and tempty barriers gather both CTAs; every CTA
    // receives the leader's commits on its own empty and tfull barriers.
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kPairBufs; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, CF::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers and TMEM exist before either uses the other's
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();

  if (warp < kCtlWarps) {
    setmaxnreg_dec<kPairCtlRegs>();
    if (warp == 0) {
      // ---------------- TMA producer (each CTA loads its own share) ----------------
      if (elect_one_sync()) {
        uint32_t it = 0;
        bool ok = true;
        const uint32_t bar0 = mapa_shared(&full[0], 0);
        for (int u = first; u < total && ok; u += stride) {
          const int tm = (u % m_groups) * 2 + rank, tn = u / m_groups;
          const int b_row = tn * kPairBN + rank * (kPairBN / 2);
          for (int kc = 0; kc < kchunks; ++kc, ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1u;
            if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, FGQ_DEVERR_PRODUCER_EMPTY)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(&full[s], CF::kTxBytes);
            const uint32_t bar = bar0 + s * 8;
            tma_load_2d_pair(sm_a + s * CF::kABytes, &tmap_a, bar, kc * BK, tm * BM);
            tma_load_2d_pair(sm_b + s * CF::kBBytes, &tmap_b, bar, kc * BK, b_row);
          }
        }
        // Before leaving: every copy into the pair's shared memory has landed
        // (the leader's full barriers see both CTAs' copies) and every MMA
        // commit addressed to this CTA's empty barriers has arrived.
        const uint32_t lo = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u;
        for (uint32_t j = lo; j < it; ++j) {
          if (leader) mbar_wait_drain(&full[j % STAGES], (j / STAGES) & 1u);
          mbar_wait_drain(&empty[j % STAGES], (j / STAGES) & 1u);
        }
      }
      __syncwarp();
    } else if (warp == 1 && leader) {
      // ---------------- MMA issuer (the leader) ----------------
      if (elect_one_sync()) {
        constexpr uint32_t idesc = idesc_e4m3_f32(2 * BM, kPairBN);
        const uint64_t dA0 = smem_desc_k_sw128(smem_u32(sm_a));
        const uint32_t a_lo0 = static_cast<uint32_t>(dA0), dhi = static_cast<uint32_t>(dA0 >> 32);
        const uint32_t b_lo0 = static_cast<uint32_t>(smem_desc_k_sw128(smem_u32(sm_b)));
        int ls = 0;
        uint32_t lph = 0;
        uint32_t it = 0;
        bool ok = true;
        for (int u = first; u < total && ok; u += stride) {
          for (int kc = 0; kc < kchunks; ++kc, ++it) {
            const uint32_t buf = it % kPairBufs, tph = (it / kPairBufs) & 1u;
            if (!mbar_wait(&tempty[buf], tph ^ 1u, abort_flag, FGQ_DEVERR_MMA_TMEM) ||
                !mbar_wait(&full[ls], lph, abort_flag, FGQ_DEVERR_MMA_FULL)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem_base + buf * kPairBN;
            const uint32_t a_lo = a_lo0 + ls * (CF::kABytes >> 4);
            const uint32_t b_lo = b_lo0 + ls * (CF::kBBytes >> 4);
#pragma unroll
            for (int kk = 0; kk < BK / 32; ++kk)
              umma_f8f6f4_pair(d, make_desc(a_lo + kk * 2, dhi), make_desc(b_lo + kk * 2, dhi),
                               idesc, kk > 0 ? 1u : 0u);
            umma_commit_pair(&empty[ls], kPairMask);
            umma_commit_pair(&tfull[buf], kPairMask);
            if (++ls == STAGES) {
              ls = 0;
              lph ^= 1u;
            }
          }
        }
        // MMAs still in flight must finish before TMEM is released.
        if (it > 0) mbar_wait_drain(&tfull[(it - 1) % kPairBufs], ((it - 1) / kPairBufs) & 1u);
      }
      __syncwarp();
    }
  } else {
    // ---------------- epilogue: promotion + store (both CTAs) ----------------
    setmaxnreg_inc<kPairEpiRegs>();
    const int ew = warp - kCtlWarps;
    const int quad = warp & 3;   // TMEM lanes this warp may access
    const int half = ew >> 2;    // which 64 of the tile's 128 columns
    const int r_in_tile = quad * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tempty0 = mapa_shared(&tempty[0], 0);
    uint32_t it = 0;
    bool ok = true;
    for (int u = first; u < total && ok; u += stride) {
      const int tm = (u % m_groups) * 2 + rank, tn = u / m_groups;
      const int row = tm * BM + r_in_tile;
      const bool row_ok = row < M;
      const int col0 = tn * kPairBN + half * HALF;
      const float* sa_row = sA + static_cast<int64_t>(row_ok ? row : 0) * kchunks;
      const float* sb_col = sB + tn;  // a 128-column tile is one scale block

      uint64_t acc[HALF / 2];
#pragma unroll
      for (int j = 0; j < HALF / 2; ++j) acc[j] = 0ull;

      float sa_next = row_ok ? __ldg(sa_row) : 0.0f;
      float sb_next = __ldg(sb_col);
      for (int kc = 0; kc < kchunks; ++kc, ++it) {
        const uint32_t buf = it % kPairBufs, tph = (it / kPairBufs) & 1u;
        const float comb = sa_next * sb_next;
        if (kc + 1 < kchunks) {  // prefetch the next chunk's scales
          sa_next = row_ok ? __ldg(sa_row + kc + 1) : 0.0f;
          sb_next = __ldg(sb_col + static_cast<int64_t>(kc + 1) * nb);
        }
        const uint64_t comb2 = pack2(__float_as_uint(comb), __float_as_uint(comb));
        // warp-uniform outcome: the TMEM loads below are warp-collective
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tfull[buf], tph, abort_flag, FGQ_DEVERR_EPI_TMEM))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + t_lane + buf * kPairBN + half * HALF;
        uint32_t ra[32], rb[32];
        tmem_ld_32x32b_x32(taddr, ra);
        tmem_ld_32x32b_x32(taddr + 32, rb);
        tmem_wait_ld_regs(ra);
        tmem_wait_ld_regs(rb);
        // every column of this buffer is in registers (the reads have
        // completed): hand it back to the leader's MMA issuer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive_relaxed(&tempty[buf]);
          else
            mbar_arrive_cluster_relaxed(tempty0 + buf * 8);
        }
        promote32(acc, ra, comb2, 0);
        promote32(acc, rb, comb2, 16);
      }
      if (!ok) break;
      if (row_ok) {
        if (OUT_BF16) {
          uint16_t* crow = static_cast<uint16_t*>(C) + static_cast<int64_t>(row) * ldc + col0;
#pragma unroll
          for (int j = 0; j < HALF / 2; j += 4) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(acc[j])),
                              __uint_as_float(static_cast<uint32_t>(acc[j] >> 32)));
            v.y = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(acc[j + 1])),
                              __uint_as_float(static_cast<uint32_t>(acc[j + 1] >> 32)));
            v.z = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(acc[j + 2])),
                              __uint_as_float(static_cast<uint32_t>(acc[j + 2] >> 32)));
            v.w = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(acc[j + 3])),
                              __uint_as_float(static_cast<uint32_t>(acc[j + 3] >> 32)));
            *reinterpret_cast<uint4*>(crow + 2 * j) = v;
          }
        } else {
          float* crow = static_cast<float*>(C) + static_cast<int64_t>(row) * ldc + col0;
#pragma unroll
          for (int j = 0; j < HALF / 2; j += 2) {
            uint4 v = make_uint4(static_cast<uint32_t>(acc[j]), static_cast<uint32_t>(acc[j] >> 32),
                                 static_cast<uint32_t>(acc[j + 1]),
                                 static_cast<uint32_t>(acc[j + 1] >> 32));
            *reinterpret_cast<uint4*>(crow + 2 * j) = v;
          }
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync();  // neither CTA leaves while its peer may still reach its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, CF::kTmemCols);
  }
}

// ---- host side -------------------------------------------------------------------

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

namespace {

// Recently encoded descriptors, keyed by everything the encoding depends
// on (base address, rows, K, box rows).  A descriptor holds no device
// state, only the address and geometry, so an entry stays valid even if
// the memory behind it is freed and reallocated at the same address.
struct MapCacheEntry {
  const void* base;
  int64_t rows, K;
  int box_rows;
  int kind;  // 0: K-major operand, 1: FP4 scale tiles
  bool valid;
  CUtensorMap map;
};
constexpr int kMapCacheSize = 64;
MapCacheEntry g_map_cache[kMapCacheSize];
int g_map_cache_next = 0;
std::mutex g_map_cache_mu;

bool encode_k_major_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                        int box_rows);
bool encode_scale_tile_map(CUtensorMap* map, const void* base, int64_t tiles, int box_tiles);

bool cached_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows,
                int kind) {
  {
    std::lock_guard<std::mutex> lock(g_map_cache_mu);
    for (const MapCacheEntry& e : g_map_cache)
      if (e.valid && e.kind == kind && e.base == base && e.rows == rows && e.K == K &&
          e.box_rows == box_rows) {
        *map = e.map;
        return true;
      }
  }
  const bool ok = kind == 0 ? encode_k_major_map(map, base, rows, K, box_rows)
                            : encode_scale_tile_map(map, base, rows, box_rows);
  if (!ok) return false;
  std::lock_guard<std::mutex> lock(g_map_cache_mu);
  MapCacheEntry& e = g_map_cache[g_map_cache_next];
  g_map_cache_next = (g_map_cache_next + 1) % kMapCacheSize;
  e.base = base;
  e.rows = rows;
  e.K = K;
  e.box_rows = box_rows;
  e.kind = kind;
  e.map = *map;
  e.valid = true;
  return true;
}

}  // namespace

// K-major E4M3 operand [rows, K] (row stride K bytes), box 128 (K) x box_rows,
// 128-byte swizzle, out-of-range rows read as zero.  Served from a small
// cache of recent descriptors (the host-side encoding then runs once per
// operand, not once per call).
bool make_k_major_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows) {
  return cached_map(map, base, rows, K, box_rows, 0);
}

// FP4 scale tiles: 512-byte tiles seen as rows of 128 32-bit words, box of
// box_tiles rows, no swizzle, zero fill past the last tile.  Cached like
// the operand descriptors.
bool make_scale_tile_map(CUtensorMap* map, const void* base, int64_t tiles, int box_tiles) {
  return cached_map(map, base, tiles, 0, box_tiles, 1);
}

namespace {

bool encode_scale_tile_map(CUtensorMap* map, const void* base, int64_t tiles, int box_tiles) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t dims[2] = {128u, static_cast<cuuint64_t>(tiles)};
  cuuint64_t strides[1] = {512u};
  cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_tiles)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides,
                      box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_k_major_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                        int box_rows) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                      box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

namespace {

template <int BN, int STAGES, bool OUT_BF16>
cudaError_t launch_cfg(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                       void* C, int64_t ldc, int M, int N, int K, cudaStream_t stream,
                       const DeviceInfo& dev) {
  using CF = Cfg<BN, STAGES>;
  auto kern = gemm_fp8_blockscaled_kernel<BN, STAGES, OUT_BF16>;
  static bool ready[64] = {};
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (!ready[dev.device]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(CF::kSmemBytes));
      if (e != cudaSuccess) return e;
      // The setmaxnreg split assumes every thread is launched with
      // kLaunchRegs registers; with fewer the epilogue's increase could
      // never be granted.
      cudaFuncAttributes attr;
      e = cudaFuncGetAttributes(&attr, kern);
      if (e != cudaSuccess) return e;
      if (attr.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
      ready[dev.device] = true;
    }
  }
  CUtensorMap ta, tb;
  if (!make_k_major_map(&ta, A, M, K, BM) || !make_k_major_map(&tb, B, N, K, BN))
    return cudaErrorInvalidValue;
  const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int grid = tiles < dev.sm_count ? tiles : dev.sm_count;
  // 32-byte stores need every row segment 32-byte aligned: C itself and the
  // row pitch (column offsets are multiples of 128 elements)
  const int64_t pitch = ldc * (OUT_BF16 ? 2 : 4);
  const int wide = (reinterpret_cast<uintptr_t>(C) % 32 == 0 && pitch % 32 == 0) ? 1 : 0;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), CF::kSmemBytes, stream, ta, tb, sA, sB, C,
                    ldc, M, N, K, wide);
}

// Clusters of two that fit on the device at once (0 when the pair kernel
// cannot run), worked out once per device together with the launch checks.
template <bool OUT_BF16>
cudaError_t pair_clusters(const DeviceInfo& dev, int* clusters) {
  auto kern = gemm_fp8_pair_kernel<OUT_BF16>;
  static std::mutex mu;
  static int cached[64] = {};
  static bool ready[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev.device]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(PairCfg::kSmemBytes));
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    // the setmaxnreg split assumes this launch register count
    if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (dev.sm_count / 2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = PairCfg::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    cached[dev.device] = n;
    ready[dev.device] = true;
  }
  *clusters = cached[dev.device];
  return cudaSuccess;
}

template <bool OUT_BF16>
cudaError_t launch_pair(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                        void* C, int64_t ldc, int M, int N, int K, int clusters,
                        cudaStream_t stream) {
  CUtensorMap ta, tb;
  if (!make_k_major_map(&ta, A, M, K, BM) || !make_k_major_map(&tb, B, N, K, kPairBN / 2))
    return cudaErrorInvalidValue;
  const int units = ((((M + BM - 1) / BM) + 1) / 2) * (N / kPairBN);
  const int grid = 2 * (units < clusters ? units : clusters);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = PairCfg::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_fp8_pair_kernel<OUT_BF16>, ta, tb, sA, sB, C, ldc, M, N, K);
}

}  // namespace

cudaError_t launch_gemm_fp8_blockscaled(const uint8_t* A, const float* sA, const uint8_t* B,
                                        const float* sB, void* C, int64_t ldc, int64_t M,
                                        int64_t N, int64_t K, int out_bf16, int mode,
                                        cudaStream_t stream, const DeviceInfo& dev) {
  (void)mode;  // power-of-two scales take the same promotion path (exact products)
  if (M == 0 || N == 0) return cudaSuccess;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  // CTA pairs when there is at least one 256 x 128 tile per pair that fits
  const int64_t pair_units = (((M + BM - 1) / BM + 1) / 2) * (N / kPairBN);
  if (kUsePairs && M > BM) {
    int clusters = 0;
    const cudaError_t e =
        out_bf16 ? pair_clusters<true>(dev, &clusters) : pair_clusters<false>(dev, &clusters);
    if (e != cudaSuccess) return e;
    if (clusters > 0 && pair_units >= clusters)
      return out_bf16 ? launch_pair<true>(A, sA, B, sB, C, ldc, m, n, k, clusters, stream)
                      : launch_pair<false>(A, sA, B, sB, C, ldc, m, n, k, clusters, stream);
  }
  const int64_t tiles256 = ((M + BM - 1) / BM) * ((N + 255) / 256);
  const bool wide = (N % 256 == 0) && tiles256 >= dev.sm_count;
  if (out_bf16) {
    return wide ? launch_cfg<256, 4, true>(A, sA, B, sB, C, ldc, m, n, k, stream, dev)
                : launch_cfg<128, 6, true>(A, sA, B, sB, C, ldc, m, n, k, stream, dev);
  }
  return wide ? launch_cfg<256, 4, false>(A, sA, B, sB, C, ldc, m, n, k, stream, dev)
              : launch_cfg<128, 6, false>(A, sA, B, sB, C, ldc, m, n, k, stream, dev);
}

namespace {

// One warp: thread 0 sets up a barrier that expects one arrival, and no
// thread ever arrives, so the bounded wait (the one every kernel here uses)
// runs out after FGQ_WAIT_NS, records its site and returns.
__global__ void selftest_wait_timeout_kernel() {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, FGQ_DEVERR_SELFTEST);
}

}  // namespace

cudaError_t launch_selftest_wait_timeout(cudaStream_t stream) {
  selftest_wait_timeout_kernel<<<1, 32, 0, stream>>>();
  return cudaGetLastError();
}

cudaError_t read_device_error_gemm(uint32_t* word, bool clear) {
  return read_unit_device_error(word, clear);
}

}  // namespace fgq
