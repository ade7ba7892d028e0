// Block-scaled FP8 GEMM for sm_103a ("Fine-Grained FP8/FP4 Quantization",
// §DeepGEMM: Tile-wise and Block-wise Scaling):
//
//   C[m,n] = sum_c sA[m,c] * sB[c, n/128] * P_c[m,n],
//   P_c    = sum_{k in chunk c} Aq[m,k] * Bq[k,n]   (one 128-wide K chunk)
//
// Design (GB300-native; the page's Hopper promotion loop is prior art):
//   - Persistent CTAs, one per SM, walking output tiles of 128 x BN with a
//     static stride schedule ("Persistent kernel (grid = SM count, internal
//     tile loop)", linear scheduler, M fastest).  Large problems run on CTA
//     pairs (clusters of two) with tcgen05.mma.cta_group::2: one 256 x 256
//     MMA tile per pair, each CTA holding 128 rows of A and 128 rows of B per
//     stage and receiving its 128 output rows in its own TMEM.  The tensor
//     core reads the peer's operands directly, so each SM fills 32 KB of
//     shared memory per K chunk instead of 48 KB, which is what bounds the
//     single-CTA 128 x 256 tile.
//   - Warp 0: TMA producer.  Each stage holds one 128-wide K chunk of A
//     (128 x 128 bytes) and B (BN x 128 bytes), 128-byte swizzled.
//   - Warp 1: one thread issues 4 tcgen05.mma (K = 32 each) per chunk into
//     one of two TMEM partial buffers (128 lanes x BN fp32 columns each),
//     then commits to the stage's "empty" and the buffer's "full" barriers.
//   - Warps 4-11: epilogue.  Per chunk they read the partial from TMEM in
//     32-column loads (the next load in flight while the current one is
//     used), multiply by sA[m,c] * sB[c, n/128] (loaded four chunks ahead)
//     and add it into fp32 accumulators held in registers (the promotion
//     step), hand the TMEM buffer back as soon as it is read, and after the
//     last chunk convert and store the tile.  Two TMEM buffers let the
//     tensor core run chunk c+1 while chunk c is promoted.
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

// BN: output columns of a tile.  Each K chunk is computed as two MMAs of
// N = BN/2 (the column halves), each with its own TMEM-full / TMEM-empty
// barrier pair, so the epilogue warps of one half drain while the tensor
// core works on the other.  CG: CTAs per MMA (1, or 2 for the paired
// tcgen05.mma.cta_group::2: its 256-row tile is split so that each CTA holds
// 128 rows of A and, for each column half, BN/4 rows of B, and receives its
// own 128 rows of the result in its TMEM).
template <int BN, int STAGES, int CG>
struct Cfg {
  static constexpr int kABytes = BM * BK;
  static constexpr int kBHalfRows = BN / 2 / CG;              // B rows per column half per CTA
  static constexpr int kBHalfBytes = kBHalfRows * BK;
  static constexpr int kBBytes = 2 * kBHalfBytes;
  static constexpr int kStageBytes = kABytes + kBBytes;      // per CTA
  static constexpr uint32_t kTxBytes = CG * kStageBytes;     // per stage of the MMA
  static constexpr int kTmemCols = 2 * BN;                   // two partial buffers
  static constexpr int kBarBytes = (2 * STAGES + 8) * 8 + 16;
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

// acc[j0 + j] += comb * partial[j] for the 32 columns held in r.  (Called
// from fully unrolled loops, so j0 is a constant and acc stays in registers.)
template <int NACC>
__device__ __forceinline__ void promote32(float (&acc)[NACC], const uint32_t (&r)[32], float comb,
                                          int j0) {
#pragma unroll
  for (int j = 0; j < 32; ++j) fma_acc(acc[j0 + j], r[j], comb);
}

// Scales of the next chunks, loaded kScaleAhead chunks before use: a
// shift register of (sA[row, c], sB[c, block]) pairs.
constexpr int kScaleAhead = 4;

// Static persistent schedule over work units.  A unit is the CG stacked
// 128-row tiles one MMA covers (CG = 2: the two CTAs of a cluster, rank r
// taking tile row CG * g + r).  Units are walked M-fastest with stride = the
// number of MMA groups, so all roles of all CTAs agree on the order.
template <int CG>
struct TileSched {
  int m_groups, n_tiles, total, first, stride, rank;
  __device__ __forceinline__ TileSched(int M, int N, int bn) {
    const int m_tiles = (M + BM - 1) / BM;
    m_groups = (m_tiles + CG - 1) / CG;
    n_tiles = (N + bn - 1) / bn;
    total = m_groups * n_tiles;
    rank = CG == 1 ? 0 : static_cast<int>(cluster_ctarank());
    first = static_cast<int>(blockIdx.x) / CG;
    stride = static_cast<int>(gridDim.x) / CG;
  }
  __device__ __forceinline__ void tile(int u, int& tm, int& tn) const {
    tm = (u % m_groups) * CG + rank;
    tn = u / m_groups;
  }
};

template <int BN, int STAGES, int CG, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_blockscaled_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                const __grid_constant__ CUtensorMap tmap_b,
                                const float* __restrict__ sA, const float* __restrict__ sB,
                                void* __restrict__ C, int64_t ldc, int M, int N, int K) {
  using CF = Cfg<BN, STAGES, CG>;
  static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair per MMA");
  constexpr int HALF = BN / 2;     // columns per epilogue warp
  constexpr int NLD = HALF / 32;   // 32-column TMEM loads per chunk
  static_assert(NLD >= 2, "the load pipeline below assumes at least two loads per chunk");
  constexpr uint16_t kPair = 0x3;  // both CTAs of the pair
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sm_a = smem;
  uint8_t* sm_b = smem + STAGES * CF::kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm_b + STAGES * CF::kBBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;  // [buffer * 2 + column half]
  uint64_t* tempty = tfull + 4;      // [buffer * 2 + column half]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TileSched<CG> sched(M, N, BN);
  const bool leader = sched.rank == 0;  // issues the MMAs (always true for CG = 1)
  const int kchunks = K / BK;
  const int nb = N / 128;

  if (threadIdx.x == 0) {
    // Only the leader's full and tempty barriers are used when CG = 2; every
    // CTA receives the leader's commits on its own empty and tfull barriers.
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 4; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], (kEpiWarps / 2) * CG);  // the four warps of one half, per CTA
    }
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc<CG>(tmem_slot, CF::kTmemCols);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  if (CG > 1)
    cluster_sync();  // both CTAs' barriers and TMEM exist before either uses the other's
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < kCtlWarps) {
    setmaxnreg_dec<kCtlRegs>();
    if (warp == 0) {
      // ---------------- TMA producer (every CTA loads its own share) ----------------
      if (elect_one_sync()) {
        const uint32_t full_cluster0 = CG > 1 ? mapa_shared(&full[0], 0) : 0u;
        uint32_t it = 0;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int u = sched.first; u < sched.total && ok; u += sched.stride) {
          int tm, tn;
          sched.tile(u, tm, tn);
          // B rows of column half h held by this CTA: BN/2 rows from
          // tn * BN + h * BN/2, split between the CTAs of a pair.
          const int b_row = tn * BN + sched.rank * CF::kBHalfRows;
          const int a_row = tm * BM;
          for (int kc = 0; kc < kchunks; ++kc, ++it) {
            if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, FGQ_DEVERR_PRODUCER_EMPTY)) {
              ok = false;
              break;
            }
            uint8_t* a_dst = sm_a + s * CF::kABytes;
            uint8_t* b_dst = sm_b + s * CF::kBBytes;
            if (CG == 1) {
              mbar_arrive_expect_tx(&full[s], CF::kTxBytes);
              tma_load_2d(a_dst, &tmap_a, &full[s], kc * BK, a_row);
              tma_load_2d(b_dst, &tmap_b, &full[s], kc * BK, b_row);
              tma_load_2d(b_dst + CF::kBHalfBytes, &tmap_b, &full[s], kc * BK, b_row + BN / 2);
            } else {
              // both CTAs' copies complete on the leader's barrier
              if (leader) mbar_arrive_expect_tx(&full[s], CF::kTxBytes);
              const uint32_t bar = full_cluster0 + 8u * s;
              tma_load_2d_pair(a_dst, &tmap_a, bar, kc * BK, a_row);
              tma_load_2d_pair(b_dst, &tmap_b, bar, kc * BK, b_row);
              tma_load_2d_pair(b_dst + CF::kBHalfBytes, &tmap_b, bar, kc * BK, b_row + BN / 2);
            }
            if (++s == STAGES) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
        // Before leaving: every copy into the pair's shared memory has landed
        // (the leader's full barriers see both CTAs' copies) and every MMA
        // commit addressed to this CTA's empty barriers has arrived.
        const uint32_t first = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j) {
          if (leader) mbar_wait_drain(&full[j % STAGES], (j / STAGES) & 1u);
          mbar_wait_drain(&empty[j % STAGES], (j / STAGES) & 1u);
        }
      }
      __syncwarp();
    } else if (warp == 1 && leader) {
      // ---------------- MMA issuer (the leader CTA of a pair) ----------------
      if (elect_one_sync()) {
        constexpr uint32_t idesc = idesc_e4m3_f32(BM * CG, BN / 2);
        // Lean issue loop: this thread shares its scheduler with two epilogue
        // warps, so per-chunk work is a few 32-bit adds per MMA.
        const uint32_t a_lo0 = smem_desc_k_sw128_lo(smem_u32(sm_a));
        const uint32_t b_lo0 = smem_desc_k_sw128_lo(smem_u32(sm_b));
        uint32_t it = 0;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int u = sched.first; u < sched.total && ok; u += sched.stride) {
          for (int kc = 0; kc < kchunks; ++kc, ++it) {
            const uint32_t buf = it & 1u, tph = (it >> 1) & 1u;
            if (!mbar_wait(&full[s], ph, abort_flag, FGQ_DEVERR_MMA_FULL)) {
              ok = false;
              break;
            }
            const uint32_t a_lo = a_lo0 + s * (CF::kABytes >> 4);
            const uint32_t b_lo = b_lo0 + s * (CF::kBBytes >> 4);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint64_t* te = &tempty[buf * 2 + h];
              if (!mbar_wait(te, tph ^ 1u, abort_flag, FGQ_DEVERR_MMA_TMEM)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t d = tmem_base + buf * BN + h * (BN / 2);
#pragma unroll
              for (int kk = 0; kk < BK / 32; ++kk)
                umma_f8f6f4<CG>(d, make_desc(a_lo + kk * 2, kSmemDescK128Hi),
                                make_desc(b_lo + h * (CF::kBHalfBytes >> 4) + kk * 2, kSmemDescK128Hi),
                                idesc, kk > 0 ? 1u : 0u);
              if (CG == 1)
                umma_commit(&tfull[buf * 2 + h]);
              else
                umma_commit_pair(&tfull[buf * 2 + h], kPair);
            }
            if (!ok) break;
            if (CG == 1)
              umma_commit(&empty[s]);
            else
              umma_commit_pair(&empty[s], kPair);
            if (++s == STAGES) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
        // MMAs still in flight must finish before TMEM is released (the last
        // commit covers every MMA issued before it).
        if (it > 0) mbar_wait_drain(&tfull[((it - 1) & 1u) * 2 + 1], ((it - 1) >> 1) & 1u);
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
    for (int u = sched.first; u < sched.total && ok; u += sched.stride) {
      int tm, tn;
      sched.tile(u, tm, tn);
      const int row = tm * BM + r_in_tile;
      const bool row_ok = row < M;
      const int col0 = tn * BN + half * HALF;
      const bool cols_ok = col0 < N;
      const int nblk = cols_ok ? col0 / 128 : nb - 1;
      const float* sa_row = sA + static_cast<int64_t>(row_ok ? row : 0) * kchunks;
      const float* sb_col = sB + nblk;

      float acc[HALF];
#pragma unroll
      for (int j = 0; j < HALF; ++j) acc[j] = 0.0f;

      float sa_q[kScaleAhead], sb_q[kScaleAhead];
#pragma unroll
      for (int i = 0; i < kScaleAhead; ++i) {
        sa_q[i] = (row_ok && i < kchunks) ? __ldg(sa_row + i) : 0.0f;
        sb_q[i] = i < kchunks ? __ldg(sb_col + static_cast<int64_t>(i) * nb) : 0.0f;
      }
      for (int kc = 0; kc < kchunks; ++kc, ++it) {
        const uint32_t buf = it & 1u, tph = (it >> 1) & 1u;
        const float comb = sa_q[0] * sb_q[0];
#pragma unroll
        for (int i = 0; i + 1 < kScaleAhead; ++i) {
          sa_q[i] = sa_q[i + 1];
          sb_q[i] = sb_q[i + 1];
        }
        const int kn = kc + kScaleAhead;
        sa_q[kScaleAhead - 1] = (row_ok && kn < kchunks) ? __ldg(sa_row + kn) : 0.0f;
        sb_q[kScaleAhead - 1] = kn < kchunks ? __ldg(sb_col + static_cast<int64_t>(kn) * nb) : 0.0f;
        // warp-uniform outcome: the TMEM loads below are warp-collective
        if (!__all_sync(0xFFFFFFFFu,
                        mbar_wait(&tfull[buf * 2 + half], tph, abort_flag, FGQ_DEVERR_EPI_TMEM))) {
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
            // every column of this buffer is in registers: hand it back to
            // the MMA issuer (the leader CTA's barrier when CG = 2)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (leader)
                mbar_arrive_relaxed(&tempty[buf * 2 + half]);
              else
                mbar_arrive_cluster_relaxed(mapa_shared(&tempty[buf * 2 + half], 0));
            }
          }
          if (q % 2 == 0)
            promote32(acc, ra, comb, 32 * q);
          else
            promote32(acc, rb, comb, 32 * q);
          if (q + 1 < NLD) {
            if (q % 2 == 0)
              tmem_wait_ld_regs(rb);
            else
              tmem_wait_ld_regs(ra);
          }
        }
      }
      if (!ok) break;
      if (row_ok && cols_ok) {
        if (OUT_BF16) {
          uint16_t* crow = static_cast<uint16_t*>(C) + static_cast<int64_t>(row) * ldc + col0;
#pragma unroll
          for (int j = 0; j < HALF; j += 8) {
            uint4 v;
            v.x = pack_bf16x2(acc[j + 0], acc[j + 1]);
            v.y = pack_bf16x2(acc[j + 2], acc[j + 3]);
            v.z = pack_bf16x2(acc[j + 4], acc[j + 5]);
            v.w = pack_bf16x2(acc[j + 6], acc[j + 7]);
            *reinterpret_cast<uint4*>(crow + j) = v;
          }
        } else {
          float* crow = static_cast<float*>(C) + static_cast<int64_t>(row) * ldc + col0;
#pragma unroll
          for (int j = 0; j < HALF; j += 4)
            *reinterpret_cast<float4*>(crow + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  if (CG > 1)
    cluster_sync();  // neither CTA leaves while its peer may still reach its memory
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, CF::kTmemCols);
  }
}

// ---- host side -------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// K-major E4M3 operand [rows, K] (row stride K bytes), box 128 (K) x box_rows,
// 128-byte swizzle, out-of-range rows read as zero.
bool make_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows) {
  auto encode = get_encode_fn();
  if (!encode) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                      box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, int STAGES, int CG, bool OUT_BF16>
cudaError_t launch_cfg(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                       void* C, int64_t ldc, int M, int N, int K, cudaStream_t stream,
                       const DeviceInfo& dev) {
  using CF = Cfg<BN, STAGES, CG>;
  auto kern = gemm_fp8_blockscaled_kernel<BN, STAGES, CG, OUT_BF16>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = CF::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;

  // Per device: shared-memory opt-in, the launch register count the
  // setmaxnreg split assumes, and how many clusters fit at once.
  static std::mutex mu;
  static int max_clusters[64] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev.device >= 64) return cudaErrorInvalidDevice;
    if (max_clusters[dev.device] == 0) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(CF::kSmemBytes));
      if (e != cudaSuccess) return e;
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      // With fewer registers per thread than kLaunchRegs the epilogue's
      // setmaxnreg increase could never be granted: refuse to launch.
      if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
      int n = dev.sm_count / CG;
      if (CG > 1) {
        cfg.gridDim = dim3(CG * n);
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
      }
      max_clusters[dev.device] = n;
    }
  }
  CUtensorMap ta, tb;
  if (!make_operand_map(&ta, A, M, K, BM) || !make_operand_map(&tb, B, N, K, CF::kBHalfRows))
    return cudaErrorInvalidValue;
  const int m_groups = ((M + BM - 1) / BM + CG - 1) / CG;
  const int units = m_groups * ((N + BN - 1) / BN);
  const int clusters = units < max_clusters[dev.device] ? units : max_clusters[dev.device];
  cfg.gridDim = dim3(CG * clusters);
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, sA, sB, C, ldc, M, N, K);
}

}  // namespace

cudaError_t launch_gemm_fp8_blockscaled(const uint8_t* A, const float* sA, const uint8_t* B,
                                        const float* sB, void* C, int64_t ldc, int64_t M,
                                        int64_t N, int64_t K, int out_bf16, int mode,
                                        cudaStream_t stream, const DeviceInfo& dev) {
  (void)mode;  // power-of-two scales take the same promotion path (exact products)
  if (M == 0 || N == 0) return cudaSuccess;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  // 256 x 256 tiles on CTA pairs (tcgen05 cta_group::2) when there are
  // enough of them to fill the GPU; 128 x 128 single-CTA tiles otherwise.
  const int64_t m_tiles = (M + BM - 1) / BM;
  const int64_t pairs256 = ((m_tiles + 1) / 2) * ((N + 255) / 256);
  const bool wide = (N % 256 == 0) && m_tiles >= 2 && 2 * pairs256 >= dev.sm_count;
  if (out_bf16) {
    return wide ? launch_cfg<256, 6, 2, true>(A, sA, B, sB, C, ldc, m, n, k, stream, dev)
                : launch_cfg<128, 6, 1, true>(A, sA, B, sB, C, ldc, m, n, k, stream, dev);
  }
  return wide ? launch_cfg<256, 6, 2, false>(A, sA, B, sB, C, ldc, m, n, k, stream, dev)
              : launch_cfg<128, 6, 1, false>(A, sA, B, sB, C, ldc, m, n, k, stream, dev);
}

cudaError_t read_device_error(uint32_t* word, bool clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
  if (e != cudaSuccess) return e;
  if (clear && v != 0) {
    unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *word = v;
  return cudaSuccess;
}

}  // namespace fgq
