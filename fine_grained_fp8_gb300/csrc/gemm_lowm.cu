// Block-scaled FP8 GEMM for few rows of A (M <= 256), sm_103a.
//
// Same result as gemm.cu ("Fine-Grained FP8/FP4 Quantization", §DeepGEMM):
//   C[m,n] = sum_c sA[m,c] * sB[c, n/128] * sum_{k in chunk c} Aq[m,k] Bq[k,n]
// but laid out for the low-M regime, where the work is streaming the weight
// once from HBM:
//   - Swapped operands: the tensor core's 128-row dimension runs over 128
//     weight rows (n), its N dimension over the M rows of A padded to MP
//     (16..256).  The partial of a 128-K chunk lands in TMEM as
//     [128 lanes = n] x [MP columns = m]; no MMA rows are spent on padding.
//   - Scheduling ("Persistent kernel (grid = SM count, internal tile loop)",
//     §Scheduler: linear and stream-K).  The work is 128-column tiles of C,
//     each a run of K chunks.  Whole waves of tiles go to the CTAs one tile
//     each (data-parallel).  When a workspace is given, the tiles left over
//     after the last whole wave are not given out whole (that would leave
//     most SMs idle for a whole tile time): their K chunks, laid end to end,
//     are cut into equal contiguous ranges, one per CTA (stream-K), so every
//     CTA streams about the same number of weight chunks.  A range that
//     covers part of a tile yields a partial tile.
//   - Stream-K fix-up: each partial tile's CTA bumps the tile's arrival
//     counter first.  The last to arrive keeps its partial in registers,
//     waits (bounded) for the others' ready flags, adds the partials in the
//     order of the CTAs' ranges (a fixed order, so results are
//     deterministic), writes C and resets the counter and flags; the others
//     write their partial to their own workspace slot and raise their flag.
//     A waiting CTA only waits for CTAs that have already arrived, i.e.
//     finished their chunks, so the wait always ends.
//   - Warp 0 = TMA producer, warp 1 = MMA issuer, warps 4-11 = promotion
//     epilogue (each warp: 32 n-rows x MP/2 columns), the same roles and
//     bounded waits as gemm.cu.
//   - Batched promotion: the partials of kBatch = 256 / MP consecutive K
//     chunks go to adjacent TMEM slices of one of two slots, and the
//     epilogue waits once per batch, promotes its chunks with the next
//     slice's load in flight, and hands the slot back.  With the tensor
//     core filling the other slot meanwhile, the per-chunk wait and load
//     latency of the epilogue is off the weight stream's critical path.
// The products sA[m, c] * sB[c, n/128] of a tile are staged in shared
// memory in windows of 16 chunks ([chunk][m]), so the epilogue reads them
// as broadcast values and promotes with one FMA per element.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "fgq_device.cuh"
#include "fgq_internal.h"
#include "fgq_quant.cuh"

namespace fgq {
namespace {

// Prefetch the box at (x, y) of a 2-D tensor map into L2 (no shared-memory
// destination, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

constexpr int BN = 128;   // weight rows per tile (the MMA's M)
constexpr int BK = 128;   // one scale chunk per stage
constexpr int kCtlWarps = 4;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (kCtlWarps + kEpiWarps);
constexpr int kLaunchRegs = 168;
constexpr uint32_t kCtlRegs = 104;
constexpr uint32_t kEpiRegs = 200;
constexpr uint32_t kEpiBarrier = 1;      // named barrier of the 256 epilogue threads
constexpr uint32_t kQuantBarrier = 2;    // named barrier closing the in-kernel quantization
constexpr int kQuantWarps = 11;          // warps 1-11 quantize A (warp 0 streams the weight)
constexpr int kMaxSmemOptin = 232448;    // 227 KB of shared memory per CTA
constexpr int kScaleWindow = 16;         // K chunks of staged activation scales
static_assert(128 * kCtlRegs + 256 * kEpiRegs <= kThreads * kLaunchRegs, "register split");

template <int MP>
struct LowCfg {
  static constexpr int kBBytes = BN * BK;        // weight tile (MMA operand A)
  static constexpr int kABytes = MP * BK;        // activation tile (MMA operand B)
  static constexpr int kStageBytes = kBBytes + kABytes;
  static constexpr int STAGES = MP <= 64 ? 6 : 4;
  // Two TMEM slots of kBatch chunk partials each (MP columns per partial).
  static constexpr int kBatch = MP >= 256 ? 1 : 256 / MP;
  static constexpr int kSlotCols = kBatch * MP;
  static constexpr int kTmemCols = 2 * kSlotCols;
  static constexpr int kScaleBytes = kScaleWindow * MP * 4;
  static constexpr int kBarBytes = (2 * STAGES + 5) * 8 + 16;
  static constexpr size_t kSmemBytes =
      1024 + static_cast<size_t>(STAGES) * kStageBytes + kScaleBytes + kBarBytes + 16;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(MP % 16 == 0 && MP >= 16 && MP <= 256, "MMA N");
  static_assert(kTmemCols == 512, "TMEM allocation");
  // Activation scales of all chunks when A is quantized in the kernel.
  static __host__ __device__ constexpr int fused_scale_bytes(int kchunks) {
    return ((kchunks * MP * 4 + 15) / 16) * 16;
  }
  static constexpr size_t fused_smem_bytes(int kchunks) {
    return 1024 + static_cast<size_t>(STAGES) * kBBytes + static_cast<size_t>(kchunks) * kABytes +
           fused_scale_bytes(kchunks) + kBarBytes + 16;
  }
  static_assert(kScaleWindow % kBatch == 0, "a batch never straddles a scale window");
  // Cluster-pair split (below): the receive buffer of the peer's partial tile
  // and its barrier, after the control words.
  static constexpr int kRecvBytes = MP * BN * 4;
  static constexpr size_t kPairSmemBytes = kSmemBytes + 64 + kRecvBytes;
  static_assert(MP > 64 || kPairSmemBytes <= 232448, "shared memory per CTA (pairs)");
};

// Loads of W consecutive TMEM columns into r[0..W-1] (r points into a
// register array at a compile-time offset).
template <int W>
__device__ __forceinline__ void tmem_ld_cols_to(uint32_t taddr, uint32_t* r);
template <>
__device__ __forceinline__ void tmem_ld_cols_to<32>(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
template <>
__device__ __forceinline__ void tmem_ld_cols_to<16>(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
template <>
__device__ __forceinline__ void tmem_ld_cols_to<8>(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
}

// Wait for outstanding TMEM loads, tying 64 destination registers to the
// wait (the second wait finds nothing outstanding and only ties the upper
// half) so that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_wait_ld_regs64(uint32_t* r) {
  tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(r));
  tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(r + 32));
}

// Bounded wait used while unwinding; ignores the abort flag.
__device__ __forceinline__ bool lowm_wait_drain(uint64_t* bar, uint32_t parity) {
  unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > FGQ_WAIT_NS) {
      record_error(FGQ_DEVERR_DRAIN);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// The work of one CTA: its stream-K range first, then its whole tiles, then
// the fix-ups it was handed.
//   - Tiles [0, dp_tiles) run whole: CTA b takes tiles b, b + G, b + 2G, ...
//   - The chunks of tiles [dp_tiles, n_tiles), laid end to end (sk_chunks of
//     them), are split among CTAs [0, sk_ctas): CTA b takes the chunks
//     [b * sk_chunks / sk_ctas, (b + 1) * sk_chunks / sk_ctas).  The host
//     keeps sk_ctas <= sk_chunks, so every range is non-empty.
//   - When some CTAs have no stream-K range (reducers = G - sk_ctas > 0),
//     stream-K tile j also gets a fix-up item on CTA sk_ctas + j % reducers,
//     after its whole tiles: that CTA, done early, usually arrives last and
//     adds the partials, so the CTAs with ranges publish and move on.
// Item i of a CTA is (tile, chunk range [c0, c1), j, kind): j is the
// stream-K tile index (tile - dp_tiles) of a partial tile or a fix-up item,
// -1 for a whole one.  The partial of CTA b for stream-K tile j goes to
// workspace slot b + j (slots are distinct: a CTA's tiles increase, and the
// next CTA starts at or after its last tile).
struct LowSched {
  int n_tiles, kchunks, dp_tiles, sk_ctas, reducers;
  long long sk_chunks;
  // Cluster-pair split (no workspace): the tiles [dp_tiles, dp_tiles +
  // pair_tiles) are split in K between the two CTAs of cluster c (tile
  // dp_tiles + c): rank 0 takes chunks [0, kchunks / 2), rank 1 the rest and
  // sends its partial to rank 0 through distributed shared memory.
  int pair_tiles;

  // One CTA's list, worked out once (the only divisions); item() then takes
  // constant time without dividing.
  struct Cta {
    int n_items, nsk, ndp;
    int j_first, c_first;  // first stream-K tile and its first chunk
    int j_last, c_last;    // last stream-K tile and the end of its range
    int red0;              // first stream-K tile this CTA fixes up (-1: none)
  };
  __device__ __forceinline__ Cta cta(int b, int G) const {
    Cta w{};
    w.red0 = -1;
    if (pair_tiles > 0) {
      const int c = b >> 1, r = b & 1, h = kchunks / 2;
      if (c < pair_tiles) {
        w.nsk = 1;
        w.j_first = w.j_last = c;
        w.c_first = r ? h : 0;
        w.c_last = r ? kchunks : h;
      }
    } else if (b < sk_ctas) {
      const long long s0 = static_cast<long long>(b) * sk_chunks / sk_ctas;
      const long long s1 = static_cast<long long>(b + 1) * sk_chunks / sk_ctas;
      if (s1 > s0) {
        w.j_first = static_cast<int>(s0 / kchunks);
        w.c_first = static_cast<int>(s0 - static_cast<long long>(w.j_first) * kchunks);
        w.j_last = static_cast<int>((s1 - 1) / kchunks);
        w.c_last = static_cast<int>(s1 - static_cast<long long>(w.j_last) * kchunks);
        w.nsk = w.j_last - w.j_first + 1;
      }
    }
    w.ndp = b < dp_tiles ? (dp_tiles - 1 - b) / G + 1 : 0;
    int nred = 0;
    const int L = n_tiles - dp_tiles;
    if (reducers > 0 && b >= sk_ctas && b - sk_ctas < reducers && b - sk_ctas < L) {
      w.red0 = b - sk_ctas;
      nred = (L - 1 - w.red0) / reducers + 1;
    }
    w.n_items = w.nsk + w.ndp + nred;
    return w;
  }
  // kind: 0 a chunk range of a tile, 1 a fix-up only (no chunks)
  __device__ __forceinline__ void item(const Cta& w, int b, int G, int i, int& tile, int& c0,
                                       int& c1, int& j, int& kind) const {
    kind = 0;
    if (i < w.nsk) {
      const int jj = w.j_first + i;
      c0 = i == 0 ? w.c_first : 0;
      c1 = jj == w.j_last ? w.c_last : kchunks;
      tile = dp_tiles + jj;
      j = (c0 == 0 && c1 == kchunks) ? -1 : jj;
      if (pair_tiles > 0) kind = 2;  // half of a tile split within the cluster
    } else if (i < w.nsk + w.ndp) {
      tile = b + (i - w.nsk) * G;
      c0 = 0;
      c1 = kchunks;
      j = -1;
    } else {
      j = w.red0 + (i - w.nsk - w.ndp) * reducers;
      tile = dp_tiles + j;
      c0 = c1 = 0;
      kind = 1;
    }
  }
  // The CTAs whose ranges meet stream-K tile j: b_lo .. b_hi (the largest b
  // with b * sk_chunks / sk_ctas <= x is ((x + 1) * sk_ctas - 1) / sk_chunks).
  __device__ __forceinline__ void seg_ctas(int j, int& b_lo, int& b_hi) const {
    const long long x0 = static_cast<long long>(j) * kchunks, x1 = x0 + kchunks - 1;
    b_lo = static_cast<int>(((x0 + 1) * sk_ctas - 1) / sk_chunks);
    b_hi = static_cast<int>(((x1 + 1) * sk_ctas - 1) / sk_chunks);
    if (b_hi > sk_ctas - 1) b_hi = sk_ctas - 1;
  }
};

// acc[off + jj] += p[jj] * c[jj] for jj < W, with c the staged multipliers
// (read as float4 broadcasts); with A quantized in the kernel the staged
// values are sA alone and the multiplier is c[jj] * sb, the same product.
template <int W, bool MUL_SB, int HALFW>
__device__ __forceinline__ void promote_cols(float (&acc)[HALFW], int off, const uint32_t* p,
                                             const float* c, float sb) {
  const float4* c4 = reinterpret_cast<const float4*>(c);
#pragma unroll
  for (int v = 0; v < W / 4; ++v) {
    const float4 m = c4[v];
    const float mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
    for (int t = 0; t < 4; ++t)
      acc[off + 4 * v + t] =
          fmaf(__uint_as_float(p[4 * v + t]), MUL_SB ? mm[t] * sb : mm[t], acc[off + 4 * v + t]);
  }
}

__device__ __forceinline__ void st_release_u32(unsigned int* p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait (bounded) until another CTA has raised *flag.  Gives up after
// FGQ_WAIT_NS of %globaltimer time, or when another warp of this CTA already
// gave up, recording FGQ_DEVERR_SK_FLAG and setting the abort flag.
__device__ __forceinline__ bool wait_flag(const unsigned int* flag, volatile int* abort) {
  if (ld_acquire_u32(flag) != 0u) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire_u32(flag) != 0u) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > FGQ_WAIT_NS) {
        record_error(FGQ_DEVERR_SK_FLAG);
        *abort = 1;
        return false;
      }
    }
  }
}

// FUSE = 0: A comes quantized (codes by TMA per stage, scales sA).  FUSE =
// kScaleFp32 + 1 or kScaleUe8m0 + 1: A comes as bf16 (a16, row stride lda)
// and is quantized here, 1x128 groups with the same arithmetic as
// fgq_quant_act_1x128, into shared memory that holds all of A's K chunks
// (codes in the 128-byte-swizzled layout a TMA load would write) and their
// scales for the whole kernel.
// PAIR: launched in clusters of two with the cluster-pair split of the
// schedule (sched.pair_tiles); the receive buffer and its barrier follow the
// control words in shared memory.
template <int MP, bool OUT_BF16, int FUSE, bool PAIR = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_lowm_kernel(const __grid_constant__ CUtensorMap tmap_w,   // Wq [N, K], box 128 x BN rows
                     const __grid_constant__ CUtensorMap tmap_a,   // Aq [M, K], box 128 x MP rows
                     const float* __restrict__ sA, const float* __restrict__ sB, void* __restrict__ C,
                     int64_t ldc, int M, int N, int K, LowSched sched,
                     float* __restrict__ partial,          // [slots][M][128] fp32 (stream-K)
                     unsigned int* __restrict__ counters,  // [stream-K tiles], zero between calls
                     unsigned int* __restrict__ flags,     // [slots], zero between calls
                     const uint16_t* __restrict__ a16, int64_t lda) {
  using CF = LowCfg<MP>;
  constexpr int STAGES = CF::STAGES;
  constexpr int HALF = MP / 2;                   // columns (m) per epilogue warp
  constexpr int LW = HALF >= 32 ? 32 : HALF;     // columns per TMEM load
  constexpr int NLD = HALF / LW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int kchunks_all = K / BK;
  uint8_t* sm_w = smem;                                   // STAGES x weight tiles
  uint8_t* sm_a = smem + STAGES * CF::kBBytes;            // activation tiles: STAGES, or all chunks
  float* sm_sa = reinterpret_cast<float*>(
      sm_a + (FUSE ? kchunks_all : STAGES) * CF::kABytes);  // [chunk][MP]: a window, or all chunks
  uint64_t* full = reinterpret_cast<uint64_t*>(
      reinterpret_cast<uint8_t*>(sm_sa) + (FUSE ? CF::fused_scale_bytes(kchunks_all) : CF::kScaleBytes));
  uint64_t* empty = full + STAGES;
  constexpr int kBatch = CF::kBatch;
  uint64_t* tfull = empty + STAGES;   // [2] slot holds a finished batch
  uint64_t* tempty = tfull + 2;       // [2] slot drained by the epilogue
  uint64_t* drain = tempty + 2;       // the MMA issuer's last commit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  uint64_t* recv_bar = reinterpret_cast<uint64_t*>(tmem_slot + 4);  // 8-byte aligned
  float* recv = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(recv_bar + 1) + 15) & ~static_cast<uintptr_t>(15));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kchunks = sched.kchunks;
  const int G = static_cast<int>(gridDim.x);
  const LowSched::Cta cw = sched.cta(blockIdx.x, G);
  const int n_items = cw.n_items;
  const int nb = N / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiWarps);
    }
    mbar_init(drain, 1);
    if (PAIR) mbar_init(recv_bar, 32 * kEpiWarps);  // every epilogue thread of the peer
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_w);
    if (!FUSE) tma_prefetch_desc(&tmap_a);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, CF::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  if (PAIR)
    cluster_sync();  // the peer's receive barrier exists before anyone arrives on it
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above (barrier set-up, TMEM allocation) may overlap the
  // previous kernel in the stream; global memory is read only after it has
  // completed.  The one exception is an L2 prefetch of this CTA's first
  // weight chunks: it returns no data and every later read goes through
  // L2, where the previous kernel's writes land, so it cannot see stale
  // bytes.  On SMs the previous kernel has already left, it starts the
  // weight stream during that kernel's last wave (M = 16 skinny sweep,
  // graph-replayed: 9.65 -> 9.27 us).
  if (threadIdx.x == 0 && n_items > 0) {
    int pnt, pc0, pc1, pj, pkind;
    sched.item(cw, blockIdx.x, G, 0, pnt, pc0, pc1, pj, pkind);
    if (pkind != 1)
      for (int kc = pc0; kc < pc1; ++kc) tma_prefetch_l2_2d(&tmap_w, kc * BK, pnt * BN);
  }
  pdl_wait();
  pdl_launch_dependents();

  if constexpr (FUSE != 0) {
    // Quantize all of A into shared memory (warp 0 starts streaming the
    // weight meanwhile).  Eight lanes per 1x128 group, as the activation
    // quantizer: lane l8 holds elements 8 l8 .. 8 l8 + 7 and 64 + 8 l8 ..
    // 64 + 8 l8 + 7.  Rows m >= M get zero codes and scale 0.
    if (warp != 0) {
      constexpr int QMODE = FUSE - 1;
      constexpr int kRounds = 6;  // groups per lane-octet with loads in flight together
      constexpr int kStride = kQuantWarps * 4;
      const int sub = lane >> 3, l8 = lane & 7;
      const int groups = MP * kchunks_all;
      // gw is the same for the whole warp (the shuffles below need all lanes)
      for (int gw = (warp - 1) * 4; gw < groups; gw += kStride * kRounds) {
        const int gb = gw + sub;
        uint4 v0[kRounds], v1[kRounds];
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
          const int g = gb + r * kStride, c = g / MP, m = g - c * MP;
          v0[r] = v1[r] = make_uint4(0, 0, 0, 0);
          if (g < groups && m < M) {
            const uint16_t* src = a16 + static_cast<int64_t>(m) * lda + c * BK;
            v0[r] = ld_stream_16(src + 8 * l8);
            v1[r] = ld_stream_16(src + 64 + 8 * l8);
          }
        }
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
          const int g = gb + r * kStride, c = g / MP, m = g - c * MP;
          uint32_t mx = __vmaxu2(absmax_pairs(v0[r]), absmax_pairs(v1[r]));
#pragma unroll
          for (int off = 4; off > 0; off >>= 1) mx = __vmaxu2(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
          const GroupScale gs = group_scale<QMODE>(max(mx & 0xFFFFu, mx >> 16));
          if (g < groups) {
            const uint2 q0 = encode8<QMODE>(v0[r], gs), q1 = encode8<QMODE>(v1[r], gs);
            // row m of chunk c: 128 bytes in its 1024-byte atom, 16-byte
            // units XOR-swizzled by m % 8 (the TMA SWIZZLE_128B layout)
            uint8_t* row = sm_a + c * CF::kABytes + (m >> 3) * 1024 + (m & 7) * 128;
            const int u0 = (l8 >> 1) ^ (m & 7), u1 = (4 + (l8 >> 1)) ^ (m & 7);
            *reinterpret_cast<uint2*>(row + u0 * 16 + (l8 & 1) * 8) = q0;
            *reinterpret_cast<uint2*>(row + u1 * 16 + (l8 & 1) * 8) = q1;
            if (l8 == 0) sm_sa[c * MP + m] = m < M ? gs.s : 0.0f;
          }
        }
      }
      // the tensor core reads these codes through the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      named_barrier_sync(kQuantBarrier, 32 * kQuantWarps);
    }
  }

  if (warp < kCtlWarps) {
    setmaxnreg_dec<kCtlRegs>();
    if (warp == 0) {
      // ---------------- TMA producer ----------------
      if (elect_one_sync()) {
        uint32_t it = 0;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int i = 0; i < n_items && ok; ++i) {
          int nt, c0, c1, jsk, kind;
          sched.item(cw, blockIdx.x, G, i, nt, c0, c1, jsk, kind);
          for (int kc = c0; kc < c1; ++kc, ++it) {
            if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, FGQ_DEVERR_PRODUCER_EMPTY)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[s], FUSE ? CF::kBBytes : CF::kStageBytes);
            tma_load_2d(sm_w + s * CF::kBBytes, &tmap_w, &full[s], kc * BK, nt * BN);
            if (!FUSE) tma_load_2d(sm_a + s * CF::kABytes, &tmap_a, &full[s], kc * BK, 0);
            if (++s == STAGES) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
        const uint32_t first = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j) lowm_wait_drain(&full[j % STAGES], (j / STAGES) & 1u);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      if (elect_one_sync()) {
        constexpr uint32_t idesc = idesc_e4m3_f32(BN, MP);
        const uint64_t dW0 = smem_desc_k_sw128(smem_u32(sm_w));
        const uint32_t w_lo0 = static_cast<uint32_t>(dW0), dhi = static_cast<uint32_t>(dW0 >> 32);
        const uint32_t a_lo0 = static_cast<uint32_t>(smem_desc_k_sw128(smem_u32(sm_a)));
        uint32_t bt = 0;  // batches issued
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int i = 0; i < n_items && ok; ++i) {
          int nt, c0, c1, jsk, kind;
          sched.item(cw, blockIdx.x, G, i, nt, c0, c1, jsk, kind);
          for (int kc = c0; kc < c1; ++kc) {
            const int j = (kc - c0) % kBatch;
            const uint32_t slot = bt & 1u;
            if (j == 0 && !mbar_wait(&tempty[slot], ((bt >> 1) & 1u) ^ 1u, abort_flag,
                                     FGQ_DEVERR_MMA_TMEM)) {
              ok = false;
              break;
            }
            if (!mbar_wait(&full[s], ph, abort_flag, FGQ_DEVERR_MMA_FULL)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem_base + slot * CF::kSlotCols + j * MP;
            const uint32_t w_lo = w_lo0 + s * (CF::kBBytes >> 4);
            // the stage's A tile, or the resident tile of chunk kc
            const uint32_t a_lo = a_lo0 + (FUSE ? kc : s) * (CF::kABytes >> 4);
#pragma unroll
            for (int kk = 0; kk < BK / 32; ++kk)
              umma_f8f6f4(d, make_desc(w_lo + kk * 2, dhi), make_desc(a_lo + kk * 2, dhi), idesc,
                             kk > 0 ? 1u : 0u);
            umma_commit(&empty[s]);
            if (j == kBatch - 1 || kc == c1 - 1) {
              umma_commit(&tfull[slot]);
              ++bt;
            }
            if (++s == STAGES) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
        // Every MMA this thread issued must finish before TMEM is released:
        // a last commit, on a barrier of its own, covers all of them (also
        // after giving up mid-batch).
        umma_commit(drain);
        lowm_wait_drain(drain, 0);
      }
      __syncwarp();
    }
  } else {
    // ---------------- epilogue: promotion, split-K reduction, store ----------------
    setmaxnreg_inc<kEpiRegs>();
    const int et = threadIdx.x - 32 * kCtlWarps;   // 0..255
    const int quad = warp & 3;
    const int half = (warp - kCtlWarps) >> 2;
    const int r_in_tile = quad * 32 + lane;         // weight row within the tile
    const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
    const int m0 = half * HALF;                     // first column (row of A) of this warp
    uint32_t bt = 0;  // batches consumed
    bool ok = true;
    for (int i = 0; i < n_items && ok; ++i) {
      int nt, c0, c1, jsk, kind;
      sched.item(cw, blockIdx.x, G, i, nt, c0, c1, jsk, kind);
      const int n = nt * BN + r_in_tile;

      float acc[HALF];
#pragma unroll
      for (int j = 0; j < HALF; ++j) acc[j] = 0.0f;
      bool ok_unit = true;
      for (int kb = c0; kb < c1; kb += kBatch, ++bt) {
        const int nbt = min(kBatch, c1 - kb);
        // Stage the window's multipliers sA[m, c] * sB[c, nt] as [chunk][m]
        // (zero for m >= M) at the start of every window of kScaleWindow
        // chunks (a whole number of batches).  Every epilogue warp runs every
        // batch (a warp that gave up on a wait only skips the work), so all
        // of them reach these barriers.  With A quantized in the kernel the
        // staged values are sA alone (all chunks), and sB is applied below.
        const int w0 = FUSE ? kb : (kb - c0) % kScaleWindow;  // row of sm_sa for chunk kb
        if (!FUSE && w0 == 0) {
          named_barrier_sync(kEpiBarrier, 32 * kEpiWarps);  // earlier readers done
          const int nck = min(kScaleWindow, c1 - kb);
          for (int e = et; e < nck * MP; e += 32 * kEpiWarps) {
            const int c = e / MP, m = e - c * MP;
            sm_sa[e] = m < M ? __ldg(sA + static_cast<int64_t>(m) * kchunks + kb + c) *
                                   __ldg(sB + static_cast<int64_t>(kb + c) * nb + nt)
                             : 0.0f;
          }
          named_barrier_sync(kEpiBarrier, 32 * kEpiWarps);
        }
        if (!ok_unit) continue;
        const uint32_t slot = bt & 1u;
        if (!__all_sync(0xFFFFFFFFu,
                        mbar_wait(&tfull[slot], (bt >> 1) & 1u, abort_flag, FGQ_DEVERR_EPI_TMEM))) {
          ok_unit = false;
          continue;
        }
        tc_fence_after();
        // partial of chunk j of the batch: TMEM columns slot*kSlotCols + j*MP
        const uint32_t taddr = tmem_base + t_lane + slot * CF::kSlotCols + m0;
        if (NLD == 1) {
          // waves of P chunks: P loads in flight, one wait, then P promotions
          constexpr int P = 64 / LW;
          for (int j0 = 0; j0 < nbt; j0 += P) {
            float sbv[P];
            uint32_t r[64];
#pragma unroll
            for (int p = 0; p < P; ++p) {
              const int j = j0 + p < nbt ? j0 + p : nbt - 1;  // repeat the last in-range chunk
              sbv[p] = FUSE ? __ldg(sB + static_cast<int64_t>(kb + j) * nb + nt) : 1.0f;
              tmem_ld_cols_to<LW>(taddr + j * MP, r + p * LW);
            }
            tmem_wait_ld_regs64(r);
#pragma unroll
            for (int p = 0; p < P; ++p) {
              if (j0 + p < nbt)
                promote_cols<LW, FUSE != 0>(acc, 0, r + p * LW, sm_sa + (w0 + j0 + p) * MP + m0,
                                            sbv[p]);
            }
          }
        } else if (NLD == 2) {
          for (int j = 0; j < nbt; ++j) {  // both halves in flight, one wait
            const float sb = FUSE ? __ldg(sB + static_cast<int64_t>(kb + j) * nb + nt) : 1.0f;
            const float* cm = sm_sa + (w0 + j) * MP + m0;
            uint32_t r[64];
            tmem_ld_cols_to<LW>(taddr + j * MP, r);
            tmem_ld_cols_to<LW>(taddr + j * MP + LW, r + LW);
            tmem_wait_ld_regs64(r);
            promote_cols<2 * LW, FUSE != 0>(acc, 0, r, cm, sb);
          }
        } else {
          // a 128-column accumulator: two 32-column loads alternate, the next
          // one in flight while the current one is promoted
          for (int j = 0; j < nbt; ++j) {
            const float sb = FUSE ? __ldg(sB + static_cast<int64_t>(kb + j) * nb + nt) : 1.0f;
            const float* cm = sm_sa + (w0 + j) * MP + m0;
            uint32_t ra[32], rb[32];
            tmem_ld_cols_to<32>(taddr + j * MP, ra);
            tmem_wait_ld_regs(ra);
#pragma unroll
            for (int q = 0; q < NLD; ++q) {
              if (q + 1 < NLD) tmem_ld_cols_to<32>(taddr + j * MP + 32 * (q + 1), q % 2 == 0 ? rb : ra);
              if (q % 2 == 0)
                promote_cols<32, FUSE != 0>(acc, 32 * q, ra, cm + 32 * q, sb);
              else
                promote_cols<32, FUSE != 0>(acc, 32 * q, rb, cm + 32 * q, sb);
              if (q + 1 < NLD) {
                if (q % 2 == 0)
                  tmem_wait_ld_regs(rb);
                else
                  tmem_wait_ld_regs(ra);
              }
            }
          }
        }
        // every partial of the batch is in registers: hand the slot back
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(&tempty[slot]);
      }
      // Every epilogue warp reaches this barrier once per item, whether it
      // finished its chunks or gave up on a wait; continue only together.
      ok = named_barrier_and(kEpiBarrier, 32 * kEpiWarps, ok_unit);
      if (!ok) break;

      // (Loops over acc are unrolled with per-element guards so that acc
      // stays in registers.)
      if (PAIR && kind == 2) {
        // Half of a tile split within the cluster: rank 1 sends its partial
        // into rank 0's receive buffer (distributed shared memory, layout
        // [HALF/4][256 threads][4]); rank 0 adds it to its own (rank 0's
        // half plus rank 1's: a fixed order) and writes C.
        if (blockIdx.x & 1) {
          const uint32_t dst = mapa_shared(recv, 0) + static_cast<uint32_t>(et) * 16;
#pragma unroll
          for (int g = 0; g < HALF / 4; ++g)
            asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst + g * 4096),
                         "f"(acc[4 * g]), "f"(acc[4 * g + 1]), "f"(acc[4 * g + 2]), "f"(acc[4 * g + 3])
                         : "memory");
          mbar_arrive_cluster(mapa_shared(recv_bar, 0));  // release: orders the stores above
        } else {
          ok = named_barrier_and(kEpiBarrier, 32 * kEpiWarps,
                                 mbar_wait_cluster(recv_bar, 0, abort_flag, FGQ_DEVERR_SK_FLAG));
          if (!ok) break;
          const float4* src = reinterpret_cast<const float4*>(recv) + et;
#pragma unroll
          for (int g = 0; g < HALF / 4; ++g) {
            const float4 v = src[g * 256];
            const float pv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int m = m0 + 4 * g + t;
              if (m < M) {
                const float sum = acc[4 * g + t] + pv[t];
                if (OUT_BF16)
                  static_cast<uint16_t*>(C)[static_cast<int64_t>(m) * ldc + n] = f32_to_bf16_rn(sum);
                else
                  static_cast<float*>(C)[static_cast<int64_t>(m) * ldc + n] = sum;
              }
            }
          }
        }
        continue;
      }
      if (jsk < 0) {  // a whole tile
#pragma unroll
        for (int j = 0; j < HALF; ++j) {
          const int m = m0 + j;
          if (m < M) {
            if (OUT_BF16)
              static_cast<uint16_t*>(C)[static_cast<int64_t>(m) * ldc + n] = f32_to_bf16_rn(acc[j]);
            else
              static_cast<float*>(C)[static_cast<int64_t>(m) * ldc + n] = acc[j];
          }
        }
        continue;  // the staged scales were last read before the barrier above
      }

      // ---- stream-K fix-up of a partial tile ----
      // Partial layout of a slot: [HALF/4 groups][256 threads][4 floats], so
      // that every epilogue thread moves its own values with 16-byte
      // accesses and a warp's accesses are 512 contiguous bytes.
      // A fix-up item contributes no partial; the tile's arrivals are its
      // range CTAs plus, when fix-ups are handed out, the reducer.
      const bool contributes = kind == 0;
      int b_lo, b_hi;
      sched.seg_ctas(jsk, b_lo, b_hi);
      if (et == 0) {
        const unsigned int arrivals = static_cast<unsigned int>(b_hi - b_lo + 1) +
                                      (sched.reducers > 0 ? 1u : 0u);
        const unsigned int prev = atomicAdd(&counters[jsk], 1u);
        *last_flag = prev + 1 == arrivals ? 1 : 0;
      }
      named_barrier_sync(kEpiBarrier, 32 * kEpiWarps);
      const bool last = *last_flag != 0;
      if (!last && !contributes) continue;  // a range CTA arrives after it and adds up
      if (!last) {
        // Publish: every thread stores its values, the barrier orders those
        // stores before thread 0's release store of the flag (release is
        // cumulative), so one release covers the whole partial tile.
        float4* my = reinterpret_cast<float4*>(partial) +
                     static_cast<int64_t>(blockIdx.x + jsk) * (HALF / 4) * 256 + et;
#pragma unroll
        for (int g = 0; g < HALF / 4; ++g)
          __stcg(my + g * 256, make_float4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3]));
        named_barrier_sync(kEpiBarrier, 32 * kEpiWarps);
        if (et == 0) st_release_u32(&flags[blockIdx.x + jsk], 1u);
        continue;
      }
      // The last to arrive: every other CTA of this tile has arrived, so it
      // has finished its chunks and is writing its partial; wait for its
      // flag (bounded), then add the partials in CTA order.
      const int me = contributes ? static_cast<int>(blockIdx.x) : -1;
      bool ready = true;
      if (et == 0) {
        for (int b = b_lo; b <= b_hi && ready; ++b)
          if (b != me) ready = wait_flag(&flags[b + jsk], abort_flag);
      }
      // thread 0's acquire loads, then the barrier, order the others' reads
      // of the partials after the peers' release stores
      ok = named_barrier_and(kEpiBarrier, 32 * kEpiWarps, ready);
      if (!ok) break;
      // GW groups of 4 values of up to P peers are loaded together, then
      // added in CTA order.
      constexpr int GW = HALF <= 16 ? HALF / 4 : (HALF <= 64 ? 4 : 2);
      constexpr int P = HALF <= 32 ? 3 : 2;
#pragma unroll
      for (int g0 = 0; g0 < HALF / 4; g0 += GW) {
        float sum[4 * GW];
#pragma unroll
        for (int t = 0; t < 4 * GW; ++t) sum[t] = 0.0f;
        for (int b0 = b_lo; b0 <= b_hi; b0 += P) {
          float4 v[P][GW];
#pragma unroll
          for (int p = 0; p < P; ++p) {
            const int b = b0 + p;
            if (b <= b_hi && b != me) {
              const float4* src = reinterpret_cast<const float4*>(partial) +
                                  static_cast<int64_t>(b + jsk) * (HALF / 4) * 256 + et;
#pragma unroll
              for (int g = 0; g < GW; ++g) v[p][g] = __ldcg(src + (g0 + g) * 256);
            }
          }
#pragma unroll
          for (int p = 0; p < P; ++p) {
            const int b = b0 + p;
            if (b > b_hi) break;
            if (b == me) {
#pragma unroll
              for (int t = 0; t < 4 * GW; ++t) sum[t] += acc[4 * g0 + t];
            } else {
#pragma unroll
              for (int g = 0; g < GW; ++g) {
                sum[4 * g] += v[p][g].x;
                sum[4 * g + 1] += v[p][g].y;
                sum[4 * g + 2] += v[p][g].z;
                sum[4 * g + 3] += v[p][g].w;
              }
            }
          }
        }
#pragma unroll
        for (int t = 0; t < 4 * GW; ++t) {
          const int m = m0 + 4 * g0 + t;
          if (m < M) {
            if (OUT_BF16)
              static_cast<uint16_t*>(C)[static_cast<int64_t>(m) * ldc + n] = f32_to_bf16_rn(sum[t]);
            else
              static_cast<float*>(C)[static_cast<int64_t>(m) * ldc + n] = sum[t];
          }
        }
      }
      if (et == 0) {  // ready for the next call
        for (int b = b_lo; b <= b_hi; ++b)
          if (b != me) flags[b + jsk] = 0u;
        counters[jsk] = 0u;
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  if (PAIR)
    cluster_sync();  // neither CTA leaves while its peer may still reach its memory
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, CF::kTmemCols);
  }
}

constexpr int kMinChunksPerRange = 4;  // shortest stream-K range worth a fix-up

int mp_for(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256; }

// The schedule of one problem and the workspace it needs.
struct LowPlan {
  LowSched sched;
  int grid;
  bool pairs;              // clusters of two with the cluster-pair split
  int slots;               // partial-tile slots (stream-K)
  size_t counter_bytes;    // per stream-K tile arrival counters (zero between calls)
  size_t flag_bytes;       // per slot ready flags (zero between calls)
  size_t partial_bytes;    // slots x MP x 128 fp32
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

LowPlan lowm_plan(int64_t M, int64_t N, int64_t K, int sm_count, bool stream_k) {
  const int T = static_cast<int>(N / BN), kc = static_cast<int>(K / BK);
  const long long W = static_cast<long long>(T) * kc;
  const int mp = mp_for(M);
  const int G = static_cast<int>(W < sm_count ? W : sm_count);
  int dp = T, sk = 0;
  if (stream_k && G > 0) {
    dp = (T / G) * G;
    const int L = T - dp;
    const long long skc = static_cast<long long>(L) * kc;
    if (L > 0) {
      // Larger partial tiles cost more to add up, so wide ones are split
      // among fewer CTAs.
      const long long smax = mp <= 64 ? (1ll << 40) : (mp == 128 ? 4 : 2);
      long long s = G;
      if (s > L * smax) s = L * smax;
      const long long by_len = skc / kMinChunksPerRange;
      if (s > (by_len > 0 ? by_len : 1)) s = by_len > 0 ? by_len : 1;
      if (skc % s == 0 && (skc / s) % kc == 0) s = 0;  // whole tiles: nothing to split
      if (s == 0) dp = T;
      sk = static_cast<int>(s);
    }
  }
  LowPlan p{};
  p.sched.n_tiles = T;
  p.sched.kchunks = kc;
  p.sched.dp_tiles = dp;
  p.sched.sk_ctas = sk;
  p.sched.sk_chunks = static_cast<long long>(T - dp) * kc;
  p.sched.pair_tiles = 0;
  // CTAs with whole tiles only take the fix-ups (when there are any)
  p.sched.reducers = (sk > 0 && dp > 0 && G > sk) ? G - sk : 0;
  if (dp == T)
    p.grid = T < sm_count ? T : sm_count;
  else
    p.grid = dp > 0 ? G : sk;
  p.pairs = false;
  const int L = T - dp;
  p.slots = sk > 0 ? sk + L - 1 : 0;
  p.counter_bytes = sk > 0 ? round256(static_cast<size_t>(L) * sizeof(unsigned int)) : 0;
  p.flag_bytes = sk > 0 ? round256(static_cast<size_t>(p.slots) * sizeof(unsigned int)) : 0;
  p.partial_bytes = static_cast<size_t>(p.slots) * mp * BN * sizeof(float);
  return p;
}

// Whole tiles, except that the tiles left after the last whole wave of G =
// 2 * clusters CTAs (or all tiles, when there are at most G / 2 of them) are
// split in K between the two CTAs of a cluster, when that leaves each
// cluster at most one such tile.  Falls back to lowm_plan(..., false).
LowPlan lowm_plan_pairs(int64_t M, int64_t N, int64_t K, int sm_count, int clusters) {
  LowPlan p = lowm_plan(M, N, K, sm_count, false);
  const int T = static_cast<int>(N / BN), kc = static_cast<int>(K / BK);
  const int G = 2 * clusters;
  if (clusters < 1 || kc < 2 || mp_for(M) > 64) return p;
  int dp, L;
  if (T <= clusters) {
    dp = 0;
    L = T;
  } else if (T > G && T % G != 0 && T % G <= clusters) {
    L = T % G;
    dp = T - L;
  } else {
    return p;
  }
  p.sched.dp_tiles = dp;
  p.sched.pair_tiles = L;
  p.sched.sk_ctas = 0;
  p.sched.sk_chunks = 0;
  p.sched.reducers = 0;
  p.grid = dp > 0 ? G : 2 * L;
  p.pairs = true;
  return p;
}

template <int MP, bool OUT_BF16>
cudaError_t launch_lowm(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                        void* C, int64_t ldc, int M, int N, int K, const LowPlan& plan,
                        void* workspace, cudaStream_t stream, const DeviceInfo& dev) {
  using CF = LowCfg<MP>;
  auto kern = gemm_lowm_kernel<MP, OUT_BF16, 0>;
  static std::mutex mu;
  static bool ready[64] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (!ready[dev.device]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(CF::kSmemBytes));
      if (e != cudaSuccess) return e;
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      // the setmaxnreg split assumes this launch register count
      if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
      ready[dev.device] = true;
    }
  }
  CUtensorMap tw, ta;
  if (!make_k_major_map(&tw, B, N, K, BN) || !make_k_major_map(&ta, A, M, K, MP))
    return cudaErrorInvalidValue;
  unsigned int* counters = nullptr;
  unsigned int* flags = nullptr;
  float* partial = nullptr;
  if (plan.sched.sk_ctas > 0) {
    uint8_t* w = static_cast<uint8_t*>(workspace);
    counters = reinterpret_cast<unsigned int*>(w);
    flags = reinterpret_cast<unsigned int*>(w + plan.counter_bytes);
    partial = reinterpret_cast<float*>(w + plan.counter_bytes + plan.flag_bytes);
  }
  return launch_pdl(kern, dim3(plan.grid), dim3(kThreads), CF::kSmemBytes, stream, tw, ta, sA, sB,
                    C, ldc, M, N, K, plan.sched, partial, counters, flags,
                    static_cast<const uint16_t*>(nullptr), int64_t{0});
}

// The cluster-pair variant: clusters of two that fit at once (cached per
// device; 0 when it cannot run), then the launch.
template <int MP, bool OUT_BF16>
cudaError_t lowm_pair_clusters(const DeviceInfo& dev, int* clusters) {
  using CF = LowCfg<MP>;
  auto kern = gemm_lowm_kernel<MP, OUT_BF16, 0, true>;
  static std::mutex mu;
  static int cached[64] = {};
  static bool ready[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev.device]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(CF::kPairSmemBytes));
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (dev.sm_count / 2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = CF::kPairSmemBytes;
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

template <int MP, bool OUT_BF16>
cudaError_t launch_lowm_pair(const uint8_t* A, const float* sA, const uint8_t* B,
                             const float* sB, void* C, int64_t ldc, int M, int N, int K,
                             const LowPlan& plan, cudaStream_t stream) {
  using CF = LowCfg<MP>;
  CUtensorMap tw, ta;
  if (!make_k_major_map(&tw, B, N, K, BN) || !make_k_major_map(&ta, A, M, K, MP))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = CF::kPairSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_lowm_kernel<MP, OUT_BF16, 0, true>, tw, ta, sA, sB, C, ldc,
                            M, N, K, plan.sched, static_cast<float*>(nullptr),
                            static_cast<unsigned int*>(nullptr),
                            static_cast<unsigned int*>(nullptr),
                            static_cast<const uint16_t*>(nullptr), int64_t{0});
}

// Whole tiles with the cluster-pair split of the tail when it applies.
template <int MP, bool OUT_BF16>
cudaError_t launch_lowm_auto(const uint8_t* A, const float* sA, const uint8_t* B,
                             const float* sB, void* C, int64_t ldc, int M, int N, int K,
                             bool pairs_allowed, cudaStream_t stream, const DeviceInfo& dev) {
  int clusters = 0;
  if (pairs_allowed) {
    const cudaError_t e = lowm_pair_clusters<MP, OUT_BF16>(dev, &clusters);
    if (e != cudaSuccess) return e;
  }
  const LowPlan plan = lowm_plan_pairs(M, N, K, dev.sm_count, clusters);
  if (plan.pairs) return launch_lowm_pair<MP, OUT_BF16>(A, sA, B, sB, C, ldc, M, N, K, plan, stream);
  return launch_lowm<MP, OUT_BF16>(A, sA, B, sB, C, ldc, M, N, K, plan, nullptr, stream, dev);
}

// A as bf16, quantized inside the kernel (FUSE = scale mode + 1); whole
// tiles only.
template <int MP, bool OUT_BF16, int FUSE>
cudaError_t launch_lowm_fused(const uint16_t* a16, int64_t lda, const uint8_t* B, const float* sB,
                              void* C, int64_t ldc, int M, int N, int K, cudaStream_t stream,
                              const DeviceInfo& dev) {
  using CF = LowCfg<MP>;
  auto kern = gemm_lowm_kernel<MP, OUT_BF16, FUSE>;
  const size_t smem = CF::fused_smem_bytes(K / BK);
  if (smem > static_cast<size_t>(kMaxSmemOptin)) return cudaErrorInvalidValue;
  static std::mutex mu;
  static bool ready[64] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (!ready[dev.device]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kMaxSmemOptin);
      if (e != cudaSuccess) return e;
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
      ready[dev.device] = true;
    }
  }
  CUtensorMap tw, ta_unused = {};
  if (!make_k_major_map(&tw, B, N, K, BN)) return cudaErrorInvalidValue;
  // The same schedule as the GEMM on quantized activations (launch_lowm_auto
  // with the same cluster count), so that the two give the same bits: the
  // tail split within clusters of two when the receive buffer fits next to
  // the resident activations.
  LowPlan plan = lowm_plan(M, N, K, dev.sm_count, false);
  const size_t pair_smem = smem + 64 + CF::kRecvBytes;
  if (pair_smem <= static_cast<size_t>(kMaxSmemOptin)) {
    int clusters = 0;
    cudaError_t e = lowm_pair_clusters<MP, OUT_BF16>(dev, &clusters);
    if (e != cudaSuccess) return e;
    plan = lowm_plan_pairs(M, N, K, dev.sm_count, clusters);
    if (plan.pairs) {
      auto pkern = gemm_lowm_kernel<MP, OUT_BF16, FUSE, true>;
      static std::mutex pmu;
      static bool pready[64] = {};
      {
        std::lock_guard<std::mutex> lock(pmu);
        if (!pready[dev.device]) {
          e = cudaFuncSetAttribute(pkern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemOptin);
          if (e != cudaSuccess) return e;
          cudaFuncAttributes fa;
          e = cudaFuncGetAttributes(&fa, pkern);
          if (e != cudaSuccess) return e;
          if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
          pready[dev.device] = true;
        }
      }
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[2];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.gridDim = dim3(plan.grid);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = pair_smem;
      cfg.stream = stream;
      cfg.attrs = attr;
      cfg.numAttrs = 2;
      return cudaLaunchKernelEx(&cfg, pkern, tw, ta_unused, static_cast<const float*>(nullptr), sB,
                                C, ldc, M, N, K, plan.sched, static_cast<float*>(nullptr),
                                static_cast<unsigned int*>(nullptr),
                                static_cast<unsigned int*>(nullptr), a16, lda);
    }
  }
  return launch_pdl(kern, dim3(plan.grid), dim3(kThreads), smem, stream, tw, ta_unused,
                    static_cast<const float*>(nullptr), sB, C, ldc, M, N, K, plan.sched,
                    static_cast<float*>(nullptr), static_cast<unsigned int*>(nullptr),
                    static_cast<unsigned int*>(nullptr), a16, lda);
}

template <bool OUT_BF16>
cudaError_t dispatch_mp(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                        void* C, int64_t ldc, int M, int N, int K, const LowPlan& plan,
                        void* workspace, cudaStream_t stream, const DeviceInfo& dev) {
  if (M <= 16)
    return launch_lowm<16, OUT_BF16>(A, sA, B, sB, C, ldc, M, N, K, plan, workspace, stream, dev);
  if (M <= 32)
    return launch_lowm<32, OUT_BF16>(A, sA, B, sB, C, ldc, M, N, K, plan, workspace, stream, dev);
  if (M <= 64)
    return launch_lowm<64, OUT_BF16>(A, sA, B, sB, C, ldc, M, N, K, plan, workspace, stream, dev);
  if (M <= 128)
    return launch_lowm<128, OUT_BF16>(A, sA, B, sB, C, ldc, M, N, K, plan, workspace, stream, dev);
  return launch_lowm<256, OUT_BF16>(A, sA, B, sB, C, ldc, M, N, K, plan, workspace, stream, dev);
}

}  // namespace

size_t lowm_workspace_bytes(int64_t M, int64_t N, int64_t K, int sm_count) {
  const LowPlan p = lowm_plan(M, N, K, sm_count, true);
  if (p.sched.sk_ctas == 0) return 256;  // never touched; a non-empty buffer keeps the contract simple
  return p.counter_bytes + p.flag_bytes + p.partial_bytes;
}

size_t lowm_workspace_zero_bytes(int64_t M, int64_t N, int64_t K, int sm_count) {
  const LowPlan p = lowm_plan(M, N, K, sm_count, true);
  return p.counter_bytes + p.flag_bytes;
}

size_t lowm_fused_smem_bytes(int64_t M, int64_t K) {
  const int kc = static_cast<int>(K / BK);
  return M <= 16 ? LowCfg<16>::fused_smem_bytes(kc) : LowCfg<32>::fused_smem_bytes(kc);
}

bool lowm_fused_fits(int64_t M, int64_t K) {
  return M >= 1 && M <= 32 && K / BK <= 4096 && lowm_fused_smem_bytes(M, K) <= kMaxSmemOptin;
}

// The fused kernel also has room for the cluster-pair receive buffer.
bool lowm_fused_pair_fits(int64_t M, int64_t K) {
  const size_t recv = M <= 16 ? LowCfg<16>::kRecvBytes : LowCfg<32>::kRecvBytes;
  return lowm_fused_fits(M, K) && lowm_fused_smem_bytes(M, K) + 64 + recv <= kMaxSmemOptin;
}

cudaError_t launch_gemm_lowm_fused(const void* a16, int64_t lda, const uint8_t* B, const float* sB,
                                   void* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                   int out_bf16, int mode, cudaStream_t stream,
                                   const DeviceInfo& dev) {
  if (M == 0) return cudaSuccess;
  if (!lowm_fused_fits(M, K)) return cudaErrorInvalidValue;
  const auto* a = static_cast<const uint16_t*>(a16);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  const bool ue = mode != 0;
  if (M <= 16) {
    if (out_bf16)
      return ue ? launch_lowm_fused<16, true, 2>(a, lda, B, sB, C, ldc, m, n, k, stream, dev)
                : launch_lowm_fused<16, true, 1>(a, lda, B, sB, C, ldc, m, n, k, stream, dev);
    return ue ? launch_lowm_fused<16, false, 2>(a, lda, B, sB, C, ldc, m, n, k, stream, dev)
              : launch_lowm_fused<16, false, 1>(a, lda, B, sB, C, ldc, m, n, k, stream, dev);
  }
  if (out_bf16)
    return ue ? launch_lowm_fused<32, true, 2>(a, lda, B, sB, C, ldc, m, n, k, stream, dev)
              : launch_lowm_fused<32, true, 1>(a, lda, B, sB, C, ldc, m, n, k, stream, dev);
  return ue ? launch_lowm_fused<32, false, 2>(a, lda, B, sB, C, ldc, m, n, k, stream, dev)
            : launch_lowm_fused<32, false, 1>(a, lda, B, sB, C, ldc, m, n, k, stream, dev);
}

cudaError_t launch_gemm_lowm(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                             void* C, int64_t ldc, int64_t M, int64_t N, int64_t K, int out_bf16,
                             bool stream_k, void* workspace, cudaStream_t stream,
                             const DeviceInfo& dev) {
  if (M == 0) return cudaSuccess;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  if (!stream_k && M <= 64) {
    // No workspace: whole tiles, the tail split within clusters of two.
    // For M <= 32 the split is taken only where the GEMM that quantizes its
    // activations itself can take it too, so that both give the same bits.
    const bool pairs = M > 32 || !lowm_fused_fits(M, K) || lowm_fused_pair_fits(M, K);
    if (M <= 16)
      return out_bf16 ? launch_lowm_auto<16, true>(A, sA, B, sB, C, ldc, m, n, k, pairs, stream, dev)
                      : launch_lowm_auto<16, false>(A, sA, B, sB, C, ldc, m, n, k, pairs, stream, dev);
    if (M <= 32)
      return out_bf16 ? launch_lowm_auto<32, true>(A, sA, B, sB, C, ldc, m, n, k, pairs, stream, dev)
                      : launch_lowm_auto<32, false>(A, sA, B, sB, C, ldc, m, n, k, pairs, stream, dev);
    return out_bf16 ? launch_lowm_auto<64, true>(A, sA, B, sB, C, ldc, m, n, k, pairs, stream, dev)
                    : launch_lowm_auto<64, false>(A, sA, B, sB, C, ldc, m, n, k, pairs, stream, dev);
  }
  const LowPlan plan = lowm_plan(M, N, K, dev.sm_count, stream_k);
  if (plan.sched.sk_ctas > 0 && workspace == nullptr) return cudaErrorInvalidValue;
  return out_bf16 ? dispatch_mp<true>(A, sA, B, sB, C, ldc, m, n, k, plan, workspace, stream, dev)
                  : dispatch_mp<false>(A, sA, B, sB, C, ldc, m, n, k, plan, workspace, stream, dev);
}

}  // namespace fgq

// ---- split-K over a fixed scratch array (no allocation) -----------------------
//
// For callers that cannot allocate device memory at all: code inside
// another allocator or a memory-pool callback, hosts that hand out a fixed
// device-memory budget up front, or embedders with no allocator of their
// own.  The split-K workspace then lives in this file-scope array: every
// GPU that loads the library holds it until the process exits, and every
// call shares it.
namespace fgq {
namespace {

static __device__ __align__(256) unsigned char g_splitk_scratch[FGQ_NOALLOC_SCRATCH_BYTES];

}  // namespace

// Unique id of the current context (cuCtxGetId), so that a cached symbol
// address is looked up again once the context it came from is gone (after
// cudaDeviceReset the module is loaded again and may sit elsewhere).
cudaError_t current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  if (get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

cudaError_t noalloc_scratch(const DeviceInfo& dev, void** ptr) {
  // The array's name in host code is only a host-side stand-in for the
  // symbol, so its device address is looked up with the device current
  // (the caller made it current): once per device, and again whenever the
  // device's context has changed since (a device reset).
  static std::mutex mu;
  static void* addr[64] = {};
  static unsigned long long ctx_of[64] = {};
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  unsigned long long ctx = 0;
  cudaError_t e = current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev.device] == nullptr || ctx_of[dev.device] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_splitk_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    addr[dev.device] = p;
    ctx_of[dev.device] = ctx;
  }
  *ptr = addr[dev.device];
  return cudaSuccess;
}

}  // namespace fgq

namespace fgq {

cudaError_t read_device_error_lowm(uint32_t* word, bool clear) {
  return read_unit_device_error(word, clear);
}

}  // namespace fgq
