// Device-side helpers for the sm_103a kernels: inline PTX for mbarriers,
// TMA (cp.async.bulk.tensor), tcgen05 (TMEM alloc, MMA, commit, loads) and
// the bounded waits every spin loop uses.
//
// Every wait here gives up after FGQ_WAIT_NS nanoseconds of %globaltimer
// time: it records the site in the library's device error word and returns
// false, so a kernel can unwind (release TMEM, return) instead of hanging.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fgq_internal.h"

namespace fgq {

// Device error word.  Zero while nothing has gone wrong; kernels OR in
// FGQ_DEVERR_* bits.  Each translation unit that includes this header has
// its own copy; the C ABI reports the OR of the kernel units' copies.
static __device__ unsigned int g_device_error = 0;

constexpr unsigned long long FGQ_WAIT_NS = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_error(unsigned int bits) {
  atomicOr(&g_device_error, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool elect_one_sync() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Named barrier `id` over `nthreads` threads (whole warps).
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ANDs a predicate over its threads: every thread
// gets the same result.
__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ---- programmatic dependent launch -----------------------------------------------

// Wait until the kernels this grid depends on (the previous kernel in the
// stream, when launched with launch_pdl) have completed and their memory
// is visible.  No-op when the launch had no programmatic dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let the next kernel in the stream (if launched with launch_pdl) start its
// set-up now; it still waits in pdl_wait() for this grid to complete.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic stream serialization: the kernel may begin
// before the previous kernel in the stream has finished, and must call
// pdl_wait() before it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Relaxed arrive: orders nothing else.  Used to hand a TMEM buffer back
// after tcgen05.wait::ld, when every read of it has already completed.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed.  Returns false
// (after recording `site`) when the wait times out or when *abort is set by
// another warp of the CTA that already gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort, unsigned int site) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > FGQ_WAIT_NS) {
        record_error(site);
        *abort = 1;
        return false;
      }
    }
  }
}

// The same bounded wait with acquire semantics at cluster scope: for a
// barrier that CTAs of the cluster arrive on with release.cluster after
// writing this CTA's shared memory.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, unsigned int site) {
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((it & 63u) == 63u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > FGQ_WAIT_NS) {
        record_error(site);
        *abort = 1;
        return false;
      }
    }
  }
}

// ---- TMA ---------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled bulk tensor copy global -> shared, completing on `bar`.
// c0 is the innermost (contiguous) coordinate in elements, c1 the row.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// 2-CTA form: the copy lands in this CTA's shared memory and completes on
// the barrier at shared::cluster address `bar_cluster`, which may belong to
// the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const void* tmap,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

// ---- clusters ------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// Arrive on a barrier given by its shared::cluster address (any CTA of the
// cluster), release semantics at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

// Relaxed arrive on a barrier of any CTA of the cluster: orders nothing
// else.  Used to hand a TMEM buffer back to the peer's MMA issuer after
// tcgen05.wait::ld, when every read of it has already completed (a release
// here would also wait for the warp's outstanding global stores).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

// Every thread of every CTA in the cluster arrives, then waits for all.
// Both CTAs of a pair run the same code to this point (a cluster is
// scheduled as a whole), so the wait ends.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// ---- tcgen05 -------------------------------------------------------------------

// TMEM allocation spanning both CTAs of a pair: one warp in each CTA
// executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4, issued by the even CTA of
// a pair: A's rows and B's rows are split between the two CTAs' shared
// memory at the same offsets, and each CTA's TMEM receives its own 128 rows
// of D.
__device__ __forceinline__ void umma_f8f6f4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2-CTA commit: arrive once on the barrier at `bar`'s offset in every CTA
// of cta_mask when every tcgen05 op issued so far by this thread has
// completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4, one CTA.
__device__ __forceinline__ void umma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= (A * 2^sfa) * (B * 2^sfb)^T, kind::mxf8f6f4 with UE8M0 scale
// factors read from TMEM (scale_vec::1X: one factor per row of A and per
// column of B for the instruction's K = 32).  Measured layout on sm_103a
// for M = 128: the factor of A's row m is at lane m, column sfa_col + m/32;
// the factor of B's column n is at lane 32*q + n%32, column sfb_col + n/32,
// where q is the TMEM lane quarter of the D row being computed, so B's
// factors are replicated in all four quarters.  idesc bits 29-30 / 4-5
// select which byte of those 32-bit cells holds A's / B's factor.
__device__ __forceinline__ void umma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem,
                                              uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Store one 32-bit value per lane into column taddr.col of the warp's 32
// TMEM lanes (lane taddr.lane + thread).
__device__ __forceinline__ void tmem_st_32x32b_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v)
               : "memory");
}

// Store four consecutive columns: a, a, a, a then b, b, b, b in the next four.
__device__ __forceinline__ void tmem_st_32x32b_x8_aabb(uint32_t taddr, uint32_t a, uint32_t b) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %1, %1, %1, %2, %2, %2, %2};" ::"r"(
                   taddr),
               "r"(a), "r"(b)
               : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, uint32_t a) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %1, %1, %1};" ::"r"(taddr), "r"(a)
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrive (once) on `bar` when every tcgen05 op issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Wait for outstanding TMEM loads, tying the 32 destination registers to
// the wait so that no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
        "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
        "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
        "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
        "+r"(r[31])
      :
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread t of the warp receives
// lane (taddr.lane + t), columns taddr.col .. +15.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
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

// Register budget changes (all warps of a warpgroup execute these).
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// acc (packed fp32 pair) += p (packed pair) * scale (packed pair), one
// rounding per lane.  volatile keeps it ordered against TMEM loads/waits.
__device__ __forceinline__ uint64_t ffma2_acc(uint64_t p, uint64_t scale, uint64_t acc) {
  uint64_t d;
  asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(p), "l"(scale), "l"(acc));
  return d;
}

__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Shared-memory matrix descriptor for a K-major operand stored in the
// 128-byte-swizzled canonical layout that a TMA SWIZZLE_128B load writes:
// rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked along M/N.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4 (unused for swizzled
//               K-major; set to 1)
//   bits 32-45  stride-dimension byte offset >> 4 (1024 bytes between atoms)
//   bits 46-47  descriptor version, 1 on this architecture
//   bits 49-51  base offset (0: atoms are 1024-byte aligned)
//   bits 61-63  swizzle mode, 2 = 128-byte swizzle
// Descriptor from its two 32-bit words.  Shared memory is below 256 KB, so
// the descriptor of an operand tile at byte offset d from another is that
// descriptor with d >> 4 added to its low word (the start field never
// carries into the next field).
__device__ __forceinline__ uint64_t make_desc(uint32_t lo, uint32_t hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
  return d;
}

__device__ __forceinline__ uint64_t smem_desc_k_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor, kind::f8f6f4, dense: D fp32, A and B E4M3, both
// K-major, shape M x N (x K = 32).
//   bits 4-5  D format (1 = f32); bits 7-9 / 10-12 A / B format (0 = E4M3);
//   bit 15 / 16 A / B major (0 = K); bits 17-22 N >> 3; bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// Instruction descriptor, kind::mxf8f6f4 (D fp32 implied), A and B E4M3,
// both K-major, UE8M0 scale factors (bit 23), scale-factor byte 0 for A
// (bits 29-30) and B (bits 4-5); OR in (id << 29) | (id << 4) to select
// byte id of the scale-factor cells.
__host__ __device__ constexpr uint32_t idesc_mx_e4m3_ue8m0(int m, int n) {
  return (0u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// ---- coalesced row stores ----------------------------------------------------------

// A warp's output rows, one per lane (lane l holds RB bytes of row l as RB/4
// 32-bit words in column order), stored to global memory so that each store
// instruction writes whole contiguous row segments instead of 16 bytes of
// 32 different rows.  The rows pass through `stage`, an SB-byte per-warp
// shared-memory buffer (16-byte aligned): in each round RR = SB / RB lanes
// write their rows into it (16-byte units XOR-swizzled by the row so the
// writes do not collide in a bank), then all 32 lanes read it back in
// row-major order and store 16 bytes at a time.  Row l goes to
// row0 + l * stride; only rows l < rows are stored.  Every lane of the warp
// must call it.
template <int RB, int SB = 2048>
__device__ __forceinline__ void warp_store_rows(uint8_t* stage, const uint32_t (&words)[RB / 4],
                                                uint8_t* row0, int64_t stride, int rows) {
  static_assert(RB % 64 == 0 && RB <= SB && (SB == 1024 || SB == 2048), "row and stage bytes");
  constexpr int RU = RB / 16;          // 16-byte units per row
  constexpr int RR = SB / RB;          // rows per round
  constexpr int NL = SB / 512;         // 16-byte loads per lane per round
  constexpr int SW = RU < 8 ? RU - 1 : 7;
  static_assert(32 % RR == 0, "rounds");
  const int lane = threadIdx.x & 31;
  const uint32_t st0 = smem_u32(stage);
#pragma unroll
  for (int k = 0; k < 32 / RR; ++k) {
    if (lane / RR == k) {
      const int rl = lane % RR;
#pragma unroll
      for (int u = 0; u < RU; ++u)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         st0 + rl * RB + ((u ^ (rl & SW)) * 16)),
                     "r"(words[4 * u]), "r"(words[4 * u + 1]), "r"(words[4 * u + 2]),
                     "r"(words[4 * u + 3])
                     : "memory");
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < NL; ++j) {
      const int q = lane + 32 * j;
      const int rl = q / RU, u = q % RU;
      uint4 v;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(st0 + rl * RB + ((u ^ (rl & SW)) * 16))
                   : "memory");
      const int r = k * RR + rl;
      if (r < rows) *reinterpret_cast<uint4*>(row0 + r * stride + u * 16) = v;
    }
    __syncwarp();
  }
}

// One 32-byte store (a whole sector) of eight 32-bit words; dst 32-byte
// aligned.
__device__ __forceinline__ void st_global_32B(void* dst, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Two fp32 -> packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 32 accumulator columns of the warp's 32 rows (lane = row; r holds fp32
// bits), converted (bf16 rounds to nearest even) and stored through the
// warp's staging buffer: rows row0 .. row0 + 31 (those below row0 + rows),
// columns col .. col + 31 of C (leading dimension ldc elements).
template <bool OUT_BF16, int SB = 2048>
__device__ __forceinline__ void warp_store32(uint8_t* stage, const uint32_t (&r)[32], void* C,
                                             int64_t ldc, int row0, int col, int rows) {
  if (OUT_BF16) {
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = cvt_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
    warp_store_rows<64, SB>(stage, w,
                            reinterpret_cast<uint8_t*>(static_cast<uint16_t*>(C) +
                                                       static_cast<int64_t>(row0) * ldc + col),
                            ldc * 2, rows);
  } else {
    warp_store_rows<128, SB>(stage, r,
                             reinterpret_cast<uint8_t*>(static_cast<float*>(C) +
                                                        static_cast<int64_t>(row0) * ldc + col),
                             ldc * 4, rows);
  }
}

// Read (and optionally clear) this translation unit's copy of the device
// error word.  Each unit with kernels that record errors exports a wrapper
// around this; the C ABI reports the OR of all of them.
static inline cudaError_t read_unit_device_error(uint32_t* word, bool clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
  if (e != cudaSuccess) return e;
  if (clear && v != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *word = v;
  return cudaSuccess;
}

// ---- numeric conversions ------------------------------------------------------

// Two fp32 -> two E4M3 codes, round to nearest even, saturating to +-448.
// Returns lo's code in bits 0-7 and hi's code in bits 8-15.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace fgq
