/*
 * fgq — fine-grained FP8 quantization and block-scaled FP8 GEMM on GB300
 * (sm_103a).  C ABI of libfgq.so.
 *
 * The method ("Fine-Grained FP8/FP4 Quantization", KernelWiki technique page):
 *   - §Scaling Granularities: activations carry one scale per 1x128 tile
 *     (one row, 128 consecutive K elements); weights carry one scale per
 *     128x128 block.
 *   - §DeepGEMM: Tile-wise and Block-wise Scaling: A and B are E4M3; the
 *     scale tensors are scale_A [M, K/128] and scale_B [K/128, N/128]; for
 *     each 128-wide K chunk the product of the FP8 tiles is multiplied by
 *     scale_A * scale_B and added into an fp32 accumulator:
 *       C[m,n] = sum_c  sA[m,c] * sB[c, n/128] * sum_{k in chunk c} Aq[m,k] Bq[k,n]
 *   - §UE8M0 vs E4M3 Scale Formats, §Blackwell: Native Block Scaling: a
 *     UE8M0 scale is a power of two 2^(e-127).
 *
 * Readings of the page fixed by this library:
 *   scale   fp32 mode:  s = amax / 448 rounded once to fp32 (448 = largest
 *           finite E4M3 value); UE8M0 mode: the smallest power of two
 *           >= that value, exponent clamped to [-127, 127].  A group whose
 *           amax is 0 gets s = 1.
 *   encode  q = E4M3(x / s): one IEEE fp32 division, then round to nearest
 *           with ties to even, magnitudes above 448 saturate to 448, sign
 *           kept (a negative value that rounds to zero gives 0x80).
 *   inputs  finite bf16 values; non-finite inputs give unspecified codes.
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers into memory the caller owns
 *     (cudaMalloc / torch allocations).  The library never allocates,
 *     frees or retains them, and never allocates device memory itself.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream and never
 *     synchronise the host.
 *   - Sizes are element counts; leading dimensions are in elements of the
 *     array they describe.
 *   - Arguments are checked before anything is launched; a rejected call
 *     returns FGQ_ERR_INVALID_ARG (or FGQ_ERR_UNSUPPORTED) and touches no
 *     memory.  A failed launch returns FGQ_ERR_CUDA.
 *   - M == 0 (or N == 0) is a valid empty problem: nothing is launched.
 */
#ifndef FGQ_H_
#define FGQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FGQ_OK = 0,
  FGQ_ERR_INVALID_ARG = 1,   /* null pointer, bad size, stride or alignment */
  FGQ_ERR_UNSUPPORTED = 2,   /* no device of a supported architecture */
  FGQ_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  FGQ_ERR_DEVICE_TIMEOUT = 4 /* a kernel gave up on a wait (see fgq_device_error) */
} fgq_status;

typedef enum { FGQ_SCALE_FP32 = 0, FGQ_SCALE_UE8M0 = 1 } fgq_scale_mode;
typedef enum { FGQ_OUT_F32 = 0, FGQ_OUT_BF16 = 1 } fgq_out_dtype;

/*
 * 1x128 tile-wise activation quantization (§Scaling Granularities,
 * per-tile 1x128; scale_A [M, K/128] from §DeepGEMM).
 *
 *   x    bf16 [M, K], row r at x + r * ldx (ldx >= K, ldx % 8 == 0),
 *        16-byte aligned.
 *   xq   E4M3 codes [M, K], row r at xq + r * ldq (ldq >= K,
 *        ldq % 16 == 0), 16-byte aligned.
 *   sx   fp32 [M, K/128] row-major (dense), 4-byte aligned.
 *   K % 128 == 0, K > 0, M >= 0.  mode: FGQ_SCALE_FP32 or FGQ_SCALE_UE8M0.
 * Per (row, group): amax over the 128 values, s from amax, q = E4M3(x/s).
 */
fgq_status fgq_quant_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                               int64_t ldq, float* sx, int mode, void* stream);

/*
 * 128x1 (transposed) activation quantization, for a weight-gradient GEMM
 * that reduces over the rows of X: groups of 128 consecutive rows of one
 * column -- the plainest extension of the 1x128 tiles of §Scaling
 * Granularities -- written in the layout fgq_gemm_fp8_blockscaled takes for
 * its A operand.  The result equals fgq_quant_act_1x128 applied to X^T.
 *
 *   x     bf16 [M, K], row m at x + m * ldx (ldx >= K, ldx % 8 == 0),
 *         16-byte aligned.
 *   xqt   E4M3 codes [K, M] row-major (dense): the code of X[m, k] at
 *         xqt[k * M + m].  16-byte aligned.
 *   sxt   fp32 [K, M/128] row-major (dense): the scale of rows
 *         128 g .. 128 g + 127 of column k at sxt[k * (M/128) + g].
 *   M % 128 == 0, K % 128 == 0, K > 0, M >= 0.  mode: FGQ_SCALE_FP32 or
 *   FGQ_SCALE_UE8M0.  Scale and encode as fgq_quant_act_1x128.
 */
fgq_status fgq_quant_act_128x1(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xqt,
                               float* sxt, int mode, void* stream);

/*
 * MXFP4 quantization (§UE8M0 vs E4M3 Scale Formats: UE8M0 scales, block
 * size 32; E2M1 values 0, 0.5, 1, 1.5, 2, 3, 4, 6 from §NVFP4 Two-Level
 * Scaling): one UE8M0 scale per 32 consecutive elements of each row.  For
 * a GEMM both operands are quantized this way along K (the weight as its
 * transpose [N, K]).
 *
 *   x    bf16 [R, K], row r at x + r * ldx (ldx >= K, ldx % 8 == 0),
 *        16-byte aligned.
 *   xq   E2M1 codes [R, K/2] bytes, row-major (dense), 4-byte aligned:
 *        element 2j of a row in the low nibble of byte j, element 2j+1 in
 *        the high nibble; code bit 3 = sign.
 *   sx   UE8M0 codes [R, K/32] bytes, row-major (dense): the scale of
 *        elements 32 g .. 32 g + 31 of row r is 2^(sx[r * K/32 + g] - 127).
 *   K % 32 == 0, K > 0, R >= 0.
 * Scale: the smallest power of two >= amax / 6 (exponent clamped at -127;
 * a zero group gets 1); each element becomes E2M1(x / s), round to nearest
 * with ties to even (x / s is exact; no element exceeds 6).
 */
fgq_status fgq_quant_mxfp4_1x32(const void* x, int64_t R, int64_t K, int64_t ldx, uint8_t* xq,
                                uint8_t* sx, void* stream);

/*
 * 128x128 block-wise weight quantization (§Scaling Granularities,
 * per-block 128x128; scale_B [K/128, N/128] from §DeepGEMM).
 *
 *   w    bf16 [K, N] (the logical weight, K = reduction dimension), row k
 *        at w + k * ldw (ldw >= N, ldw % 8 == 0), 16-byte aligned.
 *   wq   E4M3 codes stored TRANSPOSED, [N, K] row-major (dense): code of
 *        logical element (k, n) at wq[n * K + k].  This K-major layout is
 *        the operand layout of fgq_gemm_fp8_blockscaled.  16-byte aligned.
 *   sw   fp32 [K/128, N/128] row-major (dense).
 *   K % 128 == 0, N % 128 == 0, both > 0.
 * Per 128x128 block: amax over 16384 values, s from amax, q = E4M3(w/s).
 */
fgq_status fgq_quant_w_128x128(const void* w, int64_t K, int64_t N, int64_t ldw, uint8_t* wq,
                               float* sw, int mode, void* stream);

/*
 * Both operands of one block-scaled GEMM in one launch: the activations X
 * [M, K] in 1x128 groups (exactly as fgq_quant_act_1x128) and the weight W
 * [K, N] in 128x128 blocks (exactly as fgq_quant_w_128x128), one scale
 * mode for both ("Fine-Grained FP8/FP4 Quantization", §Scaling
 * Granularities; scale shapes from §DeepGEMM).  The codes and scales are
 * bit for bit those of the two separate calls; one kernel does both, so the
 * second launch's fill and drain are saved.
 *
 *   x, ldx, xq, ldq, sx   as fgq_quant_act_1x128 (unused when M == 0).
 *   w, ldw, wq, sw        as fgq_quant_w_128x128 (W [K, N], codes [N, K]).
 *   K % 128 == 0, N % 128 == 0, K > 0, N > 0, M >= 0.
 * The same argument checks as the two calls, all before any launch.
 */
fgq_status fgq_quant_operands(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                              int64_t ldq, float* sx, const void* w, int64_t N, int64_t ldw,
                              uint8_t* wq, float* sw, int mode, void* stream);

/*
 * Block-scaled FP8 GEMM (§DeepGEMM: Tile-wise and Block-wise Scaling),
 * fp32 output, fp32 scales:
 *   C[m,n] = sum_c sA[m,c] * sB[c,n/128] * sum_{k in chunk c} A[m,k] * B[k,n]
 *
 *   A    E4M3 [M, K] row-major (dense, as fgq_quant_act_1x128 writes with
 *        ldq = K), 16-byte aligned.
 *   sA   fp32 [M, K/128] row-major.
 *   B    E4M3 weight codes in the transposed [N, K] layout written by
 *        fgq_quant_w_128x128, 16-byte aligned.
 *   sB   fp32 [K/128, N/128] row-major.
 *   C    fp32 [M, N] row-major (dense), 16-byte aligned.
 *   K % 128 == 0, N % 128 == 0, K > 0, N > 0, M >= 0; M need not be a
 *   multiple of anything.
 * Each 128-wide K chunk is one tensor-core partial product in TMEM, which is
 * scaled by sA * sB and added into an fp32 accumulator (the page's
 * promotion step, done by the epilogue warps).  For M <= 32 the operands
 * are swapped so the tensor core's 128-row side runs over the weight, and
 * the 128-column tiles of C left after the last whole wave over the SMs
 * (all of them, when there are at most one per pair of SMs) are split in
 * two halves of K between the two CTAs of a cluster, the halves added
 * through distributed shared memory in a fixed order (deterministic, no
 * workspace).  Results for M <= 32 are the same bits as
 * fgq_gemm_fp8_blockscaled_fused_act on the unquantized activations.
 */
fgq_status fgq_gemm_fp8_blockscaled(const uint8_t* A, const float* sA, const uint8_t* B,
                                    const float* sB, float* C, int64_t M, int64_t N,
                                    int64_t K, void* stream);

/*
 * Same GEMM with an output type, an output leading dimension and a scale
 * mode.
 *   C      fp32 or bf16 [M, N], row m at C + m * ldc (ldc >= N; ldc % 4 == 0
 *          for fp32, ldc % 8 == 0 for bf16), 16-byte aligned.  bf16 output
 *          is the fp32 accumulator rounded to nearest even.
 *   out    FGQ_OUT_F32 or FGQ_OUT_BF16.
 *   mode   FGQ_SCALE_FP32: any positive finite scales.
 *          FGQ_SCALE_UE8M0: the caller promises every scale is a power of
 *          two (as the quantizers write in UE8M0 mode); results are the
 *          same formula.
 */
fgq_status fgq_gemm_fp8_blockscaled_ex(const uint8_t* A, const float* sA, const uint8_t* B,
                                       const float* sB, void* C, int64_t ldc, int64_t M,
                                       int64_t N, int64_t K, int out, int mode, void* stream);

/*
 * Block-scaled FP8 GEMM with stream-K scheduling for few rows of A, using a
 * caller-owned workspace ("Persistent kernel" page, §Scheduler: stream-K).
 * Same arguments and result as fgq_gemm_fp8_blockscaled_ex.
 *
 * For M <= 256: whole waves of 128-column tiles of C run one tile per SM;
 * the K chunks of the tiles left over after the last whole wave are laid
 * end to end and cut into equal contiguous ranges, one per SM, so every SM
 * streams about the same share of the weight.  A range that covers part of
 * a tile leaves an fp32 partial tile; the last CTA of that tile to finish
 * adds the partials in a fixed order (that of the ranges) and writes C, so
 * results are deterministic and identical across calls.  For M > 256 this
 * is fgq_gemm_fp8_blockscaled_ex and the workspace is not touched.
 *
 *   workspace        device memory of at least the size that
 *                    fgq_gemm_splitk_workspace_size returns for (M, N, K) on
 *                    the current device, 16-byte aligned, owned by the
 *                    caller.  It must be zero-filled before its first use;
 *                    every call that returns FGQ_OK leaves it ready for the
 *                    next (its per-tile counters and flags back at zero).  After a
 *                    call whose kernel gave up on a wait
 *                    (FGQ_ERR_DEVICE_TIMEOUT from fgq_device_error) zero it
 *                    again.  Calls that share a workspace must not overlap
 *                    on the GPU.
 *   workspace_bytes  its size; a smaller size than required returns
 *                    FGQ_ERR_INVALID_ARG.
 */
fgq_status fgq_gemm_fp8_blockscaled_splitk(const uint8_t* A, const float* sA, const uint8_t* B,
                                           const float* sB, void* C, int64_t ldc, int64_t M,
                                           int64_t N, int64_t K, int out, int mode,
                                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Block-scaled FP8 GEMM whose activations come as bf16 and are quantized
 * inside the GEMM: the quantize -> GEMM fusion the page lists for DeepGEMM
 * (the Xq round trip through memory is dropped), for few rows of A (the
 * decode regime).
 *
 * Same result as fgq_quant_act_1x128(A) followed by
 * fgq_gemm_fp8_blockscaled_ex on its codes and scales: every CTA quantizes
 * all of A (1x128 groups, scale mode `mode`, the same arithmetic as the
 * quantizer) into its shared memory and keeps it there, while the weight
 * streams through.  The codes and scales of A are not written to memory.
 *
 *   A      bf16 [M, K], row m at A + m * lda (lda >= K, lda % 8 == 0),
 *          16-byte aligned.
 *   B, sB  as fgq_gemm_fp8_blockscaled_ex (weight codes [N, K], scales
 *          [K/128, N/128]); for FGQ_SCALE_UE8M0, sB must hold powers of two.
 *   C      fp32 or bf16 [M, N], row m at C + m * ldc (as _ex).
 *   1 <= M <= 32 (M == 0 is an empty problem), and A must fit in shared
 *   memory next to the weight pipeline: M <= 16 allows K up to 7936,
 *   17 <= M <= 32 up to 3968 (K % 128 == 0).  Larger problems return
 *   FGQ_ERR_INVALID_ARG; use the quantizer and the GEMM separately.
 */
fgq_status fgq_gemm_fp8_blockscaled_fused_act(const void* A, int64_t lda, const uint8_t* B,
                                              const float* sB, void* C, int64_t ldc, int64_t M,
                                              int64_t N, int64_t K, int out, int mode,
                                              void* stream);

/*
 * MXFP4 GEMM (§UE8M0 vs E4M3 Scale Formats: UE8M0 scales, block 32; §When to
 * Use: MXFP4 for native hardware acceleration): both operands quantized by
 * fgq_quant_mxfp4_1x32 along K, the weight as its transpose,
 *   C[m,n] = sum_k e2m1(A[m,k]) 2^(sA[m,k/32]-127) e2m1(B[n,k]) 2^(sB[n,k/32]-127)
 * with the factors applied by the tensor core (block-scaled FP4 MMA) and an
 * fp32 accumulator.
 *
 *   A    E2M1 codes [M, K/2] bytes (layout of fgq_quant_mxfp4_1x32),
 *        16-byte aligned.       sA  UE8M0 codes [M, K/32], 4-byte aligned.
 *   B    E2M1 codes [N, K/2] bytes, 16-byte aligned.
 *                               sB  UE8M0 codes [N, K/32], 4-byte aligned.
 *   C    fp32 or bf16 [M, N], row m at C + m * ldc (as _ex).
 *   K % 128 == 0, N % 128 == 0, K > 0, N > 0, M >= 0.
 */
fgq_status fgq_gemm_mxfp4(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                          const uint8_t* sB, void* C, int64_t ldc, int64_t M, int64_t N,
                          int64_t K, int out, void* stream);

/*
 * NVFP4 per-tensor (global) scale (§NVFP4 Two-Level Scaling: a value is
 * global_scale * block_scale * e2m1).  The page gives no encoder; this
 * library's: g = amax / 2688 over the whole tensor (2688 = 6 * 448, the
 * largest E2M1 value times the largest E4M3 value, as the FP8 rule
 * amax / 448 at both levels), 1 for an all-zero tensor; IEEE fp32 division.
 *
 *   x    bf16 [R, K], row r at x + r * ldx (ldx >= K, ldx % 8 == 0),
 *        16-byte aligned.  K % 16 == 0, K > 0, R >= 0 (R == 0 gives 1).
 *   g    one fp32 in device memory, 4-byte aligned: written with the scale
 *        (used as scratch for the running maximum until then).
 * Finite inputs are a precondition.  Asynchronous on `stream`.
 */
fgq_status fgq_nvfp4_global_scale(const void* x, int64_t R, int64_t K, int64_t ldx, float* g,
                                  void* stream);

/*
 * NVFP4 quantization (§NVFP4 Two-Level Scaling): one E4M3 block scale per 16
 * consecutive elements of each row, under the per-tensor scale g from
 * fgq_nvfp4_global_scale (or any positive finite fp32 the caller chooses).
 * For a GEMM both operands are quantized this way along K (the weight as
 * its transpose [N, K]).
 *
 *   x    bf16 [R, K], row r at x + r * ldx (ldx >= K, ldx % 8 == 0),
 *        16-byte aligned.
 *   g    device pointer to the fp32 global scale, 4-byte aligned.
 *   xq   E2M1 codes [R, K/2] bytes, row-major (dense), 4-byte aligned:
 *        element 2j of a row in the low nibble of byte j; code bit 3 = sign.
 *   sx   E4M3 block-scale codes [R, K/16] bytes, row-major (dense).
 *   K % 16 == 0, K > 0, R >= 0.
 * Per block: s = E4M3(amax_b / (6 g)) (round to nearest even, saturating
 * at 448); D = g * s in fp32; each element becomes E2M1(x / D), round to
 * nearest even, saturating at 6; a block with D == 0 gets signed zeros.
 * Every quotient is the IEEE fp32 quotient, so codes are exact functions of
 * the inputs.  Dequantization: g * e4m3(s) * e2m1(q).
 */
fgq_status fgq_quant_nvfp4_1x16(const void* x, int64_t R, int64_t K, int64_t ldx, const float* g,
                                uint8_t* xq, uint8_t* sx, void* stream);

/*
 * NVFP4 GEMM (§NVFP4 Two-Level Scaling; §When to Use: NVFP4 with E4M3 block
 * scales for FP4 inference): both operands quantized by
 * fgq_quant_nvfp4_1x16 along K, the weight as its transpose,
 *   C[m,n] = gA gB sum_k e2m1(A[m,k]) e4m3(sA[m,k/16]) e2m1(B[n,k]) e4m3(sB[n,k/16])
 * with the block factors applied by the tensor core (block-scaled FP4 MMA
 * with E4M3 factors) into an fp32 accumulator, times gA gB (fp32) in the
 * epilogue.
 *
 *   A    E2M1 codes [M, K/2] bytes, 16-byte aligned.   sA  E4M3 codes [M, K/16], 4-byte aligned.
 *   B    E2M1 codes [N, K/2] bytes, 16-byte aligned.   sB  E4M3 codes [N, K/16], 4-byte aligned.
 *   gA, gB  device pointers to the two fp32 global scales, 4-byte aligned.
 *   C    fp32 or bf16 [M, N], row m at C + m * ldc (as _ex).
 *   K % 128 == 0, N % 128 == 0, K > 0, N > 0, M >= 0.
 */
fgq_status fgq_gemm_nvfp4(const uint8_t* A, const uint8_t* sA, const float* gA,
                          const uint8_t* B, const uint8_t* sB, const float* gB, void* C,
                          int64_t ldc, int64_t M, int64_t N, int64_t K, int out, void* stream);

/*
 * Tiled FP4 block-scale layout.  The FP4 GEMMs below with the _tiled suffix
 * take their block scales in this layout, which the tensor-map engine loads
 * without gathering; it is this library's storage format (the page gives
 * none).  For R rows of F factor bytes (F = K/32 for MXFP4, K/16 for NVFP4,
 * F % 4 == 0) the code of row r, factor f sits at byte
 *     ((r / 128) * (F / 4) + f / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + f % 4
 * of a buffer of ceil(R / 128) * 128 * F bytes: 512-byte tiles of 128 rows x
 * 4 factor bytes, each the 32-row x 16-byte tile the tensor core's factor
 * copy spreads over a 128-row TMEM tile (row m at lane m, column m / 32;
 * "Fine-Grained FP8/FP4 Quantization", §Blackwell: Native Block Scaling).
 * The bytes of rows R .. up to the next multiple of 128 are padding: the
 * calls below fill them (with the codes of zero rows, or zeros), and they
 * reach no stored output.
 *
 * fgq_fp4_scale_tiles_bytes: that buffer size.  F % 4 == 0, F > 0, R >= 0.
 * fgq_fp4_scales_to_tiles: row-major codes s [R, F] (4-byte aligned) into
 *   the tiled layout at `tiles` (4-byte aligned, the size above; padding
 *   written as zeros); device buffers, asynchronous on `stream`.  A pure
 *   permutation of the codes.
 */
fgq_status fgq_fp4_scale_tiles_bytes(int64_t R, int64_t F, size_t* bytes);
fgq_status fgq_fp4_scales_to_tiles(const uint8_t* s, int64_t R, int64_t F, uint8_t* tiles,
                                   void* stream);

/*
 * fgq_quant_mxfp4_1x32 and fgq_quant_nvfp4_1x16 with the scales written in
 * the tiled layout (s_tiles: fgq_fp4_scale_tiles_bytes(R, K/32 or K/16)
 * bytes, 16-byte aligned; padding gets the codes of zero rows) instead of
 * row-major.  Codes, scales and
 * arguments otherwise as those calls; K % 128 == 0 (MXFP4) or
 * K % 64 == 0 (NVFP4).
 */
fgq_status fgq_quant_mxfp4_1x32_tiled(const void* x, int64_t R, int64_t K, int64_t ldx,
                                      uint8_t* xq, uint8_t* s_tiles, void* stream);
fgq_status fgq_quant_nvfp4_1x16_tiled(const void* x, int64_t R, int64_t K, int64_t ldx,
                                      const float* g, uint8_t* xq, uint8_t* s_tiles, void* stream);

/*
 * fgq_gemm_mxfp4 and fgq_gemm_nvfp4 with sA and sB in the tiled layout
 * (16-byte aligned; sA for the M rows of A, sB for the N rows of the
 * transposed weight).  Same products, same arguments and limits otherwise.
 * The tensor-map engine loads each stage's factor tiles with its operand
 * tiles; once A has two 128-row tiles, pairs of CTAs (a cluster of two)
 * share each 256-row tile, each loading half of the weight tile.
 */
fgq_status fgq_gemm_mxfp4_tiled(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                                const uint8_t* sB, void* C, int64_t ldc, int64_t M, int64_t N,
                                int64_t K, int out, void* stream);
fgq_status fgq_gemm_nvfp4_tiled(const uint8_t* A, const uint8_t* sA, const float* gA,
                                const uint8_t* B, const uint8_t* sB, const float* gB, void* C,
                                int64_t ldc, int64_t M, int64_t N, int64_t K, int out,
                                void* stream);

/*
 * FP8 GEMM with power-of-two scales given as UE8M0 code tiles
 * (§Blackwell: Native Block Scaling: UE8M0 = 2^(e-127); §UE8M0 vs E4M3
 * Scale Formats).  The product is fgq_gemm_fp8_blockscaled_ex's in
 * FGQ_SCALE_UE8M0 mode; only the scales' storage differs.  Codes are the
 * biased exponent fields of the fp32 power-of-two scales, laid out like the
 * FP4 scale tiles (fgq_fp4_scales_to_tiles) with F = K/128 codes a row
 * padded to a multiple of 4: byte ((r/128)*(F4/4) + f/4)*512 + (r%32)*16 +
 * ((r%128)/32)*4 + f%4, F4 = 4*ceil(F/4), of ceil(R/128)*128*F4 bytes.
 *   activation tiles: row m's codes are those of sA[m, 0..K/128);
 *   weight tiles: row n (a column of W, a row of the transposed codes
 *   [N, K]) holds the codes of sB[c, n/128], c = 0..K/128.
 * The tensor-map engine loads the tiles with the operands, and once A has
 * two 128-row tiles pairs of CTAs share each 256-row tile (each loading
 * half of the weight tile).
 *
 * fgq_ue8m0_scale_tiles_bytes: that size for R rows (M or N).
 * fgq_ue8m0_scale_tiles_act: sA fp32 [M, K/128] (powers of two, 4-byte
 *   aligned) -> tiles (16-byte aligned).  Device buffers, async on stream.
 * fgq_ue8m0_scale_tiles_weight: sB fp32 [K/128, N/128] -> tiles for N rows.
 * fgq_gemm_fp8_ue8m0_tiled: A E4M3 [M, K] (row-major, dense), B E4M3 [N, K]
 *   (the K-major weight codes of fgq_quant_w_128x128), sA and sB the
 *   activation and weight code tiles (16-byte aligned), C as _ex.
 *   K % 128 == 0, N % 128 == 0, M >= 0.
 */
fgq_status fgq_ue8m0_scale_tiles_bytes(int64_t R, int64_t K, size_t* bytes);
/* fgq_quant_operands in FGQ_SCALE_UE8M0 mode with the scales written
 * straight into the two code tiles (sA_tiles for the M rows of A, sB_tiles
 * for the N columns of W; fgq_ue8m0_scale_tiles_bytes each; padding
 * untouched) instead of fp32 arrays: the same codes as the fp32 scales'
 * exponent fields.  Arguments and limits otherwise as fgq_quant_operands. */
fgq_status fgq_quant_operands_ue8m0_tiles(const void* x, int64_t M, int64_t K, int64_t ldx,
                                          uint8_t* xq, int64_t ldq, uint8_t* sA_tiles,
                                          const void* w, int64_t N, int64_t ldw, uint8_t* wq,
                                          uint8_t* sB_tiles, void* stream);
fgq_status fgq_ue8m0_scale_tiles_act(const float* sA, int64_t M, int64_t K, uint8_t* tiles,
                                     void* stream);
fgq_status fgq_ue8m0_scale_tiles_weight(const float* sB, int64_t K, int64_t N, uint8_t* tiles,
                                        void* stream);
fgq_status fgq_gemm_fp8_ue8m0_tiled(const uint8_t* A, const uint8_t* sA, const uint8_t* B,
                                    const uint8_t* sB, void* C, int64_t ldc, int64_t M, int64_t N,
                                    int64_t K, int out, void* stream);

/* Workspace bytes fgq_gemm_fp8_blockscaled_splitk needs for (M, N, K) on the
 * current device (depends on its SM count; 256 when the problem has no
 * partial tiles).  Same size checks as the GEMM. */
fgq_status fgq_gemm_splitk_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes);

/* Size of the fixed scratch array behind fgq_gemm_fp8_blockscaled_splitk_noalloc. */
#define FGQ_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * fgq_gemm_fp8_blockscaled_splitk without a workspace argument, for callers
 * that cannot allocate device memory: code running inside an allocator or a
 * memory-pool callback, hosts that give a library a fixed device-memory
 * budget up front, embedders with no allocator of their own.  (The page has
 * no counterpart to this; it is a convenience of this library.)
 *
 * The split-K scratch is a fixed array of FGQ_NOALLOC_SCRATCH_BYTES inside
 * the library, present on every GPU that loads it until the process exits.
 * This call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.  Arguments and result are those of
 * fgq_gemm_fp8_blockscaled_splitk.
 *   - A problem whose split-K workspace (fgq_gemm_splitk_workspace_size)
 *     exceeds FGQ_NOALLOC_SCRATCH_BYTES returns FGQ_ERR_INVALID_ARG before
 *     anything is launched.
 *   - The first call on each device looks up the array's device address;
 *     make that first call before capturing any stream on that device.
 *     A device reset (cudaDeviceReset) discards the device's context and
 *     with it that address; the first call afterwards looks it up again
 *     (the lookup is keyed by the context's id), so make that call before
 *     any capture as well.
 *   - Every call with partial tiles clears the part of the array that must
 *     start at zero (the per-tile counters and ready flags) on `stream`
 *     before its kernel runs; the rest keeps the previous call's partial
 *     results, which are always overwritten before they are read.
 *   - All calls on a device share the one array: calls that can overlap on
 *     the GPU (different streams without ordering between them) race and
 *     give wrong results.  Order them, e.g. issue them on one stream.
 */
fgq_status fgq_gemm_fp8_blockscaled_splitk_noalloc(const uint8_t* A, const float* sA,
                                                   const uint8_t* B, const float* sB, void* C,
                                                   int64_t ldc, int64_t M, int64_t N, int64_t K,
                                                   int out, int mode, void* stream);

/* Static description of a status code. */
const char* fgq_status_string(fgq_status status);

/*
 * The device error word of the current device: 0 while no kernel has given
 * up on a wait; otherwise bits naming the wait that timed out.  If `clear`
 * is nonzero the word is reset to 0.  Synchronises the current device.
 * Returns FGQ_ERR_DEVICE_TIMEOUT when the word was nonzero.
 */
fgq_status fgq_device_error(uint32_t* word, int clear);

/*
 * Diagnostic for the failure path of every kernel's waits (the pages have
 * no counterpart; it checks this library's own error reporting).  Launches
 * one warp that waits, with the same bounded wait the GEMM kernels use, on
 * an mbarrier that nothing ever completes.  After about 2 s the wait gives
 * up, sets bit 0x80 of the device error word and the kernel returns; no
 * fault, and the context stays usable.  Afterwards fgq_device_error(&w, 1)
 * returns FGQ_ERR_DEVICE_TIMEOUT with (w & 0x80) != 0 and clears the word.
 * Asynchronous on `stream`; returns FGQ_ERR_CUDA if the launch fails.
 */
fgq_status fgq_selftest_wait_timeout(void* stream);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int fgq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FGQ_H_ */
