/*
 * mxfp4.h -- C ABI of libmxfp4: block-scaled FP4 (MXFP4 / NVFP4) quantization
 * and GEMM on GB300 (sm_103a).
 *
 * Sources of the operations (web pages, by title):
 *   [MM-517169] kernelbot-amd-mxfp4-mm-517169 -- bf16 A is quantized per 1x32
 *               block to MXFP4 and multiplied with a pre-quantized MXFP4 weight
 *               B into bf16 C; its "Optimization 5" docstring motivates the fused
 *               path in which the quantized A never reaches global memory.
 *   [MM-683203] kernelbot-amd-mxfp4-mm-683203 -- the quant kernel writes scales
 *               straight into the layout the GEMM consumes; per-shape state is
 *               resolved once and the hot path allocates nothing.
 *   [NV-496271] kernelbot-nvfp4-group-gemm-496271 -- a list of (a, b, c) NVFP4
 *               problems with E4M3 scales per 16 elements in the 128x4 blocked
 *               layout, each multiplied into an fp16 C.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers named A, Aq, B, Bq, C, *_sf and workspace are DEVICE pointers
 *   (memory of the current CUDA device). `problems` in nvfp4_group_gemm is a
 *   HOST array. The caller owns all memory; the library never allocates or
 *   frees device memory and never synchronizes the stream.
 * - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *   stream. Work is enqueued on it asynchronously.
 * - Matrices are row-major. A leading dimension is given in ELEMENTS for bf16
 *   and fp16 matrices and in BYTES for packed FP4 matrices.
 * - Packed FP4 (E2M1): two codes per byte, the even-k element in the low nibble
 *   ([MM-517169] module docstring); code bit 3 is the sign, bits 0-2 index the
 *   magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 * - Scale buffers use the 128x4 blocked layout ([NV-496271] _prepare_scale_for_tma):
 *   scale (r, c) of a logical [R, C] matrix is the byte at
 *     ((r/128)*ceil(C/4) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4,
 *   and the buffer holds mxfp4_sf_bytes(R, K, vec) bytes. MXFP4 scales are
 *   E8M0 (2^(b-127)), one per 32 K-elements; NVFP4 scales are E4M3, one per 16.
 * - Alignment (violations return MXFP4_ERR_MISALIGNED): bf16 inputs A are
 *   read with 16-byte vectors (A 16-byte aligned, lda a multiple of 8);
 *   packed FP4 GEMM operands and every scale buffer a GEMM reads are loaded
 *   by TMA (16-byte aligned, packed row stride a multiple of 16 bytes);
 *   quantizer outputs need 4-byte alignment (ldq a multiple of 4); C needs
 *   only element alignment.
 * - Errors: arguments are checked on the host before anything is enqueued; a
 *   non-OK status means nothing was launched. A failed launch returns
 *   MXFP4_ERR_CUDA. There is no fallback path of any kind. Every call below
 *   that launches a kernel can also fail on the device after returning
 *   MXFP4_OK: a kernel that gives up a bounded wait leaves that call's
 *   outputs unspecified and reports it only through mxfp4_get_device_error,
 *   which a caller whose results matter checks after synchronizing.
 * - Thread safety: calls may come from several host threads; the internal
 *   plan cache is locked.
 * - Overlap of consecutive calls: GEMM and quantization launches use
 *   programmatic dependent launch. A GEMM call may start before the
 *   preceding kernel in the stream has completed and may already read its
 *   pre-quantized weights (Bq, B_sf) then; A, C, the workspace and every
 *   write wait until the preceding kernel has completed. A kernel of this
 *   library lets its successor start early only after its own wait for its
 *   predecessor, and a quantization kernel makes its codes and scales visible
 *   device-wide before it exits, so weights written by this library's
 *   quantization calls, or by work enqueued before the preceding kernel, are
 *   read in stream order. Weights written by some other kernel launched
 *   directly before a GEMM call on the same stream need an event or a copy
 *   between the two: that kernel's writes are guaranteed visible to a
 *   dependent launch only once the dependent grid has waited for it.
 */
#ifndef MXFP4_GB300_H
#define MXFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MXFP4_API __attribute__((visibility("default")))
#else
#define MXFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MXFP4_OK = 0,
    MXFP4_ERR_INVALID_ARG = 1,         /* null pointer, non-positive size, bad enum */
    MXFP4_ERR_UNSUPPORTED_SHAPE = 2,   /* K not a multiple of the scale vector, too many groups */
    MXFP4_ERR_MISALIGNED = 3,          /* pointer or row stride breaks the 16-byte rule */
    MXFP4_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes below the matching *_workspace_bytes() */
    MXFP4_ERR_CUDA = 5,                /* a CUDA runtime/driver call failed */
    MXFP4_ERR_DEVICE_TIMEOUT = 6,      /* a kernel gave up waiting (see mxfp4_get_device_error) */
    MXFP4_ERR_NO_DEVICE = 7            /* current device is not a compute capability 10.3 GPU */
} mxfp4_status_t;

/* Human-readable name of a status code (static string, never NULL). */
MXFP4_API const char *mxfp4_status_string(mxfp4_status_t status);

/* ABI version of this header; bumps on any incompatible change. */
MXFP4_API int mxfp4_abi_version(void);

/* Bytes of a blocked scale buffer for `rows` rows of `k` FP4 elements with one
 * scale per `vec` elements (vec = 32 for MXFP4, 16 for NVFP4):
 * ceil(rows/128) * ceil((k/vec)/4) * 512. Returns 0 if vec is not 16 or 32,
 * k is not a multiple of vec, or a size is not positive. */
MXFP4_API size_t mxfp4_sf_bytes(int64_t rows, int64_t k, int vec);

/* ---------------------------------------------------------- quantization -- */

/* Dynamic per-1x32 MXFP4 quantization of bf16 A [M, K] ([MM-517169] module
 * docstring steps 1-2; [MM-683203] _quant_shuffled writes the scales directly
 * in the consumer's layout). Per 32-element block along K:
 *   e = clamp(floor(log2(amax)) - 2, -127, 127), amax = 0 -> e = -127;
 *   scale byte = e + 127;  code_i = E2M1 round-half-to-even of x_i * 2^-e,
 *   saturating at +-6, IEEE sign kept (-0 -> 0x8).
 *   A    : bf16 [M, K], row stride lda elements (lda >= K, lda % 8 == 0).
 *   Aq   : out, uint8 [M, K/2], row stride ldq bytes (ldq >= K/2, ldq % 4 == 0;
 *          a multiple of 16 if Aq is later a GEMM operand).
 *   A_sf : out, blocked E8M0 scales, mxfp4_sf_bytes(M, K, 32) bytes; every pad
 *          cell is written with 0x7F (scale 1.0, [MM-683203] key trick 2).
 * K must be a positive multiple of 32. Also used to pre-quantize weights B. */
MXFP4_API mxfp4_status_t mxfp4_quantize(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq,
                              int64_t ldq, void *A_sf, void *stream);

/* Per-1x16 NVFP4 quantization of bf16 A [M, K] (the operand format of
 * [NV-496271]; the pages do not print the producer's rule, this library's
 * reading is): s = E4M3(round-to-nearest-even, saturating at 448) of
 * fp32(amax)/6; code_i = E2M1 RNE of fp32(x_i)/s (fp32 division), saturating;
 * s == 0 gives zero magnitudes with the sign kept. Same argument meaning as
 * mxfp4_quantize; A_sf holds mxfp4_sf_bytes(M, K, 16) bytes, pad cells 0x00.
 * K must be a positive multiple of 16. */
MXFP4_API mxfp4_status_t nvfp4_quantize(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq,
                              int64_t ldq, void *A_sf, void *stream);

/* ------------------------------------------------------------------ GEMM -- */

/* Workspace bytes needed by mxfp4_gemm_a4w4 and mxfp4_quant_gemm_fused for
 * this shape (split-K partial sums, tile tickets and, for the two-kernel path,
 * the quantized A). Depends only on (M, N, K). The workspace must be filled
 * with zeros before its FIRST use; every successful call leaves the counters
 * inside it at zero again (the rest is scratch), so it can be reused for any
 * later call without clearing. Calls that share one workspace must not run
 * concurrently. */
MXFP4_API size_t mxfp4_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Block-scaled MXFP4 GEMM, C = (Aq * A_sf) x (Bq * B_sf)^T ([MM-517169]
 * docstring steps 3-4 and the gemm_a4w4 call; [MM-683203] launch 2): for every
 * m < M, n < N,
 *   C[m, n] = bf16_rne( sum_k  e2m1(Aq[m,k]) 2^(A_sf[m,k/32]-127)
 *                            * e2m1(Bq[n,k]) 2^(B_sf[n,k/32]-127) ),
 * accumulated in fp32 on the tensor cores (tcgen05.mma kind::mxf4).
 *   Aq  : uint8 [M, K/2], row stride ldaq bytes;  A_sf: blocked, mxfp4_sf_bytes(M, K, 32).
 *   Bq  : uint8 [N, K/2], row stride ldbq bytes;  B_sf: blocked, mxfp4_sf_bytes(N, K, 32).
 *   C   : out, bf16 [M, N], row stride ldc elements (ldc >= N).
 *   workspace: device scratch of ws_bytes >= mxfp4_workspace_bytes(M, N, K).
 * K must be a positive multiple of 32. */
MXFP4_API mxfp4_status_t mxfp4_gemm_a4w4(const void *Aq, int64_t ldaq, const void *A_sf, const void *Bq,
                               int64_t ldbq, const void *B_sf, void *C, int64_t ldc, int64_t M,
                               int64_t N, int64_t K, void *workspace, size_t ws_bytes,
                               void *stream);

/* mxfp4_gemm_a4w4 with the epilogue extras the source pages' GEMM call
 * carries ([MM-683203] "Launch 2": bias, alpha, beta, there None / 1.0 / 0.0):
 *   C[m, n] = bf16_rne( ((alpha * acc[m, n]) + beta * C[m, n]) + bias[n] )
 * evaluated in fp32 in that order, where acc is the fp32 block-scaled product
 * of mxfp4_gemm_a4w4 and C[m, n] on the right is C's value before the call
 * (not read when beta == 0). bias: bf16 [N] (2-byte aligned) or NULL.
 * alpha and beta must be finite. alpha = 1, beta = 0, bias = NULL is exactly
 * mxfp4_gemm_a4w4. Same workspace as mxfp4_gemm_a4w4. */
MXFP4_API mxfp4_status_t mxfp4_gemm_a4w4_ex(const void *Aq, int64_t ldaq, const void *A_sf, const void *Bq,
                                            int64_t ldbq, const void *B_sf, void *C, int64_t ldc, int64_t M,
                                            int64_t N, int64_t K, float alpha, float beta, const void *bias,
                                            void *workspace, size_t ws_bytes, void *stream);

/* Dynamic MXFP4 quantization of bf16 A fused with the block-scaled GEMM
 * against pre-quantized Bq ([MM-517169] "Optimization 5"; [MM-683203] docstring).
 * Result equals mxfp4_quantize(A) followed by mxfp4_gemm_a4w4 (bit-identical
 * quantization, same accumulation contract). For small M (the activation
 * rows fit one MMA N-tile) the quantized A is formed on chip and never touches
 * global memory; for larger M the library runs the quant kernel into the
 * workspace and then the GEMM.
 *   A   : bf16 [M, K], row stride lda elements.
 *   Bq, B_sf, C, ldc, workspace: as in mxfp4_gemm_a4w4. */
MXFP4_API mxfp4_status_t mxfp4_quant_gemm_fused(const void *A, int64_t lda, const void *Bq, int64_t ldbq,
                                      const void *B_sf, void *C, int64_t ldc, int64_t M,
                                      int64_t N, int64_t K, void *workspace, size_t ws_bytes,
                                      void *stream);

/* The NVFP4 twin of mxfp4_quant_gemm_fused for small M (1 <= M <= 64):
 * dynamic NVFP4 quantization of bf16 A (per 16 elements along K: scale
 * s = E4M3_RNE_sat(fp32(amax) / 6), codes E2M1_RNE_sat(fp32(x) / s), as
 * nvfp4_quantize) fused on chip with the block-scaled GEMM against a
 * pre-quantized NVFP4 B (E2M1 [N, K/2], blocked E4M3 scales
 * mxfp4_sf_bytes(N, K, 16)):
 *   C[m, n] = fp16_rne( sum_k A_q[m, k] * B_q[n, k] )   (fp32 accumulation)
 * The quantized A never reaches global memory; no workspace. K % 16 == 0;
 * M > 64 returns MXFP4_ERR_UNSUPPORTED_SHAPE (use nvfp4_quantize and
 * nvfp4_group_gemm there). Alignment as for mxfp4_quant_gemm_fused. */
MXFP4_API mxfp4_status_t nvfp4_quant_gemm_fused(const void *A, int64_t lda, const void *Bq, int64_t ldbq,
                                                const void *B_sf, void *C, int64_t ldc, int64_t M, int64_t N,
                                                int64_t K, void *stream);

/* One problem of a grouped NVFP4 GEMM ([NV-496271] custom_kernel: each entry of
 * the problem list carries a, b, c, their scales and (m, n, k)). */
typedef struct {
    int64_t m, n, k;   /* C is [m, n]; k is the reduction length (multiple of 16) */
    const void *a;     /* uint8 [m, k/2] packed E2M1, row stride lda bytes */
    const void *sfa;   /* blocked E4M3 scales, mxfp4_sf_bytes(m, k, 16) bytes */
    const void *b;     /* uint8 [n, k/2] packed E2M1, row stride ldb bytes */
    const void *sfb;   /* blocked E4M3 scales, mxfp4_sf_bytes(n, k, 16) bytes */
    void *c;           /* out: fp16 [m, n], row stride ldc elements */
    int64_t lda, ldb, ldc;
} nvfp4_problem_t;

/* Problems a grouped call carries in its kernel parameters; a longer list
 * (any length up to 2^20) goes through a problem table that the call writes
 * into the caller's workspace (see nvfp4_group_workspace_bytes). */
#define NVFP4_MAX_GROUPS 16

/* Workspace bytes nvfp4_group_gemm needs for num_groups problems: 0 up to
 * NVFP4_MAX_GROUPS, else 640 bytes per problem (the device problem table:
 * four TMA descriptors and one problem record per group). 0 for an invalid
 * count. */
MXFP4_API size_t nvfp4_group_workspace_bytes(int num_groups);

/* Grouped NVFP4 GEMM: for each problem g,
 *   C_g[m, n] = fp16_rne( sum_k e2m1(a[m,k]) e4m3(sfa[m,k/16]) e2m1(b[n,k]) e4m3(sfb[n,k/16]) )
 * with fp32 accumulation (tcgen05.mma kind::mxf4nvf4, scale_vec::4X), all
 * groups in ONE GEMM launch scheduled tile by tile ([NV-496271] custom_kernel
 * runs one launch per group and batch index; a batch index l is flattened
 * into extra problems by the caller). `problems` is a host array of
 * num_groups entries (1 <= num_groups <= 2^20); it is read during the call
 * only. With more than NVFP4_MAX_GROUPS problems the call writes its problem
 * table into `workspace` (ws_bytes >= nvfp4_group_workspace_bytes, 64-byte
 * aligned) with small copy kernels enqueued on `stream` ahead of the GEMM, so
 * the call stays stream-ordered and can be captured in a CUDA graph; calls
 * that share a workspace must not overlap. Up to NVFP4_MAX_GROUPS problems the
 * workspace is not used (may be NULL). */
MXFP4_API mxfp4_status_t nvfp4_group_gemm(const nvfp4_problem_t *problems, int num_groups, void *workspace,
                                size_t ws_bytes, void *stream);

/* Fused RMSNorm + MXFP4 quantization of bf16 X [M, K] (row stride ldx
 * elements) with a bf16 weight [K] and eps: the activation step that
 * [MM-683203] ("hot path") fuses ahead of the GEMM, which the pages name
 * without giving its arithmetic. The reading this library takes, per row:
 *   ss  = sum_k x_k^2, exact, rounded once to fp64 (round to nearest even)
 *   r   = fp32(1 / sqrt(ss / K + eps)) computed in fp64 (r = 0 when
 *         ss / K + eps == 0)
 *   y_k = fp32(fp32(x_k * r) * weight_k)
 * and y is quantized exactly as mxfp4_quantize quantizes its input (OCP MX
 * rule per 32 values, E2M1 codes [M, K/2] with row stride ldq bytes, E8M0
 * scales in the blocked layout, mxfp4_sf_bytes(M, K, 32) bytes, pad 0x7F), so
 * the outputs feed mxfp4_gemm_a4w4 directly. The sum is exact for every
 * finite row, whatever the range of its magnitudes. Requirements: K % 32 == 0;
 * eps finite and >= 0; X and weight finite with every |y| finite; X and
 * weight 16-byte aligned, ldx * 2 a multiple of 16; Aq and A_sf 4-byte
 * aligned, ldq a multiple of 4. */
MXFP4_API mxfp4_status_t mxfp4_rmsnorm_quantize(const void *X, int64_t M, int64_t K, int64_t ldx,
                                                const void *weight, float eps, void *Aq, int64_t ldq,
                                                void *A_sf, void *stream);

/* mxfp4_rmsnorm_quantize that also stores, per row m, rstd[m] = r (the fp32
 * reciprocal the row was scaled by, as a backward pass keeps it) and
 * sumsq[m] = ss (the exactly rounded fp64 sum of squares). Either pointer may
 * be NULL (not stored); otherwise device memory of M entries, rstd 4-byte and
 * sumsq 8-byte aligned (MXFP4_ERR_MISALIGNED). Same outputs, rules and errors
 * as mxfp4_rmsnorm_quantize otherwise. */
MXFP4_API mxfp4_status_t mxfp4_rmsnorm_quantize_ex(const void *X, int64_t M, int64_t K, int64_t ldx,
                                                   const void *weight, float eps, void *Aq, int64_t ldq,
                                                   void *A_sf, float *rstd, double *sumsq, void *stream);

/* One problem of a grouped NVFP4 GEMM whose activation is still bf16: the
 * [NV-496271] problem list (custom_kernel) with A given unquantized, as a
 * mixture-of-experts layer receives it. */
typedef struct {
    int64_t m, n, k;   /* C is [m, n]; k is the reduction length (multiple of 16) */
    const void *a;     /* bf16 [m, k], row stride lda elements (lda * 2 a multiple of 16) */
    const void *b;     /* uint8 [n, k/2] packed E2M1, row stride ldb bytes */
    const void *sfb;   /* blocked E4M3 scales, mxfp4_sf_bytes(n, k, 16) bytes */
    void *c;           /* out: fp16 [m, n], row stride ldc elements */
    int64_t lda, ldb, ldc;
} nvfp4_act_problem_t;

/* Workspace bytes nvfp4_group_quant_gemm needs for these problems (every
 * group's quantized A and its scales, then the problem table for lists longer
 * than NVFP4_MAX_GROUPS), or 0 if the list is invalid. Pointers are not read. */
MXFP4_API size_t nvfp4_group_quant_gemm_workspace_bytes(const nvfp4_act_problem_t *problems, int num_groups);

/* Dynamic NVFP4 quantization of every group's bf16 A followed by the grouped
 * NVFP4 GEMM: one launch per NVFP4_MAX_GROUPS groups quantizes the A_g with
 * nvfp4_quantize's rule and layout into the workspace, then (in stream order)
 * one GEMM launch computes every C_g as nvfp4_group_gemm does from those
 * operands. `problems` is a host array of num_groups entries (1 <= num_groups
 * <= 2^20), read during the call only. `workspace`: caller-owned device
 * memory of at least nvfp4_group_quant_gemm_workspace_bytes bytes, 16-byte
 * aligned (64-byte aligned with more than NVFP4_MAX_GROUPS problems); it needs
 * no initialisation and afterwards holds the quantized A_g (layout not part of
 * the ABI). Every argument is validated before anything is enqueued; a too
 * small workspace gives MXFP4_ERR_WORKSPACE_TOO_SMALL. */
MXFP4_API mxfp4_status_t nvfp4_group_quant_gemm(const nvfp4_act_problem_t *problems, int num_groups,
                                                void *workspace, size_t ws_bytes, void *stream);

/* One problem of a grouped MXFP4 GEMM: the problem list of [NV-496271]
 * custom_kernel (a, b, c, their scales, (m, n, k)) with MXFP4 operands
 * ([MM-517169]: E2M1 codes, E8M0 scale per 32 along K) and bf16 C, the layout
 * of a mixture-of-experts layer whose experts hold MXFP4 weights. */
typedef struct {
    int64_t m, n, k;   /* C is [m, n]; k is the reduction length (multiple of 32) */
    const void *a;     /* uint8 [m, k/2] packed E2M1, row stride lda bytes */
    const void *sfa;   /* blocked E8M0 scales, mxfp4_sf_bytes(m, k, 32) bytes */
    const void *b;     /* uint8 [n, k/2] packed E2M1, row stride ldb bytes */
    const void *sfb;   /* blocked E8M0 scales, mxfp4_sf_bytes(n, k, 32) bytes */
    void *c;           /* out: bf16 [m, n], row stride ldc elements */
    int64_t lda, ldb, ldc;
} mxfp4_problem_t;

/* Problems mxfp4_group_gemm carries in its kernel parameters; longer lists
 * go through a problem table in the workspace, as for nvfp4_group_gemm. */
#define MXFP4_MAX_GROUPS 16

/* Workspace bytes mxfp4_group_gemm needs for num_groups problems (0 up to
 * MXFP4_MAX_GROUPS, else 640 bytes per problem). */
MXFP4_API size_t mxfp4_group_workspace_bytes(int num_groups);

/* Grouped MXFP4 GEMM: for each problem g,
 *   C_g[m, n] = bf16_rne( sum_k e2m1(a[m,k]) 2^(sfa[m,k/32]-127) e2m1(b[n,k]) 2^(sfb[n,k/32]-127) )
 * with fp32 accumulation (tcgen05.mma kind::mxf4, scale_vec::2X), all groups
 * in ONE GEMM launch scheduled tile by tile, as nvfp4_group_gemm does for
 * NVFP4, with the same rules for the problem list (1 <= num_groups <= 2^20)
 * and the workspace (used only with more than MXFP4_MAX_GROUPS problems). */
MXFP4_API mxfp4_status_t mxfp4_group_gemm(const mxfp4_problem_t *problems, int num_groups, void *workspace,
                                          size_t ws_bytes, void *stream);

/* Bytes of the fixed device scratch array behind mxfp4_gemm_a4w4_noalloc
 * (8 MiB). */
MXFP4_API size_t mxfp4_noalloc_scratch_bytes(void);

/* The MXFP4 GEMM of mxfp4_gemm_a4w4 for callers that cannot allocate device
 * memory -- for example a plugin running inside an engine that owns every
 * device allocation and hands it no scratch buffer, or a program whose memory
 * plan is fixed at start-up. There is no counterpart on the source pages; it
 * is a convenience of this library.
 *   Same arguments and result as mxfp4_gemm_a4w4, without the workspace: the
 *   split-K scratch (fp32 partial sums and per-tile counters) lives in one
 *   static device array of mxfp4_noalloc_scratch_bytes() bytes inside the
 *   library, which every GPU that loads the library keeps until the process
 *   exits. The call allocates nothing; it clears the counters with an
 *   asynchronous memset on `stream` before the GEMM.
 *   Shapes whose scratch would exceed the array return
 *   MXFP4_ERR_WORKSPACE_TOO_SMALL before anything is enqueued (use
 *   mxfp4_gemm_a4w4 with a caller workspace for those).
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) once for that device; make that first call before
 *   any stream capture. All calls share the array and it keeps the last
 *   call's contents: calls that overlap on the GPU (other streams, other host
 *   threads without ordering) race on it and must be serialized by the
 *   caller. */
MXFP4_API mxfp4_status_t mxfp4_gemm_a4w4_noalloc(const void *Aq, int64_t ldaq, const void *A_sf,
                                                 const void *Bq, int64_t ldbq, const void *B_sf,
                                                 void *C, int64_t ldc, int64_t M, int64_t N,
                                                 int64_t K, void *stream);

/* ------------------------------------------------------------ diagnostics -- */

/* Kernels a call can launch (mxfp4_plan_t.kernel). */
#define MXFP4_KERNEL_FUSED 1      /* fused quantization + GEMM, swap-AB, K-split clusters */
#define MXFP4_KERNEL_GEMM 2       /* single-CTA block-scaled GEMM, 128 x tile_n tiles */
#define MXFP4_KERNEL_GEMM_PAIR 3  /* CTA-pair GEMM (tcgen05 cta_group::2), 256 x 256 tiles */

/* What a call launches: the GEMM kernel, the output tile one CTA (pair:
 * one CTA pair) computes, the K-splits per tile, the number of output tiles,
 * and whether a separate quantization kernel runs first. */
typedef struct {
    int kernel;
    int tile_m, tile_n;
    int splits;
    int tiles;
    int quant_launch;
} mxfp4_plan_t;

/* The plan of mxfp4_gemm_a4w4 (which = 0), mxfp4_quant_gemm_fused
 * (which = 1) or nvfp4_quant_gemm_fused (which = 2) for an M x N x K problem
 * on the current device. Launches
 * nothing; reads the device's SM count (MXFP4_ERR_NO_DEVICE without a usable
 * GB300). Argument checks as for the calls themselves, minus the pointers. */
MXFP4_API mxfp4_status_t mxfp4_gemm_plan(int64_t M, int64_t N, int64_t K, int which, mxfp4_plan_t *out);

/* The plan of nvfp4_group_gemm / mxfp4_group_gemm for these problems
 * (pointers are not read). */
MXFP4_API mxfp4_status_t nvfp4_group_gemm_plan(const nvfp4_problem_t *problems, int num_groups,
                                               mxfp4_plan_t *out);
MXFP4_API mxfp4_status_t mxfp4_group_gemm_plan(const mxfp4_problem_t *problems, int num_groups,
                                               mxfp4_plan_t *out);

/* Reads and clears the library's device-side error word. Kernels never trap:
 * a wait that exceeds its time limit (2 s unless mxfp4_set_wait_limit_ns set
 * another) records a nonzero code there and the kernel exits cleanly, after
 * every copy and MMA it issued has landed and with its TMEM freed. Because
 * the launching call has already returned MXFP4_OK by then, this is the only
 * place such a failure shows: a call whose kernel gave up leaves its outputs
 * unspecified (the GEMM kernels skip the stores of every tile, or K-split,
 * whose inputs did not all arrive, rather than store partial sums) and may
 * leave the split-K counters of its workspace nonzero, so clear the
 * workspace before reusing it after a nonzero code. This call synchronizes
 * the current device. *code receives 0 when no kernel reported an error;
 * otherwise 1..15 (single-CTA GEMM), 16 + c (fused kernel) or 32 + c
 * (CTA-pair GEMM), c naming the wait that gave up. */
MXFP4_API mxfp4_status_t mxfp4_get_device_error(int *code);

/* K-splits of the split-K paths. The planner takes, in this order: a tuning
 * override set here, the entry of the measured table built into the library
 * for the shape (exact N and K; M by bucket), or its shape-derived rule. The
 * plan functions above report the result. */
#define MXFP4_SPLITS_GEMM 0        /* two-kernel path: bucket = 128-row tiles of M */
#define MXFP4_SPLITS_FUSED 1       /* fused MXFP4 kernel: bucket = MMA width 16/32/64 */
#define MXFP4_SPLITS_FUSED_NV 2    /* fused NVFP4 kernel: bucket = MMA width 16/32/64 */

/* Sets (splits > 0) or clears (0) a process-wide override of the K-splits of
 * every later call on `path`, clamped per call to what the kernel can run;
 * returns the previous override, or -1 for a bad argument. Meant for tuning
 * (the table is written by block_scaled_fp4_mxfp4_gb300/tune_splits.py): the
 * workspace a shape needs follows the override, so query
 * mxfp4_workspace_bytes after setting it. */
MXFP4_API int mxfp4_set_split_override(int path, int splits);

/* Entry `index` of the measured split-K table (any pointer may be NULL);
 * returns the number of entries (and fills nothing when index is out of
 * range). */
MXFP4_API int mxfp4_split_table_entry(int index, int *path, int *bucket, int64_t *n, int64_t *k, int *splits);

/* Sets the time limit, in nanoseconds, of the waits that guard work inside
 * every kernel launched afterwards (process-wide; 0 restores the default of
 * 2 s) and returns the previous limit. The waits on a kernel's exit path,
 * which keep shared memory and TMEM alive until every copy and MMA the kernel
 * issued has landed, always keep 2 s. A short limit makes the kernels give up
 * on their own: tests use it to exercise the error path without faulting the
 * GPU. Not meant for production use. */
MXFP4_API uint64_t mxfp4_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_GB300_H */
