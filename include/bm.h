/*
 * bm.h -- C ABI of the GB300 (sm_103a) BF16 BLAS3 library: GEMM and SYRK.
 *
 * The operations are the BLAS3 local compute that the distributed framework in
 * "BLASMp development notes" rests on (section 1: GEMM is the long-term base
 * and performance yardstick; stage B: SYRK's main compute is a GEMM), carried
 * out by the tensor-core GEMM mainloop that the "cp.async / ldmatrix ablation
 * plan" dissects (section 2, fixed baseline: BF16 GEMM, FP32 accumulate), and
 * the beta = 0 / beta = 1 weight-gradient GEMMs of "fused A2A/GEMM Perfetto
 * profile protocol" (official timing rules: ZeroBubble W accumulates into a
 * BF16 gradient with beta = 1).
 *
 * Conventions shared by every entry point
 *   - Storage is row-major: element (r, c) of a matrix X with leading
 *     dimension ldx sits at X[r * ldx + c]. Column-major callers use
 *     C^T = op(B)^T op(A)^T, i.e. swap A and B and the transpose flags.
 *   - A and B hold bfloat16; products accumulate in FP32 on the tensor cores;
 *     alpha and beta are applied in FP32; C is FP32 or BF16 (round to nearest
 *     even on store).
 *   - BLAS rules: when beta == 0 the input C is not read (NaN/Inf in C do not
 *     propagate); when alpha == 0 or k == 0 the result is beta * C and A, B
 *     are not read; m == 0 or n == 0 is a no-op returning BM_OK. C must not
 *     overlap A or B.
 *   - Ownership: every pointer is a DEVICE pointer owned by the caller and
 *     must stay valid until the work queued on `stream` has finished. The
 *     library allocates nothing per call; it keeps one small device status
 *     word per device, allocated on first use.
 *   - Alignment (the tensor-memory-accelerator rules quoted in the ablation
 *     plan, section 1.3: 16-byte aligned global addresses): A, B and C must be
 *     16-byte aligned and lda*2, ldb*2, ldc*sizeof(C element) multiples of 16
 *     bytes; otherwise BM_ERR_MISALIGNED and nothing is launched. The sizes
 *     m, n, k need no alignment. When a row of C (n elements) does not end
 *     on a 16-byte boundary, C is written with masked plain stores instead
 *     of tensor-memory-accelerator stores (a slower epilogue): those stores
 *     would also write the columns from n up to the next 16-byte boundary.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     Argument errors are returned synchronously before anything is queued;
 *     a failed launch returns BM_ERR_CUDA. A device-side wait that runs out
 *     of time (see bm_set_wait_timeout_ms) is reported later by
 *     bm_get_last_device_error.
 *   - Stream order holds as for any kernel: a call reads and writes memory
 *     only after the work queued before it on `stream` has completed. (Its
 *     kernel is launched early and prepares meanwhile: barriers, tensor
 *     memory, and an L2 prefetch of its first A and B tiles, which brings no
 *     data into the SM and so cannot observe an older value.)
 *   - The device must be compute capability 10.3 (GB300, sm_103a); any other
 *     device gives BM_ERR_ARCH. There is no other code path.
 */
#ifndef BM_H
#define BM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BM_API __attribute__((visibility("default")))
#else
#define BM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t / CUstream. */
typedef struct CUstream_st *bm_stream_t;

typedef enum {
    BM_OK = 0,
    BM_ERR_INVALID_VALUE = 1, /* negative size, ld too small, bad enum           */
    BM_ERR_MISALIGNED = 2,    /* pointer or leading dimension breaks the 16-B rule */
    BM_ERR_ARCH = 3,          /* current device is not compute capability 10.3   */
    BM_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed      */
    BM_ERR_TIMEOUT = 5,       /* a device-side bounded wait ran out of time       */
    BM_ERR_WORKSPACE = 6      /* workspace pointer misaligned or NULL with bytes>0 */
} bm_status;

typedef enum { BM_OP_N = 0, BM_OP_T = 1 } bm_op;
typedef enum { BM_C_F32 = 0, BM_C_BF16 = 1 } bm_ctype;
/* The same element-type enum under the names bm_dtype, BM_F32 and BM_BF16. */
typedef bm_ctype bm_dtype;
#define BM_F32 BM_C_F32
#define BM_BF16 BM_C_BF16
typedef enum { BM_LOWER = 0, BM_UPPER = 1 } bm_uplo;

/*
 * GEMM:  C[m x n] = alpha * op(A) * op(B) + beta * C
 *
 *   op(A) is m x k: A is stored [m, k] (lda >= k) when transA == BM_OP_N and
 *   [k, m] (lda >= m) when transA == BM_OP_T. op(B) is k x n: B is stored
 *   [k, n] (ldb >= n) for BM_OP_N and [n, k] (ldb >= k) for BM_OP_T.
 *   C is [m, n] with ldc >= n, element type c_type; elements of C beyond
 *   column n within ldc are never touched.
 *
 *   workspace / workspace_bytes: optional caller-owned device scratch for
 *   FP32 partial sums when tiles are split along K: all tiles when m*n is too
 *   small to fill the GPU, or the tiles of a last, partly filled wave of the
 *   persistent schedule (then the idle SMs share them). NULL/0 disables the
 *   split; the result is correct either way. The size the planner would like
 *   is bm_gemm_bf16_workspace_size(); less is accepted (fewer or no splits).
 *   The workspace must be 256-byte aligned; its contents need not be
 *   initialised and are overwritten. When only some tiles are split, the
 *   split parts run first and the last part of each region to finish sums
 *   the partials inside the GEMM kernel; the workspace then also holds one
 *   8-byte counter per region, tagged with a per-call number, so stale or
 *   random bytes are never taken for this call's counts. A call captured in
 *   a CUDA graph keeps its number on every replay; each counter is reset
 *   when its region is summed, so replays start clean. (A replay that
 *   follows a replay stopped by a device-side wait limit, BM_ERR_TIMEOUT,
 *   may find counters that replay left behind: re-capture after a timeout.)
 *   When every tile is split, a second kernel sums the partials.
 *
 *   Returns BM_OK once the work is queued on `stream`.
 */
BM_API bm_status bm_gemm_bf16(int64_t m, int64_t n, int64_t k, bm_op transA, bm_op transB,
                              float alpha, const void *A, int64_t lda, const void *B, int64_t ldb,
                              float beta, void *C, int64_t ldc, bm_ctype c_type,
                              void *workspace, size_t workspace_bytes, bm_stream_t stream);

/* Bytes of workspace that bm_gemm_bf16 would use for this shape (0 = none). */
BM_API size_t bm_gemm_bf16_workspace_size(int64_t m, int64_t n, int64_t k);

/* Size of the device scratch array that bm_gemm_bf16_noalloc uses (16 MiB). */
#define BM_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * GEMM that allocates nothing. The paper has no counterpart: this entry
 * point exists for callers that cannot call cudaMalloc, such as code that
 * runs inside a framework which owns all device memory through its own pool,
 * a plug-in called back by another library that gives it no allocator, or a
 * latency-critical path where the implicit synchronisation of cudaMalloc is
 * not acceptable.
 *
 * Same operation, arguments, layout rules and errors as bm_gemm_bf16, except
 * that there is no workspace argument. When the launch plan splits K (small
 * m * n, long k, or the tiles of a partly filled last wave), the partial sums
 * go to one file-scope device array of BM_NOALLOC_SCRATCH_BYTES that the
 * library holds on every GPU it is loaded on, until the process exits. The
 * plan is the one bm_gemm_bf16 makes when given a workspace of
 * BM_NOALLOC_SCRATCH_BYTES bytes: where a full split would need more, the
 * planner splits fewer ways so that the partials fit. Like that plan it
 * depends on beta (a tail split with beta != 0 must save more time, so such a
 * call may split fewer tiles). BM_ERR_WORKSPACE is returned, with nothing
 * launched, only if a plan ever exceeded the array, which the planner does
 * not produce. The caller still owns and passes A, B and C.
 *
 *   - The first call on a device looks up the device address of the array
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array, and it keeps the last
 *     call's contents. Nothing in it needs to start at zero (every partial
 *     that is read was written by the same call). Calls whose kernels
 *     overlap on the GPU (different streams, no ordering between them) race
 *     on it and give wrong results; order them on one stream or with events.
 *   - No cudaMalloc, cudaFree or other allocating routine is called. A
 *     device-side wait that runs out is recorded in the status word read by
 *     bm_get_last_device_error only if another entry point of this library
 *     has already created that word on the device (this call never creates
 *     it).
 */
BM_API bm_status bm_gemm_bf16_noalloc(int64_t m, int64_t n, int64_t k, bm_op transA, bm_op transB,
                                      float alpha, const void *A, int64_t lda, const void *B,
                                      int64_t ldb, float beta, void *C, int64_t ldc, bm_ctype c_type,
                                      bm_stream_t stream);

/*
 * GEMM with FP8 E4M3 operands:  C[m x n] = alpha * A * B^T + beta * C
 *
 *   The all-E4M3, FP32-accumulated matrix products of the FP8 paths in "fused
 *   A2A/GEMM Perfetto profile protocol" (FP8 section). A is [m, k] (lda >= k)
 *   and B is [n, k] (ldb >= k), both row-major with one E4M3 code per byte
 *   (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; subnormals
 *   honoured). Any per-tensor scaling of the FP8 data goes into alpha. C is
 *   FP32 or BF16 as for bm_gemm_bf16, and the workspace, BLAS rules, errors and
 *   stream behaviour are the same, except the alignment rule: lda and ldb
 *   must be multiples of 16 (bytes = elements).
 *
 *   Returns BM_OK once the work is queued on `stream`.
 */
BM_API bm_status bm_gemm_e4m3(int64_t m, int64_t n, int64_t k, float alpha, const void *A, int64_t lda,
                              const void *B, int64_t ldb, float beta, void *C, int64_t ldc,
                              bm_ctype c_type, void *workspace, size_t workspace_bytes,
                              bm_stream_t stream);

/* Bytes of workspace that bm_gemm_e4m3 would use for this shape (0 = none). */
BM_API size_t bm_gemm_e4m3_workspace_size(int64_t m, int64_t n, int64_t k);

/*
 * GEMM with MXFP8 operands:  C[m x n] = alpha * (A . SA) * (B . SB)^T + beta * C
 *
 *   The block-scaled MXFP8 GEMM of the SM103 path in "fused A2A/GEMM Perfetto
 *   profile protocol" (MXFP8 GEMM hot-path table; E4M3 data with one UE8M0
 *   scale per group of 32 consecutive elements along K, "K32 quantization
 *   group"). Element (i, p) of A stands for A[i][p] * 2^(sa - 127), where sa is
 *   the UE8M0 code of row i's group p / 32; likewise for B. A is [m, k]
 *   (lda >= k) and B is [n, k] (ldb >= k), row-major E4M3 codes as for
 *   bm_gemm_e4m3 (lda, ldb multiples of 16). Products accumulate in FP32 on the
 *   tensor cores (tcgen05.mma kind::mxf8f6f4, block-scaled); C, alpha, beta,
 *   the workspace, BLAS rules, errors and stream behaviour are as for
 *   bm_gemm_bf16.
 *
 *   Scale arrays SA (for A's m rows) and SB (for B's n rows): UE8M0 codes
 *   (value 2^(code - 127); 255 is NaN) in the tiled layout the tensor cores
 *   read, 16-byte aligned. They hold ceil(rows / 128) x ceil(k / 128) atoms of
 *   512 bytes; the code of row r, group g (elements 32 g .. 32 g + 31 of the
 *   row) is at byte
 *       ((r / 128) * ceil(k / 128) + g / 4) * 512
 *         + (r % 32) * 16 + ((r % 128) / 32) * 4 + g % 4.
 *   Entries past the last row or the last group are padding: they must not be
 *   255 (a NaN scale would turn the zeros they multiply into NaN).
 *
 *   Returns BM_OK once the work is queued on `stream`.
 */
BM_API bm_status bm_gemm_mxfp8(int64_t m, int64_t n, int64_t k, float alpha, const void *A, int64_t lda,
                               const void *SA, const void *B, int64_t ldb, const void *SB, float beta, void *C,
                               int64_t ldc, bm_ctype c_type, void *workspace, size_t workspace_bytes,
                               bm_stream_t stream);

/* Bytes of workspace that bm_gemm_mxfp8 would use for this shape (0 = none). */
BM_API size_t bm_gemm_mxfp8_workspace_size(int64_t m, int64_t n, int64_t k);

/*
 * MXFP8 quantization of a BF16 matrix: X[rows x k] -> E4M3 codes Q[rows x k]
 * and UE8M0 scales S, one per group of 32 consecutive elements of a row.
 *
 *   The "W quantize BF16 -> MXFP8" step of the SM103 MXFP8 path in "fused
 *   A2A/GEMM Perfetto profile protocol" (per group of 32: amax reduction, UE8M0
 *   scale, E4M3 conversion). The page names the steps; the rule is the OCP
 *   Microscaling (MX) v1.0 conversion: shared exponent e = floor(log2(amax)) - 8
 *   (8 is the largest E4M3 exponent), clamped to [-127, 127], scale code
 *   e + 127; each element is X / 2^e rounded to the nearest E4M3 value, ties to
 *   even, magnitudes beyond 448 saturated to 448. A group of zeros gets code 0;
 *   a group holding a NaN or an infinity gets code 255 (NaN) and NaN elements
 *   (0x7F). The last group of a row may be shorter than 32.
 *
 *   X is row-major bf16 with ldx >= k (ldx * 2 a multiple of 16 bytes); Q is
 *   row-major E4M3 with ldq >= k (a multiple of 16); Q's bytes past column k
 *   are not written. S receives ceil(rows / 128) x ceil(k / 128) atoms of 512
 *   bytes in the tiled layout of bm_gemm_mxfp8 (padding entries are set to 0),
 *   so Q and S feed bm_gemm_mxfp8 directly as A and SA, or as B and SB. All
 *   three pointers are device memory, 16-byte aligned, and must not overlap.
 *   Errors and stream behaviour as for bm_gemm_bf16.
 *
 *   Returns BM_OK once the work is queued on `stream`.
 */
BM_API bm_status bm_quantize_mxfp8(int64_t rows, int64_t k, const void *X, int64_t ldx, void *Q, int64_t ldq,
                                   void *S, bm_stream_t stream);

/*
 * SYRK:  C = alpha * op(A) * op(A)^T + beta * C   on one triangle of C[n x n]
 *
 *   op(A) is n x k: A is stored [n, k] (lda >= k) when trans == BM_OP_N
 *   (C = A A^T) and [k, n] (lda >= n) when trans == BM_OP_T (C = A^T A).
 *   uplo == BM_LOWER updates the elements with row >= column, BM_UPPER those
 *   with row <= column. The other triangle is neither read nor written.
 *   Tiles of C that lie entirely in the other triangle are not computed.
 *   C is [n, n] with ldc >= n.
 *
 *   workspace / workspace_bytes: optional caller-owned device scratch for FP32
 *   partial sums, with the rules of bm_gemm_bf16 ("Arguments + workspace" of
 *   "BLASMp development notes", stage D; the workspace need not be
 *   initialised): when the triangle has too few tiles to fill the GPU (small n,
 *   long k) every tile is split along K and a second kernel sums the partials;
 *   the tiles of a partly filled last wave may be split and summed inside the
 *   kernel. The sums write only the referenced triangle. NULL/0 disables the
 *   split; the size the planner would like is bm_syrk_bf16_workspace_size().
 *
 *   Returns BM_OK once the work is queued on `stream`.
 */
BM_API bm_status bm_syrk_bf16(bm_uplo uplo, bm_op trans, int64_t n, int64_t k, float alpha,
                              const void *A, int64_t lda, float beta, void *C, int64_t ldc,
                              bm_ctype c_type, void *workspace, size_t workspace_bytes, bm_stream_t stream);

/* Bytes of workspace that bm_syrk_bf16 would use for this shape (0 = none). */
BM_API size_t bm_syrk_bf16_workspace_size(bm_uplo uplo, int64_t n, int64_t k);

/*
 * SYR2K:  C = alpha * (op(A) * op(B)^T + op(B) * op(A)^T) + beta * C
 *         on one triangle of C[n x n]
 *
 *   The rank-2k update among the BLAS3 operators of "BLASMp development
 *   notes" (stage D adds SYR2K; stage F restructures it like SYRK). op(A) and
 *   op(B) are n x k: A, B are stored [n, k] (lda, ldb >= k) when trans ==
 *   BM_OP_N and [k, n] (lda, ldb >= n) when trans == BM_OP_T. Both products go
 *   through one FP32 accumulator per tile; uplo, the untouched other
 *   triangle, C, the workspace and the error behaviour are as for bm_syrk_bf16
 *   (a K split divides the 2k products of a tile).
 *
 *   Returns BM_OK once the work is queued on `stream`.
 */
BM_API bm_status bm_syr2k_bf16(bm_uplo uplo, bm_op trans, int64_t n, int64_t k, float alpha,
                               const void *A, int64_t lda, const void *B, int64_t ldb, float beta,
                               void *C, int64_t ldc, bm_ctype c_type, void *workspace, size_t workspace_bytes,
                               bm_stream_t stream);

/* Bytes of workspace that bm_syr2k_bf16 would use for this shape (0 = none). */
BM_API size_t bm_syr2k_bf16_workspace_size(bm_uplo uplo, int64_t n, int64_t k);

/*
 * Device-side errors. Every wait inside the kernels (on a shared-memory
 * barrier) gives up after the wait limit, records BM_ERR_TIMEOUT in the
 * device status word, frees its tensor memory and returns, so that the CUDA
 * context stays usable. This call synchronises `stream`, reads and clears
 * the status word of the current device and returns it (BM_OK if none).
 */
BM_API bm_status bm_get_last_device_error(bm_stream_t stream);

/* Wait limit of the device-side barrier waits in milliseconds (default 2000). */
BM_API void bm_set_wait_timeout_ms(uint32_t ms);

/*
 * Test hook for the bounded waits (off by default). While enabled, every CTA
 * of the next GEMM/SYRK launches leaves its first operand copy unissued, so
 * the MMA warp's wait on that stage runs out: the kernel records
 * BM_ERR_TIMEOUT, frees its tensor memory and exits, and the context stays
 * usable. Pair it with a short bm_set_wait_timeout_ms.
 */
BM_API void bm_debug_inject_stall(int enable);

/*
 * Tile override for ablations and tests (process-wide; 0 = automatic choice,
 * the default). 1: 128 x 256 tiles on single SMs; 2: 128 x 128 tiles on single
 * SMs; 3: 256 x 256 tiles on SM pairs. bm_gemm_mxfp8 takes 1 as 128 x 128
 * tiles on single SMs, 2 as 256 x 128 tiles on SM pairs and 3 as 256 x 256
 * tiles on SM pairs. Results are identical up to FP32 summation order; only
 * speed changes. Returns BM_ERR_INVALID_VALUE for other values.
 */
BM_API bm_status bm_set_tile_override(int variant);

/* Human-readable name of a status code (static storage). */
BM_API const char *bm_status_string(bm_status status);

/*
 * Resolved launch plan of a GEMM or SYRK, for reports and tests: output tile
 * (tile_m x tile_n, k-block tile_k), ring stages (of stage_kblocks k-blocks
 * each), number of output tiles
 * visited, K splits and how many tiles are split (the tiles of a last, partly
 * filled wave: split along K and summed inside the GEMM kernel, or, for bf16
 * GEMMs on 256 x 256 pair tiles where no K split pays, run as two halves of
 * their columns on two SM pairs, n_splits == 2; or all tiles when there are too
 * few to fill the GPU, split along K and summed by a second kernel), CTAs
 * launched, CTAs per output tile (2 = an SM pair working on one tile), and the
 * number of kernels one call launches. Performs the same size checks as
 * the call (no pointers are given). On a machine without a usable GPU the
 * plan assumes 152 SMs. A GEMM's plan is the one for beta == 0: with
 * beta != 0 a tail split along K needs a larger saving, so such a call may
 * split its tail tiles into N halves instead (bm_gemm_bf16_workspace_size
 * covers both). The plan does not see C: a call whose rows of C do not end on
 * a 16-byte boundary runs tiles planned as N halves whole.
 */
typedef struct {
    int32_t tile_m, tile_n, tile_k;
    int32_t stages;
    int64_t tiles;
    int32_t k_splits;
    int32_t ctas;
    int32_t cta_pair;
    int32_t kernels;
    size_t workspace_bytes;
    int64_t split_tiles;
    int32_t stage_kblocks;
    int32_t n_splits;   /* 2: the split_tiles tiles each run as two halves of their columns (no partials) */
} bm_plan;

BM_API bm_status bm_gemm_bf16_plan(int64_t m, int64_t n, int64_t k, size_t workspace_bytes, bm_plan *plan);
BM_API bm_status bm_syrk_bf16_plan(bm_uplo uplo, int64_t n, int64_t k, size_t workspace_bytes, bm_plan *plan);
/* Plan of bm_gemm_mxfp8 (tile_k = 128: one k-block is 128 E4M3 elements). */
BM_API bm_status bm_gemm_mxfp8_plan(int64_t m, int64_t n, int64_t k, size_t workspace_bytes, bm_plan *plan);

/*
 * Visit order of the output tiles of a SYRK plan (the one bm_syrk_bf16_plan
 * reports for the same arguments and no workspace), for reports and tests: tile t of the
 * persistent schedule covers rows tile_row[t] * tile_m ... and columns
 * tile_col[t] * tile_n ... of C. The tiles across the diagonal come first, one
 * per tile row, then the tiles inside the triangle. With square tiles
 * (tile_m == tile_n) those go in groups of 16 tile rows of the lower triangle,
 * each group column by column and each column's rows in order; the upper
 * triangle takes the transpose (groups of 16 tile columns, each row by row).
 * With 128 x 256 tiles they go row by row. `count` must be the plan's `tiles`;
 * the two arrays are host memory of `count` elements.
 */
BM_API bm_status bm_syrk_bf16_tile_order(bm_uplo uplo, int64_t n, int64_t k, int64_t count, int64_t *tile_row,
                                         int64_t *tile_col);

/* Library version: major * 10000 + minor * 100 + patch. */
BM_API int bm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BM_H */
