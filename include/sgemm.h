/*
 * sgemm.h -- C ABI of the GB300 (sm_103a) single-precision GEMM library.
 *
 * Operation (the definition on the page "Deep dive into the sgemmNN
 * algorithm" (lazypool blog), section "Why SGEMM matters"; argument list in
 * the style of the sgemmNN kernel signature on the same page, section
 * "The whole kernel"):
 *
 *     C <- alpha * A * B + beta * C
 *
 * with A an M x K, B a K x N and C an M x N matrix of 32-bit floats, all
 * ROW-MAJOR with leading dimensions (element strides between rows):
 *
 *     A[i][p] = A[i*lda + p],  B[p][j] = B[p*ldb + j],  C[i][j] = C[i*ldc + j]
 *
 * (row-major as in the naive kernel of page m.lqnn.cn/news/94381, section
 * 1.1).  Accumulation is in FP32 on the GPU; the summation order is the
 * library's and is fixed per kernel variant, so repeated calls with the same
 * inputs and the same variant give bit-identical results.
 *
 * Conventions (BLAS, where the pages are silent):
 *   - beta == 0: C is output only and is never read (NaN/Inf in C do not
 *     propagate).
 *   - alpha == 0 or K == 0: A and B are not read (may be NULL); C <- beta*C.
 *   - M == 0 or N == 0: nothing is done; every pointer may be NULL.
 *   - Cells outside the M x K, K x N, M x N windows (columns K..lda-1 of A,
 *     N..ldb-1 of B, N..ldc-1 of C) are never read or written.
 *   - Any 4-byte-aligned pointer and any leading dimension is accepted.  An
 *     operand the TMA cannot read as stored (not 16-byte aligned, or its
 *     leading dimension -- or batch stride -- not a multiple of 4) is either
 *     read with scalar loads by the generic variant or first copied
 *     transposed, on the GPU, into the handle's re-layout workspace, which
 *     the TMA kernels then read (whichever the library estimates faster;
 *     see sgemm_relayout_t).  Never an error, never a CPU path.
 *
 * Column-major (BLAS / Fortran order) callers: a column-major m x n matrix
 * with leading dimension ld is the row-major n x m matrix of its transpose,
 * so the column-major product C = op(A) * op(B) is the row-major product
 * C^T = op(B)^T * op(A)^T: call sgemm_run_ex with the operands swapped
 * together with their trans flags and leading dimensions (B, transB, ldb
 * first; A, transA, lda second) and M and N swapped.
 *
 * Memory and streams: all matrix pointers are DEVICE pointers owned by the
 * caller.  sgemm_run never allocates and never synchronizes: it validates
 * its arguments on the host, enqueues kernels on `stream` (a cudaStream_t
 * cast to void*, NULL for the legacy default stream) and returns.  The
 * returned status covers only what is known at enqueue time; a fault found
 * later by a kernel is reported by sgemm_get_device_status.
 *
 * Threading: one handle may be used from one host thread at a time, and its
 * calls must be ordered on the GPU (one stream, or streams ordered by
 * events): calls of the same handle share its stream-K and re-layout
 * workspaces.  Use one handle per concurrently running stream.
 *
 * Every function returns an sgemm_status_t value (as int) unless noted.
 */
#ifndef SGEMM_H
#define SGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct sgemm_ctx *sgemm_handle_t;

typedef enum {
    SGEMM_OK = 0,
    SGEMM_ERR_NULL = 1,               /* a required pointer argument is NULL          */
    SGEMM_ERR_INVALID_VALUE = 2,      /* negative size, ld below its minimum, bad enum */
    SGEMM_ERR_ALIAS = 3,              /* C overlaps A or B                             */
    SGEMM_ERR_BAD_HANDLE = 4,         /* not a live handle (never created, destroyed)  */
    SGEMM_ERR_UNSUPPORTED_DEVICE = 5, /* current device is not compute capability 10.3 */
    SGEMM_ERR_LAUNCH = 6,             /* the kernel launch was rejected                */
    SGEMM_ERR_CUDA = 7,               /* another CUDA runtime error                    */
    SGEMM_ERR_DEVICE_TIMEOUT = 8,     /* a kernel gave up a bounded wait (device side) */
    SGEMM_ERR_WRONG_DEVICE = 9,       /* current device differs from the handle's      */
    SGEMM_ERR_SCRATCH_TOO_SMALL = 10, /* sgemm_run_noalloc: problem exceeds its scratch */
    SGEMM_ERR_DEVICE_CHECK = 11       /* a device-side index check failed (builds with
                                         -DSGEMM_DEVICE_CHECKS only)                    */
} sgemm_status_t;

/* Kernel variants.  SGEMM_VARIANT_AUTO lets sgemm_run choose from the shape
 * and the alignment of the operands; the others pin one variant (for tests
 * and measurements).  A pinned TMA variant on an operand the TMA cannot read
 * as stored runs on its transposed copy (the re-layout workspace), or, when
 * the re-layout is off or the copy does not fit, is replaced by the generic
 * variant for that call. */
typedef enum {
    SGEMM_VARIANT_AUTO = 0,
    SGEMM_VARIANT_TMA_128x256 = 1,   /* TMA-fed SIMT, 128 x 256 CTA tile, 8 x 16 per thread */
    SGEMM_VARIANT_TMA_128x128 = 2,   /* TMA-fed SIMT, 128 x 128 CTA tile, 8 x 8 per thread  */
    SGEMM_VARIANT_TMA_64x64 = 3,     /* TMA-fed SIMT, 64 x 64 CTA tile, 8 x 4 per thread    */
    SGEMM_VARIANT_TMA_64x64_SPLITK = 4, /* 64 x 64 tiles, stream-K over all tiles, fixed-order sum */
    SGEMM_VARIANT_GENERIC = 5,       /* scalar loads, any alignment, 64 x 64 CTA tile       */
    SGEMM_VARIANT_SCALE = 6,         /* reported only: the C <- beta*C quick path ran       */
    SGEMM_VARIANT_TC_3XTF32 = 7,     /* tensor cores (tcgen05, TMEM), 3xTF32 split precision,
                                        128 x 256 CTA tile; FP32 inputs, outputs, tolerance   */
    SGEMM_VARIANT_TC_3XTF32_PAIR = 8,/* as TC_3XTF32 on CTA pairs (cta_group::2): 256 x 256
                                        tile per cluster of two CTAs                          */
    SGEMM_VARIANT_TC_F16_PAIR = 9,   /* sgemm_run_mixed only: BF16 / FP16 A and B on the tensor
                                        cores (kind::f16), FP32 accumulation, CTA pairs       */
    SGEMM_VARIANT_GENERIC_F16 = 10,  /* sgemm_run_mixed only: the generic variant on 16-bit
                                        inputs (any alignment)                                */
    SGEMM_VARIANT_TMA_256x128 = 11,  /* TMA-fed SIMT, 256 x 128 CTA tile, 16 warps, 8 x 8 per
                                        thread (fastest on large problems)                    */
    SGEMM_VARIANT_COUNT_ = 12
    /* sgemm_run_ex: the TMA variants serve every (transA, transB) and any
     * batch up to 65535 when A and B are 16-byte aligned and lda, ldb (and,
     * for batch > 1, strideA, strideB) are multiples of 4, and operands that
     * are not through their transposed copies (above); otherwise the generic
     * variant runs.  The tensor-core variants serve every layout
     * and batches of up to 256 products (one launch per product): they read
     * A stored M x K and B stored K x N, and an operand stored transposed is
     * first copied into that layout in the re-layout workspace (one launch
     * per copy; see sgemm_relayout_t).  Where that cannot be done (a larger
     * batch, re-layout off, copies larger than the workspace) a pinned
     * tensor-core variant acts as AUTO. */
} sgemm_variant_t;

/* Arithmetic used by SGEMM_VARIANT_AUTO.  Both modes meet the same FP32
 * contract (max |C - C_exact| within 1e-3 for K <= 1024 and 1e-2 for K <= 8192
 * on U[-1,1) data).  SGEMM_MATH_FP32 (the default) runs FP32 FMAs on the CUDA
 * cores.  SGEMM_MATH_3XTF32 lets the library use the tensor cores with the
 * 3xTF32 split-precision method (A*B = A_hi*B_hi + A_hi*B_lo + A_lo*B_hi) for
 * problems large enough to profit; its rounding errors are larger than the
 * FP32 path's (about 5x at K = 8192) but still inside the contract.  In this
 * mode SGEMM_VARIANT_AUTO takes SGEMM_VARIANT_TC_3XTF32_PAIR when there are at
 * least SMs/4 tiles of 256 x 256 and K >= 256 and the tensor-core kernels can
 * serve the call (see sgemm_variant_t), and the FP32 kernels otherwise. */
typedef enum {
    SGEMM_MATH_FP32 = 0,
    SGEMM_MATH_3XTF32 = 1
} sgemm_math_mode_t;

/* Operand re-layout of the FP32 SIMT path (sgemm_run, sgemm_run_ex, any
 * batch; the tensor-core variants' copies into the NN
 * layout use the same workspace and are off with SGEMM_RELAYOUT_OFF).  A
 * strided batch is copied matrix by matrix (an operand with batch stride 0
 * once), each copy in its own slot of the workspace.  On GB300 the SIMT kernel's main loop is
 * fastest with A stored K x M and B stored K x N (transA = 1, transB = 0:
 * one 16-byte shared-memory load then gives one k of four rows of A).  The
 * library may therefore first copy A stored M x K, or B stored N x K,
 * transposed into the handle's re-layout workspace (an HBM-bound pass,
 * about 0.6 % of the time of an 8192^3 product) and run the GEMM on the
 * copy.  Every layout forms each product in ascending k with one rounding
 * per FMA, so with the same tile variant and the same stream-K plan the
 * result is bit-identical to the call without re-layout.
 * An operand the TMA cannot read as stored (see the conventions above) is
 * copied transposed whatever its stored layout, and the other operand as
 * the estimate prefers; the generic variant runs instead when its estimate
 * is lower (small problems: about 9 us of fixed cost against the copies'
 * launches).
 *   SGEMM_RELAYOUT_AUTO (default): when the library's time estimate of the
 *     copies plus the faster kernel beats the kernel on the operands as
 *     stored by at least 1 % and the copies fit in the workspace (an
 *     operand the TMA cannot read: when they fit and beat the generic
 *     variant);
 *   SGEMM_RELAYOUT_OFF: never (an operand the TMA cannot read: the generic
 *     variant);
 *   SGEMM_RELAYOUT_ALWAYS: whenever the copies that reach transA = 1,
 *     transB = 0 fit in the workspace (tests, measurements). */
typedef enum {
    SGEMM_RELAYOUT_AUTO = 0,
    SGEMM_RELAYOUT_OFF = 1,
    SGEMM_RELAYOUT_ALWAYS = 2
} sgemm_relayout_t;

/* Element type of A and B for sgemm_run_mixed (C is always FP32). */
typedef enum {
    SGEMM_IN_BF16 = 1,  /* bfloat16: 1 sign, 8 exponent, 7 fraction bits */
    SGEMM_IN_F16 = 2    /* IEEE binary16 */
} sgemm_input_t;

/* Create a handle bound to the CURRENT CUDA device.  Requires compute
 * capability 10.3 (GB300); otherwise returns SGEMM_ERR_UNSUPPORTED_DEVICE and
 * sets *out to NULL.  Allocates the handle's device-side status word, its
 * stream-K workspace (48 MiB) and arrival counters (zeroed), and its operand
 * re-layout workspace (512 MiB: the transposes of an 8192 x 8192 A and B;
 * if that allocation fails the handle is created without it and never
 * re-lays out), and sets the kernels' shared-memory limits.  `out` must be
 * non-NULL (else SGEMM_ERR_NULL). */
int sgemm_create(sgemm_handle_t *out);

/* C <- alpha*A*B + beta*C, enqueued on `stream`; see the conventions above.
 * Argument checks, in order: handle (SGEMM_ERR_BAD_HANDLE), current device
 * (SGEMM_ERR_WRONG_DEVICE), then the rules of sgemm_check_args.  On any
 * error nothing is enqueued and C is unchanged. */
int sgemm_run(sgemm_handle_t h, int M, int N, int K, float alpha,
              const float *A, int lda, const float *B, int ldb,
              float beta, float *C, int ldc, void *stream);

/* The general form: C_b <- alpha * op(A_b) * op(B_b) + beta * C_b for b = 0 ..
 * batch-1, where op(X) = X (trans = 0) or X^T (trans = 1), op(A) is M x K,
 * op(B) is K x N, and matrix b of each operand starts `stride` elements after
 * matrix b-1 (X_b = X + b*strideX).  Row-major storage as above: A is stored
 * M x K (lda >= max(1, K)) when transA = 0 and K x M (lda >= max(1, M)) when
 * transA = 1; B is stored K x N (ldb >= max(1, N)) when transB = 0 and N x K
 * (ldb >= max(1, K)) when transB = 1.  `sgemm_run` is the case transA = transB
 * = 0, batch = 1.  Strides must be >= 0; with batch > 1 the C matrices must not
 * overlap one another (strideC at least the extent of one C window), else
 * SGEMM_ERR_INVALID_VALUE.  batch == 0 is a no-op.  The pages' sgemmNN kernel
 * (page "Deep dive into the sgemmNN algorithm") is the NN case; the transposed
 * and batched forms are the BLAS / cuBLAS conventions the pages' batched call
 * (page "GPU-accelerated matrix computation optimisation and CUDA programming
 * practice", section 4.2) uses. */
int sgemm_run_ex(sgemm_handle_t h, int transA, int transB, int M, int N, int K, float alpha,
                 const float *A, int lda, long long strideA, const float *B, int ldb, long long strideB,
                 float beta, float *C, int ldc, long long strideC, int batch, void *stream);

/* Host-only validation of sgemm_run_ex's arguments (same rules, no CUDA call). */
int sgemm_check_args_ex(int transA, int transB, int M, int N, int K, float alpha, const float *A, int lda,
                        long long strideA, const float *B, int ldb, long long strideB, float beta,
                        const float *C, int ldc, long long strideC, int batch);

/* Mixed precision: C <- alpha * op(A) * op(B) + beta * C with A and B holding
 * 16-bit values (`in_type`: SGEMM_IN_BF16 or SGEMM_IN_F16; 2 bytes per element,
 * leading dimensions in elements) and C in FP32.  op and the stored shapes as
 * in sgemm_run_ex (batch 1).  Every product of two 16-bit values is exact in
 * FP32; the products are summed in FP32 (on the tensor cores, whose FP32
 * accumulation is not round-to-nearest), then alpha, beta and C as in
 * sgemm_run.  Error contract: max |C - C_exact| within 1e-3 for K <= 1024
 * and 1e-2 for K <= 8192 on inputs of magnitude <= 1, where C_exact is the
 * exact result for the 16-bit inputs as given (the caller's rounding to 16 bits
 * is not part of it).  Page "GPU-accelerated matrix computation optimisation
 * and CUDA programming practice", section 4.1, uses this split (16-bit inputs,
 * FP32 accumulation) through a library call; here it is a kernel of this
 * library.  Runs SGEMM_VARIANT_TC_F16_PAIR when A and B are 16-byte aligned and
 * lda, ldb are multiples of 8, else SGEMM_VARIANT_GENERIC_F16 (a pinned
 * GENERIC variant also selects it).  Errors as sgemm_run_ex, plus
 * SGEMM_ERR_INVALID_VALUE for an unknown in_type. */
int sgemm_run_mixed(sgemm_handle_t h, int in_type, int transA, int transB, int M, int N, int K, float alpha,
                    const void *A, int lda, const void *B, int ldb, float beta, float *C, int ldc, void *stream);

/* Host-only validation of sgemm_run_mixed's arguments (same rules, no CUDA call). */
int sgemm_check_args_mixed(int in_type, int transA, int transB, int M, int N, int K, float alpha, const void *A,
                           int lda, const void *B, int ldb, float beta, const float *C, int ldc);

/* C <- alpha*A*B + beta*C with A, B, C in HOST memory, transfers overlapped
 * with compute.  dA, dB, dC are caller-owned DEVICE buffers of the same
 * shapes and leading dimensions (M*lda, K*ldb, M*ldc floats at least).  On a
 * handle-owned copy stream the library copies the first row panel of A (and
 * of C when beta != 0), then B in up to 8 column chunks, then the other row
 * panels; on `stream` it runs each piece of the GEMM (the same kernels and
 * rules as sgemm_run) as soon as its operands have landed -- the first row
 * panel in column blocks as B's chunks arrive, the middle panels as one
 * GEMM (two from four middle panels on, each started once its own panels
 * have landed), the last panel in column blocks; each segment's A rows may first be
 * copied transposed into the handle's re-layout workspace, once for all of
 * the segment's GEMMs -- and on a second copy stream it copies each finished
 * piece back to C while the rest computes.  Returns after enqueueing; C is complete when `stream`
 * reaches the point of the call (e.g. after cudaStreamSynchronize(stream)).
 * Page-locked host buffers give asynchronous copies; pageable ones work but
 * serialise.  The host and device windows must not be touched until then.
 * Same argument checks as sgemm_run (on the device pointers; SGEMM_ERR_NULL
 * also if a host pointer that is read or written is NULL), made before
 * anything is enqueued.  A CUDA error while enqueueing (after the checks)
 * returns SGEMM_ERR_CUDA with part of the copies and GEMMs possibly already
 * enqueued; synchronize `stream` before reusing the buffers.  The handle's
 * copy streams and events serve one call at a time: calls of the same handle
 * from several host threads must be serialised.  No allocation. */
int sgemm_run_host(sgemm_handle_t h, int M, int N, int K, float alpha,
                   const float *A, int lda, const float *B, int ldb,
                   float beta, float *C, int ldc,
                   float *dA, float *dB, float *dC, void *stream);

/* Host-only validation with exactly the rules sgemm_run applies (no CUDA call,
 * no handle): SGEMM_ERR_INVALID_VALUE if M, N or K < 0, lda < max(1, K),
 * ldb < max(1, N) or ldc < max(1, N); then, unless M == 0 or N == 0,
 * SGEMM_ERR_NULL if C is NULL, or if A or B is NULL while alpha != 0 and
 * K > 0; then SGEMM_ERR_ALIAS if the byte range of C's window overlaps that
 * of A's or B's window (only when A, B are read). */
int sgemm_check_args(int M, int N, int K, float alpha, const float *A, int lda,
                     const float *B, int ldb, float beta, const float *C, int ldc);

/* Synchronize the handle's device, then destroy it and free its device
 * memory.  SGEMM_ERR_BAD_HANDLE for NULL or an already destroyed handle. */
int sgemm_destroy(sgemm_handle_t h);

/* Pin a kernel variant for later calls of this handle (SGEMM_VARIANT_AUTO to
 * let the library choose).  SGEMM_ERR_INVALID_VALUE for an unknown value or
 * SGEMM_VARIANT_SCALE, which is chosen only by the alpha == 0 / K == 0 rule.
 * A pinned TMA variant fixes the tile; the re-layout mode still decides
 * whether operands are transposed first.  The 16-bit-input variants act as
 * SGEMM_VARIANT_AUTO for FP32 calls. */
int sgemm_set_variant(sgemm_handle_t h, int variant);

/* Set the handle's math mode (an sgemm_math_mode_t) for SGEMM_VARIANT_AUTO.
 * SGEMM_ERR_INVALID_VALUE for an unknown mode. */
int sgemm_set_math_mode(sgemm_handle_t h, int mode);

/* Set the handle's operand re-layout mode (an sgemm_relayout_t).
 * SGEMM_ERR_INVALID_VALUE for an unknown mode. */
int sgemm_set_relayout(sgemm_handle_t h, int mode);

/* Operands the handle's last successful sgemm_run / sgemm_run_ex copied
 * transposed before the GEMM: bit 0 A, bit 1 B (0 for none); -1 if `h` is
 * not a live handle. */
int sgemm_last_relayout(sgemm_handle_t h);

/* Size of the handle's re-layout workspace in floats (0 if it could not be
 * allocated, and then no operand is re-laid out); -1 if `h` is not a live
 * handle.  Transposed copies are stored with leading dimensions rounded up
 * to a multiple of 32 floats: A needs K * ceil32(M) floats per batch matrix,
 * B K * ceil32(N), both together the sum (the tensor-core variants' copies:
 * M * ceil32(K) for A, K * ceil32(N) for B). */
int64_t sgemm_relayout_capacity(sgemm_handle_t h);

/* The variant the handle's last successful sgemm_run enqueued (an
 * sgemm_variant_t), or -1 if there was none or `h` is not a live handle.
 * *splits (if non-NULL) receives the number of CTAs that share the K range of
 * a stream-K tile (rounded up; 1 when no tile was split). */
int sgemm_last_variant(sgemm_handle_t h, int *splits);

/* Number of kernel launches the handle's last successful sgemm_run /
 * sgemm_run_ex enqueued: 0 (nothing to do), one per transposed operand
 * (sgemm_last_relayout), then 1 to 3 for the GEMM: complete waves of whole
 * tiles; the stream-K CTAs of the last wave; and, for tiles larger than
 * 64 x 64, the kernel that adds the stream-K parts.  All on the same stream.
 * The 3xTF32 kernels: one launch per batch product after its copies.
 * -1 if `h` is not a live handle. */
int sgemm_last_launches(sgemm_handle_t h);

/* Wait for the handle's device to finish its work, then read and clear the
 * handle's device-side status word.  Returns SGEMM_OK, or
 * SGEMM_ERR_DEVICE_TIMEOUT if any kernel of the handle abandoned a bounded
 * wait, SGEMM_ERR_DEVICE_CHECK if a device-side index check failed (builds
 * with -DSGEMM_DEVICE_CHECKS; the check replaces the index with one in range,
 * so nothing is accessed out of bounds), or SGEMM_ERR_CUDA.  After a timeout the C of the calls since the last
 * check is undefined: some tiles may be unwritten and some may hold partial
 * sums or stale workspace contents.  On a timeout or a failed check this
 * call also clears the handle's stream-K arrival counters (a CTA that gave up
 * leaves its tile's counter unreset), so later calls on the handle are
 * correct again. */
int sgemm_get_device_status(sgemm_handle_t h);

/* Test hook: the stream-K workspace capacity, in partial tiles, that later
 * calls of the handle pass to their kernels for the device-side index checks
 * (0: the workspace's real size).  The plan still uses the real size, so a
 * limit below what a call needs makes a build with -DSGEMM_DEVICE_CHECKS
 * report SGEMM_ERR_DEVICE_CHECK for it -- every access stays inside the real
 * workspace -- and changes nothing in a build without the checks. */
int sgemm_debug_set_workspace_limit(sgemm_handle_t h, int tiles);

/* Test hook: put the handle in the state that a stream-K kernel which gave
 * up a bounded wait can leave behind -- every arrival counter nonzero and
 * the timeout bit set in the status word -- without running any kernel.
 * sgemm_get_device_status must then report the timeout and restore the
 * counters.  Synchronizes the device. */
int sgemm_debug_leave_aborted_state(sgemm_handle_t h);

/* Test hook: enqueue one small kernel that waits on a barrier nothing will
 * complete, gives up after `limit_ns` nanoseconds (clamped to [1e3, 1e9]),
 * records SGEMM_ERR_DEVICE_TIMEOUT in the handle's status word and returns.
 * It exercises the timeout path without faulting or hanging the GPU. */
int sgemm_debug_timeout_probe(sgemm_handle_t h, long long limit_ns, void *stream);

/* Measurement probe: enqueue `ctas` CTAs (0 = 4 per SM) of 256 threads, each
 * thread running 16 independent chains of packed FP32x2 FMAs for 8*iters
 * steps in registers (no memory traffic) and writing one sum to
 * sink[thread] (device memory of ctas*256 floats, caller-owned), and set
 * *flops (if non-NULL) to the FLOP the launch performs.  Timed with events
 * it gives the FP32 FMA rate the GEMM main loop is compared with.
 * SGEMM_ERR_NULL for a NULL sink; SGEMM_ERR_INVALID_VALUE if ctas < 0 or
 * iters < 1. */
int sgemm_debug_fma_probe(sgemm_handle_t h, int ctas, int iters, float *sink, long long *flops, void *stream);

/* Measurement probe of the TF32 tensor pipe: enqueue `clusters` clusters of
 * two CTAs (0 = one per pair of SMs; at most SMs/2), each issuing `iters`
 * K = 32 steps of the 3xTF32 CTA-pair kernel's MMA (tcgen05.mma
 * cta_group::2 kind::tf32, M = 256, N = 256, four K = 8 MMAs a step) on
 * operand tiles resident in shared memory, with no global-memory traffic,
 * and set *flops (if non-NULL) to the TF32 FLOP the launch performs.  Timed
 * with events it gives the measured TF32 rate; the 3xTF32 path spends three
 * TF32 MMAs per FP32 product, so its roofline is a third of it.  A wait that
 * runs out (bounded) is recorded in the handle's status word.
 * SGEMM_ERR_INVALID_VALUE if clusters < 0 or > SMs/2, or iters outside
 * 1 .. 2^20; SGEMM_ERR_WRONG_DEVICE off the handle's device. */
int sgemm_debug_tf32_probe(sgemm_handle_t h, int clusters, int iters, long long *flops, void *stream);

/* Measurement probe: `ctas` one-warp CTAs (0 = one per SM) each fill a 32 x 32
 * FP32 tile in shared memory with 0.001*(32*row + column) and read it
 * column-wise (lane l reads row l, k = 0..31) `iters` times -- the
 * transposed-operand access of page m.lqnn.cn/news/94381, section 4.2 -- with
 * a row stride of 32 floats (padded = 0: all 32 lanes in one bank, a 32-way
 * conflict per load) or 33 (padded = 1, the page's padding: 32 distinct
 * banks); lane l of CTA c writes its sum to sink[32*c + l] (ctas*32 floats,
 * caller-owned).  A control for the profiler's bank-conflict counters. */
int sgemm_debug_bank_probe(sgemm_handle_t h, int padded, int ctas, int iters, float *sink, void *stream);

/* Test hook: when `bytes` > 0, later launches of the handle's TMA variants
 * request `bytes` of dynamic shared memory instead of their own size, so a
 * value above the device limit makes the launch fail on the host
 * (SGEMM_ERR_LAUNCH) before anything runs.  0 restores normal launches. */
int sgemm_debug_set_smem_override(sgemm_handle_t h, int bytes);

/* How a call adds the partial sums of a tile whose K range is split over
 * stream-K CTAs (sgemm_debug_set_stream_k_sums).  Every mode adds a tile's
 * parts in ascending k order, so a tile split the same way gets the same
 * bits in every mode. */
typedef enum {
    SGEMM_SK_SUMS_AUTO = 0,     /* the library's choice (default) */
    SGEMM_SK_SUMS_LAST = 1,     /* the last CTA of the tile to arrive adds them all; the larger tiles
                                   split from 1.25 stream-K CTAs per tile as the 64 x 64 tile does */
    SGEMM_SK_SUMS_DEFERRED = 2, /* tiles larger than 64 x 64: every part stays in the workspace and a
                                   second kernel adds them (64 x 64 tiles: as LAST) */
    SGEMM_SK_SUMS_SHARED = 3    /* the CTAs whose K range ends in the tile wait for all its parts and
                                   add one slice of its elements each (every tile size) */
} sgemm_sk_sums_t;

/* Test hook: how later calls of the handle add the partial sums of a tile
 * whose K range is split over stream-K CTAs (sgemm_sk_sums_t).  Automatic:
 * for the tiles larger than 64 x 64, whichever of a second kernel and the
 * shared sums the library's time estimate prefers (and stream-K only where
 * it beats whole tiles); for the 64 x 64 tiles, whichever of the last CTA of
 * the tile to arrive and the shared sums it prefers (the last CTA reads the
 * parts one after another, which costs with many parts a tile).  The other
 * modes take the stream-K tail whenever a wave
 * has CTAs to spare (LAST: 1.25 per tile), so that every mode splits a call
 * the same way.  SGEMM_ERR_INVALID_VALUE for another value. */
int sgemm_debug_set_stream_k_sums(sgemm_handle_t h, int mode);

/* Test hook: cluster split-K CTAs per tile for later calls of the handle on
 * the whole-tile SIMT variants.  In cluster split-K, the `ksplit` CTAs of one
 * output tile form a thread-block cluster; CTA r takes K steps
 * [r*kt/ksplit, (r+1)*kt/ksplit) of the tile's kt steps of 32, the partial
 * tiles meet in distributed shared memory and each CTA adds a 1/ksplit slice
 * of them in ascending k order and writes it to C (one launch, no workspace).
 * 0 (the default): the library's choice, taken when all tiles x ksplit CTAs
 * fit in one wave and its time estimate beats whole tiles and stream-K.
 * 1: never.  2..8: that many CTAs per tile whenever K has at least as many
 * steps.  A tile split into ksplit parts this way gets the bits of the same
 * split through stream-K (ksplit * tiles stream-K CTAs).
 * SGEMM_ERR_INVALID_VALUE outside 0..8. */
int sgemm_debug_set_cluster_split(sgemm_handle_t h, int ksplit);

/* Test hook: the number of stream-K CTAs of later calls' stream-K plans (the
 * last wave of the whole-tile variants, and the 64 x 64 split variant); 0 (the
 * default): the library's choice.  The count is kept within what a plan
 * allows -- more CTAs than the tail has tiles (the split variant: at least
 * two per tile), at most a wave of them and the workspace's partial tiles --
 * and a call whose plan has no stream-K part is unaffected.
 * SGEMM_ERR_INVALID_VALUE for a negative count. */
int sgemm_debug_set_stream_k_ctas(sgemm_handle_t h, int ctas);

/* Test hook: how the stream-K CTAs of later calls of the handle share the K
 * steps of the tiles they split.  The K steps lie on a line, 16 positions
 * each, with `gap` positions of no work before every tile but the first; CTA
 * q of G takes the K steps whose last position falls in its equal share
 * [gap + floor(q*V/G), gap + floor((q+1)*V/G)) of the V positions.  A CTA whose
 * range runs into a further tile stores one more partial tile, and the gap
 * charges it for that with fewer K steps.  gap = 0 is the even split
 * (floor(q*T/G) .. floor((q+1)*T/G) of the T K steps).  -1 (the default): the
 * library's choice among 0, 4, .., 24, the one whose busiest CTA has the least
 * work by its estimate; 0..128: that charge, where every CTA then gets at
 * least one and at most a tile's K steps (else 0).  Any charge gives a valid
 * split whose tiles' parts are added in ascending k order; splits differ in
 * where a tile's K range is cut, so results of different charges may differ
 * in the last bits.  SGEMM_ERR_INVALID_VALUE outside -1..128. */
int sgemm_debug_set_stream_k_gap(sgemm_handle_t h, int gap);

/* Test hook: the plan sgemm_run_ex would follow for a call, computed on the
 * host with no handle, no device and no CUDA call, from the device facts a
 * handle records (`num_sms`; `ctas_per_sm`, SGEMM_VARIANT_COUNT_ entries
 * indexed by sgemm_variant_t: resident CTAs per SM of each TMA variant) and
 * its settings (re-layout workspace size in floats, re-layout mode, math
 * mode, pinned variant).  `aligned` says which operands the TMA can read as
 * stored: bit 0 A, bit 1 B, each set when the operand is 16-byte aligned with
 * its leading dimension (and batch stride) a multiple of 4 (3: both, as for
 * any call on 16-byte aligned buffers with such leading dimensions).  An
 * operand it cannot read is copied transposed into the re-layout workspace
 * when the mode allows and the copy fits and pays; else the call runs on the
 * generic kernel.  out[0..12] receives: the
 * kind (0 nothing to do, 1 the beta*C quick path, 2 tensor-core kernel, 3
 * generic kernel, 4 TMA SIMT kernel), the variant that runs, the operands
 * copied transposed first (bit 0 A, bit 1 B), the TMA operand layout (0 NN,
 * 1 TN, 2 NT), the whole tiles run in complete waves, the stream-K CTAs, the
 * tiles of the call, the kernel launches, the CTAs per stream-K tile, and how
 * the stream-K tiles' parts are added (0 by the last CTA of each tile to
 * arrive, or without stream-K; 1 by a second kernel; 2 shared by the CTAs
 * whose K range ends in the tile), the cluster split-K CTAs per tile (1:
 * none), 1 when the 3xTF32 pair kernel reads B stored N x K (an operand
 * stored K x N is then copied transposed first; 0: B stored K x N), and the
 * stream-K split's boundary charge (sgemm_debug_set_stream_k_gap; 0: the
 * even split, or no stream-K).
 * SGEMM_ERR_NULL for a NULL array, SGEMM_ERR_INVALID_VALUE for an argument out
 * of range. */
int sgemm_debug_plan(int num_sms, const int *ctas_per_sm, long long relayout_floats, int relayout_mode,
                     int math_mode, int pinned, int transA, int transB, int M, int N, int K, float alpha,
                     int batch, long long strideA, long long strideB, int aligned, int *out);

/* C <- alpha*A*B + beta*C without allocating anything, for callers that cannot
 * allocate GPU memory (allocator implementations that must not re-enter the
 * allocator, frameworks whose allocator has reserved the device memory, hosts
 * that forbid device allocation after start-up).  The pages have no
 * counterpart: this is a deployment convenience, not part of the method.
 *
 * Same arguments, rules and results as sgemm_run, but no handle: it runs the
 * 64 x 64 stream-K kernel with its partial tiles, tile counters and status word
 * in a fixed scratch array compiled into the library (8 MiB + 4 KiB + 256 B,
 * held on every GPU that loads the library until the process exits).
 * Limit: at most 512 output tiles of 64 x 64, i.e. ceil(M/64)*ceil(N/64) <= 512;
 * larger problems return SGEMM_ERR_SCRATCH_TOO_SMALL and enqueue nothing.
 * alpha == 0 or K == 0, and operands TMA cannot describe, take the same
 * scratch-free kernels as sgemm_run.  It calls no cudaMalloc or cudaFree.
 * All calls share the scratch and it keeps the last call's contents: each call
 * clears the counters and status word it uses on `stream` first, and calls that
 * overlap on the GPU (unordered streams) race and give wrong results.  The
 * first call on a device, with that device current, looks up the scratch's
 * device address and sets the kernel up; make that first call before any
 * stream capture, and do not reset the device (cudaDeviceReset) between
 * calls: the address found is kept for the life of the process.  A
 * device-side timeout leaves the tiles it hit unwritten and cannot be
 * reported by this entry point. */
int sgemm_run_noalloc(int M, int N, int K, float alpha, const float *A, int lda,
                      const float *B, int ldb, float beta, float *C, int ldc, void *stream);

/* Human-readable name of a status value (never NULL). */
const char *sgemm_status_string(int status);

/* Human-readable name of a variant value (never NULL). */
const char *sgemm_variant_name(int variant);

/* Library version, major*10000 + minor*100 + patch. */
int sgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_H */
