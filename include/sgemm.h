/*
 * sgemm.h -- C ABI of the GB300 (sm_103a) single-precision GEMM library.
 *
 * Operation.  C = A * B for row-major FP32 matrices, A (M x K), B (K x N),
 * C (M x N):  C[m, n] = sum over k of A[m, k] * B[k, n], accumulated with
 * FP32 fused multiply-adds (no TF32, no reduced-precision tensor path).
 * Definition: "Beyond Kernel 7: Closing the Gap to cuBLAS on an H100 FP32
 * GEMM", section "The operation: GEMM and the precision of the comparison"
 * (C[m, n] = sum_k A[m, k] B[k, n]; only A*B is computed, i.e. alpha = 1 and
 * beta = 0; about 2MNK operations, an FFMA counting as two).  Row-major
 * storage follows the same page's "Kernel 1" section; element (r, c) of a
 * matrix with row stride ld sits at base[r * ld + c].
 *
 * Memory and ownership.  A, B and C are DEVICE pointers owned by the caller
 * (except for sgemm_host(), which takes host memory and copies it itself);
 * the library never frees or retains them past the call.  C must not overlap
 * A or B.  C is write-only: its previous contents (NaN included) are never
 * read.  All calls are asynchronous on `stream` (0 = legacy default stream):
 * they return once the kernels are enqueued.
 *
 * Scratch.  Shapes that the split-K (Stream-K) schedule serves use a device
 * workspace.  sgemm()/sgemm_variant() take it from a cache the library keeps
 * per (device, stream): the first call that needs more than the cache holds
 * allocates it with cudaMalloc (so make that first call outside stream
 * capture); later calls reuse it.  A workspace replaced by a larger one is not
 * freed but kept until sgemm_release_workspaces(), so kernels still running
 * and CUDA graphs captured while it was current keep valid memory; a graph
 * captured with these calls must not be replayed after
 * sgemm_release_workspaces().  Calls on one stream are ordered; calls on
 * different streams use different workspaces.  Calls on one stream must not
 * be made from several host threads at the same time: the staged variant
 * copies operands into the workspace in a launch of its own, and another
 * thread's call enqueued in between would overwrite them.  Threads on
 * different streams are safe.  sgemm_release_workspaces() frees the cache.
 * Independently of that cache, the library's device image holds a fixed
 * 32 MiB array (the scratch of sgemm_streamk_static()); every process that
 * initialises a device with any entry point holds it on that device until it
 * exits, whether or not it ever calls sgemm_streamk_static().
 *
 * Errors.  Every entry point returns an sgemm_status_t and never aborts the
 * process.  Argument errors are found on the host before any launch.  A
 * device-side wait that exceeds its time limit (a pipeline that stopped
 * making progress) makes the kernel record SGEMM_ERR_TIMEOUT in a device
 * status word and return early instead of hanging; read it with
 * sgemm_query_device_status().
 */
#ifndef GB300_SGEMM_H
#define GB300_SGEMM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SGEMM_OK = 0,
  SGEMM_ERR_INVALID_VALUE = 1, /* negative size, ld too small, NULL with nonzero extent, bad variant */
  SGEMM_ERR_LAUNCH = 2,        /* a CUDA launch or API call failed (see cudaGetLastError) */
  SGEMM_ERR_TIMEOUT = 3,       /* a kernel's bounded wait expired; its output is not valid */
  SGEMM_ERR_UNSUPPORTED = 4,   /* no sm_103a device, or a size beyond 2^31 - 1 */
  SGEMM_ERR_ALLOC = 5          /* the workspace cache could not be allocated */
} sgemm_status_t;

/* Kernel variants, for sgemm_variant() and sgemm_select_variant(). */
typedef enum {
  SGEMM_VARIANT_AUTO = -1,     /* let the selector choose (what sgemm() does) */
  SGEMM_VARIANT_GUARDED = 0,   /* any shape, stride and alignment; bounds-checked scalar loads */
  SGEMM_VARIANT_TILED = 1,     /* pipelined 128x256 tiles, one output tile per CTA, no split */
  SGEMM_VARIANT_STREAMK = 2,   /* persistent CTAs: whole tiles in full waves, the rest split over K */
  SGEMM_VARIANT_TILED_SMALL = 3,   /* pipelined 128x128 tiles, one output tile per CTA */
  SGEMM_VARIANT_STREAMK_SMALL = 4, /* Stream-K schedule over 128x128 tiles */
  SGEMM_VARIANT_STAGED = 5,    /* any stride and alignment: unaligned A, B copied aligned first */
  SGEMM_VARIANT_SPECIALIZED = 6, /* Stream-K compiled for one exact shape (768^3 ... 4096^3) */
  SGEMM_VARIANT_SMALL = 7,     /* small products: 64x64 tiles, K split over CTAs, plain loads */
  SGEMM_VARIANT_COUNT = 8
} sgemm_variant_t;

/*
 * C = A * B.  M, N, K >= 0; lda >= K, ldb >= N, ldc >= N (elements).
 * M == 0 or N == 0: nothing to do, SGEMM_OK.  K == 0: C is filled with zeros
 * (the empty sum).  Any stride and alignment is accepted.  The pipelined
 * kernels read A and B by TMA, and the small-product kernel (SMALL, chosen
 * for products up to roughly 640^3 and for thin or deep shapes whose tiles
 * would leave SMs idle) with 128-bit loads: both need 16-byte-aligned base
 * addresses and row strides that are multiples of 4 floats.  An operand
 * without that property (for instance a contiguous matrix with an odd number
 * of columns) is either first copied into an aligned buffer in the workspace
 * (the staged variant; a C without it is then written with 4-byte stores) or
 * the whole product runs in the bounds-checked kernel, whichever the
 * selector estimates to be faster: the staged variant for all but very small
 * products.  Every variant gives the same result on every call (summation
 * orders are fixed); different variants may differ in rounding.
 */
sgemm_status_t sgemm(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                     const float *B, int64_t ldb, float *C, int64_t ldc, cudaStream_t stream);

/* Storage order of the operands of sgemm_ex(). */
typedef enum {
  SGEMM_ROW_MAJOR = 0, /* element (r, c) at base[r * ld + c] */
  SGEMM_COL_MAJOR = 1  /* element (r, c) at base[r + c * ld] */
} sgemm_layout_t;

/*
 * C = alpha * A * B + beta * C, the general form whose epilogue the pages
 * print ("Vectorized Memory Access ...", section 5: alpha * acc + beta * C;
 * "2D Block Tiling ...", section 5).  `layout` (an sgemm_layout_t) applies to
 * A, B and C alike; leading dimensions are row strides for SGEMM_ROW_MAJOR
 * (lda >= K, ldb >= N, ldc >= N) and column strides for SGEMM_COL_MAJOR
 * (lda >= M, ldb >= K, ldc >= M).  beta == 0 never reads C (NaN there does
 * not propagate); alpha == 0 or K == 0 gives C = beta * C without reading A
 * or B.  Column-major problems run as the row-major C^T = B^T A^T over the
 * same memory.  Otherwise as sgemm(): same kernels, selector, workspace and
 * error behaviour; sgemm(...) is sgemm_ex(SGEMM_ROW_MAJOR, ..., 1, ..., 0, ...).
 */
sgemm_status_t sgemm_ex(int layout, int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                        int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                        int64_t ldc, cudaStream_t stream);

/* Transposition of one operand of sgemm_ex2(). */
typedef enum {
  SGEMM_OP_N = 0, /* op(X) = X */
  SGEMM_OP_T = 1  /* op(X) = X^T */
} sgemm_op_t;

/*
 * C = alpha * op(A) * op(B) + beta * C with a transposition flag per operand
 * (each an sgemm_op_t): the general form of sgemm_ex(), with the alpha/beta
 * epilogue the pages print ("Vectorized Memory Access ...", section 5;
 * "2D Block Tiling ...", section 5) and the transposed / column-major operand
 * layouts of "cuSgemm" (Kernel 7 takes column-major operands).  op(A) is
 * M x K and op(B) is K x N.  The memory holds the stored matrices: A is M x K
 * when trans_a == SGEMM_OP_N and K x M when SGEMM_OP_T (op(A) = A^T); B is
 * K x N or N x K likewise.  `layout` applies to the stored A, B and C; the
 * leading dimensions are the stored matrices' (row strides for
 * SGEMM_ROW_MAJOR, column strides for SGEMM_COL_MAJOR), so for instance a
 * row-major A with trans_a == SGEMM_OP_T needs lda >= M.
 *
 * How each operand reaches the kernels (row-major view; a column-major
 * problem runs as the row-major C^T = op(B)^T op(A)^T over the same memory):
 * a transposed A is read in place by the pipelined kernels as an M-major
 * tile (TMA, no copy) when it is 16-byte aligned with lda a multiple of 4,
 * and otherwise (or for the small-product kernel) transposed into the
 * workspace first; a transposed B is always transposed into the workspace
 * first (about 8 bytes of HBM traffic per element and one extra launch).
 * sgemm_ex2 with two SGEMM_OP_N flags is sgemm_ex().  Errors, workspace and
 * C semantics as for sgemm_ex(); a flag other than SGEMM_OP_N or SGEMM_OP_T
 * returns SGEMM_ERR_INVALID_VALUE.
 */
sgemm_status_t sgemm_ex2(int layout, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                         float alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
                         float beta, float *C, int64_t ldc, cudaStream_t stream);

/*
 * C = A * B as sgemm(), with A, B and C in HOST memory: the copies to the
 * current device and back happen inside the call.  The product is the one
 * of "Beyond Kernel 7: Closing the Gap to cuBLAS on an H100 FP32 GEMM",
 * "The operation"; results are within the same bound as sgemm()'s (rows of C
 * are computed by separate launches, so bits may differ from one sgemm() call
 * over the whole product).
 *
 * Layout: row-major, element row strides lda >= K, ldb >= N, ldc >= N (any
 * alignment).  The library copies B whole, then A in row panels (one panel
 * below M = 2048, else M / 6 rows but at least 512) on a copy stream of its
 * own.  It multiplies each panel on `stream` as soon as its rows have landed,
 * and copies that panel's rows of C back on a second copy stream while the
 * next panel is multiplied.
 *
 * Ownership and ordering: asynchronous on `stream` like cudaMemcpyAsync.
 * The call returns once everything is enqueued, and C holds the product
 * when `stream` has completed; A, B and C must stay valid and unmodified
 * (C unread) until then.  Nothing of the call starts before work queued
 * earlier on `stream` has completed.  Page-locked host memory
 * (cudaHostAlloc, cudaHostRegister) gives asynchronous, overlapped copies.
 * Pageable memory works too, but CUDA may then make the copies synchronous.
 * C must not overlap A or B.
 *
 * Scratch: device staging of (M*K4 + K*N4 + M*N4) floats, K4 and N4 being K
 * and N rounded up to multiples of 4, plus the Stream-K workspace of the
 * panels.  Both come from caches the library keeps per (device, stream),
 * grown with cudaMalloc the first time a call needs more, and freed by
 * sgemm_release_workspaces().  The copy streams and events are created once
 * per (device, stream).  Calls on one stream run one after another; calls on
 * different streams have separate staging and may overlap.  As for sgemm(),
 * calls on one stream must not be made from several host threads at the same
 * time (they share that stream's staging and events).
 *
 * Errors: as sgemm() (SGEMM_ERR_ALLOC when the staging cannot be allocated);
 * M == 0 or N == 0 is a no-op, K == 0 writes zeros to C.  After an error
 * return, C's contents are undefined.
 */
sgemm_status_t sgemm_host(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                          const float *B, int64_t ldb, float *C, int64_t ldc, cudaStream_t stream);

/*
 * As sgemm() but forces `variant` (an sgemm_variant_t).  The four pipelined
 * variants (TILED, STREAMK, TILED_SMALL, STREAMK_SMALL) and SMALL given operands they
 * cannot take (a base address that is not 16-byte aligned or a row stride
 * that is not a multiple of 4) return SGEMM_ERR_INVALID_VALUE without
 * launching.  GUARDED and STAGED take any operands; STAGED copies only the
 * operands that need it, into the per-(device, stream) workspace, and then
 * runs the pipelined schedule the selector picks for the shape.
 *
 * SPECIALIZED is the size-specialized form of the pipelined kernel ("Beyond
 * Kernel 7", the size-specialized kernel of the confirmed 4096 result): the
 * instance with M, N, K and the Stream-K schedule compiled in as constants,
 * built for M = N = K = 768, 1024, 1536, 2048 and 4096 on a 152-SM GB300.  It
 * computes exactly what the generic Stream-K variant of the same schedule
 * computes (bit for bit).  The selector takes it whenever the shape, the
 * device and aligned operands allow.  Forced with operands the pipelined
 * variants cannot take it returns SGEMM_ERR_INVALID_VALUE, on any other shape
 * or device SGEMM_ERR_UNSUPPORTED, without launching.
 */
sgemm_status_t sgemm_variant(int variant, int64_t M, int64_t N, int64_t K, const float *A,
                             int64_t lda, const float *B, int64_t ldb, float *C, int64_t ldc,
                             cudaStream_t stream);

/*
 * The variant sgemm() would run for these arguments on the current device
 * (pointers are used only for their alignment), or -1 if the arguments are
 * invalid.  Launches nothing.
 */
int sgemm_select_variant(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                         const float *B, int64_t ldb, const float *C, int64_t ldc);

/*
 * Bytes of workspace the given variant (or the selected one, for
 * SGEMM_VARIANT_AUTO, assuming aligned operands) needs for this shape on the
 * current device; 0 when it needs none.  For SGEMM_VARIANT_STAGED the figure
 * includes copies of both A and B, the most that variant can need.  Returns 0
 * for invalid arguments too.
 */
size_t sgemm_workspace_size(int variant, int64_t M, int64_t N, int64_t K);

/*
 * Opt-in TF32 tensor-core mode: C = A * B with the products formed from TF32
 * inputs (FP32 exponent, 10 fraction bits) by tcgen05.mma and accumulated in
 * FP32.  Not an FP32 result: its error is bounded by about 2^-10 of
 * sum_k |A[m,k] B[k,n]| per element instead of K * 2^-24 of it; integer
 * inputs below 2^11 in magnitude whose partial sums stay below 2^24 are still
 * exact.  TF32 is the tensor-core precision the pages contrast with FP32
 * ("Beyond Kernel 7", section "The operation: GEMM and the precision of the
 * comparison"; "cuSgemm", Kernel 7).
 *
 * Same arguments and ownership as sgemm(), and any stride and alignment.
 * A 16-byte-aligned B with ldb a multiple of 4 is read in place; any other B
 * is first copied transposed, and an A without that property copied as is,
 * into the per-(device, stream) workspace, which may grow with cudaMalloc as
 * for sgemm().  A C without it is written with 4-byte stores.
 */
sgemm_status_t sgemm_tf32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                          const float *B, int64_t ldb, float *C, int64_t ldc, cudaStream_t stream);

/*
 * Reads, then clears, the device status word of the current device: the read
 * is queued on `stream` (an atomic exchange on the device), and the call
 * returns once `stream` has reached it.  Returns SGEMM_OK, or
 * SGEMM_ERR_TIMEOUT if a kernel gave up waiting since the last query.
 * *detail (may be NULL) receives a code that says which wait expired (0 when
 * none).  After a timeout the split-K arrival counters of every cached
 * workspace of the device may be stale: each is cleared on its own stream,
 * in stream order, before that stream's next call uses it, so kernels still
 * running on other streams are not disturbed.
 */
sgemm_status_t sgemm_query_device_status(cudaStream_t stream, uint32_t *detail);

/*
 * Frees every cached workspace of every device, including those replaced by
 * larger ones, and sgemm_host()'s device staging, copy streams and events
 * (synchronises each device first).  CUDA graphs captured with
 * sgemm() calls must not be replayed afterwards.
 */
void sgemm_release_workspaces(void);

/* Static description of a status code; never NULL. */
const char *sgemm_status_string(sgemm_status_t status);

/* Variant name ("guarded", "tiled", ...), or "unknown". */
const char *sgemm_variant_name(int variant);

/*
 * Test hook for the timeout path: launches one CTA that waits, with the
 * library's bounded wait and a limit of `limit_ns` nanoseconds, on a
 * shared-memory barrier nothing will ever complete.  The kernel records
 * SGEMM_ERR_TIMEOUT and returns; nothing hangs and no fault is raised.
 */
sgemm_status_t sgemm_debug_expire_wait(uint64_t limit_ns, cudaStream_t stream);

/*
 * Test hook for the Stream-K fix-up ("Beyond Kernel 7: Closing the Gap to
 * cuBLAS on an H100 FP32 GEMM", section "Kernel 14").  When `on` is nonzero,
 * pipelined and TF32 launches made after this call (by any thread of the
 * process) have the CTA (or CTA pair) that owns a split tile's first k-tiles
 * publish its partial sum like every other sharer.  It never keeps its
 * partial in registers or tensor memory, and never prefetches the others'.  The last CTA to arrive then sums every partial from the
 * workspace in CTA order.  The additions are the same sequence as on the
 * default path, so results must be bit-identical; only speed differs.  The
 * switch is process-wide; pass 0 to restore the default.  No error cases.
 */
void sgemm_debug_owner_publishes(int on);

/*
 * C = A * B with the Stream-K schedule (SGEMM_VARIANT_STREAMK), allocating
 * nothing.  The pages have no counterpart: this entry point exists for
 * callers that cannot let a library call cudaMalloc -- code that must never
 * wait on the whole device (cudaMalloc and cudaFree may synchronise it), code
 * that hands out a fixed memory budget before any work starts, and code
 * inside a framework whose own allocator owns the device memory.
 *
 * Arguments, layout and ownership are those of sgemm().  The Stream-K
 * scratch (arrival counters and partial sums of split tiles) lives in one
 * fixed 32 MiB array in the library's device image, which every GPU that
 * loads the library holds until the process exits.  No call allocates or
 * frees memory, and no library routine that does is called.
 *
 * - The first call on a device looks up the array's device address (set-up,
 *   once per device, with that device current); make that first call before
 *   any stream capture begins.
 * - Every call shares the one array: calls whose kernels overlap on the GPU
 *   (for example on two streams) race and corrupt each other's results.
 *   Order them on one stream or with events.
 * - Each call zeroes the counters it uses (an asynchronous memset on
 *   `stream`) and leaves the rest of the array as the previous call left it.
 * - Returns SGEMM_ERR_UNSUPPORTED, launching nothing, when the shape needs
 *   more scratch than the array holds (sgemm_workspace_size(
 *   SGEMM_VARIANT_STREAMK, M, N, K) > 32 MiB), and SGEMM_ERR_INVALID_VALUE
 *   for operands the pipelined kernel cannot take (a pointer not 16-byte
 *   aligned, or a row stride that is not a multiple of 4).
 */
sgemm_status_t sgemm_streamk_static(int64_t M, int64_t N, int64_t K, const float *A,
                                    int64_t lda, const float *B, int64_t ldb, float *C,
                                    int64_t ldc, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GB300_SGEMM_H */
