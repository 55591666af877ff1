/*
 * sgemm.h -- C ABI of the GB300 single-precision GEMM library
 * (libsgemm_gb300.so).
 *
 * Operation (the SGEMM of "From 1% to 94% of cuBLAS, one kernel at a time",
 * arpit2412.github.io/blog/cuda-sgemm.html, section "Napkin math for
 * 4092 x 4092", and its first kernel's per-element rule):
 *
 *     C = alpha * op(A) @ op(B) + beta * C
 *
 * with op(A) M x K, op(B) K x N, C M x N, fp32, every matrix row-major:
 * element (r, c) of a matrix with leading dimension ld is at r * ld + c
 * (the same page's storage paragraph).  Transposed operands and a strided
 * batch follow "Triton Optimization Reference (cuTile -> Triton)",
 * sections 2 (transpose by strides) and 3 (batch index with a per-batch
 * stride):
 *   transA == 0: A is stored M x K, lda >= K;  op(A)[i,k] = A[i*lda + k]
 *   transA != 0: A is stored K x M, lda >= M;  op(A)[i,k] = A[k*lda + i]
 *   transB == 0: B is stored K x N, ldb >= N;  op(B)[k,j] = B[k*ldb + j]
 *   transB != 0: B is stored N x K, ldb >= K;  op(B)[k,j] = B[j*ldb + k]
 *   C is stored M x N, ldc >= N.
 *   Batch q (0 <= q < Q) uses A + q*strideA, B + q*strideB, C + q*strideC;
 *   strides count elements; strideA or strideB may be 0 (broadcast).
 *
 * BLAS conventions where the pages are silent:
 *   - beta == 0: C is not read (NaN/Inf already in C do not propagate).
 *   - alpha == 0 or K == 0: C = beta * C; A and B are not read.
 *   - M == 0, N == 0 or Q == 0: nothing is done.
 *
 * Pointers A, B, C are DEVICE pointers owned by the caller.  The library
 * allocates no memory, never synchronises, and returns as soon as the work
 * is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream).
 * The output is valid once the stream reaches that point.
 *
 * Errors: arguments are checked on the host before anything is launched; an
 * invalid call returns SGEMM_ERR_INVALID_ARG and launches nothing.  A kernel
 * whose internal wait runs out of its bound (about a second) stops, leaves C
 * unspecified, and sets a device status word that sgemm_poll_error() reports
 * as SGEMM_ERR_TIMEOUT.  Calls are thread-safe; one call's kernels may run
 * concurrently with another call's only on different streams.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
#define SGEMM_OK 0
#define SGEMM_ERR_INVALID_ARG 1 /* a dimension, leading dimension, stride, pointer or mode */
#define SGEMM_ERR_UNSUPPORTED 2 /* valid call the library cannot run here (no sm_103 GPU) */
#define SGEMM_ERR_LAUNCH 3      /* the CUDA runtime refused a launch or attribute call    */
#define SGEMM_ERR_TIMEOUT 4     /* a kernel's bounded internal wait ran out (device word) */
#define SGEMM_ERR_SCRATCH_LIMIT 5 /* sgemm_batched_ex_noalloc: shape needs more than its scratch */

/* Contraction paths.
 *   FP32  : FP32 CUDA-core (FFMA) path; every product and sum in fp32.
 *   3XTF32: tensor-core path; each operand x is split into hi = x with its 13
 *           low mantissa bits cleared (a TF32 value) and lo = (x - hi)
 *           likewise, and the product is accumulated in fp32 as
 *           lo*hi + hi*lo + hi*hi, which meets the FP32 accuracy bound.
 *   TF32  : one tensor-core pass on tf32-rounded operands (looser accuracy,
 *           max |C - C_ref| / (|alpha| |A||B| + |beta C|) <= 2e-3).
 *   DEFAULT: the process default (sgemm_set_default_mode), initially FP32. */
#define SGEMM_MODE_DEFAULT (-1)
#define SGEMM_MODE_FP32 0
#define SGEMM_MODE_3XTF32 1
#define SGEMM_MODE_TF32 2

/* C = alpha*A@B + beta*C, no transposes, Q = 1, default mode. */
int sgemm(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
          float beta, float *C, int ldc, void *stream);

/* As sgemm, with the contraction path chosen explicitly (SGEMM_MODE_*;
 * DEFAULT means the process default): the first kernel's host signature in
 * "From 1% to 94% of cuBLAS, one kernel at a time" (M, N, K, alpha, A, B,
 * beta, C) plus the leading dimensions, the mode and the stream. */
int sgemm_ex(int mode, int M, int N, int K, float alpha, const float *A, int lda, const float *B,
             int ldb, float beta, float *C, int ldc, void *stream);

/* Strided-batched, transposed-operand form (conventions above), default mode.
 * Requires strideC >= (M-1)*ldc + N when Q > 1 (batch outputs may not
 * overlap); strides must be >= 0. */
int sgemm_batched(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                  int ldb, float beta, float *C, int ldc, int transA, int transB,
                  long long strideA, long long strideB, long long strideC, int Q, void *stream);

/* As sgemm_batched, with the contraction path chosen explicitly
 * (SGEMM_MODE_*; DEFAULT means the process default). */
int sgemm_batched_ex(int mode, int M, int N, int K, float alpha, const float *A, int lda,
                     const float *B, int ldb, float beta, float *C, int ldc, int transA,
                     int transB, long long strideA, long long strideB, long long strideC, int Q,
                     void *stream);

/* Split-K workspace.  The output is cut into tiles (256 x 128 on the FP32
 * and 3xTF32 paths, 256 x 256 on the TF32 path when the operands are
 * TMA-describable and K >= 1536, 128 x 128 for operands TMA cannot
 * describe), each computed by one persistent
 * CTA per multiprocessor or, on
 * the tensor cores, one CTA pair per two.  When the tiles do not fill a
 * whole number of waves (4092^3: 512 tiles = 6.7 waves on 76 pairs), or fill less than
 * one (small or skinny products such as the ragged 1000 x 1500 x 777 case),
 * the library can cut the tiles of the last, partial wave along K into
 * slices computed in parallel -- the split-K scheme the SGEMM worklog sees
 * cuBLAS use at 256^3 ("From 1% to 94% of cuBLAS", comparison across sizes).
 * Each slice's partial tile needs scratch memory, which the caller provides:
 *
 * sgemm_workspace_size returns the bytes of workspace the preferred plan
 * wants for this shape on the current device (0: the shape needs none, or
 * the arguments are invalid, or there is no usable device).
 *
 * sgemm_batched_ex_ws is sgemm_batched_ex plus a DEVICE workspace owned by
 * the caller: `workspace` must be 256-byte aligned when workspace_bytes > 0
 * (else SGEMM_ERR_INVALID_ARG).  The call runs the best split plan whose
 * workspace fits in workspace_bytes (with sgemm_workspace_size(...) bytes,
 * the preferred one; with NULL / 0, none), with the same results up to
 * rounding.  Every slice stores its partial tile in fp32; a second kernel,
 * enqueued on `stream` right after the first, sums each tile's slices in a
 * fixed order and applies alpha and beta, so repeated calls give identical
 * bits.  On the FP32 path the workspace also serves a transposed copy of a
 * K-inner A (when N >= 1024) and of a K-inner B (when M >= 1024), made on
 * `stream` before the product: that path runs fastest with A M-inner and B
 * N-inner.  On the tensor-core paths it serves a copy, rows padded to 128
 * bytes, of an operand TMA cannot describe (row pitch or batch stride not a
 * multiple of 4 floats, base not 16-byte aligned), which then runs on the
 * TMA-fed kernel instead of the slower direct-load one.  sgemm_workspace_size
 * counts that room for both operands.  For shapes where it pays (the
 * library's time model: the pass over the operands must cost less than the
 * product saves -- at 4092^3 yes, at 2048^3 or the batched 1024 x 1024 x 512
 * case no), the tensor-core paths instead use the workspace for the
 * operands' TF32 planes: a pass writes op(A) and op(B) K-major, rows of
 * round_up(K, 32) floats, as hi and lo planes (3xTF32: the value with its 13
 * low mantissa bits cleared, and the rest likewise) or one plane rounded to
 * nearest (TF32), 2 * (M + N) * K * 4 bytes per batch entry for 3xTF32, and
 * the product reads them through TMA with no conversion; the workspace then
 * starts with op(A)'s planes.  sgemm_workspace_size counts that room where
 * the route pays; with less, the call runs the other way.  The workspace
 * needs no initialisation; it must not be used by another call running at
 * the same time. */
size_t sgemm_workspace_size(int mode, int M, int N, int K, int Q);
int sgemm_batched_ex_ws(int mode, int M, int N, int K, float alpha, const float *A, int lda,
                        const float *B, int ldb, float beta, float *C, int ldc, int transA,
                        int transB, long long strideA, long long strideB, long long strideC,
                        int Q, void *workspace, size_t workspace_bytes, void *stream);

/* Split-K for callers that cannot allocate device memory.  (No counterpart on
 * the pages: an addition of this library.)
 *
 * Same arguments and results as sgemm_batched_ex_ws, without the workspace:
 * the partial tiles (and, on the FP32 path, a transposed operand when it
 * fits beside them) live in a fixed 24 MB scratch array inside the library
 * image.  For code that may not call cudaMalloc or may not grow a memory pool
 * at the point where it multiplies (a host callback, another library's
 * critical section, a plugin that is handed only its input and output
 * buffers).  The function allocates and frees nothing.
 *  - It splits only grids of at most half as many tiles as the GPU has
 *    multiprocessors, into as many slices as keep every slice in one wave
 *    (at most one partial tile per multiprocessor); larger grids run
 *    unsplit, exactly as sgemm_batched_ex.
 *  - Every GPU that loads the library holds the 24 MB until the process exits.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.  The address is kept for the life of the
 *    process: after a cudaDeviceReset the library image may be loaded again
 *    at another address, so do not call this function on a device that has
 *    been reset since its first call.
 *  - An operand copy the call makes first (the FP32 path's transposed
 *    operand, the tensor-core paths' copy of an operand TMA cannot describe)
 *    takes the front of the same scratch; what is left may be too small for
 *    the split, and the call then runs with fewer slices or unsplit (the
 *    same result up to rounding, only slower).
 *  - All calls on a device share the array; it needs no initialisation.
 *    Calls whose kernels overlap on the GPU (different streams, or another
 *    thread) race on the array: serialise them.
 *  - A shape whose split workspace exceeds 24 MB returns
 *    SGEMM_ERR_SCRATCH_LIMIT and launches nothing; that cannot happen on a
 *    GPU with at most ~190 multiprocessors. */
int sgemm_batched_ex_noalloc(int mode, int M, int N, int K, float alpha, const float *A, int lda,
                             const float *B, int ldb, float beta, float *C, int ldc, int transA,
                             int transB, long long strideA, long long strideB, long long strideC,
                             int Q, void *stream);

/* GEMM with 16-bit inputs and fp32 accumulation and output:
 *     C = alpha * op(A) @ op(B) + beta * C,  A and B bf16 or fp16, C fp32.
 * (The next step the SGEMM worklog's future-work list points to -- tensor
 * cores with narrower inputs -- on the same tcgen05 machinery: every
 * product of two 16-bit values is exact in fp32, so results differ from
 * the exact sum of products only by fp32 accumulation, within the FP32
 * path's tolerance.)
 *
 * `type` is SGEMM_HALF_BF16 or SGEMM_HALF_FP16; A and B are DEVICE pointers
 * to 16-bit values of that type, with the layout, leading dimensions
 * (elements) and batch strides of sgemm_batched; C, alpha and beta as there.
 * The kernel reads an operand directly when it is K-inner (A untransposed,
 * B transposed: the "A times B-transpose" layout), 16-byte aligned, and its
 * leading dimension and batch stride are multiples of 8; any other operand
 * is first copied (transposed where needed, rows padded to 64 values) into
 * the caller's DEVICE
 * workspace (256-byte aligned when workspace_bytes > 0), which also serves
 * the split-K partial tiles.  A call whose copies do not fit returns
 * SGEMM_ERR_INVALID_ARG and launches nothing.
 *
 * sgemm_half_workspace_size returns the bytes of workspace the call wants
 * for these layouts and leading dimensions (assuming 16-byte aligned
 * operands), 0 when it needs none or for invalid arguments / no usable
 * device.  K == 0 or alpha == 0 gives C = beta * C.  Errors as for
 * sgemm_batched_ex_ws; SGEMM_ERR_INVALID_ARG also for an unknown type. */
#define SGEMM_HALF_BF16 0
#define SGEMM_HALF_FP16 1
size_t sgemm_half_workspace_size(int type, int M, int N, int K, int transA, int transB, int lda,
                                 int ldb, int Q);
int sgemm_half_batched(int type, int M, int N, int K, float alpha, const void *A, int lda,
                       const void *B, int ldb, float beta, float *C, int ldc, int transA,
                       int transB, long long strideA, long long strideB, long long strideC, int Q,
                       void *workspace, size_t workspace_bytes, void *stream);

/* The product on HOST buffers.  (No counterpart on the pages, whose
 * benchmarks start with the operands on the GPU: an addition of this library
 * for callers whose data lives in host memory.)
 *
 * A, B and C are host pointers with the layout and leading dimensions of
 * sgemm_batched (one product, no batch).  The call copies op(A), op(B) and,
 * when beta != 0, C into `dev`, a DEVICE buffer the caller owns (256-byte
 * aligned, at least sgemm_host_buffer_size(...) bytes), computes there, and
 * copies C back.  op(B) is copied first; C is cut into panels of
 * `panel_rows` rows (0: the library picks as many whole rows of output tiles
 * as fit in one wave of the GPU; at most 64 panels, else
 * SGEMM_ERR_INVALID_ARG): the copy-in of one panel's rows of op(A), the
 * products of earlier panels and the copy-out of a finished one run at the
 * same time, on two copy streams the library keeps per device, on `stream`
 * for the products of even panels and on a third library stream for those of
 * odd panels (so that two products together fill the GPU); each panel's
 * product is a workspace-entry call on the device copies, which takes the
 * route the cost models pick for it.  The host link bounds
 * the call: on GB300 about 200 GB/s to the device and 184 from it, ~265 in
 * all while both directions run.  The call is asynchronous like the others:
 * C on the host holds
 * the result once `stream` has reached the end of the call (synchronise it,
 * or record an event after the call).  Host memory that is page-locked
 * (cudaHostAlloc / cudaHostRegister) is copied at full speed and overlaps;
 * pageable memory works but its copies are staged by the driver and do not
 * overlap.  Arguments are checked as in sgemm_batched_ex_ws; a CUDA error
 * part-way returns SGEMM_ERR_LAUNCH (C on the host is then unspecified).
 * The buffer must not be used by another call running at the same time.
 *
 * sgemm_host_buffer_size returns the bytes of `dev` such a call needs (0 for
 * invalid arguments or without a usable device): the three operands with
 * rows padded to a multiple of four floats, plus two split-K / transposition
 * workspaces of a panel product (one per product stream). */
size_t sgemm_host_buffer_size(int mode, int M, int N, int K, int transA, int transB,
                              int panel_rows);
int sgemm_host(int mode, int M, int N, int K, float alpha, const float *A, int lda,
               const float *B, int ldb, float beta, float *C, int ldc, int transA, int transB,
               int panel_rows, void *dev, size_t dev_bytes, void *stream);

/* Throughput probes (measurement only; no product is computed).  Launches
 * one kernel on `stream` that runs only the arithmetic instructions of a
 * path, with no operand traffic, and stores in *flops the floating-point
 * operations it performs (2 per multiply-add).  Timed with events on
 * `stream`, it gives the peak those instructions reach on this GPU at that
 * moment -- the denominator a kernel's own speed is best set against:
 *   SGEMM_PROBE_FFMA     scalar fma.rn.f32 chains      iters: loop trips, 1 .. 65536
 *   SGEMM_PROBE_FFMA2    packed fma.rn.f32x2 chains    (each trip: 128 multiply-
 *                                                       adds per thread, 1024
 *                                                       threads per multiprocessor)
 *   SGEMM_PROBE_TF32_SS  tcgen05.mma kind::tf32 M=128 N=256 K=8, both operands
 *                        in shared memory              iters: MMAs per
 *   SGEMM_PROBE_TF32_TS  kind::tf32 M=128 N=128 K=8, A in tensor memory (the
 *                        instruction of the 3xTF32 and TF32 kernels)
 *   SGEMM_PROBE_BF16_SS  kind::f16, bf16 operands, M=128 N=256 K=16
 *                                                      multiprocessor, 1 .. 2^22
 * Returns SGEMM_ERR_INVALID_ARG for an unknown kind, iters out of range or a
 * NULL flops, SGEMM_ERR_UNSUPPORTED without a compute capability 10.3 GPU,
 * SGEMM_ERR_LAUNCH if the launch fails.  The tensor-core probes end with a
 * bounded wait, reported by sgemm_poll_error like the GEMM kernels'. */
#define SGEMM_PROBE_FFMA 0
#define SGEMM_PROBE_FFMA2 1
#define SGEMM_PROBE_TF32_SS 2
#define SGEMM_PROBE_TF32_TS 3
#define SGEMM_PROBE_BF16_SS 4
int sgemm_peak_probe(int kind, long long iters, double *flops, void *stream);

/* Tuning hooks (measurement; the sweep `bench.py --tune` uses them).
 * Which kernel family runs a call is chosen per (mode, size class, batched)
 * by a table compiled into the library from that sweep, the size class
 * being round(log2(M * N * K * Q) / 3) clamped to 7..13; a class without
 * an entry follows the library's cost models.  The families ("routes"):
 *   0  AUTO     the cost models (the FP32 tile that suits the layout; on the
 *               tensor cores the raw route where its time model says it pays
 *               and both operands are TMA-describable (3xTF32: and the
 *               workspace holds their lo planes), else the TF32-planes route
 *               where it pays and the workspace holds the planes, else the
 *               CTA-pair kernel for TMA-describable operands, else the direct
 *               kernel)
 *   1  SMALL    FP32 on 64 x 64 tiles
 *   2  PAIR     tensor cores on the CTA-pair kernel, no planes
 *   3  DIRECT   tensor cores on the direct-load kernel
 *   4  PLANES   tensor cores on the planes route whenever the workspace holds
 *               the planes (sgemm_workspace_size then counts them)
 *   5  RAW      tensor cores on the caller's matrices as stored, whenever
 *               both operands are TMA-describable (16-byte aligned base,
 *               leading dimension and batch stride multiples of 4 values);
 *               3xTF32 also needs the workspace to hold the operands' lo
 *               planes (sgemm_workspace_size then counts them)
 *   6  INLINE   the RAW route with 3xTF32's lo planes made inside the product
 *               kernel from the staged operands (no pass, no workspace for
 *               planes); TF32 as RAW
 *   7  MODELS   (to force only) the cost models' choice with the table
 *               ignored: the baseline the sweep measures the others against
 * A route the call's mode cannot take means AUTO; every route computes the
 * same result within the mode's accuracy bound.
 * sgemm_tune_force(route) makes every later call in the process take that
 * route (AUTO: the table again); SGEMM_ERR_INVALID_ARG for an unknown route.
 * It is a process-wide setting: do not change it while other threads call
 * the library.  sgemm_tune_route returns the route a call of that shape
 * would take now (-1 for an invalid mode or a negative dimension). */
#define SGEMM_ROUTE_AUTO 0
#define SGEMM_ROUTE_SMALL 1
#define SGEMM_ROUTE_PAIR 2
#define SGEMM_ROUTE_DIRECT 3
#define SGEMM_ROUTE_PLANES 4
#define SGEMM_ROUTE_RAW 5
#define SGEMM_ROUTE_INLINE 6
#define SGEMM_ROUTE_MODELS 7
int sgemm_tune_force(int route);
int sgemm_tune_route(int mode, int M, int N, int K, int Q);

/* Process-wide default path used by sgemm() and sgemm_batched().  Returns
 * SGEMM_ERR_INVALID_ARG for an unknown mode (DEFAULT is not a valid value
 * here). */
int sgemm_set_default_mode(int mode);
int sgemm_get_default_mode(void);

/* Static, never-NULL description of a status code. */
const char *sgemm_status_string(int status);

/* Synchronises `stream`, then reads and clears the current device's status
 * word.  Returns SGEMM_OK, SGEMM_ERR_TIMEOUT if a kernel's bounded wait ran
 * out since the last poll, or SGEMM_ERR_LAUNCH if the stream reports a CUDA
 * error. */
int sgemm_poll_error(void *stream);

/* Self test of the bounded-wait machinery: launches one small kernel whose
 * mbarrier wait is never satisfied and whose bound is `wait_cycles` clock
 * cycles (1 .. 2^31), so that it gives up, records the timeout in the status
 * word and exits normally.  A following sgemm_poll_error() returns
 * SGEMM_ERR_TIMEOUT.  Nothing faults and the context stays usable. */
int sgemm_selftest_wait_timeout(long long wait_cycles, void *stream);

/* Number of kernels the library has enqueued in this process so far (every
 * device and stream; a failed launch is not counted).  The difference across
 * a stretch of calls is the number of kernels they launched: a GEMM call
 * launches one product kernel, plus the split-K fix-up kernel when its plan
 * splits, plus one transposition per operand the FP32 path copies, plus the
 * passes of the planes route and of the raw route's lo planes. */
unsigned long long sgemm_kernel_launches(void);

/* Slices per split tile of the most recent product kernel the library
 * planned in this process (1: not split); for tests and tuning, racy across
 * threads that call at the same time. */
int sgemm_last_split_count(void);

/* Library version, major*10000 + minor*100 + patch. */
int sgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
