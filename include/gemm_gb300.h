/*
 * gemm_gb300.h -- C ABI of the GB300 (sm_103a) dense GEMM library
 * (libgemm_gb300.so).
 *
 *   D = alpha * op(A) @ op(B) + beta * C
 *
 * The operation is the tile-level contraction of the TVM TIRx "gemm" page
 * (opening paragraph: "D = alpha*A@B + beta*C"; table "What it accepts":
 * float16 / bfloat16 operands, float32 accumulator; beta 0 -> D = A@B,
 * beta 1 -> D = A@B + C) with the general epilogue alpha * acc + beta * c_old
 * of the Phobos "@tensorcore" page (example gemm_fp16tc_fp32acc.ph), for
 * whole row-major matrices in GPU memory.
 *
 * Layout (TIRx gemm guide, section 二, dimension consistency: the
 * transpose flags only name the logical orientation, the operation is
 * normalised to A = [M,K], B = [K,N], C = D = [M,N]):
 *   A  row-major [M, K] (transA = 0) or [K, M] (transA = 1), lda = its row stride
 *   B  row-major [K, N] (transB = 0) or [N, K] (transB = 1), ldb = its row stride
 *   C  row-major [M, N], ldc = row stride (read only when beta != 0)
 *   D  row-major [M, N], ldd = row stride
 * Leading dimensions are in elements.
 *
 * Precision: A and B are both in_dtype (GEMM_F16, GEMM_BF16, or the 8-bit
 * GEMM_E4M3 / GEMM_E5M2 that the TIRx gemm guide lists among the tcgen05
 * path's precisions, section 七; one dtype for both, so mixed operand types
 * cannot be expressed); products are
 * accumulated in fp32 on the tensor cores; the epilogue computes
 * fmaf(alpha, acc, beta * c) in fp32 (alpha * acc when beta == 0) and
 * rounds to out_dtype (round-to-nearest-even for 16-bit outputs).  C has
 * out_dtype.  beta == 0 means "D zero-initialised": C is not read and may
 * be NULL, and NaNs in C do not reach D.
 *
 * Ownership and ordering: the caller owns every buffer; all four pointers
 * are device pointers valid on the current device.  gemm() enqueues its
 * work on `stream` and returns without synchronising.  The library keeps
 * one small device status block per device (allocated on the first call on
 * that device; a set-up that fails is reported by that call and tried again
 * by the next) and, per (device, stream), workspaces for stream-K partial
 * sums and repacked operands, allocated when a call first needs them and
 * grown on demand (growing one synchronises the device).  Calls are
 * thread-safe.
 *
 * Errors: gemm() returns GEMM_OK or a negative GEMM_ERR_* code.  Every
 * argument error is detected before anything is enqueued, and D is then
 * untouched.  A failure inside the kernel (a pipeline wait that exceeded
 * its time bound) is reported by gemm_poll_device_error().
 *
 * Naming: the header is gemm_gb300.h, after the library it declares
 * (libgemm_gb300.so), rather than a bare gemm.h, so that it cannot be
 * shadowed by, or shadow, another library's gemm.h on an include path.
 * The calls, their argument order and the status convention are those of
 * the planned boundary; the additions are marked where they are declared
 * (the `info` argument of gemm_poll_device_error, and gemm_mx,
 * gemm_noalloc, gemm_host and the host-only queries).
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stdint.h>

#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* = cudaStream_t; NULL is the legacy default stream */

typedef enum {
    GEMM_F16 = 0,  /* IEEE binary16 */
    GEMM_BF16 = 1, /* bfloat16 */
    GEMM_F32 = 2,  /* IEEE binary32 (outputs only) */
    GEMM_E4M3 = 3, /* 8-bit float, 1-4-3, bias 7, no infinities, S.1111.111 = NaN (operands only) */
    GEMM_E5M2 = 4, /* 8-bit float, 1-5-2, bias 15, with infinities and NaNs (operands only) */
    GEMM_E2M1 = 5  /* 4-bit float, 1-2-1, bias 1 (0, 0.5, 1, 1.5, 2, 3, 4, 6), packed two per byte,
                      even elements in the low nibble; leading dimensions count elements
                      (gemm_mx operands only) */
} gemm_dtype_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = -1,       /* negative size, flag not 0/1, ld too small, NULL buffer */
    GEMM_ERR_UNSUPPORTED_DTYPE = -2, /* in_dtype not F16/BF16, or out_dtype not F32/F16/BF16 */
    GEMM_ERR_MISALIGNED = -3,        /* a buffer not aligned to its element size */
    GEMM_ERR_ALIAS = -4,             /* D overlaps A or B, or overlaps C other than C == D with ldc == ldd */
    GEMM_ERR_ARCH = -5,              /* the current device is not an sm_103 (GB300) GPU */
    GEMM_ERR_LAUNCH = -6,            /* the kernel launch was refused */
    GEMM_ERR_CUDA = -7,              /* another CUDA runtime / driver error */
    GEMM_ERR_DEVICE_TIMEOUT = -8,    /* (gemm_poll_device_error) an in-kernel wait gave up */
    GEMM_ERR_TOO_LARGE = -9,         /* a dimension above 2^31 - 1, or a stride above 2^40 bytes */
    GEMM_ERR_UNSUPPORTED_LAYOUT = -10 /* 8-bit operands in a layout the call cannot take (see gemm_noalloc) */
} gemm_status_t;

/*
 * D = alpha * op(A) @ op(B) + beta * C on the current device, enqueued on
 * `stream`.
 *
 *   M, N, K          sizes, >= 0.  M == 0 or N == 0: nothing to do, GEMM_OK.
 *                    K == 0: the sum is empty, D = alpha * 0 + beta * C.
 *   lda, ldb         >= the stored row length of A / B (K or M, N or K) when
 *                    K > 0; ignored when K == 0.
 *   ldc              >= N when beta != 0; ignored otherwise.
 *   ldd              >= N.
 *   transA, transB   0 or 1 (see the layout above).
 *   alpha, beta      any float; beta == 0.0f selects "C not read".
 *   in_dtype         GEMM_F16, GEMM_BF16, GEMM_E4M3 or GEMM_E5M2 (A and B).
 *   out_dtype        GEMM_F32, GEMM_F16 or GEMM_BF16 (C and D).
 *   stream           CUDA stream of the current device.
 *
 * Alignment: each buffer must be aligned to its element size; any such
 * layout is computed.  Kernels:
 *   - the tcgen05 kernel (TMA copies, tensor-memory accumulators) on the
 *     caller's buffers when A, B, C, D are 16-byte aligned and lda, ldb,
 *     ldc, ldd times their element sizes are multiples of 16 bytes (TMA's
 *     rule), and 8-bit operands are K-major (A stored [M, K], transA = 0;
 *     B stored [N, K], transB = 1);
 *   - aligned fp16 / bf16 problems with K <= 32 and M*N <= 2^18: the
 *     warp-level mma.sync route, whose one-warp-per-16x8-block kernel
 *     finishes a launch sooner (GEMM_SYNC_MAX_WORK=w replaces this rule
 *     by M*N*K <= w);
 *   - other layouts with M*N*K > 2^22 (GEMM_REPACK_MIN_WORK), and every
 *     other 8-bit layout: the tcgen05 kernel on workspace copies (operands
 *     copied into 16-byte-aligned rows, 8-bit MN-major operands transposed
 *     to K-major, a misaligned D computed in workspace and copied back);
 *   - the remaining fp16 / bf16 layouts: the mma.sync route, which reads
 *     and writes element by element (one warp per 16 x 8 block of D while
 *     M*N <= 2^18 and M*N*K <= 2^24, else 128 x 128 CTA tiles staged in
 *     shared memory; GEMM_SYNC_ATOM_MAX_WORK=w replaces this rule by
 *     M*N*K <= w).
 * All accumulate in fp32 and agree within the documented tolerance.
 * GEMM_PATH=tcgen05 or mma_sync forces a kernel where it can run.
 * CUDA graphs: gemm() may be called while `stream` is being captured, as
 * long as an earlier call (outside the capture) has run on the device; it
 * then allocates nothing: stream-K splitting and the repacking route are
 * used only where this stream's workspace from earlier calls is large
 * enough (otherwise whole tiles, respectively the mma.sync kernel).  A
 * workspace that a capture used stays allocated when a later call outgrows
 * it, so the graph can be replayed after any number of other calls.
 * Returns GEMM_OK or a GEMM_ERR_* code (see gemm_status_t).
 * Setting the environment variable GEMM_LOG=1 prints each call's plan or
 * rejection reason to stderr; GEMM_MAX_SMS=n (n >= 2) plans the persistent
 * grid for at most n SMs, leaving the others to other work on the GPU.
 */
GEMM_API int gemm(void* D, const void* A, const void* B, const void* C,
         int64_t M, int64_t N, int64_t K,
         int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd,
         int transA, int transB, float alpha, float beta,
         int in_dtype, int out_dtype, struct CUstream_st* stream);

/*
 * gemm_mx -- gemm() with MX block-scaled 8-bit operands:
 *
 *   D[i][j] = alpha * sum_k (sa(i, k) * op(A)[i][k]) * (sb(j, k) * op(B)[k][j])
 *             + beta * C[i][j],
 *   sa(i, k) = 2^(SFA[i * ld_sfa + k / 32] - 127),
 *   sb(j, k) = 2^(SFB[j * ld_sfb + k / 32] - 127).
 *
 * The TIRx gemm guide (section 七) lists block scaling with separate A and
 * B scale factors ("SFA/SFB") among the tcgen05 path's modes without
 * defining it; this is the OCP Microscaling (MX) reading: every 32
 * consecutive K elements of a row of op(A) share one UE8M0 scale byte, and
 * likewise every 32 of a column of op(B).  A scale byte e stands for
 * 2^(e - 127); e = 255 is NaN and makes its 32 products NaN.
 *
 *   SFA, SFB         device pointers: SFA row-major [M, ceil(K/32)] bytes with
 *                    row stride ld_sfa, SFB row-major [N, ceil(K/32)] with row
 *                    stride ld_sfb (rows of SFB are columns of op(B),
 *                    whatever transB says).  Any byte alignment.  Not read
 *                    when K == 0 (may then be NULL).
 *   ld_sfa, ld_sfb   >= ceil(K/32) when K > 0.
 *   in_dtype         GEMM_E4M3, GEMM_E5M2 or GEMM_E2M1 (else
 *                    GEMM_ERR_UNSUPPORTED_DTYPE).  E2M1 (fp4, the guide's
 *                    other gemm_async precision) is packed: element e of a
 *                    row-major operand (e = row * ld + col) is the low nibble
 *                    of byte e / 2 when e is even, the high nibble when odd.
 *                    It must be K-major (A stored [M, K], transA = 0; B
 *                    stored [N, K], transB = 1; else
 *                    GEMM_ERR_UNSUPPORTED_LAYOUT) with K, lda and ldb even
 *                    (else GEMM_ERR_INVALID_ARG).
 *   everything else  as for gemm().
 *
 * Kernel: tcgen05.mma kind::mxf8f6f4 with 256 x 224 tiles on a CTA pair
 * for f32 D and 256 x 192 for 16-bit D (128-row tiles on one SM when
 * M <= 128); each call first rearranges the scales into 512-byte chunks in
 * a workspace of this (device, stream) (about (M + 1.14 N) * K / 32 bytes
 * for f32 D, (M + 1.33 N) * K / 32 for 16-bit D), then runs the product.
 * Layouts that are not K-major 16-byte aligned go through the same
 * repacking as gemm()'s 8-bit operands.  D must not overlap SFA or SFB
 * (GEMM_ERR_ALIAS).  Under CUDA graph capture nothing is allocated: the
 * workspaces must exist from an earlier call of at least the same size on
 * the stream, else GEMM_ERR_CUDA.
 */
GEMM_API int gemm_mx(void* D, const void* A, const void* B, const void* C,
                     const void* SFA, const void* SFB,
                     int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd,
                     int64_t ld_sfa, int64_t ld_sfb,
                     int transA, int transB, float alpha, float beta,
                     int in_dtype, int out_dtype, struct CUstream_st* stream);

/*
 * A static, human-readable name for a gemm_status_t value (never NULL).
 *
 * The status convention stands in for the error path of the TIRx gemm
 * guide (section 二, "What it accepts", its closing paragraph on dispatch
 * failure: a variant that cannot take the call raises DispatchFail, and
 * when no variant can, the reasons are collected into one RuntimeError).  Across a C ABI there are no exceptions, so each
 * reason the guide gives for refusing a call becomes a negative code,
 * returned before anything is enqueued, and this call names it.
 */
GEMM_API const char* gemm_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears a status record of the
 * current device.  The device has up to two: gemm()'s (gemm_mx() and
 * gemm_host() share it), created by the first gemm() call on the device,
 * and gemm_noalloc()'s, the static array set up by its first call.  Only
 * records that exist are read: this call creates nothing and allocates
 * nothing, so callers of gemm_noalloc() may use it too.  Each record keeps
 * the first in-kernel wait that gave up (GEMM_WAIT_TIMEOUT_NS, default
 * 2 s) since it was last cleared; a kernel that gave up stopped early and
 * left its D partly written.
 *
 * Returns GEMM_OK (no record holds an error), GEMM_ERR_DEVICE_TIMEOUT
 * (one record held a timeout; that record is cleared -- when both hold
 * one, gemm()'s is reported first and the other by the next poll), or
 * GEMM_ERR_CUDA when the stream reports a CUDA error.  When `info` is not
 * NULL it receives four ints: code, block, wait site, detail (all zero
 * when GEMM_OK is returned).
 *
 * Source: the TIRx gemm guide's error path (see gemm_status_string) turns
 * dispatch failures into errors the caller sees; an asynchronous kernel
 * can only report after the fact, so this poll is how its failures reach
 * the caller.  The `info` argument is this library's addition: the
 * single-argument poll(stream) planned for the boundary gives the code
 * alone.
 */
GEMM_API int gemm_poll_device_error(struct CUstream_st* stream, int* info);

/*
 * Host-only query (no GPU needed): the persistent kernel's tile order.
 * The pages have no counterpart of the host-only queries (this one and the
 * three below); they expose this library's scheduler and planner so that
 * tests and callers can check what a call will run without a GPU.
 * For a grid of num_m x num_n output tiles rasterised in groups of group_m
 * tile rows, writes the (m, n) tile coordinates of tile index `tile`.
 * Returns GEMM_OK, or GEMM_ERR_INVALID_ARG for out-of-range arguments.
 */
GEMM_API int gemm_tile_coords(int tile, int num_m, int num_n, int group_m, int* m_blk, int* n_blk);

/*
 * Host-only query (no GPU needed): the kernel configuration gemm() would
 * choose for these sizes on a GPU with num_sms SMs (fp16 operands, B stored
 * [K, N], f32 D; gemm_plan_layout below takes the others).  out[0..9] receive:
 * cta_pair (1 = 2-SM tiles), tile_m, tile_n, number of tiles, grid size
 * (CTAs), dynamic shared memory bytes, epilogue warps, operand pipeline
 * stages, stream-K tiles (trailing tiles split along K; 0 = every tile
 * whole), and the bytes of the per-stream workspace the stream-K tiles
 * need.  Returns GEMM_OK or an error code.
 */
GEMM_API int gemm_plan(int64_t M, int64_t N, int64_t K, int num_sms, int64_t* out);

/*
 * Host-only query (no GPU needed): gemm_plan() for a layout and types --
 * transB (1: B stored [N, K]), in_dtype (GEMM_F16, GEMM_BF16, GEMM_E4M3 or
 * GEMM_E5M2) and out_dtype (GEMM_F32, GEMM_F16 or GEMM_BF16) -- with the
 * same out[0..9].  8-bit operands are planned K-major, the layout gemm()
 * runs them in.  The plan can differ with the layout: with f32 D and
 * K-major B, tiles 224 columns wide are chosen when they fill the last wave
 * better than 256-wide ones.  gemm_plan(M, N, K, num_sms, out) equals
 * gemm_plan_layout(M, N, K, 0, GEMM_F16, GEMM_F32, num_sms, out).  Returns
 * GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_TOO_LARGE or
 * GEMM_ERR_UNSUPPORTED_DTYPE.
 */
GEMM_API int gemm_plan_layout(int64_t M, int64_t N, int64_t K, int transB, int in_dtype, int out_dtype,
                              int num_sms, int64_t* out);

/*
 * Host-only query (no GPU needed): the work of one persistent worker
 * (cluster) under the kernel's schedule.  num_tiles tiles of `iters`
 * pipeline stages each; the last sk_tiles tiles are split along K evenly
 * across the `workers` workers; the others are dealt whole, round-robin.
 * Writes up to max_units records of 6 ints (tile, first stage, end stage,
 * stream-K tile index or -1, contributor index, number of contributors) to
 * `out` and returns the number of units of this worker (possibly more than
 * max_units), or GEMM_ERR_INVALID_ARG.
 */
GEMM_API int gemm_schedule_units(int num_tiles, int iters, int workers, int sk_tiles, int worker, int* out,
                                 int max_units);

/*
 * gemm_noalloc -- gemm() for callers that cannot allocate device memory.
 *
 * The pages have no counterpart of this call; it exists for users of this
 * library.  gemm() obtains its device status record with cudaMalloc the
 * first time it runs on a device.  Some callers cannot allow that: code
 * that owns all of the device's memory through its own pool or budget,
 * code running where CUDA allocation calls are not permitted (for example
 * from a stream callback), or code that must not add allocations to a
 * process it does not own.  gemm_noalloc() computes what gemm() computes,
 * with the same arguments, rules and return codes, through the same
 * kernels, but never calls cudaMalloc, cudaFree or any other allocating
 * routine.  Without workspace it does not split tiles along K (stream-K)
 * and does not repack: fp16 / bf16 layouts off TMA's 16-byte grid run on
 * the mma.sync kernel whatever their size, and 8-bit operands must already
 * be K-major and 16-byte aligned (else GEMM_ERR_UNSUPPORTED_LAYOUT, before
 * anything is enqueued).  The kernel's scratch (its 16-byte status record) lives in a
 * fixed 256-byte array inside the library, which every GPU that loads the
 * library holds until the process exits.  The scratch does not grow with
 * the problem, so no problem size exceeds it; a build whose record did not
 * fit the array would return GEMM_ERR_TOO_LARGE.
 *
 *   - The first call on each device does a one-time set-up (device queries,
 *     the kernels' shared-memory limit, and the device address of the
 *     static array via cudaGetSymbolAddress).  Make that first call before
 *     any stream capture.
 *   - All gemm_noalloc() calls on a device share the one status record.
 *     It is zero when the library is loaded and keeps the first pipeline
 *     wait that gave up (the kernel then stops early, leaving D partly
 *     written) until gemm_poll_device_error() reads and clears it; no
 *     gemm_noalloc() call clears it.  Calls whose kernels overlap on the
 *     GPU (different streams) race on it: a timeout in either is reported,
 *     but the record says which call's kernel wrote first, not which call
 *     the caller meant to check.
 *   - gemm_poll_device_error() reads this record without allocating, so it
 *     is the way to learn whether a gemm_noalloc() call completed.
 */
GEMM_API int gemm_noalloc(void* D, const void* A, const void* B, const void* C,
                          int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd,
                          int transA, int transB, float alpha, float beta,
                          int in_dtype, int out_dtype, struct CUstream_st* stream);

/*
 * gemm_host -- gemm() with A, B, C and D in host memory.
 *
 * The pages have no counterpart of this call; it is the entry point for
 * callers whose matrices live on the host.  Same arguments, layouts, rules
 * and results as gemm(), except that the four pointers are host pointers
 * (pinned memory -- cudaMallocHost / cudaHostAlloc / cudaHostRegister --
 * lets the copies run asynchronously at full speed; pageable memory works,
 * with copies that block the calling thread).
 *
 *   - The library stages the operands in device buffers it owns (one set
 *     per (device, stream), grown on demand, kept until the process exits)
 *     and pipelines the work over row panels of D on three streams: the
 *     host-to-device copies of later panels, the products of earlier ones
 *     (on `stream`, through gemm()) and the device-to-host copies of
 *     finished ones overlap.
 *   - Stream order: the copies of A, B and C start after the work already
 *     enqueued on `stream`, and D is complete on the host when `stream`
 *     has completed this call (for example after cudaStreamSynchronize).
 *     The host buffers must stay unchanged until then.
 *   - Consecutive calls on one stream are ordered; calls on one stream from
 *     several threads must be serialised by the caller.
 *   - CUDA graphs: a call inside a capture of `stream` needs the staging
 *     set up by an earlier call on that stream with at least these sizes
 *     (else GEMM_ERR_CUDA); the captured copies then read and write the
 *     same host buffers on every replay.  Staging that a capture used
 *     stays allocated when later calls outgrow it, so replays stay valid.
 * Returns GEMM_OK or a GEMM_ERR_* code; argument errors (including host
 * buffers that overlap) are detected before anything is enqueued.  An
 * error from a later step (a CUDA call, or gemm() refusing a panel) leaves
 * the copies already enqueued ordered before the rest of `stream`, as on
 * success: the host buffers must stay unchanged until `stream` has
 * completed; D is then partly written.
 */
GEMM_API int gemm_host(void* D, const void* A, const void* B, const void* C,
                       int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd,
                       int transA, int transB, float alpha, float beta,
                       int in_dtype, int out_dtype, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
