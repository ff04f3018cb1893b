/*
 * mxgemm.h -- C ABI of libmxgemm.so: the MX block-scaled NT GEMM on one
 * NVIDIA GB300 (sm_103a).
 *
 *   C[M,N] = sum_j 2^(SA[m,j]-127) * 2^(SB[n,j]-127) * sum_{t<32} a[m,32j+t] * b[n,32j+t]
 *
 * with A (M x K) and B (N x K) both stored row-major ("NT": K is the contiguous
 * dimension of both operands), one E8M0 scale per 32 consecutive K values,
 * FP32 accumulation and FP32 or BF16 output.
 *
 * Where the operation is defined:
 *  - "Accelerating PyTorch on AMD GPUs with FlyDSL" (English digest), section
 *    "API compatibility is not universal input coverage": the MXFP scaled GEMM
 *    needs specific row/column layouts, one E8M0 scale per 32 values along K,
 *    and K divisible by 128; incompatible layouts may add copies.
 *  - Same page, section "Performance numbers need their baselines": the MXFP8 /
 *    MXFP4 scaled GEMMs are timed from already-quantised inputs; quantisation,
 *    compilation and initial tuning are outside the measurement.
 *  - AI-compiler daily digest of 2026-10-22, item 1 (FlyDSL): the scaled GEMMs
 *    scale blocks of 1 x 32 values with E8M0 scales and accumulate in FP32.
 *  - Element encodings (not printed on the pages; OCP MX): MXFP8 elements are
 *    E4M3 (bias 7, max 448, 0x7F/0xFF NaN), MXFP4 elements are E2M1 packed two
 *    per byte (element 2i in the low nibble), E8M0 is 2^(code-127) with 0xFF NaN.
 *
 * Conventions for every call:
 *  - Pointers named A, B, SA, SB, C, src, dst, workspace are DEVICE pointers
 *    (cudaMalloc / PyTorch CUDA memory on the current device).  The caller owns
 *    all device memory; the library never allocates device memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Launching calls are stream-ordered and asynchronous; they return once the
 *    work is enqueued.
 *  - Every call returns an int status: MXGEMM_OK (0) or a negative MXGEMM_ERR_*.
 *    Arguments are validated before anything is launched; on an error nothing
 *    is launched and no output is touched.  No call aborts or throws.
 *  - A plan is a host object; it is not thread-safe (one thread per plan).
 *  - On its first use on a device the library caches per-device state: the
 *    kernels' shared-memory opt-in, the device addresses of its own device
 *    variables (the status word, the stream-K arrival counters, the
 *    mxgemm_run_noalloc scratch) and the
 *    device's properties.  cudaDeviceReset discards what the cache refers to;
 *    a process that resets a device must not call this library on that
 *    device again (the cached addresses would be stale).
 */
#ifndef MXGEMM_H
#define MXGEMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MXGEMM_API __attribute__((visibility("default")))
#else
#define MXGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element format of A and B (both operands use the same format). */
typedef enum {
    MXGEMM_FMT_MXFP8_E4M3 = 1, /* one E4M3 code per byte: row = K bytes        */
    MXGEMM_FMT_MXFP4_E2M1 = 2, /* two E2M1 codes per byte: row = K/2 bytes     */
    MXGEMM_FMT_BF16 = 3        /* plain BF16, no scales: row = 2K bytes         */
} mxgemm_format_t;

/* Output element type of C (row-major M x N, leading dimension N). */
typedef enum {
    MXGEMM_OUT_F32 = 1,  /* FP32: the accumulator, unrounded                     */
    MXGEMM_OUT_BF16 = 2  /* BF16: the FP32 accumulator rounded to nearest-even   */
} mxgemm_out_t;

/* Status codes. */
#define MXGEMM_OK                   0
#define MXGEMM_ERR_ARG             -1  /* NULL pointer or unknown enum / flag      */
#define MXGEMM_ERR_SHAPE           -2  /* M, N <= 0, K <= 0 or K % 128 != 0        */
#define MXGEMM_ERR_ALIGN           -3  /* a device pointer is not 16-byte aligned  */
#define MXGEMM_ERR_WORKSPACE       -4  /* workspace NULL or smaller than required  */
#define MXGEMM_ERR_ARCH            -5  /* current device is not sm_103             */
#define MXGEMM_ERR_CUDA            -6  /* a CUDA runtime/driver call failed        */
#define MXGEMM_ERR_DEVICE_TIMEOUT  -7  /* a kernel gave up waiting (see below)     */
#define MXGEMM_ERR_UNSUPPORTED     -8  /* valid request this build does not serve  */
#define MXGEMM_ERR_DEVICE_BOUNDS   -9  /* debug build: a kernel skipped an access  */

/* Plan flags (mxgemm_plan_create).  0 = the library's per-shape heuristic. */
#define MXGEMM_PLAN_FORCE_BN128     (1u << 0)  /* force a 128-wide N tile             */
#define MXGEMM_PLAN_FORCE_BN256     (1u << 1)  /* force a 256-wide N tile             */
#define MXGEMM_PLAN_FORCE_NOSWAP    (1u << 2)  /* never compute C^T = B*A^T           */
#define MXGEMM_PLAN_FORCE_SWAP      (1u << 3)  /* always compute C^T = B*A^T          */
#define MXGEMM_PLAN_FORCE_PAIR      (1u << 4)  /* 256-row tiles on CTA pairs          */
#define MXGEMM_PLAN_FORCE_SINGLE    (1u << 5)  /* 128-row tiles, one CTA per tile     */
/* (bit 6 is not a flag: passing it gives MXGEMM_ERR_ARG)                     */
#define MXGEMM_PLAN_STREAMK         (1u << 7)  /* spread the last wave's k-stages     */
#define MXGEMM_PLAN_SPLITK_SHIFT    8          /* bits 8..15: forced split-K (0=auto) */
#define MXGEMM_PLAN_NO_STREAMK      (1u << 16) /* whole tiles only (no stream-K)      */
#define MXGEMM_PLAN_FORCE_BN192     (1u << 17) /* 256 x 192 tiles on CTA pairs        */

/* Run flags (mxgemm_run). */
#define MXGEMM_RUN_SA_PRELAYOUT     (1u << 0)  /* SA is already in the tile layout    */
#define MXGEMM_RUN_SB_PRELAYOUT     (1u << 1)  /* SB is already in the tile layout    */
#define MXGEMM_RUN_PREPARED         (1u << 2)  /* mxgemm_prepare ran on this workspace */
#define MXGEMM_RUN_B_STATIC         (1u << 3)  /* no kernel still running writes B    */

typedef struct mxgemm_plan *mxgemm_plan_t;

/*
 * Create a plan for C[M,N] = A[M,K] * B[N,K]^T.
 *   fmt:   mxgemm_format_t; out: mxgemm_out_t; flags: MXGEMM_PLAN_* (0 = auto).
 *   MXGEMM_FMT_BF16 plans the plain BF16 NT GEMM on the same kernels (the
 *   FlyDSL page's BF16 "NT GEMM" comparison set, section "Performance numbers
 *   need their baselines"): K a multiple of 64, SA / SB not read (may be NULL),
 *   no workspace for scales.
 * Validates the shape (M, N >= 1; K >= 128 and K % 128 == 0, per the FlyDSL
 * page's K constraint), checks that the current device is an sm_103 part,
 * chooses the tile shape, operand roles (swap-AB), split-K and stream-K, and
 * sizes the workspace.  Host memory only.  On success *plan receives a new plan.
 * Stream-K (256-wide tiles): when the last wave of tiles would leave more than
 * 10% of the SMs idle, its tiles are cut along K between CTAs and each cut
 * tile's partial sums are added in k order inside the kernel (the result does
 * not depend on the run); MXGEMM_PLAN_STREAMK forces it where the last wave is
 * under 95% full, MXGEMM_PLAN_NO_STREAMK keeps whole tiles.
 * 256 x 192 CTA-pair tiles are planned where 256-wide pair tiles would fill
 * less than a wave of pairs and could not be split two ways within one;
 * MXGEMM_PLAN_FORCE_BN192 forces them (MXGEMM_ERR_UNSUPPORTED where pair tiles
 * cannot serve the shape: MXFP4 with K % 256 != 0; MXGEMM_ERR_ARG together
 * with another tile-width, single-CTA or stream-K flag).
 */
MXGEMM_API int mxgemm_plan_create(mxgemm_plan_t *plan, int64_t M, int64_t N, int64_t K,
                       int fmt, int out, uint32_t flags);

/* Free a plan (NULL is accepted). */
MXGEMM_API int mxgemm_plan_destroy(mxgemm_plan_t plan);

/*
 * Bytes of device workspace mxgemm_run needs for this plan (0 for NULL plan):
 * the tile-layout copies of SA and SB (unless both are passed pre-laid-out),
 * split-K partial sums, and for stream-K plans the cut tiles' partial sums.
 * The workspace holds nothing between calls.  Alignment: 256 bytes.
 * A stream-K plan's arrival counters live in a device array inside the
 * library (64 Ki counters per device): each plan takes its own range when it
 * is created and returns it when destroyed, and every completed launch leaves
 * its counters at zero, so no launch zeroes anything first.  Consequences: two
 * launches of the same plan must not overlap on the GPU (order them, as for a
 * shared workspace); launches of different plans may.  If the array is full, a
 * new plan keeps its counters in its workspace instead (zeroed by every run).
 * A launch that gave up on a wait (MXGEMM_ERR_DEVICE_TIMEOUT) may leave
 * counters nonzero: read the status with mxgemm_device_status(stream, 1),
 * which then zeroes the array, before any further launch.
 */
MXGEMM_API size_t mxgemm_workspace_bytes(mxgemm_plan_t plan);

/*
 * Write a one-line, NUL-terminated description of the plan's choices
 * (tile, roles, split, grid) into buf (at most len bytes).
 */
MXGEMM_API int mxgemm_plan_describe(mxgemm_plan_t plan, char *buf, size_t len);

/*
 * Bytes of a tile-layout scale tensor for `rows` operand rows and K:
 *   ceil(rows/128) * 128 * (K/32).  Returns 0 if rows < 1 or K % 128 != 0.
 */
MXGEMM_API size_t mxgemm_sf_bytes(int64_t rows, int64_t K);

/*
 * Scale relayout: row-major E8M0 scales -> the tensor-core tile layout.
 *   src: rows x (K/32) bytes, row-major (scale of row r, K-block j at r*(K/32)+j).
 *   dst: mxgemm_sf_bytes(rows, K) bytes.  Layout: 512-byte tiles ordered
 *        [ceil(rows/128)][K/128]; inside the tile of row block R and K-tile T,
 *        the scale of row r = 128R + 32q + p (q < 4, p < 32) and K-block
 *        j = 4T + c (c < 4) sits at byte p*16 + q*4 + c.  Rows past `rows`
 *        are filled with code 127 (x1.0).
 * This is the copy the FlyDSL page warns about ("incompatible layouts may
 * introduce copies"); it is a separate, HBM-bound kernel so its cost can be
 * timed on its own.  A weight's scales need it once; pass the result to
 * mxgemm_run with MXGEMM_RUN_SB_PRELAYOUT to skip it afterwards.
 * Errors: MXGEMM_ERR_ARG (NULL), MXGEMM_ERR_SHAPE, MXGEMM_ERR_ALIGN (src or
 * dst not 16-byte aligned), MXGEMM_ERR_CUDA (launch failed).
 */
MXGEMM_API int mxgemm_relayout_scales(const uint8_t *src, int64_t rows, int64_t K,
                           uint8_t *dst, void *stream);

/* Input element type of mxgemm_quantize. */
#define MXGEMM_IN_F32               1          /* FP32, 4 bytes per value             */
#define MXGEMM_IN_BF16              2          /* BF16, 2 bytes per value             */

/* Quantise flags (mxgemm_quantize). */
#define MXGEMM_QUANT_SF_TILED       (1u << 0)  /* write scales in the tile layout     */

/*
 * MX quantiser: x [rows, K] (FP32 or BF16, row-major) -> element codes in the
 * operand format mxgemm_run reads, plus one E8M0 scale per 32 values along K.
 * The step that precedes the GEMM: the FlyDSL page (English digest, section
 * "Performance numbers need their baselines") times the scaled GEMMs from
 * already-quantised inputs and prints no quantisation formula.  The recipe
 * used here, per row and 32-value block (the same reading as the oracle):
 *     s = max(floor(log2 amax) - e_max, -127)   e_max = 8 (E4M3), 2 (E2M1);
 *     an all-zero block takes s = 0; scale code = s + 127;
 *     code = x / 2^s rounded to the nearest E4M3 / E2M1 value, ties to even,
 *            saturating at +-448 / +-6 (a zero keeps the sign of x);
 *     a block holding a NaN or an infinity: scale code 0xFF, all codes 0.
 *   fmt:      mxgemm_format_t of the codes.
 *   in_dtype: MXGEMM_IN_F32 or MXGEMM_IN_BF16.
 *   x:        device, rows x K values, 32-byte aligned, read-only.
 *   codes:    device, rows x K bytes (MXFP8) or rows x K/2 bytes (MXFP4,
 *             element 2i in the low nibble), 16-byte aligned; overwritten.
 *   scales:   device, 16-byte aligned; overwritten.  Without flags:
 *             rows x K/32 bytes row-major (the SA/SB input of mxgemm_run).
 *             With MXGEMM_QUANT_SF_TILED: mxgemm_sf_bytes(rows, K) bytes in
 *             the tile layout of mxgemm_relayout_scales (padding rows = 127),
 *             ready for mxgemm_run with MXGEMM_RUN_SA_PRELAYOUT (or _SB_) --
 *             this skips the relayout copy the FlyDSL page ("API
 *             compatibility is not universal input coverage") warns about.
 *   K:        multiple of 32; a multiple of 128 with MXGEMM_QUANT_SF_TILED.
 * One stream-ordered kernel launch, no allocation.
 * Errors: MXGEMM_ERR_ARG (NULL pointer, unknown fmt / in_dtype / flag),
 * MXGEMM_ERR_SHAPE (rows < 1, K not as above), MXGEMM_ERR_ALIGN,
 * MXGEMM_ERR_ARCH, MXGEMM_ERR_CUDA (launch failed).
 */
MXGEMM_API int mxgemm_quantize(int fmt, int in_dtype, const void *x, int64_t rows, int64_t K,
                               void *codes, uint8_t *scales, uint32_t flags, void *stream);

/*
 * Run the GEMM on `stream`.
 *   A:  M x K codes (fmt-dependent bytes per row, row-major, 16-byte aligned)
 *   SA: M x K/32 scales, row-major -- or, with MXGEMM_RUN_SA_PRELAYOUT,
 *       mxgemm_sf_bytes(M,K) bytes in the tile layout of mxgemm_relayout_scales
 *   B, SB: the same for the N x K operand (MXGEMM_RUN_SB_PRELAYOUT)
 *   C:  M x N output, row-major, element type per the plan's `out`
 *   workspace / ws_bytes: at least mxgemm_workspace_bytes(plan) bytes
 *       (may be NULL/0 if that is 0)
 * Enqueues (1) the relayout of whichever scales are not pre-laid-out and
 * (2) the persistent tcgen05 block-scaled GEMM kernel (3) a split-K reduce if
 * the plan splits K.  MXFP8 plans on 256-row CTA-pair tiles with
 * K % 512 == 0 (their description says "sa=in-kernel") lay out row-major SA
 * inside the GEMM kernel instead of step (1): one CTA of each pair loads the
 * pair's row-major scales and writes the tile layout in shared memory.
 * Inputs are read-only; C is fully overwritten.
 * MXGEMM_RUN_B_STATIC: the caller promises that B (the weight) is not written
 * by any kernel that may still be running on `stream` when this call starts
 * (weights loaded once and only read; the preceding kernels produce A).  The
 * GEMM's CTAs may then start loading B before the preceding kernel completes
 * (programmatic dependent launch); A, SA and SB are still read only after it.
 * Used by the weight-streaming decode plans ("lean" in their description);
 * other plans ignore it.  Breaking the promise gives wrong results, not a fault.
 * A plan belongs to the device that was current when it was created; running
 * it with another device current returns MXGEMM_ERR_ARG.
 * Errors: MXGEMM_ERR_ARG, MXGEMM_ERR_ALIGN, MXGEMM_ERR_WORKSPACE,
 * MXGEMM_ERR_CUDA.  A device-side wait that exceeds its limit is reported by
 * mxgemm_device_status(), not here (the call is asynchronous).
 */
MXGEMM_API int mxgemm_run(mxgemm_plan_t plan, const void *A, const uint8_t *SA,
               const void *B, const uint8_t *SB, void *C,
               void *workspace, size_t ws_bytes, uint32_t run_flags, void *stream);

/*
 * Step (1) of mxgemm_run on its own: lays out whichever of SA / SB is not
 * flagged MXGEMM_RUN_S{A,B}_PRELAYOUT into `workspace` in one launch on
 * `stream` (none when there is nothing to lay out); a plan whose stream-K
 * counters did not fit in the library's array also has them reset here.  A
 * following mxgemm_run on the same workspace and stream with
 * MXGEMM_RUN_PREPARED (plus the same PRELAYOUT flags) then enqueues only the
 * GEMM (and its split-K reduce): the scales laid out here are read from the
 * workspace, so mxgemm_run's SA / SB arguments without a PRELAYOUT flag are
 * not read and may be NULL -- except SA for a plan that lays it out inside the
 * GEMM ("sa=in-kernel" in its description): mxgemm_prepare leaves SA alone
 * and mxgemm_run reads it.  Lets a caller time
 * or schedule the two steps separately (the extra layout copies the FlyDSL page
 * warns about are step (1)).  Nothing else may use the workspace in between.
 *   SA, SB:  row-major scales as for mxgemm_run (pre-laid-out ones not read;
 *            all ignored for MXGEMM_FMT_BF16)
 * Errors: MXGEMM_ERR_ARG (NULL plan, unknown flag, missing scales, another
 * device current), MXGEMM_ERR_ALIGN, MXGEMM_ERR_WORKSPACE, MXGEMM_ERR_CUDA.
 * mxgemm_run_noalloc rejects MXGEMM_RUN_PREPARED (its scratch is internal).
 */
MXGEMM_API int mxgemm_prepare(mxgemm_plan_t plan, const uint8_t *SA, const uint8_t *SB,
                   void *workspace, size_t ws_bytes, uint32_t run_flags, void *stream);

/* Time limit, in nanoseconds of GPU global time, of every barrier wait inside
 * the GEMM kernels launched by mxgemm_run, mxgemm_run_noalloc and
 * mxgemm_grouped_run (mxgemm_selftest_stall uses 20 ms). */
#define MXGEMM_WAIT_LIMIT_NS 2000000000ull

/*
 * Synchronise `stream` and return the library's sticky device status on the
 * current device: MXGEMM_OK, or MXGEMM_ERR_DEVICE_TIMEOUT if any kernel since
 * the last reset gave up on a barrier wait (every wait in the kernels has a
 * time limit of MXGEMM_WAIT_LIMIT_NS, two seconds; on expiry the kernel records
 * the error, drains its own in-flight work and exits instead of hanging).  If
 * `reset` is nonzero the status is cleared after reading; if it was a timeout,
 * the library's stream-K arrival counters are zeroed as well (call it with no
 * other launch of this library in flight on the device).  MXGEMM_ERR_CUDA if
 * the synchronisation itself fails.
 */
MXGEMM_API int mxgemm_device_status(void *stream, int reset);

/*
 * Self-test of the device timeout path: launches the GEMM of `plan` with its
 * loader switched off, so no data ever arrives and every barrier wait in the
 * kernel expires after ~20 ms.  The kernel then records
 * MXGEMM_ERR_DEVICE_TIMEOUT, frees its TMEM and exits; C is left unwritten.
 * SA and SB are taken as pre-laid-out and are not read.  Returns the launch
 * status; read the device status with mxgemm_device_status().  Used by the
 * test suite to show that a stalled kernel returns instead of hanging.
 */
MXGEMM_API int mxgemm_selftest_stall(mxgemm_plan_t plan, const void *A, const uint8_t *SA,
                          const void *B, const uint8_t *SB, void *C,
                          void *workspace, size_t ws_bytes, void *stream);

/*
 * Debug build.  The library is also built with MXGEMM_DEBUG defined
 * (libmxgemm_debug.so beside libmxgemm.so; the Python binding loads it when
 * the environment variable MXGEMM_DEBUG=1).  Same entry points; in it
 *   - every plain global load and store of the GEMM kernels (C or the split-K
 *     slabs, the stream-K partial sums and arrival counters) is checked
 *     against its buffer's extent, vector stores also against their
 *     alignment; a failing access is skipped and MXGEMM_ERR_DEVICE_BOUNDS is
 *     written to the device status word (no trap);
 *   - mxgemm_run and mxgemm_run_noalloc fill C with NaN (all-ones bytes)
 *     before the GEMM, so an element no kernel writes reads back as NaN;
 *   - mxgemm_run, mxgemm_run_noalloc and mxgemm_grouped_run synchronise their
 *     stream and return the device status word (so they cannot be captured in
 *     a CUDA graph).
 * mxgemm_debug_build() returns 1 in the debug build, 0 in the release build.
 */
MXGEMM_API int mxgemm_debug_build(void);

/*
 * Self-test of the debug build's bounds checks: runs `plan` (arguments as for
 * mxgemm_run) with the GEMM kernel told that C ends one row early, so the
 * stores of the last row are out of its range.  The debug build skips them
 * (the last row of C keeps the NaN fill; with swap-AB tiles, whose stores run
 * down the columns of C, every 32-row group of stores that touches it) and
 * returns MXGEMM_ERR_DEVICE_BOUNDS, the rest of C being the product; clear
 * the status afterwards with mxgemm_device_status(stream, 1).  Plans that
 * split K (C written by the reduce pass) give MXGEMM_ERR_UNSUPPORTED, and so
 * does the release build.
 */
MXGEMM_API int mxgemm_selftest_bounds(mxgemm_plan_t plan, const void *A, const uint8_t *SA, const void *B,
                                      const uint8_t *SB, void *C, void *workspace, size_t ws_bytes,
                                      uint32_t run_flags, void *stream);

/*
 * mxgemm_run without a workspace argument, for callers that cannot allocate
 * device memory.  (The FlyDSL pages have no counterpart: this is an interface
 * convenience of this library, not part of the method.)
 *
 * Who needs it: callers that own only their inputs and outputs and may not
 * call cudaMalloc (or any allocating routine) around a GEMM -- e.g. a serving
 * loop whose device memory was planned once at start-up, where a cudaMalloc
 * would synchronise the device and can fail once memory is fragmented, or a
 * plain C host program with no allocator of its own to hand a workspace over.
 *
 * The scratch it uses instead (tile-layout scales, split-K partial sums) is
 * one static device array of MXGEMM_NOALLOC_SCRATCH_BYTES inside the library.
 * Every GPU that loads the library holds that array until the process exits.
 *   - Plans whose mxgemm_workspace_bytes() exceeds MXGEMM_NOALLOC_SCRATCH_BYTES
 *     are rejected with MXGEMM_ERR_WORKSPACE before anything is launched.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents.  Calls that overlap on the GPU (different streams without
 *     ordering between them, or several host threads) race on it: order them.
 *     Nothing in the array needs to start at zero -- each call rewrites every
 *     byte it later reads.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: after a cudaDeviceReset of that device it is stale (see the
 *     conventions at the top of this file).
 * Arguments, results and errors are otherwise those of mxgemm_run.  No
 * cudaMalloc, cudaFree or other allocating call is made.
 */
#define MXGEMM_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
MXGEMM_API int mxgemm_run_noalloc(mxgemm_plan_t plan, const void *A, const uint8_t *SA,
                                  const void *B, const uint8_t *SB, void *C,
                                  uint32_t run_flags, void *stream);

/*
 * Grouped (mixture-of-experts) MX GEMM.  G groups ("experts"); group e owns the
 * token rows [offsets[e], offsets[e+1]) of A and of C and the weight rows
 * [e*N, (e+1)*N) of B:
 *     C[r, n] = sum_j 2^(SA[r,j]-127) * 2^(SB[e*N+n,j]-127) * sum_{t<32} a[r,32j+t] * b[e*N+n,32j+t]
 * for every row r of group e, i.e. one MX NT GEMM per group.  The FlyDSL page
 * (English digest, "Performance numbers need their baselines") times grouped
 * GEMMs with uniform groups, varied projection dimensions and uneven expert
 * loads; the AI-compiler daily of 2026-10-22 (item 1) names persistent expert
 * scheduling.  Here one persistent kernel walks the tiles of all groups; each
 * CTA reads the offsets from device memory, so group sizes may be produced on
 * the GPU (by a router) without a host round trip.
 */
typedef struct mxgemm_grouped_plan *mxgemm_grouped_plan_t;

/*
 * Plan a grouped GEMM for `groups` groups (1..512), `rows` token rows in total
 * (the row count of A and C: T), N weight rows per group (a multiple of 128,
 * so that every group's weight scales start on a 128-row scale tile) and K
 * (a multiple of 128).  fmt / out as for mxgemm_plan_create; flags: any of
 * MXGEMM_PLAN_FORCE_{SWAP,NOSWAP,BN128,BN256,PAIR,SINGLE} (others:
 * MXGEMM_ERR_ARG).  By default the weights fill the 128-row MMA dimension
 * (swap-AB) when the expected tokens per group, rows / groups, are at most
 * 64, and groups of at least 512 tokens on average run 256 x 256 CTA-pair
 * tiles (token tiles of 256 rows inside each group; not swapped, N >= 256,
 * MXFP4 with K % 256 == 0).  Host memory only.
 * Errors: MXGEMM_ERR_ARG, MXGEMM_ERR_SHAPE, MXGEMM_ERR_UNSUPPORTED (sizes past
 * the kernel's 32-bit indices), MXGEMM_ERR_ARCH.
 */
MXGEMM_API int mxgemm_grouped_plan_create(mxgemm_grouped_plan_t *plan, int64_t groups, int64_t rows, int64_t N,
                                          int64_t K, int fmt, int out, uint32_t flags);

/* Free a grouped plan (NULL is accepted). */
MXGEMM_API int mxgemm_grouped_plan_destroy(mxgemm_grouped_plan_t plan);

/* Device workspace bytes of mxgemm_grouped_run (0 for NULL): the tokens'
 * per-group tile-layout scales and the weights' tile-layout scales. */
MXGEMM_API size_t mxgemm_grouped_workspace_bytes(mxgemm_grouped_plan_t plan);

/* One-line description of the grouped plan's choices. */
MXGEMM_API int mxgemm_grouped_plan_describe(mxgemm_grouped_plan_t plan, char *buf, size_t len);

/*
 * Run the grouped GEMM on `stream`.
 *   group_offsets: device, G + 1 int64 row offsets, non-decreasing, in
 *       [0, rows]; 8-byte aligned.  Read on the device by every launch.
 *       Rows of C outside every group are not written.  Offsets that break
 *       these rules give unspecified results but no out-of-range access: each
 *       group's rows are clamped to [0, rows] before use.
 *   A, SA: rows x K codes (K or K/2 bytes per row) and rows x K/32 row-major
 *       scales (laid out per group inside the call).
 *   B, SB: G*N x K codes (group e's weight in rows [e*N, (e+1)*N)) and G*N x
 *       K/32 row-major scales -- or, with MXGEMM_RUN_SB_PRELAYOUT, the tile
 *       layout of mxgemm_relayout_scales over all G*N rows (a weight's scales
 *       need laying out once).
 *   C: rows x N, row-major, element type per the plan.
 * All device pointers but group_offsets 16-byte aligned.  Launches: the
 * per-group token-scale relayout, the weight-scale relayout (unless
 * pre-laid-out) and the persistent grouped GEMM kernel.
 * Errors: MXGEMM_ERR_ARG (NULL, unknown run flag, a plan of another device),
 * MXGEMM_ERR_ALIGN, MXGEMM_ERR_WORKSPACE, MXGEMM_ERR_CUDA.
 */
MXGEMM_API int mxgemm_grouped_run(mxgemm_grouped_plan_t plan, const int64_t *group_offsets, const void *A,
                                  const uint8_t *SA, const void *B, const uint8_t *SB, void *C, void *workspace,
                                  size_t ws_bytes, uint32_t run_flags, void *stream);

/*
 * Scale-placement checker for MXFP4 dot products ("Deciding Scale Placement in
 * MXFP4 Dot Products with Integer Arithmetic", AI-compiler daily digest of
 * 2026-10-22, item 2): for each scale pair (sa[p], sb[p]) (E8M0 codes 0..254)
 * and every tuple of k (1..4) E2M1 elements per operand -- 16^(2k) tuples,
 * numbered t = sum a_i << 4i + sum b_i << 4(k+i) over the 4-bit codes --
 * compare, in binary32 with every operation rounded to nearest even and no
 * fused multiply-add (f_a = 2^(sa-127), f_b = 2^(sb-127)):
 *     pre  = tree( (a_i f_a) (b_i f_b) )      scales applied to the elements
 *     post = (tree( a_i b_i ) f_a) f_b        scales applied to the sum
 *     rn   = sum a_i b_i * 2^(sa+sb-254) rounded once to binary32
 * with tree(n) = tree(first ceil(n/2)) + tree(rest); equal = both NaN or equal
 * values.  Writes counts[3p] = #(pre != post), counts[3p+1] = #(pre == rn),
 * counts[3p+2] = #(post == rn), first_diff[p] = the smallest t with
 * pre != post, or -1; a scale code outside 0..254 gives -1 in all four.
 *   sa, sb: device int32[npairs]; counts: device int64[3*npairs]; first_diff:
 *   device int64[npairs].  Stream-ordered; k = 4 costs 4.3e9 tuples per pair.
 * Errors: MXGEMM_ERR_ARG (NULL), MXGEMM_ERR_SHAPE (k, npairs outside 1..4,
 * 1..2^24), MXGEMM_ERR_ALIGN, MXGEMM_ERR_ARCH, MXGEMM_ERR_CUDA.
 */
MXGEMM_API int mxgemm_placement_scan(int k, const int *sa, const int *sb, int npairs, long long *counts,
                                     long long *first_diff, void *stream);

/*
 * Tensor-pipe rate probe: the ceiling the GEMM kernels are measured against.
 * Every SM (cta_group 1) or CTA pair (cta_group 2, clusters of 2) holds four
 * operand sets in shared memory and issues `stages` k-stages of back-to-back
 * tcgen05.mma into one TMEM accumulator, with no global loads; each k-stage
 * is 128 bytes of K per row (4 MMAs: K = 32 for MXFP8, 64 for MXFP4 (two per
 * 128-element scale tile), 16 for BF16), M = 128 per CTA (256 per pair) and
 * N = `n` (128 or 256) columns.  scale_copies = 1 also issues, per k-stage,
 * the tcgen05.cp copies of the stage's scale chunks into TMEM that a GEMM
 * k-stage issues (ignored for BF16).  The operand values are fixed finite
 * codes with scale 1; the products are not read.
 *   fmt:     MXGEMM_FMT_MXFP8_E4M3, MXGEMM_FMT_MXFP4_E2M1 or MXGEMM_FMT_BF16
 *   stages:  16 .. 2^22 (4 * stages MMAs per unit; ~4096 lasts ~1 ms)
 *   result:  host double[4], written on success:
 *            [0] cycles per MMA (SM clock, mean over units),
 *            [1] SM clock during the run in GHz (clock64 over globaltimer),
 *            [2] dense PFLOP/s of the whole GPU (all units' MMAs over the
 *                span from the first unit's start to the last unit's end),
 *            [3] units that ran (SMs, or pairs).
 * Synchronous: launches a short warm-up and the measured kernel on `stream`
 * and waits for them.  Uses a static device array of the library (no
 * allocation); calls must not overlap.  Each unit waits for its MMAs with a
 * two-second limit.
 * Errors: MXGEMM_ERR_ARG (NULL result, fmt / cta_group / n / scale_copies /
 * stages out of range), MXGEMM_ERR_ARCH, MXGEMM_ERR_CUDA,
 * MXGEMM_ERR_DEVICE_TIMEOUT (a unit's wait expired).
 */
MXGEMM_API int mxgemm_probe_tensor_rate(int fmt, int cta_group, int n, int scale_copies, int stages,
                                        double *result, void *stream);

/* Static, human-readable name of a status code. */
MXGEMM_API const char *mxgemm_status_str(int status);

/* Library version: major*10000 + minor*100 + patch. */
MXGEMM_API int mxgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXGEMM_H */
