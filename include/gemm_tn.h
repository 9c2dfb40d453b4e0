/*
 * gemm_tn.h -- C ABI of the GB300 (sm_103a) fp16 TN GEMM library.
 *
 * Operation (page "Reading CuTe's make_tiled_mma: how one MMA tiles into a
 * matrix", section "Fix the matrices and directions first"):
 *
 *     D(m,n) = C(m,n) + sum_{k<K} A(m,k) * B(n,k)
 *
 * with A of logical shape (M,K), B of logical shape (N,K) -- B(n,k) is the
 * usual right-hand matrix read as B_math(k,n) -- and C/D of shape (M,N).
 * "TN" names the operand form of the tensor-core instruction, not a memory
 * order; memory order is given separately per operand.
 *
 * Operand views (page "CuTe Layout to Tensor Core", sections 1 "the outermost
 * level: a matrix is a Shape + Stride layout" and 2 "Tensor = Pointer +
 * Layout"): an operand is a pointer plus a two-mode shape:stride layout in
 * which one mode is stride-1.
 *   A, a_major == GEMM_TN_MAJOR_K : (M,K):(ldA,1), ldA >= K
 *   A, a_major == GEMM_TN_MAJOR_MN: (M,K):(1,ldA), ldA >= M
 *   B, b_major == GEMM_TN_MAJOR_K : (N,K):(ldB,1), ldB >= K
 *   B, b_major == GEMM_TN_MAJOR_MN: (N,K):(1,ldB), ldB >= N
 *   C/D                           : (M,N):(ldC,1), ldC >= N
 * All elements are IEEE binary16.
 *
 * C and D share one buffer: each element of C is read before the element of
 * D at the same position is written.  (Page "Reading CuTe's retile_D",
 * section "How the two fragments are handed to the MMA", accumulates the
 * product onto C in place.)  gemm_tn_scaled and gemm_tn_batched below add
 * the alpha / beta form with a separate D, and a batch of problems.
 *
 * Accumulation (same page, section "From CuTe's name to the instruction";
 * make_tiled_mma page, section "Fix the matrices and directions first"):
 *   GEMM_TN_ACC_F32: the products are summed in fp32, C is converted to fp32
 *                    and added, and the sum is rounded once to fp16
 *                    (round-to-nearest-even): the F32F16F16F32 form.
 *   GEMM_TN_ACC_F16: the products are summed in an fp16 accumulator and C is
 *                    added in fp16: the F16F16F16F16 form.
 *
 * Ownership: the caller owns A, B, C and D (device memory); the library never
 * frees or retains caller memory.  Workspaces (the skinny path's split-K
 * partial sums, stream-K partial tiles, repacked strided operands) come from
 * a memory pool the library creates for each device on the first call of
 * an entry point that may need one: taken with cudaMallocFromPoolAsync on
 * the call's stream and returned with cudaFreeAsync on the same stream, so
 * calls on different streams never share them.  The pool keeps up to 1 GiB
 * cached between calls and lives until process exit (see
 * gemm_tn_skinny_noalloc for a variant that neither allocates nor creates
 * the pool).  When the pool cannot serve a request, a workspace the caller
 * asked for (the skinny path, an explicit K split, the forced repack route)
 * makes the call return GEMM_TN_ERR_NO_MEMORY with nothing enqueued; one
 * the library chose by itself (an automatic K split, stream-K, the
 * automatic repack route) is dropped and the call runs without it.
 *
 * Graphs: the first call on a device sets the library up (kernel attributes,
 * the workspace pool); after that, calls can be recorded by stream capture
 * and replayed (the workspace of the skinny and stream-K paths is then a
 * graph memory node).
 *
 * Ordering: every call is asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream).  It returns once the kernels are enqueued; D is
 * valid after the stream has been synchronised.  Calls on one stream are
 * ordered; calls that may overlap on different streams must not share an
 * output buffer.  All pointers are device pointers of the current device.
 *
 * Errors: every function returns a gemm_tn_status and never aborts or throws.
 * Argument checks run before anything is enqueued, so an error return from
 * them leaves the stream untouched.
 */
#ifndef GEMM_TN_H_
#define GEMM_TN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GEMM_TN_API __attribute__((visibility("default")))
#else
#define GEMM_TN_API
#endif

typedef enum {
  GEMM_TN_MAJOR_K = 0,  /* the K mode is stride-1 */
  GEMM_TN_MAJOR_MN = 1  /* the M (for A) or N (for B) mode is stride-1 */
} gemm_tn_major;

typedef enum {
  GEMM_TN_ACC_F32 = 0,
  GEMM_TN_ACC_F16 = 1
} gemm_tn_accum;

typedef enum {
  GEMM_TN_OK = 0,
  GEMM_TN_ERR_INVALID_ARG = 1,     /* negative or too large size, ld too small,
                                      NULL pointer with a nonzero extent, bad
                                      enum, CD overlapping A or B */
  GEMM_TN_ERR_ALIGNMENT = 2,       /* a pointer not 16-byte aligned or an ld
                                      that is not a multiple of 8 elements */
  GEMM_TN_ERR_UNSUPPORTED = 3,     /* no device of compute capability 10.3 */
  GEMM_TN_ERR_CUDA = 4,            /* a CUDA runtime / driver call failed */
  GEMM_TN_ERR_DEVICE_TIMEOUT = 5,  /* a bounded wait inside a kernel expired;
                                      that launch's D is not valid */
  GEMM_TN_ERR_NO_MEMORY = 6        /* a workspace (split-K or stream-K partial
                                      sums, repacked operands) could not be
                                      allocated */
} gemm_tn_status;

typedef enum {
  GEMM_TN_PATH_AUTO = 0,    /* skinny path with K-major A and B and fp32
                               accumulation for M <= 192, and for M <= 256
                               when N <= 14336, once K is long enough to
                               stream (K >= 2048 for M <= 32, 4096 for
                               M <= 64, 8192 above); persistent tile path
                               otherwise */
  GEMM_TN_PATH_LARGE = 1,   /* persistent tile kernels: 256x256 tiles on one
                               CTA or on a CTA pair, or 128xBN tiles */
  GEMM_TN_PATH_SKINNY = 2,  /* swapped-operand split-K kernel + reduction;
                               needs M <= 256, K-major A and B and fp32
                               accumulation */
  GEMM_TN_PATH_STRIDED_COPY = 3,   /* gemm_tn_strided_ex only: threads gather
                                      operands into shared memory; no
                                      workspace */
  GEMM_TN_PATH_STRIDED_REPACK = 4  /* gemm_tn_strided_ex only: repack views
                                      TMA cannot read into pooled buffers,
                                      then the tile kernels */
} gemm_tn_path;

/* Extra controls for gemm_tn_ex.  Zero-initialise and set what you need;
 * every zero field means "the library's default". */
typedef struct {
  int path;             /* gemm_tn_path */
  int split_k;          /* skinny path: at most this many CTAs share the K
                           loops of the output tiles, in ranges of equal
                           length (0 = one per SM).  Large path
                           with tile_kernel 1: K splits per 128-row tile;
                           with tile_kernel 2: K splits per 256 x 256 pair
                           tile; fp32 accumulation only (0 = none; with
                           tile_kernel 0 the library splits by itself when
                           the tiles would leave more than half the SMs
                           idle and K is long enough) */
  int tile_n;           /* large path, output tile width (0: the library's
                           choice).  128-row tiles (tile_kernel 1): 64, 128
                           or 256; the library takes 128 when N <= 128 or
                           when 128 x 256 tiles would leave half the SMs
                           idle, 64 when even 128 x 128 tiles would and K is
                           not split, else 256.  CTA-pair tiles (only with
                           tile_kernel 2; not with a K split): 128, 160,
                           192, 224 or 256 with a K-major B, 128 or 256
                           with an N-major B; the library takes the width
                           whose waves of tiles over the SM pairs finish
                           soonest.  Other values, or a width the chosen
                           kernel cannot run, are GEMM_TN_ERR_INVALID_ARG */
  int sync_check;       /* nonzero: synchronise `stream` after the launch and
                           return GEMM_TN_ERR_DEVICE_TIMEOUT if a kernel gave
                           up waiting (the sticky device error word is read
                           and cleared) */
  uint64_t timeout_ns;  /* limit of every in-kernel wait (0 = 1 s) */
  int test_stall;       /* TEST ONLY: nonzero makes the producer of the first
                           tile withhold one pipeline stage, so that the
                           consumer's bounded wait expires and the kernel
                           reports GEMM_TN_ERR_DEVICE_TIMEOUT instead of
                           hanging */
  int tile_kernel;      /* large path: 0 = choose (2 with a K split when
                           few 256 x 256 tiles have K loops of at least
                           2 x 4096; else 1 with 128 x 128 tiles (or
                           128 x 64) when 128 x 256 tiles would fill at most
                           half the SMs; else 2 when M and N exceed 128;
                           else 1),
                           1 = single-CTA 128 x tile_n
                           tiles, 2 = CTA-pair 256 x 256 tiles (two SMs per
                           tile, tcgen05 cta_group::2), 3 = single-CTA
                           256 x 256 tiles (tile_n is ignored by 2 and 3) */
  int stream_k;         /* CTA-pair kernel, fp32 accumulation, 256-wide
                           tiles: unless -1, when the last round of tiles
                           would leave at least half the pairs idle, its
                           tiles run as 2-4 K splits each (partial sums
                           through a workspace, added in a fixed order with
                           C once by a second kernel); 0 (default) = on.
                           Single-CTA 256 x 256 kernel, fp32 accumulation:
                           1 = split the last, partial wave of tiles over all
                           SMs (stream-K: K ranges of equal length, partial
                           sums through a workspace, added in a fixed order),
                           0 (default) or -1 = never.  The default is off
                           because the split's finishing work (partials
                           pulled through one SM per tile at the end of the
                           kernel) cost about as much as the balanced wave
                           saved on every shape measured.  The split needs a
                           workspace from the library's pool; without one
                           the call runs unsplit. */
  int test_fail_alloc;  /* TEST ONLY: nonzero makes every workspace request
                           of this call fail as an exhausted pool would, so
                           that the handling of that case can be checked:
                           the skinny path and an explicitly requested K
                           split (split_k with tile_kernel 1 or 2) return
                           GEMM_TN_ERR_NO_MEMORY with nothing enqueued; a K
                           split or stream-K the library would choose runs
                           the unsplit kernel instead; gemm_tn_strided_ex
                           falls back to the copy producer unless the
                           repack route was forced. */
  int k_stage;          /* CTA-pair kernel: K depth of a pipeline stage, 64
                           or 128 (0 = the library's choice); other values
                           are GEMM_TN_ERR_INVALID_ARG */
  int trace;            /* nonzero: the call's GEMM kernel (not a K split's
                           reduction) stamps a phase trace per CTA into the
                           library's trace buffer, which gemm_tn_trace_read
                           returns (the buffer is cleared on the stream
                           first; one buffer per device, so traced calls
                           that overlap on the GPU mix their records) */
  int host_panel_rows;  /* gemm_tn_host: rows of M per panel (rounded up to a
                           multiple of 8; 0 = the library's choice: all of M
                           up to 1024 rows, else panels of ceil(M / 8)
                           rounded up to 256 rows and at least 512 -- without
                           host_inputs_ready the last one cut into a half
                           and two quarters so that little work is left
                           after the last copy-in; more than 64 panels are
                           merged to 64) */
  int host_inputs_ready; /* gemm_tn_host: nonzero declares that A, B and C
                           already hold their values when the call is made
                           (nothing enqueued earlier on `stream` writes
                           them), so their copies to the device need not
                           wait for that work: they start once the copies
                           in of earlier gemm_tn_host calls are done, and
                           back-to-back calls overlap.  D is still written
                           only after the earlier work on `stream`. */
} gemm_tn_options;

/*
 * D = C + A.B^T in place in CD, as described at the top of this file.
 *
 *   M, N, K      sizes, each in [0, 2^31 - 1].  M == 0 or N == 0 is a no-op;
 *                K == 0 leaves CD unchanged (D = C) without a launch.
 *   A, ldA       (M,K) operand storage and its leading dimension in elements
 *   a_major      gemm_tn_major of A
 *   B, ldB       (N,K) operand storage and its leading dimension
 *   b_major      gemm_tn_major of B
 *   CD, ldC      (M,N) row-major storage of C on entry and D on return
 *   accum_dtype  gemm_tn_accum
 *   stream       cudaStream_t the work is enqueued on
 *
 * Alignment: A, B, CD 16-byte aligned; ldA, ldB, ldC multiples of 8 (the
 * tensor-memory-access unit moves 16-byte rows).
 */
GEMM_TN_API int gemm_tn(int64_t M, int64_t N, int64_t K,
                        const void* A, int64_t ldA, int a_major,
                        const void* B, int64_t ldB, int b_major,
                        void* CD, int64_t ldC,
                        int accum_dtype, void* stream);

/* gemm_tn with explicit controls; opts may be NULL (same as gemm_tn). */
GEMM_TN_API int gemm_tn_ex(int64_t M, int64_t N, int64_t K,
                           const void* A, int64_t ldA, int a_major,
                           const void* B, int64_t ldB, int b_major,
                           void* CD, int64_t ldC,
                           int accum_dtype, void* stream,
                           const gemm_tn_options* opts);

/*
 * Scaled, batched form:
 *
 *     D_l = alpha * A_l . B_l^T + beta * C_l        for l < batch
 *
 * Page "cute(7) simple_gemm", section 8.1, checks the kernel against
 * cuBLAS's alpha / beta GEMM (D = alpha A.B^T + beta C); page "CuTe Layout
 * to Tensor Core", section 4 (local_tile), gives the extra coordinate that
 * indexes a batch.  Per problem the views are those of gemm_tn, with a
 * separate D: (M,N):(ldD,1).  Problem l's operand X starts strideX elements
 * after problem l-1's:  A_l = A + l*strideA, and so on.
 *
 *   alpha, beta  fp32 scalars.  alpha == 0 or K == 0: the product term is
 *                absent and A, B are not read (D = beta * C); beta == 0: C is
 *                not read and may be NULL (NaN or Inf stored there cannot
 *                reach D).  These are the BLAS conventions.
 *   precision    fp32 accumulation: fma(alpha, acc, beta * C) in fp32,
 *                rounded once to fp16.  fp16 accumulation: the products are
 *                summed in fp16 as in gemm_tn; with alpha = beta = 1, C is
 *                added in fp16 (exactly gemm_tn), otherwise the fp16 sum is
 *                scaled and C added in fp32 and rounded once.
 *   strides      used only when batch > 1, in elements, multiples of 8:
 *                strideA: 0 (one A for every problem) or at least one view
 *                  (M*ldA K-major, K*ldA M-major); strideB likewise;
 *                strideC: any value >= 0 (0 = one C for every problem);
 *                strideD: at least M*ldD (the problems' D do not overlap);
 *                every (batch-1)*stride at most 2^61 (INVALID_ARG above).
 *   aliasing     D may be C itself (same pointer, ldD == ldC, strideD ==
 *                strideC): each C element is read before the D element at
 *                its position is written.  Otherwise D must not overlap C;
 *                D must never overlap A or B.
 *   alignment    A, B, C, D 16-byte aligned, ld* multiples of 8
 *                (GEMM_TN_ERR_ALIGNMENT otherwise; gemm_tn_strided takes
 *                arbitrary strides for the unscaled, single-problem form).
 *   paths        one problem that GEMM_TN_PATH_AUTO sends to the skinny
 *                split-K path (small M, long K, K-major operands, fp32
 *                accumulation) takes it here too; everything else
 *                runs the tile kernels with the batch folded into the tile
 *                list (tile t belongs to problem t / tiles-per-problem).
 *   returns      as gemm_tn; M, N or batch == 0 is a no-op.
 */
GEMM_TN_API int gemm_tn_batched(int64_t M, int64_t N, int64_t K, int64_t batch, float alpha,
                                const void* A, int64_t ldA, int64_t strideA, int a_major,
                                const void* B, int64_t ldB, int64_t strideB, int b_major,
                                float beta, const void* C, int64_t ldC, int64_t strideC,
                                void* D, int64_t ldD, int64_t strideD, int accum_dtype,
                                void* stream);

/* gemm_tn_batched with explicit controls (opts may be NULL); the controls
 * mean what they mean for gemm_tn_ex. */
GEMM_TN_API int gemm_tn_batched_ex(int64_t M, int64_t N, int64_t K, int64_t batch, float alpha,
                                   const void* A, int64_t ldA, int64_t strideA, int a_major,
                                   const void* B, int64_t ldB, int64_t strideB, int b_major,
                                   float beta, const void* C, int64_t ldC, int64_t strideC,
                                   void* D, int64_t ldD, int64_t strideD, int accum_dtype,
                                   void* stream, const gemm_tn_options* opts);

/* One problem of the scaled form: D = alpha * A.B^T + beta * C
 * (gemm_tn_batched with batch 1). */
GEMM_TN_API int gemm_tn_scaled(int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                               int64_t ldA, int a_major, const void* B, int64_t ldB, int b_major,
                               float beta, const void* C, int64_t ldC, void* D, int64_t ldD,
                               int accum_dtype, void* stream);

/*
 * D = C + A.B^T for operand views with arbitrary element strides (the layout
 * page, sections 1-2: a matrix is any shape:stride view; neither mode needs
 * to be stride-1):
 *   A(m,k) = A[m*sAm + k*sAk],  B(n,k) = B[n*sBn + k*sBk],
 *   C/D(m,n) = CD[m*sCm + n*sCn]     (strides in elements, all >= 0)
 * The accumulation modes and in-place semantics are those of gemm_tn.
 * It accepts layouts gemm_tn rejects: leading dimensions that are not
 * multiples of 8, pointers that are only 2-byte aligned, and views with no
 * stride-1 mode.  Two routes:
 *   - repack: operands whose view TMA cannot read are first copied into
 *     row-major buffers from the library's stream-ordered pool (see
 *     Ownership at the top of this file), the tile kernels run
 *     on them, and D is scattered back when its view needed a copy;
 *   - copy producer: one kernel whose threads gather 16-byte K chunks
 *     through the strides straight into shared memory; no workspace.
 * gemm_tn_strided picks repack for problems of at least 2^24 multiply-adds
 * and falls back to the copy producer when the pool cannot serve the
 * workspace; gemm_tn_strided_ex can force either (gemm_tn_options.path =
 * GEMM_TN_PATH_STRIDED_REPACK / _COPY; timeout_ns also applies).
 * Errors: GEMM_TN_ERR_INVALID_ARG for negative sizes or strides, NULL with a
 * nonzero extent, a C/D view in which two coordinates share an element, or
 * C/D overlapping A or B; GEMM_TN_ERR_ALIGNMENT for a pointer that is not
 * 2-byte aligned; GEMM_TN_ERR_NO_MEMORY when the repack route is forced and
 * the pool cannot serve it.  M == 0, N == 0 or K == 0 enqueue nothing.
 */
GEMM_TN_API int gemm_tn_strided(int64_t M, int64_t N, int64_t K,
                                const void* A, int64_t sAm, int64_t sAk,
                                const void* B, int64_t sBn, int64_t sBk,
                                void* CD, int64_t sCm, int64_t sCn,
                                int accum_dtype, void* stream);

/* gemm_tn_strided with explicit controls (opts may be NULL); only `path`
 * (0, GEMM_TN_PATH_STRIDED_COPY or GEMM_TN_PATH_STRIDED_REPACK) and
 * `timeout_ns` are read. */
GEMM_TN_API int gemm_tn_strided_ex(int64_t M, int64_t N, int64_t K,
                                   const void* A, int64_t sAm, int64_t sAk,
                                   const void* B, int64_t sBn, int64_t sBk,
                                   void* CD, int64_t sCm, int64_t sCn,
                                   int accum_dtype, void* stream,
                                   const gemm_tn_options* opts);

/*
 * D = alpha * A.B^T + beta * C with A, B, C and D in HOST memory: the
 * operands, layouts, accumulation modes and rounding are those of
 * gemm_tn_scaled (A, B, C and D views as in gemm_tn; D may be C itself with
 * ldD == ldC, but no other overlap of C and D is accepted), and the results
 * are bit-identical to gemm_tn_scaled on device copies of the same arrays.
 *
 * The call copies B to the device, then A, C and D in panels of rows of M
 * (gemm_tn_options.host_panel_rows), and overlaps the transfers with the
 * work: panel i's GEMM runs on `stream` as soon as its A and C rows have
 * arrived, while the next panels' rows are copied in on one of the
 * library's copy streams and the finished panels' D rows are copied out on
 * another.  Host-to-device and device-to-host copies share the host link, so
 * a call of this kind is bound by its copies: per call about
 * (bytes of A, B and C) / (host-to-device rate) plus the last panel's GEMM
 * and copy-out.
 *
 * Ordering and ownership: the work is ordered after everything enqueued on
 * `stream` before the call, and everything enqueued on `stream` after the
 * call is ordered after all of it (the copy streams are joined back).  The
 * call returns once the work is enqueued: A, B and C must not be written,
 * and D not read, until `stream` has passed the call
 * (cudaStreamSynchronize).  The host arrays should be page-locked
 * (cudaHostAlloc / cudaHostRegister): copies from pageable memory are
 * staged by the driver and do not overlap.  The device copies live in a
 * workspace of N x K for B plus three panels of A (panel rows x K) and of
 * C/D (panel rows x N).  The library keeps two such workspaces per device
 * for this entry point, used by alternate calls, each reused once the call
 * before last is done with it, grown (with a host wait for the calls still
 * using them) when a call needs more than any earlier one, and kept until
 * the process exits; under stream capture the workspace is taken from the
 * library's pool in `stream`'s order instead (a graph memory node).
 * Concurrent calls from several host threads are serialised while they
 * enqueue (the copy streams are the library's, one pair per device).
 *
 * With gemm_tn_options.host_inputs_ready the copies in are ordered only
 * after the copies in of earlier gemm_tn_host calls on the device (see the
 * option), so that a stream of independent calls keeps the host link busy
 * across call boundaries.
 *
 * Only host_panel_rows, host_inputs_ready, sync_check and the large-path controls of
 * gemm_tn_options (path, tile_kernel, tile_n, split_k, stream_k, k_stage,
 * timeout_ns) are read; they apply to every panel's GEMM.
 * Errors: GEMM_TN_ERR_INVALID_ARG for negative or too large sizes, an ld
 * smaller than its row, NULL with a nonzero extent, or C and D overlapping
 * other than exactly; GEMM_TN_ERR_NO_MEMORY when the pool cannot serve the
 * workspace (nothing enqueued); GEMM_TN_ERR_CUDA when a copy or launch
 * fails.  M == 0 or N == 0 enqueues nothing.
 */
GEMM_TN_API int gemm_tn_host(int64_t M, int64_t N, int64_t K, float alpha,
                             const void* A, int64_t ldA, int a_major,
                             const void* B, int64_t ldB, int b_major,
                             float beta, const void* C, int64_t ldC,
                             void* D, int64_t ldD, int accum_dtype, void* stream,
                             const gemm_tn_options* opts);

/* Synchronise `stream`, then read and clear the device error word that a
 * kernel sets when one of its bounded waits expires.  Returns GEMM_TN_OK,
 * GEMM_TN_ERR_DEVICE_TIMEOUT (and, if detail != NULL, the raw word: bits
 * 16-23 the role that gave up -- 1 producer, 2 MMA issuer, 3 epilogue -- and
 * bits 0-15 the pipeline stage), or GEMM_TN_ERR_CUDA. */
GEMM_TN_API int gemm_tn_check_device_error(void* stream, uint32_t* detail);

/* Phase trace of the last launch made with gemm_tn_options.trace on the
 * current device: GEMM_TN_TRACE_SLOTS 64-bit words per CTA, for the first
 * GEMM_TN_TRACE_CTAS CTAs of the grid (blockIdx.x order):
 *   0 kernel entry            1 after the wait for the previous kernel
 *   2 first stage complete    3 last accumulator committed (MMA issuer)
 *   4 first accumulator ready 5 last output chunk issued (first epilogue warp)
 *   6 that warp's stores done 7 exit (before tensor memory is freed)
 *   8 SM id                   9 work units (tiles or segments) of the CTA
 *  10 SM cycle counter at entry  11 SM cycle counter at exit
 * Times are the GPU's global nanosecond timer; 0 marks a point the CTA did
 * not pass (or a kernel that does not stamp it: the skinny kernel stores
 * partial sums, so its slot 6 stays 0).  Synchronises `stream`, then copies
 * max_ctas records (at most GEMM_TN_TRACE_CTAS) to `out` (host memory of
 * max_ctas * GEMM_TN_TRACE_SLOTS words) and sets *recorded (if non-NULL) to
 * the number of CTAs with an entry stamp.  Returns GEMM_TN_OK,
 * GEMM_TN_ERR_INVALID_ARG (out NULL, max_ctas < 0) or GEMM_TN_ERR_CUDA. */
#define GEMM_TN_TRACE_SLOTS 12
#define GEMM_TN_TRACE_CTAS 512
GEMM_TN_API int gemm_tn_trace_read(void* stream, uint64_t* out, int max_ctas, int* recorded);

/* Which path gemm_tn would take for these sizes and majors (gemm_tn_path). */
GEMM_TN_API int gemm_tn_plan_path(int64_t M, int64_t N, int64_t K, int a_major,
                                  int b_major);

/* Number of kernel launches the last successful gemm_tn, gemm_tn_ex,
 * gemm_tn_scaled, gemm_tn_batched[_ex] or gemm_tn_strided[_ex] call on this
 * host thread enqueued (0 for the no-op cases). */
GEMM_TN_API int gemm_tn_last_launch_count(void);

/* Names of the kernels the last successful call of any entry point above or
 * gemm_tn_skinny_noalloc on this host thread enqueued, '+'-separated
 * ("" after a no-op call).  Static storage; never NULL. */
GEMM_TN_API const char* gemm_tn_last_kernels(void);

/* Static, NUL-terminated name of a gemm_tn_status value. */
GEMM_TN_API const char* gemm_tn_status_string(int status);

/* Size of the fixed scratch array behind gemm_tn_skinny_noalloc: 16 MiB,
 * held in device memory on every GPU that loads this library, until the
 * process exits. */
#define GEMM_TN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * The skinny path (M <= 64, K-major A and B, GEMM_TN_ACC_F32) without any
 * device allocation.  The source pages have no counterpart of this entry
 * point; it exists for callers that cannot let a library allocate device
 * memory behind their back:
 *   - latency-sensitive loops, where cudaMalloc/cudaFree can synchronise the
 *     device and stall every stream;
 *   - processes whose framework allocator has already reserved nearly all
 *     device memory, where a library's own cudaMalloc can fail at an
 *     unpredictable moment;
 *   - programs that must fix their device-memory footprint up front.
 * gemm_tn's skinny path takes its split-K partial sums' workspace from the
 * library's memory pool on every call.  This entry point computes the same
 * thing with the same kernels, but keeps the partial sums in one fixed
 * array of GEMM_TN_NOALLOC_SCRATCH_BYTES compiled into the library, so no
 * call ever allocates or frees device memory.
 *
 * Arguments, views and results are those of gemm_tn, restricted to
 * M <= 64, a_major == b_major == GEMM_TN_MAJOR_K and
 * accum_dtype == GEMM_TN_ACC_F32.  The caller still owns and passes A, B and
 * CD.
 *
 * Limits and behaviour:
 *   - returns GEMM_TN_ERR_INVALID_ARG, before enqueuing anything, when the
 *     arguments are outside that restriction or when the problem needs more
 *     partial-sum scratch than GEMM_TN_NOALLOC_SCRATCH_BYTES (the need is
 *     (SMs) x (tiles one CTA touches) x 128 x round_up(M,16) x 4 bytes; the
 *     M=16, N=K=16384 problem needs about 2.5 MiB);
 *   - the first call on each device sets the library up there (reads the
 *     device's attributes, raises the kernels' shared-memory limits, looks
 *     up the driver's tensor-map encoder) and looks up the array's device
 *     address (cudaGetSymbolAddress, with that device current); none of
 *     this allocates device memory, and unlike the other entry points this
 *     one never creates the library's workspace pool.  Make that first call
 *     before any stream capture on that device;
 *   - every call on a device shares the one array, and the array keeps
 *     whatever the last call left in it.  Nothing in it needs to start at
 *     zero (each partial sum is written before it is read within a call),
 *     but calls that can overlap on the GPU -- for example on two streams
 *     without ordering between them -- race on the array and produce wrong
 *     results.  Order such calls on one stream or with events.
 */
GEMM_TN_API int gemm_tn_skinny_noalloc(int64_t M, int64_t N, int64_t K,
                                       const void* A, int64_t ldA, int a_major,
                                       const void* B, int64_t ldB, int b_major,
                                       void* CD, int64_t ldC,
                                       int accum_dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_TN_H_ */
