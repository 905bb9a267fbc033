/*
 * sgemm_gb300.h - C ABI of the GB300 (sm_103a) single-precision GEMM library.
 *
 * The operation is the problem statement mysgemm(M, N, K, alpha, A, B, beta,
 * C) of "NVIDIA_SGEMM_PRACTICE" (section "kernel 1", and the launch comment
 * of section "kernel 2"):
 *
 *     C[m][n] = alpha * sum_{k<K} A[m][k] * B[k][n] + beta * C[m][n]
 *
 * on row-major float32 matrices: A is M x K, B is K x N, C is M x N.  The
 * pages use packed matrices; here each matrix has a leading dimension (the
 * distance in elements between consecutive rows), so the pages' case is
 * lda = K, ldb = N, ldc = N.
 *
 * Conventions shared by every entry point below:
 *   - A, B, C are device pointers owned by the caller (except sgemm_host).
 *     The library never frees or retains them beyond the call.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *     unless stated otherwise.
 *   - Return value: 0 on success; -i when the i-th argument (1-based) is
 *     invalid; a positive cudaError_t value when a CUDA call fails; or one of
 *     the SGEMM_ERR_* codes (all > 10000).
 *   - Argument rules: M, N, K >= 0; lda >= max(1, K); ldb >= max(1, N);
 *     ldc >= max(1, N); A and B must be non-NULL when alpha != 0 and K > 0;
 *     C must be non-NULL when M > 0 and N > 0; C must not overlap A or B.
 *   - Quick returns: M == 0 or N == 0 does nothing.  alpha == 0 or K == 0
 *     computes C = beta * C without reading A or B.  beta == 0 makes C
 *     write-only: its old contents (NaN included) never reach the result.
 *   - Results are deterministic: the same call on the same device gives the
 *     same bits every time (no floating-point atomics).
 *   - Accuracy: every element lies within
 *     1e-4 * (|alpha| * sum_k |A[m][k] * B[k][n]| + |beta * C[m][n]|)
 *     of the exact result, on every path.
 *   - Calls from several host threads on different streams are safe.
 *   - The tensor-core kernels are launched with programmatic stream
 *     serialization: one may begin its on-chip set-up while the kernel ahead
 *     of it on the stream finishes, but it reads and writes no global memory
 *     before that kernel has completed, so stream order is unchanged.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that this header does not
 * need the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *sgemm_stream_t;

/* Status codes beyond 0 / -i / cudaError_t. */
#define SGEMM_ERR_DEVICE_TIMEOUT     10001 /* a bounded on-device wait gave up */
#define SGEMM_ERR_NO_DEVICE          10002 /* no CUDA device is usable        */
#define SGEMM_ERR_UNSUPPORTED_DEVICE 10003 /* device is not compute 10.3     */
#define SGEMM_ERR_WORKSPACE          10004 /* split-K workspace unavailable   */
#define SGEMM_ERR_INTERNAL           10005 /* planner found no kernel         */
#define SGEMM_ERR_SCRATCH_LIMIT      10006 /* sgemm_noalloc: problem needs more
                                              split-K scratch than its fixed
                                              array holds                      */
#define SGEMM_ERR_OUT_OF_BOUNDS      10007 /* a library built with SGEMM_DEBUG
                                              found a kernel address outside
                                              its matrix (the access was
                                              skipped; C is unspecified)      */

/* Algorithm selector for sgemm_ex / sgemm_host. */
#define SGEMM_ALGO_AUTO   0 /* planner picks the faster path                  */
#define SGEMM_ALGO_FFMA   1 /* register-blocked fp32 FMA on the CUDA cores    */
#define SGEMM_ALGO_TF32X3 2 /* tcgen05 tensor cores, fp32 split into hi + lo
                               tf32 parts, hi*hi + hi*lo + lo*hi accumulated
                               in fp32 in tensor memory                        */

/* Flags for sgemm_ex. */
/* SGEMM_FLAG_TILE_ROWS(r): 3xTF32 path only, force r C rows per tile
 * (r in 16, 32, 64, 128, 192, 256); 0 lets the planner choose. */
#define SGEMM_FLAG_TILE_ROWS(r) ((((r) / 16) & 0xFF) << 8)
/* SGEMM_FLAG_WHOLE_TILES: 3xTF32 path only, keep whole tiles in the last
 * wave instead of splitting the leftover tiles along K over idle SMs. */
#define SGEMM_FLAG_WHOLE_TILES 2
/* SGEMM_FLAG_SPLIT_TAIL: 3xTF32 path only, split the leftover tiles of a
 * partly empty last wave along K whenever there are any, even where the
 * planner's run-time estimate prefers whole tiles (for tuning and tests).
 * Ignored with an explicit split count; WHOLE_TILES wins over it. */
#define SGEMM_FLAG_SPLIT_TAIL 4
/* SGEMM_FLAG_NO_A_COPY: 3xTF32 path only.  An A whose rows are not 16-byte
 * aligned (lda % 4 != 0 or a misaligned pointer) and that is far smaller
 * than B (M * 32 <= N, the im2col shapes) is otherwise copied first,
 * on the call's stream, into a library buffer with rows padded to 4 floats
 * (2 * M * K * 4 bytes of traffic), so that its tiles come by TMA.  With the
 * flag the kernel loads such an A itself.  Both give the same bits. */
#define SGEMM_FLAG_NO_A_COPY (1 << 16)
/* SGEMM_FLAG_B_ROWS_LOADED: 3xTF32 path only.  A B whose rows are not
 * 16-byte aligned (ldb % 4 != 0) but whose start is, with K >= 4, is
 * otherwise copied by TMA as four tensors, one per residue class of rows
 * k % 4 (the rows of a class lie 4 * ldb floats apart, a multiple of 16
 * bytes).  With the flag the kernel loads such a B itself.  Both give the
 * same bits. */
#define SGEMM_FLAG_B_ROWS_LOADED (1 << 17)
/* CTA pairs (3xTF32 path): clusters of two CTAs on neighbouring SMs share
 * one tensor-core MMA (tcgen05 cta_group::2) over a tile of 256 columns,
 * each CTA holding half of the tile's A rows (half the shared-memory traffic
 * and producer work per MMA, deeper pipelines).  They need A's rows 16-byte
 * aligned and B copied by TMA (its rows aligned, or as residue classes).
 * The planner runs tiles of 256 rows on pairs; tiles of 192 rows only with
 * SGEMM_FLAG_PAIRS.  Whole tiles give the same bits either way; tiles split
 * along K may differ in rounding (their K slices can differ).
 * SGEMM_FLAG_PAIRS: pairs for tiles of 192 or 256 rows whenever possible.
 * SGEMM_FLAG_NO_PAIRS: never pairs (wins over SGEMM_FLAG_PAIRS). */
#define SGEMM_FLAG_PAIRS (1 << 18)
#define SGEMM_FLAG_NO_PAIRS (1 << 19)
#define SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE 1 /* test only: one pipeline arrive
                                              is withheld and the on-device
                                              wait budget is cut to ~1 ms, so
                                              the bounded wait runs out; the
                                              call then reports
                                              SGEMM_ERR_DEVICE_TIMEOUT through
                                              sgemm_check_status and C is
                                              unspecified                      */

/*
 * sgemm - C = alpha * A * B + beta * C, planner-chosen path.
 *
 * Arguments 1-12 in the order of the problem statement, with leading
 * dimensions after each matrix and the stream last.  Same as
 * sgemm_ex(..., SGEMM_ALGO_AUTO, 0, 0).
 */
int sgemm(int M, int N, int K, float alpha,
          const float *A, int lda,
          const float *B, int ldb,
          float beta, float *C, int ldc,
          sgemm_stream_t stream);

/*
 * sgemm_ex - as sgemm, with explicit choices.
 *
 *   algo   (13): SGEMM_ALGO_AUTO / _FFMA / _TF32X3.
 *   splits (14): 0 = planner's choice; s >= 1 forces s slices of K (clamped
 *                to the number of K tiles).  With s > 1 each slice writes a
 *                partial tile to a library-owned workspace and the last slice
 *                to finish adds the partials in slice order, so the result
 *                does not depend on timing.
 *   flags  (15): 0, or any of SGEMM_FLAG_TILE_ROWS(r),
 *                SGEMM_FLAG_WHOLE_TILES, SGEMM_FLAG_SPLIT_TAIL and
 *                SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE (tests only).  Any other bit, or a tile height that is not
 *                supported, is rejected.
 *
 * AUTO takes the 3xTF32 path, except for short, shallow A (M <= 32,
 * K <= 48, no forced split count).  That goes to the FFMA path's wide-N
 * kernel, which streams B and C at HBM speed in exact fp32.  An explicit
 * SGEMM_ALGO_FFMA uses that kernel up to K = 64.
 *
 * Scheduling (3xTF32 path): persistent CTAs, one per SM.  The planner
 * estimates the run time of each tile height, split count and last-wave
 * treatment from measured per-tile costs and takes the fastest.  With few
 * output tiles K is split (splits).  With a partly empty last wave, whole
 * waves keep whole tiles and the leftover tiles may be cut into K slices,
 * one per otherwise idle SM (split tail).  Tiles shared by several units are
 * finished by the last unit to arrive, which adds the partial tiles in a
 * fixed order, so the result does not depend on timing.
 *
 * The split-K workspace is owned by the library, kept per device and stream,
 * grown on demand (a synchronous cudaMalloc, so make the first call of a
 * given size outside stream capture) and released by sgemm_release().  After
 * such a first call on a stream, calls on it can be captured into a CUDA
 * graph: a call then only encodes tensor maps on the host and launches.
 */
int sgemm_ex(int M, int N, int K, float alpha,
             const float *A, int lda,
             const float *B, int ldb,
             float beta, float *C, int ldc,
             sgemm_stream_t stream, int algo, int splits, int flags);

/*
 * sgemm_host - C = alpha * A * B + beta * C on HOST buffers, synchronous.
 *
 * A, B, C are host pointers (pinned memory gives full copy bandwidth and
 * lets the copies overlap the GEMMs).  The call copies A, B (and C when
 * beta != 0) to library-owned device buffers on the current device, runs
 * the GEMM, copies C back and waits for completion.  From 64 MB of traffic
 * and 512 rows up it runs as up to 12 row blocks of C (128-row multiples,
 * the last one taking any remainder): B goes up first, each block's rows of
 * A (and C) follow on an upload stream, a block's GEMM starts once its rows
 * have landed, and its rows of C return on a download stream while later
 * blocks compute.  On the 3xTF32 path the block sizes come from simulating
 * that timeline with the planner's run-time model of each block's GEMM (a
 * small first block so the GEMMs start early, a small last one, equal
 * blocks between); sgemm_host_blocks reports them.  A call with fewer rows
 * and at least 8192 columns runs as up to 12 column blocks (1024-column
 * multiples) the same way, with A first and pitched copies of the blocks'
 * columns of B and C.  Each block is a planned
 * GEMM of its own, so the schedule, and with it the rounding of each
 * element's sum, may differ from one sgemm_ex call over the whole matrix
 * (the accuracy bound is the same).
 * Same argument rules and return codes as sgemm_ex; algo as in sgemm_ex.
 * The device buffers are kept for reuse and freed by sgemm_release().
 * Calls from several host threads at once race on those buffers.
 */
int sgemm_host(int M, int N, int K, float alpha,
               const float *A, int lda,
               const float *B, int ldb,
               float beta, float *C, int ldc, int algo);

/*
 * sgemm_host_blocks - how sgemm_host would cut a call into blocks, without
 * running it.
 *
 * Host-only: makes no CUDA call when num_sms > 0 (num_sms = 0 queries the
 * current device; the pair form is then sized for num_sms / 2 CTA pairs).
 * M, N, K, lda, ldb, ldc, alpha, beta, algo as in sgemm_host (no buffers).
 * Sets *axis to 0 for row blocks of C or 1 for column blocks, writes up to
 * max_sizes block sizes (rows, or columns) in call order to sizes, and
 * returns the block count: 1 when the call runs as one GEMM (sizes[0] is
 * then M).  Returns -i for an invalid argument (the i-th argument of this
 * function, 1-based), or a negative sgemm error code from the device query.
 */
int sgemm_host_blocks(int M, int N, int K, int lda, int ldb, int ldc, float alpha, float beta, int algo,
                      int num_sms, int *axis, int *sizes, int max_sizes);

/*
 * sgemm_plan_info - what the planner would launch, without launching.
 *
 * Host-only: makes no CUDA call when num_sms > 0 (num_sms = 0 queries the
 * current device).  Arguments as in sgemm_ex; the pointers are only used for
 * alignment and may be any values.  Writes up to `ninfo` ints to `info`:
 *   [0] path (SGEMM_ALGO_FFMA or SGEMM_ALGO_TF32X3)
 *   [1] tile rows of C      [2] tile columns of C
 *   [3] K splits            [4] work units (tiles * splits)
 *   [5] grid size (CTAs)    [6] pipeline stages
 *   [7] 1 if A is read with 16-byte vector loads
 *   [8] 1 if B is read with 16-byte vector loads
 *   [9] workspace bytes needed
 *   [10] leftover tiles split along K after the whole waves (0 = none)
 *   [11] 1 for the FFMA path's wide-N kernel (M <= 32, K <= 64: A resident
 *        in shared memory, B streamed, persistent CTAs), else 0
 *   [12] 1 when the tiles run on CTA pairs (SGEMM_FLAG_PAIRS; tile columns
 *        then 256, grid = 2 x pairs), else 0
 * Returns 0, or -i for an invalid argument (the i-th argument of this
 * function, 1-based).
 */
int sgemm_plan_info(int M, int N, int K, const void *A, int lda,
                    const void *B, int ldb, const void *C, int ldc,
                    int algo, int splits, int flags, float alpha, float beta,
                    int num_sms, int *info, int ninfo);

/*
 * sgemm_check_status - wait for `stream`, then read and clear the device
 * status words of the current device: the one of every allocating entry
 * point and the one of sgemm_noalloc.  Returns 0, SGEMM_ERR_DEVICE_TIMEOUT
 * if a kernel launched since the last check gave up a bounded wait (or met
 * a work split it cannot finish, which the planner never produces),
 * SGEMM_ERR_OUT_OF_BOUNDS (SGEMM_DEBUG builds only) if a kernel computed an
 * address outside its matrix, or a positive cudaError_t.  When a word was set, it also waits for the whole
 * device and clears the split-K arrival counters that word's kernels use.
 * Allocates no device memory.
 */
int sgemm_check_status(sgemm_stream_t stream);

/* sgemm_status_string - static, human-readable text for any return code. */
const char *sgemm_status_string(int status);

/*
 * sgemm_release - free every library-owned device buffer (workspaces, host
 * call staging buffers) on all devices.  Waits for the device first.  Not
 * safe while another thread is inside a call of this library.
 */
int sgemm_release(void);

/*
 * sgemm_noalloc - C = alpha * A * B + beta * C on the 3xTF32 path without
 * allocating any device memory.  (The pages have no counterpart: this entry
 * point exists for callers of this library.)
 *
 * Who needs it: callers that cannot let a library allocate device memory
 * behind their back - programs that reserve the whole GPU for their own
 * memory pool up front, where a hidden cudaMalloc fails or breaks their
 * accounting, and latency-sensitive loops in which cudaMalloc/cudaFree's
 * implicit device-wide synchronisation would stall other streams.
 *
 * Same arguments, rules and results as
 * sgemm_ex(..., stream, SGEMM_ALGO_TF32X3, splits, 0); the caller still
 * passes A, B and C.  The split-K partial tiles and arrival counters live in
 * fixed arrays compiled into the library: 16 MiB of partials (units x 128 x
 * tile rows floats) and 4096 counters (one per output tile), held on every
 * GPU that loads the library until the process exits.  A plan that needs
 * more returns SGEMM_ERR_SCRATCH_LIMIT before anything runs.  The call never
 * calls cudaMalloc, cudaFree or any allocating routine.
 *
 * Set-up: the first call on a device with M > 0 and N > 0 (with that device
 * current) resolves the arrays' device addresses with cudaGetSymbolAddress.
 * Under CUDA's lazy module loading (the default) that is also when the
 * arrays and the device code of every kernel this entry point can launch
 * are loaded onto the device, which takes device memory (16 MiB for the
 * arrays, plus the code): make that first call before reserving the
 * device's memory for a pool, and before any stream capture.  A call with
 * alpha == 0 and beta == 1 does the set-up and nothing else (C, which must
 * be a non-NULL device pointer, is neither read nor written); after it,
 * later calls leave the device's free memory unchanged.
 * Sharing: every call uses the same arrays, which keep the previous call's
 * contents.  The arrival counters start at zero and each call leaves them
 * at zero.  Calls whose work overlaps on the GPU - on different streams, or
 * from several host threads at once - race on the arrays and give wrong
 * results: serialise them.
 * Status: a bounded on-device wait that gives up (only a broken GPU does,
 * or the test hook below) leaves C unspecified and sets this entry point's
 * device status word.  sgemm_check_status reads and clears it, and then
 * clears the arrival counters; until that check, later split-K calls of
 * this entry point may give wrong results.
 */
int sgemm_noalloc(int M, int N, int K, float alpha,
                  const float *A, int lda,
                  const float *B, int ldb,
                  float beta, float *C, int ldc,
                  sgemm_stream_t stream, int splits);

/*
 * sgemm_noalloc_debug_flags - test hook: debug flags for the next
 * sgemm_noalloc call that launches a GEMM (it consumes them; later calls run
 * normally).  flags (1): 0 or SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE, which makes
 * that call's bounded wait run out after about 1 ms, so that its failure is
 * reported by sgemm_check_status.  Returns 0, or -1 for other bits.
 */
int sgemm_noalloc_debug_flags(int flags);

/*
 * sgemm_t - C = alpha * op(A) * op(B) + beta * C, with op(X) = X or X^T
 * (BLAS transa / transb in row-major storage).  The pages fix both operands
 * row-major ("NVIDIA_SGEMM_PRACTICE", section "kernel 1"); this is the
 * transposed-operand extension a BLAS caller expects.
 *
 *   transa (1): 0: A is M x K, lda >= K.  1: A is stored K x M (op(A) = A^T),
 *               lda >= M.
 *   transb (2): 0: B is K x N, ldb >= N.  1: B is stored N x K, ldb >= K.
 *   M, N, K, alpha, A, lda, B, ldb, beta, C, ldc (3-13): as in sgemm, with
 *               the storage above.  C is M x N row-major, ldc >= N.
 *   stream (14), algo (15): as in sgemm_ex.
 *
 * A transposed operand is first copied, transposed, into a library-owned
 * buffer of this stream (grown on demand like the split-K workspace,
 * released by sgemm_release).  The planned GEMM then runs on the copy, so a
 * transposed operand costs one extra read and write of it.  Calls on the
 * same stream from several threads race on that buffer.  Returns 0, -i for
 * the i-th argument, a positive cudaError_t, or SGEMM_ERR_WORKSPACE.
 */
int sgemm_t(int transa, int transb, int M, int N, int K, float alpha,
            const float *A, int lda,
            const float *B, int ldb,
            float beta, float *C, int ldc,
            sgemm_stream_t stream, int algo);

/*
 * sgemm_strided_batched - for b in [0, batch):
 *   C_b = alpha * op(A_b) * op(B_b) + beta * C_b,
 * where X_b = X + b * strideX elements (X in A, B, C), op as in sgemm_t.
 * The pages' per-image im2col GEMMs are such a batch.
 *
 *   strideA (9), strideB (12): >= 0; 0 shares one matrix across the batch.
 *   strideC (16): the C matrices must not overlap, so for batch > 1 at least
 *                 (M - 1) * ldc + N.
 *   batch (17): >= 0.
 *   The other arguments are as in sgemm_t, renumbered.
 *
 * On the 3xTF32 path (AUTO, except the wide-N FFMA shapes) the whole batch
 * is one launch: the schedule's tiles run over every matrix, so a batch of
 * small GEMMs fills the GPU.  Transposed operands are first copied,
 * transposed, into this stream's buffer (as in sgemm_t), all matrices at
 * once.  The batch runs instead as one planned GEMM per matrix, in order on
 * `stream`, on the FFMA path, when alpha = 0 or K = 0, when the tile count
 * exceeds 2^31 / 16, or when the C matrices overlap A's or B's memory.
 * 16-byte strides (multiples of 4 elements) keep the tensor-map copies;
 * other strides use element loads.
 * Returns 0, -i for the i-th argument, or the first failing call's status.
 */
int sgemm_strided_batched(int transa, int transb, int M, int N, int K, float alpha,
                          const float *A, int lda, long long strideA,
                          const float *B, int ldb, long long strideB,
                          float beta, float *C, int ldc, long long strideC,
                          int batch, sgemm_stream_t stream, int algo);

/*
 * sgemm_conv2d - Y = alpha * conv2d(X, Wt) + beta * Y in fp32, as an
 * implicit GEMM: the im2col lowering that gives the skinny GEMM shapes of
 * "UNIVERSAL_SGEMM_CUDA" (its shape list: filters x (channels * KH * KW)
 * times (channels * KH * KW) x output pixels) is never stored; the kernel's
 * producers read each B element straight from the input image.  The pages
 * give only the lowered shapes; the layer is the usual one: a
 * cross-correlation (the filter is not flipped) with zero padding,
 *   Y[b][f][oh][ow] = alpha * sum_{c,kh,kw} Wt[f][c][kh][kw] *
 *                     X[b][c][oh*stride_h + kh*dil_h - pad_h][ow*stride_w + kw*dil_w - pad_w]
 *                     + beta * Y[b][f][oh][ow],
 * input positions outside the image reading as 0.
 *
 *   nb (1), C (2), H (3), W (4): X is nb x C x H x W, packed NCHW; nb, C >= 0,
 *                 H, W >= 1.
 *   F (5), KH (6), KW (7): Wt is F x C x KH x KW, packed OIHW; F >= 0,
 *                 KH, KW >= 1, and the dilated filter fits in the padded
 *                 image (else -6 / -7).
 *   stride_h, stride_w (8, 9) >= 1; pad_h, pad_w (10, 11) >= 0;
 *   dil_h, dil_w (12, 13) >= 1.
 *   alpha (14), X (15), Wt (16), beta (17): device pointers for X and Wt,
 *                 read only; not read when alpha == 0 or C == 0.
 *   Y (18):       device pointer, nb x F x OH x OW packed NCHW with
 *                 OH = (H + 2 pad_h - dil_h (KH - 1) - 1) / stride_h + 1 and
 *                 OW likewise; must not overlap X or Wt.  beta == 0: Y is
 *                 not read.
 *   stream (19):  as in sgemm.
 *   algo (20):    SGEMM_ALGO_TF32X3: the 3xTF32 tensor kernel, producers
 *                 gathering B.  SGEMM_ALGO_FFMA: the wide-N FFMA kernel's
 *                 convolution form (resident filter, slabs of the im2col
 *                 matrix gathered by cp.async), only for F <= 32 and
 *                 C * KH * KW <= 64 (else -20).  SGEMM_ALGO_AUTO: FFMA for
 *                 F <= 32 and C * KH * KW <= 48, else TF32X3.
 * Limits: a padded image with its filter reach, times C + 1, below 2^31
 * elements (32-bit offsets in the gather; else -2), OH * OW < 2^31 (else -3).
 * The tensor path reads the filter through a tensor map: its rows (C * KH *
 * KW floats) are first copied to 16-byte aligned rows in a library buffer of
 * this stream (as in sgemm_t) when they are not aligned, and reordered to
 * OHWI (k over the channels at each tap) when C is a multiple of 16.  Layers
 * with padding may also get a zero-bordered copy of the input there (see
 * sgemm_conv2d_ex).  Accuracy and status reporting are those of sgemm_ex with the
 * TF32X3 path: the same bound per output element, with the sum over the
 * filter taps that fall inside the image.  Returns 0, -i for the i-th
 * argument, a positive cudaError_t, or SGEMM_ERR_WORKSPACE.
 */
int sgemm_conv2d(int nb, int C, int H, int W, int F, int KH, int KW,
                 int stride_h, int stride_w, int pad_h, int pad_w, int dil_h, int dil_w,
                 float alpha, const float *X, const float *Wt, float beta, float *Y,
                 sgemm_stream_t stream, int algo);

/*
 * sgemm_conv2d_ex - sgemm_conv2d with flags (21):
 *   SGEMM_CONV_NO_PAD_COPY: never make the zero-bordered copy of the input.
 *     For a layer with padding, fewer than 16-multiple channels and at most
 *     kConvTabMax (2048) taps, the library otherwise copies the input once
 *     into this stream's transpose buffer, at most 1 GiB, with zero borders,
 *     so that the gather needs no bounds checks.  With the flag, or above that
 *     size, the gather checks every tap against the image instead (slower,
 *     no extra memory).
 *   Other bits: -21.  Everything else as sgemm_conv2d.
 */
#define SGEMM_CONV_NO_PAD_COPY 1
int sgemm_conv2d_ex(int nb, int C, int H, int W, int F, int KH, int KW,
                    int stride_h, int stride_w, int pad_h, int pad_w, int dil_h, int dil_w,
                    float alpha, const float *X, const float *Wt, float beta, float *Y,
                    sgemm_stream_t stream, int algo, int flags);

/* sgemm_version - library version as 10000*major + 100*minor + patch. */
int sgemm_version(void);

/*
 * sgemm_tf32_mma_rate - measure the tensor cores' rate on the MMA form the
 * 3xTF32 path issues (tcgen05.mma kind::tf32, M = 128, N = n, K = 8, A from
 * tensor memory, B from shared memory, fp32 accumulator), on the current
 * device.  This is measurement, not GEMM: the pages time their kernels
 * against a device peak ("NVIDIA_SGEMM_PRACTICE", overview table), and this
 * call supplies the tf32 peak the way the kernel uses the tensor cores.
 *
 *   n      (1): MMA N, a multiple of 16 in [16, 256].
 *   iters  (2): MMAs per SM, >= 1 (about 150 cycles each at n = 256).
 *   stream (3): stream the two launches (warm-up, timed) are ordered on;
 *               the call waits for them.
 *   tflops (4): out, raw tf32 TFLOP/s = SMs x iters x 2 x 128 x n x 8 / time.
 *
 * Returns 0, -i for a bad argument, a positive cudaError_t,
 * SGEMM_ERR_UNSUPPORTED_DEVICE, or SGEMM_ERR_DEVICE_TIMEOUT if the bounded
 * wait for the MMAs gave up.  Allocates nothing on the device.
 */
int sgemm_tf32_mma_rate(int n, int iters, sgemm_stream_t stream, double *tflops);

/*
 * sgemm_ffma_rate - measure the CUDA cores' fp32 FMA rate on the current
 * device: the peak of the FFMA path (the pages estimate theirs from core
 * counts and clocks, "matmul_opt.cu", its theoretical-peak paragraph; this
 * call measures it).  Every SM runs 2048 threads, each with 16 independent
 * FMA chains.  Measurement, not GEMM.
 *
 *   packed (1): 0 = scalar fma.rn.f32; 1 = packed fma.rn.f32x2 (two FMAs per
 *               instruction, the form the FFMA kernels issue).
 *   iters  (2): steps per thread, >= 1 (16 FMAs each).
 *   stream (3): stream the two launches (warm-up, timed) are ordered on;
 *               the call waits for them.
 *   tflops (4): out, fp32 TFLOP/s = 2 x FMAs / time.
 *
 * Returns 0, -i for a bad argument, a positive cudaError_t or
 * SGEMM_ERR_UNSUPPORTED_DEVICE.  Allocates nothing on the device.
 */
int sgemm_ffma_rate(int packed, int iters, sgemm_stream_t stream, double *tflops);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
