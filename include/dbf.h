/*
 * dbf.h - C ABI of the packed double-binary matmul library (libdbf.so).
 *
 * The operation (LoRDBA - "Adaptación Binaria Doble de Bajo Rango", section 2,
 * Metodología / Arquitectura Central; and "Addition is almost all you need:
 * Compressing large language models with double binary factorization",
 * section 2, Formulación Matemática / Cálculo en la inferencia):
 *
 *     y = sum_{i=1..ell} alpha_i . B1 (beta_i . (B2 (gamma_i . x)))
 *
 * for every token row x of a batch, i.e. y = x dW^T with
 * dW = sum_i diag(alpha_i) B1 diag(beta_i) B2 diag(gamma_i).
 * B1 in {+1,-1}^{N x R} and B2 in {+1,-1}^{R x M} are stored at one bit per
 * entry; alpha_i, beta_i, gamma_i are fp16 per-channel scales.  The two sign
 * contractions replace multiplications by additions and subtractions (same
 * sections: "Núcleo de Inferencia" on the LoRDBA page, the evaluation order
 * on the DBF page).
 *
 * Conventions for every call:
 *   - Pointers named d_* or documented as "device" are CUDA device memory
 *     owned by the caller; the library keeps no pointer after a call returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream.
 *   - The library never allocates device memory.  Scratch space is passed in
 *     as `workspace` (device, 256-byte aligned, at least the size the
 *     matching *_workspace_bytes call returns).
 *   - fp16 and bf16 values are passed as uint16_t bit patterns.
 *   - Return value: DBF_OK (0) or a negative DBF_ERR_* code for errors the
 *     host can see (bad argument, alignment, workspace too small, CUDA launch
 *     error).  Errors seen on the device (a bounded wait that ran out, an
 *     invalid segment table) are recorded in a device status word that
 *     dbf_check_status() reads and clears.
 *   - T = 0 (no tokens) is a no-op that returns DBF_OK.
 *   - The matmul kernels use programmatic dependent launch: they start while
 *     the kernel before them on the stream finishes, and they read factor
 *     memory (packed signs, scales, and the d_adapters table of
 *     dbf_matmul_segmented) before waiting for it; they wait before reading
 *     x, y and the segment tables.  Only kernels that allow this overlap let
 *     it happen (a kernel that does not is complete before the next one
 *     starts): this library's matmul kernels, which never write factor
 *     memory.  So factor memory may come from any earlier copy or kernel,
 *     except a kernel of the caller's that itself allows the overlap.
 */
#ifndef DBF_H
#define DBF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
enum {
    DBF_OK = 0,
    DBF_ERR_INVALID_ARG = -1,  /* null pointer, bad size, ell out of [1,4]   */
    DBF_ERR_ALIGNMENT = -2,    /* a pointer lacks the stated alignment        */
    DBF_ERR_UNSUPPORTED = -3,  /* shape outside what the kernels handle       */
    DBF_ERR_WORKSPACE = -4,    /* workspace null or smaller than required     */
    DBF_ERR_CUDA = -5,         /* a CUDA runtime call or launch failed        */
    DBF_ERR_TIMEOUT = -6,      /* device: a bounded wait ran out              */
    DBF_ERR_DEVICE_ARG = -7,   /* device: segment table out of range          */
    DBF_ERR_NUMERIC = -8,      /* device: a Cholesky pivot was not positive   */
    DBF_ERR_BOUNDS = -9        /* device, debug build only: an index checked
                                  by the kernels was out of range; the access
                                  was skipped                                  */
};

/* Kernel path selection for dbf_matmul_path (dbf_matmul uses DBF_PATH_AUTO). */
enum {
    DBF_PATH_AUTO = 0,     /* decode for T <= dbf_decode_max_tokens(), else prefill */
    DBF_PATH_DECODE = 1,   /* fused sign-accumulate skinny GEMM (mma.sync, register unpack) */
    DBF_PATH_PREFILL = 2   /* tcgen05 GEMM, signs unpacked into tensor memory */
};

/*
 * One set of factors.  All pointers are device memory.
 *   B1    uint32 [N][ldw1]  packed rows of B1 (R sign bits each), 16-byte aligned
 *   B2    uint32 [R][ldw2]  packed rows of B2 (M sign bits each), 16-byte aligned
 *   alpha fp16   [ell][N]   term-major, 16-byte aligned
 *   beta  fp16   [ell][R]
 *   gamma fp16   [ell][M]
 * Packing: bit j of word w of a row is the sign of column 32*w + j (1 = +1,
 * 0 = -1); bits past the last column must be 0 (dbf_pack writes them so).
 * ldw1 >= ceil(R/32), ldw2 >= ceil(M/32); any such stride is accepted.
 * 1 <= ell <= 4; N, M, R >= 1.
 */
typedef struct dbf_factors {
    int32_t N, M, R, ell;
    int32_t ldw1, ldw2;
    const uint32_t *B1;
    const uint32_t *B2;
    const uint16_t *alpha;
    const uint16_t *beta;
    const uint16_t *gamma;
} dbf_factors;

/*
 * dbf_pack: signs (device int8 [rows][cols], row-major, row stride = cols)
 * -> words (device uint32 [rows][ldw]).  Bit j of word w of row r is 1 when
 * signs[r][32w+j] > 0, else 0; so +1 -> 1, -1 -> 0, and 0 (sign(0)) counts
 * as -1 unless callers map it to +1 first.  Bits and words past ceil(cols/32)
 * words are written as 0.  Storage format: one bit per binary factor entry
 * (LoRDBA page, section 2, "Eficiencia de Almacenamiento"); the bit order is
 * this library's own.  ldw >= ceil(cols/32); words 16-byte aligned.
 */
int dbf_pack(const int8_t *signs, int64_t rows, int64_t cols,
             uint32_t *words, int64_t ldw, void *stream);

/* dbf_unpack: inverse of dbf_pack, writes +1/-1 int8 [rows][cols]. */
int dbf_unpack(const uint32_t *words, int64_t rows, int64_t cols, int64_t ldw,
               int8_t *signs, void *stream);

/*
 * dbf_transpose_packed: packed sign matrix -> packed transpose.
 *   words    device uint32 [rows][ldw], a rows x cols sign matrix in the
 *            dbf_pack format (ldw >= ceil(cols/32))
 *   words_t  device uint32 [cols][ldw_t], receives the cols x rows transpose
 *            in the same format (ldw_t >= ceil(rows/32)); pad bits and pad
 *            words are written as 0
 * Both 4-byte aligned.  Setup operation for the backward product (the sign
 * matrices transposed once per factor set).
 */
int dbf_transpose_packed(const uint32_t *words, int64_t rows, int64_t cols, int64_t ldw,
                         uint32_t *words_t, int64_t ldw_t, void *stream);

/*
 * dbf_factors_transposed: descriptor of the backward (input-gradient) product
 *     dx = dy dW = sum_i gamma_i . B2^T (beta_i . (B1^T (alpha_i . dy)))
 * for dy [T][N] -> dx [T][M], the gradient that training through the
 * sign-factor product needs (LoRDBA page, section 2, Pipeline de
 * Entrenamiento: carriers and scales are trained jointly).  It has the form
 * of the forward product with N' = M, M' = N, B1' = B2^T, B2' = B1^T,
 * alpha' = gamma, beta' = beta, gamma' = alpha, so dbf_matmul (any path) with
 * *out computes dx.  Host only: fills *out from f and the two transposes
 * (from dbf_transpose_packed):
 *   B2T  device uint32 [M][ldw_b2t], transpose of B2 (ldw_b2t >= ceil(R/32))
 *   B1T  device uint32 [R][ldw_b1t], transpose of B1 (ldw_b1t >= ceil(N/32))
 * 16-byte aligned.  The scale vectors are shared with f (no copy).
 */
int dbf_factors_transposed(const dbf_factors *f, const uint32_t *B2T, int32_t ldw_b2t,
                           const uint32_t *B1T, int32_t ldw_b1t, dbf_factors *out);

/*
 * dbf_backward: everything training needs from one backward pass through the
 * product (LoRDBA page, section 2, Pipeline de Entrenamiento: the sign
 * carriers and the scales are trained jointly), for the output gradient dy of
 * L = sum_t <dy_t, y_t>:
 *     dx[t]       = sum_i gamma_i . B2^T (beta_i . B1^T (alpha_i . dy_t))
 *     dalpha_i[n] = sum_t dy_t[n] * (B1 (beta_i . B2 (gamma_i . x_t)))[n]
 *     dbeta_i[r]  = sum_t (B1^T (alpha_i . dy_t))[r] * (B2 (gamma_i . x_t))[r]
 *     dgamma_i[k] = sum_t x_t[k] * (B2^T (beta_i . B1^T (alpha_i . dy_t)))[k]
 *   f, ft     host pointers: the factors and their transposed descriptor
 *             (dbf_factors_transposed; only its sign matrices are read, the
 *             scales come from f); shapes must match (ft->N == f->M, ...)
 *   x         device bf16 [T][M], the forward input
 *   dy        device bf16 [T][N]
 *   dx        device bf16 [T][M], or NULL to skip writing dx
 *   dalpha    device fp32 [ell][N], dbeta fp32 [ell][R], dgamma fp32 [ell][M]:
 *             overwritten (zeroed first, then accumulated with atomics, so
 *             the last bits vary from run to run)
 *   workspace device, >= dbf_backward_workspace_bytes(f, T), 256-byte aligned
 * Runs on the prefill (tensor-core) kernels for every T: the forward is
 * recomputed (x -> V, H; then V -> dalpha without writing y), then the
 * transposed product gives dbeta, dx and dgamma: six launches, 2x the FLOPs
 * of one forward call.  Intermediates are fp16 as in the forward product.
 * All device pointers 16-byte aligned.  Asynchronous on `stream`; errors as
 * dbf_matmul.  The workspace must not be shared with concurrent calls.
 */
int dbf_backward(const dbf_factors *f, const dbf_factors *ft, const uint16_t *x,
                 const uint16_t *dy, int64_t T, uint16_t *dx, float *dalpha,
                 float *dbeta, float *dgamma, void *workspace, size_t ws_bytes,
                 void *stream);

/* Device workspace (bytes) dbf_backward needs for this shape and token count. */
size_t dbf_backward_workspace_bytes(const dbf_factors *f, int64_t T);

/*
 * dbf_matmul_grouped: G independent products in one call,
 *     ys[p] = sum_i alpha_i . B1 (beta_i . (B2 (gamma_i . xs[p])))  with fs[p],
 * for projections whose middle dimension R differs from one to the next (the
 * DBF page, section 2 "Control Granular de Compresión" and section 3: the
 * compression ratio is set per layer through the middle dimension, giving
 * non-uniform bits per layer), or any N and M.
 *   fs      host array of G descriptors (device pointers inside), one ell for all
 *   G       1 .. 16
 *   xs, ys  host arrays of G device pointers: bf16 [T][fs[p].M] and [T][fs[p].N],
 *           16-byte aligned
 *   T, accumulate, workspace, stream as dbf_matmul; workspace >=
 *           dbf_grouped_workspace_bytes(fs, G, T)
 * T <= dbf_decode_max_tokens(): two launches for the whole group (one per
 * decode stage; every problem keeps its own shape), instead of one or two per
 * problem.  Larger T: each problem runs the prefill kernels in turn.  Errors
 * as dbf_matmul; DBF_ERR_UNSUPPORTED for G > 16 or when no common tile plan
 * fits the group.
 */
int dbf_matmul_grouped(const dbf_factors *fs, int32_t G, const uint16_t *const *xs,
                       uint16_t *const *ys, int64_t T, int accumulate, void *workspace,
                       size_t ws_bytes, void *stream);

/* Device workspace (bytes) dbf_matmul_grouped needs; 0 for invalid arguments. */
size_t dbf_grouped_workspace_bytes(const dbf_factors *fs, int32_t G, int64_t T);

/* Kernels one dbf_matmul_grouped call launches; -1 for invalid arguments. */
int dbf_grouped_launch_count(const dbf_factors *fs, int32_t G, int64_t T);

/*
 * dbf_matmul_hostio_batch: L independent dbf_matmul_hostio calls (host x in,
 * host y out, each with its own factors fs[l]) pipelined over four slots of
 * device buffers: the copy of x[l+1] to the device and of y[l-1] back to the
 * host run while the kernels of call l run, on the library's own copy-in,
 * compute and read-back streams, which start after the work already queued on
 * `stream` and which `stream` waits for at the end (capturable in a CUDA graph
 * that captures `stream`).
 *   fs              host array of L descriptors
 *   x_host, y_host  host arrays of L host pointers, bf16 [T][fs[l].M] and
 *                   [T][fs[l].N]; page-locked memory for the copies to overlap
 *   workspace       device, >= dbf_hostio_batch_workspace_bytes(fs, L, T)
 * Consecutive calls whose host buffers follow one another inside one
 * page-locked allocation (e.g. one [L][T][M] buffer sliced per call) share
 * one copy each way, up to 32 calls per copy (fewer in the first and last
 * copies of a batch, so the pipeline fills and drains quickly); other calls
 * are copied one by one.  L = 0 or T = 0 is a no-op.  Host-thread safe (an internal lock); the
 * pipeline streams are shared per device, so concurrent batches serialise.
 * Errors as dbf_matmul; after an error the pipeline is still joined back
 * into `stream`, and calls of the batch may or may not have run.
 */
int dbf_matmul_hostio_batch(const dbf_factors *fs, int32_t L, const uint16_t *const *x_host,
                            uint16_t *const *y_host, int64_t T, int accumulate,
                            void *workspace, size_t ws_bytes, void *stream);

/* Device workspace (bytes) of dbf_matmul_hostio_batch; 0 for invalid arguments. */
size_t dbf_hostio_batch_workspace_bytes(const dbf_factors *fs, int32_t L, int64_t T);

/* Device workspace (bytes) dbf_matmul needs for this shape and token count. */
size_t dbf_workspace_bytes(const dbf_factors *f, int64_t T);

/* Largest T that DBF_PATH_AUTO sends to the decode kernels. */
int dbf_decode_max_tokens(void);

/*
 * dbf_matmul: y = sum_i alpha_i . B1 (beta_i . (B2 (gamma_i . x))) per row.
 *   f          host pointer to a dbf_factors whose pointers are device memory
 *   x          device bf16 [T][M] row-major, 16-byte aligned
 *   y          device bf16 [T][N] row-major, 16-byte aligned
 *   accumulate 0: y = branch;  1: y = bf16(y + branch) (y read, then written)
 * Arithmetic (both kernel paths): gamma_i * x is formed in fp32 and rounded
 * once to fp16; the sign sums u = B2 (gamma_i * x) accumulate in fp32;
 * beta_i * u is formed in fp32 and rounded once to fp16; the sums
 * B1 (beta_i * u) accumulate in fp32; sum_i alpha_i * (...) (+ y) is formed
 * in fp32 and rounded once to bf16 (round to nearest even).
 * Preconditions: |gamma_i * x| and |beta_i * u| stay below 65504 (fp16 range
 * of the intermediates).  Integer inputs (integer x, unit scales) give the
 * exactly rounded result only while |x| <= 2048 and |u| <= 2048, the range
 * in which fp16 holds every integer; |y| needs no bound beyond fp32's 2^24.
 */
int dbf_matmul(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y,
               int accumulate, void *workspace, size_t ws_bytes, void *stream);

/* As dbf_matmul, with an explicit kernel path (DBF_PATH_*).  Both paths
 * compute the same product; the choice only affects speed. */
int dbf_matmul_path(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y,
                    int accumulate, void *workspace, size_t ws_bytes, void *stream,
                    int path);

/* Workspace bytes for dbf_matmul_path with an explicit path. */
size_t dbf_workspace_bytes_path(const dbf_factors *f, int64_t T, int path);

/*
 * dbf_matmul_hostio: the same call with HOST activations and outputs.
 *   x_host  bf16 [T][M] in host memory (pinned for asynchronous copies)
 *   y_host  bf16 [T][N] in host memory; read first when accumulate = 1
 * The call copies x_host into the workspace, runs dbf_matmul, and copies y
 * back, all on `stream`; y_host is valid after the stream synchronises.
 * Workspace: dbf_hostio_workspace_bytes(f, T), device memory.
 */
size_t dbf_hostio_workspace_bytes(const dbf_factors *f, int64_t T);
int dbf_matmul_hostio(const dbf_factors *f, const uint16_t *x_host, int64_t T,
                      uint16_t *y_host, int accumulate, void *workspace,
                      size_t ws_bytes, void *stream);

/*
 * dbf_matmul_segmented: a sorted token batch routed to many adapters
 * (multi-adapter serving of unmerged adapters, S-LoRA / Punica style, as on
 * the LoRDBA page, section 1).  Tokens [off[s], off[s+1]) use adapter
 * seg_adapter[s]; each segment is one dbf_matmul with that adapter's factors.
 *   d_adapters    device array of n_adapters dbf_factors; every entry must
 *                 have the given N, M, R and ell
 *   x, y          device bf16 [T][M], [T][N]
 *   d_seg_offsets device int32 [S+1], non-decreasing, off[0] = 0, off[S] = T
 *   d_seg_adapter device int32 [S], each in [0, n_adapters)
 * Rows of y outside every segment are not written.  The table is read on the
 * device (no host synchronisation); an out-of-range entry skips that segment
 * and records DBF_ERR_DEVICE_ARG for dbf_check_status.  With S <= 1024 every
 * chunk of a segment (as many tokens as the launch's column tile holds) gets
 * its own thread-block cluster, found by a scan of the offsets on the device;
 * larger S give a cluster per segment, which runs the segment's chunks in
 * turn.  The results are the same bits either way.
 */
size_t dbf_segmented_workspace_bytes(int32_t N, int32_t M, int32_t R, int32_t ell,
                                     int64_t T, int32_t S);
int dbf_matmul_segmented(const dbf_factors *d_adapters, int32_t n_adapters,
                         int32_t N, int32_t M, int32_t R, int32_t ell,
                         const uint16_t *x, int64_t T, uint16_t *y,
                         const int32_t *d_seg_offsets, const int32_t *d_seg_adapter,
                         int32_t S, int accumulate, void *workspace, size_t ws_bytes,
                         void *stream);

/*
 * dbf_launch_count: number of kernel launches one dbf_matmul_path call makes
 * for these factors, T and path (the fused decode kernel: 1; the two-stage
 * decode kernels: 2; prefill: 3).  Host only, touches no device memory.
 * Returns 0 for T <= 0 or invalid arguments.
 * dbf_segmented_launch_count: the same for dbf_matmul_segmented.
 */
int dbf_launch_count(const dbf_factors *f, int64_t T, int path);
int dbf_segmented_launch_count(int32_t N, int32_t M, int32_t R, int32_t ell, int64_t T, int32_t S);

/*
 * dbf_check_status: synchronises `stream`, then returns and clears the device
 * status word of the current device (DBF_OK when no kernel recorded an
 * error).  A CUDA error from the synchronisation returns DBF_ERR_CUDA.
 */
int dbf_check_status(void *stream);

/*
 * dbf_selftest_bounded_wait: launches one block that waits on an mbarrier
 * nobody arrives on, with the library's bounded wait and a limit of
 * `limit_us` microseconds (1..2000000).  The wait gives up, records
 * DBF_ERR_TIMEOUT in the device status word and the block exits normally;
 * the CUDA context stays usable.  For tests of the failure path.
 */
int dbf_selftest_bounded_wait(int64_t limit_us, void *stream);

/*
 * dbf_selftest_split_gemm: C = alpha * A B^T + beta * C on the tensor-core
 * GEMM that dbf_factorize uses for its P-update and T F^T (each operand split
 * into two tf32 parts, three tf32 products per term, fp32 accumulation; DBF
 * page, section 2, the ADMM P-update).  For tests of that kernel.
 *   A  device fp32 [m][lda], B device fp32 [n][ldb], C device fp32 [m][ldc]
 *      (all row-major; K = kk columns of A and B are used)
 *   lower  1: tiles of C wholly above the diagonal (128 x 256 tiles) are
 *          left untouched
 *   workspace  device, >= dbf_selftest_split_gemm_workspace_bytes(m, n, kk),
 *              256-byte aligned (the split forms of A and B)
 * 1 <= m, n, kk <= 65535 and lda, ldb >= kk, ldc >= n, else
 * DBF_ERR_INVALID_ARG / DBF_ERR_UNSUPPORTED.  Asynchronous on `stream`.
 */
size_t dbf_selftest_split_gemm_workspace_bytes(int32_t m, int32_t n, int32_t kk);
int dbf_selftest_split_gemm(int32_t m, int32_t n, int32_t kk, float alpha, const float *A, int64_t lda,
                            const float *B, int64_t ldb, float beta, float *C, int64_t ldc, int lower,
                            void *workspace, size_t ws_bytes, void *stream);

/*
 * dbf_selftest_decode_one_launch: the decode path's two stages (x -> V and
 * V -> y, DBF page, section 2, "Cálculo en la inferencia": the gamma, B2,
 * beta, B1, alpha chain) in ONE cooperative launch, with a grid-wide barrier
 * between the stage that writes V and the stage that reads it, instead of two
 * launches.  The comparison arm of the two-launch form that dbf_matmul takes
 * for large R; for tests and timing.
 *   f, x, T, y, accumulate, workspace, ws_bytes, stream: as dbf_matmul_path
 *      with DBF_PATH_DECODE (1 <= T <= dbf_decode_max_tokens(); T = 0 does
 *      nothing).  Any R; the same stage code, arithmetic and summation
 *      order as the two-launch form, so the result is bit for bit that of
 *      dbf_matmul_path with DBF_PATH_DECODE wherever that call takes the
 *      two launches (R > 256).
 *   barrier  device, two uint32 words, 8-byte aligned, zero before the first
 *      call; every call that completes advances the first word by 1024
 *      (modulo 2^32) and leaves the second at 0, ready for the next call.
 *      Calls that may overlap on the GPU need a pair each.
 * DBF_ERR_UNSUPPORTED (reason in dbf_last_cuda_error()) when the two stages'
 * tile plans split K over different cluster sizes (neither of them 1), when
 * their shared memory together exceeds a CTA's, or when the grid cannot be
 * resident at once; DBF_ERR_INVALID_ARG for a missing or misaligned
 * barrier or T above the decode range.  A barrier wait that runs out (1 s)
 * records DBF_ERR_TIMEOUT; the call's y is then undefined and the barrier
 * words must be zeroed again.  Grids above 1024 CTAs are DBF_ERR_UNSUPPORTED.
 */
int dbf_selftest_decode_one_launch(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y,
                                   int accumulate, void *workspace, size_t ws_bytes, uint32_t *barrier,
                                   void *stream);

/*
 * dbf_matmul_decode_noalloc: dbf_matmul_path(..., DBF_PATH_DECODE) for
 * callers that cannot allocate device memory for a call: serving loops that
 * must never take cudaMalloc's implicit device synchronisation on the token
 * path, runtimes whose device memory is one arena planned at start-up, and
 * plug-in hosts that hand a library only its inputs and outputs.  The papers
 * have no counterpart; this is a deployment variant of the decode path.
 *   Arguments as dbf_matmul (f, x, T, y, accumulate, stream); no workspace.
 *   Result: bit for bit the result of dbf_matmul_path with DBF_PATH_DECODE
 *   (the same argument checks, kernels and device status word).
 *   Scratch: a 2 MiB static device array inside the library, held by every
 *   GPU that loads the library until the process exits.  Calls needing more
 *   than 2 MiB (dbf_workspace_bytes_path(f, T, DBF_PATH_DECODE), i.e.
 *   ell * T * round_up(R, 64) * 2 bytes rounded up to 256) are rejected with
 *   DBF_ERR_WORKSPACE before any device work, with the reason in
 *   dbf_last_cuda_error().
 *   The first call on each device (with that device current) looks up the
 *   array's device address (cudaGetSymbolAddress, no allocation); make that
 *   first call before any stream capture.
 *   Every call shares the one array and the array keeps the last call's
 *   contents; the kernels write every element of it they read before reading
 *   it, so nothing needs clearing, but calls that overlap on the GPU
 *   (concurrent streams, or several host threads on one device) race on it:
 *   serialise them.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
int dbf_matmul_decode_noalloc(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y,
                              int accumulate, void *stream);

/* ------------------------------------------------ dense factorization */
/*
 * Parameters of dbf_factorize.  The pages give the steps of the optimiser,
 * not its schedule; these are the counts and the penalty it runs with.
 */
typedef struct dbf_factorize_params {
    int32_t outer;        /* alternating rounds (A-step, then B-step), >= 0 */
    int32_t inner;        /* ADMM iterations in each step, >= 0              */
    int32_t power_iters;  /* power iterations of each SVID rank-1 step, >= 0 */
    float rho_rel;        /* ADMM penalty as a multiple of mean(diag(F F^T)), > 0 */
} dbf_factorize_params;

/*
 * dbf_factorize: double binary factorization of a dense matrix,
 *     W ~ (a . A . m^T)(B . b^T),  m = m_left . m_right,
 * ("Addition is almost all you need: Compressing large language models
 * with double binary factorization", section 2, Formulación Matemática and
 * Algoritmo de Optimización).  Each round fixes one factor and fits the
 * other by ADMM with the SVID projection:
 *     A-step  min 1/2 ||W - P Q||^2,  P = diag(a) A diag(m_left),
 *             Q = diag(m_right) B diag(b) fixed;
 *     B-step  the same on W^T for Q^T = diag(b) B^T diag(m_right), P fixed;
 *     ADMM    P = (T F^T + rho (Z - U)) (F F^T + rho I)^-1,
 *             Z = SVID(P + U), U = U + P - Z,
 *             rho = rho_rel * mean(diag(F F^T)) (rho_rel if F is zero),
 *             started from Z = the factor being replaced, U = 0;
 *     SVID(Y) = sign(Y) (sign(0) = +1) times r c^T, c from power_iters
 *             power iterations on |Y| from the all-ones direction
 *             (v = |Y|^T |Y| v, normalised), r = |Y| c.
 * The result of each step is the last Z.  With m = m_left . m_right the
 * factors are those of dbf_factors with ell = 1: alpha = a, B1 = A,
 * beta = m, B2 = B, gamma = b (pack A and B with dbf_pack, scales to fp16).
 *   W        device fp32 [N][M] row-major (read only)
 *   a, A, m_left    device fp32 [N], int8 [N][k] (+1/-1), fp32 [k]: the
 *                   left factor; read as the start of the first A-step (a
 *                   zero a starts it at Z = 0), overwritten with the result
 *   m_right, B, b   device fp32 [k], int8 [k][M] (+1/-1), fp32 [M]: the
 *                   right factor, fixed in the first A-step, overwritten
 *   workspace  device, >= dbf_factorize_workspace_bytes(N, M, k), 256-byte
 *              aligned, not shared with concurrent calls
 * Computes to fp32 accuracy: the P-update and T F^T products on the tensor
 * cores from operands split into two tf32 parts (three products per term),
 * F F^T and the inverse on fp32 SIMT GEMMs, a blocked Cholesky; the reductions have a
 * fixed order, so a rerun gives the same bits.  Limits: 1 <= N, M <= 65535,
 * 1 <= k <= 16384, else DBF_ERR_UNSUPPORTED; null pointers or params out of
 * range give DBF_ERR_INVALID_ARG.  Asynchronous on `stream`; a pivot that
 * is not positive (possible only for a tiny rho_rel) is recorded as
 * DBF_ERR_NUMERIC for dbf_check_status and the step continues.
 * outer = 0 or inner = 0 leaves the factors as given.
 */
int dbf_factorize(const float *W, int64_t N, int64_t M, int64_t k, const dbf_factorize_params *params,
                  float *a, int8_t *A, float *m_left, float *m_right, int8_t *B, float *b,
                  void *workspace, size_t ws_bytes, void *stream);

/* Device workspace (bytes) dbf_factorize needs; 0 for sizes out of range. */
size_t dbf_factorize_workspace_bytes(int64_t N, int64_t M, int64_t k);

/* Kernels one dbf_factorize call launches; -1 for arguments out of range. */
int dbf_factorize_launch_count(int64_t N, int64_t M, int64_t k, const dbf_factorize_params *params);

/*
 * dbf_factorize_weighted: the factorization with importance weights (the
 * DBF page, section 2, Importancia de Entradas y Salidas: input activation
 * norms and output gradient norms weight the approximation error), i.e.
 * the same steps for the objective
 *     || diag(d_out) (W - W_hat) diag(d_in) ||_F.
 * Because diag(d_out) P and Q diag(d_in) keep the factored form, it runs
 * dbf_factorize on W' = diag(d_out) W diag(d_in) from the start
 * (d_out . a, A, m_left; m_right, B, b . d_in) and divides the weights out
 * of a and b at the end.
 *   d_out, d_in  device fp32 [N], [M], positive and finite; an entry that is
 *                not leaves its scale unconverted and records
 *                DBF_ERR_DEVICE_ARG for dbf_check_status
 * Other arguments, limits and errors as dbf_factorize; the workspace is
 * dbf_factorize_weighted_workspace_bytes(N, M, k) (W' after the plain
 * scratch).  Unit weights give the bits of dbf_factorize.
 * After an error return (DBF_ERR_CUDA from a launch), a, A, m_left,
 * m_right, B and b are undefined: the weights are divided back out of a and
 * b on that path too when the context still accepts launches, but the
 * rounds may have stopped part-way.
 */
int dbf_factorize_weighted(const float *W, int64_t N, int64_t M, int64_t k, const dbf_factorize_params *params,
                           const float *d_out, const float *d_in, float *a, int8_t *A, float *m_left,
                           float *m_right, int8_t *B, float *b, void *workspace, size_t ws_bytes,
                           void *stream);

/* Device workspace (bytes) dbf_factorize_weighted needs; 0 for sizes out of range. */
size_t dbf_factorize_weighted_workspace_bytes(int64_t N, int64_t M, int64_t k);

/* Kernels one dbf_factorize_weighted call launches (dbf_factorize's + 5); -1 for
 * arguments out of range. */
int dbf_factorize_weighted_launch_count(int64_t N, int64_t M, int64_t k, const dbf_factorize_params *params);

/* Human-readable text for a DBF_* code (static string). */
const char *dbf_status_string(int code);

/* Text of the last CUDA error the library saw on this thread (static buffer). */
const char *dbf_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DBF_H */
