/*
 * tgemm — fused tensor-core GEMM with an in-kernel epilogue, for GB300 (sm_103a).
 *
 *     C[i, j] = epi( sum_{k<K} A[i, k] * B[k, j]  (+ bias[j]) )    0 <= i < M, 0 <= j < N
 *
 * The operation is the GEMM of "从零开始学习 TileLang：从 Python、PyTorch 到高性能
 * GPU Kernel 的完整开发教程", ch.10 §10.1 (C_ij = sum_k A_ik B_kj, 2MNK flops,
 * §10.9), with the epilogue of its §10.8 "GEMM Epilogue 融合" (relu(a @ b + bias),
 * bias indexed by the output column, applied before the write-back), the
 * C = ReLU(A @ B) kernel of "Writing high-performance kernels in TileLang"
 * ("Écrivons un GEMM"), the Bias (N,) operand of "TileLang で GPU カーネル設計を
 * 解説" §4, and the load -> GEMM -> activation -> store tile fusion of
 * "【CUDA】TileFusion".  Precision follows the tutorial's §10.7 recipe: fp16 or
 * bf16 inputs, tensor-core products, fp32 accumulation, one final rounding to
 * the input dtype (round to nearest even).  ReLU maps x <= 0 (including -0.0)
 * to +0.0 and keeps NaN.  The GELU epilogue (below) is the bias + GELU fusion
 * of "TileLang で GPU カーネル設計を解説" §4.
 *
 * Layout: every matrix is row-major with an explicit leading dimension (row
 * pitch, in elements): A[i, k] at A + i*lda + k, B[k, j] at B + k*ldb + j,
 * C[i, j] at C + i*ldc + j.  bias has N contiguous elements.  All four arrays
 * hold the same dtype.  Elements of C outside 0 <= j < N (the pitch padding)
 * are never written.
 *
 * Ownership: the caller owns every buffer; the library never frees, retains or
 * reads a pointer after the enqueued work completes.
 */
#ifndef TGEMM_H
#define TGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *tgemm_stream_t;   /* same handle as cudaStream_t; NULL = legacy default stream */

typedef enum { TGEMM_F16 = 0, TGEMM_BF16 = 1 } tgemm_dtype;

/*
 * GELU is the tanh form of "TileLang で GPU カーネル設計を解説" §4, written there
 * as a sigmoid: gelu(x) = x / (1 + exp(-1.5957691216 * (x + 0.044715 x^3))),
 * applied after the bias; evaluated in fp32 with CUDA's fast exponential.
 */
typedef enum {
    TGEMM_EPI_NONE = 0,       /* C = A.B                 */
    TGEMM_EPI_RELU = 1,       /* C = max(A.B, 0)         */
    TGEMM_EPI_BIAS = 2,       /* C = A.B + bias          */
    TGEMM_EPI_BIAS_RELU = 3,  /* C = max(A.B + bias, 0)  */
    TGEMM_EPI_GELU = 4,       /* C = gelu(A.B)           */
    TGEMM_EPI_BIAS_GELU = 5   /* C = gelu(A.B + bias)    */
} tgemm_epilogue;

typedef enum {
    TGEMM_OK = 0,
    TGEMM_ERR_INVALID_ARG = 1,        /* bad size, pitch, NULL pointer, dtype or epilogue   */
    TGEMM_ERR_ALIGNMENT = 2,          /* a base pointer is not 16-byte aligned               */
    TGEMM_ERR_UNSUPPORTED_DEVICE = 3, /* no CUDA device, or the current device is not CC 10.3 */
    TGEMM_ERR_ALIAS = 4,              /* C's byte range overlaps A, B or bias                */
    TGEMM_ERR_CUDA = 5,               /* a CUDA runtime/driver call or a launch failed       */
    TGEMM_ERR_TIMEOUT = 6,            /* a kernel gave up on a pipeline wait (device status) */
    TGEMM_ERR_SCRATCH_LIMIT = 7,      /* tgemm_run_noalloc: repacked operands exceed its fixed scratch */
    TGEMM_ERR_DEBUG_CHECK = 8         /* debug build: a device-side bounds / alignment check failed
                                         and the access was skipped (device status) */
} tgemm_status;

/*
 * tgemm_run — enqueue C = epi(A.B + bias) on `stream` (device pointers).
 *
 * Arguments: A [M x lda], B [K x ldb], bias [N] (may be NULL unless the
 * epilogue uses it: BIAS, BIAS_RELU, BIAS_GELU), C [M x ldc], all device
 * pointers in `dtype`.
 *
 * Errors are reported synchronously, before anything is enqueued, and leave C
 * untouched:
 *   M, N or K < 0; lda < K, ldb < N or ldc < N; a NULL A, B or C when the
 *   problem is not empty; a NULL bias with a BIAS epilogue; an unknown dtype or
 *   epilogue                                              -> TGEMM_ERR_INVALID_ARG
 *   a base pointer (A, B, C, bias) not 16-byte aligned    -> TGEMM_ERR_ALIGNMENT
 *   C's byte range overlapping A's, B's or bias's         -> TGEMM_ERR_ALIAS
 *   no device, or a current device other than CC 10.3    -> TGEMM_ERR_UNSUPPORTED_DEVICE
 *   a pointer the driver does not know as device memory   -> TGEMM_ERR_INVALID_ARG
 *   a failed CUDA call or launch                          -> TGEMM_ERR_CUDA
 *
 * Degenerate sizes: M == 0 or N == 0 enqueues nothing and returns TGEMM_OK;
 * K == 0 writes epi(bias) (the empty sum is 0).
 *
 * Any pitch >= the logical width is accepted.  When lda or ldb is not a
 * multiple of 8 elements (tensor-memory-access copies need 16-byte row
 * strides) the operand is first repacked on the GPU into a 16-byte-pitched
 * scratch buffer drawn stream-ordered from a library-owned memory pool and
 * returned to it on `stream`; when ldc is not a multiple of 8 the epilogue
 * stores C with plain masked stores instead of tensor-memory-access stores.
 * The library may read (never write) any element of the declared input
 * arrays, pitch padding included: a padded element only ever feeds outputs
 * outside C's M x N, which are not stored.
 *
 * Environment overrides of the work plan, for testing and tuning only (results
 * change at most by the split-K note below): TGEMM_FORCE_CFG (tile shape:
 * 256, 192, 128, 64, 256x2, 224x2, 128x2, or 256x4: two 256 x 256 CTA pairs
 * stacked in M that share B by cluster multicast), TGEMM_SPLIT_K (k ranges
 * for every tile), TGEMM_TAIL_SPLIT (the last partial wave's tiles: 0 = kept
 * whole, 1 = cut into column parts only), TGEMM_GROUP_M (row-blocks per
 * column sweep), TGEMM_NO_B3D (one copy per 64-column sub-tile of B).
 * TGEMM_TEST_STALL=1 (testing the failure path only) makes the GEMM kernel of
 * each call announce 16 bytes that never arrive for its first operand slot: its
 * operand wait runs out after 2 s, the kernel records TGEMM_ERR_TIMEOUT in the
 * device status word, drains and returns (C is left incomplete).
 * TGEMM_TRACE_MAX_GROUPS caps the persistent CTA groups in trace builds
 * (compiled with -DTGEMM_TRACE, never the product build) and is ignored
 * otherwise.
 *
 * Problems with too few output tiles to fill the GPU (few rows, e.g. decode
 * shapes) split the k loop of each tile across CTAs: fp32 partial sums go to
 * pool scratch and the last CTA to finish a tile region adds them in a fixed
 * order before the epilogue, so results are deterministic; they may differ
 * in the last bits from an unsplit run (different summation order).  The
 * arrival counters of those regions live in a small buffer the library keeps
 * for each stream it has launched such work on (8 bytes per region, at least
 * 4 KiB, drawn from its pool and kept until the process exits); calls on one
 * stream are ordered, so they share it safely.  Kernels are enqueued as
 * programmatic dependent launches: their set-up may overlap the end of the
 * stream's previous kernel, but they touch no global memory before that
 * kernel has completed, so stream order holds as for any launch.  Larger
 * problems whose tiles leave a last, partial wave cut those tiles the same
 * way (2-4 k ranges, each at least 16 k-blocks, when the pieces fit one wave;
 * same determinism, and those tiles may differ in the last bits from an
 * unsplit run), else into narrower column parts, which change no result bit.
 *
 * Asynchrony: returns once the work is enqueued; the caller synchronises.
 * Thread safety: safe to call from several host threads.
 */
tgemm_status tgemm_run(const void *A, const void *B, const void *bias, void *C,
                       int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldc,
                       tgemm_dtype dtype, tgemm_epilogue epilogue, tgemm_stream_t stream);

/*
 * tgemm_run_ex — tgemm_run with either operand stored transposed (the
 * transpose_A / transpose_B options of T.gemm in "Writing high-performance
 * kernels in TileLang", "Écrivons un GEMM"; the column-major B of
 * "【CUDA】TileFusion").  The product is still C = epi(A.B + bias) with A
 * M x K and B K x N:
 *   transpose_a = 0: A[i, k] at A + i*lda + k   (stored [M, lda], lda >= K)
 *   transpose_a = 1: A[i, k] at A + k*lda + i   (stored [K, lda], lda >= M)
 *   transpose_b = 0: B[k, j] at B + k*ldb + j   (stored [K, ldb], ldb >= N)
 *   transpose_b = 1: B[k, j] at B + j*ldb + k   (stored [N, ldb], ldb >= K:
 *                    the [out_features, in_features] weight layout)
 * The tensor cores read either major directly; nothing is transposed in
 * memory.  Errors as tgemm_run (a transpose flag other than 0 or 1 ->
 * TGEMM_ERR_INVALID_ARG).
 */
tgemm_status tgemm_run_ex(const void *A, const void *B, const void *bias, void *C,
                          int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldb, int64_t ldc,
                          tgemm_dtype dtype, tgemm_epilogue epilogue,
                          int transpose_a, int transpose_b, tgemm_stream_t stream);

/*
 * tgemm_run_host — the same operation on HOST buffers (pinned or pageable),
 * end to end: device buffers are drawn from the library's stream-ordered pool,
 * A, B and bias are copied host -> device on `stream`, tgemm_run is enqueued,
 * C is copied device -> host, and the buffers are returned to the pool.
 * The call returns after enqueueing; C_host is valid once `stream` has been
 * synchronised (with pageable memory the copies themselves may block).
 * Same arguments, pitches and errors as tgemm_run (no device-pointer check).
 */
tgemm_status tgemm_run_host(const void *A_host, const void *B_host, const void *bias_host,
                            void *C_host, int64_t M, int64_t N, int64_t K,
                            int64_t lda, int64_t ldb, int64_t ldc,
                            tgemm_dtype dtype, tgemm_epilogue epilogue, tgemm_stream_t stream);

/*
 * tgemm_run_noalloc — tgemm_run for callers that must not allocate GPU memory.
 * (No counterpart on the pages: this is a deployment variant of the same
 * operation.)
 *
 * Who needs it: code whose device memory is reserved up front by another
 * allocator (a framework's caching allocator that holds most of HBM, so a
 * library-side cudaMalloc/cudaMallocAsync can fail or fragment that reserve),
 * latency-bound loops that avoid allocation calls because they can block or
 * synchronise, and deployments that forbid any allocation after start-up.
 *
 * What differs from tgemm_run: nothing is allocated.  The only scratch this
 * operation needs — the repacked copy of A and/or B when lda or ldb is not a
 * multiple of 8 elements — lives in a fixed device array inside the library of
 * TGEMM_NOALLOC_SCRATCH_BYTES (64 MiB), which every GPU that loads the library
 * holds until the process exits.  Each repacked operand takes
 * rows * round_up(width, 8) * 2 bytes, rounded up to 256 bytes; if the
 * operands that need repacking do not fit together, the call returns
 * TGEMM_ERR_SCRATCH_LIMIT before enqueueing anything.  Operands whose pitch is
 * already a multiple of 8 use no scratch at all.
 *
 * Sharing: every call, on every stream and host thread, uses the same array,
 * so two calls that may overlap on the GPU race on it; order them (one
 * stream, or events).  The array keeps the previous call's contents; nothing
 * in it needs to start at zero, because each call writes every scratch
 * element it reads before reading it.
 *
 * Set-up: the first call on each device (with that device current) looks up
 * the device address of the array once; make that first call before any
 * stream capture.
 *
 * Arguments, layout and the other error codes are those of tgemm_run.
 * Results: this variant never splits the k loop (the fp32 partial sums would
 * need scratch), while tgemm_run splits it for problems with few output tiles
 * and may split the tiles of a last, partial wave.  The two therefore agree
 * bit for bit wherever tgemm_run's plan has no k split (tgemm_plan reports
 * split_k == 1) and whenever every partial sum is exact (small-integer
 * inputs); otherwise both are within the same error bound of the exact
 * result and may differ in the last bits.
 */
#define TGEMM_NOALLOC_SCRATCH_BYTES (64ull << 20)
tgemm_status tgemm_run_noalloc(const void *A, const void *B, const void *bias, void *C,
                               int64_t M, int64_t N, int64_t K,
                               int64_t lda, int64_t ldb, int64_t ldc,
                               tgemm_dtype dtype, tgemm_epilogue epilogue, tgemm_stream_t stream);

/* Static, human-readable name of a status code (never NULL). */
const char *tgemm_status_string(tgemm_status status);

/*
 * tgemm_last_device_status — read and clear the device-side status word of the
 * current device.  Kernels bound every pipeline wait by a time limit; a wait
 * that runs out records TGEMM_ERR_TIMEOUT here and the kernel returns early
 * (its output is then invalid).  In the debug build a failed device-side check
 * records TGEMM_ERR_DEBUG_CHECK, and the first error since the last call is
 * kept (the release build keeps the last).  Synchronises the device.  Returns TGEMM_OK when no kernel has reported an
 * error since the last call.
 */
tgemm_status tgemm_last_device_status(void);

/*
 * tgemm_debug_last_check — the debug build (libtgemm_debug.so, compiled with
 * -DTGEMM_DEBUG; the Python binding loads it when TGEMM_DEBUG=1 is set): the
 * id of the first device-side check that failed since the last call, then
 * cleared; 0 when none failed.  The checks guard the error classes the
 * TileLang tutorial names for hand-written kernels: 1 / 2 a TMA load of A /
 * B whose innermost coordinate is not 16-byte aligned, 3 a TMA store of C
 * starting at a negative, unaligned or out-of-range coordinate, 4 a plain
 * store of C outside its (M - 1) * ldc + N elements, 5 a split-K partial
 * outside its scratch, 6 an arrival counter outside its buffer, 7 an
 * attention output store outside O, 8 a repack store outside its
 * destination.  The failing access is skipped (nothing traps); a skipped
 * copy leaves its pipeline slot incomplete, which the bounded waits end.
 * Synchronises the device.  Returns -1 in the release build, which compiles
 * no checks.  Testing only: TGEMM_DEBUG_PLANT=c_store makes the debug build's
 * bound for C one row short, so that check 4 fires on C's last row (whose
 * stores are then skipped).
 */
int tgemm_debug_last_check(void);

/* Library version, e.g. 0x000100 for 0.1.0. */
int tgemm_version(void);

/*
 * tgemm_attention_fwd — enqueue the attention forward pass (the output of
 * FlashAttention, "TileLang で GPU カーネル設計を解説" §6) on `stream`:
 *
 *   O[b, i, h, :] = sum_j softmax_j(scale * Q[b, i, h, :] . K[b, j, h, :]) V[b, j, h, :],
 *   scale = 1 / sqrt(dim),
 *
 * over all keys j < seq, or only j <= i when causal = 1.
 *
 * Arguments: Q, K, V, O device pointers in `dtype` (fp16 or bf16), each a
 * dense [batch, seq, heads, dim] array (dim contiguous, then heads, then seq,
 * then batch), 16-byte aligned; O must not overlap Q, K or V.  dim must be 64.
 * Ownership stays with the caller; the call only reads Q, K, V and writes O.
 *
 * Arithmetic: scores and P.V products accumulate in fp32; the softmax runs
 * blockwise over 128 keys at a time with a running maximum and sum (the
 * online softmax), P is rounded to `dtype` before it multiplies V, and each
 * output row is divided by the fp32 sum of the unrounded P and rounded once
 * to `dtype` (round-to-nearest-even).
 *
 * Returns TGEMM_ERR_INVALID_ARG (negative sizes, dim != 64, causal not 0/1,
 * bad dtype, batch or heads above 65535, a NULL or host pointer for a
 * non-empty problem), TGEMM_ERR_ALIGNMENT, TGEMM_ERR_ALIAS,
 * TGEMM_ERR_UNSUPPORTED_DEVICE, TGEMM_ERR_CUDA; TGEMM_OK once enqueued.
 * An empty problem (batch, seq or heads 0) enqueues nothing.
 */
tgemm_status tgemm_attention_fwd(const void *Q, const void *K, const void *V, void *O,
                                 int64_t batch, int64_t seq, int64_t heads, int64_t dim,
                                 int causal, tgemm_dtype dtype, tgemm_stream_t stream);

/*
 * tgemm_plan — the work plan tgemm_run (and tgemm_run_ex / tgemm_run_host per
 * chunk) uses for an M x N x K problem on a GPU with num_sms SMs.  Host logic
 * only: no device is touched, so it also answers on a machine without a GPU.
 * The transposed layouts do not change the plan; tgemm_run_noalloc uses it
 * with split_k forced to 1.
 *
 * out (caller-owned, 10 int32 entries):
 *   [0] tile width BN (columns)      [1] CTAs per tile (1; 2 for a pair: 256 rows;
 *                                        4 for two pairs sharing B: 512 rows)
 *   [2] shared-memory ring stages    [3] tiles = ceil(M / (128 * [1])) * ceil(N / BN)
 *   [4] persistent CTA groups launched (CTAs = [4] * [1])
 *   [5] split_k (1: no k split)      [6] first tile split in k (tiles from here on)
 *   [7] first narrow tile            [8] column parts of each narrow tile (1: none);
 *                                        tiles [7] .. [6]-1 are cut into [8] parts
 *   [9] work units of the persistent loop
 *
 * The tile-shape rule and the plan are heuristics: they may change between
 * versions without changing any result beyond the split-K note of tgemm_run.
 * Returns TGEMM_ERR_INVALID_ARG if out is NULL, num_sms < 2, or a size is
 * below 1 or above INT32_MAX; TGEMM_OK otherwise.
 */
tgemm_status tgemm_plan(int64_t M, int64_t N, int64_t K, int num_sms, int32_t *out);

#ifdef __cplusplus
}
#endif

#endif /* TGEMM_H */
