/*
 * sgemm.h: C ABI of the GB300 (sm_103a) single-precision GEMM library.
 *
 * Operation, for every entry point below:
 *
 *     C = alpha * (A . B) + beta * C
 *
 * with A an M x K, B a K x N and C an M x N matrix of fp32 values, all row-major: element
 * (r, c) of a matrix with leading dimension ld sits at index r * ld + c. This is the SGEMM of
 * "a CUDA matmul" (section 00, and the naive kernel of section 02, whose strides are the
 * packed lda = K, ldb = N, ldc = N generalised here), and the GEMM definition of the "GEMM
 * scrapbook" (each cell of C is one row of A dotted with one column of B).
 *
 * Conventions shared by all entry points
 * --------------------------------------
 * Memory and ownership: A, B and C are device pointers owned by the caller (for example
 *   torch CUDA tensors). The library keeps no reference to them after the call returns.
 *   No entry point allocates device memory on every call: workspaces are allocated on first
 *   use (per device and stream: stream-K and split-K partial sums, repacked or transposed
 *   operand copies, the staged product of an unaligned C, the 3xTF32 / TF32 split operands;
 *   per device: the host-memory path's buffers), grown when a larger problem needs more, and
 *   kept until sgemm_release_workspace(). sgemm_noalloc() uses none of them.
 * Streams: every compute call is asynchronous on `stream` (a cudaStream_t; NULL means the
 *   legacy default stream) and does not synchronise. Results are visible to later work on
 *   the same stream.
 * alpha and beta (BLAS convention): beta == 0 means C is write-only (NaN or Inf already in
 *   C does not reach the result). alpha == 0 or K == 0 means C = beta * C, and A and B are
 *   not read (they may then be NULL).
 * Degenerate sizes: M == 0, N == 0 or batch == 0 is a no-op that returns SGEMM_OK without
 *   touching any pointer.
 * Alignment: none is required. 16-byte aligned pointers with leading dimensions (and batch
 *   strides) that are multiples of 4 elements select the TMA fast path; anything else runs a
 *   cp.async path with the same arithmetic.
 * Aliasing: C must not overlap A or B (undefined result, as in BLAS).
 * Accuracy: the SIMT entry points accumulate in fp32 with fused multiply-adds in ascending k
 *   for every output cell; the result differs from the exact value by rounding only.
 * Errors: argument errors return SGEMM_ERR_INVALID_VALUE before any device work is queued.
 *   A failed launch returns SGEMM_ERR_LAUNCH. Every wait inside a kernel is bounded; a wait
 *   that expires sets a device error word, makes the kernel return early (its output is then
 *   undefined) and is reported as SGEMM_ERR_TIMEOUT by sgemm_device_status(). A readable
 *   message for the calling thread's last non-OK return is given by sgemm_last_error().
 * Thread safety: calls from several host threads are safe; each thread has its own
 *   sgemm_last_error() text.
 */
#ifndef DENSE_FP32_GEMM_08_GB300_SGEMM_H
#define DENSE_FP32_GEMM_08_GB300_SGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sgemm_status {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_VALUE = 1, /* bad size, leading dimension, stride or NULL pointer */
    SGEMM_ERR_LAUNCH = 2,        /* the CUDA runtime refused a launch or a setup call */
    SGEMM_ERR_TIMEOUT = 3,       /* a bounded wait inside a kernel expired */
    SGEMM_ERR_UNSUPPORTED = 4    /* valid arguments this build cannot run (e.g. no GPU) */
} sgemm_status_t;

/* Operand form (BLAS transa / transb, row-major storage). */
typedef enum sgemm_op {
    SGEMM_OP_N = 0, /* the operand as stored: A is M x K (lda >= K), B is K x N (ldb >= N) */
    SGEMM_OP_T = 1  /* its transpose: A stored K x M (lda >= M), B stored N x K (ldb >= K) */
} sgemm_op_t;

/* Arithmetic path (the accuracy / speed knob of sgemm_ex). */
typedef enum sgemm_path {
    SGEMM_PATH_SIMT = 0,   /* fp32 FMAs on the SIMT cores: the sgemm() path */
    SGEMM_PATH_3XTF32 = 1, /* three TF32 tensor-core products: the sgemm_3xtf32() path */
    SGEMM_PATH_TF32 = 2    /* one TF32 tensor-core product: the sgemm_tf32() path */
} sgemm_path_t;

/* Activation of the fused epilogue (sgemm_fused). */
typedef enum sgemm_activation {
    SGEMM_ACT_NONE = 0,
    SGEMM_ACT_RELU = 1,      /* max(x, 0); NaN stays NaN */
    SGEMM_ACT_GELU = 2,      /* 0.5 x (1 + erf(x / sqrt 2))  (Hendrycks & Gimpel 2016) */
    SGEMM_ACT_GELU_TANH = 3, /* 0.5 x (1 + tanh(sqrt(2 / pi) (x + 0.044715 x^3))) */
    SGEMM_ACT_SILU = 4       /* x / (1 + exp(-x))  (Elfwing, Uchibe & Doya 2018) */
} sgemm_activation_t;

/*
 * C = alpha * (A . B) + beta * C on the FP32 SIMT path ("GEMM scrapbook": 2D block tiling
 * with register outer products, float4 loads, warp tiling and double buffering; here a
 * multi-stage TMA or cp.async shared-memory ring and paired fp32 FMAs).
 *   M, N, K   >= 0.
 *   A         M x K, lda >= max(1, K).   B   K x N, ldb >= max(1, N).
 *   C         M x N, ldc >= max(1, N).
 *   A, B may be NULL only when alpha == 0 or K == 0; C may be NULL only when M or N is 0.
 *   stream    cudaStream_t or NULL.
 * Any alignment. When C's rows are not 16-byte aligned (an ldc that is not a multiple of 4, or
 * a misaligned C), beta != 0 and M * N is at least 2^22, the product is computed into an
 * aligned workspace of 4 * M * N' bytes (N' = N rounded up to a multiple of 4) and a second
 * pass applies alpha, beta (and, for sgemm_fused on this path, the bias and activation) to C:
 * the same fp32 arithmetic as the single-pass epilogue, so the result is the same bit for bit.
 */
sgemm_status_t sgemm(int64_t M, int64_t N, int64_t K, float alpha,
                     const float *A, int64_t lda, const float *B, int64_t ldb,
                     float beta, float *C, int64_t ldc, void *stream);

/*
 * `batch` independent products: problem b uses A + b * strideA, B + b * strideB and
 * C + b * strideC (element strides), each with the sizes and leading dimensions above.
 *   batch >= 0; strideA, strideB >= 0 (0 broadcasts one operand); strideC >= M * ldc when
 *   batch > 1 (the C matrices of different problems must not overlap).
 */
sgemm_status_t sgemm_strided_batched(int64_t M, int64_t N, int64_t K, float alpha,
                                     const float *A, int64_t lda, int64_t strideA,
                                     const float *B, int64_t ldb, int64_t strideB,
                                     float beta, float *C, int64_t ldc, int64_t strideC,
                                     int64_t batch, void *stream);

/*
 * The same operation on the tensor cores (tcgen05 MMA, accumulators in tensor memory),
 * emulating fp32 with three TF32 products. Each operand value x is split as
 * x = big + small with big = tf32_rna(x) and small = tf32_rna(x - big); the accumulators
 * receive small_A.big_B + big_A.small_B + big_A.big_B. The pages mention tensor cores (TF32
 * at twice the FP32 rate) only in passing, as the way past the SIMT kernels ("GEMM
 * scrapbook", closing remarks); the three-product split itself is not on the pages (it is the
 * published 3xTF32 method). Same arguments, errors and conventions as sgemm(), with any
 * alignment. A pre-pass writes the split operands into a per-(device, stream) workspace of
 * 16 * batch * (M + N) * K' bytes (K' = K rounded up to a multiple of 4), allocated on first
 * use and kept until sgemm_release_workspace().
 * Non-finite inputs propagate as in fp32. Accuracy: held to the same normalised error bound
 * as the SIMT path (measured at K = 16384 on N(0, 1) inputs: 3.6e-6, with the k-blocks
 * spread over two tensor-memory accumulators that the epilogue sums in fp32).
 */
sgemm_status_t sgemm_3xtf32(int64_t M, int64_t N, int64_t K, float alpha,
                            const float *A, int64_t lda, const float *B, int64_t ldb,
                            float beta, float *C, int64_t ldc, void *stream);

/* Batched form of sgemm_3xtf32; the arguments are those of sgemm_strided_batched. */
sgemm_status_t sgemm_3xtf32_strided_batched(int64_t M, int64_t N, int64_t K, float alpha,
                                            const float *A, int64_t lda, int64_t strideA,
                                            const float *B, int64_t ldb, int64_t strideB,
                                            float beta, float *C, int64_t ldc,
                                            int64_t strideC, int64_t batch, void *stream);

/*
 * The fast, lower-accuracy tensor-core mode: each operand value is rounded to TF32
 * (tf32_rna, 10 explicit mantissa bits) and one TF32 product per multiply-add accumulates in
 * fp32 tensor memory. The pages quote the TF32 tensor rate at twice the FP32 rate ("GEMM
 * scrapbook", closing remarks). Accuracy: each product is off by at most (2u + u^2)|a b| with
 * u = 2^-11, so the normalised error is bounded by about 9.8e-4 (plus fp32 accumulation),
 * not by the fp32 bound of the other entry points. Same arguments, errors and conventions as
 * sgemm(), any alignment; the rounded operands live in the same kind of per-(device, stream)
 * workspace as the 3xTF32 path (half its size).
 */
sgemm_status_t sgemm_tf32(int64_t M, int64_t N, int64_t K, float alpha,
                          const float *A, int64_t lda, const float *B, int64_t ldb,
                          float beta, float *C, int64_t ldc, void *stream);

/* Batched form of sgemm_tf32; the arguments are those of sgemm_strided_batched. */
sgemm_status_t sgemm_tf32_strided_batched(int64_t M, int64_t N, int64_t K, float alpha,
                                          const float *A, int64_t lda, int64_t strideA,
                                          const float *B, int64_t ldb, int64_t strideB,
                                          float beta, float *C, int64_t ldc,
                                          int64_t strideC, int64_t batch, void *stream);

/*
 * The same product as sgemm(), for callers that must not have the library allocate device
 * memory: an application that hands its whole memory budget to its own pool, so that a
 * cudaMalloc from a library would fail or fragment that pool; or code that cannot afford
 * the device-wide synchronisation that cudaMalloc and cudaFree may cause. The pages have no
 * counterpart for this entry point.
 *
 * It always runs the persistent stream-K kernel with 128 x 256 tiles and keeps that kernel's
 * partial sums and flags in one array compiled into the library (20 MiB of partial-sum slots
 * for up to 160 CTAs, plus 8 KiB of flags). Every GPU on which the library is loaded holds
 * this array until the process exits. It calls no cudaMalloc, cudaFree or other allocating
 * routine. A, B, C and all conventions are those of sgemm().
 *
 * Set-up: the first call on each device looks up that device's copy of the array and sets
 * the kernel's attributes; make that first call before any stream capture.
 * Sharing: every call uses the same array, which keeps the previous call's contents; each
 * call clears the flags it needs, on `stream`, before its kernel runs. Calls whose work
 * overlaps on the GPU (for example on two streams at once) race on the array and may
 * produce wrong results: order them on one stream or synchronise between them.
 * Limits: returns SGEMM_ERR_UNSUPPORTED, with a message naming the need, when its stream-K
 * schedule would use more than 160 CTAs (more scratch than the array holds), or when A or B
 * is not 16-byte aligned with lda and ldb multiples of 4.
 */
sgemm_status_t sgemm_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                             const float *A, int64_t lda, const float *B, int64_t ldb,
                             float beta, float *C, int64_t ldc, void *stream);

/*
 * C = alpha * (op(A) . op(B)) + beta * C with op(X) = X or X^T, on the chosen path. The pages
 * multiply row-major A by row-major B only ("a CUDA matmul", section 02); the transposed
 * forms are the BLAS generalisation. op(A) is M x K and op(B) is K x N; a transposed operand
 * is stored with its rows and columns swapped (A: K x M with lda >= max(1, M); B: N x K with
 * ldb >= max(1, K)). Column-major callers can use the identity C^T = B^T A^T: a column-major
 * M x N product is the row-major N x M product with A and B exchanged.
 * On the SIMT path each transposed operand is first transposed once into a per-(device,
 * stream) workspace; the TF32 paths transpose inside their split pre-pass. Arguments,
 * errors and conventions are otherwise those of sgemm() / sgemm_strided_batched(); an
 * unknown `transa`, `transb` or `path` returns SGEMM_ERR_INVALID_VALUE.
 */
sgemm_status_t sgemm_ex(sgemm_op_t transa, sgemm_op_t transb, sgemm_path_t path,
                        int64_t M, int64_t N, int64_t K, float alpha,
                        const float *A, int64_t lda, const float *B, int64_t ldb,
                        float beta, float *C, int64_t ldc, void *stream);

/* Batched form of sgemm_ex (strides as in sgemm_strided_batched, of the stored operands). */
sgemm_status_t sgemm_ex_strided_batched(sgemm_op_t transa, sgemm_op_t transb, sgemm_path_t path,
                                        int64_t M, int64_t N, int64_t K, float alpha,
                                        const float *A, int64_t lda, int64_t strideA,
                                        const float *B, int64_t ldb, int64_t strideB,
                                        float beta, float *C, int64_t ldc, int64_t strideC,
                                        int64_t batch, void *stream);

/*
 * Fused epilogue for layer-shaped products ("GEMM scrapbook": a language model is mostly
 * projections and feed-forward GEMMs; the bias, activation and residual around them are the
 * BLAS-external part fused here):
 *
 *     C = act(alpha * op(A) . op(B) + bias) + beta * C
 *
 * bias: N floats added to every row (device pointer, shared by every batch entry), or NULL.
 * act: applied after the bias and before the beta * C term, so act(x W + b) is beta = 0 and
 * x W + b + residual is act = SGEMM_ACT_NONE with beta = 1 and C holding the residual. Every
 * path, operand form and kernel applies the epilogue in registers before the single write of
 * C; when alpha == 0 or K == 0 the result is act(bias) + beta * C. Arguments and errors are
 * those of sgemm_ex / sgemm_ex_strided_batched; an unknown activation returns
 * SGEMM_ERR_INVALID_VALUE. The activations use CUDA's erff / tanhf / expf.
 */
sgemm_status_t sgemm_fused(sgemm_op_t transa, sgemm_op_t transb, sgemm_path_t path,
                           int64_t M, int64_t N, int64_t K, float alpha,
                           const float *A, int64_t lda, const float *B, int64_t ldb,
                           float beta, float *C, int64_t ldc, const float *bias,
                           sgemm_activation_t act, void *stream);

/* Batched form of sgemm_fused (one bias vector for all batch entries). */
sgemm_status_t sgemm_fused_strided_batched(sgemm_op_t transa, sgemm_op_t transb,
                                           sgemm_path_t path, int64_t M, int64_t N, int64_t K,
                                           float alpha, const float *A, int64_t lda,
                                           int64_t strideA, const float *B, int64_t ldb,
                                           int64_t strideB, float beta, float *C, int64_t ldc,
                                           int64_t strideC, int64_t batch, const float *bias,
                                           sgemm_activation_t act, void *stream);

/*
 * The product with A, B and C in HOST memory (same sizes, leading dimensions, alpha / beta
 * rules and argument errors as sgemm()). The call returns when C holds the result. B is
 * uploaded once; the rows of A (and of C when beta != 0) travel in chunks (at least M / 8
 * rows, grown until a chunk holds half a wave of tiles) through two device buffers each,
 * uploaded on an internal stream while the previous chunk is computed on `stream` (the SIMT
 * path) and the one before it is downloaded on another internal stream. The first chunk is
 * computed in K slices of growing size (256, 384, 512, ... rows of B), each starting when its
 * part of B has arrived (the slices accumulate in fp32, like stream-K pieces). With pinned (page-locked) host memory the copies
 * overlap the computation; pageable memory works but the copies then serialise. Device
 * buffers of about 4 * (K * N + 2 * chunk * (K + N)) bytes (rows padded to 16 bytes) are kept
 * per device until sgemm_release_workspace(); calls on the same device run one at a time.
 */
sgemm_status_t sgemm_host(int64_t M, int64_t N, int64_t K, float alpha,
                          const float *A, int64_t lda, const float *B, int64_t ldb,
                          float beta, float *C, int64_t ldc, void *stream);

/* Static text for a status code (never NULL). */
const char *sgemm_status_string(sgemm_status_t status);

/* Detail message for the calling thread's most recent non-OK return ("" if none). */
const char *sgemm_last_error(void);

/*
 * Synchronises `stream`, then reads and clears the device error word of the current device.
 * Returns SGEMM_ERR_TIMEOUT if a kernel's bounded wait expired since the previous call,
 * SGEMM_ERR_LAUNCH if the stream reports a CUDA error, SGEMM_OK otherwise.
 */
sgemm_status_t sgemm_device_status(void *stream);

/*
 * Failure-path self-test (diagnostic, not part of the product's arithmetic). Queues on
 * `stream` a one-thread kernel whose wait can never be satisfied: which = 0 waits on an
 * mbarrier phase no thread completes, which = 1 waits for a flag value nothing stores. The
 * wait is bounded like every wait in the library's kernels: after about 2 s the kernel raises
 * the device error word and returns, so the next sgemm_device_status(stream) returns
 * SGEMM_ERR_TIMEOUT and the CUDA context stays usable. Returns SGEMM_ERR_INVALID_VALUE for
 * another `which`.
 */
sgemm_status_t sgemm_selftest_bounded_wait(int which, void *stream);

/* Frees every workspace: stream-K and split-K partial sums, repacked and transposed operand
 * copies, TF32 split operands and the host-memory path's buffers (the next call that needs
 * one allocates it again). Synchronises the device first. */
sgemm_status_t sgemm_release_workspace(void);

/*
 * Kernel configurations (tile shape, pipeline depth, loader, tile schedule) of the SIMT
 * path. sgemm_num_configs() is the table size; sgemm_config_name(i) a static name
 * (NULL when i is out of range).
 */
int sgemm_num_configs(void);
const char *sgemm_config_name(int id);

/*
 * The configuration the dispatcher picks for these arguments (the id in the table above),
 * or -1 when no kernel would run (degenerate sizes, alpha == 0, K == 0, invalid arguments).
 * Reads no device memory.
 */
int sgemm_select_config(int64_t M, int64_t N, int64_t K, float alpha,
                        const float *A, int64_t lda, const float *B, int64_t ldb,
                        const float *C, int64_t ldc, int64_t batch);

/*
 * Forces configuration `id` for subsequent SIMT calls from every thread (-1 restores the
 * per-shape table). A forced configuration that cannot run an operand's alignment falls
 * back to the table's choice. Returns SGEMM_ERR_INVALID_VALUE for an unknown id.
 * The environment variable SGEMM_FORCE_CONFIG=<id> sets the same at load time.
 */
sgemm_status_t sgemm_force_config(int id);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_FP32_GEMM_08_GB300_SGEMM_H */
