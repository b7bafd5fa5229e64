/*
 * gemm_gb300.h -- C ABI of a GEMM library for one NVIDIA GB300 GPU (sm_103a).
 *
 * Every entry point computes the general matrix product of the copecc.github.io "GEMM"
 * page (section "核心问题与运算特征"):
 *
 *     C = alpha * op(A) * op(B) + beta * C          op(A): M x K, op(B): K x N, C: M x N
 *
 * with each C[i][j] the dot product of row i of op(A) and column j of op(B) (the same
 * section; also yekq.top "LeetGPU 第二题", section "题目描述").
 *
 * Layout.  All matrices are ROW-MAJOR.  A leading dimension is the element distance
 * between the first elements of two consecutive stored rows, and may exceed the logical
 * row length when rows are padded (copecc "GEMM" page, section "Leading Dimension (lda,
 * ldb, ldc)").  The transpose flags choose how a buffer is read (the role the op
 * arguments play in cublasSgemm on the ssxxe.cn page, section "三、cuBLAS 实现方式探究",
 * restated for row-major storage):
 *     opA = GEMM_OP_N: A stored M x K, op(A)[i][k] = A[i*lda + k], lda >= max(1, K)
 *     opA = GEMM_OP_T: A stored K x M, op(A)[i][k] = A[k*lda + i], lda >= max(1, M)
 *     opB = GEMM_OP_N: B stored K x N, op(B)[k][j] = B[k*ldb + j], ldb >= max(1, N)
 *     opB = GEMM_OP_T: B stored N x K, op(B)[k][j] = B[j*ldb + k], ldb >= max(1, K)
 *     C stored M x N, C[i][j] at C[i*ldc + j], ldc >= max(1, N)
 *
 * Ownership.  A, B and C are device memory owned by the caller (host memory for the
 * *_host entry points); the library never frees or retains them.  C must not overlap A or
 * B.  The library keeps scratch per (device, stream): a split-K workspace (64 MB and 8192
 * counters), two buffers for transposed fp32 operands and, for the *_host entry points, a
 * staging area; each is allocated when first needed, grown when a larger problem needs it
 * (after the stream's earlier work), kept until exit, and never allocated while the stream
 * is being captured (a call then takes a path that needs no new scratch, except where host
 * matrices must be staged).  At most 16 streams per device hold each kind: calls on further
 * streams run without split-K or transposition (same results within the stated bounds,
 * slower), and a *_host call on a further stream first synchronises the device and releases
 * the other streams' staging areas.  The *_host calls enqueue their work one host thread at
 * a time.
 *
 * Asynchrony.  A call validates its arguments on the host, launches on `stream` (a
 * cudaStream_t passed as void*; NULL means the legacy default stream of the current
 * device) and returns without waiting.  The return value reports argument errors and
 * launch errors only; gemm_get_device_status() reports errors raised inside a kernel.
 * Nothing aborts or exits the process.
 *
 * BLAS conventions.  M == 0 or N == 0: nothing is launched and GEMM_OK is returned.
 * K == 0 or alpha == 0: C = beta * C.  beta == 0: C is written without being read, so
 * NaN or Inf already in C does not propagate.  alpha and beta are host values.
 *
 * Thread safety.  Calls may come from several host threads.  Calls on one stream from
 * different threads must not overlap in time (a call may grow that stream's scratch while
 * the other enqueues work that uses it); calls that write the same C concurrently race, as
 * with any BLAS.
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stdint.h>

/* Symbols of this header are the only ones the shared library exports. */
#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { GEMM_OP_N = 0, GEMM_OP_T = 1 } gemm_op_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1,  /* bad size, op, leading dimension or NULL pointer */
    GEMM_ERR_MISALIGNED = 2,     /* pointer or leading dimension breaks the alignment rule */
    GEMM_ERR_UNSUPPORTED = 3,    /* size beyond the library's limits (see each call) */
    GEMM_ERR_LAUNCH = 4,         /* the CUDA runtime refused the launch */
    GEMM_ERR_DEVICE_TIMEOUT = 5, /* a kernel gave up waiting on a barrier (bounded wait) */
    GEMM_ERR_NO_DEVICE = 6       /* no usable sm_103 device is current */
} gemm_status_t;

/*
 * Strict-FP32 GEMM (SGEMM) on the CUDA cores: every product and sum is an IEEE fp32
 * fused multiply-add, never TF32 and never a reduced-precision tensor operation.
 * A, B, C: 4-byte aligned fp32 device pointers; any leading dimension is accepted (the
 * 16-byte vector paths are used only where pointer and leading dimension allow them).
 * Above 1e10 flops, an operand whose rows run along K (op(A) = N, op(B) = T) may first be
 * transposed into this stream's scratch buffer (8 bytes of traffic per element) so that
 * the kernel reads it with 16-byte copies; the result does not depend on it.
 * Limits: M, N, K < 2^31.
 */
GEMM_API gemm_status_t gemm_sgemm_f32(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N, int64_t K,
                             float alpha, const float *A, int64_t lda, const float *B,
                             int64_t ldb, float beta, float *C, int64_t ldc, void *stream);

/*
 * fp16-input GEMM with fp32 accumulation and fp32 output on the tcgen05 tensor cores
 * (the mixed-precision mode of the copecc "GEMM" page, section "Batched 执行与混合精度", and
 * of the dandandamowang.xyz "GEMM优化（二）" page): products of IEEE binary16 inputs are
 * summed in fp32, then C = alpha * sum + beta * C in fp32.
 * A, B: IEEE binary16 bit patterns (uint16_t), 2-byte aligned, any lda, ldb; an odd byte
 * address gives GEMM_ERR_MISALIGNED.  The tensor-memory-access unit reads rows only from a
 * 16-byte aligned base with a leading dimension that is a multiple of 8 elements; an operand
 * laid out otherwise is read by loader warps of the same kernel instead (each row copied as
 * the aligned 16-byte blocks that cover it, then shifted into place in shared memory; rows
 * at the ends of the operand's storage or cut by the matrix edge element by element), with
 * no extra launch and no scratch memory, at a fraction of the TMA path's rate.
 * C: fp32, 4-byte aligned, any ldc.
 * Limits: M, N, K < 2^31; lda, ldb < 2^35 elements.
 */
GEMM_API gemm_status_t gemm_hgemm_f16f32(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                int64_t K, float alpha, const uint16_t *A, int64_t lda,
                                const uint16_t *B, int64_t ldb, float beta, float *C,
                                int64_t ldc, void *stream);

/*
 * bfloat16-input GEMM with fp32 accumulation and fp32 output on the tcgen05 tensor cores:
 * the BF16 case of the mixed-precision mode of the copecc "GEMM" page, section "Batched 执行与
 * 混合精度" (FP16/BF16 inputs, FP32 accumulation).  Same rules as gemm_hgemm_f16f32, with
 * A and B holding bfloat16 bit patterns (the upper halves of IEEE binary32 values).
 */
GEMM_API gemm_status_t gemm_bgemm_bf16f32(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                          int64_t K, float alpha, const uint16_t *A, int64_t lda,
                                          const uint16_t *B, int64_t ldb, float beta, float *C,
                                          int64_t ldc, void *stream);

/*
 * Strided-batched forms (copecc "GEMM" page, section "Batched 执行与混合精度": one call runs
 * `batch` GEMMs of the same M, N, K whose operands sit strideA, strideB and strideC elements
 * apart).  Problem b computes
 *     C_b = alpha * op(A_b) * op(B_b) + beta * C_b,   X_b = X + b * strideX,
 * with the row-major rules of the single calls.  A stride of 0 shares that operand between
 * all problems; strideC must keep the outputs apart: strideC >= (M - 1) * ldc + N when
 * batch > 1 (else GEMM_ERR_INVALID_VALUE).  batch == 0 launches nothing.  A 16-bit
 * operand whose batch stride is not a multiple of 8 elements is read by the loader warps,
 * like one with an unaligned leading dimension (see gemm_hgemm_f16f32).
 * Limits: batch <= 2^31.
 */
GEMM_API gemm_status_t gemm_sgemm_f32_strided_batched(gemm_op_t opA, gemm_op_t opB, int64_t M,
                                                      int64_t N, int64_t K, float alpha,
                                                      const float *A, int64_t lda, int64_t strideA,
                                                      const float *B, int64_t ldb, int64_t strideB,
                                                      float beta, float *C, int64_t ldc,
                                                      int64_t strideC, int64_t batch, void *stream);

GEMM_API gemm_status_t gemm_hgemm_f16f32_strided_batched(gemm_op_t opA, gemm_op_t opB, int64_t M,
                                                         int64_t N, int64_t K, float alpha,
                                                         const uint16_t *A, int64_t lda,
                                                         int64_t strideA, const uint16_t *B,
                                                         int64_t ldb, int64_t strideB, float beta,
                                                         float *C, int64_t ldc, int64_t strideC,
                                                         int64_t batch, void *stream);

GEMM_API gemm_status_t gemm_bgemm_bf16f32_strided_batched(gemm_op_t opA, gemm_op_t opB, int64_t M,
                                                          int64_t N, int64_t K, float alpha,
                                                          const uint16_t *A, int64_t lda,
                                                          int64_t strideA, const uint16_t *B,
                                                          int64_t ldb, int64_t strideB, float beta,
                                                          float *C, int64_t ldc, int64_t strideC,
                                                          int64_t batch, void *stream);

/*
 * The three products on matrices in HOST memory: same arguments, layouts, leading-dimension
 * rules, results and errors as gemm_sgemm_f32, gemm_hgemm_f16f32 and gemm_bgemm_bf16f32,
 * but A, B and C are host pointers (page-locked, from cudaHostAlloc / cudaHostRegister /
 * torch pin_memory, for the call to stay asynchronous; pageable memory works too, with the
 * copies then synchronising as cudaMemcpyAsync does for it).  The source pages have no
 * counterpart: they copy operands in and results out around the kernel by hand.
 *
 * In order on `stream`, the call copies each stored operand -- and C when beta != 0 -- to a
 * device staging area of this (device, stream) pair as one contiguous copy that keeps the
 * caller's leading dimension, runs the device GEMM there, and copies the M x N elements of
 * C back into the caller's C (the row padding of an ldc > N matrix is neither read when
 * beta == 0 nor ever written).  It returns after enqueueing: A, B and C must stay alive and
 * unchanged until the stream has passed the call (cudaStreamSynchronize, or an event), and
 * C holds the result only then.  Calls on different streams overlap on the GPU (the copies
 * of one with the GEMM of another); calls on one stream run one after the other.
 *
 * The staging area is allocated by the first call on a stream and reallocated -- after
 * synchronising that stream -- when a larger problem arrives; it is kept until the process
 * exits (see Thread safety above for calls sharing a stream).  Returns GEMM_ERR_UNSUPPORTED without enqueueing anything when the area would have
 * to be (re)allocated while the stream is being captured, when device memory for it cannot
 * be had, or when a matrix spans more than 2^40 elements; GEMM_ERR_LAUNCH when a copy
 * cannot be enqueued (after the input copies, C may then be partly written or not at all).
 */
GEMM_API gemm_status_t gemm_sgemm_f32_host(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                           int64_t K, float alpha, const float *A, int64_t lda,
                                           const float *B, int64_t ldb, float beta, float *C,
                                           int64_t ldc, void *stream);
GEMM_API gemm_status_t gemm_hgemm_f16f32_host(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                              int64_t K, float alpha, const uint16_t *A, int64_t lda,
                                              const uint16_t *B, int64_t ldb, float beta, float *C,
                                              int64_t ldc, void *stream);
GEMM_API gemm_status_t gemm_bgemm_bf16f32_host(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                               int64_t K, float alpha, const uint16_t *A, int64_t lda,
                                               const uint16_t *B, int64_t ldb, float beta, float *C,
                                               int64_t ldc, void *stream);

/*
 * Allocation-free variant of gemm_sgemm_f32, for callers that must not allocate device
 * memory while they run: a framework whose own allocator owns the device memory and
 * forbids other cudaMalloc calls, or a latency-critical caller that cannot afford the
 * blocking, device-wide synchronisation or late failure of an allocation.  The source
 * pages have no counterpart to this entry point.
 *
 * Same arguments, rules and result as gemm_sgemm_f32 (strict FP32, row-major, caller-owned
 * A, B, C), computed by the split-K kernel (64 x 64 tiles, K split over up to 16 CTAs whose
 * partial tiles are added in a fixed order).  Its scratch -- arrival counters and partial
 * tiles -- lives in one statically sized device array of 16 MiB + 16 KiB that the library
 * holds on every GPU that loads it, until the process exits; the call itself never calls
 * cudaMalloc, cudaFree or any allocating routine.
 *
 * The K split count S is reduced until the split's scratch fits the array: at most 4096
 * tiles of 64 x 64 and tiles * S <= 1024 partial tiles.  S = 1 uses no scratch, so problems
 * too large to split still run (unsplit).
 * Limits: M, N, K < 2^31; larger sizes return GEMM_ERR_UNSUPPORTED without launching anything.
 * The first call on a device looks up the device address of the scratch array (with that
 * device current); make that first call before capturing the stream into a graph.
 * Every call shares the one array, whose contents persist between calls: the call clears
 * the counters it needs on `stream` before its kernel, but two calls whose work overlaps on
 * the GPU (e.g. on different streams) race on the array and corrupt each other's results.
 */
GEMM_API gemm_status_t gemm_sgemm_f32_noalloc(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                              int64_t K, float alpha, const float *A, int64_t lda,
                                              const float *B, int64_t ldb, float beta, float *C,
                                              int64_t ldc, void *stream);

/*
 * Waits for `stream`, then returns and clears the error word that kernels of this library
 * set on the current device when a bounded barrier wait expires (GEMM_ERR_DEVICE_TIMEOUT),
 * or GEMM_OK.  A kernel that sets the word leaves its output tile unwritten.  After a
 * timeout it also synchronises every stream of the current device that owns a split-K
 * workspace and zeroes that workspace's arrival counters, which an abandoned wait may have
 * left raised.
 */
GEMM_API gemm_status_t gemm_get_device_status(void *stream);

/* Static, human-readable name of a status code. */
GEMM_API const char *gemm_status_string(gemm_status_t status);

/* Library version as 10000 * major + 100 * minor + patch. */
GEMM_API int gemm_version(void);

/*
 * Number of kernels this process has launched through the library so far, on every device
 * and stream (GEMM kernels and the operand re-layout and scaling kernels).  For accounting:
 * the difference across a region counts the library's launches in it.  Needs no GPU.
 */
GEMM_API uint64_t gemm_kernel_launches(void);

/*
 * Measured FP32 fused multiply-add throughput of the current device, in TFLOP/s (2 flops
 * per multiply-add), written to *tflops: the strict-FP32 path's roofline denominator, next
 * to the figure derived from SM count x 128 FP32 lanes x 2 x clock.  A kernel of
 * independent packed multiply-add chains (fma.rn.f32x2) fills every SM; one untimed launch,
 * then the best of three launches timed with CUDA events on `stream` (synchronises it;
 * about a millisecond of GPU time).  Returns GEMM_ERR_INVALID_VALUE for a NULL output,
 * GEMM_ERR_NO_DEVICE without a current device, GEMM_ERR_LAUNCH when a launch or an event
 * fails (then *tflops is 0).
 */
GEMM_API gemm_status_t gemm_measure_fp32_fma_peak(void *stream, double *tflops);

/*
 * The tile configurations of the strict-FP32 path (a host function: needs no GPU), for
 * tools and tests.  Configuration `index` (0, 1, ... in the order the planner considers
 * them) is written to *out: its one-letter name, block tile BM x BN, K slice BK, thread tile
 * TM x TN, ring stages, threads per CTA, the CTAs per SM it is compiled for, the padding of
 * each [k][x] stage row in floats (0: XOR-swizzled rows), and its dynamic shared memory,
 * STAGES * BK * (BM + BN + 2 * pad) * 4 bytes -- the footprint arithmetic of the ssxxe.cn
 * GEMM page, section "2.1 矩阵分块利用Shared Memory", BK * (BM + BN) * 4 bytes per stage,
 * plus the padding.  Returns GEMM_ERR_INVALID_VALUE for an index past the last
 * configuration or a NULL output.
 */
typedef struct {
    char name;
    int bm, bn, bk, tm, tn, stages, threads, ctas_per_sm, row_pad, smem_bytes;
} gemm_sgemm_config_t;
GEMM_API gemm_status_t gemm_sgemm_config(int index, gemm_sgemm_config_t *out);

/*
 * Tile raster used by the kernels (a host function: needs no GPU).  It maps the t-th tile
 * of a tiles_m x tiles_n grid of output tiles to (tile_m, tile_n) so that consecutive
 * tiles sweep a group of 2^log_group tile rows column by column, which keeps the operand
 * tiles they share resident in L2 (copecc "GEMM" page, section "线程块网格重排 (Thread Block
 * Swizzling)"; with tiles_m = 2^log_group this is exactly that section's mapping).  The
 * last group may be shorter.  Returns GEMM_ERR_INVALID_VALUE for t outside the grid,
 * non-positive grid sizes, log_group outside [0, 16] or NULL outputs.
 */
GEMM_API gemm_status_t gemm_tile_raster(int64_t t, int64_t tiles_m, int64_t tiles_n, int log_group,
                               int64_t *tile_m, int64_t *tile_n);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
