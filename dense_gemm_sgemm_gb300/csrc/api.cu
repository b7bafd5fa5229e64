// Host side of the C ABI: argument validation, BLAS quick returns and dispatch to the
// SGEMM (CUDA-core FFMA) and HGEMM (tcgen05) launchers.  No device memory is allocated.
#include <cuda_runtime.h>

#include <mutex>

#include "gemm_internal.h"
#include "sgemm_kernel.cuh"

namespace gemm {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ok[kMaxDevices];

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

bool aligned(const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }
}  // namespace

bool current_device(DeviceInfo &info)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev_ok[dev]) {
        DeviceInfo d{};
        d.device = dev;
        int optin = 0;
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        d.smem_optin = size_t(optin);
        g_dev[dev] = d;
        g_dev_ok[dev] = true;
    }
    info = g_dev[dev];
    return true;
}

// Shared argument checks of both precisions (row-major rules of include/gemm_gb300.h).
static gemm_status_t check_common(int opA, int opB, int64_t M, int64_t N, int64_t K,
                                  const void *A, int64_t lda, const void *B, int64_t ldb,
                                  const void *C, int64_t ldc, bool need_ab)
{
    if ((opA != GEMM_OP_N && opA != GEMM_OP_T) || (opB != GEMM_OP_N && opB != GEMM_OP_T))
        return GEMM_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
    const int64_t min_lda = opA == GEMM_OP_N ? K : M;
    const int64_t min_ldb = opB == GEMM_OP_N ? N : K;
    if (lda < (min_lda > 1 ? min_lda : 1) || ldb < (min_ldb > 1 ? min_ldb : 1) ||
        ldc < (N > 1 ? N : 1))
        return GEMM_ERR_INVALID_VALUE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return GEMM_OK;
    if (C == nullptr) return GEMM_ERR_INVALID_VALUE;
    if (need_ab && (A == nullptr || B == nullptr)) return GEMM_ERR_INVALID_VALUE;
    return GEMM_OK;
}

static gemm_status_t from_cuda(cudaError_t e)
{
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

}  // namespace gemm

using namespace gemm;

namespace gemm {

// Batch rules shared by every strided-batched call: batch >= 0, strides >= 0, and the
// outputs of different problems must not overlap (strideC covers one M x N matrix).
static gemm_status_t check_batch(int64_t M, int64_t N, int64_t ldc, int64_t strideA, int64_t strideB,
                                 int64_t strideC, int64_t batch)
{
    if (batch < 0 || strideA < 0 || strideB < 0 || strideC < 0) return GEMM_ERR_INVALID_VALUE;
    if (batch > 1 && M > 0 && N > 0 && strideC < (M - 1) * ldc + N) return GEMM_ERR_INVALID_VALUE;
    if (batch > (int64_t(1) << 31)) return GEMM_ERR_UNSUPPORTED;
    return GEMM_OK;
}

static gemm_status_t sgemm_impl(int opA, int opB, int64_t M, int64_t N, int64_t K, float alpha,
                                const float *A, int64_t lda, int64_t strideA, const float *B,
                                int64_t ldb, int64_t strideB, float beta, float *C, int64_t ldc,
                                int64_t strideC, int64_t batch, void *stream)
{
    const bool need_ab = K > 0 && alpha != 0.0f;
    gemm_status_t s = check_common(opA, opB, M, N, K, A, lda, B, ldb, C, ldc, need_ab);
    if (s != GEMM_OK) return s;
    s = check_batch(M, N, ldc, strideA, strideB, strideC, batch);
    if (s != GEMM_OK || M == 0 || N == 0 || batch == 0) return s;
    if (!aligned(C, 4) || (need_ab && (!aligned(A, 4) || !aligned(B, 4))))
        return GEMM_ERR_MISALIGNED;
    DeviceInfo dev;
    if (!current_device(dev) || dev.cc_major != 10 || dev.cc_minor != 3) return GEMM_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!need_ab) {
        if (beta == 1.0f) return GEMM_OK;
        return from_cuda(launch_scale_batched(M, N, beta, C, ldc, strideC, batch, st));
    }
    return from_cuda(launch_sgemm(dev, opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C,
                                  ldc, strideC, batch, st));
}

static gemm_status_t tc_impl(int dtype, int opA, int opB, int64_t M, int64_t N, int64_t K, float alpha,
                             const uint16_t *A, int64_t lda, int64_t strideA, const uint16_t *B,
                             int64_t ldb, int64_t strideB, float beta, float *C, int64_t ldc,
                             int64_t strideC, int64_t batch, void *stream)
{
    const bool need_ab = K > 0 && alpha != 0.0f;
    gemm_status_t s = check_common(opA, opB, M, N, K, A, lda, B, ldb, C, ldc, need_ab);
    if (s != GEMM_OK) return s;
    s = check_batch(M, N, ldc, strideA, strideB, strideC, batch);
    if (s != GEMM_OK || M == 0 || N == 0 || batch == 0) return s;
    if (!aligned(C, 4)) return GEMM_ERR_MISALIGNED;
    if (need_ab && (!aligned(A, 2) || !aligned(B, 2))) return GEMM_ERR_MISALIGNED;
    if (need_ab && (lda > (int64_t(1) << 35) || ldb > (int64_t(1) << 35) || strideA > (int64_t(1) << 38) ||
                    strideB > (int64_t(1) << 38)))
        return GEMM_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if (!current_device(dev) || dev.cc_major != 10 || dev.cc_minor != 3) return GEMM_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!need_ab) {
        if (beta == 1.0f) return GEMM_OK;
        return from_cuda(launch_scale_batched(M, N, beta, C, ldc, strideC, batch, st));
    }
    // Operands the tensor-memory-access unit cannot read (base not 16-byte aligned, leading
    // dimension or batch stride not a multiple of 8 elements) are read by the kernel's loader
    // warps instead, in the same launch.
    return launch_hgemm(dev, dtype, opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
                        strideC, batch, st);
}

// Matrices in host memory: each operand is staged on the device with the caller's leading
// dimension, so it moves as one contiguous copy (a pitched host-to-device copy of rows this
// short runs several times slower); then the device path runs on the staged matrices and C
// comes back, only its M x N elements (a pitched copy when ldc > N leaves the row padding
// of the caller's C untouched).  Everything is ordered on `stream`.
template <class T, class DeviceCall>
static gemm_status_t host_impl(int opA, int opB, int64_t M, int64_t N, int64_t K, float alpha,
                               const T *A, int64_t lda, const T *B, int64_t ldb, float beta,
                               float *C, int64_t ldc, void *stream, DeviceCall device_call)
{
    const bool need_ab = K > 0 && alpha != 0.0f;
    gemm_status_t s = check_common(opA, opB, M, N, K, A, lda, B, ldb, C, ldc, need_ab);
    if (s != GEMM_OK || M == 0 || N == 0) return s;
    // Elements a rows x cols matrix with leading dimension ld spans; -1 when too large.
    constexpr int64_t kMaxElems = int64_t(1) << 40;
    auto extent = [](int64_t rows, int64_t cols, int64_t ld) -> int64_t {
        if (rows == 0 || cols == 0) return 0;
        if (ld > 0 && rows - 1 > (kMaxElems - cols) / ld) return -1;
        return (rows - 1) * ld + cols;
    };
    const int64_t nA = need_ab ? extent(opA == GEMM_OP_N ? M : K, opA == GEMM_OP_N ? K : M, lda) : 0;
    const int64_t nB = need_ab ? extent(opB == GEMM_OP_N ? K : N, opB == GEMM_OP_N ? N : K, ldb) : 0;
    const int64_t nC = extent(M, N, ldc);
    if (nA < 0 || nB < 0 || nC < 0) return GEMM_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if (!current_device(dev) || dev.cc_major != 10 || dev.cc_minor != 3) return GEMM_ERR_NO_DEVICE;
    auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
    const size_t bA = up(size_t(nA) * sizeof(T)), bB = up(size_t(nB) * sizeof(T));
    const size_t bC = up(size_t(nC) * sizeof(float));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // held until this call's copies and kernels are enqueued (see host_staging)
    std::lock_guard<std::mutex> lk(host_call_mutex());
    char *base = static_cast<char *>(host_staging(dev.device, st, bA + bB + bC));
    if (base == nullptr) return GEMM_ERR_UNSUPPORTED;
    T *dA = reinterpret_cast<T *>(base), *dB = reinterpret_cast<T *>(base + bA);
    float *dC = reinterpret_cast<float *>(base + bA + bB);
    if ((nA > 0 && cudaMemcpyAsync(dA, A, size_t(nA) * sizeof(T), cudaMemcpyDefault, st) != cudaSuccess) ||
        (nB > 0 && cudaMemcpyAsync(dB, B, size_t(nB) * sizeof(T), cudaMemcpyDefault, st) != cudaSuccess) ||
        (beta != 0.0f && cudaMemcpyAsync(dC, C, size_t(nC) * sizeof(float), cudaMemcpyDefault, st) != cudaSuccess)) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    s = device_call(need_ab ? dA : nullptr, need_ab ? dB : nullptr, dC, st);
    if (s != GEMM_OK) return s;
    const cudaError_t e =
        ldc == N ? cudaMemcpyAsync(C, dC, size_t(M) * size_t(N) * sizeof(float), cudaMemcpyDefault, st)
                 : cudaMemcpy2DAsync(C, size_t(ldc) * sizeof(float), dC, size_t(ldc) * sizeof(float),
                                     size_t(N) * sizeof(float), size_t(M), cudaMemcpyDefault, st);
    if (e != cudaSuccess) cudaGetLastError();
    return from_cuda(e);
}

}  // namespace gemm

extern "C" {

gemm_status_t gemm_sgemm_f32_host(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N, int64_t K,
                                  float alpha, const float *A, int64_t lda, const float *B,
                                  int64_t ldb, float beta, float *C, int64_t ldc, void *stream)
{
    return host_impl(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream,
                     [&](const float *dA, const float *dB, float *dC, cudaStream_t st) {
                         return sgemm_impl(opA, opB, M, N, K, alpha, dA, lda, 0, dB, ldb, 0, beta, dC, ldc,
                                           0, 1, st);
                     });
}

gemm_status_t gemm_hgemm_f16f32_host(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                     int64_t K, float alpha, const uint16_t *A, int64_t lda,
                                     const uint16_t *B, int64_t ldb, float beta, float *C,
                                     int64_t ldc, void *stream)
{
    return host_impl(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream,
                     [&](const uint16_t *dA, const uint16_t *dB, float *dC, cudaStream_t st) {
                         return tc_impl(kInF16, opA, opB, M, N, K, alpha, dA, lda, 0, dB, ldb, 0, beta,
                                        dC, ldc, 0, 1, st);
                     });
}

gemm_status_t gemm_bgemm_bf16f32_host(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                      int64_t K, float alpha, const uint16_t *A, int64_t lda,
                                      const uint16_t *B, int64_t ldb, float beta, float *C,
                                      int64_t ldc, void *stream)
{
    return host_impl(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream,
                     [&](const uint16_t *dA, const uint16_t *dB, float *dC, cudaStream_t st) {
                         return tc_impl(kInBf16, opA, opB, M, N, K, alpha, dA, lda, 0, dB, ldb, 0, beta,
                                        dC, ldc, 0, 1, st);
                     });
}

gemm_status_t gemm_sgemm_f32(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N, int64_t K,
                             float alpha, const float *A, int64_t lda, const float *B,
                             int64_t ldb, float beta, float *C, int64_t ldc, void *stream)
{
    return sgemm_impl(opA, opB, M, N, K, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc, 0, 1, stream);
}

gemm_status_t gemm_sgemm_f32_strided_batched(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                             int64_t K, float alpha, const float *A, int64_t lda,
                                             int64_t strideA, const float *B, int64_t ldb,
                                             int64_t strideB, float beta, float *C, int64_t ldc,
                                             int64_t strideC, int64_t batch, void *stream)
{
    return sgemm_impl(opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc, strideC,
                      batch, stream);
}

gemm_status_t gemm_hgemm_f16f32(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                int64_t K, float alpha, const uint16_t *A, int64_t lda,
                                const uint16_t *B, int64_t ldb, float beta, float *C,
                                int64_t ldc, void *stream)
{
    return tc_impl(kInF16, opA, opB, M, N, K, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc, 0, 1, stream);
}

gemm_status_t gemm_hgemm_f16f32_strided_batched(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                                int64_t K, float alpha, const uint16_t *A, int64_t lda,
                                                int64_t strideA, const uint16_t *B, int64_t ldb,
                                                int64_t strideB, float beta, float *C, int64_t ldc,
                                                int64_t strideC, int64_t batch, void *stream)
{
    return tc_impl(kInF16, opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc, strideC,
                   batch, stream);
}

gemm_status_t gemm_bgemm_bf16f32(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N, int64_t K,
                                 float alpha, const uint16_t *A, int64_t lda, const uint16_t *B,
                                 int64_t ldb, float beta, float *C, int64_t ldc, void *stream)
{
    return tc_impl(kInBf16, opA, opB, M, N, K, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc, 0, 1, stream);
}

gemm_status_t gemm_bgemm_bf16f32_strided_batched(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                                 int64_t K, float alpha, const uint16_t *A, int64_t lda,
                                                 int64_t strideA, const uint16_t *B, int64_t ldb,
                                                 int64_t strideB, float beta, float *C, int64_t ldc,
                                                 int64_t strideC, int64_t batch, void *stream)
{
    return tc_impl(kInBf16, opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
                   strideC, batch, stream);
}

gemm_status_t gemm_get_device_status(void *stream)
{
    DeviceInfo dev;
    if (!current_device(dev)) return GEMM_ERR_NO_DEVICE;
    return read_and_clear_device_status(static_cast<cudaStream_t>(stream));
}

const char *gemm_status_string(gemm_status_t status)
{
    switch (status) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_VALUE: return "GEMM_ERR_INVALID_VALUE: bad size, op, leading dimension or pointer";
    case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED: pointer or leading dimension breaks the alignment rule";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED: size beyond the library limits";
    case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH: the CUDA runtime refused the launch";
    case GEMM_ERR_DEVICE_TIMEOUT: return "GEMM_ERR_DEVICE_TIMEOUT: a kernel gave up on a bounded barrier wait";
    case GEMM_ERR_NO_DEVICE: return "GEMM_ERR_NO_DEVICE: no usable sm_103 device is current";
    }
    return "unknown gemm_status_t";
}

int gemm_version(void) { return 100; }

uint64_t gemm_kernel_launches(void) { return gemm::launches_so_far(); }

gemm_status_t gemm_sgemm_config(int index, gemm_sgemm_config_t *out)
{
    if (out == nullptr) return GEMM_ERR_INVALID_VALUE;
    auto fill = [out](char name, auto cfg) {
        using C = decltype(cfg);
        *out = gemm_sgemm_config_t{name, C::BM, C::BN, C::BK, C::TM, C::TN, C::STAGES, sg::kThreads,
                                   C::MIN_BLOCKS, C::PAD, C::SMEM_BYTES};
        return GEMM_OK;
    };
    switch (index) {
    case 0: return fill('L', sg::CfgL{});
    case 1: return fill('M', sg::CfgM{});
    case 2: return fill('S', sg::CfgS{});
    default: return GEMM_ERR_INVALID_VALUE;
    }
}

gemm_status_t gemm_tile_raster(int64_t t, int64_t tiles_m, int64_t tiles_n, int log_group,
                               int64_t *tile_m, int64_t *tile_n)
{
    if (tile_m == nullptr || tile_n == nullptr || tiles_m <= 0 || tiles_n <= 0 ||
        log_group < 0 || log_group > 16 || t < 0 || t >= tiles_m * tiles_n)
        return GEMM_ERR_INVALID_VALUE;
    int64_t tm = 0, tn = 0;
    raster(t, tiles_m, tiles_n, log_group, tm, tn);
    *tile_m = tm;
    *tile_n = tn;
    return GEMM_OK;
}

}  // extern "C"
