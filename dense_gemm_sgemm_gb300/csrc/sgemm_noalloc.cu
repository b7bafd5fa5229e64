// gemm_sgemm_f32_noalloc: the split-K SGEMM with its scratch in a fixed, statically sized
// device array instead of memory obtained from cudaMalloc.
//
// Who needs it: code that may not allocate device memory at call time -- for example a
// host framework whose own allocator owns all device memory and forbids any other
// cudaMalloc, or a real-time or safety-critical caller that must never hit an allocation
// (cudaMalloc can block, synchronise the device, or fail when memory is fragmented).
// gemm_sgemm_f32 allocates its split-K workspace once per stream on first use; this entry
// point never calls cudaMalloc, cudaFree or any other allocating routine.
//
// The price: the scratch array below exists on every GPU that loads this library, for as
// long as the process lives, and bounds how far a problem's K is split (a problem too large
// to split within it runs unsplit, which needs no scratch).
#include <cuda_runtime.h>

#include <mutex>

#include "sgemm_kernel.cuh"

namespace gemm {
namespace {

using namespace sg;

// Scratch layout: kNoallocCounters arrival counters (one per 64 x 64 tile), then the partial
// tiles (splits x tiles x 64 x 64 fp32).
constexpr int kNoallocCounters = 4096;
constexpr size_t kNoallocCounterBytes = size_t(kNoallocCounters) * sizeof(unsigned int);
constexpr size_t kNoallocPartialBytes = size_t(16) << 20;  // 16 MiB = 1024 partial tiles
constexpr size_t kNoallocScratchBytes = kNoallocCounterBytes + kNoallocPartialBytes;
constexpr size_t kTileBytes = size_t(CfgS::BM) * CfgS::BN * sizeof(float);

static __device__ __align__(256) unsigned char g_sgemm_noalloc_scratch[kNoallocScratchBytes];

// Device address of the scratch array on each device.  In host code the symbol is only a
// stand-in, so the address is looked up once per device, with that device current.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_have[kMaxDevices];
unsigned char *g_addr[kMaxDevices];

bool scratch_address(int dev, unsigned char **out)
{
    if (dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_have[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_sgemm_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return false;
        }
        g_addr[dev] = static_cast<unsigned char *>(ptr);
        g_have[dev] = true;
    }
    *out = g_addr[dev];
    return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace gemm

using namespace gemm;

extern "C" GEMM_API gemm_status_t gemm_sgemm_f32_noalloc(gemm_op_t opA, gemm_op_t opB, int64_t M,
                                                         int64_t N, int64_t K, float alpha,
                                                         const float *A, int64_t lda, const float *B,
                                                         int64_t ldb, float beta, float *C,
                                                         int64_t ldc, void *stream)
{
    // Argument rules are those of gemm_sgemm_f32.
    if ((opA != GEMM_OP_N && opA != GEMM_OP_T) || (opB != GEMM_OP_N && opB != GEMM_OP_T))
        return GEMM_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
    const int64_t min_lda = opA == GEMM_OP_N ? K : M, min_ldb = opB == GEMM_OP_N ? N : K;
    if (lda < (min_lda > 1 ? min_lda : 1) || ldb < (min_ldb > 1 ? min_ldb : 1) || ldc < (N > 1 ? N : 1))
        return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return GEMM_OK;
    if (C == nullptr) return GEMM_ERR_INVALID_VALUE;
    if (M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff) return GEMM_ERR_UNSUPPORTED;
    if (K == 0 || alpha == 0.0f) {
        // No product: C = beta * C, which needs no scratch.
        if (reinterpret_cast<uintptr_t>(C) & 3u) return GEMM_ERR_MISALIGNED;
        DeviceInfo dev;
        if (!current_device(dev) || dev.cc_major != 10 || dev.cc_minor != 3) return GEMM_ERR_NO_DEVICE;
        if (beta == 1.0f) return GEMM_OK;
        return launch_scale(M, N, beta, C, ldc, static_cast<cudaStream_t>(stream)) == cudaSuccess
                   ? GEMM_OK : GEMM_ERR_LAUNCH;
    }
    if (A == nullptr || B == nullptr) return GEMM_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 3u)
        return GEMM_ERR_MISALIGNED;

    // Grid of 64 x 64 tiles and K splits: enough splits to fill one wave of three CTAs per
    // SM, at most 16, at least two 16-wide K slices each.  A split count above one needs an
    // arrival counter per tile and a partial tile per split and tile in the scratch array;
    // where they would not fit, fewer splits are taken, down to one, which uses no scratch.
    const int64_t tiles_m = (M + CfgS::BM - 1) / CfgS::BM, tiles_n = (N + CfgS::BN - 1) / CfgS::BN;
    const int64_t tiles = tiles_m * tiles_n;
    const int64_t KT = (K + CfgS::BK - 1) / CfgS::BK;
    DeviceInfo dev;
    if (!current_device(dev) || dev.cc_major != 10 || dev.cc_minor != 3) return GEMM_ERR_NO_DEVICE;
    const int64_t target = int64_t(dev.num_sms) * CfgS::MIN_BLOCKS;
    int64_t S = (target + tiles / 2) / tiles;
    S = S < 1 ? 1 : (S > 16 ? 16 : S);
    while (S > 1 && (KT / S < 2 || tiles > kNoallocCounters ||
                     size_t(tiles) * S * kTileBytes > kNoallocPartialBytes))
        --S;

    // The address lookup is the per-device set-up of the first call, split or not.
    unsigned char *scratch = nullptr;
    if (!scratch_address(dev.device, &scratch)) return GEMM_ERR_LAUNCH;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents; the arrival counters must start at zero.
    if (S > 1 && cudaMemsetAsync(scratch, 0, size_t(tiles) * sizeof(unsigned int), st) != cudaSuccess)
        return GEMM_ERR_LAUNCH;

    SgemmParams p{};
    p.M = M; p.N = N; p.K = K;
    p.A = A; p.lda = lda; p.B = B; p.ldb = ldb; p.C = C; p.ldc = ldc;
    p.alpha = alpha; p.beta = beta;
    p.log_group = 3;
    p.batch = 1;
    p.c_vec = aligned16(C) && (ldc % 4) == 0;
    p.tiles_m = tiles_m;
    p.tiles_n = tiles_n;
    p.splits = static_cast<int>(S);
    p.kt_per_split = static_cast<int>((KT + S - 1) / S);
    p.counters = reinterpret_cast<unsigned int *>(scratch);
    p.ws = reinterpret_cast<float *>(scratch + kNoallocCounterBytes);
    const bool a_vec = aligned16(A) && lda % 4 == 0, b_vec = aligned16(B) && ldb % 4 == 0;
    const int a_mode = opA == GEMM_OP_N ? (a_vec ? kKVec : kKT) : (a_vec ? kMnVec : kMnScalar);
    const int b_mode = opB == GEMM_OP_T ? kKT : (b_vec ? kMnVec : kMnScalar);
    return launch_SS(dev.device, a_mode, b_mode, p, st) == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}
