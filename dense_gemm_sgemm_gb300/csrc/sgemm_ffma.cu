// Strict-FP32 SGEMM: host-side planning (tile configuration, split-K, workspace) and the
// beta-only kernel.  The kernel template is in sgemm_kernel.cuh; each tile configuration is
// compiled in its own sgemm_cfg_*.cu.
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "sgemm_kernel.cuh"

namespace gemm {
namespace {

using namespace sg;

__global__ void scale_kernel(int64_t M, int64_t N, float beta, float *__restrict__ C, int64_t ldc)
{
    const int64_t total = M * N;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = e / N, j = e % N;
        float *c = C + i * ldc + j;
        *c = beta == 0.0f ? 0.0f : beta * *c;
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- split-K planning
constexpr size_t kWsBytes = kWorkspaceBytes;
constexpr size_t kWsCounters = kWorkspaceCounters;

// A launch plan: tile configuration ('L' = 128 x 128, 'S' = 64 x 64) and K splits.
struct Plan {
    char cfg;
    int splits;
};

// Plan rule, fitted to measurements on GB300 (fp32, flushed L2):
//  * when the 128 x 128 tiles alone give every SM a tile, use them unsplit (best per-flop
//    throughput: 8 x 8 outer products, 128-bit fragment reads);
//  * otherwise use 64 x 64 tiles (three CTAs per SM) and split K so that the grid fills one
//    wave of num_sms * 3 CTAs, with at most 16 splits and at least two 16-wide slices each.
// Split-K needs the workspace: at most kWsCounters tiles and kWsBytes of partial tiles.
// GEMM_GB300_SGEMM_PLAN="S:4" (configuration and splits) overrides the rule, for sweeps.
Plan choose_plan(int64_t M, int64_t N, int64_t K, int64_t batch, int num_sms, bool allow_split)
{
    // a batch multiplies the tiles (and the split-K partials) of one problem
    const int KT = static_cast<int>((K + 15) / 16);
    const int64_t tiles_l = ((M + CfgL::BM - 1) / CfgL::BM) * ((N + CfgL::BN - 1) / CfgL::BN) * batch;
    const int64_t tiles_s = ((M + CfgS::BM - 1) / CfgS::BM) * ((N + CfgS::BN - 1) / CfgS::BN) * batch;
    auto fits = [&](int64_t tiles, int bm, int bn, int S) {
        return S == 1 || (allow_split && S <= KT && tiles <= int64_t(kWsCounters) &&
                          size_t(tiles) * S * bm * bn * 4 <= kWsBytes);
    };
    Plan plan{'L', 1};
    if (tiles_l < num_sms) {
        const int64_t target = int64_t(num_sms) * CfgS::MIN_BLOCKS;
        int S = static_cast<int>((target + tiles_s / 2) / tiles_s);
        S = S < 1 ? 1 : (S > 16 ? 16 : S);
        while (S > 1 && (KT / S < 2 || !fits(tiles_s, CfgS::BM, CfgS::BN, S))) --S;
        plan = {'S', S};
    }
    if (const char *e = std::getenv("GEMM_GB300_SGEMM_PLAN")) {
        if ((e[0] == 'L' || e[0] == 'S') && e[1] == ':') {
            const int f = std::atoi(e + 2);
            const bool l = e[0] == 'L';
            if (f >= 1 && fits(l ? tiles_l : tiles_s, l ? CfgL::BM : CfgS::BM, l ? CfgL::BN : CfgS::BN, f))
                plan = {e[0], f};
        }
    }
    return plan;
}

}  // namespace

cudaError_t launch_sgemm(const DeviceInfo &dev, int opA, int opB, int64_t M, int64_t N,
                         int64_t K, float alpha, const float *A, int64_t lda, int64_t strideA,
                         const float *B, int64_t ldb, int64_t strideB, float beta, float *C,
                         int64_t ldc, int64_t strideC, int64_t batch, cudaStream_t stream)
{
    SgemmParams p{};
    p.M = M; p.N = N; p.K = K;
    p.A = A; p.lda = lda; p.B = B; p.ldb = ldb; p.C = C; p.ldc = ldc;
    p.alpha = alpha; p.beta = beta;
    p.log_group = 3;
    p.batch = batch;
    p.stride_a = batch > 1 ? strideA : 0;
    p.stride_b = batch > 1 ? strideB : 0;
    p.stride_c = batch > 1 ? strideC : 0;
    // 16-byte paths need every problem's base aligned: strides divisible by 4 elements
    const bool strides4 = batch <= 1 || (strideA % 4 == 0 && strideB % 4 == 0);
    p.c_vec = aligned16(C) && (ldc % 4) == 0 && (batch <= 1 || strideC % 4 == 0);
    // op(A) = N stores A as M x K, rows along k: staged K-major.  op(A) = T stores K x M,
    // rows along m: staged [k][m].  B likewise with n in place of m (op(B) = T is K-major).
    // 16-byte copies need a 16-byte aligned base and a leading dimension divisible by 4.
    const bool a_vec = aligned16(A) && lda % 4 == 0 && strides4;
    const bool b_vec = aligned16(B) && ldb % 4 == 0 && strides4;
    Plan plan = choose_plan(M, N, K, batch, dev.num_sms, true);
    StreamWorkspace w;
    if (plan.splits > 1 && !stream_workspace(dev.device, stream, w))
        plan = choose_plan(M, N, K, batch, dev.num_sms, false);  // no workspace: plan without split
    const int bm = plan.cfg == 'L' ? CfgL::BM : CfgS::BM, bn = plan.cfg == 'L' ? CfgL::BN : CfgS::BN;
    const int KT = static_cast<int>((K + 15) / 16);
    const bool transposed = plan.cfg == 'L' ? KContigModes<CfgL>::kTransposed : KContigModes<CfgS>::kTransposed;
    const int k_vec_a = transposed ? kKT : (a_vec ? kKVec : kKScalar);
    const int k_vec_b = transposed ? kKT : (b_vec ? kKVec : kKScalar);
    const int a_mode = opA == GEMM_OP_N ? k_vec_a : (a_vec ? kMnVec : kMnScalar);
    const int b_mode = opB == GEMM_OP_T ? k_vec_b : (b_vec ? kMnVec : kMnScalar);
    p.tiles_m = (M + bm - 1) / bm;
    p.tiles_n = (N + bn - 1) / bn;
    p.splits = plan.splits;
    p.kt_per_split = (KT + plan.splits - 1) / plan.splits;
    if (plan.splits > 1) {
        p.ws = w.data;
        p.counters = w.counters;
        return plan.cfg == 'L' ? launch_LS(dev.device, a_mode, b_mode, p, stream)
                               : launch_SS(dev.device, a_mode, b_mode, p, stream);
    }
    return plan.cfg == 'L' ? launch_L(dev.device, a_mode, b_mode, p, stream)
                           : launch_S(dev.device, a_mode, b_mode, p, stream);
}

cudaError_t launch_scale_batched(int64_t M, int64_t N, float beta, float *C, int64_t ldc,
                                 int64_t strideC, int64_t batch, cudaStream_t stream)
{
    for (int64_t b = 0; b < batch; ++b) {
        const cudaError_t e = launch_scale(M, N, beta, C + b * strideC, ldc, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_scale(int64_t M, int64_t N, float beta, float *C, int64_t ldc,
                         cudaStream_t stream)
{
    const int64_t total = M * N;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    scale_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(M, N, beta, C, ldc);
    return cudaGetLastError();
}

}  // namespace gemm
