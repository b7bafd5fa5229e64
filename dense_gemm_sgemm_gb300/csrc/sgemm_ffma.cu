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

// One tile configuration as the host sees it, with its cost-model constants (microseconds,
// fitted by least squares on log time to 1,600 timed launches on GB300: ten M x N shapes from
// 256^2 to 3072^2, K = 128 / 513 / 1024 / 4096, op(A) = N and T, every configuration and split
// count below; the rule picks a plan within 1.6% of the fastest measured one on average, and
// within 1.8% over 1,900 launches re-measured after the 128-row tiles moved to 32-wide slices,
// where a refit gained nothing; refit on 3,840 launches -- the same shapes with beta = -0.5
// and with beta = 0 -- after the 64 x 64 tile's lane-quad layout and padded stages made it
// faster: 1.4% from the fastest plan on average (geometric), was 2.6%; 1.6% on 3,840
// launches re-measured after the 128 x 64 tile moved to padded 16-wide slices, where a refit
// gained nothing).
struct CfgDesc {
    char name;  // 'L' = 128 x 128 (8 x 8 per thread), 'M' = 128 x 64 (8 x 4), 'S' = 64 x 64 (4 x 4)
    int bm, bn, bk, min_blocks;
    bool a_k_major;  // a K-contiguous A is staged [x][k] (else transposed to [k][x])
    int max_splits;
    double us_slice;   // one K slice of one CTA, per co-resident CTA of the same SM
    double us_fixed;   // per wave of CTAs: prologue, epilogue, launch ramp
    double us_split;   // per split: partial-tile traffic and the fixed-order sum
    cudaError_t (*launch)(int, int, int, const SgemmParams &, cudaStream_t);
    cudaError_t (*launch_split)(int, int, int, const SgemmParams &, cudaStream_t);
};

using Launcher = cudaError_t (*)(int, int, int, const SgemmParams &, cudaStream_t);

template <class C>
constexpr CfgDesc desc(char name, int max_splits, double us_slice, double us_fixed, double us_split,
                       Launcher l, Launcher ls)
{
    return CfgDesc{name, C::BM, C::BN, C::BK, C::MIN_BLOCKS, mode_allowed<C>(kKVec), max_splits,
                   us_slice, us_fixed, us_split, l, ls};
}

const CfgDesc kCfgs[] = {
    desc<CfgL>('L', 4, 1.348, 2.682, 1.846, launch_L, launch_LS),
    desc<CfgM>('M', 12, 0.791, 2.395, 0.725, launch_M, launch_MS),
    desc<CfgS>('S', 16, 0.403, 1.511, 0.150, launch_S, launch_SS),
};

const CfgDesc *find_cfg(char name)
{
    for (const CfgDesc &c : kCfgs)
        if (c.name == name) return &c;
    return nullptr;
}

// A launch plan: tile configuration, K splits, and the number of leading tiles that run
// whole (0: every tile is split; see SgemmParams::full_tiles).
struct Plan {
    const CfgDesc *cfg;
    int splits;
    int64_t full_tiles;
};

// Plan rule: the (configuration, splits) pair of least modelled time.  CTAs run in waves of
// num_sms * min_blocks; the CTAs that share an SM share its FMA pipes, so a wave lasts
// (slices per CTA) * (CTAs on the busiest SM) * us_slice + us_fixed, and every split adds
// us_split.  Splits come from {1, 2, 3, 4, 6, 8, 12, 16} (at most max_splits, at least two
// K slices each) and cost 2% extra in the comparison, so near ties keep K whole.
// Split-K needs the workspace: at most kWsCounters tiles and kWsBytes of partial tiles.
// GEMM_GB300_SGEMM_PLAN="S:4" (configuration and splits) overrides the rule, for sweeps; an
// unsplit override still gets the last-wave split below unless GEMM_GB300_SGEMM_TAIL=0.
Plan choose_plan(int64_t M, int64_t N, int64_t K, int64_t batch, int num_sms, bool allow_split)
{
    // a batch multiplies the tiles (and the split-K partials) of one problem.  KT counts K in
    // 16-wide units (the cost model's unit); a configuration splits its own, BK-wide slices.
    const int64_t KT = (K + 15) / 16;
    auto tiles = [&](const CfgDesc &c) { return ((M + c.bm - 1) / c.bm) * ((N + c.bn - 1) / c.bn) * batch; };
    auto fits = [&](const CfgDesc &c, int S) {
        return S == 1 || (allow_split && S <= (K + c.bk - 1) / c.bk && S <= c.max_splits &&
                          tiles(c) <= int64_t(kWsCounters) && size_t(tiles(c)) * S * c.bm * c.bn * 4 <= kWsBytes);
    };
    auto cost = [&](const CfgDesc &c, int S) {
        const int64_t ctas = tiles(c) * S;
        const double kps = double((KT + S - 1) / S);
        const int64_t slots = int64_t(num_sms) * c.min_blocks;
        const int64_t full = ctas / slots, rem = ctas % slots;
        double t = double(full) * (kps * c.min_blocks * c.us_slice + c.us_fixed);
        if (rem > 0) t += kps * double((rem + num_sms - 1) / num_sms) * c.us_slice + c.us_fixed;
        if (S > 1) t = (t + S * c.us_split) * 1.02;
        return t;
    };
    static const int kSplits[] = {1, 2, 3, 4, 6, 8, 12, 16};
    Plan plan{find_cfg('L'), 1, 0};
    double best = -1.0;
    for (const CfgDesc &c : kCfgs)
        for (int S : kSplits) {
            if (!fits(c, S) || (S > 1 && KT / S < 2)) continue;
            const double t = cost(c, S);
            if (best < 0.0 || t < best) {
                best = t;
                plan = {&c, S, 0};
            }
        }
    if (const char *e = std::getenv("GEMM_GB300_SGEMM_PLAN")) {
        const CfgDesc *c = find_cfg(e[0]);
        if (c != nullptr && e[1] == ':') {
            const int f = std::atoi(e + 2);
            if (f >= 1 && fits(*c, f)) plan = {c, f, 0};
        }
    }
    // Last partial wave of the 128 x 128 tile (two CTAs per SM).  A CTA alone on its SM runs
    // about twice as fast as one sharing it, so a last wave of tail <= num_sms tiles already
    // takes ~1/2 of a full wave.  Split S ways, it takes ~1/(2S) when S * tail <= num_sms
    // (each split still alone) or ~1/S when S * tail fits two per SM.  The split is taken when
    // it reaches 0.4 or less (4096^3: 112 tail tiles, no split pays; 5120^2 x 2048: 80 tail
    // tiles in 3 splits, 1762 -> 1736 us).  At least 4 K slices per split.
    const char *tail_env = std::getenv("GEMM_GB300_SGEMM_TAIL");  // "0": never split the last wave
    if (plan.splits == 1 && batch == 1 && allow_split && plan.cfg->name == 'L' &&
        !(tail_env && tail_env[0] == '0')) {
        const CfgDesc &c = *plan.cfg;
        const int64_t t = tiles(c), slots = int64_t(num_sms) * c.min_blocks, tail = t % slots;
        if (t >= slots && tail > 0 && tail <= int64_t(num_sms) && tail <= int64_t(kWsCounters)) {
            double best_rel = 0.4;
            int best_s = 0;
            for (int S = 2; S <= c.max_splits; ++S) {
                if (KT / S < 4 || S > (K + c.bk - 1) / c.bk || size_t(tail) * S * c.bm * c.bn * 4 > kWsBytes)
                    continue;
                const double rel = tail * S <= num_sms ? 1.0 / (2 * S) : (tail * S <= slots ? 1.0 / S : 1.0);
                if (rel <= best_rel) {
                    best_rel = rel;
                    best_s = S;
                }
            }
            if (best_s > 0) plan = {&c, best_s, t - tail};
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
    Plan plan = choose_plan(M, N, K, batch, dev.num_sms, true);
    // Two splits of every 64 x 64 tile run as two-CTA clusters that hand the partial over
    // through distributed shared memory; every other split plan needs the stream's workspace.
    // GEMM_GB300_SGEMM_PAIR=0 keeps the workspace hand-off (for tests).
    const char *pair_env = std::getenv("GEMM_GB300_SGEMM_PAIR");
    const bool pair_ok = pair_env == nullptr || pair_env[0] != '0';
    auto cluster_pair = [&](const Plan &pl) {
        return pl.splits == 2 && pl.full_tiles == 0 && pl.cfg->name == 'S' && pair_ok;
    };
    StreamWorkspace w;
    if (plan.splits > 1 && !cluster_pair(plan) && !stream_workspace(dev.device, stream, w))
        plan = choose_plan(M, N, K, batch, dev.num_sms, false);  // no workspace: plan without split
    const CfgDesc &cfg = *plan.cfg;
    if (batch <= 1) strideA = strideB = strideC = 0;

    // Tiles that stage every operand [k][x] read a K-contiguous operand through 4-byte
    // transposing copies.  On large problems that operand is transposed once into scratch
    // instead and then read with straight 16-byte copies, which makes the GEMM 6-12% faster
    // (measured at 4096^3 and 16384 x 16384 x 1024).  The transposition moves 8 bytes per
    // element of the operand: relative to the GEMM's 2 M N K flops that is 1-2% when the
    // other output dimension is 2048 or more, and its launch is negligible above 1e10 flops.
    // Without scratch the transposing copies remain.
    if (!cfg.a_k_major && (plan.splits == 1 || plan.full_tiles > 0) &&
        2.0 * double(M) * double(N) * double(K) * double(batch) >= 1e10) {
        const int64_t kOther = 2048;
        const float *t = nullptr;
        int64_t ldt = 0, st = 0;
        if (opA == GEMM_OP_N && N >= kOther &&
            transpose_f32_operand(dev.device, stream, 0, A, M, K, lda, strideA, batch, &t, &ldt, &st)) {
            A = t; lda = ldt; strideA = st; opA = GEMM_OP_T;
        }
        if (opB == GEMM_OP_T && M >= kOther &&
            transpose_f32_operand(dev.device, stream, 1, B, N, K, ldb, strideB, batch, &t, &ldt, &st)) {
            B = t; ldb = ldt; strideB = st; opB = GEMM_OP_N;
        }
    }

    SgemmParams p{};
    p.M = M; p.N = N; p.K = K;
    p.A = A; p.lda = lda; p.B = B; p.ldb = ldb; p.C = C; p.ldc = ldc;
    p.alpha = alpha; p.beta = beta;
    p.log_group = 3;
    p.batch = batch;
    p.stride_a = strideA;
    p.stride_b = strideB;
    p.stride_c = strideC;
    // 16-byte paths need every problem's base aligned: strides divisible by 4 elements
    const bool strides4 = strideA % 4 == 0 && strideB % 4 == 0;
    p.c_vec = aligned16(C) && (ldc % 4) == 0 && strideC % 4 == 0;
    // op(A) = N stores A as M x K, rows along k; op(A) = T stores K x M, rows along m.  B
    // likewise with n in place of m (op(B) = T is K-contiguous).  16-byte copies need a
    // 16-byte aligned base and a leading dimension divisible by 4.
    const bool a_vec = aligned16(A) && lda % 4 == 0 && strides4;
    const bool b_vec = aligned16(B) && ldb % 4 == 0 && strides4;
    const int KT = static_cast<int>((K + cfg.bk - 1) / cfg.bk);  // this configuration's slices
    // K-contiguous operands (op(A) = N, op(B) = T): see mode_allowed
    const int a_mode = opA == GEMM_OP_N ? (cfg.a_k_major && a_vec ? kKVec : kKT)
                                        : (a_vec ? kMnVec : kMnScalar);
    const int b_mode = opB == GEMM_OP_T ? kKT : (b_vec ? kMnVec : kMnScalar);
    p.tiles_m = (M + cfg.bm - 1) / cfg.bm;
    p.tiles_n = (N + cfg.bn - 1) / cfg.bn;
    p.splits = plan.splits;
    p.full_tiles = plan.full_tiles;
    p.kt_per_split = (KT + plan.splits - 1) / plan.splits;
    if (plan.splits > 1) {
        p.ws = w.data;
        p.counters = w.counters;
        if (plan.full_tiles > 0) {
            // The whole tiles run in the kernel without split-K code (the split variant needs
            // more registers and would slow every tile), then the split last wave.
            SgemmParams pw = p;
            pw.splits = 1;
            const cudaError_t e = cfg.launch(dev.device, a_mode, b_mode, pw, stream);
            if (e != cudaSuccess) return e;
            p.cta_offset = plan.full_tiles;
        }
        // Two splits of every 64 x 64 tile: the pair forms a cluster and hands its partial
        // over through distributed shared memory instead of the workspace (the same sum,
        // p0 + p1).
        if (cluster_pair(plan)) return launch_SP(dev.device, a_mode, b_mode, p, stream);
        return cfg.launch_split(dev.device, a_mode, b_mode, p, stream);
    }
    return cfg.launch(dev.device, a_mode, b_mode, p, stream);
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
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches();
    return e;
}

}  // namespace gemm
