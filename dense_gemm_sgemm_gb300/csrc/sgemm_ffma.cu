// Strict-FP32 SGEMM on the CUDA cores of sm_103a.
//
// C = alpha * op(A) * op(B) + beta * C, row-major (copecc.github.io "GEMM" page, section
// "核心问题与运算特征").  The kernel follows the blocking the pages build up, re-designed
// for Blackwell:
//   * block tile BM x BN, K sliced by BK and staged in shared memory (copecc "共享内存分块";
//     ssxxe.cn section "2.1"), as a STAGES-deep cp.async ring instead of the pages'
//     register double buffer (ssxxe.cn section "2.3") -- the copy engine fills slot s+3
//     while the FMA units work on slot s, with one __syncthreads per K slice;
//   * each thread owns a TM x TN outer-product tile split into 4 x 4 blocks spaced BM/2
//     (BN/2) apart (copecc "二维寄存器分块"; ssxxe.cn section "2.2"), read from shared memory
//     with 128-bit loads (copecc "向量化访存");
//   * both operands live in shared memory as [k][m] / [k][n] with the 16-byte chunk index
//     XOR-ed with (k mod 8) (copecc "共享内存填充与重排", Swizzling), which keeps the
//     transposing 4-byte copies, the 16-byte copies and the fragment reads all free of bank
//     conflicts without padding;
//   * the products are fused multiply-adds on packed fp32 pairs (fma.rn.f32x2 through
//     __ffma2_rn), IEEE fp32 with round-to-nearest-even and no TF32;
//   * ragged M, N and K are handled by zero-filled copies (cp.async src-size 0) and
//     predicated stores (yekq.top "LeetGPU 第二题", the 1001 x 513 x 777 case);
//   * the 1-D grid is rasterised in groups of tile rows (copecc "线程块网格重排").
#include <cuda_runtime.h>

#include <atomic>

#include "gemm_internal.h"

namespace gemm {
namespace {

constexpr int kThreads = 256;

// Operand loader modes.
constexpr int kMnVec = 0;     // global rows run along k, 16-byte copies (aligned)
constexpr int kMnScalar = 1;  // global rows run along k, 4-byte copies (any ld)
constexpr int kKContig = 2;   // global rows run along m (or n), 4-byte transposing copies

struct SgemmParams {
    int64_t M, N, K;
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    float *C;
    int64_t ldc;
    float alpha, beta;
    int64_t tiles_m, tiles_n;
    int log_group;
    int c_vec;  // C base 16-byte aligned and ldc % 4 == 0
};

template <int BM_, int BN_, int BK_, int TM_, int TN_, int STAGES_, int MIN_BLOCKS_>
struct Cfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, TM = TM_, TN = TN_, STAGES = STAGES_;
    static constexpr int MIN_BLOCKS = MIN_BLOCKS_;
    static constexpr int TY = BM / TM, TX = BN / TN;  // thread grid
    static constexpr int MB = TM / 4, NB = TN / 4;    // 4-wide blocks per thread
    static constexpr int M_STRIDE = BM / MB, N_STRIDE = BN / NB;
    static constexpr int A_STAGE = BK * BM, B_STAGE = BK * BN;  // floats per stage
    static constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
    static_assert(TY * TX == kThreads, "one thread per TM x TN tile");
    static_assert(TX % 8 == 0 && TY % 4 == 0, "a warp covers 4 x 8 threads");
    static_assert(TM % 4 == 0 && TN % 4 == 0, "128-bit fragment loads");
    static_assert(BM % 32 == 0 && BN % 32 == 0 && BK % 8 == 0, "swizzle needs 8 chunks per row");
};

using CfgLarge = Cfg<128, 128, 16, 8, 8, 4, 2>;
using CfgSmall = Cfg<64, 64, 16, 4, 4, 4, 2>;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Float offset of element (k, x) in a [BK][W] stage: 16-byte chunk index XOR (k mod 8).
template <int W>
__device__ __forceinline__ int swz(int k, int x)
{
    return k * W + ((((x >> 2) ^ (k & 7)) << 2) | (x & 3));
}

// Copies BK x W slices of one operand into shared memory, one slice per call.  The
// per-thread parts of every address (row, column, bank) are fixed at construction; a call
// only adds the slice offset, so the unrolled copies use immediate offsets.
//   X    stored matrix, ld its leading dimension
//   ext  extent of the m (or n) dimension, x0 the tile origin along it
template <int MODE, int W, int BK>
struct SliceLoader;

// Rows of X run along k (op(A) = T, op(B) = N), aligned: 16-byte copies.
template <int W, int BK>
struct SliceLoader<kMnVec, W, BK> {
    static constexpr int CPR = W / 4;            // 16-byte chunks per k row
    static constexpr int R = BK * CPR / kThreads;  // copies per thread
    static constexpr int KSTEP = kThreads / CPR;   // k distance between a thread's copies
    static_assert(BK * CPR % kThreads == 0 && KSTEP % 8 == 0, "");
    const float *p;   // element (kb, x) of the current slice
    int64_t ld;
    int kb;           // first k row of this thread
    uint32_t bytes;   // valid bytes of this thread's chunk (ragged n tail)
    uint32_t dst0;    // byte offset in a stage
    __device__ __forceinline__ SliceLoader(const float *X, int64_t ld_, int64_t ext, int64_t x0, int tid)
    {
        const int c = tid % CPR;
        kb = tid / CPR;
        ld = ld_;
        const int64_t rem = ext - (x0 + 4 * c);
        bytes = rem <= 0 ? 0u : (rem >= 4 ? 16u : static_cast<uint32_t>(rem * 4));
        p = X + kb * ld + (bytes ? x0 + 4 * c : 0);
        dst0 = static_cast<uint32_t>(kb * W + ((c ^ (kb & 7)) << 2)) * 4u;
    }
    __device__ __forceinline__ void load(uint32_t stage, const float *base, int64_t k0, int64_t K) const
    {
        const float *q = p + k0 * ld;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const bool ok = bytes && (k0 + kb + r * KSTEP < K);
            cp_async16(stage + dst0 + r * KSTEP * W * 4, ok ? q + r * KSTEP * ld : base, ok ? bytes : 0u);
        }
    }
};

// Rows of X run along k, unaligned pointer or ld: 4-byte copies.
template <int W, int BK>
struct SliceLoader<kMnScalar, W, BK> {
    static constexpr int R = BK * W / kThreads;
    static constexpr int KSTEP = kThreads / W;
    static_assert(BK * W % kThreads == 0 && kThreads % W == 0, "");
    const float *p;
    int64_t ld;
    int kb, x;
    bool x_ok;
    __device__ __forceinline__ SliceLoader(const float *X, int64_t ld_, int64_t ext, int64_t x0, int tid)
    {
        x = tid % W;
        kb = tid / W;
        ld = ld_;
        x_ok = x0 + x < ext;
        p = X + kb * ld + (x_ok ? x0 + x : 0);
    }
    __device__ __forceinline__ void load(uint32_t stage, const float *base, int64_t k0, int64_t K) const
    {
        const float *q = p + k0 * ld;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int k = kb + r * KSTEP;
            const bool ok = x_ok && (k0 + k < K);
            cp_async4(stage + static_cast<uint32_t>(swz<W>(k, x)) * 4u, ok ? q + r * KSTEP * ld : base,
                      ok ? 4u : 0u);
        }
    }
};

// Rows of X run along m or n (op(A) = N, op(B) = T): 4-byte copies that transpose.  Each
// warp copies a 4 (x) by 8 (k) patch -- lanes 0-3 take four rows of X, lanes in steps of 4
// walk 8 consecutive k -- and the swizzle spreads its 32 stores over all 32 banks.
template <int W, int BK>
struct SliceLoader<kKContig, W, BK> {
    static constexpr int RX = W / 32;               // patches per thread along x
    static constexpr int RK = BK / 8;               // patches per thread along k
    static_assert(W % 32 == 0 && BK % 8 == 0 && kThreads == 256, "");
    const float *p;   // element (x0 + xb, kb) of X for the current slice
    int64_t ld;
    int kb;
    uint32_t row_ok;  // bit i: row xb + 32 i inside the matrix
    uint32_t dst0;
    __device__ __forceinline__ SliceLoader(const float *X, int64_t ld_, int64_t ext, int64_t x0, int tid)
    {
        const int lane = tid & 31, warp = tid >> 5;
        const int xb = 4 * warp + (lane & 3);
        kb = lane >> 2;
        ld = ld_;
        row_ok = 0;
#pragma unroll
        for (int i = 0; i < RX; ++i)
            if (x0 + xb + 32 * i < ext) row_ok |= 1u << i;
        p = X + (row_ok & 1u ? (x0 + xb) * ld : 0) + kb;
        dst0 = static_cast<uint32_t>(kb * W + (((warp ^ kb)) << 2) + (lane & 3)) * 4u;
    }
    __device__ __forceinline__ void load(uint32_t stage, const float *base, int64_t k0, int64_t K) const
    {
        const float *q = p + k0;
#pragma unroll
        for (int rk = 0; rk < RK; ++rk) {
            const bool k_ok = k0 + kb + 8 * rk < K;
#pragma unroll
            for (int rx = 0; rx < RX; ++rx) {
                const bool ok = k_ok && ((row_ok >> rx) & 1u);
                cp_async4(stage + dst0 + static_cast<uint32_t>(8 * rk * W + 32 * rx) * 4u,
                          ok ? q + int64_t(32 * rx) * ld + 8 * rk : base, ok ? 4u : 0u);
            }
        }
    }
};

template <class C, int A_MODE, int B_MODE>
__global__ void __launch_bounds__(kThreads, C::MIN_BLOCKS) sgemm_ffma_kernel(const SgemmParams p)
{
    extern __shared__ __align__(16) float smem[];
    float *sA = smem;
    float *sB = smem + C::STAGES * C::A_STAGE;

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int ty = (warp / (C::TX / 8)) * 4 + (lane >> 3);
    const int tx = (warp % (C::TX / 8)) * 8 + (lane & 7);

    int64_t tm, tn;
    raster(blockIdx.x, p.tiles_m, p.tiles_n, p.log_group, tm, tn);
    const int64_t m0 = tm * C::BM, n0 = tn * C::BN;
    const int KT = static_cast<int>((p.K + C::BK - 1) / C::BK);

    const uint32_t sA_addr = smem_addr(sA), sB_addr = smem_addr(sB);
    const SliceLoader<A_MODE, C::BM, C::BK> la(p.A, p.lda, p.M, m0, tid);
    const SliceLoader<B_MODE, C::BN, C::BK> lb(p.B, p.ldb, p.N, n0, tid);
    auto load_tile = [&](int slot, int kt) {
        const int64_t k0 = int64_t(kt) * C::BK;
        la.load(sA_addr + slot * C::A_STAGE * 4, p.A, k0, p.K);
        lb.load(sB_addr + slot * C::B_STAGE * 4, p.B, k0, p.K);
    };

#pragma unroll
    for (int s = 0; s < C::STAGES - 1; ++s) {
        if (s < KT) load_tile(s, s);
        cp_async_commit();
    }

    float2 acc[C::TM][C::TN / 2];
#pragma unroll
    for (int i = 0; i < C::TM; ++i)
#pragma unroll
        for (int j = 0; j < C::TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);

    for (int kt = 0; kt < KT; ++kt) {
        cp_async_wait<C::STAGES - 2>();
        __syncthreads();  // slice kt is visible; every thread is done with slot (kt-1)
        const int nt = kt + C::STAGES - 1;
        if (nt < KT) load_tile(nt % C::STAGES, nt);
        cp_async_commit();

        const float *As = sA + (kt % C::STAGES) * C::A_STAGE;
        const float *Bs = sB + (kt % C::STAGES) * C::B_STAGE;
#pragma unroll
        for (int k = 0; k < C::BK; ++k) {
            float a[C::TM], b[C::TN];
#pragma unroll
            for (int i = 0; i < C::MB; ++i) {
                const int c = (i * C::M_STRIDE) / 4 + ty;
                const float4 v =
                    *reinterpret_cast<const float4 *>(As + k * C::BM + ((c ^ (k & 7)) << 2));
                a[4 * i + 0] = v.x; a[4 * i + 1] = v.y; a[4 * i + 2] = v.z; a[4 * i + 3] = v.w;
            }
#pragma unroll
            for (int j = 0; j < C::NB; ++j) {
                const int c = (j * C::N_STRIDE) / 4 + tx;
                const float4 v =
                    *reinterpret_cast<const float4 *>(Bs + k * C::BN + ((c ^ (k & 7)) << 2));
                b[4 * j + 0] = v.x; b[4 * j + 1] = v.y; b[4 * j + 2] = v.z; b[4 * j + 3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < C::TM; ++i) {
                const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
                for (int j = 0; j < C::TN / 2; ++j)
                    acc[i][j] = __ffma2_rn(ai, make_float2(b[2 * j], b[2 * j + 1]), acc[i][j]);
            }
        }
    }
    cp_async_wait<0>();

    // Epilogue: C = alpha * acc + beta * C, beta == 0 never reads C.
    const float alpha = p.alpha, beta = p.beta;
#pragma unroll
    for (int i = 0; i < C::TM; ++i) {
        const int64_t gm = m0 + (i / 4) * C::M_STRIDE + ty * 4 + (i % 4);
        if (gm >= p.M) continue;
        float *crow = p.C + gm * p.ldc;
#pragma unroll
        for (int jb = 0; jb < C::NB; ++jb) {
            const int64_t gn = n0 + jb * C::N_STRIDE + tx * 4;
            const float2 lo = acc[i][2 * jb], hi = acc[i][2 * jb + 1];
            float v[4] = {lo.x, lo.y, hi.x, hi.y};
            if (p.c_vec && gn + 3 < p.N) {
                float4 o;
                if (beta != 0.0f) {
                    const float4 cin = *reinterpret_cast<const float4 *>(crow + gn);
                    o.x = fmaf(alpha, v[0], beta * cin.x);
                    o.y = fmaf(alpha, v[1], beta * cin.y);
                    o.z = fmaf(alpha, v[2], beta * cin.z);
                    o.w = fmaf(alpha, v[3], beta * cin.w);
                } else {
                    o = make_float4(alpha * v[0], alpha * v[1], alpha * v[2], alpha * v[3]);
                }
                *reinterpret_cast<float4 *>(crow + gn) = o;
            } else {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    if (gn + jj < p.N) {
                        const float r = beta != 0.0f ? fmaf(alpha, v[jj], beta * crow[gn + jj])
                                                     : alpha * v[jj];
                        crow[gn + jj] = r;
                    }
                }
            }
        }
    }
}

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

template <class C, int A_MODE, int B_MODE>
cudaError_t launch_cfg(int dev_id, const SgemmParams &p, cudaStream_t stream)
{
    auto kern = sgemm_ffma_kernel<C, A_MODE, B_MODE>;
    // The shared-memory opt-in is a per-device function attribute: set it once per device.
    static std::atomic<uint64_t> attr_set{0};
    const uint64_t bit = uint64_t(1) << (dev_id & 63);
    if (!(attr_set.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(bit, std::memory_order_release);
    }
    const int64_t tiles = p.tiles_m * p.tiles_n;
    if (tiles > 0x7fffffff) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(tiles), kThreads, C::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

template <class C, int A_MODE>
cudaError_t launch_b(int dev_id, int b_mode, const SgemmParams &p, cudaStream_t s)
{
    switch (b_mode) {
    case kMnVec: return launch_cfg<C, A_MODE, kMnVec>(dev_id, p, s);
    case kMnScalar: return launch_cfg<C, A_MODE, kMnScalar>(dev_id, p, s);
    default: return launch_cfg<C, A_MODE, kKContig>(dev_id, p, s);
    }
}

template <class C>
cudaError_t launch_ab(int dev_id, int a_mode, int b_mode, SgemmParams p, cudaStream_t s)
{
    p.tiles_m = (p.M + C::BM - 1) / C::BM;
    p.tiles_n = (p.N + C::BN - 1) / C::BN;
    switch (a_mode) {
    case kMnVec: return launch_b<C, kMnVec>(dev_id, b_mode, p, s);
    case kMnScalar: return launch_b<C, kMnScalar>(dev_id, b_mode, p, s);
    default: return launch_b<C, kKContig>(dev_id, b_mode, p, s);
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_sgemm(const DeviceInfo &dev, int opA, int opB, int64_t M, int64_t N,
                         int64_t K, float alpha, const float *A, int64_t lda, const float *B,
                         int64_t ldb, float beta, float *C, int64_t ldc, cudaStream_t stream)
{
    SgemmParams p{};
    p.M = M; p.N = N; p.K = K;
    p.A = A; p.lda = lda; p.B = B; p.ldb = ldb; p.C = C; p.ldc = ldc;
    p.alpha = alpha; p.beta = beta;
    p.log_group = 3;
    p.c_vec = aligned16(C) && (ldc % 4) == 0;
    // op(A) = N stores A as M x K: rows run along k, so A is K-contiguous.  op(A) = T
    // stores K x M: rows run along m.  The same holds for B with n in place of m.
    const int a_mode = opA == GEMM_OP_N ? kKContig
                       : (aligned16(A) && lda % 4 == 0 ? kMnVec : kMnScalar);
    const int b_mode = opB == GEMM_OP_T ? kKContig
                       : (aligned16(B) && ldb % 4 == 0 ? kMnVec : kMnScalar);
    // Large tiles when they give every SM at least one tile, else the 64 x 64 tile so that
    // small problems still spread over the chip.
    const int64_t large_tiles = ((M + 127) / 128) * ((N + 127) / 128);
    if (large_tiles >= dev.num_sms) return launch_ab<CfgLarge>(dev.device, a_mode, b_mode, p, stream);
    return launch_ab<CfgSmall>(dev.device, a_mode, b_mode, p, stream);
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
