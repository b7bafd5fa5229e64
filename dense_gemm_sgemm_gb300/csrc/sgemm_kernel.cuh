// Strict-FP32 SGEMM on the CUDA cores of sm_103a: the kernel template.
//
// C = alpha * op(A) * op(B) + beta * C, row-major (copecc.github.io "GEMM" page, section
// "核心问题与运算特征").  The kernel follows the blocking the pages build up, re-designed
// for Blackwell:
//   * block tile BM x BN, K sliced by BK and staged in shared memory (copecc "共享内存分块";
//     ssxxe.cn section "2.1"), as a STAGES-deep cp.async ring instead of the pages'
//     register double buffer (ssxxe.cn section "2.3") -- the copies of slice s+STAGES-1 are
//     in flight while the FMA units work on slice s, with one __syncthreads per K slice;
//   * each thread owns a TM x TN outer-product tile split into 4 x 4 blocks spaced BM/2
//     (BN/2) apart (copecc "二维寄存器分块"; ssxxe.cn section "2.2");
//   * operands whose stored rows run along k (op(A) = T, op(B) = N) are staged [k][x] with
//     straight copies and read with 128-bit loads (copecc "向量化访存"); K-contiguous ones
//     (op(A) = N, op(B) = T) are either transposed by 4-byte copies into a [k][x] stage or,
//     for A on the 4 x 4 tile, staged [x][k] and read four k per 128-bit load; copies are
//     16 bytes where pointer and leading dimension are aligned, 4 bytes otherwise;
//   * bank conflicts are avoided as copecc "共享内存填充与重排" describes, both ways: the
//     128 x 128 tile XOR-swizzles 16-byte chunk indices (Swizzling, no extra memory); the
//     4 x 4 and 8 x 4 tiles pad each [k][x] row by one chunk (Padding), which costs 6% more
//     shared memory but turns every fragment and copy address into a per-thread base plus a
//     constant -- their inner loops were issue-bound on the swizzle arithmetic;
//   * the products are fused multiply-adds on packed fp32 pairs (fma.rn.f32x2 through
//     __ffma2_rn), IEEE fp32 with round-to-nearest-even and no TF32;
//   * ragged M, N and K are handled by zero-filled copies (cp.async src-size below the copy
//     size) and predicated stores (yekq.top "LeetGPU 第二题", the 1001 x 513 x 777 case);
//   * the 1-D grid is rasterised in groups of tile rows (copecc "线程块网格重排");
//   * optionally K is split over several CTAs (for every tile, or for the last partial wave)
//     whose partial tiles are summed in a fixed order by the last one to finish
//     (deterministic split-K); two splits of a 4 x 4-thread tile instead form a two-CTA
//     cluster and the first reads the second's partial from its shared memory (same order);
//   * each lane quad of the 4 x 4 and 8 x 4 tiles is a 2 x 2 block of the thread grid, so a
//     128-bit fragment load reads at most two distinct 16-byte chunks per quad (2 cycles).
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "gemm_internal.h"

namespace gemm {
namespace sg {

constexpr int kThreads = 256;

// Operand staging modes: shared-memory orientation x copy width.
constexpr int kMnVec = 0;     // stored rows run along k: stage [k][x], 16-byte copies
constexpr int kMnScalar = 1;  // stored rows run along k: stage [k][x], 4-byte copies
constexpr int kKVec = 2;      // stored rows run along x: stage [x][k], 16-byte copies
constexpr int kKT = 4;        // stored rows run along x: stage [k][x], 4-byte copies that transpose
__host__ __device__ constexpr bool is_k_major(int mode) { return mode == kKVec; }

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
    // Split-K: tiles [0, full_tiles) of a problem run whole, one CTA each; every later tile
    // runs as `splits` CTAs, split s summing k slices [s*kt_per_split, (s+1)*kt_per_split).
    // CTA b of a problem (blockIdx.x) takes tile b when b < full_tiles, else tile
    // full_tiles + (b - full_tiles) / splits, split (b - full_tiles) % splits.  full_tiles = 0
    // splits every tile; a positive full_tiles splits only the last, partial wave, and the
    // host then launches the whole tiles (without split-K code) and the split ones apart:
    // a launch covers CTAs [cta_offset, cta_offset + gridDim.x).
    int64_t full_tiles, cta_offset;
    int splits, kt_per_split;
    float *ws;               // splits x tiles partial tiles (splits > 1 only)
    unsigned int *counters;  // one arrival counter per tile, zero between launches
    // Strided batch: problem blockIdx.z of a launch (batch problems in all); element offsets
    // between consecutive problems' A, B and C (0: shared operand).
    int64_t batch, stride_a, stride_b, stride_c;
};

template <int BM_, int BN_, int BK_, int TM_, int TN_, int STAGES_, int MIN_BLOCKS_>
struct Cfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, TM = TM_, TN = TN_, STAGES = STAGES_;
    static constexpr int MIN_BLOCKS = MIN_BLOCKS_;
    static constexpr int TY = BM / TM, TX = BN / TN;  // thread grid
    static constexpr int MB = TM / 4, NB = TN / 4;    // 4-wide blocks per thread
    static constexpr int M_STRIDE = BM / MB, N_STRIDE = BN / NB;
    // [k][x] stage rows: the 4 x 4 and 8 x 4 tiles pad each row by one 16-byte chunk, so every
    // fragment and copy address is a per-thread base plus a constant; the 8 x 8 tile, whose
    // register budget has room for the swizzle arithmetic, XOR-swizzles chunks.
    static constexpr int PAD = TM * TN <= 32 ? 4 : 0;
    static constexpr int A_STAGE = BK * (BM + PAD), B_STAGE = BK * (BN + PAD);  // floats per stage
    static constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
    static constexpr bool PAIR_M = TM > TN;  // accumulator pairs along the longer side
    static_assert(TY * TX == kThreads, "one thread per TM x TN tile");
    static_assert(TX % 8 == 0 && TY % 4 == 0, "a warp covers 4 x 8 threads");
    static_assert(TM % 4 == 0 && TN % 4 == 0, "128-bit fragment loads");
    static_assert(BM % 32 == 0 && BN % 32 == 0, "swizzle needs 8 chunks per [k][x] row");
    static_assert(BK == 16 || TM >= 8, "[x][k] stages (4 x 4 tiles) hold four 16-byte chunks per row");
    static_assert(M_STRIDE % 16 == 0 && N_STRIDE % 16 == 0, "row swizzle repeats every 16 rows");
};

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

__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Thread-block cluster helpers (the two K splits of a tile in one cluster).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Float offset of element (k, x) in a [BK][W] stage: 16-byte chunk index XOR (k mod 8).
template <int W, int PAD>
__device__ __forceinline__ int swz_mn(int k, int x)
{
    if constexpr (PAD > 0) return k * (W + PAD) + x;
    return k * W + ((((x >> 2) ^ (k & 7)) << 2) | (x & 3));
}

// Float offset of element (x, k) in a [W][16] stage: chunk index (k / 4) XOR ((x / 4) mod 4).
__device__ __forceinline__ int swz_k(int x, int k)
{
    return x * 16 + ((((k >> 2) ^ ((x >> 2) & 3)) << 2) | (k & 3));
}

// Copies BK x W slices of one operand into shared memory, one slice per call.  The
// per-thread parts of every address (row, column, bank) are fixed at construction; a call
// only adds the slice offset, so the unrolled copies use immediate offsets.
//   X    stored matrix, ld its leading dimension (passed to load() from the parameters)
//   ext  extent of the m (or n) dimension, x0 the tile origin along it
template <int MODE, int W, int BK, int PAD>
struct SliceLoader;

// Stored rows run along k, aligned: 16-byte copies into [k][x].
template <int W, int BK, int PAD>
struct SliceLoader<kMnVec, W, BK, PAD> {
    static constexpr int CPR = W / 4;              // 16-byte chunks per k row
    static constexpr int R = BK * CPR / kThreads;  // copies per thread
    static constexpr int KSTEP = kThreads / CPR;   // k distance between a thread's copies
    static_assert(BK * CPR % kThreads == 0 && (KSTEP % 8 == 0 || 8 % KSTEP == 0), "");
    const float *p;   // element (kb, x) of slice 0
    int kb;           // first k row of this thread
    int c;            // 16-byte chunk of this thread within a k row
    uint32_t bytes;   // valid bytes of this thread's chunk (ragged x tail)
    uint32_t dst0;    // byte offset in a stage
    __device__ __forceinline__ SliceLoader(const float *X, int64_t ld, int64_t ext, int64_t x0, int tid)
    {
        c = tid % CPR;
        kb = tid / CPR;
        const int64_t rem = ext - (x0 + 4 * c);
        bytes = rem <= 0 ? 0u : (rem >= 4 ? 16u : static_cast<uint32_t>(rem * 4));
        p = X + kb * ld + (bytes ? x0 + 4 * c : 0);
        dst0 = static_cast<uint32_t>(PAD > 0 ? kb * (W + PAD) + 4 * c : kb * W + ((c ^ (kb & 7)) << 2)) * 4u;
    }
    // Byte offset of copy r: rows KSTEP apart keep the swizzle of row kb when KSTEP is a
    // multiple of 8; otherwise each row takes its own.
    __device__ __forceinline__ uint32_t dst(int r) const
    {
        if constexpr (PAD > 0) {
            return dst0 + r * KSTEP * (W + PAD) * 4;
        } else if constexpr (KSTEP % 8 == 0) {
            return dst0 + r * KSTEP * W * 4;
        } else {
            const int k = kb + r * KSTEP;
            return static_cast<uint32_t>(k * W + ((c ^ (k & 7)) << 2)) * 4u;
        }
    }
    template <bool FULL>
    __device__ __forceinline__ void load(uint32_t stage, const float *base, int64_t ld, int64_t k0,
                                         int64_t K) const
    {
        const float *q = p + k0 * ld;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const bool ok = bytes && (FULL || k0 + kb + r * KSTEP < K);
            cp_async16(stage + dst(r), ok ? q + r * KSTEP * ld : base, ok ? bytes : 0u);
        }
    }
};

// Stored rows run along k, unaligned pointer or ld: 4-byte copies into [k][x].
template <int W, int BK, int PAD>
struct SliceLoader<kMnScalar, W, BK, PAD> {
    static constexpr int R = BK * W / kThreads;
    static constexpr int KSTEP = kThreads / W;
    static_assert(BK * W % kThreads == 0 && kThreads % W == 0, "");
    const float *p;
    int kb, x;
    bool x_ok;
    __device__ __forceinline__ SliceLoader(const float *X, int64_t ld, int64_t ext, int64_t x0, int tid)
    {
        x = tid % W;
        kb = tid / W;
        x_ok = x0 + x < ext;
        p = X + kb * ld + (x_ok ? x0 + x : 0);
    }
    template <bool FULL>
    __device__ __forceinline__ void load(uint32_t stage, const float *base, int64_t ld, int64_t k0,
                                         int64_t K) const
    {
        const float *q = p + k0 * ld;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int k = kb + r * KSTEP;
            const bool ok = x_ok && (FULL || k0 + k < K);
            cp_async4(stage + static_cast<uint32_t>(swz_mn<W, PAD>(k, x)) * 4u, ok ? q + r * KSTEP * ld : base,
                      ok ? 4u : 0u);
        }
    }
};

// Stored rows run along x (K contiguous), aligned: 16-byte copies into [x][k].  Four
// consecutive threads take the four chunks of one 64-byte row.
template <int W, int BK, int PAD>
struct SliceLoader<kKVec, W, BK, PAD> {
    static constexpr int R = W * 4 / kThreads;  // rows per thread
    static constexpr int XSTEP = kThreads / 4;   // row distance between a thread's copies
    static_assert(W * 4 % kThreads == 0 && XSTEP % 16 == 0, "");
    const float *p;   // element (x0 + xb, 4c) of X
    int c4;           // first k of this thread's chunk
    uint32_t row_ok;  // bit r: row xb + r * XSTEP inside the matrix
    uint32_t dst0;
    __device__ __forceinline__ SliceLoader(const float *X, int64_t ld, int64_t ext, int64_t x0, int tid)
    {
        const int xb = tid / 4;
        c4 = 4 * (tid % 4);
        row_ok = 0;
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (x0 + xb + r * XSTEP < ext) row_ok |= 1u << r;
        p = X + (row_ok & 1u ? (x0 + xb) * ld : 0) + c4;
        dst0 = static_cast<uint32_t>(swz_k(xb, c4)) * 4u;
    }
    template <bool FULL>
    __device__ __forceinline__ void load(uint32_t stage, const float *base, int64_t ld, int64_t k0,
                                         int64_t K) const
    {
        const int64_t rem = K - (k0 + c4);
        const uint32_t bytes = FULL ? 16u : (rem <= 0 ? 0u : (rem >= 4 ? 16u : static_cast<uint32_t>(rem * 4)));
        const float *q = p + k0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const bool ok = bytes && ((row_ok >> r) & 1u);
            cp_async16(stage + dst0 + r * XSTEP * BK * 4, ok ? q + int64_t(r * XSTEP) * ld : base,
                       ok ? bytes : 0u);
        }
    }
};

// Stored rows run along x, staged transposed as [k][x] with 4-byte copies.  Each warp
// copies a 4 (x) by 8 (k) patch -- lanes 0-3 take four rows of X, lanes in steps of 4 walk
// 8 consecutive k -- and the swizzle spreads its 32 stores over all 32 banks.  Costs more
// copy instructions than a K-major stage but keeps the 128-bit fragment reads.
template <int W, int BK, int PAD>
struct SliceLoader<kKT, W, BK, PAD> {
    static constexpr int RX = W / 32;  // patches per thread along x
    static constexpr int RK = BK / 8;  // patches per thread along k
    static_assert(W % 32 == 0 && BK % 8 == 0 && kThreads == 256, "");
    const float *p;   // element (x0 + xb, kb) of X
    int kb;
    uint32_t row_ok;  // bit i: row xb + 32 i inside the matrix
    uint32_t dst0;
    __device__ __forceinline__ SliceLoader(const float *X, int64_t ld, int64_t ext, int64_t x0, int tid)
    {
        const int lane = tid & 31, warp = tid >> 5;
        const int xb = 4 * warp + (lane & 3);
        kb = lane >> 2;
        row_ok = 0;
#pragma unroll
        for (int i = 0; i < RX; ++i)
            if (x0 + xb + 32 * i < ext) row_ok |= 1u << i;
        p = X + (row_ok & 1u ? (x0 + xb) * ld : 0) + kb;
        dst0 = static_cast<uint32_t>(PAD > 0 ? kb * (W + PAD) + 4 * warp + (lane & 3)
                                             : kb * W + ((warp ^ kb) << 2) + (lane & 3)) * 4u;
    }
    template <bool FULL>
    __device__ __forceinline__ void load(uint32_t stage, const float *base, int64_t ld, int64_t k0,
                                         int64_t K) const
    {
        const float *q = p + k0;
#pragma unroll
        for (int rk = 0; rk < RK; ++rk) {
            const bool k_ok = FULL || k0 + kb + 8 * rk < K;
#pragma unroll
            for (int rx = 0; rx < RX; ++rx) {
                const bool ok = k_ok && ((row_ok >> rx) & 1u);
                cp_async4(stage + dst0 + static_cast<uint32_t>(8 * rk * (W + PAD) + 32 * rx) * 4u,
                          ok ? q + int64_t(32 * rx) * ld + 8 * rk : base, ok ? 4u : 0u);
            }
        }
    }
};

// Fragment loads.  A thread's T values of an operand are 4-wide blocks STRIDE apart,
// starting at row (or column) 4 * t4 of the tile.
// [k][x] stages: the values at one k, two 128-bit loads per 8 values.
template <int W, int T, int STRIDE, int PAD>
__device__ __forceinline__ void load_frag_mn(const float *stage, int k, int t4, float (&v)[T])
{
#pragma unroll
    for (int b = 0; b < T / 4; ++b) {
        const int c = (b * STRIDE) / 4 + t4;
        const float4 f = *reinterpret_cast<const float4 *>(
            stage + (PAD > 0 ? k * (W + PAD) + 4 * c : k * W + ((c ^ (k & 7)) << 2)));
        v[4 * b + 0] = f.x; v[4 * b + 1] = f.y; v[4 * b + 2] = f.z; v[4 * b + 3] = f.w;
    }
}

// [x][k] stages: the values at k .. k+G-1 (G = 2 or 4, k a multiple of G, so all of them
// lie in one 16-byte chunk), one 64- or 128-bit load per row.
template <int G, int T, int STRIDE>
__device__ __forceinline__ void load_frag_k_group(const float *stage, int k, int t4, float (&v)[G][T])
{
    static_assert(G == 2 || G == 4, "k groups of 2 or 4");
#pragma unroll
    for (int b = 0; b < T / 4; ++b)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int x = b * STRIDE + 4 * t4 + i;
            if constexpr (G == 4) {
                const float4 f = *reinterpret_cast<const float4 *>(stage + swz_k(x, k));
                v[0][4 * b + i] = f.x;
                v[1][4 * b + i] = f.y;
                v[2][4 * b + i] = f.z;
                v[3][4 * b + i] = f.w;
            } else {
                const float2 f = *reinterpret_cast<const float2 *>(stage + swz_k(x, k));
                v[0][4 * b + i] = f.x;
                v[1][4 * b + i] = f.y;
            }
        }
}

// The TM x TN accumulators of one thread, held as packed fp32 pairs for fma.rn.f32x2.
// PAIR_M = false pairs neighbours along n (element (i, j) lives in v[i][j / 2]); PAIR_M = true
// pairs neighbours along m (element (i, j) lives in v[i / 2][j]).  One operand of each packed
// multiply-add is a pair straight out of a 128-bit fragment load; the other is a broadcast
// value, which costs register moves, so the pairing follows the longer thread-tile side.
template <int TM, int TN, bool PAIR_M>
struct Acc {
    static constexpr int R = PAIR_M ? TM / 2 : TM, S = PAIR_M ? TN : TN / 2;
    float2 v[R][S];

    __device__ __forceinline__ void zero()
    {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < S; ++c) v[r][c] = make_float2(0.f, 0.f);
    }
    __device__ __forceinline__ float &at(int i, int j)
    {
        if constexpr (PAIR_M) {
            float2 &q = v[i >> 1][j];
            return (i & 1) ? q.y : q.x;
        } else {
            float2 &q = v[i][j >> 1];
            return (j & 1) ? q.y : q.x;
        }
    }
    // acc += a b^T for one k (a: TM values along m, b: TN values along n).
    __device__ __forceinline__ void fma(const float (&a)[TM], const float (&b)[TN])
    {
        if constexpr (PAIR_M) {
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const float2 bj = make_float2(b[j], b[j]);
#pragma unroll
                for (int r = 0; r < R; ++r)
                    v[r][j] = __ffma2_rn(make_float2(a[2 * r], a[2 * r + 1]), bj, v[r][j]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
                for (int c = 0; c < S; ++c)
                    v[i][c] = __ffma2_rn(ai, make_float2(b[2 * c], b[2 * c + 1]), v[i][c]);
            }
        }
    }
};

template <class C, int A_MODE, int B_MODE, bool SPLIT, bool PAIR>
__device__ __forceinline__ void sgemm_tile(const SgemmParams &p, const float *__restrict__ A,
                                           const float *__restrict__ B, float *__restrict__ Cmat,
                                           int64_t tile, int split, int nsplit, int64_t slot);

// PAIR: every tile is split in two and the launch forms clusters of two CTAs, the two splits
// of one tile (cluster rank = split); see the hand-off in sgemm_tile.
template <class C, int A_MODE, int B_MODE, bool SPLIT, bool PAIR = false>
__global__ void __launch_bounds__(kThreads, C::MIN_BLOCKS) sgemm_ffma_kernel(const SgemmParams p)
{
    // One problem per CTA: problem blockIdx.z of this launch (the host launches batches of
    // more than 65535 problems in chunks).
    const int64_t z = blockIdx.z;
    const int64_t b = blockIdx.x + p.cta_offset;
    int64_t tile = b, slot = 0;
    int split = 0, nsplit = 1;
    if (SPLIT && b >= p.full_tiles) {
        const int64_t r = b - p.full_tiles;
        tile = p.full_tiles + r / p.splits;
        split = static_cast<int>(r % p.splits);
        nsplit = p.splits;
        slot = z * (p.tiles_m * p.tiles_n - p.full_tiles) + (tile - p.full_tiles);
    }
    sgemm_tile<C, A_MODE, B_MODE, SPLIT, PAIR>(p, p.A + z * p.stride_a, p.B + z * p.stride_b,
                                               p.C + z * p.stride_c, tile, split, nsplit, slot);
}

// One output tile (or one K split of it) of one problem.  slot numbers the split tile's
// partials and arrival counter among all split tiles of the launch.
template <class C, int A_MODE, int B_MODE, bool SPLIT, bool PAIR>
__device__ __forceinline__ void sgemm_tile(const SgemmParams &p, const float *__restrict__ A,
                                           const float *__restrict__ B, float *__restrict__ Cmat,
                                           int64_t tile, int split, int nsplit, int64_t slot)
{
    static_assert(!PAIR || (SPLIT && C::TM * C::TN <= 16), "cluster pairs: split 4 x 4 tiles");
    extern __shared__ __align__(16) float smem[];
    float *sA = smem;
    float *sB = smem + C::STAGES * C::A_STAGE;

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    // A warp covers 4 x 8 threads of the thread grid.  A 128-bit shared load costs two
    // cycles while each group of four consecutive lanes reads at most two distinct 16-byte
    // chunks, four cycles when it reads four (measured on sm_103a).  The 4 x 4 and 8 x 4
    // tiles, whose inner loops are bound by those loads, therefore lay each lane quad out as
    // a 2 x 2 block (lane bits 0 and 4 pick the row, bits 1..3 the column): two cycles for
    // both operands instead of two for A and four for B.  The 8 x 8 tile keeps rows of eight
    // lanes: there the quad layout made ptxas spill.
    constexpr bool kQuadBlocks = C::TM * C::TN <= 32;
    const int ty = (warp / (C::TX / 8)) * 4 + (kQuadBlocks ? ((lane & 1) | ((lane >> 4) << 1)) : (lane >> 3));
    const int tx = (warp % (C::TX / 8)) * 8 + (kQuadBlocks ? (((lane >> 1) & 1) | (((lane >> 2) & 3) << 1)) : (lane & 7));

    int64_t tm, tn;
    raster(tile, p.tiles_m, p.tiles_n, p.log_group, tm, tn);
    const int64_t m0 = tm * C::BM, n0 = tn * C::BN;
    const int KT_all = static_cast<int>((p.K + C::BK - 1) / C::BK);
    const int kt0 = split * p.kt_per_split;
    const int KT = nsplit > 1 ? min(KT_all - kt0, p.kt_per_split) : KT_all;  // slices of this CTA

    const uint32_t sA_addr = smem_addr(sA), sB_addr = smem_addr(sB);
    const SliceLoader<A_MODE, C::BM, C::BK, C::PAD> la(A, p.lda, p.M, m0, tid);
    const SliceLoader<B_MODE, C::BN, C::BK, C::PAD> lb(B, p.ldb, p.N, n0, tid);
    // Copies that read nothing (zero fill) still need a valid address: the parameter-space
    // bases, which cost no registers.
    // On the 4 x 4 tile with 4-byte copies (many copies per FMA), slices that lie wholly
    // inside K skip the per-copy K bounds checks (ragged 1001 x 777 x 513: 41.4 -> 40.0 us).
    // Elsewhere the second copy path costs more than it saves (1024^2 x 1024: +7%).
    constexpr bool kFullSliceFastPath =
        C::TM * C::TN <= 16 && (A_MODE == kKT || A_MODE == kMnScalar || B_MODE == kKT || B_MODE == kMnScalar);
    auto load_tile = [&](int slot, int kt) {
        const int64_t k0 = int64_t(kt0 + kt) * C::BK;
        const uint32_t sa = sA_addr + slot * C::A_STAGE * 4, sb = sB_addr + slot * C::B_STAGE * 4;
        if (kFullSliceFastPath && k0 + C::BK <= p.K) {
            la.template load<true>(sa, p.A, p.lda, k0, p.K);
            lb.template load<true>(sb, p.B, p.ldb, k0, p.K);
        } else {
            la.template load<false>(sa, p.A, p.lda, k0, p.K);
            lb.template load<false>(sb, p.B, p.ldb, k0, p.K);
        }
    };

#pragma unroll
    for (int s = 0; s < C::STAGES - 1; ++s) {
        if (s < KT) load_tile(s, s);
        cp_async_commit();
    }

    // The epilogue reads C when beta != 0: ask L2 for this thread's rows now, so the reads
    // at the end do not wait for DRAM.
    if (p.beta != 0.0f && split == 0) {
#pragma unroll
        for (int i = 0; i < C::TM; ++i) {
            const int64_t gm = m0 + (i / 4) * C::M_STRIDE + ty * 4 + (i % 4);
#pragma unroll
            for (int jb = 0; jb < C::NB; ++jb) {
                const int64_t gn = n0 + jb * C::N_STRIDE + tx * 4;
                if (gm < p.M && gn < p.N) prefetch_l2(Cmat + gm * p.ldc + gn);
            }
        }
    }

    Acc<C::TM, C::TN, C::PAIR_M> acc;
    acc.zero();

    // K-major ([x][k]) operands are read KG consecutive k at a time, one 64- or 128-bit load per
    // row; [k][x] operands one k at a time.
    constexpr int KG = (!is_k_major(A_MODE) && !is_k_major(B_MODE)) ? 1 : (C::TM * C::TN <= 32 ? 4 : 2);
    for (int kt = 0; kt < KT; ++kt) {
        cp_async_wait<C::STAGES - 2>();
        __syncthreads();  // slice kt is visible; every thread is done with slot (kt-1)
        const int nt = kt + C::STAGES - 1;
        if (nt < KT) load_tile(nt % C::STAGES, nt);
        cp_async_commit();

        const float *As = sA + (kt % C::STAGES) * C::A_STAGE;
        const float *Bs = sB + (kt % C::STAGES) * C::B_STAGE;
#pragma unroll
        for (int k = 0; k < C::BK; k += KG) {
            float ag[KG][C::TM], bg[KG][C::TN];
            if constexpr (is_k_major(A_MODE)) load_frag_k_group<KG, C::TM, C::M_STRIDE>(As, k, ty, ag);
            if constexpr (is_k_major(B_MODE)) load_frag_k_group<KG, C::TN, C::N_STRIDE>(Bs, k, tx, bg);
#pragma unroll
            for (int kk = 0; kk < KG; ++kk) {
                float a[C::TM], b[C::TN];
                if constexpr (is_k_major(A_MODE)) {
#pragma unroll
                    for (int i = 0; i < C::TM; ++i) a[i] = ag[kk][i];
                } else {
                    load_frag_mn<C::BM, C::TM, C::M_STRIDE, C::PAD>(As, k + kk, ty, a);
                }
                if constexpr (is_k_major(B_MODE)) {
#pragma unroll
                    for (int j = 0; j < C::TN; ++j) b[j] = bg[kk][j];
                } else {
                    load_frag_mn<C::BN, C::TN, C::N_STRIDE, C::PAD>(Bs, k + kk, tx, b);
                }
                acc.fma(a, b);
            }
        }
    }
    cp_async_wait<0>();

    // Small-tile split kernels read their C values (beta != 0) before the split-K hand-off,
    // so the split that arrives last does not wait for them after it (C is written only by
    // that split).
    const float alpha = p.alpha, beta = p.beta;
    auto row_of = [&](int i) { return m0 + (i / 4) * C::M_STRIDE + ty * 4 + (i % 4); };
    auto col_of = [&](int jb) { return n0 + jb * C::N_STRIDE + tx * 4; };
    constexpr bool kSmallTile = C::TM * C::TN <= 16;
    float4 cin[kSmallTile ? C::TM : 1][kSmallTile ? C::NB : 1];
    auto read_c = [&]() {
#pragma unroll
        for (int i = 0; i < C::TM; ++i) {
            const int64_t gm = row_of(i);
            const float *crow = Cmat + (gm < p.M ? gm * p.ldc : 0);
#pragma unroll
            for (int jb = 0; jb < C::NB; ++jb) {
                const int64_t gn = col_of(jb);
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (gm < p.M) {
                    if (p.c_vec && gn + 3 < p.N) {
                        v = *reinterpret_cast<const float4 *>(crow + gn);
                    } else {
                        v.x = gn + 0 < p.N ? crow[gn + 0] : 0.0f;
                        v.y = gn + 1 < p.N ? crow[gn + 1] : 0.0f;
                        v.z = gn + 2 < p.N ? crow[gn + 2] : 0.0f;
                        v.w = gn + 3 < p.N ? crow[gn + 3] : 0.0f;
                    }
                }
                cin[i][jb] = v;
            }
        }
    };
    if constexpr (kSmallTile) {
        if (beta != 0.0f && (!PAIR || split == 0)) read_c();
    }

    if constexpr (PAIR) {
        // The two K splits of this tile are one cluster.  Split 1 leaves its partial tile in
        // its own (now idle) operand ring, thread-major; after a cluster barrier split 0 reads
        // it through distributed shared memory, adds it to its own (p0 + p1, the order of the
        // global hand-off below) and writes C; a second barrier keeps split 1's shared memory
        // alive until then.  No global round trip, fence or arrival counter.  Both CTAs of a
        // cluster are resident together, and both pass both barriers on every path.
        constexpr int Q = C::TM * C::TN / 4;  // float4 per thread
        constexpr int QR = C::TN / 4;         // float4 per accumulator row
        __syncthreads();  // every warp is done reading the ring
        float4 *part = reinterpret_cast<float4 *>(smem);
        if (split == 1) {
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const int i = q / QR, j = 4 * (q % QR);
                part[q * kThreads + tid] = make_float4(acc.at(i, j), acc.at(i, j + 1), acc.at(i, j + 2), acc.at(i, j + 3));
            }
        }
        cluster_sync();
        if (split == 1) {
            cluster_sync();
            return;
        }
        const uint32_t peer = map_to_rank(smem_addr(part), 1u);
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const float4 u = ld_cluster_f4(peer + static_cast<uint32_t>(q * kThreads + tid) * 16u);
            const int i = q / QR, j = 4 * (q % QR);
            acc.at(i, j) += u.x; acc.at(i, j + 1) += u.y; acc.at(i, j + 2) += u.z; acc.at(i, j + 3) += u.w;
        }
        cluster_sync();
    } else if (SPLIT && nsplit > 1) {
        // Deterministic split-K: every split stores its partial tile, and the split that
        // arrives last adds all partials in split order 0, 1, ..., splits-1 -- the same
        // order whichever CTA finishes last -- before the epilogue.
        constexpr int Q = C::TM * C::TN / 4;  // float4 per thread
        constexpr int QR = C::TN / 4;         // float4 per accumulator row
        const int64_t tile4 = int64_t(C::BM) * C::BN / 4;
        float4 *all = reinterpret_cast<float4 *>(p.ws) + slot * nsplit * tile4;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int i = q / QR, j = 4 * (q % QR);
            __stcg(all + split * tile4 + q * kThreads + tid,
                   make_float4(acc.at(i, j), acc.at(i, j + 1), acc.at(i, j + 2), acc.at(i, j + 3)));
        }
        __threadfence();
        __shared__ unsigned int s_last;
        __syncthreads();
        if (tid == 0) {
            const unsigned int prev = atomicAdd(p.counters + slot, 1u);
            s_last = prev == static_cast<unsigned int>(nsplit - 1);
            if (s_last) p.counters[slot] = 0;  // ready for the next launch
        }
        __syncthreads();
        const bool last = s_last != 0;
        __syncthreads();  // s_last is read before another problem of the batch reuses it
        if (!last) return;
        __threadfence();
        // One round per split, Q independent loads in flight per round.
        for (int s2 = 0; s2 < nsplit; ++s2) {
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const float4 u = __ldcg(all + s2 * tile4 + q * kThreads + tid);
                const int i = q / QR, j = 4 * (q % QR);
                if (s2 == 0) {
                    acc.at(i, j) = u.x; acc.at(i, j + 1) = u.y; acc.at(i, j + 2) = u.z; acc.at(i, j + 3) = u.w;
                } else {
                    acc.at(i, j) += u.x; acc.at(i, j + 1) += u.y; acc.at(i, j + 2) += u.z; acc.at(i, j + 3) += u.w;
                }
            }
        }
    }

    // Epilogue: C = alpha * acc + beta * C, beta == 0 never reads C.
    if constexpr (!kSmallTile) {
        // Large thread tiles (long-running CTAs): one pass, read-modify-write per 4-vector.
#pragma unroll
        for (int i = 0; i < C::TM; ++i) {
            const int64_t gm = row_of(i);
            if (gm >= p.M) continue;
            float *crow = Cmat + gm * p.ldc;
#pragma unroll
            for (int jb = 0; jb < C::NB; ++jb) {
                const int64_t gn = col_of(jb);
                const float v[4] = {acc.at(i, 4 * jb), acc.at(i, 4 * jb + 1), acc.at(i, 4 * jb + 2),
                                    acc.at(i, 4 * jb + 3)};
                if (p.c_vec && gn + 3 < p.N) {
                    float4 o;
                    if (beta != 0.0f) {
                        const float4 cin = *reinterpret_cast<const float4 *>(crow + gn);
                        o = make_float4(fmaf(alpha, v[0], beta * cin.x), fmaf(alpha, v[1], beta * cin.y),
                                        fmaf(alpha, v[2], beta * cin.z), fmaf(alpha, v[3], beta * cin.w));
                    } else {
                        o = make_float4(alpha * v[0], alpha * v[1], alpha * v[2], alpha * v[3]);
                    }
                    *reinterpret_cast<float4 *>(crow + gn) = o;
                } else {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (gn + jj < p.N)
                            crow[gn + jj] = beta != 0.0f ? fmaf(alpha, v[jj], beta * crow[gn + jj]) : alpha * v[jj];
                }
            }
        }
        return;
    }
    // Small thread tiles (short-lived CTAs, where the epilogue is a large share of the time):
    // every read of C was issued above, all in flight together; then every store.
    if (beta != 0.0f) {
#pragma unroll
        for (int i = 0; i < C::TM; ++i) {
#pragma unroll
            for (int jb = 0; jb < C::NB; ++jb) {
                const float4 c4 = cin[i][jb];
                float &v0 = acc.at(i, 4 * jb), &v1 = acc.at(i, 4 * jb + 1);
                float &v2 = acc.at(i, 4 * jb + 2), &v3 = acc.at(i, 4 * jb + 3);
                v0 = fmaf(alpha, v0, beta * c4.x);
                v1 = fmaf(alpha, v1, beta * c4.y);
                v2 = fmaf(alpha, v2, beta * c4.z);
                v3 = fmaf(alpha, v3, beta * c4.w);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < C::TM; ++i)
#pragma unroll
            for (int j = 0; j < C::TN; ++j) acc.at(i, j) *= alpha;
    }
#pragma unroll
    for (int i = 0; i < C::TM; ++i) {
        const int64_t gm = row_of(i);
        if (gm >= p.M) continue;
        float *crow = Cmat + gm * p.ldc;
#pragma unroll
        for (int jb = 0; jb < C::NB; ++jb) {
            const int64_t gn = col_of(jb);
            const float v[4] = {acc.at(i, 4 * jb), acc.at(i, 4 * jb + 1), acc.at(i, 4 * jb + 2),
                                acc.at(i, 4 * jb + 3)};
            if (p.c_vec && gn + 3 < p.N) {
                *reinterpret_cast<float4 *>(crow + gn) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    if (gn + jj < p.N) crow[gn + jj] = v[jj];
            }
        }
    }
}

template <class C, bool SPLIT, int A_MODE, int B_MODE, bool PAIR = false>
cudaError_t launch_cfg(int dev_id, const SgemmParams &p, cudaStream_t stream)
{
    auto kern = sgemm_ffma_kernel<C, A_MODE, B_MODE, SPLIT, PAIR>;
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
    const int64_t ctas = SPLIT ? p.full_tiles + (tiles - p.full_tiles) * p.splits - p.cta_offset
                               : (p.full_tiles > 0 ? p.full_tiles : tiles);
    if (ctas > 0x7fffffff) return cudaErrorInvalidConfiguration;
    // gridDim.z holds at most 65535 problems: larger batches go in consecutive launches on the
    // same stream (which also keeps their split-K workspace use in order).
    constexpr int64_t kMaxZ = 65535;
    for (int64_t b0 = 0; b0 < p.batch; b0 += kMaxZ) {
        SgemmParams q = p;
        q.batch = p.batch - b0 < kMaxZ ? p.batch - b0 : kMaxZ;
        q.A = p.A + b0 * p.stride_a;
        q.B = p.B + b0 * p.stride_b;
        q.C = p.C + b0 * p.stride_c;
        const dim3 grid(static_cast<unsigned>(ctas), 1u, static_cast<unsigned>(q.batch));
        if constexpr (PAIR) {
            // Clusters of the two splits of a tile (CTAs 2t and 2t + 1 of the grid).
            if (p.splits != 2 || p.full_tiles != 0 || p.cta_offset != 0 || ctas % 2 != 0)
                return cudaErrorInvalidValue;
            cudaLaunchConfig_t cfg{};
            cfg.gridDim = grid;
            cfg.blockDim = dim3(kThreads, 1, 1);
            cfg.dynamicSmemBytes = C::SMEM_BYTES;
            cfg.stream = stream;
            cudaLaunchAttribute attr{};
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = 2;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, q);
            if (e != cudaSuccess) return e;
        } else {
            kern<<<grid, kThreads, C::SMEM_BYTES, stream>>>(q);
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        count_launches();
    }
    return cudaSuccess;
}

// Staging modes each tile configuration is instantiated for: thread tiles 8 rows high keep
// 128-bit [k][x] fragment reads (transposing copies of K-contiguous operands, kKT); the 4 x 4
// tile stages an aligned K-contiguous A [x][k] with 16-byte copies (kKVec, read four k per
// 128-bit load) and every other K-contiguous operand through transposing copies (kKT: an
// unaligned A needs 4-byte copies either way and the [k][x] stage reads faster -- ragged
// 1001 x 777 x 513 43.7 -> 41.7 us; [x][k] reads of B rows 4t .. 4t+3 would fall into the
// same 16 banks).
template <class C>
constexpr bool mode_allowed(int mode)
{
    if (C::TM >= 8) return mode == kMnVec || mode == kMnScalar || mode == kKT;
    return mode == kMnVec || mode == kMnScalar || mode == kKVec || mode == kKT;
}

template <class C, bool SPLIT, int A_MODE, int B_MODE, bool PAIR>
cudaError_t launch_if_allowed(int dev_id, const SgemmParams &p, cudaStream_t s)
{
    if constexpr (mode_allowed<C>(A_MODE) && mode_allowed<C>(B_MODE))
        return launch_cfg<C, SPLIT, A_MODE, B_MODE, PAIR>(dev_id, p, s);
    else
        return cudaErrorInvalidValue;
}

template <class C, bool SPLIT, int A_MODE, bool PAIR>
cudaError_t launch_b(int dev_id, int b_mode, const SgemmParams &p, cudaStream_t s)
{
    switch (b_mode) {
    case kMnVec: return launch_if_allowed<C, SPLIT, A_MODE, kMnVec, PAIR>(dev_id, p, s);
    case kMnScalar: return launch_if_allowed<C, SPLIT, A_MODE, kMnScalar, PAIR>(dev_id, p, s);
    case kKVec: return launch_if_allowed<C, SPLIT, A_MODE, kKVec, PAIR>(dev_id, p, s);
    case kKT: return launch_if_allowed<C, SPLIT, A_MODE, kKT, PAIR>(dev_id, p, s);
    default: return cudaErrorInvalidValue;
    }
}

// Launches configuration C for the given staging modes.  p.tiles_m/tiles_n, p.splits and
// p.kt_per_split must already describe the grid of C.  PAIR: two splits per tile as
// two-CTA clusters (p.splits == 2, every tile split).
template <class C, bool SPLIT, bool PAIR = false>
cudaError_t launch_ab(int dev_id, int a_mode, int b_mode, const SgemmParams &p, cudaStream_t s)
{
    if (!mode_allowed<C>(a_mode)) return cudaErrorInvalidValue;
    switch (a_mode) {
    case kMnVec: return launch_b<C, SPLIT, kMnVec, PAIR>(dev_id, b_mode, p, s);
    case kMnScalar: return launch_b<C, SPLIT, kMnScalar, PAIR>(dev_id, b_mode, p, s);
    case kKVec: return launch_b<C, SPLIT, kKVec, PAIR>(dev_id, b_mode, p, s);
    case kKT: return launch_b<C, SPLIT, kKT, PAIR>(dev_id, b_mode, p, s);
    default: return cudaErrorInvalidValue;
    }
}

// Tile configurations (one translation unit each, see sgemm_cfg_*.cu).
using CfgL = Cfg<128, 128, 32, 8, 8, 3, 2>;  // 8 x 8 per thread, two CTAs per SM
using CfgM = Cfg<128, 64, 16, 8, 4, 4, 3>;   // 8 x 4 per thread (pairs along m), three CTAs per SM
using CfgS = Cfg<64, 64, 16, 4, 4, 4, 3>;    // 4 x 4 per thread, three CTAs per SM
// The 128 x 128 tile takes 32-wide K slices in 3 stages: half the per-slice barriers and ring
// turns of 16-wide slices (3% faster at 4096^3).  The 128 x 64 tile had them too (up to 7% at
// K = 4096 against swizzled 16-wide slices), but three CTAs per SM of padded 32-wide stages do
// not fit in shared memory, and padded 16-wide slices in 4 stages beat both (768 x 1024 x 513:
// 41.6 -> 35.6 us, 1536^2 x 513: 66.2 -> 62.1 us).  The 4 x 4 tile keeps 16-wide slices
// ([x][k] stages of four 16-byte chunks).
static_assert(CfgS::BK == 16, "the [x][k] fragment loads read 16-wide slices");

// Launchers defined in the configuration translation units.
cudaError_t launch_L(int dev_id, int a_mode, int b_mode, const SgemmParams &p, cudaStream_t s);
cudaError_t launch_LS(int dev_id, int a_mode, int b_mode, const SgemmParams &p, cudaStream_t s);
cudaError_t launch_M(int dev_id, int a_mode, int b_mode, const SgemmParams &p, cudaStream_t s);
cudaError_t launch_MS(int dev_id, int a_mode, int b_mode, const SgemmParams &p, cudaStream_t s);
cudaError_t launch_S(int dev_id, int a_mode, int b_mode, const SgemmParams &p, cudaStream_t s);
cudaError_t launch_SS(int dev_id, int a_mode, int b_mode, const SgemmParams &p, cudaStream_t s);
cudaError_t launch_SP(int dev_id, int a_mode, int b_mode, const SgemmParams &p, cudaStream_t s);

}  // namespace sg
}  // namespace gemm
