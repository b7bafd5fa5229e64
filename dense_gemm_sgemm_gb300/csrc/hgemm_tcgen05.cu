// fp16-input / fp32-accumulate GEMM on the tcgen05 tensor cores of sm_103a.
//
// C = alpha * op(A) * op(B) + beta * C with A, B in IEEE binary16 and C in fp32
// (copecc.github.io "GEMM" page, sections "核心问题与运算特征" and "Batched 执行与混合精度";
// dandandamowang.xyz "GEMM优化（二）": fp16 inputs, fp32 accumulator).  The pages reach the
// tensor cores through WMMA fragments on one warp at a time; on Blackwell the same
// contraction is issued by ONE thread as tcgen05.mma, with operands read straight from
// shared memory through matrix descriptors and the fp32 accumulator kept in tensor memory
// (TMEM).  The kernel is persistent and warp-specialised:
//
//   warp 0      TMA producer: one elected lane streams BK-wide K slices of the A and B
//               tiles into a shared-memory ring (cp.async.bulk.tensor with 128-byte
//               swizzle; the pages' cp.async double buffer of the "v4" section, moved to
//               the tensor-memory-access unit and deepened);
//   warp 1      MMA issuer and TMEM owner: allocates 512 TMEM columns (two 128 x 256 fp32
//               accumulators), issues 4 tcgen05.mma (K=16) per slice and returns each
//               slice to the producer with tcgen05.commit;
//   warps 2-5   epilogue: tcgen05.ld the finished accumulator (one TMEM lane = one row of
//               the tile), pass each 32 x 32 piece through a shared staging tile so that
//               C = alpha * acc + beta * C is read and written in 128-byte row segments,
//               while warp 1 already accumulates the next tile into the other buffer.
//
// Two forms.  PAIR = true (any problem of at least two 128-row tile rows): clusters of two
// CTAs on neighbouring SMs compute a 256 x 256 tile with tcgen05.mma.cta_group::2 (M=256,
// N=256).  Each CTA loads only its own 128 rows of A and its own 128 columns of B, a
// 32 KB stage per K slice, and the MMA reads the B halves of both CTAs: per SM this moves
// two thirds of the bytes of a one-CTA 128 x 256 tile through L2 and shared memory, and
// lets 6 stages fit.  Only the first CTA of the pair (rank 0) issues MMAs; both CTAs' TMA
// loads complete on its "full" barriers, and its commits release the "empty" barriers of
// both CTAs.  PAIR = false: one CTA computes a 128 x 256 tile with cta_group::1 MMAs from
// a 4-stage ring of 48 KB stages.
//
// WIDE (pairs, problems of at least a full wave with beta = 0): 256 x 512 pair tiles, two
// N = 256 MMAs per K step into one 512-column accumulator per CTA; each CTA loads 256 of the B
// columns (4 stages of 48 KB).  A quarter fewer bytes cross from L2 per flop -- the measured
// limit of the 256 x 256 tiles.  Each tile's epilogue no longer overlaps the next tile's
// MMAs, so it only stages C and leaves the stores to the TMA unit (cp.async.bulk.tensor),
// alternating two staging tiles per warp.
//
// The last, partial wave of tiles is split so that more SMs share it: into K halves whose
// fp32 partial sums are exchanged (each half finishes half of the tile's columns), or into
// N halves.
//
// Tiles are visited in the grouped raster of the copecc "线程块网格重排" section.  Ragged M,
// N and K need no special code: TMA fills out-of-range elements with zeros, which add
// nothing to the dot products, and the epilogue predicates its stores.
//
// Every wait on an mbarrier is bounded: when a wait expires the kernel records
// GEMM_ERR_DEVICE_TIMEOUT in g_device_status, stops all roles, waits (bounded) for its own
// copies and MMAs in flight, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "gemm_internal.h"

namespace gemm {

// Error word raised by kernels whose bounded barrier waits expire (0 = no error).
__device__ unsigned int g_device_status = 0;

namespace {

constexpr int BM = 128, BN = 256, BK = 64, UMMA_K = 16;  // BM: rows per CTA
constexpr int kThreads = 192;  // 6 warps
constexpr int kLdgThreads = 192;  // issuer warps 6-7 and fixer warps 8-11 of the loader form
template <bool LDG>
constexpr int threads_of() { return LDG ? kThreads + kLdgThreads : kThreads; }
constexpr int kAccCols = BN;        // fp32 columns per accumulator
constexpr int kTmemCols = 2 * BN;   // two accumulators
constexpr int A_STAGE_BYTES = BM * BK * 2;  // 16 KB
constexpr int EPI_BYTES = 4 * 32 * 32 * 4;  // a 32 x 32 fp32 staging tile per epilogue warp
constexpr int kBarBytes = 256;
constexpr int kLogGroup = 3;  // default raster group: 2^3 tile rows (or tile-pair rows)

// Ring geometry of the forms: a CTA of a pair holds half of the B columns.  The loader form
// keeps, per stage, a 16-byte side slot for every stage row (the ninth block of a row that is
// not 16-byte aligned), and fewer stages: its copies pass through the L1 data array, whose
// size -- what the shared-memory carve-out leaves of the 256 KB -- bounds the bytes they can
// have in flight (4 stages of a pair: 164 KB carve-out, 92 KB of L1).
// WIDE (pairs only): 256 x 512 pair tiles, each CTA holding 256 of the 512 B columns, 4 stages
// of 48 KB.
template <bool PAIR, bool LDG = false, bool WIDE = false>
struct Ring {
    static constexpr int kStages = WIDE ? 4 : LDG ? (PAIR ? 4 : 3) : (PAIR ? 6 : 4);
    static constexpr int kBRows = WIDE ? BN : PAIR ? BN / 2 : BN;
    static constexpr int kBStageBytes = kBRows * BK * 2;  // 16 KB or 32 KB
    static constexpr int kStageBytes = A_STAGE_BYTES + kBStageBytes;
    static constexpr int kSideBytes = LDG ? (BM + kBRows) * 16 : 0;  // per stage
    // TMA-read forms: two staging tiles per epilogue warp (TMA stores of C alternate between
    // them); the loader form stores C with plain stores from one
    static constexpr int kEpiBytes = LDG ? EPI_BYTES : 2 * EPI_BYTES;
    static constexpr int kSmemBytes =
        kStages * (kStageBytes + kSideBytes) + kEpiBytes + kBarBytes + 1024;  // + alignment slack
};
static_assert(Ring<true, false, true>::kSmemBytes <= 227 * 1024 &&
                  Ring<true>::kSmemBytes <= 227 * 1024 && Ring<false>::kSmemBytes <= 227 * 1024 &&
                  Ring<true, true>::kSmemBytes <= 227 * 1024 && Ring<false, true>::kSmemBytes <= 227 * 1024,
              "one CTA per SM within the 227 KB opt-in limit");
template <bool LDG>
constexpr int max_smem_of() { return Ring<true, LDG>::kSmemBytes > Ring<false, LDG>::kSmemBytes ? Ring<true, LDG>::kSmemBytes : Ring<false, LDG>::kSmemBytes; }
constexpr int kMaxSmemBytes = max_smem_of<false>() > max_smem_of<true>() ? max_smem_of<false>() : max_smem_of<true>();

struct HgemmParams {
    int64_t M, N, K;
    float *C;
    int64_t ldc;
    float alpha, beta;
    int64_t tiles_m, tiles_n, num_tiles;
    int num_kb;
    int c_vec;               // C base 16-byte aligned and ldc % 4 == 0
    uint64_t timeout_ns;     // limit of every barrier wait
    int inject_stall;        // test hook: 1 = the producer never fills the first slice of its
                             // first unit; 2 = nor of a first K half of the tail
    // Work units.  Units [0, full_tiles) are whole 128 x 256 tiles over all of K.  Each tile
    // of the last, partial wave becomes two units, so twice as many SMs share that wave:
    //   tail_mode kTailN: the left and right 128 x 128 halves (every element still summed by
    //     one CTA over all of K, so no result bit changes);
    //   tail_mode kTailK: the first and second half of the K slices.  Each half stores in ws
    //     its fp32 partial sums of the other half's 128 columns, waits for the other half's
    //     arrival (counters), adds the other half's partial to its own columns and writes
    //     them: every element is the sum of the two K halves' partial sums, the same bits
    //     whichever half adds.
    // Every K slice costs the ring's round-trip latency whatever the unit's width, so K
    // halves finish the wave in half the time and N halves do not.
    int64_t full_tiles, num_units;
    int tail_mode;
    float *ws;               // kTailK: 2 partial tiles per split tile (per CTA of a cluster)
    unsigned int *counters;  // kTailK: one arrival counter per split tile, zero between launches
    // Strided batch: batch problems share M, N, K; work units count tiles (or tile pairs)
    // of every problem, problem b owning units [b * per_batch, (b + 1) * per_batch).
    int64_t batch, per_batch;
    int a_batched, b_batched;  // 0: the operand is shared by every problem (stride 0)
    int64_t stride_c;          // elements between consecutive C matrices
    uint32_t ab_format;        // instruction-descriptor input type: 0 = fp16, 1 = bf16
    int log_group;             // raster group of 2^log_group tile (pair) rows
    int tile_n;                // columns of a tile: 256, or 512 for the wide pair tiles
    int c_tma;                 // beta == 0, TMA-read operands: C is written by TMA stores through map_c
    // Operands the tensor-memory-access unit cannot read (base not 16-byte aligned, leading
    // dimension or batch stride not a multiple of 8 elements) are read by the loader warps:
    // pointer, leading dimension and batch stride of the stored matrix, in elements.
    int a_ldg, b_ldg;
    const uint16_t *a_ptr, *b_ptr;
    int64_t lda, ldb, stride_a, stride_b;
};

constexpr int kTailNone = 0, kTailN = 1, kTailK = 2;

// Work unit u: tile t, column offset and width within it, K slices [kb0, kb1), and for a
// K-half unit its half (0 or 1) and the index of its tile among the split tiles (else -1).
struct Unit {
    int64_t t, split_slot;
    int n_off, width, kb0, kb1, khalf;
};

__device__ __forceinline__ Unit decode_unit(const HgemmParams &p, int64_t u)
{
    Unit x{u, -1, 0, p.tile_n, 0, p.num_kb, -1};
    if (u >= p.full_tiles && p.tail_mode != kTailNone) {
        const int64_t r = u - p.full_tiles;
        const int h = static_cast<int>(r & 1);
        x.t = p.full_tiles + (r >> 1);
        if (p.tail_mode == kTailN) {
            x.n_off = h * (BN / 2);
            x.width = BN / 2;
        } else {
            const int mid = p.num_kb / 2;
            x.kb0 = h ? mid : 0;
            x.kb1 = h ? p.num_kb : mid;
            x.khalf = h;
            x.split_slot = r >> 1;
        }
    }
    return x;
}

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// CLUSTER: acquire at cluster scope, for phases completed by release arrivals of threads of
// the other CTA of a pair.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    if constexpr (CLUSTER)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    return ok != 0;
}

// Waits for the phase of parity `parity` to complete.  Gives up (returns false) when the
// CTA-wide abort flag is raised or after timeout_ns nanoseconds.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int *abort_flag,
                                          uint64_t timeout_ns)
{
    if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > timeout_ns) return false;
        }
    }
}

// OR of `pred` over the 128 threads of the four epilogue warps (named barrier 1); every one
// of them must call it.
__device__ __forceinline__ bool epilogue_any(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void raise_abort(volatile int *abort_flag)
{
    *abort_flag = 1;
    atomicOr(&g_device_status, 1u);
}

// Box of a 3-D tensor map (columns, rows, problem of the batch) into shared memory.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Store of a box of shared memory at `src` to a 3-D tensor (C), tracked by this thread's bulk
// async-groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int32_t c0, int32_t c1, int32_t c2)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// The same copy issued by a CTA of a two-CTA pair whose completion is counted on an
// mbarrier that may sit in either CTA of the pair (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int32_t c0, int32_t c1, int32_t c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// shared::cluster address of the variable at shared::cta address `addr` in CTA `rank` of
// this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive (release at cluster scope) on an mbarrier given by its shared::cluster address,
// which may be in another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc], fp16/bf16 inputs, fp32 accumulate.  PAIR:
// issued by rank 0 of a CTA pair for both CTAs (M = 256: each CTA's descriptors name its
// own 128 rows of A and its own half of the B columns at the same shared-memory offsets;
// each CTA's TMEM receives its own 128 rows of D).
template <bool PAIR>
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    if constexpr (PAIR) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}

// Arrives on the mbarrier at shared::cluster address `bar` (this CTA's or, for a pair, the
// peer's) once every tcgen05.mma issued so far by this thread has completed.
template <bool PAIR>
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    if constexpr (PAIR)
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
    else
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
}

// TMEM allocation by one whole warp; for a pair, one warp of each CTA calls it together and
// both receive the same columns.
template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t cols)
{
    if constexpr (PAIR) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
}

template <bool PAIR>
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t cols)
{
    if constexpr (PAIR)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld_32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns of this thread's TMEM lane (one load round trip).
__device__ __forceinline__ void tmem_ld_64(uint32_t taddr, float (&v)[64])
{
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a tcgen05 operand tile stored with the 128-byte
// swizzle (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B):
//   bits  0-13 start address >> 4       bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4  bits 46-47 descriptor version (1)
//   bits 49-51 base offset (0: tiles are 1024-byte aligned)
//   bits 61-63 layout (2 = 128-byte swizzle)
// K-major tiles (rows along M or N, 64 fp16 of K per 128-byte row): the stride byte
// offset is the distance between 8-row groups (1024 bytes); the leading offset is unused.
// MN-major tiles (rows along K, 64 fp16 of M or N per row): the leading byte offset is the
// distance between 64-element column blocks, the stride byte offset between 8-row groups.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t((addr >> 4) & 0x3FFFu)) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of kind::f16: D fp32 (bits 4-5 = 1), A and B fp16 (bits 7-9 and
// 10-12 = 0), A/B major-ness in bits 15/16 (0 = K-major, 1 = MN-major), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28 (M = 128 for one CTA, 256 for a pair).
__host__ __device__ constexpr uint32_t make_idesc(int a_mn, int b_mn, int n, int m)
{
    return (1u << 4) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
           (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

// ------------------------------------------------------------------ loader warps
// For an operand whose rows TMA cannot address (its copies need a 16-byte aligned base and
// 16-byte multiples as row and batch strides), the loader form of the kernel fills the same
// swizzled stages as TMA would, in two roles:
//   issuer warps 6-7  copy each stage row as the aligned 16-byte blocks that cover it with
//                     cp.async (the cp.async producer of dandandamowang "GEMM优化（二）",
//                     section 5 (v4)); completion is counted on the stage's "copied" barrier
//                     (cp.async.mbarrier.arrive), so they never wait for their own copies and
//                     run ahead as far as the ring has free slots;
//   fixer warps 8-11  wait for a stage's copies, shift the rows that do not start on a 16-byte
//                     boundary into place, order the stage before the tensor cores' reads
//                     (proxy fence) and announce it on the (rank 0) full barrier.
// Both roles decide row by row with the same functions below, so they agree on which rows
// were copied as blocks and which need shifting.
constexpr int kIssuers = 64, kFixers = 128;

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t dst, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t src)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(src)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ldg_u16(const uint16_t *p)
{
    return __ldcg(reinterpret_cast<const unsigned short *>(p));
}

// OR of `pred` over the COUNT threads of named barrier ID; every one of them must call it.
template <int ID, int COUNT>
__device__ __forceinline__ bool group_any(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "n"(ID), "n"(COUNT)
        : "memory");
    return r != 0;
}

// Stage row r of an operand for the K slice at k0 holds 64 elements of one row of the stored
// matrix `mat` (leading dimension ld): for a K-major operand (MN = false) row `first + r` from
// column k0, for an MN-major one row k0 + r % 64 from column first + 64 (r / 64) -- the boxes
// TMA would copy.  Chunk c of row r belongs at dst + 128 r + 16 (c ^ (r % 8)), the 128-byte
// swizzle of the tensor maps.  Elements outside the stored matrix (mn x K for K-major, K x mn
// for MN-major) are zeros.  A row entirely inside the matrix is copied as the aligned 16-byte
// blocks that cover it: block b into the place of chunk b and, when the row starts delta > 0
// bytes into a block ("shifted"), block 8 into side + 16 r.  These blocks reach up to 14 bytes
// before and 16 after the row's 128, always inside the operand's own storage
// [mat, mat + (rows - 1) ld + cols) -- a row whose blocks would not be (at the very start or
// end of that storage), and a row cut by the matrix edge, is read element by element.
struct RowPlan {
    uintptr_t a0;      // first block
    int64_t grow, gcol;  // stored row and column of the row's element 0
    int64_t left;      // elements of the row inside the matrix from gcol (0: outside)
    bool blocks, shifted;
};

template <bool MN>
__device__ __forceinline__ RowPlan row_plan(const uint16_t *mat, int64_t ld, int64_t mn, int64_t K, int64_t first,
                                            int64_t k0, int r)
{
    const int64_t rows_total = MN ? K : mn, cols_total = MN ? mn : K;
    RowPlan x;
    x.grow = MN ? k0 + (r & 63) : first + r;
    x.gcol = MN ? first + 64 * (r >> 6) : k0;
    x.left = x.grow < rows_total ? cols_total - x.gcol : 0;
    const uintptr_t s = reinterpret_cast<uintptr_t>(mat + x.grow * ld + x.gcol);
    x.a0 = s & ~uintptr_t(15);
    const uintptr_t lo = reinterpret_cast<uintptr_t>(mat);
    const uintptr_t hi = lo + 2u * uintptr_t((rows_total - 1) * ld + cols_total);
    x.blocks = x.left >= 64 && (x.a0 == s || (x.a0 >= lo && x.a0 + 144u <= hi));
    x.shifted = x.blocks && x.a0 != s;
    return x;
}

// True when every row of the R-row box is inside the matrix and its blocks inside the
// storage: the rows need no individual checks.
template <bool MN>
__device__ __forceinline__ bool box_interior(int64_t mn, int64_t K, int64_t first, int64_t k0, int R)
{
    return MN ? (k0 + 64 <= K && first + 64 * (R / 64) <= mn && (k0 > 0 || first >= 8) &&
                 (k0 + 64 < K || first + 64 * (R / 64) + 8 <= mn))
              : (first + R <= mn && k0 + 64 <= K && (first > 0 || k0 >= 8) && (first + R < mn || k0 + 72 <= K));
}

// Issuer thread ti (0..63) copies chunk c = ti % 8 of rows ti / 8 + 8 i, i < R / 8.  Rows
// congruent modulo 8 lie a multiple of 16 bytes apart (16 ld bytes, or 128 across MN-major
// boxes), so all of this thread's rows share one offset within a 16-byte block.  Rows read
// element by element are stored before this returns (in groups of 8 chunks, so the loads of
// a group are in flight together).
template <bool MN, int R>
__device__ __forceinline__ void ldg_issue(uint32_t dst, uint32_t side, const uint16_t *mat, int64_t ld,
                                          int64_t mn, int64_t K, int64_t first, int64_t k0, int ti)
{
    constexpr int N = R / 8;  // rows of this thread
    const int c = ti & 7, rho = ti >> 3;
    if (box_interior<MN>(mn, K, first, k0, R)) {
        const uintptr_t s = reinterpret_cast<uintptr_t>(MN ? mat + (k0 + rho) * ld + first : mat + (first + rho) * ld + k0);
        const uintptr_t a0 = s & ~uintptr_t(15);
        const uintptr_t ld16 = 16u * uintptr_t(ld);  // bytes between rows 8 apart
        const bool shifted = a0 != s;
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const int r = rho + 8 * i;
            const uintptr_t a = a0 + (MN ? uintptr_t(i & 7) * ld16 + uintptr_t(i >> 3) * 128u : uintptr_t(i) * ld16);
            cp_async_16(dst + uint32_t(r) * 128u + (uint32_t(c ^ rho) << 4), reinterpret_cast<const void *>(a + 16u * c));
            if (shifted && c == 7) cp_async_16(side + 16u * uint32_t(r), reinterpret_cast<const void *>(a + 128u));
        }
        return;
    }
#pragma unroll
    for (int i0 = 0; i0 < N; i0 += 8) {
        uint4 v[8];
        uint32_t store = 0;
#pragma unroll
        for (int j = 0; j < 8 && i0 + j < N; ++j) {
            const int r = rho + 8 * (i0 + j);
            const RowPlan x = row_plan<MN>(mat, ld, mn, K, first, k0, r);
            const uint32_t sdst = dst + uint32_t(r) * 128u + (uint32_t(c ^ rho) << 4);
            v[j] = make_uint4(0u, 0u, 0u, 0u);
            if (x.blocks) {
                cp_async_16(sdst, reinterpret_cast<const void *>(x.a0 + 16u * c));
                if (x.shifted && c == 7) cp_async_16(side + 16u * uint32_t(r), reinterpret_cast<const void *>(x.a0 + 128u));
                continue;
            }
            const int64_t left = x.left - 8 * c;
            const int nv = left <= 0 ? 0 : left >= 8 ? 8 : int(left);
            if (nv > 0) {
                const uint16_t *src = mat + x.grow * ld + x.gcol + 8 * c;
                uint32_t e[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) e[k] = k < nv ? ldg_u16(src + k) : 0u;
                v[j] = make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
            }
            store |= 1u << j;
        }
#pragma unroll
        for (int j = 0; j < 8 && i0 + j < N; ++j)
            if ((store >> j) & 1u) {
                const int r = rho + 8 * (i0 + j);
                st_shared_v4(dst + uint32_t(r) * 128u + (uint32_t(c ^ rho) << 4), v[j]);
            }
    }
}

// Fixer thread tf (0..127, fixer warp w = tf / 32, lanes 8g..8g+7 one row) shifts, in
// iteration i < R / 16, row w + 4 (i % 2) + 8 (g + 4 (i / 2)) if it was copied shifted: chunk
// c = tf % 8 becomes bytes [delta, delta + 16) of block c followed by block c + 1 (block 8 from
// the side slot).  The rows of one warp instruction are congruent modulo 8 and share delta,
// so the word selection does not diverge; the eight lanes of a row read before any writes.
// Every fixer thread must call this.
template <bool MN, int R>
__device__ __forceinline__ void ldg_fix(uint32_t dst, uint32_t side, const uint16_t *mat, int64_t ld,
                                        int64_t mn, int64_t K, int64_t first, int64_t k0, int tf)
{
    const int w = tf >> 5, g = (tf >> 3) & 3, c = tf & 7;
    const bool interior = box_interior<MN>(mn, K, first, k0, R);
    // offset of residue rho's rows within their 16-byte blocks (the same in every row
    // congruent to rho modulo 8, see ldg_issue)
    const uint32_t mat_b = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(mat));
    const uint32_t seed = (MN ? mat_b + 2u * uint32_t(first) + 2u * uint32_t(ld) * uint32_t(k0)
                              : mat_b + 2u * uint32_t(ld) * uint32_t(first) + 2u * uint32_t(k0)) & 15u;
#pragma unroll
    for (int i = 0; i < R / 16; ++i) {
        const int rho = w + 4 * (i & 1), r = rho + 8 * (g + 4 * (i >> 1));
        const uint32_t delta = (seed + 2u * uint32_t(ld) * uint32_t(rho)) & 15u;
        const bool fix = interior ? delta != 0 : row_plan<MN>(mat, ld, mn, K, first, k0, r).shifted;
        const uint32_t pos = dst + uint32_t(r) * 128u + (uint32_t(c ^ rho) << 4);
        const uint32_t pos1 = c < 7 ? dst + uint32_t(r) * 128u + (uint32_t((c + 1) ^ rho) << 4)
                                    : side + 16u * uint32_t(r);
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (fix) {
            const uint4 x = ld_shared_v4(pos), y = ld_shared_v4(pos1);
            const uint32_t sh = (delta & 3u) * 8u;
            auto f = [sh](uint32_t lo, uint32_t hi) { return __funnelshift_r(lo, hi, sh); };
            switch (delta >> 2) {
            case 0: o = make_uint4(f(x.x, x.y), f(x.y, x.z), f(x.z, x.w), f(x.w, y.x)); break;
            case 1: o = make_uint4(f(x.y, x.z), f(x.z, x.w), f(x.w, y.x), f(y.x, y.y)); break;
            case 2: o = make_uint4(f(x.z, x.w), f(x.w, y.x), f(y.x, y.y), f(y.y, y.z)); break;
            default: o = make_uint4(f(x.w, y.x), f(y.x, y.y), f(y.y, y.z), f(y.z, y.w)); break;
            }
        }
        __syncwarp();
        if (fix) st_shared_v4(pos, o);
    }
}

// ------------------------------------------------------------------ the kernel
// PAIR = false: one CTA per 128 x 256 tile.  PAIR = true: units count tile pairs along M;
// the CTA of cluster rank r computes tile row 2 * pair_row + r, and rank 0 issues the
// pair's MMAs.  LDG = true: four more warps (6-9) load the operands flagged a_ldg / b_ldg
// into the ring themselves and warp 10 relays their slices to the MMA issuer; the producer
// warp still arms each slice and copies the other operand (if any) by TMA.
template <int A_MN, int B_MN, bool PAIR, bool LDG, bool WIDE = false>
__global__ void __launch_bounds__(threads_of<LDG>(), 1)
hgemm_tcgen05_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                     const __grid_constant__ CUtensorMap map_b_half,
                     const __grid_constant__ CUtensorMap map_b_quarter,
                     const __grid_constant__ CUtensorMap map_c, const HgemmParams p)
{
    static_assert(!WIDE || (PAIR && !LDG), "wide tiles: pairs of TMA-read operands");
    using R = Ring<PAIR, LDG, WIDE>;
    // WIDE: one 512-column accumulator (no double buffer: a tile's epilogue runs before the
    // next tile's MMAs), two N = 256 MMAs per K step
    constexpr int kAccs = WIDE ? 1 : 2;
    constexpr int kAccColsT = WIDE ? 2 * BN : kAccCols;
    constexpr int STAGES = R::kStages;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);

    const uint32_t sA = base;                                // STAGES x 16 KB
    const uint32_t sB = base + STAGES * A_STAGE_BYTES;       // STAGES x (16 or 32) KB
    float4 *epi_tiles = reinterpret_cast<float4 *>(smem + STAGES * R::kStageBytes);
    uint8_t *bar_area = smem + STAGES * R::kStageBytes + R::kEpiBytes;
    const uint32_t bar0 = smem_u32(bar_area);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bar_area + 8 * (2 * STAGES + 5));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 8 * (2 * STAGES + 5) + 4);
    // loader form: the issuer threads' arrivals (and the completion of their copies) of a slice
    auto copied_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 6 + s); };
    const uint32_t side0 = bar0 + kBarBytes;  // STAGES x kSideBytes (loader form)
    static_assert(8 * (3 * STAGES + 6) <= kBarBytes, "barrier area");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Unit schedule: CTAs (or pairs) stride over the units; the raster runs over tiles (or
    // tile pairs along M).
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const int64_t unit0 = PAIR ? int64_t(cluster_id_x()) : int64_t(blockIdx.x);
    const int64_t ustride = PAIR ? int64_t(cluster_count_x()) : int64_t(gridDim.x);
    const int64_t rows_r = PAIR ? (p.tiles_m + 1) / 2 : p.tiles_m;
    constexpr int kEpiArrivals = PAIR ? 8 : 4;  // one per epilogue warp of every CTA

    if (threadIdx.x == 0) {
        // the arming arrival of rank 0's producer, and with loader warps one arrival of the
        // fixer warps of each CTA once the loaders' part of the slice is in place
        constexpr uint32_t kFullArrivals = LDG ? 1u + (PAIR ? 2u : 1u) : 1u;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), kFullArrivals);
            mbar_init(empty_bar(s), 1);  // the MMA issuer's commit
            if (LDG) mbar_init(copied_bar(s), 2 * kIssuers);  // an arrival and a copy completion each
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), kEpiArrivals);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!(LDG && p.a_ldg)) tma_prefetch_desc(&map_a);
        if (!(LDG && p.b_ldg)) {
            tma_prefetch_desc(&map_b);
            tma_prefetch_desc(&map_b_half);
            tma_prefetch_desc(&map_b_quarter);
        }
    }
    // A pair allocates TMEM together, so the peer must be running; its barriers must also
    // exist before the other CTA's copies, commits and arrivals reach them.
    if (PAIR) cluster_sync();
    if (warp == 1) tmem_alloc<PAIR>(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
    tc_fence_before();
    // a pair: both CTAs hold their columns before rank 0's MMAs can write them
    if (PAIR) cluster_sync();
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const uint64_t tmo = p.timeout_ns;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (each CTA fills its own ring)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0, fill_parity = 0;  // per stage: a fill was issued / its parity
            bool ok = true;
            for (int64_t u = unit0; ok && u < p.num_units; u += ustride) {
                const Unit x = decode_unit(p, u);
                const int64_t t = x.t;
                const int n_off = x.n_off, width = x.width;
                int64_t tm, tn;
                const int64_t bt = t / p.per_batch;
                raster(t - bt * p.per_batch, rows_r, p.tiles_n, p.log_group, tm, tn);
                if (PAIR) tm = 2 * tm + rank;
                const int32_t ba = p.a_batched ? static_cast<int32_t>(bt) : 0;
                const int32_t bb = p.b_batched ? static_cast<int32_t>(bt) : 0;
                const int32_t m0 = static_cast<int32_t>(tm * BM);
                // a pair's CTA loads B columns [n0, n0 + bw) of the unit
                const int bw = PAIR ? width / 2 : width;
                const int32_t n0 = static_cast<int32_t>(tn * BN) + n_off + (PAIR ? int32_t(rank) * bw : 0);
                // bytes that complete a slice on the (rank 0) full barrier: both CTAs' for a
                // pair, of the operands copied by TMA
                const bool tma_a = !(LDG && p.a_ldg), tma_b = !(LDG && p.b_ldg);
                const uint32_t bytes = (PAIR ? 2u : 1u) * ((tma_a ? uint32_t(A_STAGE_BYTES) : 0u) +
                                                           (tma_b ? uint32_t(bw) * BK * 2 : 0u));
                for (int kb = x.kb0; kb < x.kb1; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, tmo)) {
                        raise_abort(abort_flag);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = PAIR ? map_to_rank(full_bar(stage), 0) : full_bar(stage);
                    if (rank == 0) mbar_expect_tx(full_bar(stage), bytes);
                    filled |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    const bool stall = kb == x.kb0 && ((p.inject_stall == 1 && u == unit0) ||
                                                       (p.inject_stall == 2 && x.khalf == 0));
                    if (!stall) {
                        const int32_t k0 = kb * BK;
                        const uint32_t a_dst = sA + stage * A_STAGE_BYTES;
                        const uint32_t b_dst = sB + stage * R::kBStageBytes;
                        auto load = [&](uint32_t dst, const CUtensorMap *map, int32_t c0, int32_t c1, int32_t c2) {
                            if (PAIR) tma_load_3d_pair(dst, map, fb, c0, c1, c2);
                            else tma_load_3d(dst, map, fb, c0, c1, c2);
                        };
                        if (!tma_a) {
                        } else if (A_MN) {  // A stored K x M: two 64 (m) x 64 (k) boxes
                            load(a_dst, &map_a, m0, k0, ba);
                            load(a_dst + 8192, &map_a, m0 + 64, k0, ba);
                        } else {     // A stored M x K: one 64 (k) x 128 (m) box
                            load(a_dst, &map_a, k0, m0, ba);
                        }
                        if (WIDE) {  // pieces h of 128 columns at tile columns 256 h + 128 rank
                            for (int h = 0; h < 2; ++h) {
                                const int32_t nb = static_cast<int32_t>(tn * (2 * BN)) + 256 * h + 128 * int32_t(rank);
                                if (B_MN) {
                                    load(b_dst + 16384 * h, &map_b, nb, k0, bb);
                                    load(b_dst + 16384 * h + 8192, &map_b, nb + 64, k0, bb);
                                } else {
                                    load(b_dst + 16384 * h, &map_b_half, k0, nb, bb);
                                }
                            }
                        } else if (!tma_b) {
                        } else if (B_MN) {  // B stored K x N: bw / 64 boxes of 64 (n) x 64 (k)
                            for (int j = 0; j < bw / 64; ++j) load(b_dst + 8192 * j, &map_b, n0 + 64 * j, k0, bb);
                        } else {     // B stored N x K: one 64 (k) x bw (n) box
                            load(b_dst, bw == BN ? &map_b : bw == BN / 2 ? &map_b_half : &map_b_quarter, k0, n0, bb);
                        }
                        if (bytes == 0) filled &= ~(1u << stage);  // no copy of this CTA's in flight
                    } else {
                        filled &= ~(1u << stage);  // nothing in flight on this slot
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                if (PAIR) {
                    // This CTA's copies complete on rank 0's barriers, which it cannot wait on:
                    // give the copies already issued time to land before its shared memory
                    // may go away (a TMA load of one stage takes microseconds).
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 2000000ull) {
                    }
                } else {
                    // Let the copies already issued land before the CTA's shared memory goes away.
                    for (int s = 0; s < STAGES; ++s)
                        if ((filled >> s) & 1u) {
                            const volatile int no_abort = 0;
                            mbar_wait(full_bar(s), (fill_parity >> s) & 1u, &no_abort, 100000000ull);
                        }
                }
            } else if (PAIR) {
                // Wait for the last release of every slot, so that no commit from rank 0 is
                // still on its way to this CTA's barriers when it exits.
                for (int i = 0; i < STAGES; ++i) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, tmo)) {
                        raise_abort(abort_flag);
                        break;
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (rank 0 of a pair issues for both CTAs)
            constexpr int kM = PAIR ? 2 * BM : BM;
            const uint32_t fmt = (p.ab_format << 7) | (p.ab_format << 10);  // A and B input type
            const uint32_t idesc_full = make_idesc(A_MN, B_MN, BN, kM) | fmt;
            const uint32_t idesc_half = make_idesc(A_MN, B_MN, BN / 2, kM) | fmt;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true, issued = false;
            for (int64_t u = unit0; ok && u < p.num_units; u += ustride) {
                const Unit x = decode_unit(p, u);
                const uint32_t idesc = (WIDE || x.width == BN) ? idesc_full : idesc_half;
                if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, abort_flag, tmo)) {
                    raise_abort(abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + uint32_t(acc * kAccColsT);
                for (int kb = x.kb0; kb < x.kb1; ++kb) {
                    // the peer's loader warps complete slices by release arrivals at cluster scope
                    if (!mbar_wait<LDG && PAIR>(full_bar(stage), phase, abort_flag, tmo)) {
                        raise_abort(abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_tile = sA + stage * A_STAGE_BYTES;
                    const uint32_t b_tile = sB + stage * R::kBStageBytes;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        // K-major: step 32 bytes along the swizzled 128-byte row.
                        // MN-major: step 16 rows of 128 bytes.
                        const uint64_t ad = A_MN ? smem_desc(a_tile + k * 2048, 8192, 1024)
                                                 : smem_desc(a_tile + k * 32, 16, 1024);
                        const uint32_t accumulate = (kb > x.kb0 || k > 0) ? 1u : 0u;
#pragma unroll
                        for (int h = 0; h < (WIDE ? 2 : 1); ++h) {  // WIDE: the two 256-column halves
                            const uint32_t bt = b_tile + 16384u * h;
                            const uint64_t bd = B_MN ? smem_desc(bt + k * 2048, 8192, 1024) : smem_desc(bt + k * 32, 16, 1024);
                            umma_f16<PAIR>(d_tmem + 256u * h, ad, bd, idesc, accumulate);
                        }
                    }
                    issued = true;
                    // the slot is free once these MMAs have read it (a pair: in both CTAs)
                    umma_commit<PAIR>(empty_bar(stage));
                    if (PAIR) umma_commit<PAIR>(map_to_rank(empty_bar(stage), 1));  // the peer's slot
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit<PAIR>(accf_bar(acc));  // accumulator complete
                if (PAIR) umma_commit<PAIR>(map_to_rank(accf_bar(acc), 1));
                if (++acc == kAccs) { acc = 0; acc_phase ^= 1u; }
            }
            if (!ok && issued) {
                // Wait for the MMAs in flight before TMEM is released.
                umma_commit<PAIR>(drain_bar);
                const volatile int no_abort = 0;
                mbar_wait(drain_bar, 0, &no_abort, 100000000ull);
            }
        }
    } else if (LDG && warp >= (kThreads + kIssuers) / 32) {
        // ---------------- fixer warps (loader form): wait for a slice's copies, shift its
        // unaligned rows into place, order the slice before the tensor cores' reads (proxy
        // fence; these threads have no copies of their own in flight) and announce it.
        const int tf = threadIdx.x - (kThreads + kIssuers);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int64_t u = unit0; ok && u < p.num_units; u += ustride) {
            const Unit x = decode_unit(p, u);
            int64_t tm, tn;
            const int64_t bt = x.t / p.per_batch;
            raster(x.t - bt * p.per_batch, rows_r, p.tiles_n, p.log_group, tm, tn);
            if (PAIR) tm = 2 * tm + rank;
            const int bw = PAIR ? x.width / 2 : x.width;
            const int64_t m0 = tm * BM;
            const int64_t n0 = tn * BN + x.n_off + (PAIR ? int64_t(rank) * bw : 0);
            const uint16_t *a_mat = p.a_ptr + (p.a_batched ? bt * p.stride_a : 0);
            const uint16_t *b_mat = p.b_ptr + (p.b_batched ? bt * p.stride_b : 0);
            for (int kb = x.kb0; kb < x.kb1; ++kb) {
                bool got = true;
                if (tf == 0) got = mbar_wait(copied_bar(stage), phase, abort_flag, tmo);
                if (group_any<3, kFixers>(!got)) {
                    if (tf == 0) raise_abort(abort_flag);
                    ok = false;
                    break;
                }
                const int64_t k0 = int64_t(kb) * BK;
                const uint32_t side = side0 + uint32_t(stage) * R::kSideBytes;
                if (p.a_ldg) ldg_fix<A_MN != 0, BM>(sA + stage * A_STAGE_BYTES, side, a_mat, p.lda, p.M, p.K, m0, k0, tf);
                if (p.b_ldg) {
                    const uint32_t b_dst = sB + stage * R::kBStageBytes, b_side = side + BM * 16;
                    if (bw == 256) ldg_fix<B_MN != 0, 256>(b_dst, b_side, b_mat, p.ldb, p.N, p.K, n0, k0, tf);
                    else if (bw == 128) ldg_fix<B_MN != 0, 128>(b_dst, b_side, b_mat, p.ldb, p.N, p.K, n0, k0, tf);
                    else ldg_fix<B_MN != 0, 64>(b_dst, b_side, b_mat, p.ldb, p.N, p.K, n0, k0, tf);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                asm volatile("bar.sync 3, %0;" ::"n"(kFixers) : "memory");
                if (tf == 0) {
                    if (PAIR) mbar_arrive_cluster(map_to_rank(full_bar(stage), 0));
                    else mbar_arrive(full_bar(stage));
                }
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
    } else if (LDG && warp >= kThreads / 32) {
        // ---------------- issuer warps (loader form): copy each slice once its slot is free;
        // the copies complete on the slot's copied barrier, so these warps never wait for them.
        const int ti = threadIdx.x - kThreads;
        int stage = 0;
        uint32_t phase = 0;
        for (int64_t u = unit0; u < p.num_units; u += ustride) {
            const Unit x = decode_unit(p, u);
            int64_t tm, tn;
            const int64_t bt = x.t / p.per_batch;
            raster(x.t - bt * p.per_batch, rows_r, p.tiles_n, p.log_group, tm, tn);
            if (PAIR) tm = 2 * tm + rank;
            const int bw = PAIR ? x.width / 2 : x.width;
            const int64_t m0 = tm * BM;
            const int64_t n0 = tn * BN + x.n_off + (PAIR ? int64_t(rank) * bw : 0);
            const uint16_t *a_mat = p.a_ptr + (p.a_batched ? bt * p.stride_a : 0);
            const uint16_t *b_mat = p.b_ptr + (p.b_batched ? bt * p.stride_b : 0);
            bool ok = true;
            for (int kb = x.kb0; kb < x.kb1; ++kb) {
                bool got = true;
                if (ti == 0) got = mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, tmo);
                if (group_any<2, kIssuers>(!got)) {
                    if (ti == 0) raise_abort(abort_flag);
                    ok = false;
                    break;
                }
                const int64_t k0 = int64_t(kb) * BK;
                const uint32_t side = side0 + uint32_t(stage) * R::kSideBytes;
                if (p.a_ldg) ldg_issue<A_MN != 0, BM>(sA + stage * A_STAGE_BYTES, side, a_mat, p.lda, p.M, p.K, m0, k0, ti);
                if (p.b_ldg) {
                    const uint32_t b_dst = sB + stage * R::kBStageBytes, b_side = side + BM * 16;
                    if (bw == 256) ldg_issue<B_MN != 0, 256>(b_dst, b_side, b_mat, p.ldb, p.N, p.K, n0, k0, ti);
                    else if (bw == 128) ldg_issue<B_MN != 0, 128>(b_dst, b_side, b_mat, p.ldb, p.N, p.K, n0, k0, ti);
                    else ldg_issue<B_MN != 0, 64>(b_dst, b_side, b_mat, p.ldb, p.N, p.K, n0, k0, ti);
                }
                // one arrival when this thread's copies have landed, one now (release of the
                // element-wise stores above)
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(copied_bar(stage)) : "memory");
                mbar_arrive(copied_bar(stage));
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
        }
        // no copy may land after the CTA's shared memory is gone
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    } else {
        // ---------------- epilogue (warps 2..5; TMEM lane quarter = warp % 4)
        const int quarter = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        int cbuf = 0;  // with TMA stores: the staging tile of the next chunk
        const float alpha = p.alpha, beta = p.beta;
        for (int64_t u = unit0; u < p.num_units; u += ustride) {
            const Unit x = decode_unit(p, u);
            const int64_t t = x.t;
            const int n_off = x.n_off, width = x.width;
            int64_t tm, tn;
            const int64_t bt = t / p.per_batch;
            raster(t - bt * p.per_batch, rows_r, p.tiles_n, p.log_group, tm, tn);
            if (PAIR) tm = 2 * tm + rank;
            // The four epilogue warps leave together or not at all: a K-half unit below
            // synchronises them, so none may have given up on a unit the others continue.
            const bool got = mbar_wait(accf_bar(acc), acc_phase, abort_flag, tmo);
            if (epilogue_any(!got)) {
                raise_abort(abort_flag);
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(acc * kAccColsT);
            // C = alpha * acc + beta * C for chunk c (32 columns) of the warp's 32 rows; v holds
            // this lane's row.  The rows go through the warp's staging tile (16-byte chunks
            // XOR-swizzled by row: conflict-free both ways), so that each store instruction
            // writes four 128-byte row segments instead of 32 scattered 16-byte pieces.
            float4 *tile = epi_tiles + quarter * 256 * (LDG ? 1 : 2);
            const int64_t row0 = tm * BM + quarter * 32;  // first row of this warp
            auto store_chunk = [&](int c, const float *v) {
                const int64_t gn0 = tn * p.tile_n + n_off + c * 32;
                if (gn0 >= p.N) return;  // the same for the whole warp
                if (!LDG && p.c_tma) {
                    // beta == 0: alpha * acc into one of the warp's two staging tiles (laid out
                    // as the tensor map's 128-byte swizzle), then one lane stores the 32 x 32
                    // box by TMA (clipped at the edges of C) while the warp goes on
                    float4 *tb = tile + 256 * cbuf;
                    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                    __syncwarp();  // the store that last read this tile has read it
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        tb[lane * 8 + (j ^ (lane & 7))] = make_float4(alpha * v[4 * j], alpha * v[4 * j + 1],
                                                                      alpha * v[4 * j + 2], alpha * v[4 * j + 3]);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&map_c, smem_u32(tb), static_cast<int32_t>(gn0), static_cast<int32_t>(row0),
                                     static_cast<int32_t>(bt));
                        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                    }
                    cbuf ^= 1;
                    return;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    tile[lane * 8 + (j ^ (lane & 7))] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                __syncwarp();
                const int q = lane & 7;
                const int64_t gn = gn0 + 4 * q;
                const bool vec = p.c_vec && gn + 3 < p.N;
                float *cbase = p.C + bt * p.stride_c + gn;
                // every read of C in flight before the first store
                float4 ci[8];
                if (vec && beta != 0.0f) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int64_t gm = row0 + 4 * i + (lane >> 3);
                        ci[i] = gm < p.M ? *reinterpret_cast<const float4 *>(cbase + gm * p.ldc)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = 4 * i + (lane >> 3);
                    const int64_t gm = row0 + r;
                    const float4 a = tile[r * 8 + (q ^ (r & 7))];
                    if (gm >= p.M) continue;
                    float *dst = cbase + gm * p.ldc;
                    if (vec) {
                        float4 o;
                        if (beta != 0.0f) {
                            o = make_float4(fmaf(alpha, a.x, beta * ci[i].x), fmaf(alpha, a.y, beta * ci[i].y),
                                            fmaf(alpha, a.z, beta * ci[i].z), fmaf(alpha, a.w, beta * ci[i].w));
                        } else {
                            o = make_float4(alpha * a.x, alpha * a.y, alpha * a.z, alpha * a.w);
                        }
                        *reinterpret_cast<float4 *>(dst) = o;
                    } else {
                        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            if (gn + jj < p.N)
                                dst[jj] = beta != 0.0f ? fmaf(alpha, av[jj], beta * dst[jj]) : alpha * av[jj];
                    }
                }
                __syncwarp();  // the tile is read before the next chunk overwrites it
            };
            if (x.khalf < 0 && LDG) {
#pragma unroll 1
                for (int c = 0; c < width / 32; ++c) {
                    float v[32];
                    __syncwarp();  // tcgen05.ld is warp-collective: reconverge after the predicated stores
                    tmem_ld_32(taddr + c * 32, v);
                    store_chunk(c, v);
                }
            } else if (x.khalf < 0) {
                // 64 columns per TMEM load round trip (every unit width is a multiple of 64; the
                // loader form, limited to 168 registers a thread, keeps 32)
#pragma unroll 1
                for (int c = 0; c < width / 32; c += 2) {
                    float v[64];
                    __syncwarp();
                    tmem_ld_64(taddr + c * 32, v);
                    store_chunk(c, v);
                    store_chunk(c + 1, v + 32);
                }
            } else {
                // K half h finishes columns [128 h, 128 h + 128) of the tile.  It publishes
                // its partial sums of the other half's columns, counts its arrival, waits
                // (bounded) for the other K half's arrival, copies that half's partial of
                // its own columns into the operand ring -- idle now: a split unit is its
                // CTA's last unit and every load into the ring has landed -- with 16-byte
                // cp.async, adds it and writes C.  Partials are thread-major (float4 q of
                // epilogue thread e at q * 128 + e), so every warp access is 512 contiguous
                // bytes.  Both halves belong to this grid, which never exceeds the resident
                // capacity, so the wait ends unless a fault aborts the kernel.
                const int e = threadIdx.x - 64;
                const int h = x.khalf;
                const int64_t slot = PAIR ? 2 * x.split_slot + rank : x.split_slot;
                constexpr int QH = BN / 8;  // float4 per row of a half tile
                float4 *mine = reinterpret_cast<float4 *>(p.ws) + (slot * 2 + h) * (QH * 128) + e;
                const float4 *other = reinterpret_cast<const float4 *>(p.ws) + (slot * 2 + (h ^ 1)) * (QH * 128) + e;
#pragma unroll 1
                for (int cc = 0; cc < BN / 64; ++cc) {
                    float v[32];
                    __syncwarp();
                    tmem_ld_32(taddr + ((h ^ 1) * (BN / 64) + cc) * 32, v);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        __stcg(mine + (cc * 8 + j) * 128, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps' partials
                bool failed = false;
                if (threadIdx.x == 64) {
                    unsigned int *ctr = p.counters + slot;
                    __threadfence();  // release this CTA's partial (cumulative over the barrier)
                    atomicAdd(ctr, 1u);
                    const uint64_t t0 = global_timer_ns();
                    for (uint32_t it = 0;; ++it) {
                        uint32_t seen;
                        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(ctr) : "memory");
                        if (seen >= 2u) break;
                        if ((it & 15u) == 0 && (*abort_flag || global_timer_ns() - t0 > tmo)) {
                            failed = true;
                            break;
                        }
                    }
                    if (!failed) {
                        __threadfence();  // acquire the other half's partial for the whole CTA
                        // both halves have seen both arrivals: the second to get here resets
                        if (atomicAdd(ctr, 1u) == 3u) *ctr = 0u;
                    }
                }
                if (epilogue_any(failed)) {
                    raise_abort(abort_flag);
                } else {
                    static_assert(QH * 128 * 16 <= STAGES * R::kStageBytes, "the ring holds a partial half tile");
                    const uint32_t stage_dst = sA + uint32_t(e) * 16u;
#pragma unroll 8
                    for (int q = 0; q < QH; ++q)
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(stage_dst + uint32_t(q) * 2048u),
                                     "l"(other + q * 128)
                                     : "memory");
                    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
                    const float4 *staged = reinterpret_cast<const float4 *>(smem) + e;
#pragma unroll 1
                    for (int cc = 0; cc < BN / 64; ++cc) {
                        const int c = h * (BN / 64) + cc;
                        float v[32];
                        __syncwarp();
                        tmem_ld_32(taddr + c * 32, v);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 o = staged[(cc * 8 + j) * 128];
                            v[4 * j] += o.x; v[4 * j + 1] += o.y; v[4 * j + 2] += o.z; v[4 * j + 3] += o.w;
                        }
                        store_chunk(c, v);
                    }
                }
            }
            // accumulator may be overwritten: one arrival per warp on the issuer's barrier
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR) mbar_arrive_cluster(map_to_rank(acce_bar(acc), 0));
                else mbar_arrive(acce_bar(acc));
            }
            if (++acc == kAccs) { acc = 0; acc_phase ^= 1u; }
        }
        // every TMA store of C has completed (and read its staging tile) before the CTA ends
        if (!LDG && p.c_tma && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // neither CTA leaves or frees TMEM while the other may still use it
    tc_fence_after();
    if (warp == 1) tmem_free<PAIR>(tmem_base, kTmemCols);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    });
    return fn;
}

// 3-D tensor map over `batch` row-major matrices of `rows` x `cols` (cols contiguous) with
// leading dimension ld, `bstride` elements apart, read in boxes of box_cols x box_rows x 1
// with the 128-byte swizzle.  A shared operand (bstride 0) is one matrix (batch extent 1).
bool make_map(CUtensorMap *map, const uint16_t *ptr, int64_t rows, int64_t cols, int64_t ld,
              uint32_t box_cols, uint32_t box_rows, int64_t batch, int64_t bstride, int bf16)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const bool shared = bstride == 0 || batch <= 1;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(shared ? 1 : batch)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2,
                                   static_cast<cuuint64_t>(shared ? ld : bstride) * 2};
    const cuuint32_t box[3] = {box_cols, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
              const_cast<uint16_t *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Maps {
    CUtensorMap a, b, b_half, b_quarter, c;
};

// 3-D tensor map over `batch` row-major fp32 matrices M x N (leading dimension ldc, `bstride`
// elements apart) written in 32 x 32 boxes with the 128-byte swizzle (the layout of the
// epilogue's staging tiles).
bool make_map_c(CUtensorMap *map, float *ptr, int64_t M, int64_t N, int64_t ldc, int64_t batch, int64_t bstride)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const bool single = bstride == 0 || batch <= 1;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M),
                                static_cast<cuuint64_t>(single ? 1 : batch)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldc) * 4,
                                   static_cast<cuuint64_t>(single ? ldc * M : bstride) * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// Largest number of two-CTA clusters of the pair kernel that can be resident at once (0: none).
template <int A_MN, int B_MN, bool LDG, bool WIDE = false>
int max_pair_clusters(int dev_id)
{
    static std::atomic<int> cached[64];
    static std::atomic<uint64_t> known{0};
    const uint64_t bit = uint64_t(1) << (dev_id & 63);
    if (known.load(std::memory_order_acquire) & bit) return cached[dev_id & 63].load();
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(threads_of<LDG>(), 1, 1);
    cfg.dynamicSmemBytes = Ring<true, LDG, WIDE>::kSmemBytes;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, hgemm_tcgen05_kernel<A_MN, B_MN, true, LDG, WIDE>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cached[dev_id & 63].store(n);
    known.fetch_or(bit, std::memory_order_release);
    return n;
}

template <int A_MN, int B_MN, bool PAIR, bool LDG, bool WIDE = false>
cudaError_t set_smem_attr(int dev_id)
{
    static std::atomic<uint64_t> attr_set{0};
    const uint64_t bit = uint64_t(1) << (dev_id & 63);
    if (attr_set.load(std::memory_order_acquire) & bit) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(hgemm_tcgen05_kernel<A_MN, B_MN, PAIR, LDG, WIDE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Ring<PAIR, LDG, WIDE>::kSmemBytes);
    if (e == cudaSuccess) attr_set.fetch_or(bit, std::memory_order_release);
    return e;
}

// Plans the unit schedule and launches.  With pairs, units are tile pairs along M.
template <int A_MN, int B_MN, bool LDG>
cudaError_t launch_t(const DeviceInfo &dev, const Maps &m, HgemmParams p, cudaStream_t stream)
{
    // GEMM_GB300_HGEMM_PAIR=0: one CTA per tile even where pairs would be used
    const char *pair_env = std::getenv("GEMM_GB300_HGEMM_PAIR");
    // GEMM_GB300_HGEMM_TAIL: "0" no tail split, "n" N halves, otherwise the rule below
    const char *tail_env = std::getenv("GEMM_GB300_HGEMM_TAIL");
    const char tail_want = tail_env && tail_env[0] ? tail_env[0] : 'a';
    bool pair = p.tiles_m >= 2 && !(pair_env && pair_env[0] == '0');
    int max_clusters = 0;
    if (pair) {
        if (set_smem_attr<A_MN, B_MN, true, LDG>(dev.device) != cudaSuccess) return cudaGetLastError();
        max_clusters = max_pair_clusters<A_MN, B_MN, LDG>(dev.device);
        pair = max_clusters > 0;
    }
    // Wide pair tiles (256 x 512): a quarter less L2-to-SM traffic per flop, but the single
    // 512-column accumulator leaves each tile's epilogue exposed.  Used when beta == 0 and C
    // can be written by TMA stores (16-byte aligned, ldc and batch stride multiples of 4), so
    // the epilogue hands its stores to the TMA unit and returns the accumulator quickly (with
    // beta = 1 and plain stores 16384 x 4096 x 4096 ran 21% slower), when there is at least one
    // full wave of wide tiles, and when their waves take no longer than the 256 x 256 tiles'.
    // A wide tile costs 1.75 pair tiles (measured: 4096^3 1.75, 8192^3 1.79); the pair tiles'
    // partial last wave costs half a tile in K halves (below), a whole one otherwise; the wide
    // tiles' last wave is not split.  So 8192^3 takes wide tiles (7 waves, 12.25 pair-tile
    // times against 13.5), 4096 x 2560 does not (2 waves, 3.5 against 2.5).
    // GEMM_GB300_HGEMM_WIDE=0 never, =1 whenever pairs are used (for tests).
    if (!LDG && pair && p.tile_n == BN) {
        const char *wide_env = std::getenv("GEMM_GB300_HGEMM_WIDE");
        const char want = wide_env && wide_env[0] ? wide_env[0] : 'a';
        const int64_t per_batch_w = ((p.tiles_m + 1) / 2) * ((p.N + 2 * BN - 1) / (2 * BN));
        const int64_t work_w = per_batch_w * p.batch;
        const int64_t wc = max_clusters;
        const int64_t work_n = ((p.tiles_m + 1) / 2) * p.tiles_n * p.batch;
        const int64_t full_n = work_n / wc, tail_n = work_n % wc;
        const double waves_n = double(full_n) + (tail_n == 0 ? 0.0 : (2 * tail_n <= wc && p.num_kb >= 8) ? 0.5 : 1.0);
        const double waves_w = 1.75 * double((work_w + wc - 1) / wc);
        const bool c_tma_ok = p.c_tma != 0;
        if (want != '0' && (want == '1' || (c_tma_ok && work_w >= wc && waves_w <= waves_n)) &&
            set_smem_attr<A_MN, B_MN, true, false, true>(dev.device) == cudaSuccess) {
            const int max_w = max_pair_clusters<A_MN, B_MN, false, true>(dev.device);
            if (max_w > 0) {
                p.tile_n = 2 * BN;
                p.tiles_n = (p.N + 2 * BN - 1) / (2 * BN);
                const Maps &mw = m;
                p.per_batch = per_batch_w;
                p.full_tiles = work_w;
                p.num_units = work_w;
                p.tail_mode = kTailNone;
                const int64_t clusters = work_w < max_w ? work_w : max_w;
                cudaLaunchConfig_t cfg{};
                cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
                cfg.blockDim = dim3(kThreads, 1, 1);
                cfg.dynamicSmemBytes = Ring<true, false, true>::kSmemBytes;
                cfg.stream = stream;
                cudaLaunchAttribute attr{};
                attr.id = cudaLaunchAttributeClusterDimension;
                attr.val.clusterDim.x = 2;
                attr.val.clusterDim.y = 1;
                attr.val.clusterDim.z = 1;
                cfg.attrs = &attr;
                cfg.numAttrs = 1;
                const cudaError_t e = cudaLaunchKernelEx(&cfg, hgemm_tcgen05_kernel<A_MN, B_MN, true, false, true>, mw.a,
                                                         mw.b, mw.b_half, mw.b_quarter, mw.c, p);
                if (e == cudaSuccess) count_launches();
                return e;
            }
        } else {
            cudaGetLastError();
        }
    }
    // Whole tiles (or pairs) for the full waves; when the last wave would leave more than
    // half of the workers idle, its tiles are split in two units each: K halves when there
    // are at least 8 K slices and the stream's workspace holds the partial tiles, else N
    // halves.
    p.per_batch = pair ? ((p.tiles_m + 1) / 2) * p.tiles_n : p.num_tiles;
    const int64_t work = p.per_batch * p.batch;
    const int64_t workers_max = pair ? max_clusters : dev.num_sms;
    const int64_t workers = work < workers_max ? work : workers_max;
    p.full_tiles = work;
    p.num_units = work;
    p.tail_mode = kTailNone;
    const int64_t full = (work / workers) * workers, tail = work - full;
    if (tail > 0 && 2 * tail <= workers && tail_want != '0') {
        const int64_t split_tiles = tail * (pair ? 2 : 1);  // CTA tiles of the split units
        StreamWorkspace w;
        if (tail_want != 'n' && p.num_kb >= 8 && split_tiles <= int64_t(kWorkspaceCounters) &&
            size_t(split_tiles) * 2 * BM * BN * sizeof(float) <= kWorkspaceBytes &&
            stream_workspace(dev.device, stream, w)) {
            p.tail_mode = kTailK;
            p.ws = w.data;
            p.counters = w.counters;
        } else {
            p.tail_mode = kTailN;
        }
        p.full_tiles = full;
        p.num_units = full + 2 * tail;
    }
    if (!pair) {
        cudaError_t e = set_smem_attr<A_MN, B_MN, false, LDG>(dev.device);
        if (e != cudaSuccess) return e;
        hgemm_tcgen05_kernel<A_MN, B_MN, false, LDG>
            <<<static_cast<unsigned>(workers), threads_of<LDG>(), Ring<false, LDG>::kSmemBytes, stream>>>(
                m.a, m.b, m.b_half, m.b_quarter, m.c, p);
        const cudaError_t le = cudaGetLastError();
        if (le == cudaSuccess) count_launches();
        return le;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * workers), 1, 1);
    cfg.blockDim = dim3(threads_of<LDG>(), 1, 1);
    cfg.dynamicSmemBytes = Ring<true, LDG>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, hgemm_tcgen05_kernel<A_MN, B_MN, true, LDG>, m.a, m.b, m.b_half,
                                             m.b_quarter, m.c, p);
    if (e == cudaSuccess) count_launches();
    return e;
}

}  // namespace

gemm_status_t launch_hgemm(const DeviceInfo &dev, int dtype, int opA, int opB, int64_t M, int64_t N,
                           int64_t K, float alpha, const uint16_t *A, int64_t lda, int64_t strideA,
                           const uint16_t *B, int64_t ldb, int64_t strideB, float beta, float *C,
                           int64_t ldc, int64_t strideC, int64_t batch, cudaStream_t stream)
{
    if (dev.smem_optin < size_t(kMaxSmemBytes)) return GEMM_ERR_NO_DEVICE;
    const int a_mn = opA == GEMM_OP_T;  // A stored K x M
    const int b_mn = opB == GEMM_OP_N;  // B stored K x N
    const int bf = dtype == kInBf16;
    // An operand TMA can read: 16-byte aligned base, leading dimension and batch stride
    // multiples of 8 elements (16 bytes).  Any other 2-byte aligned operand goes through the
    // loader warps (odd byte addresses are refused before this point).
    auto tma_ok = [&](const void *ptr, int64_t ld, int64_t stride) {
        return reinterpret_cast<uintptr_t>(ptr) % 16 == 0 && ld % 8 == 0 && (batch <= 1 || stride % 8 == 0);
    };
    const bool a_ldg = !tma_ok(A, lda, strideA), b_ldg = !tma_ok(B, ldb, strideB);
    Maps m;
    std::memset(&m, 0, sizeof(m));
    bool ok_a = true, ok_b = true;
    if (!a_ldg)
        ok_a = a_mn ? make_map(&m.a, A, K, M, lda, 64, BK, batch, strideA, bf)
                    : make_map(&m.a, A, M, K, lda, BK, BM, batch, strideA, bf);
    if (b_ldg) {
    } else if (b_mn) {  // 64 (n) x 64 (k) boxes serve every unit width
        ok_b = make_map(&m.b, B, K, N, ldb, 64, BK, batch, strideB, bf);
        m.b_half = m.b;
        m.b_quarter = m.b;
    } else {     // B stored N x K: boxes of 256, 128 and 64 rows
        ok_b = make_map(&m.b, B, N, K, ldb, BK, BN, batch, strideB, bf) &&
               make_map(&m.b_half, B, N, K, ldb, BK, BN / 2, batch, strideB, bf) &&
               make_map(&m.b_quarter, B, N, K, ldb, BK, BN / 4, batch, strideB, bf);
    }
    if (!ok_a || !ok_b) return GEMM_ERR_MISALIGNED;
    const bool c_vec = (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (ldc % 4 == 0) && (batch <= 1 || strideC % 4 == 0);
    // beta == 0 with operands read by TMA: the epilogue writes C by TMA stores.  Only when N is
    // a multiple of 4 as well: a store box cut by the right edge of C is written in whole
    // 16-byte pieces (measured: with N = 383 and ldc = 384 the padding column 383 was written),
    // so every piece must lie inside or outside C.
    const bool c_tma = !a_ldg && !b_ldg && beta == 0.0f && c_vec && N % 4 == 0 &&
                       make_map_c(&m.c, C, M, N, ldc, batch, batch > 1 ? strideC : 0);

    HgemmParams p{};
    p.M = M; p.N = N; p.K = K;
    p.C = C; p.ldc = ldc;
    p.alpha = alpha; p.beta = beta;
    p.tiles_m = (M + BM - 1) / BM;
    p.tiles_n = (N + BN - 1) / BN;
    p.num_tiles = p.tiles_m * p.tiles_n;
    p.num_kb = static_cast<int>((K + BK - 1) / BK);
    p.c_vec = (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (ldc % 4 == 0) && (batch <= 1 || strideC % 4 == 0);
    p.batch = batch;
    p.a_batched = batch > 1 && strideA != 0;
    p.b_batched = batch > 1 && strideB != 0;
    p.stride_c = batch > 1 ? strideC : 0;
    p.ab_format = bf ? 1u : 0u;
    p.tile_n = BN;
    p.c_tma = c_tma;
    p.a_ldg = a_ldg;
    p.b_ldg = b_ldg;
    p.a_ptr = A;
    p.b_ptr = B;
    p.lda = lda;
    p.ldb = ldb;
    p.stride_a = strideA;
    p.stride_b = strideB;
    p.timeout_ns = 2000000000ull;
    p.inject_stall = 0;
    // GEMM_GB300_HGEMM_GROUP=g (sweeps only): a raster group of 2^g tile (pair) rows
    p.log_group = kLogGroup;
    if (const char *e = std::getenv("GEMM_GB300_HGEMM_GROUP"); e && e[0] >= '0' && e[0] <= '9' && !e[1])
        p.log_group = e[0] - '0';
    if (const char *e = std::getenv("GEMM_GB300_TEST_INJECT_STALL"); e && (e[0] == '1' || e[0] == '2')) {
        p.inject_stall = e[0] - '0';
        p.timeout_ns = 20000000ull;
    }
    cudaError_t e;
    if (a_ldg || b_ldg) {
        if (a_mn) e = b_mn ? launch_t<1, 1, true>(dev, m, p, stream) : launch_t<1, 0, true>(dev, m, p, stream);
        else e = b_mn ? launch_t<0, 1, true>(dev, m, p, stream) : launch_t<0, 0, true>(dev, m, p, stream);
    } else {
        if (a_mn) e = b_mn ? launch_t<1, 1, false>(dev, m, p, stream) : launch_t<1, 0, false>(dev, m, p, stream);
        else e = b_mn ? launch_t<0, 1, false>(dev, m, p, stream) : launch_t<0, 0, false>(dev, m, p, stream);
    }
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

gemm_status_t read_and_clear_device_status(cudaStream_t stream)
{
    unsigned int word = 0;
    const unsigned int zero = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_LAUNCH;
    if (cudaMemcpyFromSymbol(&word, g_device_status, sizeof(word)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    if (word) {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) reset_workspace_counters(dev);
        return GEMM_ERR_DEVICE_TIMEOUT;
    }
    return GEMM_OK;
}

}  // namespace gemm
