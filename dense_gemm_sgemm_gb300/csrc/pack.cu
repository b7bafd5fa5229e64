// Operand re-layout into per-stream scratch: packing of 16-bit operands whose layout the
// tensor-memory-access unit cannot read, and transposition of K-contiguous fp32 operands.
//
// TMA needs a 16-byte aligned base and row (and batch) strides that are multiples of 16
// bytes.  An fp16 / bf16 operand with an odd leading dimension, an unaligned base or an
// unaligned batch stride is first copied by pack_rows_u16 into a scratch buffer with the
// leading dimension rounded up to 8 elements, then read from there.  The copy moves
// 2 bytes per element in each direction, which is small next to the 2*M*N*K flops of any
// GEMM large enough to care.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "gemm_internal.h"

namespace gemm {
namespace {

// dst[b][r][c] = src[b][r][c] for c < cols, 0 for cols <= c < ldp (the row padding).
// Each thread writes one aligned 16-byte group of 8 elements.
__global__ void pack_rows_u16(const uint16_t *__restrict__ src, int64_t ld, int64_t stride,
                              uint16_t *__restrict__ dst, int64_t ldp, int64_t rows, int64_t cols,
                              int64_t batch)
{
    const int64_t groups_per_row = ldp / 8;
    const int64_t total = batch * rows * groups_per_row;
    for (int64_t g = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; g < total;
         g += int64_t(gridDim.x) * blockDim.x) {
        const int64_t cg = g % groups_per_row;
        const int64_t rb = g / groups_per_row;
        const int64_t r = rb % rows, b = rb / rows;
        const uint16_t *s = src + b * stride + r * ld + cg * 8;
        uint16_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = cg * 8 + e < cols ? s[e] : uint16_t(0);
        uint4 w;
        w.x = uint32_t(v[0]) | (uint32_t(v[1]) << 16);
        w.y = uint32_t(v[2]) | (uint32_t(v[3]) << 16);
        w.z = uint32_t(v[4]) | (uint32_t(v[5]) << 16);
        w.w = uint32_t(v[6]) | (uint32_t(v[7]) << 16);
        *reinterpret_cast<uint4 *>(dst + (b * rows + r) * ldp + cg * 8) = w;
    }
}

// One growable scratch buffer per (device, stream) for re-laid-out operands A and B.
struct PackBuffers {
    void *ptr[2] = {nullptr, nullptr};
    size_t bytes[2] = {0, 0};
};
std::mutex g_mu;
std::map<std::pair<int, cudaStream_t>, PackBuffers> g_bufs;

// A buffer of at least `bytes` for operand slot `which` (0 = A, 1 = B) of this stream.
// Grows by reallocation (after the stream's earlier work using it has finished); never
// allocates while the stream is being captured.
void *pack_buffer(int dev, cudaStream_t stream, int which, size_t bytes)
{
    std::lock_guard<std::mutex> lk(g_mu);
    PackBuffers &pb = g_bufs[{dev, stream}];
    if (pb.bytes[which] >= bytes) return pb.ptr[which];
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return nullptr;
    }
    if (pb.ptr[which]) {
        if (cudaStreamSynchronize(stream) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        cudaFree(pb.ptr[which]);
        pb.ptr[which] = nullptr;
        pb.bytes[which] = 0;
    }
    void *p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    pb.ptr[which] = p;
    pb.bytes[which] = bytes;
    return p;
}

// dst[b][c][r] = src[b][r][c] through a 64 x 65 shared tile, 256 threads: each thread issues
// its 16 loads (rows ty + 4i of one column) before any store, so enough reads are in flight
// to keep HBM busy; reads and writes are 128-byte row segments per warp.  Columns r >= rows
// of dst (row padding) are left unwritten.
constexpr int kTT = 64;
__global__ void __launch_bounds__(256) transpose_f32(const float *__restrict__ src, int64_t ld, int64_t stride,
                                                     float *__restrict__ dst, int64_t ldt, int64_t stride_t,
                                                     int64_t rows, int64_t cols)
{
    __shared__ float tile[kTT][kTT + 1];
    const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
    const int64_t r0 = int64_t(blockIdx.y) * kTT, c0 = int64_t(blockIdx.x) * kTT;
    const float *s = src + int64_t(blockIdx.z) * stride;
    float *d = dst + int64_t(blockIdx.z) * stride_t;
    float v[kTT / 4];
#pragma unroll
    for (int i = 0; i < kTT / 4; ++i) {
        const int64_t r = r0 + ty + 4 * i, c = c0 + tx;
        v[i] = r < rows && c < cols ? __ldg(s + r * ld + c) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < kTT / 4; ++i) tile[ty + 4 * i][tx] = v[i];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTT / 4; ++i) {
        const int64_t c = c0 + ty + 4 * i, r = r0 + tx;
        if (c < cols && r < rows) d[c * ldt + r] = tile[tx][ty + 4 * i];
    }
}

}  // namespace

bool transpose_f32_operand(int dev, cudaStream_t stream, int which, const float *src, int64_t rows,
                           int64_t cols, int64_t ld, int64_t stride, int64_t batch, const float **out,
                           int64_t *ld_out, int64_t *stride_out)
{
    const int64_t ldt = (rows + 3) / 4 * 4;
    const int64_t nb = stride == 0 ? 1 : batch;  // a shared operand is transposed once
    const int64_t grid_y = (rows + kTT - 1) / kTT, grid_x = (cols + kTT - 1) / kTT;
    if (grid_y > 65535 || grid_x > 0x7fffffff) return false;
    const size_t bytes = size_t(nb) * size_t(cols) * size_t(ldt) * 4;
    float *dst = static_cast<float *>(pack_buffer(dev, stream, which, bytes > 0 ? bytes : 16));
    if (dst == nullptr) return false;
    for (int64_t b0 = 0; b0 < nb; b0 += 65535) {
        const int64_t nz = nb - b0 < 65535 ? nb - b0 : 65535;
        const dim3 grid(static_cast<unsigned>(grid_x), static_cast<unsigned>(grid_y), static_cast<unsigned>(nz));
        transpose_f32<<<grid, 256, 0, stream>>>(src + b0 * stride, ld, stride, dst + b0 * cols * ldt, ldt,
                                                        cols * ldt, rows, cols);
        if (cudaGetLastError() != cudaSuccess) return false;
        count_launches();
    }
    *out = dst;
    *ld_out = ldt;
    *stride_out = stride == 0 ? 0 : cols * ldt;
    return true;
}

bool pack_u16_operand(int dev, cudaStream_t stream, int which, const uint16_t *src, int64_t rows,
                      int64_t cols, int64_t ld, int64_t stride, int64_t batch, const uint16_t **out,
                      int64_t *ld_out, int64_t *stride_out)
{
    const int64_t ldp = (cols + 7) / 8 * 8;
    const int64_t nb = stride == 0 ? 1 : batch;  // a shared operand is packed once
    const size_t bytes = size_t(nb) * size_t(rows) * size_t(ldp) * 2;
    uint16_t *dst = static_cast<uint16_t *>(pack_buffer(dev, stream, which, bytes > 0 ? bytes : 16));
    if (dst == nullptr) return false;
    const int64_t total = nb * rows * (ldp / 8);
    int64_t blocks = (total + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    if (blocks < 1) blocks = 1;
    pack_rows_u16<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(src, ld, stride, dst, ldp, rows, cols, nb);
    if (cudaGetLastError() != cudaSuccess) return false;
    count_launches();
    *out = dst;
    *ld_out = ldp;
    *stride_out = stride == 0 ? 0 : rows * ldp;
    return true;
}

}  // namespace gemm
