// Operand re-layout into per-stream scratch: transposition of K-contiguous fp32 operands,
// so that the SGEMM kernel reads both operands as 16-byte [k][x] rows.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "gemm_internal.h"

namespace gemm {
namespace {

// One growable scratch buffer per (device, stream) for transposed operands A and B.
struct PackBuffers {
    void *ptr[2] = {nullptr, nullptr};
    size_t bytes[2] = {0, 0};
};
std::mutex g_mu;
std::map<std::pair<int, cudaStream_t>, PackBuffers> g_bufs;

// A buffer of at least `bytes` for operand slot `which` (0 = A, 1 = B) of this stream.
// Grows by reallocation (after the stream's earlier work using it has finished); never
// allocates while the stream is being captured, nor for a new stream once kMaxScratchStreams
// streams of the device hold buffers (the caller then reads the operand untransposed).
void *pack_buffer(int dev, cudaStream_t stream, int which, size_t bytes)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_bufs.find({dev, stream}) == g_bufs.end()) {
        int held = 0;
        for (const auto &kv : g_bufs) held += kv.first.first == dev;
        if (held >= kMaxScratchStreams) return nullptr;
    }
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

}  // namespace gemm
