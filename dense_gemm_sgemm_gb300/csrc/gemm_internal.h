// Internal declarations shared by the host API and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/gemm_gb300.h"

namespace gemm {

// Grouped tile raster (copecc "GEMM" page, section "线程块网格重排"): consecutive tile
// indices walk down a group of 2^log_group tile rows before moving to the next tile
// column, so the tiles running at the same time share A rows and B columns in L2.
__host__ __device__ __forceinline__ void raster(int64_t t, int64_t tiles_m, int64_t tiles_n,
                                                int log_group, int64_t &tm, int64_t &tn)
{
    const int64_t group_rows = int64_t(1) << log_group;
    const int64_t per_group = group_rows * tiles_n;
    const int64_t g = t / per_group;
    const int64_t first = g * group_rows;
    int64_t rows = tiles_m - first;
    if (rows > group_rows) rows = group_rows;
    const int64_t r = t - g * per_group;
    tm = first + r % rows;
    tn = r / rows;
}

struct DeviceInfo {
    int device;
    int num_sms;
    int cc_major, cc_minor;
    size_t smem_optin;
};

// Cached per-device properties of the current device; false if there is none.
bool current_device(DeviceInfo &info);

// Scratch kept per (device, stream) -- split-K workspace, transposition buffers, host
// staging -- exists for at most kMaxScratchStreams streams per device and kind: a caller
// cycling through many short-lived streams must not accumulate it without bound.  Calls on
// further streams take the paths that need no scratch (no split-K, no transposition); the
// host-memory entry points release the other streams' staging instead (see host_staging).
constexpr int kMaxScratchStreams = 16;

// Split-K workspace of one (device, stream): kWorkspaceBytes of partial tiles and
// kWorkspaceCounters arrival counters that are zero between kernels.
constexpr size_t kWorkspaceBytes = size_t(64) << 20;
constexpr size_t kWorkspaceCounters = 8192;
struct StreamWorkspace {
    float *data = nullptr;
    unsigned int *counters = nullptr;
};
// False when no workspace exists and none can be allocated now (during capture, or when
// kMaxScratchStreams other streams of the device hold one).
bool stream_workspace(int dev, cudaStream_t stream, StreamWorkspace &out);
// Zeroes the arrival counters of every workspace of device `dev` (after a kernel gave up on
// a bounded wait and may have left counters raised).  Synchronises those streams.
void reset_workspace_counters(int dev);
// Device staging area of at least `bytes` for the host-memory entry points, one per
// (device, stream), grown by reallocation after synchronising the stream.  A new stream
// beyond kMaxScratchStreams first synchronises the device and frees the other streams'
// areas.  The caller holds host_call_mutex() from before this call until the call's copies
// and kernels are enqueued, so no other host call is using an area being freed.  nullptr
// when it would have to be (re)allocated while the stream is being captured, or allocation
// fails.
void *host_staging(int dev, cudaStream_t stream, size_t bytes);
std::mutex &host_call_mutex();

// Launchers (return cudaSuccess or the launch error).  Arguments are already validated.
// A batch of `batch` problems: operand b of problem i starts `stride` elements after that
// of problem i-1 (stride 0: all problems share the operand).
cudaError_t launch_sgemm(const DeviceInfo &dev, int opA, int opB, int64_t M, int64_t N,
                         int64_t K, float alpha, const float *A, int64_t lda, int64_t strideA,
                         const float *B, int64_t ldb, int64_t strideB, float beta, float *C,
                         int64_t ldc, int64_t strideC, int64_t batch, cudaStream_t stream);

cudaError_t launch_scale(int64_t M, int64_t N, float beta, float *C, int64_t ldc,
                         cudaStream_t stream);

// 16-bit input types of the tensor-core path.
constexpr int kInF16 = 0;
constexpr int kInBf16 = 1;

// Returns GEMM_OK, GEMM_ERR_MISALIGNED or GEMM_ERR_LAUNCH.  A and B need only 2-byte
// alignment: operands that TMA cannot read go through the kernel's loader warps.
gemm_status_t launch_hgemm(const DeviceInfo &dev, int dtype, int opA, int opB, int64_t M,
                           int64_t N, int64_t K, float alpha, const uint16_t *A, int64_t lda,
                           int64_t strideA, const uint16_t *B, int64_t ldb, int64_t strideB,
                           float beta, float *C, int64_t ldc, int64_t strideC, int64_t batch,
                           cudaStream_t stream);

// Writes the transpose of an fp32 operand (batch x rows x cols, leading dimension ld, batch
// stride stride; stride 0 = shared) into this stream's scratch buffer `which` (0 = A, 1 = B)
// as batch x cols x rows with the leading dimension rounded up to 4 (16-byte aligned rows).
// Returns the transposed pointer, leading dimension and stride; false when no buffer can be
// had or the shape exceeds the grid limits.
bool transpose_f32_operand(int dev, cudaStream_t stream, int which, const float *src, int64_t rows,
                           int64_t cols, int64_t ld, int64_t stride, int64_t batch, const float **out,
                           int64_t *ld_out, int64_t *stride_out);

// C = beta * C for every problem of a batch (alpha == 0 or K == 0).
cudaError_t launch_scale_batched(int64_t M, int64_t N, float beta, float *C, int64_t ldc,
                                 int64_t strideC, int64_t batch, cudaStream_t stream);

// Counts kernel launches of the library (gemm_kernel_launches).
void count_launches(uint64_t n = 1);
uint64_t launches_so_far();

// Reads and clears the device error word (synchronises `stream`).
gemm_status_t read_and_clear_device_status(cudaStream_t stream);

}  // namespace gemm
