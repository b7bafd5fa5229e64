// Per-(device, stream) workspace of the split-K paths of both kernels, and the library's
// kernel-launch counter.
//
// One workspace per (device, stream): calls on the same stream are ordered and may share it;
// calls on different streams never do.  It is allocated once, on the first call on that
// stream that splits K, kept until the process exits, and never allocated while the stream
// is being captured (the call then runs without splitting).  Every kernel that uses the
// arrival counters leaves them at zero when it finishes -- unless it gave up on a bounded
// wait, after which reset_workspace_counters() restores them.
#include <cuda_runtime.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "gemm_internal.h"

namespace gemm {
namespace {
std::atomic<uint64_t> g_launches{0};
std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, StreamWorkspace> g_ws;
}  // namespace

bool stream_workspace(int dev, cudaStream_t stream, StreamWorkspace &out)
{
    std::lock_guard<std::mutex> lk(g_ws_mu);
    auto it = g_ws.find({dev, stream});
    if (it != g_ws.end()) {
        out = it->second;
        return true;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return false;
    }
    StreamWorkspace w;
    if (cudaMalloc(&w.data, kWorkspaceBytes) != cudaSuccess ||
        cudaMalloc(&w.counters, kWorkspaceCounters * sizeof(unsigned int)) != cudaSuccess ||
        cudaMemset(w.counters, 0, kWorkspaceCounters * sizeof(unsigned int)) != cudaSuccess) {
        cudaGetLastError();
        if (w.data) cudaFree(w.data);
        if (w.counters) cudaFree(w.counters);
        return false;
    }
    g_ws[{dev, stream}] = w;
    out = w;
    return true;
}

void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

uint64_t launches_so_far() { return g_launches.load(std::memory_order_relaxed); }

void reset_workspace_counters(int dev)
{
    std::lock_guard<std::mutex> lk(g_ws_mu);
    for (auto &kv : g_ws)
        if (kv.first.first == dev) {
            cudaStreamSynchronize(kv.first.second);
            cudaMemset(kv.second.counters, 0, kWorkspaceCounters * sizeof(unsigned int));
        }
    cudaGetLastError();
}

}  // namespace gemm
