// Per-(device, stream) workspace of the split-K paths of both kernels, the per-stream
// staging area of the host-memory entry points, and the library's kernel-launch counter.
//
// One workspace per (device, stream): calls on the same stream are ordered and may share it;
// calls on different streams never do.  It is allocated once, on the first call on that
// stream that splits K through the workspace, kept until the process exits, and never
// allocated while the stream is being captured or once kMaxScratchStreams streams of the
// device hold one (the call then runs without splitting).  Every kernel that uses the arrival
// counters leaves them at zero when it finishes -- unless it gave up on a bounded wait, after
// which reset_workspace_counters() restores them.
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
    int held = 0;
    for (const auto &kv : g_ws) held += kv.first.first == dev;
    if (held >= kMaxScratchStreams) return false;
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

namespace {
struct Staging {
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_host_call_mu;
std::map<std::pair<int, cudaStream_t>, Staging> g_stage;
}  // namespace

std::mutex &host_call_mutex() { return g_host_call_mu; }

void *host_staging(int dev, cudaStream_t stream, size_t bytes)
{
    auto it = g_stage.find({dev, stream});
    if (it != g_stage.end() && it->second.bytes >= bytes && it->second.ptr) return it->second.ptr;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return nullptr;
    }
    if (it == g_stage.end()) {
        int held = 0;
        for (const auto &kv : g_stage) held += kv.first.first == dev;
        if (held >= kMaxScratchStreams) {
            // Every host call holds host_call_mutex() until its work is enqueued, and the
            // device synchronisation waits for all enqueued work: no area is still in use.
            if (cudaDeviceSynchronize() != cudaSuccess) {
                cudaGetLastError();
                return nullptr;
            }
            for (auto jt = g_stage.begin(); jt != g_stage.end();) {
                if (jt->first.first == dev) {
                    cudaFree(jt->second.ptr);
                    jt = g_stage.erase(jt);
                } else {
                    ++jt;
                }
            }
        }
    }
    Staging &sg = g_stage[{dev, stream}];
    if (sg.ptr) {
        // Earlier calls on this stream may still be copying through the old area.
        if (cudaStreamSynchronize(stream) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        cudaFree(sg.ptr);
        sg.ptr = nullptr;
        sg.bytes = 0;
    }
    // Round up to 2 MiB so a run of slightly larger problems does not reallocate each time.
    const size_t want = (bytes + (size_t(2) << 20) - 1) & ~((size_t(2) << 20) - 1);
    void *p = nullptr;
    if (cudaMalloc(&p, want) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    sg.ptr = p;
    sg.bytes = want;
    return p;
}

void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

uint64_t launches_so_far() { return g_launches.load(std::memory_order_relaxed); }

void reset_workspace_counters(int dev)
{
    std::lock_guard<std::mutex> lk(g_ws_mu);
    // The whole device, not each workspace's stream: a stream may have been destroyed since.
    cudaDeviceSynchronize();
    for (auto &kv : g_ws)
        if (kv.first.first == dev) cudaMemset(kv.second.counters, 0, kWorkspaceCounters * sizeof(unsigned int));
    cudaDeviceSynchronize();
    cudaGetLastError();
}

}  // namespace gemm
