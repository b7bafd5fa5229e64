"""Per-stream scratch stays bounded when a caller cycles through many streams.

The split-K workspace, the buffers of transposed fp32 operands and the staging area of the
host-memory entry points are kept per (device, stream) for at most 16 streams per device.
Calls on further streams take the paths without that scratch (no split-K, no transposition)
or, for the host-memory entry points, release the other streams' staging first.  Every
result is compared with the CPU oracle.
"""
import pytest
import torch

import dense_gemm_sgemm_gb300 as g
from dense_gemm_sgemm_gb300 import gemm_get_device_status, workloads
from tests import parity

pytestmark = pytest.mark.gpu

STREAMS = 24
CAP = 16


def test_many_short_lived_streams_bounded_scratch_and_correct():
    split = workloads.sgemm_256()                                   # 16 tiles: split-K workspace
    tail = workloads.Workload("scratch_tail_2300x2560x512", "f16", 2300, 2560, 512, seed=61)  # K-half units
    big = workloads.Workload("scratch_transpose_2048", "f32", 2048, 2048, 2048, seed=62)      # A transposed
    cases = [split, tail, big]
    inputs = {w.name: workloads.make_inputs(w) for w in cases}
    devs = {w.name: parity.to_device(inputs[w.name]) for w in cases}
    refs = {w.name: parity.oracle_full(w, inputs[w.name]) for w in cases}
    outs = {w.name: [torch.empty(w.M, w.ldc, device="cuda") for _ in range(STREAMS)] for w in cases}
    host = workloads.make_inputs(split)
    pinned = {k: v.pin_memory() for k, v in host.items()}
    host_out = [torch.empty(split.M, split.N).pin_memory() for _ in range(STREAMS)]
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for i in range(STREAMS):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for w in cases:
                d = devs[w.name]
                fn = g.gemm_sgemm_f32 if w.dtype == "f32" else g.gemm_hgemm_f16f32
                fn(w.opA, w.opB, w.M, w.N, w.K, w.alpha, d["A"], w.lda, d["B"], w.ldb, w.beta,
                   outs[w.name][i], w.ldc, s)
            g.gemm_sgemm_f32_host("N", "N", split.M, split.N, split.K, 1.0, pinned["A"], split.lda,
                                  pinned["B"], split.ldb, 0.0, host_out[i], split.ldc, s)
        s.synchronize()
        del s  # a short-lived stream
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    free1, _ = torch.cuda.mem_get_info()
    # per stream at most: 64 MB workspace, one 16 MB transposed operand, a 2 MiB staging area
    per_stream = (64 << 20) + (16 << 20) + (2 << 20) + (1 << 20)
    assert free0 - free1 <= CAP * per_stream + (256 << 20), (free0 - free1) / 2**20
    for w in cases:
        ref, absdot = refs[w.name]
        for i in range(STREAMS):
            parity.assert_close(w, outs[w.name][i].cpu().numpy(), ref, absdot, None,
                                where=f" ({w.name}, stream {i})")
    ref, absdot = refs[split.name]
    for i in range(STREAMS):
        parity.assert_close(split, host_out[i].numpy(), ref, absdot, None, where=f" (host entry, stream {i})")
