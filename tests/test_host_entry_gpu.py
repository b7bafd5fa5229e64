"""The host-memory entry points (gemm_*_host) against the CPU oracle: staging copies in,
device GEMM, copy out, for all three input types, both op flags, padded leading
dimensions, page-locked and pageable buffers, and calls overlapped on several streams."""
import numpy as np
import pytest
import torch

from dense_gemm_sgemm_gb300 import (gemm_bgemm_bf16f32_host, gemm_get_device_status,
                                    gemm_hgemm_f16f32_host, gemm_kernel_launches,
                                    gemm_sgemm_f32_host, workloads)
from tests import parity

pytestmark = pytest.mark.gpu

HOST_FN = {"f32": gemm_sgemm_f32_host, "f16": gemm_hgemm_f16f32_host,
           "bf16": gemm_bgemm_bf16f32_host}
SENTINEL = 12345.0


def _host_inputs(w, pinned=True):
    inputs = workloads.make_inputs(w)
    host = {k: v.clone() for k, v in inputs.items()}
    if w.pad[2]:
        host["C"][:, w.N:] = SENTINEL  # row padding of C: never written by the call
    if pinned:
        host = {k: v.pin_memory() for k, v in host.items()}
    return inputs, host


def _run(w, host, stream=None):
    HOST_FN[w.dtype](w.opA, w.opB, w.M, w.N, w.K, w.alpha, host["A"], w.lda, host["B"], w.ldb,
                     w.beta, host["C"], w.ldc, stream)


def _check(w, inputs, host, integer=False):
    ref, absdot = parity.oracle_full(w, inputs)
    got = host["C"].numpy()
    cin = inputs["C"].numpy()[:, : w.N] if w.beta != 0.0 else None
    parity.assert_close(w, got[:, : w.N], ref, absdot, cin, integer=integer)
    if w.pad[2]:
        assert (got[:, w.N:] == SENTINEL).all(), "row padding of C was written"


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("opA,opB", [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")])
@pytest.mark.parametrize("beta", [0.0, -0.5])
def test_host_entry_matches_the_oracle(dtype, opA, opB, beta):
    w = workloads.Workload(f"host_{dtype}_{opA}{opB}", dtype, 301, 263, 197, opA, opB,
                           alpha=1.5, beta=beta, seed=71, pad=(3, 5, 7))
    inputs, host = _host_inputs(w)
    _run(w, host)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    _check(w, inputs, host)


def test_host_entry_headline_integer_bit_exact_and_launch_count():
    # The ragged 1001 x 777 x 513 shape with integer inputs: every partial sum exact.
    w = workloads.Workload("host_ragged_int", "f32", 1001, 777, 513, seed=72, dist_a="int4",
                           dist_b="int4")
    inputs, host = _host_inputs(w)
    before = gemm_kernel_launches()
    _run(w, host)
    torch.cuda.synchronize()
    assert gemm_kernel_launches() - before >= 1
    assert gemm_get_device_status() == 0
    _check(w, inputs, host, integer=True)


def test_host_entry_pageable_buffers():
    w = workloads.Workload("host_pageable", "f32", 200, 150, 100, alpha=0.5, beta=2.0, seed=73,
                           pad=(0, 0, 4))
    inputs, host = _host_inputs(w, pinned=False)
    _run(w, host)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    _check(w, inputs, host)


def test_host_entry_numpy_operands():
    w = workloads.Workload("host_numpy", "f16", 128, 96, 80, "T", "N", beta=1.0, seed=74)
    inputs, _ = _host_inputs(w, pinned=False)
    a = parity.np_in(inputs["A"], "f16").copy()
    b = parity.np_in(inputs["B"], "f16").copy()
    c = inputs["C"].numpy().copy()
    gemm_hgemm_f16f32_host(w.opA, w.opB, w.M, w.N, w.K, w.alpha, a, w.lda, b, w.ldb, w.beta, c,
                           w.ldc)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    _check(w, inputs, {"C": torch.from_numpy(c)})


def test_host_entry_calls_overlapped_on_three_streams():
    # Six independent problems over three streams, two calls per stream: each call's
    # staging area belongs to its stream, so overlapping calls never share one.
    streams = [torch.cuda.Stream() for _ in range(3)]
    cases = []
    for i in range(6):
        w = workloads.Workload(f"host_stream_{i}", "f32", 257 + 31 * i, 190 + 17 * i, 160 + 9 * i,
                               alpha=1.0 + i, beta=0.25 * i, seed=80 + i)
        inputs, host = _host_inputs(w)
        cases.append((w, inputs, host))
    for i, (w, _, host) in enumerate(cases):
        _run(w, host, streams[i % 3])
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    for w, inputs, host in cases:
        _check(w, inputs, host)


def test_host_entry_quick_returns():
    # M == 0: nothing happens; K == 0: C = beta * C through the staging area.
    c = torch.arange(12, dtype=torch.float32).reshape(3, 4).pin_memory()
    a = torch.ones(3, 1).pin_memory()
    b = torch.ones(1, 4).pin_memory()
    before = gemm_kernel_launches()
    gemm_sgemm_f32_host("N", "N", 0, 4, 1, 1.0, a, 1, b, 4, 0.0, c, 4)
    assert gemm_kernel_launches() == before
    gemm_sgemm_f32_host("N", "N", 3, 4, 0, 1.0, a, 1, b, 4, 0.5, c, 4)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    assert torch.equal(c, torch.arange(12, dtype=torch.float32).reshape(3, 4) * 0.5)


def test_host_entry_rejects_device_tensors():
    d = torch.zeros(4, 4, device="cuda")
    with pytest.raises(ValueError):
        gemm_sgemm_f32_host("N", "N", 4, 4, 4, 1.0, d, 4, d, 4, 0.0, d, 4)


def test_host_entry_staging_grows_with_the_problem():
    # A small call, then a larger one on the same stream: the staging area is reallocated
    # after the small call's copies have finished, and both results are right.
    s = torch.cuda.Stream()
    small = workloads.Workload("host_small", "bf16", 64, 64, 64, seed=75)
    large = workloads.Workload("host_large", "bf16", 1500, 1300, 700, beta=1.0, seed=76,
                               dist_a="int4", dist_b="int4", dist_c="int4")
    i1, h1 = _host_inputs(small)
    i2, h2 = _host_inputs(large)
    _run(small, h1, s)
    _run(large, h2, s)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    _check(small, i1, h1)
    _check(large, i2, h2, integer=True)
