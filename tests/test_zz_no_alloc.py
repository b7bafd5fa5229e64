"""gemm_sgemm_f32_noalloc: the split-K SGEMM for callers that must not allocate.

Some callers cannot let a library call cudaMalloc while they run -- a framework whose own
allocator owns the device memory, or a latency-critical path where an allocation could
block, synchronise the device or fail.  This entry point keeps its split-K scratch in a
fixed device array inside the library.  These tests call it through the C ABI, twice in a
row (the second call reuses the scratch the first one left behind), and check each result
against the CPU oracle and against gemm_sgemm_f32 on the same inputs.  The file is named to
be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_sgemm_gb300 import (GemmError, gemm_get_device_status, gemm_sgemm_f32,
                                    gemm_sgemm_f32_noalloc, workloads)
from tests import parity

pytestmark = pytest.mark.gpu

CASES = [
    workloads.sgemm_ragged(),                       # 208 tiles, split 2
    workloads.sgemm_256(),                          # 16 tiles, split 8
    workloads.Workload("noalloc_opT_pad", "f32", 300, 200, 700, "T", "T", alpha=0.5, beta=2.0,
                       seed=31, pad=(3, 1, 2)),    # unaligned lds, both operands transposed
    # 4096 tiles of 64 x 64: too many to split within the scratch array, so K is not split
    workloads.Workload("noalloc_unsplit_4096x4096x96", "f32", 4096, 4096, 96, alpha=1.0,
                       beta=-1.0, seed=32),
]


def _call(fn, w, dev, c_init):
    C = c_init.clone()
    fn(w.opA, w.opB, w.M, w.N, w.K, w.alpha, dev["A"], w.lda, dev["B"], w.ldb, w.beta, C, w.ldc)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    return C


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_matches_oracle_and_gemm_sgemm_f32_on_two_calls_in_a_row(w):
    inputs = workloads.make_inputs(w)
    dev = parity.to_device(inputs)
    ref, absdot = parity.oracle_full(w, inputs)
    cin = inputs["C"].numpy()[:, : w.N] if w.beta != 0.0 else None
    lib = _call(gemm_sgemm_f32, w, dev, dev["C"]).cpu().numpy()[:, : w.N]
    first = _call(gemm_sgemm_f32_noalloc, w, dev, dev["C"])
    second = _call(gemm_sgemm_f32_noalloc, w, dev, dev["C"])
    for got in (first, second):
        g = got.cpu().numpy()[:, : w.N]
        parity.assert_close(w, g, ref, absdot, cin, where=" (against the oracle)")
        parity.assert_close(w, g, lib, absdot, cin, where=" (against gemm_sgemm_f32)")
    # the split-K sum has a fixed order: the two calls agree bit for bit
    f, s2 = first[:, : w.N].contiguous(), second[:, : w.N].contiguous()
    assert torch.equal(f.view(torch.int32), s2.view(torch.int32))
    if w.ldc > w.N:  # padding columns of C are never written
        assert torch.isnan(first[:, w.N:]).all() and torch.isnan(second[:, w.N:]).all()


def test_sizes_beyond_the_limit_are_refused_without_launch():
    # M = 2^31 is beyond the entry point's limit: refused on the host, nothing launched
    A = torch.zeros(16, device="cuda")
    with pytest.raises(GemmError) as e:
        gemm_sgemm_f32_noalloc("N", "N", 1 << 31, 1, 1, 1.0, A, 1, A, 1, 0.0, A, 1)
    assert e.value.status == 3  # GEMM_ERR_UNSUPPORTED


def test_integer_inputs_bit_exact_against_oracle():
    w = workloads.Workload("noalloc_int", "f32", 320, 192, 1024, seed=9, dist_a="int4",
                           dist_b="int4")
    inputs = workloads.make_inputs(w)
    dev = parity.to_device(inputs)
    ref = oracle.gemm("N", "N", w.M, w.N, w.K, 1.0, inputs["A"].numpy(), w.lda,
                      inputs["B"].numpy(), w.ldb)
    for _ in range(2):
        C = _call(gemm_sgemm_f32_noalloc, w, dev, dev["C"])
        assert np.array_equal(C.cpu().numpy().view(np.uint32), ref.view(np.uint32))
