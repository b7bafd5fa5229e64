"""Parity of the tensor-core path with wide pair tiles (256 x 512, one 512-column accumulator).

Large problems (three or more full waves of wide tiles) take this form by default;
GEMM_GB300_HGEMM_WIDE=1 forces it on the small and ragged shapes below, =0 keeps 256 x 256
tiles.  The wide tile issues the same tcgen05.mma instructions (M = 256, N = 256, K = 16, in
the same K order) for each output element, so both forms must agree bit for bit; every
element is also compared with the CPU oracle.
"""
import itertools

import pytest
import torch

import dense_gemm_sgemm_gb300 as g
from dense_gemm_sgemm_gb300 import gemm_get_device_status, gemm_kernel_launches, workloads
from tests import parity

pytestmark = pytest.mark.gpu


def _run(w, inputs, monkeypatch, wide):
    monkeypatch.setenv("GEMM_GB300_HGEMM_WIDE", wide)
    dev = parity.to_device(inputs)
    n0 = gemm_kernel_launches()
    parity.run_library(w, dev)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    assert gemm_kernel_launches() - n0 == 1
    return dev["C"]


def _pad8(cols):
    return (-cols) % 8


@pytest.mark.parametrize("beta", [-0.5, 0.0])
@pytest.mark.parametrize("opA,opB", list(itertools.product("NT", "NT")))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_wide_tiles_full_oracle_and_same_bits(opA, opB, dtype, beta, monkeypatch):
    # 6 pair rows (the last one half outside M), N = 1240: 3 wide tiles, the last cut at 216
    # columns; ragged K; padded C rows that must stay untouched.  beta = 0 with ldc a multiple
    # of 4 writes C through TMA stores (clipped at the edges of C).
    M, N, K = 1408 + 77, 1240, 904
    w0 = workloads.Workload("probe", dtype, M, N, K, opA, opB)
    w = workloads.Workload(f"wide_{dtype}_{opA}{opB}", dtype, M, N, K, opA, opB, alpha=1.25, beta=beta,
                           seed=81, pad=(_pad8(w0.a_shape[1]), _pad8(w0.b_shape[1]), 3 if beta else 4))
    inputs = workloads.make_inputs(w)
    wide = _run(w, inputs, monkeypatch, "1")
    narrow = _run(w, inputs, monkeypatch, "0")
    assert torch.equal(wide[:, : w.N].contiguous().view(torch.int32), narrow[:, : w.N].contiguous().view(torch.int32))
    assert torch.isnan(wide[:, w.N:]).all()  # row padding of C never written
    parity.check_full(w, inputs, wide[:, : w.N].contiguous())


def test_edge_of_c_not_a_multiple_of_four_columns(monkeypatch):
    # beta = 0, C aligned, ldc = 384 but N = 383: the last 16-byte piece of each row straddles
    # the edge, so C is written without TMA stores; the padding column must stay untouched
    w = workloads.Workload("c_edge_383", "f16", 65, 383, 8, alpha=-0.5, seed=84, pad=(0, 1, 1))
    inputs = workloads.make_inputs(w)
    for wide in ("0", "1"):
        out = _run(w, inputs, monkeypatch, wide)
        assert torch.isnan(out[:, w.N:]).all()
        parity.check_full(w, inputs, out[:, : w.N].contiguous())


def test_wide_tiles_integer_bit_exact_several_per_cluster(monkeypatch):
    # 16 pair rows x 5 wide tiles = 80 units on 76 clusters: some run two tiles, so a tile's
    # MMAs wait for the previous tile's epilogue to drain the single accumulator
    w = workloads.Workload("wide_int", "f16", 4096, 2560, 1024, seed=82, dist_a="int4", dist_b="int4")
    inputs = workloads.make_inputs(w)
    out = _run(w, inputs, monkeypatch, "1")
    parity.check_full(w, inputs, out, integer=True)


def test_wide_tiles_strided_batched(monkeypatch):
    monkeypatch.setenv("GEMM_GB300_HGEMM_WIDE", "1")
    batch, M, N, K = 3, 520, 760, 328
    gen = torch.Generator().manual_seed(83)
    A = (torch.rand(batch, M, K, generator=gen) * 2 - 1).half()
    B = (torch.rand(batch, N, K, generator=gen) * 2 - 1).half()
    C = (torch.rand(batch, M, N, generator=gen) * 2 - 1)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    g.gemm_hgemm_f16f32_strided_batched("N", "T", M, N, K, 0.5, dA, K, M * K, dB, K, N * K, 2.0, dC, N, M * N,
                                        batch)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    for b in range(batch):
        w = workloads.Workload(f"wide_batched_{b}", "f16", M, N, K, "N", "T", alpha=0.5, beta=2.0)
        inputs = {"A": A[b], "B": B[b], "C": C[b]}
        parity.check_full(w, inputs, dC[b])


def test_wide_expired_wait_is_reported_and_context_survives(monkeypatch):
    monkeypatch.setenv("GEMM_GB300_HGEMM_WIDE", "1")
    M, N, K = 256, 512, 256
    A = torch.randint(-2, 3, (M, K), device="cuda").half()
    B = torch.randint(-2, 3, (K, N), device="cuda").half()
    C = torch.zeros(M, N, device="cuda")
    assert gemm_get_device_status() == 0
    monkeypatch.setenv("GEMM_GB300_TEST_INJECT_STALL", "1")
    g.gemm_hgemm_f16f32("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N)
    assert gemm_get_device_status() == 5  # GEMM_ERR_DEVICE_TIMEOUT
    monkeypatch.delenv("GEMM_GB300_TEST_INJECT_STALL")
    g.gemm_hgemm_f16f32("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    assert torch.equal(C, A.float() @ B.float())
