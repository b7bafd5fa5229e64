"""Edge cases of both paths against the CPU oracle: IEEE special values, very long K, single
row / single column problems and extreme 16-bit inputs."""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_sgemm_gb300 import (gemm_bgemm_bf16f32, gemm_get_device_status, gemm_hgemm_f16f32,
                                    gemm_sgemm_f32, workloads)
from tests import parity

pytestmark = pytest.mark.gpu

FN = {"f32": gemm_sgemm_f32, "f16": gemm_hgemm_f16f32, "bf16": gemm_bgemm_bf16f32}
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _gemm(dtype, opA, opB, M, N, K, alpha, A, B, beta, C):
    """Runs the library on CPU tensors (stored shapes, unit column stride); returns C."""
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    FN[dtype](opA, opB, M, N, K, alpha, dA, A.shape[1], dB, B.shape[1], beta, dC, C.shape[1])
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    return dC.cpu()


def _oracle(dtype, opA, opB, M, N, K, alpha, A, B, beta, C):
    return oracle.gemm(opA, opB, M, N, K, alpha, parity.np_in(A, dtype), A.shape[1],
                       parity.np_in(B, dtype), B.shape[1], beta, C.numpy(), C.shape[1], dtype=dtype,
                       want_absdot=True)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_nan_and_inf_propagate_as_in_ieee_arithmetic(dtype):
    # Small-integer operands, then: a NaN in row 3 of A (row 3 of C is NaN), +Inf in row 7 of
    # A at k = 5 with B[5][j] = 0 for even j (Inf * 0 = NaN there, +/-Inf elsewhere), and
    # -Inf in column 11 of B at k = 2 (column 11 of C is -/+Inf or NaN).
    M, N, K = 130, 136, 64
    g = torch.Generator().manual_seed(61)
    A = torch.randint(-3, 4, (M, K), generator=g).to(torch.float32)
    B = torch.randint(1, 4, (K, N), generator=g).to(torch.float32)
    A[3, 10] = float("nan")
    A[7, 5] = float("inf")
    B[5, 0::2] = 0.0
    B[2, 11] = float("-inf")
    A, B = A.to(TORCH[dtype]), B.to(TORCH[dtype])
    C = torch.zeros(M, N)
    got = _gemm(dtype, "N", "N", M, N, K, 1.0, A, B, 0.0, C).numpy()
    ref, absdot = _oracle(dtype, "N", "N", M, N, K, 1.0, A, B, 0.0, C)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isposinf(got), np.isposinf(ref))
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    assert np.isnan(ref).any() and np.isinf(ref).any()
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])  # small integers: exact


@pytest.mark.parametrize("opA,opB", [("N", "N"), ("T", "T")])
def test_very_long_k_integer_bit_exact_sgemm(opA, opB):
    # 64 x 64 output, K = 65536: a deep split-K plan; integer partial sums stay exact
    w = workloads.Workload(f"longk_{opA}{opB}", "f32", 64, 72, 65536, opA, opB, seed=62,
                           dist_a="int4", dist_b="int4")
    inputs = workloads.make_inputs(w)
    dev = parity.to_device(inputs)
    parity.run_library(w, dev)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    parity.check_full(w, inputs, dev["C"], integer=True)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_very_long_k_integer_bit_exact_tensor_core(dtype):
    w = workloads.Workload(f"longk_{dtype}", dtype, 256, 256, 16384, seed=63, dist_a="int4",
                           dist_b="int4")
    inputs = workloads.make_inputs(w)
    dev = parity.to_device(inputs)
    parity.run_library(w, dev)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    parity.check_full(w, inputs, dev["C"], integer=True)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("M,N,K", [(1, 1000, 777), (999, 1, 333), (1, 1, 4096), (3, 5, 1)])
@pytest.mark.parametrize("opA,opB", [("N", "N"), ("T", "T")])
def test_single_row_and_single_column(dtype, M, N, K, opA, opB):
    w = workloads.Workload(f"vec_{M}x{N}x{K}", dtype, M, N, K, opA, opB, alpha=-0.5, beta=0.25,
                           seed=64)
    inputs = workloads.make_inputs(w)
    dev = parity.to_device(inputs)
    parity.run_library(w, dev)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    parity.check_full(w, inputs, dev["C"])


def test_fp16_extremes_subnormals_and_largest_finite():
    # fp16 subnormals (down to 2^-24) and values near the largest finite 65504: the products
    # are exact in fp32 and far from its range limits.
    M, N, K = 128, 256, 96
    g = torch.Generator().manual_seed(65)
    sub = torch.tensor([2.0 ** -24, 3 * 2.0 ** -24, 2.0 ** -15, -2.0 ** -20])
    big = torch.tensor([65504.0, -65504.0, 32768.0, 61440.0])
    A = sub[torch.randint(0, 4, (M, K), generator=g)]
    B = big[torch.randint(0, 4, (K, N), generator=g)]
    A[:, ::3] = big[torch.randint(0, 4, (M, (K + 2) // 3), generator=g)] / 65536.0
    A, B = A.half(), B.half()
    C = torch.randn(M, N, generator=g)
    w = workloads.Workload("f16_extremes", "f16", M, N, K, alpha=0.75, beta=0.5)
    got = _gemm("f16", "N", "N", M, N, K, 0.75, A, B, 0.5, C).numpy()
    ref, absdot = _oracle("f16", "N", "N", M, N, K, 0.75, A, B, 0.5, C)
    parity.assert_close(w, got, ref, absdot, C.numpy())


def test_bf16_wide_exponent_range():
    # bf16 keeps fp32's exponent range: operands from 2^-60 to 2^60 (products within fp32)
    M, N, K = 128, 128, 64
    g = torch.Generator().manual_seed(66)
    ea = torch.randint(-60, 61, (M, K), generator=g).to(torch.float32)
    eb = torch.randint(-60, 61, (K, N), generator=g).to(torch.float32)
    A = (torch.rand(M, K, generator=g) + 0.5) * torch.pow(2.0, ea)
    B = (torch.rand(K, N, generator=g) - 0.5) * torch.pow(2.0, eb)
    A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    C = torch.zeros(M, N)
    w = workloads.Workload("bf16_range", "bf16", M, N, K)
    got = _gemm("bf16", "N", "N", M, N, K, 1.0, A, B, 0.0, C).numpy()
    ref, absdot = _oracle("bf16", "N", "N", M, N, K, 1.0, A, B, 0.0, C)
    parity.assert_close(w, got, ref, absdot, None)


@pytest.mark.parametrize("dtype,plan", [("f32", "L:1"), ("f32", "L:3"), ("f32", "M:2"), ("f32", "S:1"),
                                        ("f32", "S:2"), ("f32", "S:5"), ("f16", None), ("bf16", None)])
def test_writes_stay_inside_c(dtype, plan, monkeypatch):
    # C is the first M rows of a larger NaN-filled buffer with padded rows (ldc > N): after
    # the call every element outside the M x N matrix -- the row padding and two guard rows
    # after it -- must still be NaN, on every tile configuration and split path.
    if plan:
        monkeypatch.setenv("GEMM_GB300_SGEMM_PLAN", plan)
    M, N, K, ldc = 333, 290, 200, 301
    g = torch.Generator().manual_seed(67)
    A = (torch.rand(M, K, generator=g) * 2 - 1).to(TORCH[dtype])
    B = (torch.rand(K, N, generator=g) * 2 - 1).to(TORCH[dtype])
    buf = torch.full(((M + 2) * ldc,), float("nan"), device="cuda")
    C = buf[: M * ldc].view(M, ldc)
    FN[dtype]("N", "N", M, N, K, 1.0, A.cuda(), K, B.cuda(), N, 0.0, C, ldc)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    full = buf.view(M + 2, ldc).cpu()
    assert not torch.isnan(full[:M, :N]).any()
    assert torch.isnan(full[:M, N:]).all(), "row padding written"
    assert torch.isnan(full[M:]).all(), "guard rows after C written"
