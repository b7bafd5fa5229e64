"""bf16 inputs (gemm_bgemm_bf16f32) and the strided-batched forms of all three paths,
against the CPU oracle problem by problem."""
import itertools

import numpy as np
import pytest
import torch

import dense_gemm_sgemm_gb300 as g
import oracle
from dense_gemm_sgemm_gb300 import GemmError, gemm_get_device_status, workloads
from tests import parity

pytestmark = pytest.mark.gpu


def _pad8(cols, extra=0):
    return (-cols) % 8 + 8 * extra


# ------------------------------------------------------------------------------ bf16
@pytest.mark.parametrize("opA,opB", list(itertools.product("NT", "NT")))
def test_bf16_small_full_oracle(opA, opB):
    M, N, K = 260, 300, 200
    w0 = workloads.Workload("probe", "bf16", M, N, K, opA, opB)
    w = workloads.Workload(f"bf16_{opA}{opB}", "bf16", M, N, K, opA, opB, alpha=0.5, beta=-1.0,
                           seed=41, pad=(_pad8(w0.a_shape[1]), _pad8(w0.b_shape[1], 1), 1))
    inputs = workloads.make_inputs(w)
    dev = parity.to_device(inputs)
    parity.run_library(w, dev)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    parity.check_full(w, inputs, dev["C"][:, : w.N].contiguous())


def test_bf16_integer_bit_exact_and_large_full_oracle():
    w = workloads.Workload("bf16_int", "bf16", 2304, 2560, 512, opB="T", seed=42,
                           dist_a="int4", dist_b="int4")
    inputs = workloads.make_inputs(w)
    dev = parity.to_device(inputs)
    parity.run_library(w, dev)
    torch.cuda.synchronize()
    parity.check_full(w, inputs, dev["C"], integer=True)
    w = workloads.Workload("bf16_4096", "bf16", 4096, 4096, 4096, seed=43)
    inputs = workloads.make_inputs(w)
    dev = parity.to_device(inputs)
    parity.run_library(w, dev)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    parity.check_full(w, inputs, dev["C"])


# --------------------------------------------------------------------- strided batched
def _batched_case(dtype, batch, M, N, K, opA, opB, share_a=False, share_b=False, alpha=1.25,
                  beta=0.5, seed=0):
    """Operands of a batch laid out with padded strides; returns tensors and strides."""
    gen = torch.Generator().manual_seed(seed)
    a_rows, a_cols = (M, K) if opA == "N" else (K, M)
    b_rows, b_cols = (K, N) if opB == "N" else (N, K)
    align = 8 if dtype != "f32" else 1
    lda = a_cols + (-a_cols) % align + align
    ldb = b_cols + (-b_cols) % align
    ldc = N + 3
    sA = 0 if share_a else a_rows * lda + align * 3
    sB = 0 if share_b else b_rows * ldb + align * 5
    sC = M * ldc + 7
    nA = (batch - 1) * sA + a_rows * lda
    nB = (batch - 1) * sB + b_rows * ldb
    nC = (batch - 1) * sC + M * ldc
    A = torch.rand(nA, generator=gen) * 2 - 1
    B = torch.rand(nB, generator=gen) * 2 - 1
    C = torch.rand(nC, generator=gen) * 2 - 1
    if dtype == "f16":
        A, B = A.half(), B.half()
    elif dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    return dict(A=A, B=B, C=C, lda=lda, ldb=ldb, ldc=ldc, sA=sA, sB=sB, sC=sC, M=M, N=N, K=K,
                opA=opA, opB=opB, alpha=alpha, beta=beta, batch=batch, dtype=dtype)


def _check_batched(c):
    fn = {"f32": g.gemm_sgemm_f32_strided_batched, "f16": g.gemm_hgemm_f16f32_strided_batched,
          "bf16": g.gemm_bgemm_bf16f32_strided_batched}[c["dtype"]]
    dA, dB, dC = c["A"].cuda(), c["B"].cuda(), c["C"].cuda()
    fn(c["opA"], c["opB"], c["M"], c["N"], c["K"], c["alpha"], dA, c["lda"], c["sA"], dB, c["ldb"],
       c["sB"], c["beta"], dC, c["ldc"], c["sC"], c["batch"])
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    got = dC.cpu()
    npA, npB = parity.np_in(c["A"], c["dtype"]), parity.np_in(c["B"], c["dtype"])
    npC = c["C"].numpy()
    w = workloads.Workload("batched", c["dtype"], c["M"], c["N"], c["K"], c["opA"], c["opB"],
                           alpha=c["alpha"], beta=c["beta"])
    for b in range(c["batch"]):
        a0, b0, c0 = b * c["sA"], b * c["sB"], b * c["sC"]
        ref, absdot = oracle.gemm(c["opA"], c["opB"], c["M"], c["N"], c["K"], c["alpha"],
                                  npA[a0:], c["lda"], npB[b0:], c["ldb"], c["beta"],
                                  npC[c0:c0 + c["M"] * c["ldc"]], c["ldc"], dtype=c["dtype"],
                                  want_absdot=True)
        out = got[c0:c0 + c["M"] * c["ldc"]].reshape(c["M"], c["ldc"]).numpy()
        cin = npC[c0:c0 + c["M"] * c["ldc"]].reshape(c["M"], c["ldc"])[:, : c["N"]]
        parity.assert_close(w, out[:, : c["N"]], ref, absdot, cin, where=f" problem {b}")
        # the padding between problems and after each row is never written
        pad = got[c0:c0 + c["M"] * c["ldc"]].reshape(c["M"], c["ldc"])[:, c["N"]:]
        assert torch.equal(pad, c["C"][c0:c0 + c["M"] * c["ldc"]].reshape(c["M"], c["ldc"])[:, c["N"]:])
        if b + 1 < c["batch"]:
            gap = got[c0 + c["M"] * c["ldc"]: (b + 1) * c["sC"]]
            assert torch.equal(gap, c["C"][c0 + c["M"] * c["ldc"]: (b + 1) * c["sC"]])


@pytest.mark.parametrize("opA,opB", list(itertools.product("NT", "NT")))
def test_sgemm_strided_batched(opA, opB):
    _check_batched(_batched_case("f32", 5, 130, 97, 70, opA, opB, seed=1))


def test_sgemm_strided_batched_shared_operand_and_split_k():
    # small problems with a long K: the planner splits K, tiles numbered across the batch
    _check_batched(_batched_case("f32", 3, 64, 96, 1024, "N", "N", share_a=True, seed=2))
    _check_batched(_batched_case("f32", 4, 200, 64, 513, "T", "N", share_b=True, beta=0.0, seed=3))


@pytest.mark.parametrize("share", ["none", "a", "b"])
def test_sgemm_strided_batched_transposed_first(share, monkeypatch):
    # large enough for the transposition of K-contiguous operands into scratch (see
    # test_sgemm_gpu); a shared operand is transposed once
    monkeypatch.setenv("GEMM_GB300_SGEMM_PLAN", "L:1")
    _check_batched(_batched_case("f32", 2, 2050, 2049, 600, "N", "T", share_a=share == "a",
                                 share_b=share == "b", seed=4))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("opA,opB", [("N", "N"), ("N", "T"), ("T", "N")])
def test_tensor_core_strided_batched(dtype, opA, opB):
    # 3 problems x 6 tile pairs: units of different problems share the persistent grid
    _check_batched(_batched_case(dtype, 3, 300, 520, 192, opA, opB, seed=4))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tensor_core_strided_batched_unaligned_strides_through_the_loader(dtype):
    c = _batched_case(dtype, 3, 200, 136, 100, "N", "T", seed=6)
    # shift every problem's operands by an odd number of elements
    c["sA"] += 3
    c["sB"] += 1
    c["A"] = torch.cat([c["A"], torch.zeros(3 * 3, dtype=c["A"].dtype)])
    c["B"] = torch.cat([c["B"], torch.zeros(3, dtype=c["B"].dtype)])
    _check_batched(c)


def test_tensor_core_strided_batched_shared_b():
    _check_batched(_batched_case("f16", 4, 256, 256, 128, "N", "T", share_b=True, seed=5))


def test_batched_argument_rules():
    A = torch.zeros(1 << 16, device="cuda")
    H = torch.zeros(1 << 16, device="cuda", dtype=torch.float16)
    with pytest.raises(GemmError) as e:  # outputs of consecutive problems overlap
        g.gemm_sgemm_f32_strided_batched("N", "N", 8, 8, 8, 1.0, A, 8, 64, A, 8, 64, 0.0, A, 8,
                                         32, 2)
    assert e.value.status == 1
    with pytest.raises(GemmError) as e:  # negative batch
        g.gemm_sgemm_f32_strided_batched("N", "N", 8, 8, 8, 1.0, A, 8, 64, A, 8, 64, 0.0, A, 8,
                                         64, -1)
    assert e.value.status == 1
    with pytest.raises(GemmError) as e:  # odd byte address
        g.gemm_hgemm_f16f32_strided_batched("N", "N", 8, 8, 8, 1.0, H.data_ptr() + 1, 8, 64, H, 8,
                                            64, 0.0, A, 8, 64, 2)
    assert e.value.status == 2
    # batch == 0 is a no-op
    g.gemm_sgemm_f32_strided_batched("N", "N", 8, 8, 8, 1.0, A, 8, 64, A, 8, 64, 0.0, A, 8, 64, 0)
