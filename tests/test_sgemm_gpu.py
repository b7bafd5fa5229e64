"""Parity of the strict-FP32 path (gemm_sgemm_f32) against the CPU oracle."""
import itertools

import numpy as np
import pytest
import torch

from dense_gemm_sgemm_gb300 import GemmError, gemm_get_device_status, gemm_sgemm_f32, workloads
from tests import parity

pytestmark = pytest.mark.gpu


def _run(w, inputs=None):
    inputs = inputs if inputs is not None else workloads.make_inputs(w)
    dev = parity.to_device(inputs)
    parity.run_library(w, dev)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    return inputs, dev


def test_256_cube_uniform():
    w = workloads.sgemm_256()
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"])


def test_256_cube_integer_bit_exact():
    w = workloads.sgemm_256(integer=True)
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"], integer=True)


def test_ragged_1001x777x513_alpha_beta():
    w = workloads.sgemm_ragged()
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"])


@pytest.mark.parametrize("mn", workloads.SWEEP_MN)
def test_sweep_full_oracle(mn):
    # every element of the M = N sweep (K = 1024), up to 16384^2, against the full oracle
    w = workloads.sgemm_sweep(mn)
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"])


def test_4096_cube_full_oracle():
    w = workloads.sgemm_cube(4096)
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"])


_EDGE = [1, 2, 3, 5, 7, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257]


def _fuzz_cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M, N, K = (int(rng.choice(_EDGE)) for _ in range(3))
        out.append((M, N, K))
    return out


@pytest.mark.parametrize("opA,opB", list(itertools.product("NT", "NT")))
def test_fuzz_shapes_ops_padding(opA, opB):
    for i, (M, N, K) in enumerate(_fuzz_cases(24, seed=10 * "NT".index(opA) + "NT".index(opB))):
        pad = (i % 3, (i // 3) % 3, i % 2)  # unaligned lds exercise the 4-byte loaders
        beta = 0.0 if i % 2 == 0 else -0.75
        w = workloads.Workload(f"fuzz_{M}x{N}x{K}_{opA}{opB}", "f32", M, N, K, opA, opB,
                               alpha=1.25, beta=beta, seed=100 + i, pad=pad)
        inputs, dev = _run(w)
        parity.check_full(w, inputs, dev["C"][:, : w.N].contiguous() if pad[2] else dev["C"])
        if pad[2]:  # padding columns of C are never written
            assert torch.isnan(dev["C"][:, w.N:]).all()


# Every tile configuration (L 128 x 128, M 128 x 64, S 64 x 64), with and without split K,
# through the plan override, on shapes with ragged tails in M, N and K and both copy widths.
@pytest.mark.parametrize("plan", ["L:1", "L:3", "M:1", "M:2", "M:5", "S:1", "S:2", "S:3", "S:6"])
def test_every_tile_configuration(plan, monkeypatch):
    monkeypatch.setenv("GEMM_GB300_SGEMM_PLAN", plan)
    for i, (opA, opB) in enumerate(itertools.product("NT", "NT")):
        for j, (M, N, K) in enumerate([(300, 200, 333), (129, 65, 160)]):
            pad = (j, j, 0) if i % 2 == 0 else (0, 0, 3 * j)
            w = workloads.Workload(f"plan{plan}_{M}x{N}x{K}_{opA}{opB}", "f32", M, N, K, opA,
                                   opB, alpha=0.75, beta=0.5 if j == 0 else 0.0,
                                   seed=200 + 4 * i + j, pad=pad)
            inputs, dev = _run(w)
            parity.check_full(w, inputs, dev["C"][:, : w.N].contiguous() if pad[2] else dev["C"])
            if pad[2]:
                assert torch.isnan(dev["C"][:, w.N:]).all(), "row padding of C was written"
        wi = workloads.Workload(f"plan{plan}_int_{opA}{opB}", "f32", 257, 191, 515, opA, opB,
                                seed=300 + i, dist_a="int4", dist_b="int4")
        inputs, dev = _run(wi)
        parity.check_full(wi, inputs, dev["C"], integer=True)


# Two K splits of every 64 x 64 tile run as two-CTA clusters that hand the partial over
# through distributed shared memory; the workspace hand-off sums in the same order (p0 + p1),
# so both give the same bits -- on the ragged headline shape (both operands with 4-byte
# copies), an aligned batch and a shape whose second split has fewer slices.
@pytest.mark.parametrize("shape", [(1001, 777, 513, "N", "N", 1), (512, 384, 1024, "T", "N", 3),
                                   (130, 200, 48, "N", "T", 1)])
def test_cluster_pair_split_matches_workspace_split(shape, monkeypatch):
    M, N, K, opA, opB, batch = shape
    monkeypatch.setenv("GEMM_GB300_SGEMM_PLAN", "S:2")
    w = workloads.Workload(f"pair_{M}x{N}x{K}", "f32", M, N, K, opA, opB, alpha=1.5, beta=-0.5,
                           seed=91)
    inputs = workloads.make_inputs(w)
    outs = []
    for pair in ("1", "0"):
        monkeypatch.setenv("GEMM_GB300_SGEMM_PAIR", pair)
        _, dev = _run(w, inputs)
        outs.append(dev["C"].cpu())
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))
    parity.check_full(w, inputs, outs[0].cuda())
    if batch > 1:
        # strided batch of `batch` problems through the same plan: each equals its single call
        from dense_gemm_sgemm_gb300 import gemm_sgemm_f32_strided_batched

        g = torch.Generator().manual_seed(92)
        a_shape, b_shape = w.a_shape, w.b_shape
        A = torch.rand(batch, *a_shape, generator=g) * 2 - 1
        B = torch.rand(batch, *b_shape, generator=g) * 2 - 1
        Cin = torch.rand(batch, M, N, generator=g) * 2 - 1
        res = []
        for pair in ("1", "0"):
            monkeypatch.setenv("GEMM_GB300_SGEMM_PAIR", pair)
            dC = Cin.cuda()
            gemm_sgemm_f32_strided_batched(opA, opB, M, N, K, 1.5, A.cuda(), a_shape[1],
                                           a_shape[0] * a_shape[1], B.cuda(), b_shape[1],
                                           b_shape[0] * b_shape[1], -0.5, dC, N, M * N, batch)
            torch.cuda.synchronize()
            assert gemm_get_device_status() == 0
            res.append(dC.cpu())
        assert torch.equal(res[0].view(torch.int32), res[1].view(torch.int32))


# An unsplit 128 x 128 plan whose last wave is small runs that wave's tiles as K splits in a
# second launch (fixed-order sum by the last split); GEMM_GB300_SGEMM_TAIL=0 turns that off.
# 2304^2: 324 tiles of 128 x 128 (one wave of 304 + 20 -> 4 splits); the 128 x 64 and 64 x 64
# plans run unsplit (covered here as the reference behaviour).
@pytest.mark.parametrize("plan", ["L:1", "M:1", "S:1"])
@pytest.mark.parametrize("opA,opB", [("N", "N"), ("T", "T")])
def test_last_wave_split(plan, opA, opB, monkeypatch):
    monkeypatch.setenv("GEMM_GB300_SGEMM_PLAN", plan)
    wi = workloads.Workload(f"tail_int_{plan}_{opA}{opB}", "f32", 2304, 2304, 300, opA, opB,
                            seed=41, dist_a="int4", dist_b="int4", pad=(1, 0, 0))
    inputs, dev = _run(wi)
    parity.check_full(wi, inputs, dev["C"], integer=True)
    w = workloads.Workload(f"tail_{plan}_{opA}{opB}", "f32", 2304, 2300, 300, opA, opB,
                           alpha=0.5, beta=-1.5, seed=42)
    inputs, dev = _run(w)
    split = dev["C"].clone()
    parity.check_full(w, inputs, split)
    monkeypatch.setenv("GEMM_GB300_SGEMM_TAIL", "0")
    dev["C"].copy_(inputs["C"].cuda())
    parity.run_library(w, dev)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    parity.check_full(w, inputs, dev["C"])


# Large problems on the 128-row tiles transpose a K-contiguous operand into scratch first
# (op(A) = N when N >= 2048, op(B) = T when M >= 2048, at 1e10 flops or more): unaligned
# leading dimensions, ragged K and both operands at once.
@pytest.mark.parametrize("opA,opB", [("N", "N"), ("N", "T"), ("T", "T")])
def test_large_k_contiguous_operands_are_transposed_first(opA, opB, monkeypatch):
    monkeypatch.setenv("GEMM_GB300_SGEMM_PLAN", "L:1")
    w = workloads.Workload(f"pretranspose_{opA}{opB}", "f32", 3100, 3079, 531, opA, opB,
                           alpha=0.5, beta=0.25, seed=31, pad=(1, 3, 0), dist_a="int4",
                           dist_b="int4", dist_c="int4")
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"], integer=True)


@pytest.mark.parametrize("opA,opB", list(itertools.product("NT", "NT")))
def test_integer_bit_exact_all_ops(opA, opB):
    w = workloads.Workload(f"int_{opA}{opB}", "f32", 300, 200, 1024, opA, opB, seed=7,
                           dist_a="int4", dist_b="int4")
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"], integer=True)


def test_misaligned_pointers_take_scalar_paths():
    # Views that start one element into their buffers are 4-byte but not 16-byte aligned.
    M, N, K = 150, 130, 70
    g = torch.Generator().manual_seed(21)
    Abuf = torch.rand(M * K + 1, generator=g) * 2 - 1
    Bbuf = torch.rand(K * N + 1, generator=g) * 2 - 1
    Cbuf = torch.rand(M * N + 1, generator=g) * 2 - 1
    for opA, opB in itertools.product("NT", "NT"):
        w = workloads.Workload(f"misaligned_{opA}{opB}", "f32", M, N, K, opA, opB, alpha=0.5,
                               beta=2.0)
        inputs = {"A": Abuf[1:].reshape(w.a_shape).clone(), "B": Bbuf[1:].reshape(w.b_shape).clone(),
                  "C": Cbuf[1:].reshape(M, N).clone()}
        dA, dB, dC = Abuf.cuda(), Bbuf.cuda(), Cbuf.cuda()
        gemm_sgemm_f32(opA, opB, M, N, K, 0.5, dA[1:], w.lda, dB[1:], w.ldb, 2.0, dC[1:], N)
        torch.cuda.synchronize()
        parity.check_full(w, inputs, dC[1:].reshape(M, N))


def test_beta_zero_ignores_nan_and_k_zero_alpha_zero():
    M, N, K = 70, 90, 40
    A = torch.randn(M, K, device="cuda")
    B = torch.randn(K, N, device="cuda")
    C = torch.full((M, N), float("nan"), device="cuda")
    gemm_sgemm_f32("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N)
    torch.cuda.synchronize()
    assert torch.isfinite(C).all()
    Cin = torch.randn(M, N, device="cuda")
    C = Cin.clone()
    gemm_sgemm_f32("N", "N", M, N, 0, 1.0, None, K, None, N, 0.5, C, N)  # K == 0
    torch.cuda.synchronize()
    assert torch.equal(C, Cin * 0.5)
    C = Cin.clone()
    gemm_sgemm_f32("N", "N", M, N, K, 0.0, A, K, B, N, 0.0, C, N)  # alpha == 0, beta == 0
    torch.cuda.synchronize()
    assert torch.equal(C, torch.zeros_like(C))
    C = Cin.clone()
    gemm_sgemm_f32("N", "N", M, N, K, 0.0, A, K, B, N, 1.0, C, N)  # nothing to do
    torch.cuda.synchronize()
    assert torch.equal(C, Cin)
    gemm_sgemm_f32("N", "N", 0, N, K, 1.0, A, K, B, N, 0.0, C, N)  # empty M
    gemm_sgemm_f32("N", "N", M, 0, K, 1.0, A, K, B, N, 0.0, C, 1)  # empty N


def test_invalid_arguments_raise_before_launch():
    A = torch.zeros(4, 4, device="cuda")
    with pytest.raises(GemmError) as e:
        gemm_sgemm_f32("N", "N", 4, 4, 4, 1.0, A, 3, A, 4, 0.0, A, 4)  # lda < K
    assert e.value.status == 1
    with pytest.raises(GemmError) as e:
        gemm_sgemm_f32("N", "N", 4, 4, 4, 1.0, 0, 4, A, 4, 0.0, A, 4)  # NULL A
    assert e.value.status == 1
    base = A.data_ptr() + 2  # not 4-byte aligned
    with pytest.raises(GemmError) as e:
        gemm_sgemm_f32("N", "N", 2, 2, 2, 1.0, base, 4, A, 4, 0.0, A, 4)
    assert e.value.status == 2


def test_streams_are_respected():
    w = workloads.sgemm_ragged()
    inputs = workloads.make_inputs(w)
    dev = parity.to_device(inputs)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        parity.run_library(w, dev)
    s.synchronize()
    parity.check_full(w, inputs, dev["C"])
