"""The seeded synthetic inputs and the work/byte counts the benchmark's roofline uses.

No GPU: these pin the input recipe (seed, draw order, distributions, fp16/bf16 rounding,
NaN-filled C when beta == 0, NaN row padding) and the per-GEMM figures -- 2 M N K flop, and
algorithmic bytes s_in (M K + K N) + 4 M N (1 + [beta != 0]) (each input read once, C
written once and read when beta != 0) -- with values worked out by hand.
"""
import math

import pytest
import torch

from dense_gemm_sgemm_gb300 import workloads


def test_same_seed_same_bits_and_draw_order():
    w = workloads.Workload("probe", "f32", 5, 7, 3, alpha=2.0, beta=0.5, seed=11)
    a1, a2 = workloads.make_inputs(w), workloads.make_inputs(w)
    for k in "ABC":
        assert torch.equal(a1[k].view(torch.int32), a2[k].view(torch.int32))
    # draw order A, B, C from one generator seeded with w.seed, uniform[-1, 1] = rand * 2 - 1
    g = torch.Generator().manual_seed(11)
    A = torch.rand(5, 3, generator=g) * 2 - 1
    B = torch.rand(3, 7, generator=g) * 2 - 1
    C = torch.rand(5, 7, generator=g) * 2 - 1
    assert torch.equal(a1["A"], A) and torch.equal(a1["B"], B) and torch.equal(a1["C"], C)


def test_beta_zero_fills_c_with_nan_and_padding_is_nan():
    w = workloads.Workload("probe", "f32", 4, 6, 5, opA="T", opB="T", seed=3, pad=(2, 1, 3))
    x = workloads.make_inputs(w)
    assert x["A"].shape == (5, 4 + 2) and x["B"].shape == (6, 5 + 1) and x["C"].shape == (4, 6 + 3)
    assert (w.lda, w.ldb, w.ldc) == (6, 6, 9)
    assert torch.isnan(x["C"]).all()
    assert torch.isnan(x["A"][:, 4:]).all() and torch.isnan(x["B"][:, 5:]).all()
    assert not torch.isnan(x["A"][:, :4]).any() and not torch.isnan(x["B"][:, :5]).any()


@pytest.mark.parametrize("dtype,tdtype", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_16_bit_inputs_are_the_fp32_draws_rounded(dtype, tdtype):
    w32 = workloads.Workload("probe", "f32", 9, 8, 7, seed=5)
    w16 = workloads.Workload("probe", dtype, 9, 8, 7, seed=5)
    x32, x16 = workloads.make_inputs(w32), workloads.make_inputs(w16)
    assert x16["A"].dtype == tdtype and x16["B"].dtype == tdtype and x16["C"].dtype == torch.float32
    assert torch.equal(x16["A"], x32["A"].to(tdtype)) and torch.equal(x16["B"], x32["B"].to(tdtype))


def test_distributions():
    w = workloads.Workload("probe", "f32", 64, 64, 64, seed=7, dist_a="int4", dist_b="u11")
    x = workloads.make_inputs(w)
    A, B = x["A"], x["B"]
    assert torch.equal(A, A.round()) and A.min() >= -4 and A.max() <= 4 and len(torch.unique(A)) == 9
    assert B.min() >= -1 and B.max() <= 1 and not torch.equal(B, B.round())


def test_named_workloads_follow_the_recipe_table():
    # (M, N, K, opA, opB, alpha, beta, seed, dtype)
    table = {
        "sgemm_256cube": (256, 256, 256, "N", "N", 1.0, 0.0, 0, "f32"),
        "sgemm_256cube_int": (256, 256, 256, "N", "N", 1.0, 0.0, 0, "f32"),
        "sgemm_ragged_1001x777x513": (1001, 777, 513, "N", "N", 1.5, -0.5, 1, "f32"),
        "sgemm_sweep_128x128x1024": (128, 128, 1024, "N", "N", 1.0, 0.0, 2, "f32"),
        "sgemm_sweep_16384x16384x1024": (16384, 16384, 1024, "N", "N", 1.0, 0.0, 2, "f32"),
        "sgemm_4096cube": (4096, 4096, 4096, "N", "N", 1.0, 0.0, 2, "f32"),
        "hgemm_8192x8192x8192": (8192, 8192, 8192, "N", "N", 1.0, 0.0, 3, "f16"),
        "hgemm_2048x2048x1024_int": (2048, 2048, 1024, "N", "N", 1.0, 0.0, 3, "f16"),
        "linear_16384x4096x4096_opBT": (16384, 4096, 4096, "N", "T", 1.0, 1.0, 4, "f16"),
    }
    for name, (M, N, K, opA, opB, alpha, beta, seed, dtype) in table.items():
        w = workloads.by_name(name)
        assert (w.M, w.N, w.K, w.opA, w.opB, w.alpha, w.beta, w.seed, w.dtype) == \
            (M, N, K, opA, opB, alpha, beta, seed, dtype), name
    assert workloads.by_name("sgemm_256cube_int").dist_a == "int4"
    assert workloads.by_name("hgemm_2048x2048x1024_int").dist_b == "int4"
    lin = workloads.by_name("linear_16384x4096x4096_opBT")
    assert (lin.dist_a, lin.dist_b, lin.dist_c) == ("n01", "n002", "n01_1")
    assert lin.b_shape == (4096, 4096) and lin.a_shape == (16384, 4096)


def test_flops_and_algorithmic_bytes_by_hand():
    rag = workloads.by_name("sgemm_ragged_1001x777x513")
    assert rag.flops == 2 * 1001 * 777 * 513 == 797_999_202
    # fp32 inputs read once (4 (1001*513 + 513*777) = 3_648_456), C written and read (beta != 0:
    # 8 * 1001 * 777 = 6_222_216)
    assert rag.algorithmic_bytes == 9_870_672
    head = workloads.by_name("hgemm_8192x8192x8192")
    assert head.flops == 2 * 8192 ** 3
    # fp16 A and B (2 * 2 * 8192^2 = 268_435_456) + fp32 C written once (268_435_456)
    assert head.algorithmic_bytes == 536_870_912
    lin = workloads.by_name("linear_16384x4096x4096_opBT")
    # 2 (16384*4096 + 4096*4096) + 8 * 16384 * 4096 (beta = 1: C read and written)
    assert lin.algorithmic_bytes == 2 * (16384 * 4096 + 4096 * 4096) + 8 * 16384 * 4096 == 704_643_072
    assert math.isclose(head.flops / head.algorithmic_bytes, 2048.0)
