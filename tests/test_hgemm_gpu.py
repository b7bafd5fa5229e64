"""Parity of the fp16-input / fp32-accumulate tcgen05 path (gemm_hgemm_f16f32)."""
import itertools

import numpy as np
import pytest
import torch

import dense_gemm_sgemm_gb300 as g
from dense_gemm_sgemm_gb300 import GemmError, gemm_get_device_status, gemm_hgemm_f16f32, workloads
from tests import parity

pytestmark = pytest.mark.gpu


def _run(w, inputs=None):
    inputs = inputs if inputs is not None else workloads.make_inputs(w)
    dev = parity.to_device(inputs)
    parity.run_library(w, dev)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    return inputs, dev


def _pad8(cols, extra=0):
    return (-cols) % 8 + 8 * extra


def test_small_full_oracle_all_ops():
    for opA, opB in itertools.product("NT", "NT"):
        M, N, K = 200, 300, 136
        w0 = workloads.Workload("probe", "f16", M, N, K, opA, opB)
        pad = (_pad8(w0.a_shape[1]), _pad8(w0.b_shape[1]), 0)
        w = workloads.Workload(f"hgemm_small_{opA}{opB}", "f16", M, N, K, opA, opB, alpha=1.0,
                               beta=0.0, seed=11, pad=pad)
        inputs, dev = _run(w)
        parity.check_full(w, inputs, dev["C"])


@pytest.mark.parametrize("opA,opB", list(itertools.product("NT", "NT")))
def test_integer_bit_exact(opA, opB):
    M, N, K = 384, 640, 1024
    w = workloads.Workload(f"hgemm_int_{opA}{opB}", "f16", M, N, K, opA, opB, seed=5,
                           dist_a="int4", dist_b="int4")
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"], integer=True)


@pytest.mark.parametrize("opA,opB", list(itertools.product("NT", "NT")))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_pair_and_single_cta_paths_full_oracle(opA, opB, dtype, monkeypatch):
    # Two-CTA tiles (tcgen05.mma.cta_group::2, each CTA holding its own A rows and half of the
    # B columns) and one-CTA tiles on the same problem: an odd number of 128-row tile rows
    # (the last pair has no second row), ragged N and K, several tiles per CTA.
    M, N, K = 1408 + 77, 2048 + 40, 904
    w0 = workloads.Workload("probe", dtype, M, N, K, opA, opB)
    pad = (_pad8(w0.a_shape[1]), _pad8(w0.b_shape[1]), 0)
    w = workloads.Workload(f"hgemm_pairs_{dtype}_{opA}{opB}", dtype, M, N, K, opA, opB,
                           alpha=1.25, beta=-0.5, seed=31, pad=pad)
    inputs = workloads.make_inputs(w)
    for pair in (True, False):
        if not pair:
            monkeypatch.setenv("GEMM_GB300_HGEMM_PAIR", "0")
        _, dev = _run(w, inputs)
        parity.check_full(w, inputs, dev["C"])


def test_persistent_tiles_and_double_buffered_accumulator():
    # 18 x 10 = 180 tiles of 128 x 256: several CTAs run two tiles through both TMEM buffers
    w = workloads.Workload("hgemm_2304x2560x192", "f16", 2304, 2560, 192, alpha=0.75, beta=0.5,
                           seed=8)
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"])


_EDGE = [1, 7, 8, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383]


@pytest.mark.parametrize("opA,opB", list(itertools.product("NT", "NT")))
def test_fuzz_ragged_shapes(opA, opB):
    rng = np.random.default_rng(10 * "NT".index(opA) + "NT".index(opB) + 77)
    for i in range(12):
        M, N, K = (int(rng.choice(_EDGE)) for _ in range(3))
        w0 = workloads.Workload("probe", "f16", M, N, K, opA, opB)
        pad = (_pad8(w0.a_shape[1], i % 2), _pad8(w0.b_shape[1], (i // 2) % 2), i % 3)
        beta = 0.0 if i % 2 == 0 else 1.5
        w = workloads.Workload(f"hgemm_fuzz_{M}x{N}x{K}_{opA}{opB}", "f16", M, N, K, opA, opB,
                               alpha=-0.5, beta=beta, seed=200 + i, pad=pad)
        inputs, dev = _run(w)
        C = dev["C"]
        parity.check_full(w, inputs, C[:, : w.N].contiguous() if pad[2] else C)
        if pad[2]:
            assert torch.isnan(C[:, w.N:]).all()


@pytest.mark.parametrize("n", workloads.HGEMM_SQUARE)
def test_square_full_oracle(n):
    w = workloads.hgemm_square(n)
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"])


def test_square_integer_2048_bit_exact():
    w = workloads.hgemm_square(2048, integer=True, K=1024)
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"], integer=True)


def test_linear_layer_opBT_beta1_full_oracle():
    w = workloads.linear_fp16()
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"])


def test_odd_byte_addresses_are_refused():
    A = torch.zeros(64, 72, dtype=torch.float16, device="cuda")
    C = torch.zeros(64, 64, device="cuda")
    with pytest.raises(GemmError) as e:
        gemm_hgemm_f16f32("N", "N", 8, 8, 8, 1.0, A.data_ptr() + 1, 72, A, 72, 0.0, C, 64)
    assert e.value.status == 2


def test_beta_zero_ignores_nan():
    M, N, K = 300, 504, 200  # lda = 200 and ldb = 504 are multiples of 8
    A = torch.randn(M, K, device="cuda").half()
    B = torch.randn(K, N, device="cuda").half()
    C = torch.full((M, N), float("nan"), device="cuda")
    gemm_hgemm_f16f32("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N)
    torch.cuda.synchronize()
    assert torch.isfinite(C).all()


# The last, partial wave of tiles is split in two units per tile: K halves by default (at
# least 8 K slices; the half that finishes second adds the other's fp32 partial), N halves
# through GEMM_GB300_HGEMM_TAIL=n, none with GEMM_GB300_HGEMM_TAIL=0.
TAIL_MODES = ["auto", "n"]


def _tail_env(monkeypatch, mode, pair=True):
    if mode != "auto":
        monkeypatch.setenv("GEMM_GB300_HGEMM_TAIL", mode)
    if not pair:
        monkeypatch.setenv("GEMM_GB300_HGEMM_PAIR", "0")


@pytest.mark.parametrize("pair", [True, False])
@pytest.mark.parametrize("mode", TAIL_MODES)
def test_tail_wave_split_units_full_oracle(mode, pair, monkeypatch):
    # 18 x 10 = 180 tiles of 128 x 256 (90 tile pairs for the two-CTA MMA): the tiles of the
    # last wave run as two units each on different SMs.
    _tail_env(monkeypatch, mode, pair)
    w = workloads.Workload("hgemm_tail_2300x2560x512", "f16", 2300, 2560, 512, alpha=0.75,
                           beta=0.5, seed=12, pad=(0, 0, 3))
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"][:, : w.N].contiguous())
    assert torch.isnan(dev["C"][:, w.N:]).all()


@pytest.mark.parametrize("mode", TAIL_MODES)
@pytest.mark.parametrize("opB", ["N", "T"])
def test_tail_wave_split_units_integer_bit_exact(opB, mode, monkeypatch):
    _tail_env(monkeypatch, mode)
    w = workloads.Workload(f"hgemm_tail_int_{opB}", "f16", 2304, 2600, 1000, opB=opB, seed=13,
                           dist_a="int4", dist_b="int4", pad=(0, (-2600) % 8 if opB == "N" else 0, 0))
    inputs, dev = _run(w)
    parity.check_full(w, inputs, dev["C"], integer=True)


def test_tail_n_halves_change_no_bit(monkeypatch):
    # Each output element is summed by one CTA over all of K either way.
    w = workloads.Workload("hgemm_tail_same_bits", "f16", 2304, 2560, 640, seed=14)
    monkeypatch.setenv("GEMM_GB300_HGEMM_TAIL", "n")
    inputs, dev = _run(w)
    with_halves = dev["C"].clone()
    monkeypatch.setenv("GEMM_GB300_HGEMM_TAIL", "0")
    dev["C"].copy_(inputs["C"].cuda())
    parity.run_library(w, dev)
    torch.cuda.synchronize()
    assert torch.equal(with_halves.view(torch.int32), dev["C"].view(torch.int32))


def test_tail_k_halves_deterministic_and_counters_reset():
    # Whichever K half finishes second, the two partials sum to the same bits; the arrival
    # counters are back at zero after every launch, so repeated launches agree.
    w = workloads.Workload("hgemm_tail_k_repeat", "f16", 2304, 2560, 640, alpha=1.0, beta=1.0,
                           seed=15)
    inputs = workloads.make_inputs(w)
    dev = parity.to_device(inputs)
    outs = []
    for _ in range(4):
        dev["C"].copy_(inputs["C"].cuda())
        parity.run_library(w, dev)
        torch.cuda.synchronize()
        assert gemm_get_device_status() == 0
        outs.append(dev["C"].clone())
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))
    parity.check_full(w, inputs, outs[0])
