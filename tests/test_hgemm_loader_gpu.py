"""Parity of the tensor-core path on 16-bit operands that TMA cannot read.

TMA copies rows only from a 16-byte aligned base with a leading dimension (and batch stride)
that is a multiple of 8 elements.  Any other 2-byte aligned operand is read by the loader
warps of the same kernel: each row is copied as the aligned 16-byte blocks that cover it
(cp.async) and shifted into place in shared memory where it starts off a 16-byte boundary;
rows at the ends of the operand's storage or cut by the matrix edge are read element by
element, with zero fill outside the matrix.  Each case is compared with the CPU oracle
element by element.
"""
import itertools

import numpy as np
import pytest
import torch

import dense_gemm_sgemm_gb300 as g
from dense_gemm_sgemm_gb300 import gemm_get_device_status, gemm_kernel_launches, workloads
from tests import parity

pytestmark = pytest.mark.gpu

FN = {"f16": g.gemm_hgemm_f16f32, "bf16": g.gemm_bgemm_bf16f32}


def _shifted(t: torch.Tensor, off: int) -> torch.Tensor:
    """A flat device copy of t starting `off` elements after a 256-byte aligned base."""
    flat = torch.zeros(t.numel() + off, dtype=t.dtype)
    flat[off:] = t.reshape(-1)
    return flat.cuda()[off:]


def _run(w, inputs, off_a=0, off_b=0, calls=1):
    dA, dB = _shifted(inputs["A"], off_a), _shifted(inputs["B"], off_b)
    dC = inputs["C"].cuda()
    outs = []
    for _ in range(calls):
        dC.copy_(inputs["C"])
        n0 = gemm_kernel_launches()
        FN[w.dtype](w.opA, w.opB, w.M, w.N, w.K, w.alpha, dA, w.lda, dB, w.ldb, w.beta, dC, w.ldc)
        launches = gemm_kernel_launches() - n0
        torch.cuda.synchronize()
        assert gemm_get_device_status() == 0
        assert launches == 1  # the loader warps run inside the GEMM kernel: no pre-pass
        outs.append(dC[:, : w.N].contiguous())
    return outs


# (extra elements per row of A and B, base offsets of A and B in elements): each names the
# alignment of the rows the loader warps see.
LAYOUTS = {
    "odd_ld": ((1, 3), (0, 0)),          # rows alternate 2- and 4-byte alignment (and all classes mod 16)
    "ld_4byte": ((2, 6), (0, 0)),        # rows 4-byte aligned (shifted by 4, 8 or 12 bytes)
    "ld_8byte": ((4, 4), (0, 0)),        # rows 8-byte aligned (shifted by 8 bytes on odd rows)
    "base_2byte": ((0, 0), (1, 1)),      # aligned leading dimensions, every row 2-byte aligned
    "base_odd_ld": ((1, 1), (3, 1)),     # both
    "a_only": ((1, 0), (0, 0)),          # A through the loader, B by TMA
    "b_only": ((0, 0), (0, 1)),          # A by TMA, B through the loader
}


def _workload(name, dtype, M, N, K, opA, opB, layout, **kw):
    (pa, pb), _ = LAYOUTS[layout]
    w0 = workloads.Workload("probe", dtype, M, N, K, opA, opB)
    # pad on top of a multiple of 8, so the chosen residue is exactly the layout's
    pad = ((-w0.a_shape[1]) % 8 + pa, (-w0.b_shape[1]) % 8 + pb, kw.pop("pad_c", 0))
    return workloads.Workload(name, dtype, M, N, K, opA, opB, pad=pad, **kw)


@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("opA,opB", list(itertools.product("NT", "NT")))
def test_alignment_classes_full_oracle(opA, opB, layout):
    # ragged in every dimension, three 128-row tile rows (two-CTA pairs plus an odd row)
    w = _workload(f"loader_{layout}_{opA}{opB}", "f16", 300, 270, 333, opA, opB, layout,
                  alpha=0.75, beta=0.25, seed=51)
    inputs = workloads.make_inputs(w)
    _, (oa, ob) = LAYOUTS[layout]
    for out in _run(w, inputs, oa, ob, calls=2):
        parity.check_full(w, inputs, out)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("opA,opB", list(itertools.product("NT", "NT")))
def test_single_cta_tiles_full_oracle(opA, opB, dtype):
    # M <= 128: one-CTA tiles (cta_group::1), several tile columns, K tail inside a chunk
    w = _workload(f"loader_single_{dtype}_{opA}{opB}", dtype, 100, 700, 203, opA, opB, "base_odd_ld",
                  alpha=-1.5, beta=0.5, seed=52)
    inputs = workloads.make_inputs(w)
    (out,) = _run(w, inputs, 3, 1)
    parity.check_full(w, inputs, out)


@pytest.mark.parametrize("pair", [True, False])
@pytest.mark.parametrize("mode", ["auto", "n"])
def test_split_tail_units_full_oracle(mode, pair, monkeypatch):
    # 180 tiles: the last wave runs as K-half (auto) or N-half units, read by the loader warps
    if mode != "auto":
        monkeypatch.setenv("GEMM_GB300_HGEMM_TAIL", mode)
    if not pair:
        monkeypatch.setenv("GEMM_GB300_HGEMM_PAIR", "0")
    w = _workload("loader_tail_2300x2560x512", "f16", 2300, 2560, 512, "N", "T", "odd_ld",
                  alpha=0.75, beta=0.5, seed=53, pad_c=3)
    inputs = workloads.make_inputs(w)
    (out,) = _run(w, inputs)
    parity.check_full(w, inputs, out)


@pytest.mark.parametrize("opA,opB", [("N", "N"), ("T", "T")])
def test_integer_bit_exact_large(opA, opB):
    # several waves of tile pairs, every K slice through the loader (odd leading dimensions)
    w = _workload(f"loader_int_{opA}{opB}", "f16", 2048, 2304, 1024, opA, opB, "odd_ld", seed=54,
                  dist_a="int4", dist_b="int4")
    inputs = workloads.make_inputs(w)
    (out,) = _run(w, inputs, 1, 0)
    parity.check_full(w, inputs, out, integer=True)


def test_4096_cube_odd_leading_dimensions_full_oracle():
    w = _workload("loader_4096cube", "f16", 4096, 4096, 4096, "N", "N", "odd_ld", seed=3)
    inputs = workloads.make_inputs(w)
    (out,) = _run(w, inputs)
    parity.check_full(w, inputs, out)


def test_loader_matches_tma_path_bit_for_bit():
    # The same values laid out for TMA and for the loader: the tensor cores see identical
    # shared-memory tiles, so the results agree bit for bit.
    w_tma = workloads.Workload("loader_same_tma", "f16", 1000, 1032, 776, "N", "N", alpha=1.0,
                               beta=0.0, seed=55)
    w_ldg = _workload("loader_same_ldg", "f16", 1000, 1032, 776, "N", "N", "base_odd_ld", seed=55)
    inputs = workloads.make_inputs(w_tma)
    (ref,) = _run(w_tma, inputs)
    (ld_a, ld_b) = (w_ldg.lda, w_ldg.ldb)
    padded = {"A": torch.full((w_ldg.M, ld_a), float("nan")).half(),
              "B": torch.full((w_ldg.K, ld_b), float("nan")).half(), "C": inputs["C"]}
    padded["A"][:, : w_ldg.K] = inputs["A"][:, : w_ldg.K]
    padded["B"][:, : w_ldg.N] = inputs["B"][:, : w_ldg.N]
    (out,) = _run(w_ldg, padded, 3, 1)
    assert torch.equal(ref.view(torch.int32), out.view(torch.int32))
    assert np.isfinite(out.cpu().numpy()).all()  # NaN row padding is never read
