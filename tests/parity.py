"""Shared helpers of the parity tests: run the library, run the oracle, compare.

Acceptance (per element, from the definition of the method and the stated tolerances):
    |C - C_ref| <= tol * (|alpha| * sum_k |a_ik b_kj| + |beta| * |Cin_ij|) + ulp32(|C_ref|)
with tol = 1e-5 for strict FP32 and 2e-3 for fp16 (and bf16) inputs with fp32
accumulation, and bit equality when every input is a small integer (all partial sums are
then exact in fp32).  The 16-bit inputs are the rounded values both sides consume, so the
tolerance covers only the fp32 accumulation, whose error does not depend on the input type.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dense_gemm_sgemm_gb300 import gemm_bgemm_bf16f32, gemm_hgemm_f16f32, gemm_sgemm_f32, workloads

TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


def to_device(inputs: dict) -> dict:
    return {k: v.cuda() for k, v in inputs.items()}


def run_library(w: workloads.Workload, dev: dict, stream=None):
    fn = {"f32": gemm_sgemm_f32, "f16": gemm_hgemm_f16f32, "bf16": gemm_bgemm_bf16f32}[w.dtype]
    fn(w.opA, w.opB, w.M, w.N, w.K, w.alpha, dev["A"], w.lda, dev["B"], w.ldb, w.beta,
       dev["C"], w.ldc, stream)


def np_in(t: torch.Tensor, dtype: str):
    """numpy view of an operand: fp32 values, or the raw bits of fp16 / bf16 values."""
    t = t.contiguous().cpu()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    a = t.numpy()
    return a.view(np.uint16) if dtype == "f16" else a


_np_in = np_in


def oracle_full(w: workloads.Workload, inputs: dict):
    """Oracle C (M x N) and absdot for the whole problem."""
    return oracle.gemm(w.opA, w.opB, w.M, w.N, w.K, w.alpha, _np_in(inputs["A"], w.dtype),
                       w.lda, _np_in(inputs["B"], w.dtype), w.ldb, w.beta,
                       inputs["C"].numpy(), w.ldc, dtype=w.dtype, want_absdot=True)


def oracle_points(w: workloads.Workload, inputs: dict, rows, cols):
    return oracle.gemm_points(w.opA, w.opB, w.M, w.N, w.K, w.alpha,
                              _np_in(inputs["A"], w.dtype), w.lda,
                              _np_in(inputs["B"], w.dtype), w.ldb, w.beta,
                              inputs["C"].numpy(), w.ldc, rows, cols, dtype=w.dtype)


def assert_close(w, got, ref, absdot, cin, integer=False, where=""):
    got = np.asarray(got, dtype=np.float32)
    ref = np.asarray(ref, dtype=np.float32)
    assert got.shape == ref.shape
    if integer:
        bad = got.view(np.uint32) != ref.view(np.uint32)
        if bad.any():
            i = np.argwhere(bad)[0]
            raise AssertionError(f"{w.name}{where}: not bit-exact at {tuple(i)}: "
                                 f"{got[tuple(i)]} vs {ref[tuple(i)]} ({bad.sum()} elements)")
        return
    bound = oracle.tolerance_bound(ref, absdot, w.alpha, w.beta, cin, TOL[w.dtype])
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bad = ~(err <= bound)  # NaN in got counts as bad
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{w.name}{where}: {bad.sum()} elements out of bound; first at "
                             f"{i}: got {got[i]} ref {ref[i]} err {err[i]:.3e} bound {bound[i]:.3e}")


def check_full(w, inputs, dev_c, integer=False, rows_per_chunk=2048):
    """Every element of C against the full oracle product (compared in row chunks, so the
    largest problems need only a few GB of host memory beyond the oracle's result)."""
    ref, absdot = oracle_full(w, inputs)
    got = dev_c.cpu().numpy()[:, : w.N]
    cin = inputs["C"].numpy()[:, : w.N] if w.beta != 0.0 else None
    for r0 in range(0, w.M, rows_per_chunk):
        r1 = min(w.M, r0 + rows_per_chunk)
        assert_close(w, got[r0:r1], ref[r0:r1], absdot[r0:r1],
                     None if cin is None else cin[r0:r1], integer,
                     where=f" (rows {r0}..{r1 - 1})" if w.M > rows_per_chunk else "")
