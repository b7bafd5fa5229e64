"""Pins of the acceptance rule that decides every floating-point parity test (CPU only).

The rule, from the stated tolerances of the method (1e-5 of sum_k |a_ik b_kj| for strict
FP32, 2e-3 for 16-bit inputs with fp32 accumulation), scaled by |alpha| and extended by the
beta term and one fp32 ulp of the reference for the final rounding:

    |C - C_ref| <= tol * (|alpha| * sum_k |a_ik b_kj| + |beta| * |Cin_ij|) + ulp32(|C_ref|)

Each expected bound below was worked out by hand (the ulp of a float32 in [2^e, 2^(e+1)) is
2^(e-23)) and is written as a literal, so a slip in oracle.tolerance_bound -- a dropped
|alpha|, the beta term read when beta == 0, the wrong tolerance for a type, the ulp taken at
the wrong magnitude -- fails one of them.  The negative tests check that tests.parity
rejects a result just outside the bound and accepts one just inside.
"""
import numpy as np
import pytest

import oracle
from dense_gemm_sgemm_gb300 import workloads
from tests import parity


def _bound(ref, absdot, alpha, beta, cin, tol):
    return float(oracle.tolerance_bound(np.array([ref], dtype=np.float32), np.array([absdot]),
                                        alpha, beta, None if cin is None else np.array([cin]),
                                        tol)[0])


def test_stated_tolerances():
    assert parity.TOL == {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


@pytest.mark.parametrize("ref,absdot,alpha,beta,cin,tol,expected", [
    # negative alpha: 1e-5 * 2 * 1000 + 2^-24 (0.75 lies in [0.5, 1))
    (0.75, 1000.0, -2.0, 0.0, None, 1e-5, 0.020000059604644775),
    # beta == 0: a NaN Cin is never part of the bound
    (0.75, 1000.0, -2.0, 0.0, float("nan"), 1e-5, 0.020000059604644775),
    # both terms: 1e-5 * 1.5 * 10 + 1e-5 * 0.5 * 3 + 2^-23
    (1.0, 10.0, 1.5, -0.5, 3.0, 1e-5, 0.00016511920928955078),
    # fp16 inputs: 2e-3 * 0.5 + 2e-3 * 0.25 + 2^-22 (|-2| lies in [2, 4))
    (-2.0, 0.5, 1.0, 1.0, -0.25, 2e-3, 0.0015002384185791016),
    # the ulp floor on either side of a power of two
    (2.0, 0.0, 1.0, 0.0, None, 1e-5, 2.384185791015625e-07),
    (1.99999988079071044921875, 0.0, 1.0, 0.0, None, 1e-5, 1.1920928955078125e-07),
    (-0.5, 0.0, 1.0, 0.0, None, 1e-5, 5.9604644775390625e-08),
    # an exact zero: the smallest fp32 subnormal, 2^-149
    (0.0, 0.0, 1.0, 0.0, None, 1e-5, 1.401298464324817e-45),
])
def test_bound_on_hand_worked_cases(ref, absdot, alpha, beta, cin, tol, expected):
    got = _bound(ref, absdot, alpha, beta, cin, tol)
    assert got == pytest.approx(expected, rel=1e-12, abs=0.0)


def _w(dtype, alpha=1.0, beta=0.0):
    return workloads.Workload("pin", dtype, 1, 1, 1, alpha=alpha, beta=beta)


def _check(w, got, ref, absdot, cin=None):
    parity.assert_close(w, np.array([[got]], dtype=np.float32), np.array([[ref]], dtype=np.float32),
                        np.array([[absdot]]), None if cin is None else np.array([[cin]]))


def test_result_just_inside_the_bound_passes_and_just_outside_fails():
    # bound = 1e-5 * 100 + 2^-24 = 1.0000596e-3; fp32 rounding of 0.5 + d is below 3e-8
    w = _w("f32")
    _check(w, 0.5 + 0.99e-3, 0.5, 100.0)
    _check(w, 0.5 - 0.99e-3, 0.5, 100.0)
    with pytest.raises(AssertionError):
        _check(w, 0.5 + 1.01e-3, 0.5, 100.0)
    with pytest.raises(AssertionError):
        _check(w, 0.5 - 1.01e-3, 0.5, 100.0)


def test_negative_alpha_scales_the_bound_by_its_magnitude():
    w = _w("f32", alpha=-1.0)
    _check(w, 0.5 + 0.99e-3, 0.5, 100.0)
    with pytest.raises(AssertionError):
        _check(w, 0.5 + 1.01e-3, 0.5, 100.0)


def test_beta_term_widens_the_bound_only_when_beta_is_nonzero():
    # tol * |beta| * |Cin| = 1e-5 * 0.5 * 400 = 2e-3 on top of 1e-5 * 100 = 1e-3
    _check(_w("f32", beta=-0.5), 0.5 + 2.9e-3, 0.5, 100.0, cin=400.0)
    with pytest.raises(AssertionError):
        _check(_w("f32", beta=-0.5), 0.5 + 3.1e-3, 0.5, 100.0, cin=400.0)


def test_the_type_selects_the_tolerance():
    # 0.1 off with sum |ab| = 100: inside 2e-3 * 100 = 0.2 (16-bit inputs), far outside the
    # FP32 bound of 1e-3
    _check(_w("f16"), 0.6, 0.5, 100.0)
    _check(_w("bf16"), 0.6, 0.5, 100.0)
    with pytest.raises(AssertionError):
        _check(_w("f32"), 0.6, 0.5, 100.0)


def test_nan_result_fails():
    with pytest.raises(AssertionError):
        _check(_w("f32"), float("nan"), 0.5, 100.0)


def test_integer_mode_demands_identical_bits():
    ref = np.array([[3.0]], dtype=np.float32)
    one_ulp_up = np.nextafter(ref, np.float32(4.0))
    parity.assert_close(_w("f32"), ref.copy(), ref, np.array([[1.0]]), None, integer=True)
    with pytest.raises(AssertionError):
        parity.assert_close(_w("f32"), one_ulp_up, ref, np.array([[1.0]]), None, integer=True)
    # -0.0 and +0.0 differ in their bits
    with pytest.raises(AssertionError):
        parity.assert_close(_w("f32"), np.array([[-0.0]], dtype=np.float32),
                            np.array([[0.0]], dtype=np.float32), np.array([[0.0]]), None,
                            integer=True)


# Plausible slips, each planted into a copy of tolerance_bound's own source: every one must
# break at least one of the hand-worked cases above.
_MUTANTS = {
    "alpha sign kept": ("abs(alpha)", "alpha"),
    "alpha dropped": ("rel_tol * abs(alpha) * ", "rel_tol * "),
    "beta term always read": ("if beta != 0.0 and cin is not None:", "if cin is not None:"),
    "beta term dropped": ("bound = bound + rel_tol * abs(beta)", "bound = bound + 0.0 * abs(beta)"),
    "ulp of the next power of two": ("np.spacing(r)", "np.spacing(2 * r)"),
    "ulp dropped": ("return bound + ulp", "return bound"),
    "ulp in fp64": ("np.asarray(ref, dtype=np.float32)", "np.asarray(ref, dtype=np.float64)"),
}


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_planted_mistakes_are_caught(name):
    import inspect
    import textwrap

    src = textwrap.dedent(inspect.getsource(oracle.tolerance_bound))
    old, new = _MUTANTS[name]
    assert old in src, f"mutation site for {name!r} not found"
    ns = {"np": np}
    exec(compile(src.replace(old, new, 1), "<mutant>", "exec"), ns)
    mutant = ns["tolerance_bound"]
    cases = test_bound_on_hand_worked_cases.pytestmark[0].args[1]
    caught = False
    for ref, absdot, alpha, beta, cin, tol, expected in cases:
        got = float(mutant(np.array([ref], dtype=np.float32), np.array([absdot]), alpha, beta,
                           None if cin is None else np.array([cin]), tol)[0])
        if not got == pytest.approx(expected, rel=1e-12, abs=0.0):
            caught = True
            break
    assert caught, f"the mutant {name!r} passes every hand-worked case"
