"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes the oracle to something independent of its own code: exact rational
arithmetic on tiny shapes, numpy's own binary16 decoding, closed forms (identity,
permutation, rank-1), alpha/beta linearity, the worked examples printed on the pages
(tests/golden/), and numpy's fp64 matrix product.  ``test_planted_mistakes_are_caught``
compiles deliberately broken copies of the oracle and checks that these pins reject each.
"""
import ctypes
import itertools
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import golden_io

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ----------------------------------------------------------------------------- helpers
def _bf16_bits(values64):
    """bfloat16 bit patterns of float64 values (rounded by torch, round to nearest even)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(values64, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _store(logical, op, pad, dtype):
    """Stored buffer (flat) and ld of a logical matrix for the given op and row padding."""
    mat = np.asarray(logical, dtype=np.float64)
    stored = mat if op == "N" else mat.T
    rows, cols = stored.shape
    ld = cols + pad
    buf = np.full((rows, ld), np.nan, dtype=np.float64)
    buf[:, :cols] = stored
    if dtype == "bf16":
        return _bf16_bits(buf).reshape(-1), ld
    np_t = np.float32 if dtype == "f32" else np.float16
    return buf.astype(np_t).reshape(-1), ld


def _brute(Alog, Blog, alpha, beta, Clog):
    """Exact rational C = alpha*A*B + beta*C over Python Fractions, then rounded to fp32."""
    M, K = np.shape(Alog)
    N = np.shape(Blog)[1]
    out = np.empty((M, N), dtype=np.float32)
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(float(Alog[i][k])) * Fraction(float(Blog[k][j]))
            r = Fraction(alpha) * s
            if beta != 0:
                r += Fraction(beta) * Fraction(float(Clog[i][j]))
            out[i, j] = np.float32(float(r))
    return out


def _values(rng, shape, family):
    if family == "int":
        return rng.integers(-4, 5, size=shape).astype(np.float64)
    # dyadic rationals with few significant bits: exact in fp16, fp32 and fp64 products
    return rng.integers(-12, 13, size=shape).astype(np.float64) / 4.0


def _same(a, b):
    a = np.asarray(a, dtype=np.float32)
    b = np.asarray(b, dtype=np.float32)
    return a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32))


# ------------------------------------------------------- brute force on tiny shapes
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_brute_force_exact_rationals(dtype):
    rng = np.random.default_rng(1234)
    cases = 0
    for M, N, K in itertools.product(range(1, 8), range(1, 6), range(1, 4)):
        for opA, opB, pad in itertools.product("NT", "NT", (0, 3)):
            family = "int" if (M + N + K + pad) % 2 == 0 else "dyadic"
            Alog = _values(rng, (M, K), family)
            Blog = _values(rng, (K, N), family)
            Clog = _values(rng, (M, N), "dyadic")
            alpha, beta = (1.0, 0.0) if family == "int" else (0.75, -1.25)
            A, lda = _store(Alog, opA, pad, dtype)
            B, ldb = _store(Blog, opB, pad, dtype)
            Cin, ldc = _store(Clog, "N", pad, "f32")
            got = oracle.gemm(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, Cin, ldc,
                              dtype=dtype, threads=1)
            want = _brute(Alog, Blog, alpha, beta, Clog)
            assert _same(got, want), (M, N, K, opA, opB, pad, dtype)
            cases += 1
    assert cases == 7 * 5 * 3 * 8


def test_half_decoder_matches_numpy_on_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    lib = oracle._load()
    got = np.array([lib.gemm_oracle_half_to_double(int(b)) for b in bits])
    both_nan = np.isnan(want) & np.isnan(got)
    assert np.all(both_nan | (got == want))
    assert np.array_equal(np.signbit(got[~both_nan]), np.signbit(want[~both_nan]))


def test_bf16_decoder_matches_torch_on_every_bit_pattern():
    import torch

    bits = np.arange(1 << 16, dtype=np.uint16)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    both_nan = np.isnan(want) & np.isnan(got)
    assert np.all(both_nan | (got == want))
    assert np.array_equal(np.signbit(got[~both_nan]), np.signbit(want[~both_nan]))


# ----------------------------------------------------------------- closed forms
@pytest.mark.parametrize("opA,opB", list(itertools.product("NT", "NT")))
def test_identity_and_permutation(opA, opB):
    rng = np.random.default_rng(7)
    M, K = 37, 53
    Alog = rng.uniform(-1, 1, size=(M, K)).astype(np.float32).astype(np.float64)
    I = np.eye(K)
    A, lda = _store(Alog, opA, 2, "f32")
    Ib, ldi = _store(I, opB, 1, "f32")
    got = oracle.gemm(opA, opB, M, K, K, 1.0, A, lda, Ib, ldi)
    assert _same(got, Alog.astype(np.float32))  # A * I = A
    perm = rng.permutation(M)
    P = np.zeros((M, M))
    P[np.arange(M), perm] = 1.0
    Pb, ldp = _store(P, opA, 0, "f32")
    A2, lda2 = _store(Alog, opB, 0, "f32")
    got = oracle.gemm(opA, opB, M, K, M, 1.0, Pb, ldp, A2, lda2)
    assert _same(got, Alog[perm].astype(np.float32))  # P * A permutes the rows of A


@pytest.mark.parametrize("K", [1, 2, 5, 64, 1000])
def test_rank1_closed_form(K):
    rng = np.random.default_rng(K)
    M, N = 19, 23
    u = rng.integers(-8, 9, size=M).astype(np.float64)
    v = 2.0 ** rng.integers(-6, 7, size=N)
    Alog = np.outer(u, np.ones(K))  # u * 1^T
    Blog = np.outer(np.ones(K), v)  # 1 * v^T
    for opA, opB in itertools.product("NT", "NT"):
        A, lda = _store(Alog, opA, 0, "f32")
        B, ldb = _store(Blog, opB, 0, "f32")
        got = oracle.gemm(opA, opB, M, N, K, 1.0, A, lda, B, ldb)
        assert _same(got, (K * np.outer(u, v)).astype(np.float32))


def test_alpha_beta_linearity_and_degenerate_cases():
    rng = np.random.default_rng(3)
    M, N, K = 24, 31, 40
    A = _values(rng, (M, K), "int").astype(np.float32)
    B = _values(rng, (K, N), "int").astype(np.float32)
    Cin = _values(rng, (M, N), "dyadic").astype(np.float32)
    a1, a2, beta = 0.5, -1.25, 0.75
    c12 = oracle.gemm("N", "N", M, N, K, a1 + a2, A, K, B, N, beta, Cin, N)
    c1 = oracle.gemm("N", "N", M, N, K, a1, A, K, B, N, beta, Cin, N)
    c0 = oracle.gemm("N", "N", M, N, K, 1.0, A, K, B, N)
    assert _same(c12, c1 + np.float32(a2) * c0)
    # K == 0: the product is empty, C = beta * Cin
    c = oracle.gemm("N", "N", M, N, 0, 3.0, np.zeros(1, np.float32), 1,
                    np.zeros(1, np.float32), N, beta, Cin, N)
    assert _same(c, np.float32(beta) * Cin)
    # alpha == 0: C = beta * Cin
    c = oracle.gemm("N", "N", M, N, K, 0.0, A, K, B, N, beta, Cin, N)
    assert _same(c, np.float32(beta) * Cin)
    # beta == 0 never reads Cin (NaN and Inf do not propagate)
    poison = np.full((M, N), np.nan, np.float32)
    poison[0, 0] = np.inf
    c = oracle.gemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, poison, N)
    assert np.isfinite(c).all() and _same(c, c0)


# ------------------------------------------------------------- the pages' examples
def test_leading_dimension_worked_example():
    g = golden_io.read("ld_padded_2x3.txt")
    rows, cols, ld = (golden_io.scalar(g, k) for k in ("rows", "cols", "ld"))
    logical = np.array([float(x) for x in g["logical"][0]]).reshape(rows, cols)
    storage = np.array([np.nan if x == "pad" else float(x) for x in g["storage"][0]],
                       dtype=np.float32)
    assert storage.size == rows * ld
    I = np.eye(cols, dtype=np.float32).reshape(-1)
    got = oracle.gemm("N", "N", rows, cols, cols, 1.0, storage, ld, I, cols)
    assert _same(got, logical.astype(np.float32))
    # the same storage read as op(A) = T is the 3 x 2 transpose
    got = oracle.gemm("T", "N", cols, rows, rows, 1.0, storage, ld,
                      np.eye(rows, dtype=np.float32).reshape(-1), rows)
    assert _same(got, logical.T.astype(np.float32))


def test_row_major_swap_worked_example():
    g = golden_io.read("rowmajor_swap_2x3x4.txt")
    M, N, K = (golden_io.scalar(g, k) for k in ("M", "N", "K"))
    rng = np.random.default_rng(11)
    A = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    B = rng.integers(-4, 5, size=(K, N)).astype(np.float32)
    C = oracle.gemm("N", "N", M, N, K, 1.0, A, K, B, N)
    # Column-major reading: the B buffer is B^T (N x K) and the A buffer is A^T (K x M).
    # In row-major terms that is op = T on each buffer, with the operands swapped.
    D = oracle.gemm("T", "T", N, M, K, 1.0, B, N, A, K)  # D = B^T A^T = C^T, N x M
    ct_column_major_memory = D.T.reshape(-1)  # column-major storage of D
    assert _same(ct_column_major_memory, C.reshape(-1))
    names = g["ct_memory_order"][0]
    idx = [int(n[1]) * N + int(n[2]) for n in names]
    assert _same(ct_column_major_memory, C.reshape(-1)[idx])


# ------------------------------------------------------------- library cross-check
@pytest.mark.parametrize("opA,opB", list(itertools.product("NT", "NT")))
@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_against_numpy_fp64_product(opA, opB, dtype):
    rng = np.random.default_rng(5)
    M, N, K = 67, 45, 129
    np_t = np.float32 if dtype == "f32" else np.float16
    Alog = rng.uniform(-1, 1, size=(M, K)).astype(np_t).astype(np.float64)
    Blog = rng.uniform(-1, 1, size=(K, N)).astype(np_t).astype(np.float64)
    Clog = rng.uniform(-1, 1, size=(M, N)).astype(np.float32).astype(np.float64)
    A, lda = _store(Alog, opA, 1, dtype)
    B, ldb = _store(Blog, opB, 2, dtype)
    got, absdot = oracle.gemm(opA, opB, M, N, K, 1.5, A, lda, B, ldb, -0.5,
                              Clog.astype(np.float32), N, dtype=dtype, want_absdot=True)
    want = (1.5 * (Alog @ Blog) - 0.5 * Clog).astype(np.float32)
    ulps = np.abs(got.view(np.int32).astype(np.int64) - want.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1
    assert np.allclose(absdot, np.abs(Alog) @ np.abs(Blog), rtol=1e-12, atol=0)


def test_points_threads_and_full_agree():
    rng = np.random.default_rng(9)
    M, N, K = 50, 70, 90
    A = rng.standard_normal((K, M)).astype(np.float32)  # stored for opA = T
    B = rng.standard_normal((N, K)).astype(np.float32)  # stored for opB = T
    Cin = rng.standard_normal((M, N)).astype(np.float32)
    c1 = oracle.gemm("T", "T", M, N, K, 0.3, A, M, B, K, 2.0, Cin, N, threads=1)
    c8 = oracle.gemm("T", "T", M, N, K, 0.3, A, M, B, K, 2.0, Cin, N, threads=8)
    assert _same(c1, c8)
    rows = rng.integers(0, M, 200)
    cols = rng.integers(0, N, 200)
    pts, _ = oracle.gemm_points("T", "T", M, N, K, 0.3, A, M, B, K, 2.0, Cin, N, rows, cols)
    assert _same(pts, c1[rows, cols])
    # i-k-j (op(B) = N) and per-element (op(B) = T) orders give the same bits
    Bn = np.ascontiguousarray(B.T)
    cn = oracle.gemm("T", "N", M, N, K, 0.3, A, M, Bn, N, 2.0, Cin, N)
    assert _same(cn, c1)


def test_bad_arguments_are_rejected():
    z = np.zeros(16, np.float32)
    with pytest.raises(ValueError):
        oracle.gemm("N", "N", 2, 2, 4, 1.0, z, 3, z, 2)  # lda < K
    with pytest.raises(ValueError):
        oracle.gemm("N", "T", 2, 2, 4, 1.0, z, 4, z, 3)  # ldb < K for op(B) = T
    with pytest.raises(ValueError):
        oracle.gemm("X", "N", 2, 2, 2, 1.0, z, 2, z, 2)


# ------------------------------------------------------------ planted mistakes
_MUTANTS = {
    "opA_T_index_transposed": ("k * j->lda + i", "i * j->lda + k"),
    "opB_T_index_transposed": ("c * j->ldb + k", "k * j->ldb + c"),
    "last_k_dropped": ("for (int64_t k = 0; k < j->K; ++k) {\n        double p",
                       "for (int64_t k = 0; k + 1 < j->K; ++k) {\n        double p"),
    "beta_sign_flipped": ("if (j->beta != 0.0) r += j->beta", "if (j->beta != 0.0) r -= j->beta"),
    "half_exponent_bias_off_by_one": ("expo - 25", "expo - 24"),
    "alpha_ignored_in_row_kernel": ("double r = j->alpha * acc[c];", "double r = acc[c];"),
    "bf16_bits_misplaced": ("uint32_t bits = (uint32_t)h << 16;", "uint32_t bits = (uint32_t)h << 15;"),
}


def _compile_mutant(tmp_path, name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gemm_oracle.c")).read()
    assert old in src, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-pthread", str(path), "-o", str(so),
                    "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    return lib


def _pins_pass_with(lib):
    """Re-run a compact subset of the pins above against another build of the oracle."""
    saved = oracle._lib
    try:
        i64, dbl, ip, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_int, ctypes.c_void_p
        full = [ip, ip, i64, i64, i64, dbl, vp, i64, vp, i64, dbl, vp, i64, vp, i64, vp, i64, ip]
        for nm in ("gemm_oracle_f32", "gemm_oracle_f16", "gemm_oracle_bf16"):
            getattr(lib, nm).argtypes = full
            getattr(lib, nm).restype = ctypes.c_int
        for dec in ("gemm_oracle_half_to_double", "gemm_oracle_bf16_to_double"):
            getattr(lib, dec).argtypes = [ctypes.c_uint16]
            getattr(lib, dec).restype = ctypes.c_double
        oracle._lib = lib
        rng = np.random.default_rng(2024)
        for dtype in ("f32", "f16", "bf16"):
            for (M, N, K), opA, opB in itertools.product([(3, 4, 3), (5, 2, 2), (2, 3, 1)],
                                                         "NT", "NT"):
                Alog = _values(rng, (M, K), "dyadic")
                Blog = _values(rng, (K, N), "dyadic")
                Clog = _values(rng, (M, N), "dyadic")
                A, lda = _store(Alog, opA, 1, dtype)
                B, ldb = _store(Blog, opB, 1, dtype)
                got = oracle.gemm(opA, opB, M, N, K, 0.75, A, lda, B, ldb, -1.25,
                                  Clog.astype(np.float32), N, dtype=dtype, threads=1)
                if not _same(got, _brute(Alog, Blog, 0.75, -1.25, Clog)):
                    return False
        return True
    finally:
        oracle._lib = saved


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_planted_mistakes_are_caught(tmp_path, name):
    old, new = _MUTANTS[name]
    lib = _compile_mutant(tmp_path, name, old, new)
    assert not _pins_pass_with(lib), f"planted mistake {name} was not caught"


def test_unmutated_copy_passes_the_same_pins(tmp_path):
    lib = _compile_mutant(tmp_path, "identity", "#include <math.h>", "#include <math.h>")
    assert _pins_pass_with(lib)
