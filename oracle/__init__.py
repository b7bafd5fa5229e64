"""CPU oracle for C = alpha*op(A)*op(B) + beta*C -- TEST INFRASTRUCTURE ONLY.

This package is the correctness anchor of the GPU library.  Only the test-suite, the
smoke check and the CPU-baseline leg of ``bench.py`` may import it; the library itself
never does, and the two share no code.  The arithmetic lives in ``gemm_oracle.c`` (plain
C, fp64 accumulation in k order, one thread per row range); this module compiles it with
gcc and marshals numpy arrays into it.

Definition followed (copecc.github.io "GEMM" page, section "核心问题与运算特征", and
yekq.top "LeetGPU 第二题", section "题目描述")::

    C[i][j] = fl32( alpha * sum_k opA(i,k) * opB(k,j) + beta * Cin[i][j] )

with the row-major leading-dimension convention of the copecc "Leading Dimension" section.
beta == 0 never reads Cin.  fp16 inputs are passed as their raw bit patterns and decoded
exactly by the C code.

Every function here is pinned by ``tests/test_oracle_pins.py`` (exact-rational brute
force, identity/permutation, rank-1 closed forms, alpha/beta linearity, the worked
examples of the pages stored under ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

OP_N = 0
OP_T = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into oracle/_build/liboracle.so (portable C, no ISA flags)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, dbl, ip = ctypes.c_int64, ctypes.c_double, ctypes.c_int
        vp = ctypes.c_void_p
        full = [ip, ip, i64, i64, i64, dbl, vp, i64, vp, i64, dbl, vp, i64, vp, i64, vp, i64, ip]
        pts = [ip, ip, i64, i64, i64, dbl, vp, i64, vp, i64, dbl, vp, i64, vp, vp, i64, vp, vp, ip]
        for name, args in (("gemm_oracle_f32", full), ("gemm_oracle_f16", full),
                           ("gemm_oracle_bf16", full), ("gemm_oracle_f32_points", pts),
                           ("gemm_oracle_f16_points", pts), ("gemm_oracle_bf16_points", pts)):
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        for dec in ("gemm_oracle_half_to_double", "gemm_oracle_bf16_to_double"):
            getattr(lib, dec).argtypes = [ctypes.c_uint16]
            getattr(lib, dec).restype = ctypes.c_double
        _lib = lib
        return lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _op(op) -> int:
    if op in (OP_N, "N", "n"):
        return OP_N
    if op in (OP_T, "T", "t"):
        return OP_T
    raise ValueError(f"op must be 'N' or 'T', got {op!r}")


def _flat(x, dtype):
    """Contiguous 1-D view of x with the given element type (fp16/bf16 passed as raw bits)."""
    a = np.asarray(x)
    if dtype == "bf16":
        if a.dtype != np.uint16:
            raise TypeError("bf16 operands must be uint16 bit patterns")
    elif dtype == "f16":
        if a.dtype == np.float16:
            a = a.view(np.uint16)
        if a.dtype != np.uint16:
            raise TypeError("fp16 operands must be numpy float16 or uint16 bit patterns")
    else:
        if a.dtype != np.float32:
            raise TypeError("fp32 operands must be numpy float32")
    return np.ascontiguousarray(a).reshape(-1)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check_extent(name, buf, rows, cols, ld):
    if rows == 0 or cols == 0:
        return
    need = (rows - 1) * ld + cols
    if buf.size < need:
        raise ValueError(f"{name}: buffer has {buf.size} elements, needs {need}")


def gemm(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta=0.0, Cin=None, ldcin=None,
         dtype="f32", want_absdot=False, threads=None):
    """Full oracle product.  Returns C (M x N float32) and, if asked, absdot (M x N fp64)."""
    opA, opB = _op(opA), _op(opB)
    A = _flat(A, dtype)
    B = _flat(B, dtype)
    _check_extent("A", A, M if opA == OP_N else K, K if opA == OP_N else M, lda)
    _check_extent("B", B, K if opB == OP_N else N, N if opB == OP_N else K, ldb)
    cin = None
    if beta != 0.0:
        if Cin is None:
            raise ValueError("beta != 0 needs Cin")
        cin = _flat(Cin, "f32")
        ldcin = N if ldcin is None else ldcin
        _check_extent("Cin", cin, M, N, ldcin)
    C = np.empty((M, N), dtype=np.float32)
    ab = np.empty((M, N), dtype=np.float64) if want_absdot else None
    fn = {"f32": _load().gemm_oracle_f32, "f16": _load().gemm_oracle_f16,
          "bf16": _load().gemm_oracle_bf16}[dtype]
    rc = fn(opA, opB, M, N, K, float(alpha), _ptr(A), lda, _ptr(B), ldb, float(beta),
            _ptr(cin), ldcin or 0, _ptr(C), max(N, 1), _ptr(ab), max(N, 1),
            threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return (C, ab) if want_absdot else C


def gemm_points(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, Cin, ldcin, rows, cols,
                dtype="f32", threads=None):
    """Oracle value and absdot of C at the listed (row, col) positions only."""
    opA, opB = _op(opA), _op(opB)
    A = _flat(A, dtype)
    B = _flat(B, dtype)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in length")
    cin = None
    if beta != 0.0:
        cin = _flat(Cin, "f32")
    out = np.empty(rows.size, dtype=np.float32)
    ab = np.empty(rows.size, dtype=np.float64)
    fn = {"f32": _load().gemm_oracle_f32_points, "f16": _load().gemm_oracle_f16_points,
          "bf16": _load().gemm_oracle_bf16_points}[dtype]
    rc = fn(opA, opB, M, N, K, float(alpha), _ptr(A), lda, _ptr(B), ldb, float(beta),
            _ptr(cin), ldcin or 0, _ptr(rows), _ptr(cols), rows.size, _ptr(out), _ptr(ab),
            threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out, ab


def half_to_double(bits: int) -> float:
    """The oracle's own binary16 decoder (exposed so the tests can pin it)."""
    return float(_load().gemm_oracle_half_to_double(int(bits) & 0xFFFF))


def bf16_to_double(bits: int) -> float:
    """The oracle's own bfloat16 decoder (exposed so the tests can pin it)."""
    return float(_load().gemm_oracle_bf16_to_double(int(bits) & 0xFFFF))


def tolerance_bound(ref, absdot, alpha, beta, cin, rel_tol):
    """Per-element acceptance bound of the parity tests.

    |C - C_ref| <= rel_tol * (|alpha| * sum_k |a_ik b_kj| + |beta| * |Cin_ij|) + ulp32(|C_ref|).
    The last term allows the single final rounding to fp32.
    """
    bound = rel_tol * abs(alpha) * np.asarray(absdot, dtype=np.float64)
    if beta != 0.0 and cin is not None:
        bound = bound + rel_tol * abs(beta) * np.abs(np.asarray(cin, dtype=np.float64))
    r = np.abs(np.asarray(ref, dtype=np.float32))
    ulp = np.spacing(r).astype(np.float64)
    return bound + ulp
