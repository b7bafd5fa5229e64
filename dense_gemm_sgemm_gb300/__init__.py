"""GEMM for one NVIDIA GB300 GPU: C = alpha * op(A) * op(B) + beta * C, row-major.

Thin Python face of the C ABI in include/gemm_gb300.h.  The functions take torch CUDA
tensors (or raw device addresses as ints), pass their addresses, sizes and the current
CUDA stream to the library, and raise GemmError on a non-OK status.  All arithmetic runs
in the library's CUDA kernels; torch only owns the memory and the stream.

    gemm_sgemm_f32(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc)
    gemm_hgemm_f16f32(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc)
    gemm_bgemm_bf16f32(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc)
    gemm_*_strided_batched(opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
                           beta, C, ldc, strideC, batch)
    gemm_*_host(... same as the single calls, A, B, C in host memory ...)
"""
from __future__ import annotations

import ctypes

from ._lib import GEMM_OP_N, GEMM_OP_T, STATUS, GemmError, library_path, load

__all__ = [
    "GEMM_OP_N", "GEMM_OP_T", "GemmError", "gemm_sgemm_f32", "gemm_hgemm_f16f32",
    "gemm_bgemm_bf16f32", "gemm_sgemm_f32_strided_batched", "gemm_hgemm_f16f32_strided_batched",
    "gemm_bgemm_bf16f32_strided_batched", "gemm_sgemm_f32_noalloc", "gemm_sgemm_f32_host",
    "gemm_hgemm_f16f32_host", "gemm_bgemm_bf16f32_host",
    "gemm_get_device_status", "gemm_status_string", "gemm_version", "gemm_tile_raster",
    "gemm_kernel_launches", "gemm_measure_fp32_fma_peak", "gemm_sgemm_configs",
    "library_path", "load", "matmul",
]


def _op(op) -> int:
    if op in (GEMM_OP_N, "N", "n"):
        return GEMM_OP_N
    if op in (GEMM_OP_T, "T", "t"):
        return GEMM_OP_T
    raise ValueError(f"op must be 'N' or 'T', got {op!r}")


def _addr(x, want_dtype=None) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    import torch

    if not isinstance(x, torch.Tensor):
        raise TypeError("operands must be torch tensors or device addresses")
    if not x.is_cuda:
        raise ValueError("operands must live in CUDA device memory")
    if want_dtype is not None and x.dtype != want_dtype:
        raise TypeError(f"expected {want_dtype}, got {x.dtype}")
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != 0:
        raise GemmError(status, what)


def gemm_sgemm_f32(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    import torch

    st = load().gemm_sgemm_f32(_op(opA), _op(opB), M, N, K, alpha, _addr(A, torch.float32), lda,
                               _addr(B, torch.float32), ldb, beta, _addr(C, torch.float32), ldc,
                               _stream(stream))
    _check(st, "gemm_sgemm_f32")


def gemm_hgemm_f16f32(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    import torch

    st = load().gemm_hgemm_f16f32(_op(opA), _op(opB), M, N, K, alpha, _addr(A, torch.float16),
                                  lda, _addr(B, torch.float16), ldb, beta,
                                  _addr(C, torch.float32), ldc, _stream(stream))
    _check(st, "gemm_hgemm_f16f32")


def gemm_bgemm_bf16f32(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    import torch

    st = load().gemm_bgemm_bf16f32(_op(opA), _op(opB), M, N, K, alpha, _addr(A, torch.bfloat16),
                                   lda, _addr(B, torch.bfloat16), ldb, beta,
                                   _addr(C, torch.float32), ldc, _stream(stream))
    _check(st, "gemm_bgemm_bf16f32")


_BATCHED = {
    "f32": ("gemm_sgemm_f32_strided_batched", "float32"),
    "f16": ("gemm_hgemm_f16f32_strided_batched", "float16"),
    "bf16": ("gemm_bgemm_bf16f32_strided_batched", "bfloat16"),
}


def _batched(kind, opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
             strideC, batch, stream):
    import torch

    name, dt = _BATCHED[kind]
    dt = getattr(torch, dt)
    st = getattr(load(), name)(_op(opA), _op(opB), M, N, K, alpha, _addr(A, dt), lda, strideA,
                               _addr(B, dt), ldb, strideB, beta, _addr(C, torch.float32), ldc,
                               strideC, batch, _stream(stream))
    _check(st, name)


def gemm_sgemm_f32_strided_batched(opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
                                   beta, C, ldc, strideC, batch, stream=None):
    _batched("f32", opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
             strideC, batch, stream)


def gemm_hgemm_f16f32_strided_batched(opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
                                      beta, C, ldc, strideC, batch, stream=None):
    _batched("f16", opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
             strideC, batch, stream)


def gemm_bgemm_bf16f32_strided_batched(opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb,
                                       strideB, beta, C, ldc, strideC, batch, stream=None):
    _batched("bf16", opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
             strideC, batch, stream)


def gemm_sgemm_f32_noalloc(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    """gemm_sgemm_f32 for callers that must not allocate device memory during the call.

    The split-K scratch is a fixed 16 MiB + 16 KiB device array owned by the library (no
    cudaMalloc ever); K is split only as far as the array holds the partial tiles (problems
    too large for that run unsplit), and calls that overlap on the GPU must not share the array.
    """
    import torch

    st = load().gemm_sgemm_f32_noalloc(_op(opA), _op(opB), M, N, K, alpha, _addr(A, torch.float32),
                                       lda, _addr(B, torch.float32), ldb, beta,
                                       _addr(C, torch.float32), ldc, _stream(stream))
    _check(st, "gemm_sgemm_f32_noalloc")


def _host_addr(x, torch_dtype: str, np_dtypes) -> int:
    """Address of a host matrix: a CPU torch tensor, a numpy array or an int address."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    import numpy as np

    if isinstance(x, np.ndarray):
        if x.dtype not in [np.dtype(d) for d in np_dtypes]:
            raise TypeError(f"expected numpy {np_dtypes}, got {x.dtype}")
        return x.ctypes.data
    import torch

    if not isinstance(x, torch.Tensor):
        raise TypeError("host operands must be CPU torch tensors, numpy arrays or addresses")
    if x.is_cuda:
        raise ValueError("the *_host entry points take host memory; use the device calls")
    if x.dtype != getattr(torch, torch_dtype):
        raise TypeError(f"expected torch.{torch_dtype}, got {x.dtype}")
    return x.data_ptr()


def _host_call(name, in_dtype, np_in, opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
               stream):
    st = getattr(load(), name)(_op(opA), _op(opB), M, N, K, alpha,
                               _host_addr(A, in_dtype, np_in), lda,
                               _host_addr(B, in_dtype, np_in), ldb, beta,
                               _host_addr(C, "float32", ["float32"]), ldc, _stream(stream))
    _check(st, name)


def gemm_sgemm_f32_host(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    """gemm_sgemm_f32 on host matrices: copies in, GEMM and copy out, in order on the
    stream; C holds the result once the stream has passed the call (pin the buffers for
    the call to be asynchronous)."""
    _host_call("gemm_sgemm_f32_host", "float32", ["float32"], opA, opB, M, N, K, alpha, A, lda,
               B, ldb, beta, C, ldc, stream)


def gemm_hgemm_f16f32_host(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    """gemm_hgemm_f16f32 on host matrices (see gemm_sgemm_f32_host)."""
    _host_call("gemm_hgemm_f16f32_host", "float16", ["float16", "uint16"], opA, opB, M, N, K,
               alpha, A, lda, B, ldb, beta, C, ldc, stream)


def gemm_bgemm_bf16f32_host(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    """gemm_bgemm_bf16f32 on host matrices (see gemm_sgemm_f32_host); numpy operands hold
    the bfloat16 bit patterns as uint16."""
    _host_call("gemm_bgemm_bf16f32_host", "bfloat16", ["uint16"], opA, opB, M, N, K, alpha, A,
               lda, B, ldb, beta, C, ldc, stream)


def gemm_get_device_status(stream=None) -> int:
    """Status code of the device error word (waits for the stream, then clears it)."""
    return int(load().gemm_get_device_status(_stream(stream)))


def gemm_status_string(status: int) -> str:
    return load().gemm_status_string(int(status)).decode()


def gemm_version() -> int:
    return int(load().gemm_version())


def gemm_kernel_launches() -> int:
    """Kernels this process has launched through the library so far (for accounting)."""
    return int(load().gemm_kernel_launches())


def gemm_measure_fp32_fma_peak(stream=None) -> float:
    """Measured FP32 multiply-add throughput of the current device in TFLOP/s (packed FMA
    chains on every SM, best of three event-timed launches; synchronises the stream)."""
    out = ctypes.c_double(0.0)
    _check(load().gemm_measure_fp32_fma_peak(_stream(stream), ctypes.byref(out)),
           "gemm_measure_fp32_fma_peak")
    return out.value


def gemm_sgemm_configs():
    """The strict-FP32 path's tile configurations as dicts (host function, no GPU)."""
    from ._lib import SgemmConfig

    out, i = [], 0
    while True:
        c = SgemmConfig()
        if load().gemm_sgemm_config(i, ctypes.byref(c)) != 0:
            return out
        d = {f: getattr(c, f) for f, _ in SgemmConfig._fields_}
        d["name"] = d["name"].decode()
        out.append(d)
        i += 1


def gemm_tile_raster(t, tiles_m, tiles_n, log_group):
    """(tile_m, tile_n) of tile t under the library's grouped raster (host function)."""
    tm, tn = ctypes.c_int64(), ctypes.c_int64()
    st = load().gemm_tile_raster(t, tiles_m, tiles_n, log_group, ctypes.byref(tm),
                                 ctypes.byref(tn))
    _check(st, "gemm_tile_raster")
    return tm.value, tn.value


def matmul(A, B, C=None, alpha=1.0, beta=0.0, opA="N", opB="N", stream=None):
    """Tensor-level convenience over the two entry points.

    A and B are 2-D CUDA tensors holding the STORED matrices (row stride = leading
    dimension, unit column stride); fp32 operands go to gemm_sgemm_f32, fp16 operands to
    gemm_hgemm_f16f32, bf16 operands to gemm_bgemm_bf16f32.  C (fp32, M x N) is created
    when omitted (then beta must be 0).
    """
    import torch

    for x in (A, B):
        if x.dim() != 2 or x.stride(1) != 1:
            raise ValueError("operands must be 2-D with unit column stride")
    M = A.shape[0] if _op(opA) == GEMM_OP_N else A.shape[1]
    K = A.shape[1] if _op(opA) == GEMM_OP_N else A.shape[0]
    N = B.shape[1] if _op(opB) == GEMM_OP_N else B.shape[0]
    kb = B.shape[0] if _op(opB) == GEMM_OP_N else B.shape[1]
    if kb != K:
        raise ValueError(f"inner dimensions differ: {K} vs {kb}")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if C.shape != (M, N) or C.stride(1) != 1 or C.dtype != torch.float32:
        raise ValueError("C must be fp32, M x N, unit column stride")
    fn = {torch.float32: gemm_sgemm_f32, torch.float16: gemm_hgemm_f16f32,
          torch.bfloat16: gemm_bgemm_bf16f32}[A.dtype]
    fn(opA, opB, M, N, K, alpha, A, max(A.stride(0), 1), B, max(B.stride(0), 1), beta, C,
       max(C.stride(0), 1), stream)
    return C
