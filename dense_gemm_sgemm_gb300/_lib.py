"""ctypes binding of include/gemm_gb300.h (argument marshalling only).

The shared library is built in-tree by ``dense_gemm_sgemm_gb300.build``.  Nothing here
computes any part of a GEMM: every call goes to the CUDA library, and a missing library is
an ImportError, never a silent fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading


GEMM_OP_N = 0
GEMM_OP_T = 1

STATUS = {
    0: "GEMM_OK",
    1: "GEMM_ERR_INVALID_VALUE",
    2: "GEMM_ERR_MISALIGNED",
    3: "GEMM_ERR_UNSUPPORTED",
    4: "GEMM_ERR_LAUNCH",
    5: "GEMM_ERR_DEVICE_TIMEOUT",
    6: "GEMM_ERR_NO_DEVICE",
}

# Every symbol include/gemm_gb300.h declares, with (restype, argtypes).
_i64, _f32, _int, _vp = ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_void_p
_GEMM_ARGS = [_int, _int, _i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _vp]
_BATCHED_ARGS = [_int, _int, _i64, _i64, _i64, _f32, _vp, _i64, _i64, _vp, _i64, _i64, _f32, _vp,
                 _i64, _i64, _i64, _vp]
SIGNATURES = {
    "gemm_sgemm_f32": (_int, _GEMM_ARGS),
    "gemm_hgemm_f16f32": (_int, _GEMM_ARGS),
    "gemm_bgemm_bf16f32": (_int, _GEMM_ARGS),
    "gemm_sgemm_f32_strided_batched": (_int, _BATCHED_ARGS),
    "gemm_hgemm_f16f32_strided_batched": (_int, _BATCHED_ARGS),
    "gemm_bgemm_bf16f32_strided_batched": (_int, _BATCHED_ARGS),
    "gemm_sgemm_f32_noalloc": (_int, _GEMM_ARGS),
    "gemm_sgemm_f32_host": (_int, _GEMM_ARGS),
    "gemm_hgemm_f16f32_host": (_int, _GEMM_ARGS),
    "gemm_bgemm_bf16f32_host": (_int, _GEMM_ARGS),
    "gemm_get_device_status": (_int, [_vp]),
    "gemm_status_string": (ctypes.c_char_p, [_int]),
    "gemm_version": (_int, []),
    "gemm_kernel_launches": (ctypes.c_uint64, []),
    "gemm_measure_fp32_fma_peak": (_int, [_vp, ctypes.POINTER(ctypes.c_double)]),
    "gemm_tile_raster": (_int, [_i64, _i64, _i64, _int, ctypes.POINTER(_i64),
                                ctypes.POINTER(_i64)]),
    "gemm_sgemm_config": (_int, [_int, _vp]),
}

class SgemmConfig(ctypes.Structure):
    """gemm_sgemm_config_t of include/gemm_gb300.h."""
    _fields_ = [("name", ctypes.c_char)] + [(f, ctypes.c_int) for f in (
        "bm", "bn", "bk", "tm", "tn", "stages", "threads", "ctas_per_sm", "row_pad", "smem_bytes")]


_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = STATUS.get(status, f"status {status}")
        super().__init__(f"{what}: {name}" if what else name)


def library_path() -> str:
    from . import build as _build

    return _build.LIB_PATH


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """The loaded CUDA library; raises ImportError when it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise ImportError(
                    f"{path} is missing: build it with `python -m dense_gemm_sgemm_gb300.build`")
            from . import build as _build

            _build.build()
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib
