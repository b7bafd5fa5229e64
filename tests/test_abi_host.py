"""Host-side checks of the C ABI that need no GPU: the library loads, exports every symbol
the header declares, validates arguments before touching a device, and its tile raster
reproduces the worked example of the pages."""
import ctypes
import os
import re

import pytest

import dense_gemm_sgemm_gb300 as g
from dense_gemm_sgemm_gb300 import _lib, build
from tests import golden_io

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "gemm_gb300.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "gemm_sgemm_f32" in names and "gemm_hgemm_f16f32" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_status_strings_and_version(lib):
    for code, name in _lib.STATUS.items():
        assert g.gemm_status_string(code).startswith(name)
    assert "unknown" in g.gemm_status_string(99)
    assert g.gemm_version() >= 100


def test_tile_raster_matches_block_swizzle_example(lib):
    d = golden_io.read("block_swizzle_16.txt")
    log_tile = golden_io.scalar(d, "log_tile")
    count = golden_io.scalar(d, "count")
    side = 1 << log_tile
    assert count == side * side
    picture = [[int(x) for x in row] for row in d["row"]]
    for t in range(count):
        tm, tn = g.gemm_tile_raster(t, side, side, log_tile)
        assert picture[tm][tn] == t


@pytest.mark.parametrize("tiles_m,tiles_n,log_group", [(7, 5, 1), (13, 9, 3), (1, 40, 2), (33, 1, 4)])
def test_tile_raster_is_a_bijection_with_grouped_order(lib, tiles_m, tiles_n, log_group):
    seen = set()
    prev = None
    for t in range(tiles_m * tiles_n):
        tm, tn = g.gemm_tile_raster(t, tiles_m, tiles_n, log_group)
        assert 0 <= tm < tiles_m and 0 <= tn < tiles_n
        seen.add((tm, tn))
        if prev is not None and tm // (1 << log_group) == prev[0] // (1 << log_group):
            assert tn >= prev[1]  # within a group, columns never go back
        prev = (tm, tn)
    assert len(seen) == tiles_m * tiles_n
    with pytest.raises(g.GemmError):
        g.gemm_tile_raster(tiles_m * tiles_n, tiles_m, tiles_n, log_group)


def test_argument_validation_needs_no_device(lib):
    f = lib.gemm_sgemm_f32
    h = lib.gemm_hgemm_f16f32
    P = 4096  # a fake, never dereferenced address: every call below returns before any launch
    assert f(2, 0, 4, 4, 4, 1.0, P, 4, P, 4, 0.0, P, 4, None) == 1      # bad op
    assert f(0, 0, -1, 4, 4, 1.0, P, 4, P, 4, 0.0, P, 4, None) == 1     # negative M
    assert f(0, 0, 4, 4, 4, 1.0, P, 3, P, 4, 0.0, P, 4, None) == 1      # lda < K
    assert f(1, 0, 4, 4, 4, 1.0, P, 3, P, 4, 0.0, P, 4, None) == 1      # lda < M (op T)
    assert f(0, 1, 4, 4, 5, 1.0, P, 5, P, 4, 0.0, P, 4, None) == 1      # ldb < K (op T)
    assert f(0, 0, 4, 4, 4, 1.0, P, 4, P, 4, 0.0, P, 3, None) == 1      # ldc < N
    assert f(0, 0, 4, 4, 4, 1.0, None, 4, P, 4, 0.0, P, 4, None) == 1   # NULL A
    assert f(0, 0, 4, 4, 4, 1.0, P, 4, P, 4, 0.0, None, 4, None) == 1   # NULL C
    assert f(0, 0, 0, 4, 4, 1.0, None, 4, None, 4, 0.0, None, 4, None) == 0  # empty: no launch
    assert f(0, 0, 1 << 31, 4, 4, 1.0, P, 4, P, 4, 0.0, P, 4, None) == 3
    assert f(0, 0, 4, 4, 4, 1.0, P + 2, 4, P, 4, 0.0, P, 4, None) == 2  # A not 4-byte aligned
    assert h(0, 0, 4, 4, 8, 1.0, P + 1, 8, P, 8, 0.0, P, 4, None) == 2  # A not 2-byte aligned
    assert h(0, 0, 4, 4, 8, 1.0, P, 8, P + 3, 8, 0.0, P, 4, None) == 2  # B not 2-byte aligned
    assert h(0, 0, 4, 4, 8, 1.0, P, 8, P, 8, 0.0, P + 2, 4, None) == 2  # C not 4-byte aligned
    # K == 0 or alpha == 0 does not need A or B
    assert f(0, 0, 0, 0, 0, 0.0, None, 1, None, 1, 0.0, None, 1, None) == 0


def test_binding_refuses_cpu_tensors(lib):
    import torch

    x = torch.zeros(4, 4)
    with pytest.raises(ValueError):
        g.gemm_sgemm_f32("N", "N", 4, 4, 4, 1.0, x, 4, x, 4, 0.0, x, 4, stream=0)


def test_host_entry_validation_needs_no_device(lib):
    # The *_host entry points validate like the device calls before any copy or allocation.
    P = 4096  # never dereferenced: every call below returns first
    for f in (lib.gemm_sgemm_f32_host, lib.gemm_hgemm_f16f32_host, lib.gemm_bgemm_bf16f32_host):
        assert f(2, 0, 4, 4, 4, 1.0, P, 4, P, 4, 0.0, P, 4, None) == 1      # bad op
        assert f(0, 0, 4, 4, 4, 1.0, P, 3, P, 4, 0.0, P, 4, None) == 1      # lda < K
        assert f(0, 0, 4, 4, 4, 1.0, P, 4, P, 4, 0.0, P, 3, None) == 1      # ldc < N
        assert f(0, 0, 4, 4, 4, 1.0, None, 4, P, 4, 0.0, P, 4, None) == 1   # NULL A
        assert f(0, 0, 4, 4, 4, 1.0, P, 4, P, 4, 0.0, None, 4, None) == 1   # NULL C
        assert f(0, 0, 0, 4, 4, 1.0, None, 4, None, 4, 0.0, None, 4, None) == 0  # empty: nothing
        assert f(0, 0, 1 << 31, 4, 4, 1.0, P, 4, P, 4, 0.0, P, 4, None) == 3


def test_binding_host_entry_refuses_wrong_types(lib):
    import numpy as np
    import torch

    a = np.zeros((4, 4), dtype=np.float64)
    with pytest.raises(TypeError):
        g.gemm_sgemm_f32_host("N", "N", 4, 4, 4, 1.0, a, 4, a, 4, 0.0, a, 4, stream=0)
    with pytest.raises(TypeError):
        t = torch.zeros(4, 4, dtype=torch.float16)
        g.gemm_sgemm_f32_host("N", "N", 4, 4, 4, 1.0, t, 4, t, 4, 0.0, t, 4, stream=0)
    with pytest.raises(TypeError):
        g.gemm_sgemm_f32_host("N", "N", 4, 4, 4, 1.0, [1.0], 4, [1.0], 4, 0.0, [1.0], 4, stream=0)


def test_fma_peak_probe_rejects_a_null_output_without_a_device(lib):
    assert lib.gemm_measure_fp32_fma_peak(None, ctypes.POINTER(ctypes.c_double)()) == 1


def test_config_table_follows_the_pages_footprint_arithmetic(lib):
    # The pages' worked example (ssxxe.cn GEMM page, section 2.1): a 128 x 128 block tile with
    # BK = 8 holds BK * (BM + BN) * 4 = 8192 bytes of fp32 tiles and does 32 flop per byte
    # loaded.  The library's configurations account their shared memory the same way per
    # ring stage (plus one 16-byte chunk of padding per padded [k][x] row), fit the CTAs per
    # SM they are compiled for, and the 128 x 128 one has the example's intensity.
    d = golden_io.read("smem_footprint.txt")
    BM, BN, BK = (golden_io.scalar(d, k) for k in ("BM", "BN", "BK"))
    assert BK * (BM + BN) * 4 == golden_io.scalar(d, "smem_bytes")
    assert 2 * BM * BN * BK / ((BM + BN) * BK * 4) == golden_io.scalar(d, "flop_per_byte")
    configs = g.gemm_sgemm_configs()
    assert [c["name"] for c in configs] == ["L", "M", "S"]
    for c in configs:
        assert c["smem_bytes"] == c["stages"] * c["bk"] * (c["bm"] + c["bn"] + 2 * c["row_pad"]) * 4
        assert c["threads"] == (c["bm"] // c["tm"]) * (c["bn"] // c["tn"])
        assert c["row_pad"] in (0, 4)
        assert c["ctas_per_sm"] * (c["smem_bytes"] + 1024) <= 228 * 1024  # 228 KB per SM
    L = [c for c in configs if (c["bm"], c["bn"]) == (BM, BN)][0]
    assert 2 * L["bm"] * L["bn"] * L["bk"] / ((L["bm"] + L["bn"]) * L["bk"] * 4) == \
        golden_io.scalar(d, "flop_per_byte")
    c = g.load().gemm_sgemm_config(len(configs), ctypes.byref(_lib.SgemmConfig()))
    assert c == 1  # past the last configuration
