"""The library's measured FP32 multiply-add ceiling (the strict-FP32 roofline denominator)."""
import ctypes

import pytest
import torch

import dense_gemm_sgemm_gb300 as lib

pytestmark = pytest.mark.gpu


def test_fma_peak_probe_is_within_the_unit_count_bound():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    derived = sms * 128 * 2 * 2.07e9 / 1e12  # FP32 lanes x 2 flop x the maximum SM clock
    before = lib.gemm_kernel_launches()
    tf = lib.gemm_measure_fp32_fma_peak()
    assert lib.gemm_kernel_launches() - before == 4  # one untimed, three timed
    assert lib.gemm_get_device_status() == 0
    # A chain kernel cannot beat the lanes at the maximum clock; well below half of it means
    # the probe does not measure the FMA pipe.
    assert 0.5 * derived < tf <= 1.03 * derived, (tf, derived)


def test_fma_peak_probe_rejects_a_null_output():
    st = lib.load().gemm_measure_fp32_fma_peak(None, ctypes.POINTER(ctypes.c_double)())
    assert st == 1  # GEMM_ERR_INVALID_VALUE
