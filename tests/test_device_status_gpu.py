"""Failure detection without a GPU fault: the tensor-core kernel bounds every barrier wait.

GEMM_GB300_TEST_INJECT_STALL=1 makes the producer announce the first K slice without ever
loading it, so the MMA warp's wait on that slice can never succeed.  With the hook the
library also shortens the wait limit to 20 ms.  The kernel must give up, record
GEMM_ERR_DEVICE_TIMEOUT, stop its other warps, free its tensor memory and return; the host
reads the status and the context stays usable for the next call.

GEMM_GB300_TEST_INJECT_STALL=2 does the same to the first K half of every split tile of the
last wave, so the CTAs running the second halves wait for a partner that never arrives:
that cross-CTA wait must expire too, and the arrival counters it leaves raised must be
cleared when the status is read (the next split-K call would otherwise go wrong).
"""
import pytest
import torch

from dense_gemm_sgemm_gb300 import gemm_get_device_status, gemm_hgemm_f16f32

pytestmark = pytest.mark.gpu

TIMEOUT = 5  # GEMM_ERR_DEVICE_TIMEOUT


@pytest.mark.parametrize("M", [128, 256])  # one CTA per tile, and a two-CTA cluster
def test_expired_wait_is_reported_and_context_survives(monkeypatch, M):
    N, K = 256, 256
    A = torch.randint(-2, 3, (M, K), device="cuda").half()
    B = torch.randint(-2, 3, (K, N), device="cuda").half()
    C = torch.zeros(M, N, device="cuda")
    assert gemm_get_device_status() == 0
    monkeypatch.setenv("GEMM_GB300_TEST_INJECT_STALL", "1")
    gemm_hgemm_f16f32("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N)
    assert gemm_get_device_status() == TIMEOUT
    assert gemm_get_device_status() == 0  # reading clears the word
    monkeypatch.delenv("GEMM_GB300_TEST_INJECT_STALL")
    gemm_hgemm_f16f32("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N)
    torch.cuda.synchronize()
    assert gemm_get_device_status() == 0
    assert torch.equal(C, A.float() @ B.float())


def test_expired_wait_for_the_other_k_half_is_reported_and_counters_reset(monkeypatch):
    # 18 x 10 tiles of 128 x 256 (90 two-CTA pairs): 76 pairs whole, 14 in K halves
    M, N, K = 2304, 2560, 512
    g = torch.Generator(device="cuda").manual_seed(5)
    A = torch.randint(-2, 3, (M, K), device="cuda", generator=g).half()
    B = torch.randint(-2, 3, (K, N), device="cuda", generator=g).half()
    C = torch.zeros(M, N, device="cuda")
    ref = A.float() @ B.float()
    assert gemm_get_device_status() == 0
    monkeypatch.setenv("GEMM_GB300_TEST_INJECT_STALL", "2")
    gemm_hgemm_f16f32("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N)
    assert gemm_get_device_status() == TIMEOUT
    monkeypatch.delenv("GEMM_GB300_TEST_INJECT_STALL")
    for _ in range(2):  # the split tiles' counters start from zero again
        C.zero_()
        gemm_hgemm_f16f32("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N)
        torch.cuda.synchronize()
        assert gemm_get_device_status() == 0
        assert torch.equal(C, ref)
