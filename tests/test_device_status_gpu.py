"""Failure detection without a GPU fault: the tensor-core kernel bounds every barrier wait.

GEMM_GB300_TEST_INJECT_STALL=1 makes the producer announce the first K slice without ever
loading it, so the MMA warp's wait on that slice can never succeed.  With the hook the
library also shortens the wait limit to 20 ms.  The kernel must give up, record
GEMM_ERR_DEVICE_TIMEOUT, stop its other warps, free its tensor memory and return; the host
reads the status and the context stays usable for the next call.
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
