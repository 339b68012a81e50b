"""Failure detection without a GPU fault: a bounded wait that nothing satisfies expires,
the kernel records POETX_ERR_TIMEOUT and returns, and the context stays usable."""
import numpy as np
import pytest
import torch

from gpu_util import DEV, P, host  # noqa: F401

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives(P):
    assert P.poetx_get_device_error() == 0
    P.poetx_selftest_timeout(2000)  # 2 ms
    assert P.poetx_get_device_error() == 7  # POETX_ERR_TIMEOUT
    assert 40000 < P.poetx_timeout_site() < 50000  # the self-test's wait (file id 4)
    assert P.poetx_get_device_error() == 0  # cleared by the read
    X = torch.randn(8, 64, device=DEV).to(torch.bfloat16)
    Y = torch.empty_like(X)
    p = torch.arange(64, dtype=torch.int32, device=DEV).flip(0).contiguous()
    P.poetx_perm_gather(X, p, Y)
    np.testing.assert_array_equal(host(Y), host(X)[:, ::-1])


def test_host_errors_raise(P):
    X = torch.randn(8, 64, device=DEV).to(torch.bfloat16)
    G = torch.randn(2, 100, 100, device=DEV).to(torch.bfloat16)
    with pytest.raises(P.PoetxError) as e:
        P.poetx_blockdiag_mm(X, G, torch.empty_like(X))
    assert e.value.status == 2
