"""Helpers shared by the GPU parity tests (device transfer, library fixture, tolerances)."""
import numpy as np
import pytest
import torch

DEV = "cuda:0"

# Tolerances (relative Frobenius error, max over blocks where the output is blocked):
#   fp32 CNP and the fp32 layer: 1e-5; bf16 layer outputs and gradients: 2e-2.
#   A single bf16 product (one GEMM whose output is rounded to bf16 once): its error is the
#   output rounding, at most 2^-9 relative per element (RMS about 1.1e-3), so 1e-2 is used.
TOL_F32 = 1e-5
TOL_BF16_LAYER = 2e-2
TOL_BF16_STEP = 1e-2


def dev(a, dtype):
    return torch.tensor(np.asarray(a), dtype=dtype, device=DEV)


def host(t):
    if t.dtype in (torch.int8, torch.int32, torch.int64, torch.uint8):
        return t.cpu().numpy()
    return t.float().cpu().numpy().astype(np.float64)


@pytest.fixture(scope="session")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from orthogonal_reparameterized_gb300 import build
    build.build()
    import orthogonal_reparameterized_gb300.poetx as P
    P.lib()
    torch.cuda.set_device(0)
    return P


@pytest.fixture(params=[0, 1], ids=["tcgen05", "cudacore"])
def engine(request, P):
    """Runs a test once with the tensor-core kernels and once with the CUDA-core ones."""
    P.poetx_set_gemm_engine(request.param)
    yield request.param
    P.poetx_set_gemm_engine(0)
