"""The workspace-free CNP forward (poetx_cnp_fwd_noalloc), for callers that cannot allocate
device memory (a plugin inside a host application that owns all device allocations, or a
path where a device-synchronizing cudaMalloc is not acceptable).  It must give what the
ordinary entry point gives, call after call, although every call reuses the same fixed
scratch inside the library.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import DEV, P, TOL_F32, dev, host  # noqa: F401
from orthogonal_reparameterized_gb300 import inputs

pytestmark = pytest.mark.gpu


def _outs(nblk, b):
    return (torch.empty(nblk, b, b, device=DEV),
            torch.empty(nblk, b, b, dtype=torch.bfloat16, device=DEV),
            torch.empty(nblk, b, b, dtype=torch.bfloat16, device=DEV))


@pytest.mark.parametrize("nblk,b", [(16, 256), (3, 100), (8, 512)])
def test_noalloc_matches_cnp_fwd_on_two_calls(P, nblk, b):
    lib = P.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):  # the second call finds the first call's data in the scratch
        q = dev(inputs.cnp_inputs(900 + call, nblk, b, 0.02 * (call + 1)), torch.float32)
        G, Gb, Gt = _outs(nblk, b)
        st = lib.poetx_cnp_fwd_noalloc(ctypes.c_void_p(q.data_ptr()), nblk, b, 3,
                                       ctypes.c_void_p(G.data_ptr()), ctypes.c_void_p(Gb.data_ptr()),
                                       ctypes.c_void_p(Gt.data_ptr()), stream)
        assert st == 0, P.status_str(st)
        R, Rb, Rt = _outs(nblk, b)
        P.poetx_cnp_fwd(q, b, R, Rb, Rt)
        torch.cuda.synchronize()
        assert O.rel_fro(host(G), host(R), per_block=True) <= TOL_F32
        assert O.rel_fro(host(Gb), host(Rb), per_block=True) <= TOL_F32
        assert O.rel_fro(host(Gt), host(Rt), per_block=True) <= TOL_F32
        assert O.rel_fro(host(G), O.cnp_forward(host(q), b), per_block=True) <= TOL_F32
    assert P.poetx_get_device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(P):
    lib = P.lib()
    b = 512
    nblk = P.CNP_NOALLOC_MAX_ELEMS // (b * b) + 1
    q = torch.zeros(1, device=DEV)
    st = lib.poetx_cnp_fwd_noalloc(ctypes.c_void_p(q.data_ptr()), nblk, b, 3,
                                   ctypes.c_void_p(q.data_ptr()), None, None, None)
    assert st == 5  # POETX_ERR_WORKSPACE, nothing launched
    assert lib.poetx_cnp_fwd_noalloc(ctypes.c_void_p(q.data_ptr()), 4, 64, 2,
                                     ctypes.c_void_p(q.data_ptr()), None, None, None) == 6
