"""Parity of the fp32 Cayley-Neumann kernels with the fp64 oracle: max over blocks of the
relative Frobenius error <= 1e-5, plus exact special cases."""
import numpy as np
import pytest
import torch

import oracle as O
from conftest import read_golden, read_golden_kv  # noqa: F401
from gpu_util import DEV, P, TOL_F32, dev, engine, host  # noqa: F401
from orthogonal_reparameterized_gb300 import inputs

pytestmark = pytest.mark.gpu


def _fwd(P, q, b):
    nblk = q.shape[0]
    G = torch.empty(nblk, b, b, device=DEV)
    Gb = torch.empty(nblk, b, b, dtype=torch.bfloat16, device=DEV)
    Gt = torch.empty(nblk, b, b, dtype=torch.bfloat16, device=DEV)
    P.poetx_cnp_fwd(dev(q, torch.float32), b, G, Gb, Gt)
    return G, Gb, Gt


@pytest.mark.parametrize("nblk,b,std", [(5, 2, 0.3), (3, 3, 0.3), (4, 5, 0.2), (8, 32, 0.01),
                                        (6, 64, 0.02), (3, 100, 0.02), (4, 128, 0.02),
                                        (3, 256, 0.02), (2, 512, 0.02), (2, 256, 0.2)])
def test_cnp_fwd_parity(P, engine, nblk, b, std):
    q = inputs.cnp_inputs(11, nblk, b, std)
    G, Gb, Gt = _fwd(P, q, b)
    ref = O.cnp_forward(q, b)
    assert O.rel_fro(host(G), ref, per_block=True) <= TOL_F32
    # the bf16 copies are the round-to-nearest-even of the fp32 result, and Gt its transpose
    np.testing.assert_array_equal(host(Gb), host(G.to(torch.bfloat16)))
    np.testing.assert_array_equal(host(Gt), np.swapaxes(host(Gb), 1, 2))


def test_cnp_fwd_golden_b2(P):
    rows = read_golden("cnp_b2.txt")
    q = np.array([[r[0]] for r in rows])
    G, _, _ = _fwd(P, q, 2)
    for j, r in enumerate(rows):
        np.testing.assert_allclose(host(G)[j], [[r[1], r[2]], [r[3], r[4]]], rtol=2e-7, atol=1e-6)


def test_cnp_fwd_zero_is_identity(P, engine):
    for b in (2, 64, 256):
        G, _, _ = _fwd(P, np.zeros((3, b * (b - 1) // 2)), b)
        np.testing.assert_array_equal(host(G), np.broadcast_to(np.eye(b), (3, b, b)))


@pytest.mark.parametrize("nblk,b,splits,std", [(5, 2, 1, 0.3), (4, 5, 3, 0.2), (8, 32, 1, 0.01),
                                               (6, 64, 4, 0.02), (3, 100, 2, 0.02),
                                               (4, 128, 1, 0.02), (3, 256, 5, 0.02),
                                               (2, 512, 2, 0.02)])
def test_cnp_bwd_parity(P, engine, nblk, b, splits, std):
    q = inputs.cnp_inputs(12, nblk, b, std)
    dG = inputs.dG_inputs(13, splits, nblk, b)
    dq = torch.empty(nblk, b * (b - 1) // 2, device=DEV)
    P.poetx_cnp_bwd(dev(q, torch.float32), dev(dG, torch.float32), b, dq)
    ref = O.cnp_backward(q, dG, b)
    assert O.rel_fro(host(dq), ref, per_block=True) <= TOL_F32


def test_cnp_bwd_golden_b2_and_accumulate(P):
    rows = read_golden("cnp_b2_grad.txt")
    q = np.array([[r[0]] for r in rows])
    dG = np.array([[[r[1], r[2]], [r[3], r[4]]] for r in rows])
    dq = dev(np.ones((len(rows), 1)), torch.float32)
    P.poetx_cnp_bwd(dev(q, torch.float32), dev(dG, torch.float32), 2, dq, accumulate=True)
    np.testing.assert_allclose(host(dq)[:, 0], [1 + r[5] for r in rows], rtol=1e-6, atol=1e-6)


def test_cnp_bwd_zero_q(P):
    b = 64
    dG = inputs.dG_inputs(14, 1, 3, b)
    dq = torch.empty(3, b * (b - 1) // 2, device=DEV)
    P.poetx_cnp_bwd(dev(np.zeros((3, b * (b - 1) // 2)), torch.float32), dev(dG, torch.float32),
                    b, dq)
    iu = np.triu_indices(b, 1)
    ref = (2 * (dG[0][:, iu[0], iu[1]] - dG[0][:, iu[1], iu[0]])).astype(np.float32)
    np.testing.assert_array_equal(host(dq).astype(np.float32), ref)


@pytest.mark.parametrize("b", [64, 128, 256, 512])
def test_cnp_sweep_full_size(P, engine, b):
    """The 4096 x 4096 layer of the block-size sweep: 4096/b blocks on each side."""
    nblk = 2 * 4096 // b
    q = inputs.cnp_inputs(20260308, nblk, b, 0.02)
    G, _, _ = _fwd(P, q, b)
    assert O.rel_fro(host(G), O.cnp_forward(q, b), per_block=True) <= TOL_F32
    dG = inputs.dG_inputs(20260308, 1, nblk, b)
    dq = torch.empty(nblk, b * (b - 1) // 2, device=DEV)
    P.poetx_cnp_bwd(dev(q, torch.float32), dev(dG, torch.float32), b, dq)
    assert O.rel_fro(host(dq), O.cnp_backward(q, dG, b), per_block=True) <= TOL_F32


def test_cnp_deterministic(P, engine):
    b, nblk = 256, 4
    q = dev(inputs.cnp_inputs(15, nblk, b, 0.02), torch.float32)
    dG = dev(inputs.dG_inputs(15, 3, nblk, b), torch.float32)
    outs = []
    for _ in range(2):
        dq = torch.empty(nblk, b * (b - 1) // 2, device=DEV)
        P.poetx_cnp_bwd(q, dG, b, dq)
        outs.append(host(dq))
    np.testing.assert_array_equal(outs[0], outs[1])
