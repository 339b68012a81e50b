"""Parity of the product kernels (block-diagonal multiply, block weight gradient, frozen-
weight contraction) with the fp64 oracle, on the tensor-core engine and on the CUDA-core
engine, at sizes that span several tiles with a ragged token tail."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import DEV, P, TOL_BF16_STEP, TOL_F32, dev, engine, host  # noqa: F401

pytestmark = pytest.mark.gpu
RNG = np.random.default_rng(99)


def _bf(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16)


def _rand_bf16(shape, std=1.0):
    return _bf(RNG.standard_normal(shape) * std)


@pytest.mark.parametrize("N,nblk,b", [(300, 4, 64), (129, 3, 128), (517, 2, 256), (200, 2, 512),
                                      (64, 1, 256), (1, 2, 64)])
@pytest.mark.parametrize("trans", [False, True])
def test_blockdiag_bf16(P, engine, N, nblk, b, trans):
    X = _rand_bf16((N, nblk * b)).to(DEV)
    G = _rand_bf16((nblk, b, b), 1 / np.sqrt(b)).to(DEV)
    Y = torch.empty_like(X)
    P.poetx_blockdiag_mm(X, G, Y, trans=trans)
    ref = O.blockdiag_mm(host(X), host(G), transpose=trans)
    assert O.rel_fro(host(Y), ref) <= TOL_BF16_STEP


def test_blockdiag_bf16_colscale(P, engine):
    N, nblk, b = 260, 2, 128
    X = _rand_bf16((N, nblk * b)).to(DEV)
    G = _rand_bf16((nblk, b, b), 1 / np.sqrt(b)).to(DEV)
    s = torch.rand(nblk * b, device=DEV) + 0.5
    Y = torch.empty_like(X)
    P.poetx_blockdiag_mm(X, G, Y, trans=True, col_scale=s)
    ref = O.blockdiag_mm(host(X), host(G), transpose=True) * host(s)[None, :]
    assert O.rel_fro(host(Y), ref) <= TOL_BF16_STEP


@pytest.mark.parametrize("N,nblk,b", [(300, 4, 64), (517, 2, 256), (200, 2, 512)])
@pytest.mark.parametrize("trans", [False, True])
def test_blockdiag_bf16_out_perm(P, engine, N, nblk, b, trans):
    """Product stored through a column permutation: bit-identical to the product followed
    by the standalone scatter."""
    X = _rand_bf16((N, nblk * b)).to(DEV)
    G = _rand_bf16((nblk, b, b), 1 / np.sqrt(b)).to(DEV)
    perm = torch.tensor(RNG.permutation(nblk * b), dtype=torch.int32, device=DEV)
    Y = torch.empty_like(X)
    P.poetx_blockdiag_mm(X, G, Y, trans=trans, out_perm=perm)
    Z = torch.empty_like(X)
    P.poetx_blockdiag_mm(X, G, Z, trans=trans)
    ref = torch.empty_like(X)
    P.poetx_perm_scatter(Z, perm, ref)
    np.testing.assert_array_equal(host(Y), host(ref))
    assert O.rel_fro(host(Y), O.perm_scatter(O.blockdiag_mm(host(X), host(G), trans),
                                             host(perm))) <= TOL_BF16_STEP


@pytest.mark.parametrize("N,nblk,b,splits", [(300, 4, 64, 3), (1000, 2, 128, 4),
                                             (517, 2, 256, 2), (256, 1, 512, 1),
                                             (100, 2, 256, 4), (0, 2, 64, 2)])
def test_wgrad_bf16(P, engine, N, nblk, b, splits):
    X = _rand_bf16((N, nblk * b)).to(DEV)
    dY = _rand_bf16((N, nblk * b)).to(DEV)
    dG = torch.full((splits, nblk, b, b), float("nan"), device=DEV)
    P.poetx_blockdiag_wgrad(X, dY, b, dG)
    chunk = 64 * -(-N // (64 * splits)) if N else 64
    Xh, dYh = host(X), host(dY)
    for s in range(splits):
        sl = slice(s * chunk, min(N, (s + 1) * chunk))
        ref = O.blockdiag_wgrad(Xh[sl], dYh[sl], b)
        got = host(dG[s])
        if sl.start >= N:
            np.testing.assert_array_equal(got, 0.0)
        else:
            # fp32 output: only the fp32 accumulation order differs from the fp64 sum
            assert O.rel_fro(got, ref) <= 1e-5


@pytest.mark.parametrize("N,m,n", [(300, 512, 768), (129, 256, 256), (1, 512, 256),
                                   (640, 1024, 512), (4100, 2048, 1024),
                                   # enough 256 x 256 tiles for the 2-CTA pair kernel, in
                                   # one direction each, odd count of 128-row tiles
                                   (2600, 1024, 8192), (2600, 8192, 1024)])
@pytest.mark.parametrize("trans", [False, True])
def test_wprime_bf16(P, engine, N, m, n, trans):
    W = _rand_bf16((n, m), 1 / np.sqrt(m)).to(DEV)
    A = _rand_bf16((N, n if trans else m)).to(DEV)
    C = torch.empty(N, m if trans else n, dtype=torch.bfloat16, device=DEV)
    P.poetx_wprime_gemm(A, W, C, trans=trans)
    ref = host(A) @ (host(W) if trans else host(W).T)
    assert O.rel_fro(host(C), ref) <= TOL_BF16_STEP


@pytest.mark.parametrize("trans", [False, True])
@pytest.mark.parametrize("N,m,n", [(300, 512, 768),
                                   # several tiles per SM, a ragged last token tile
                                   (2600, 4096, 2816)])
def test_wprime_int8(P, engine, trans, N, m, n):
    Wq = torch.randint(-127, 128, (n, m), dtype=torch.int8, device=DEV)
    s = (torch.rand(n, device=DEV) + 0.5) / 127
    A = _rand_bf16((N, n if trans else m)).to(DEV)
    C = torch.empty(N, m if trans else n, dtype=torch.bfloat16, device=DEV)
    P.poetx_wprime_gemm(A, Wq, C, trans=trans, w_scale=s)
    Wd = host(Wq).astype(np.float64)
    if trans:  # A already carries the row scale
        ref = host(A) @ Wd
    else:
        ref = (host(A) @ Wd.T) * host(s)[None, :]
    assert O.rel_fro(host(C), ref) <= TOL_BF16_STEP


def test_products_f32(P):
    N, nblk, b = 70, 3, 32
    X = torch.randn(N, nblk * b, device=DEV)
    G = torch.randn(nblk, b, b, device=DEV)
    for trans in (False, True):
        Y = torch.empty_like(X)
        P.poetx_blockdiag_mm(X, G, Y, trans=trans)
        assert O.rel_fro(host(Y), O.blockdiag_mm(host(X), host(G), trans)) <= TOL_F32
    dG = torch.empty(2, nblk, b, b, device=DEV)
    dY = torch.randn_like(X)
    P.poetx_blockdiag_wgrad(X, dY, b, dG)
    assert O.rel_fro(host(dG.sum(0)), O.blockdiag_wgrad(host(X), host(dY), b)) <= TOL_F32
    W = torch.randn(48, 96, device=DEV)
    A = torch.randn(N, 96, device=DEV)
    C = torch.empty(N, 48, device=DEV)
    P.poetx_wprime_gemm(A, W, C)
    assert O.rel_fro(host(C), host(A) @ host(W).T) <= TOL_F32
    A2 = torch.randn(N, 48, device=DEV)
    C2 = torch.empty(N, 96, device=DEV)
    P.poetx_wprime_gemm(A2, W, C2, trans=True)
    assert O.rel_fro(host(C2), host(A2) @ host(W)) <= TOL_F32


def test_engines_agree_bitwise_on_exact_inputs(P):
    """Small-integer inputs make every fp32 partial sum exact, so both engines must give
    identical bits (any layout or descriptor slip shows up as a mismatch)."""
    N, m, n = 256, 512, 256
    A = torch.randint(-3, 4, (N, m), device=DEV).to(torch.bfloat16)
    W = torch.randint(-3, 4, (n, m), device=DEV).to(torch.bfloat16)
    outs = []
    for e in (0, 1):
        P.poetx_set_gemm_engine(e)
        C = torch.empty(N, n, dtype=torch.bfloat16, device=DEV)
        P.poetx_wprime_gemm(A, W, C)
        outs.append(host(C))
    P.poetx_set_gemm_engine(0)
    ref = host(A) @ host(W).T
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[1], host(torch.tensor(ref).to(torch.bfloat16)))
