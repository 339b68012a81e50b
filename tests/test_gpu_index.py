"""Bit-exact parity of the index / data-movement kernels with the oracle: packed triangle
unpack and gradient pack, permutation gather/scatter, the merge into W', the quantiser."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import DEV, P, dev, host  # noqa: F401

pytestmark = pytest.mark.gpu
RNG = np.random.default_rng(2024)


@pytest.mark.parametrize("nblk,b", [(3, 2), (2, 5), (4, 32), (3, 100), (2, 256), (1, 512)])
def test_triu_unpack_bit_exact(P, nblk, b):
    q = RNG.standard_normal((nblk, b * (b - 1) // 2)).astype(np.float32)
    Q = torch.empty(nblk, b, b, device=DEV)
    P.poetx_triu_unpack(dev(q, torch.float32), b, Q)
    np.testing.assert_array_equal(host(Q), O.triu_unpack(q.astype(np.float64), b))


@pytest.mark.parametrize("nblk,b", [(3, 2), (2, 7), (4, 64), (2, 300)])
@pytest.mark.parametrize("acc", [False, True])
def test_triu_grad_pack_bit_exact(P, nblk, b, acc):
    X = RNG.standard_normal((nblk, b, b)).astype(np.float32)
    d0 = RNG.standard_normal((nblk, b * (b - 1) // 2)).astype(np.float32)
    dq = dev(d0, torch.float32)
    P.poetx_triu_grad_pack(dev(X, torch.float32), dq, accumulate=acc)
    # fp32 subtraction (and addition) are correctly rounded on both sides
    ref = O.triu_grad_pack(X.astype(np.float64)).astype(np.float32)
    if acc:
        ref = (d0 + ref).astype(np.float32)
    np.testing.assert_array_equal(host(dq).astype(np.float32), ref)


def _perms(D):
    return {"random": RNG.permutation(D), "identity": np.arange(D),
            "reversal": np.arange(D)[::-1].copy(),
            "swap": np.r_[1, 0, np.arange(2, D)]}


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.int8])
# shapes reach every ring layout of the kernel: one-warp groups with deep rings that wrap many
# times (20000 x 256), two-warp groups (4096 wide), whole-CTA groups (14336), and rows so
# long that one CTA fills an SM (32768)
@pytest.mark.parametrize("N,D", [(1, 64), (37, 256), (300, 2048), (20000, 256), (64, 4096),
                                 (5, 14336), (3, 32768)])
def test_perm_gather_scatter_bit_exact(P, dtype, N, D):
    if dtype == torch.int8:
        X = torch.randint(-128, 127, (N, D), dtype=torch.int8, device=DEV)
    else:
        X = torch.randn(N, D, device=DEV).to(dtype)
    for name, p in _perms(D).items():
        pt = dev(p, torch.int32)
        Y = torch.empty_like(X)
        P.poetx_perm_gather(X, pt, Y)
        ref = O.perm_gather(host(X), p)
        np.testing.assert_array_equal(host(Y), ref, err_msg=name)
        Z = torch.empty_like(X)
        P.poetx_perm_scatter(Y, pt, Z)
        np.testing.assert_array_equal(host(Z), O.perm_scatter(ref, p), err_msg=name)
        np.testing.assert_array_equal(host(Z), host(X), err_msg=name)


def _rand_rows(dtype, N, D):
    if dtype == torch.int8:
        return torch.randint(-128, 127, (N, D), dtype=torch.int8, device=DEV)
    return torch.randn(N, D, device=DEV).to(dtype)


# the widest rows each element type takes: the staged 2-byte index and one row fill the
# shared memory of an SM; one 16-byte vector wider is refused on the host, before any launch
@pytest.mark.parametrize("dtype,D", [(torch.float32, 37528), (torch.bfloat16, 56304),
                                     (torch.int8, 65520)])
def test_perm_widest_rows(P, dtype, D):
    X = _rand_rows(dtype, 3, D)
    p = RNG.permutation(D)
    pt = dev(p, torch.int32)
    Y = torch.empty_like(X)
    P.poetx_perm_gather(X, pt, Y)
    np.testing.assert_array_equal(host(Y), O.perm_gather(host(X), p))
    Z = torch.empty_like(X)
    P.poetx_perm_scatter(Y, pt, Z)
    np.testing.assert_array_equal(host(Z), host(X))
    wide = D + 16 // X.element_size()
    Xw = _rand_rows(dtype, 3, wide)
    with pytest.raises(Exception):
        P.poetx_perm_gather(Xw, dev(np.arange(wide), torch.int32), torch.empty_like(Xw))


def test_perm_index_not_16_byte_aligned(P):
    """An index starting 4 bytes past a 16-byte boundary is staged one element at a time."""
    N, D = 64, 4096
    p = RNG.permutation(D)
    buf = dev(np.r_[0, p], torch.int32)
    pt = buf[1:]
    assert pt.data_ptr() % 16 == 4
    X = _rand_rows(torch.bfloat16, N, D)
    Y = torch.empty_like(X)
    P.poetx_perm_gather(X, pt, Y)
    np.testing.assert_array_equal(host(Y), O.perm_gather(host(X), p))
    Z = torch.empty_like(X)
    P.poetx_perm_scatter(X, pt, Z)
    np.testing.assert_array_equal(host(Z), O.perm_scatter(host(X), p))


def test_perm_empty(P):
    X = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    P.poetx_perm_gather(X, dev(np.arange(64), torch.int32), torch.empty_like(X))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.int8])
@pytest.mark.parametrize("n,m", [(64, 128), (512, 2048), (13824, 5120)])
def test_merge_perm_bit_exact(P, dtype, n, m):
    pn, pm = RNG.permutation(n), RNG.permutation(m)
    if dtype == torch.int8:
        W = torch.randint(-127, 128, (n, m), dtype=torch.int8, device=DEV)
        s = torch.rand(n, device=DEV)
        sp = torch.empty_like(s)
    else:
        W = torch.randn(n, m, device=DEV).to(dtype)
        s = sp = None
    Wp = torch.empty_like(W)
    P.poetx_merge_perm(W, dev(pn, torch.int32), dev(pm, torch.int32), Wp, s, sp)
    np.testing.assert_array_equal(host(Wp), O.merge_perm(host(W), pn, pm))
    if s is not None:
        np.testing.assert_array_equal(host(sp), host(s)[pn])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.int8])
@pytest.mark.parametrize("n,m,n_pad,m_pad", [(200, 144, 256, 192), (72, 2048, 128, 2048),
                                             (512, 48, 512, 64)])
def test_merge_perm_padded_bit_exact(P, dtype, n, m, n_pad, m_pad):
    """The merge into a zero-padded weight (ragged last blocks): the [n, m] corner is the
    plain merge, every padding row, column and scale is 0 (the buffers start as garbage)."""
    pn, pm = RNG.permutation(n), RNG.permutation(m)
    if dtype == torch.int8:
        W = torch.randint(-127, 128, (n, m), dtype=torch.int8, device=DEV)
        s = torch.rand(n, device=DEV)
        sp = torch.full((n_pad,), float("nan"), device=DEV)
        Wp = torch.full((n_pad, m_pad), 5, dtype=torch.int8, device=DEV)
    else:
        W = torch.randn(n, m, device=DEV).to(dtype)
        s = sp = None
        Wp = torch.full((n_pad, m_pad), float("nan"), device=DEV).to(dtype)
    P.poetx_merge_perm_padded(W, dev(pn, torch.int32), dev(pm, torch.int32), Wp, s, sp)
    ref = np.zeros((n_pad, m_pad))
    ref[:n, :m] = O.merge_perm(host(W), pn, pm)
    np.testing.assert_array_equal(host(Wp), ref)
    if s is not None:
        np.testing.assert_array_equal(host(sp)[:n], host(s)[pn])
        assert np.all(host(sp)[n:] == 0)


@pytest.mark.parametrize("n,m", [(7, 33), (64, 4096), (13824, 5120)])
def test_quantize_bit_exact(P, n, m):
    W = (RNG.standard_normal((n, m)) / np.sqrt(m)).astype(np.float32)
    W[n // 2] = 0.0
    Wq = torch.empty(n, m, dtype=torch.int8, device=DEV)
    s = torch.empty(n, device=DEV)
    P.poetx_quantize_rows_int8(dev(W, torch.float32), Wq, s)
    rq, rs = O.quantize_rows_int8(W)
    np.testing.assert_array_equal(host(Wq), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
