"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test checks one oracle function against a closed form, a hand-worked example from
``tests/golden`` (with its source), a library special case, finite differences or an
invariant the pages state.  A plausible slip anywhere in the oracle (dropped term, sign,
transposed operand, wrong index order, wrong permutation direction) fails at least one.
"""
import numpy as np
import pytest

import oracle as O
from conftest import read_golden, read_golden_kv

RNG = np.random.default_rng(12345)


def _rand_q(nblk, b, std=0.3):
    return RNG.standard_normal((nblk, b * (b - 1) // 2)) * std


# ------------------------------------------------------------------ triu storage (S1)
@pytest.mark.parametrize("b", [2, 3, 5, 8])
def test_triu_unpack_bruteforce(b):
    q = _rand_q(3, b)
    Q = O.triu_unpack(q, b)
    for blk in range(3):
        k = 0
        for i in range(b):
            assert Q[blk, i, i] == 0.0
            for j in range(i + 1, b):
                assert Q[blk, i, j] == q[blk, k]
                assert Q[blk, j, i] == -q[blk, k]
                k += 1


def test_triu_order_is_numpy_triu_indices():
    b = 7
    q = np.arange(1, b * (b - 1) // 2 + 1, dtype=float)[None]
    Q = O.triu_unpack(q, b)[0]
    iu = np.triu_indices(b, 1)
    np.testing.assert_array_equal(Q[iu], q[0])


@pytest.mark.parametrize("b", [2, 4, 9])
def test_triu_grad_pack_is_adjoint_of_unpack(b):
    q = _rand_q(2, b)
    X = RNG.standard_normal((2, b, b))
    lhs = np.sum(O.triu_unpack(q, b) * X)
    rhs = np.sum(q * O.triu_grad_pack(X))
    assert abs(lhs - rhs) < 1e-12 * max(1.0, abs(lhs))


# ------------------------------------------------------------------ CNP forward (S2)
def test_cnp_zero_is_identity():
    for b in (2, 5, 32):
        G = O.cnp_forward(np.zeros((3, b * (b - 1) // 2)), b)
        np.testing.assert_array_equal(G, np.broadcast_to(np.eye(b), G.shape))


def test_cnp_golden_b2():
    for q, g00, g01, g10, g11 in read_golden("cnp_b2.txt"):
        G = O.cnp_forward(np.array([[q]]), 2)[0]
        np.testing.assert_allclose(G, [[g00, g01], [g10, g11]], rtol=0, atol=1e-15)


def test_cnp_golden_b4_direct_sum():
    # q01 = 0.5, q23 = 0.25, all other pairs 0 -> G = diag(G(0.5), G(0.25)) (cnp_b2.txt)
    q = np.zeros((1, 6))
    q[0, 0] = 0.5   # pair (0,1)
    q[0, 5] = 0.25  # pair (2,3)
    G = O.cnp_forward(q, 4)[0]
    ref = np.zeros((4, 4))
    ref[:2, :2] = [[0.5625, 0.75], [-0.75, 0.5625]]
    ref[2:, 2:] = [[0.87890625, 0.46875], [-0.46875, 0.87890625]]
    np.testing.assert_allclose(G, ref, rtol=0, atol=1e-15)


@pytest.mark.parametrize("b", [3, 8, 33])
def test_cnp_equals_eq9_expansion_and_factorisation(b):
    """eq. 9's expanded polynomial and the factorisation (I+Q)^2 (I+Q^2) agree with the
    product definition (I+Q)(I+Q+Q^2+Q^3)."""
    q = _rand_q(4, b, 0.1)
    G = O.cnp_forward(q, b)
    Q = O.triu_unpack(q, b)
    I = np.eye(b)
    Q2 = Q @ Q
    eq9 = 2 * (Q + Q2 + Q2 @ Q) + Q2 @ Q2 + I
    fac = (I + Q) @ (I + Q) @ (I + Q2)
    np.testing.assert_allclose(G, eq9, rtol=0, atol=1e-13)
    np.testing.assert_allclose(G, fac, rtol=0, atol=1e-13)


@pytest.mark.parametrize("b", [4, 16, 64])
def test_cnp_orthogonality_defect_closed_form(b):
    """Powers of Q commute, so G^T G = (I+Q^2)^2 (I-Q)^2 (I+Q)^2 = (I - Q^4)^2 exactly."""
    q = _rand_q(3, b, 0.05)
    G = O.cnp_forward(q, b)
    Q = O.triu_unpack(q, b)
    Q4 = np.linalg.matrix_power(Q, 4)
    I = np.eye(b)
    ref = (I - Q4) @ (I - Q4)
    np.testing.assert_allclose(np.swapaxes(G, 1, 2) @ G, ref, rtol=0, atol=1e-13)


def test_cnp_defect_shrinks_with_q():
    """||G^T G - I|| = ||2Q^4 - Q^8|| -> halving Q shrinks the defect ~16x."""
    b = 32
    q = _rand_q(2, b, 0.02)
    d = []
    for s in (1.0, 0.5, 0.25):
        G = O.cnp_forward(q * s, b)
        d.append(np.linalg.norm(np.swapaxes(G, 1, 2) @ G - np.eye(b)))
    assert d[0] < 1e-2
    for a, c in zip(d, d[1:]):
        assert 14.0 < a / c < 17.0


@pytest.mark.parametrize("b", [4, 24])
def test_cnp_vs_exact_cayley(b):
    """G - (I+Q)(I-Q)^-1 = -(I+Q) Q^4 (I-Q)^-1 (truncation of the Neumann series after Q^3),
    with the exact Cayley transform computed by a library solve."""
    q = _rand_q(2, b, 0.1)
    G = O.cnp_forward(q, b)
    Q = O.triu_unpack(q, b)
    I = np.eye(b)
    for j in range(2):
        inv = np.linalg.solve((I - Q[j]).T, I).T  # (I - Q)^-1
        cay = (I + Q[j]) @ inv
        err = -(I + Q[j]) @ np.linalg.matrix_power(Q[j], 4) @ inv
        np.testing.assert_allclose(G[j] - cay, err, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ CNP backward (S14)
def test_cnp_backward_golden_b2():
    for q, a, bb, c, d, dq in read_golden("cnp_b2_grad.txt"):
        got = O.cnp_backward(np.array([[q]]), np.array([[[a, bb], [c, d]]]), 2)
        assert abs(got[0, 0] - dq) < 1e-13


def test_cnp_backward_zero_q():
    """At Q = 0, G = I + 2Q + O(Q^2): dL/dQ = 2 dG, so dq_ij = 2 (dG_ij - dG_ji)."""
    b = 6
    dG = RNG.standard_normal((2, b, b))
    dq = O.cnp_backward(np.zeros((2, b * (b - 1) // 2)), dG, b)
    iu = np.triu_indices(b, 1)
    ref = 2 * (dG[:, iu[0], iu[1]] - dG[:, iu[1], iu[0]])
    np.testing.assert_allclose(dq, ref, rtol=0, atol=1e-14)


@pytest.mark.parametrize("b,order", [(2, 3), (3, 3), (5, 3), (8, 3), (5, 1), (5, 2), (4, 5)])
def test_cnp_backward_finite_differences(b, order):
    q = _rand_q(2, b, 0.3)
    dG = RNG.standard_normal((2, b, b))
    dq = O.cnp_backward(q, dG, b, order)
    h = 1e-6
    fd = np.zeros_like(q)
    for blk in range(2):
        for k in range(q.shape[1]):
            qp, qm = q.copy(), q.copy()
            qp[blk, k] += h
            qm[blk, k] -= h
            fd[blk, k] = (np.sum(dG * O.cnp_forward(qp, b, order))
                          - np.sum(dG * O.cnp_forward(qm, b, order))) / (2 * h)
    np.testing.assert_allclose(dq, fd, rtol=1e-7, atol=1e-8)


def test_cnp_backward_sums_partials():
    b = 5
    q = _rand_q(3, b)
    parts = RNG.standard_normal((4, 3, b, b))
    np.testing.assert_allclose(O.cnp_backward(q, parts, b),
                               O.cnp_backward(q, parts.sum(0), b), rtol=0, atol=1e-12)


# ------------------------------------------------------------------ permutations (S3/S7/S15)
def test_perm_gather_scatter_bruteforce():
    X = RNG.standard_normal((3, 7))
    p = RNG.permutation(7).astype(np.int32)
    Xt = O.perm_gather(X, p)
    for t in range(3):
        for i in range(7):
            assert Xt[t, i] == X[t, p[i]]
    Y = O.perm_scatter(Xt, p)
    np.testing.assert_array_equal(Y, X)
    for t in range(3):
        for i in range(7):
            assert Y[t, p[i]] == Xt[t, i]


def test_merge_perm_equals_permutation_matrices():
    """W' = Phi_n^T W0 Phi_m with Phi = Psi^T and Psi the gather matrix (Psi v)_i = v_pi[i]."""
    n, m = 6, 9
    W0 = RNG.standard_normal((n, m))
    pn = RNG.permutation(n)
    pm = RNG.permutation(m)
    Psi_n = np.eye(n)[pn]
    Psi_m = np.eye(m)[pm]
    ref = Psi_n @ W0 @ Psi_m.T
    np.testing.assert_array_equal(O.merge_perm(W0, pn, pm), ref)
    np.testing.assert_array_equal(O.merge_perm(W0, np.arange(n), np.arange(m)), W0)


# ------------------------------------------------------------------ quantiser (S16)
def test_quantize_rows_int8_properties():
    W = (RNG.standard_normal((20, 33)) * 0.1).astype(np.float32)
    W[3] = 0.0
    Wq, s = O.quantize_rows_int8(W)
    assert Wq.dtype == np.int8 and s.dtype == np.float32
    assert s[3] == 1.0 and not Wq[3].any()
    for r in range(20):
        if r == 3:
            continue
        amax = np.max(np.abs(W[r]))
        assert s[r] == np.float32(amax) / np.float32(127)
        c = np.argmax(np.abs(W[r]))
        assert abs(int(Wq[r, c])) == 127
        # rounding bound of a correctly rounded quotient, then round-to-nearest
        err = np.abs(W[r].astype(np.float64) - Wq[r].astype(np.float64) * s[r])
        assert np.all(err <= 0.5 * s[r] * (1 + 1e-6) + 1e-12)
    assert np.abs(Wq.astype(int)).max() <= 127


def test_quantize_round_half_even_bruteforce():
    # w/s lands exactly on .5 ties: numpy rint rounds half to even
    W = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5]], dtype=np.float32)
    Wq, s = O.quantize_rows_int8(W)
    assert s[0] == 1.0
    np.testing.assert_array_equal(Wq[0], [127, 0, 2, 2, 0, -2])


# ------------------------------------------------------------------ the layer
def _layer(m, n, b, N, seed=0, qstd=0.2):
    r = np.random.default_rng(seed)
    return dict(
        x=r.standard_normal((N, m)), dy=r.standard_normal((N, n)),
        W0=r.standard_normal((n, m)) / np.sqrt(m),
        perm_m=r.permutation(m), perm_n=r.permutation(n),
        q_R=r.standard_normal((m // b, b * (b - 1) // 2)) * qstd,
        q_P=r.standard_normal((n // b, b * (b - 1) // 2)) * qstd)


def _blkdiag(G):
    nblk, b, _ = G.shape
    D = np.zeros((nblk * b, nblk * b))
    for j in range(nblk):
        D[j * b:(j + 1) * b, j * b:(j + 1) * b] = G[j]
    return D


def test_layer_golden_zero_q():
    g = read_golden_kv("layer_tiny.txt")
    x = np.array(g["zero_q.x"])
    W0 = np.array(g["zero_q.W0"])
    pm = np.array(g["zero_q.perm_m"][0], dtype=int)
    pn = np.array(g["zero_q.perm_n"][0], dtype=int)
    dy = np.array(g["zero_q.dy"])
    r = O.poetx_layer(x, dy, W0, pm, pn, np.zeros((2, 1)), np.zeros((2, 1)), 2)
    np.testing.assert_allclose(r["y"], g["zero_q.y"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(r["dx"], g["zero_q.dx"], rtol=0, atol=1e-14)


def test_layer_golden_rot():
    g = read_golden_kv("layer_tiny.txt")
    r = O.poetx_layer(np.array(g["rot.x"]), np.zeros((1, 2)), np.array(g["rot.W0"]),
                      np.array([0, 1]), np.array([0, 1]), np.array(g["rot.q_R"]),
                      np.array(g["rot.q_P"]), 2)
    np.testing.assert_allclose(r["y"], g["rot.y"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("m,n,b,N", [(8, 8, 4, 3), (12, 8, 4, 5), (16, 32, 8, 4)])
def test_layer_zero_q_is_plain_linear(m, n, b, N):
    L = _layer(m, n, b, N)
    L["q_R"][:] = 0
    L["q_P"][:] = 0
    r = O.poetx_layer(L["x"], L["dy"], L["W0"], L["perm_m"], L["perm_n"], L["q_R"],
                      L["q_P"], b)
    np.testing.assert_allclose(r["y"], L["x"] @ L["W0"].T, rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["dx"], L["dy"] @ L["W0"], rtol=0, atol=1e-13)


@pytest.mark.parametrize("m,n,b,N", [(8, 8, 4, 3), (12, 8, 4, 5), (16, 32, 8, 4)])
def test_layer_equals_weight_centric_form(m, n, b, N):
    """Input-centric chain == x W_eff^T with W_eff = R W0 P, R = Psi_n^T D_P^T Psi_n,
    P = Psi_m^T D_R^T Psi_m built from dense matrices (POET-X summary, "Background" and
    "Core method": R_i = Psi^T Diag(G~) Psi; POET skill page, Step 1: W = R W0 P)."""
    L = _layer(m, n, b, N)
    r = O.poetx_layer(L["x"], L["dy"], L["W0"], L["perm_m"], L["perm_n"], L["q_R"],
                      L["q_P"], b)
    Psi_m = np.eye(m)[L["perm_m"]]
    Psi_n = np.eye(n)[L["perm_n"]]
    R = Psi_n.T @ _blkdiag(r["G_P"]).T @ Psi_n
    P = Psi_m.T @ _blkdiag(r["G_R"]).T @ Psi_m
    W_eff = R @ L["W0"] @ P
    np.testing.assert_allclose(r["y"], L["x"] @ W_eff.T, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dx"], L["dy"] @ W_eff, rtol=0, atol=1e-12)


def test_merged_weight_equals_four_explicit_permutations():
    """POET-X summary, "Core method" §2: merging Phi_n^T W Phi_m gives the same output as
    applying all four permutations around the un-merged W0."""
    m, n, b, N = 12, 8, 4, 5
    L = _layer(m, n, b, N)
    G_R = O.cnp_forward(L["q_R"], b)
    G_P = O.cnp_forward(L["q_P"], b)
    pm, pn = L["perm_m"], L["perm_n"]
    # four permutations: gather -> blockdiag -> scatter -> W0 -> gather -> blockdiag -> scatter
    a = O.perm_scatter(O.blockdiag_mm(O.perm_gather(L["x"], pm), G_R), pm)
    bb = a @ L["W0"].T
    y4 = O.perm_scatter(O.blockdiag_mm(O.perm_gather(bb, pn), G_P), pn)
    y2 = O.layer_forward(L["x"], O.merge_perm(L["W0"], pn, pm), pm, pn, G_R, G_P)["y"]
    np.testing.assert_allclose(y2, y4, rtol=0, atol=1e-13)


def test_spectrum_preserved_with_orthogonal_blocks():
    """With exactly orthogonal blocks the singular values of W_eff equal those of W0
    (POET-X summary, "Background"; POET skill page, "Reference")."""
    m, n, b = 16, 12, 4
    L = _layer(m, n, b, 1)
    r = np.random.default_rng(7)
    G_R = np.stack([np.linalg.qr(r.standard_normal((b, b)))[0] for _ in range(m // b)])
    G_P = np.stack([np.linalg.qr(r.standard_normal((b, b)))[0] for _ in range(n // b)])
    Wp = O.merge_perm(L["W0"], L["perm_n"], L["perm_m"])
    # W_eff^T = response of the chain to the identity batch
    W_effT = O.layer_forward(np.eye(m), Wp, L["perm_m"], L["perm_n"], G_R, G_P)["y"]
    s1 = np.linalg.svd(W_effT, compute_uv=False)
    s0 = np.linalg.svd(L["W0"], compute_uv=False)
    np.testing.assert_allclose(s1, s0, rtol=0, atol=1e-13)


# ------------------------------------------------------------------ merge-then-reinitialize
def test_merge_reinit_zero_q_returns_w0():
    """With the factors at the identity the merge writes back exactly the frozen weight."""
    m, n, b = 12, 8, 4
    L = _layer(m, n, b, 1)
    Wp = O.merge_perm(L["W0"], L["perm_n"], L["perm_m"])
    W0n = O.merge_reinit(Wp, L["perm_m"], L["perm_n"], 0 * L["q_R"], 0 * L["q_P"], b)
    np.testing.assert_allclose(W0n, L["W0"], rtol=0, atol=1e-15)


def test_merge_reinit_closed_form_b2():
    """b = 2, identity permutations: Q = [[0, t], [-t, 0]] gives Q^2 = -t^2 I, so
    G = (I + Q)(I + Q + Q^2 + Q^3) = (1 - t^2) [[1 - t^2, 2t], [-2t, 1 - t^2]] (by hand), and
    the merged weight is G_P^T W0 G_R^T (POET skill page, Step 1 and Step 4)."""
    def G2(t):
        return (1 - t * t) * np.array([[1 - t * t, 2 * t], [-2 * t, 1 - t * t]])
    W0 = np.array([[0.5, -1.25], [2.0, 0.75]])
    tR, tP = 0.3, -0.2
    W0n = O.merge_reinit(W0, np.array([0, 1]), np.array([0, 1]), np.array([[tR]]),
                         np.array([[tP]]), 2)
    np.testing.assert_allclose(W0n, G2(tP).T @ W0 @ G2(tR).T, rtol=0, atol=1e-15)


@pytest.mark.parametrize("m,n,b", [(8, 8, 4), (12, 8, 4), (16, 32, 8)])
def test_merge_reinit_equals_dense_R_W0_P(m, n, b):
    """W0_new = R W0 P with R = Psi_n^T D_P^T Psi_n and P = Psi_m^T D_R^T Psi_m built as dense
    matrices (POET skill page, Step 1: W = R W0 P; Step 4 writes it back into W0)."""
    L = _layer(m, n, b, 1)
    Wp = O.merge_perm(L["W0"], L["perm_n"], L["perm_m"])
    W0n = O.merge_reinit(Wp, L["perm_m"], L["perm_n"], L["q_R"], L["q_P"], b)
    Psi_m = np.eye(m)[L["perm_m"]]
    Psi_n = np.eye(n)[L["perm_n"]]
    R = Psi_n.T @ _blkdiag(O.cnp_forward(L["q_P"], b)).T @ Psi_n
    P = Psi_m.T @ _blkdiag(O.cnp_forward(L["q_R"], b)).T @ Psi_m
    np.testing.assert_allclose(W0n, R @ L["W0"] @ P, rtol=0, atol=1e-13)


def test_merge_reinit_preserves_the_layer_with_new_permutations():
    """After the merge, q = 0 and freshly drawn permutations, the layer computes the same
    outputs and input gradients as before (the purpose of the step)."""
    m, n, b, N = 16, 24, 4, 7
    L = _layer(m, n, b, N, seed=3)
    Wp = O.merge_perm(L["W0"], L["perm_n"], L["perm_m"])
    before = O.poetx_layer(L["x"], L["dy"], L["W0"], L["perm_m"], L["perm_n"], L["q_R"],
                           L["q_P"], b)
    W0n = O.merge_reinit(Wp, L["perm_m"], L["perm_n"], L["q_R"], L["q_P"], b)
    r = np.random.default_rng(9)
    pm2, pn2 = r.permutation(m), r.permutation(n)
    after = O.poetx_layer(L["x"], L["dy"], W0n, pm2, pn2, 0 * L["q_R"], 0 * L["q_P"], b)
    np.testing.assert_allclose(after["y"], before["y"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(after["dx"], before["dx"], rtol=0, atol=1e-12)


def test_merge_reinit_singular_values_within_cnp_bound():
    """G is a polynomial in the skew Q, so it is normal with singular values 1 - lambda^4
    for the eigenvalues +-i lambda of Q (|1 + i l| |1 + i l - l^2 - i l^3| = (1 + l^2)
    (1 - l^2)).  Hence sigma_k(W0_new) / sigma_k(W0) lies in [(1 - lR^4)(1 - lP^4), 1]
    with lR, lP the largest |eigenvalue| over the blocks of each side."""
    m, n, b = 16, 12, 4
    L = _layer(m, n, b, 1, seed=5, qstd=0.15)
    Wp = O.merge_perm(L["W0"], L["perm_n"], L["perm_m"])
    W0n = O.merge_reinit(Wp, L["perm_m"], L["perm_n"], L["q_R"], L["q_P"], b)
    lam = lambda q: max(np.abs(np.linalg.eigvals(Qj)).max() for Qj in O.triu_unpack(q, b))
    lo = (1 - lam(L["q_R"]) ** 4) * (1 - lam(L["q_P"]) ** 4)
    assert lo < 1 - 1e-6  # the bound is not trivial here
    ratio = np.linalg.svd(W0n, compute_uv=False) / np.linalg.svd(L["W0"], compute_uv=False)
    assert np.all(ratio <= 1 + 1e-12) and np.all(ratio >= lo - 1e-12), (ratio, lo)


# ------------------------------------------------------------------ optimizer on triu(q)
def test_adam_first_step_closed_form():
    """t = 1 from zero state: m_hat = g and v_hat = g^2 exactly, so the step is
    -lr g / (|g| + eps) (Kingma & Ba, Algorithm 1); |g| near eps separates eps outside the
    square root from eps inside it."""
    g = np.array([3.0, -2e-8, 1e-8, -0.5, 0.0])
    q = np.array([0.1, 0.2, -0.3, 0.4, 0.5])
    z = np.zeros_like(g)
    qn, m, v = O.adam_step(q, g, z, z, 1, lr=0.01, eps=1e-8)
    np.testing.assert_allclose(qn, q - 0.01 * g / (np.abs(g) + 1e-8), rtol=0, atol=1e-16)
    np.testing.assert_allclose(m, 0.1 * g, rtol=1e-15, atol=0)
    np.testing.assert_allclose(v, 0.001 * g * g, rtol=1e-12, atol=0)


def test_adam_constant_gradient_is_bias_free():
    """With a constant gradient the bias corrections make m_hat = g and v_hat = g^2 at every
    step, so T steps move q by exactly T lr g / (|g| + eps)."""
    g = np.array([0.7, -1.3, 2e-3])
    q = np.array([1.0, -1.0, 0.25])
    m = v = np.zeros_like(g)
    qt = q.copy()
    for t in range(1, 8):
        qt, m, v = O.adam_step(qt, g, m, v, t, lr=1e-3, beta1=0.8, beta2=0.95, eps=1e-6)
    np.testing.assert_allclose(qt, q - 7 * 1e-3 * g / (np.abs(g) + 1e-6), rtol=0, atol=1e-14)


def test_adam_weight_decay_alone_and_zero_gradient():
    q = np.array([0.5, -2.0])
    z = np.zeros_like(q)
    qn, m, v = O.adam_step(q, z, z, z, 3, lr=0.1, weight_decay=0.01)
    np.testing.assert_allclose(qn, q * (1 - 0.1 * 0.01), rtol=0, atol=1e-16)
    qn, _, _ = O.adam_step(q, z, z, z, 3, lr=0.1)
    np.testing.assert_array_equal(qn, q)


@pytest.mark.parametrize("m,n,b,N", [(8, 8, 4, 3), (12, 8, 4, 2)])
def test_layer_backward_finite_differences(m, n, b, N):
    L = _layer(m, n, b, N, seed=3, qstd=0.3)
    r = O.poetx_layer(L["x"], L["dy"], L["W0"], L["perm_m"], L["perm_n"], L["q_R"],
                      L["q_P"], b)

    def loss(x, qR, qP):
        G_R = O.cnp_forward(qR, b)
        G_P = O.cnp_forward(qP, b)
        Wp = O.merge_perm(L["W0"], L["perm_n"], L["perm_m"])
        y = O.layer_forward(x, Wp, L["perm_m"], L["perm_n"], G_R, G_P)["y"]
        return np.sum(L["dy"] * y)

    h = 1e-6
    for key, grad in (("q_R", r["dq_R"]), ("q_P", r["dq_P"]), ("x", r["dx"])):
        base = {"x": L["x"], "qR": L["q_R"], "qP": L["q_P"]}
        name = {"q_R": "qR", "q_P": "qP", "x": "x"}[key]
        arr = base[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, mm = arr.copy(), arr.copy()
            p[idx] += h
            mm[idx] -= h
            fd[idx] = (loss(**{**base, name: p}) - loss(**{**base, name: mm})) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8)


def test_token_shards_sum_to_full_batch_gradient():
    """dq and dG are sums over tokens: the sum over token shards equals the full batch
    (the data-parallel exchange of the POET-X summary, "Practice notes" §4)."""
    m, n, b, N = 16, 8, 4, 10
    L = _layer(m, n, b, N)
    full = O.poetx_layer(L["x"], L["dy"], L["W0"], L["perm_m"], L["perm_n"], L["q_R"],
                         L["q_P"], b)
    acc_R = 0
    acc_P = 0
    for sl in (slice(0, 3), slice(3, 7), slice(7, 10)):
        s = O.poetx_layer(L["x"][sl], L["dy"][sl], L["W0"], L["perm_m"], L["perm_n"],
                          L["q_R"], L["q_P"], b)
        acc_R = acc_R + s["dq_R"]
        acc_P = acc_P + s["dq_P"]
        np.testing.assert_allclose(s["y"], full["y"][sl], rtol=0, atol=1e-13)
    np.testing.assert_allclose(acc_R, full["dq_R"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(acc_P, full["dq_P"], rtol=0, atol=1e-12)


def test_row_helpers_match_full():
    m, n, b, N = 16, 8, 4, 6
    L = _layer(m, n, b, N)
    r = O.poetx_layer(L["x"], L["dy"], L["W0"], L["perm_m"], L["perm_n"], L["q_R"],
                      L["q_P"], b)
    rows = [1, 4]
    np.testing.assert_allclose(
        O.layer_forward_rows(L["x"][rows], r["Wp"], L["perm_m"], L["perm_n"], r["G_R"],
                             r["G_P"]), r["y"][rows], rtol=0, atol=1e-14)
    np.testing.assert_allclose(
        O.dx_rows(L["dy"][rows], r["Wp"], L["perm_m"], L["perm_n"], r["G_R"], r["G_P"]),
        r["dx"][rows], rtol=0, atol=1e-14)


def test_rel_fro():
    a = np.ones((2, 3, 3))
    b = a.copy()
    b[1] *= 1.1
    assert O.rel_fro(a, a) == 0.0
    assert abs(O.rel_fro(b, a, per_block=True) - 0.1) < 1e-12


# ------------------------------------------------------------------ ragged last block (N4)
def _ragged(m, n, b, N, seed, qstd=0.3):
    r = np.random.default_rng(seed)
    nR, nP = -(-m // b), -(-n // b)
    return {"x": r.standard_normal((N, m)), "dy": r.standard_normal((N, n)),
            "W0": r.standard_normal((n, m)) / np.sqrt(m), "perm_m": r.permutation(m),
            "perm_n": r.permutation(n),
            "q_R": r.standard_normal((nR, b * (b - 1) // 2)) * qstd,
            "q_P": r.standard_normal((nP, b * (b - 1) // 2)) * qstd}


def test_block_sizes():
    assert O.block_sizes(10, 4) == [4, 4, 2]
    assert O.block_sizes(8, 4) == [4, 4]
    assert O.block_sizes(9, 4) == [4, 4, 1]
    assert O.block_sizes(3, 4) == [3]


@pytest.mark.parametrize("m,n,b,N", [(10, 7, 4, 3), (9, 6, 4, 2), (6, 13, 5, 2)])
def test_ragged_layer_finite_differences(m, n, b, N):
    """Every gradient of L = <dy, y> (x, the parameters of every block including the ragged
    last ones) against central differences of the ragged forward."""
    L = _ragged(m, n, b, N, seed=m * 31 + n)
    r = O.poetx_layer_ragged(L["x"], L["dy"], L["W0"], L["perm_m"], L["perm_n"], L["q_R"],
                             L["q_P"], b)

    def loss(x, qR, qP):
        return np.sum(L["dy"] * O.poetx_layer_ragged(x, L["dy"], L["W0"], L["perm_m"],
                                                     L["perm_n"], qR, qP, b)["y"])

    h = 1e-6
    base = {"x": L["x"], "qR": L["q_R"], "qP": L["q_P"]}
    for name, grad in (("qR", r["dq_R"]), ("qP", r["dq_P"]), ("x", r["dx"])):
        arr = base[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, mm = arr.copy(), arr.copy()
            p[idx] += h
            mm[idx] -= h
            fd[idx] = (loss(**{**base, name: p}) - loss(**{**base, name: mm})) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8)


def test_ragged_entries_outside_the_last_block_are_not_parameters():
    """Changing an entry (i, k) with k >= r of the last block's row changes nothing, and its
    gradient is zero; for b = 4, r = 2 only the pair (0, 1) is a parameter."""
    m, n, b, N = 10, 8, 4, 3
    L = _ragged(m, n, b, N, seed=5)
    r0 = O.poetx_layer_ragged(L["x"], L["dy"], L["W0"], L["perm_m"], L["perm_n"], L["q_R"],
                              L["q_P"], b)
    q2 = L["q_R"].copy()
    q2[2, 1:] += 0.7          # pairs (0,2), (0,3), (1,2), (1,3), (2,3) of the last block
    r1 = O.poetx_layer_ragged(L["x"], L["dy"], L["W0"], L["perm_m"], L["perm_n"], q2,
                              L["q_P"], b)
    np.testing.assert_array_equal(r0["y"], r1["y"])
    assert np.all(r0["dq_R"][2, 1:] == 0) and r0["dq_R"][2, 0] != 0


def test_ragged_zero_q_is_plain_linear():
    m, n, b, N = 11, 9, 4, 5
    L = _ragged(m, n, b, N, seed=7)
    z = lambda a: 0 * a
    r = O.poetx_layer_ragged(L["x"], L["dy"], L["W0"], L["perm_m"], L["perm_n"], z(L["q_R"]),
                             z(L["q_P"]), b)
    np.testing.assert_allclose(r["y"], L["x"] @ L["W0"].T, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(r["dx"], L["dy"] @ L["W0"], rtol=1e-13, atol=1e-13)


def test_ragged_blocks_have_the_closed_form_defect():
    """Each block, ragged or not, is the CNP of its own skew block: G^T G = (I - Q^4)^2
    (Q^4 symmetric), and a block of one feature is the 1 x 1 identity."""
    b, d = 4, 9
    q = _rand_q(3, b)
    Gs = O.cnp_forward_ragged(q, b, d)
    assert [G.shape[0] for G in Gs] == [4, 4, 1]
    assert Gs[2].tolist() == [[1.0]]
    for j, G in enumerate(Gs[:2]):
        Q = O.triu_unpack(q[j:j + 1], b)[0]
        Q4 = np.linalg.matrix_power(Q, 4)
        np.testing.assert_allclose(G.T @ G, (np.eye(b) - Q4) @ (np.eye(b) - Q4), atol=1e-12)
    Gs2 = O.cnp_forward_ragged(q, b, 7)       # last block of 3: pairs (0,1), (0,2), (1,2)
    Q3 = np.array([[0, q[1, 0], q[1, 1]], [-q[1, 0], 0, q[1, 3]], [-q[1, 1], -q[1, 3], 0]])
    Q34 = np.linalg.matrix_power(Q3, 4)
    np.testing.assert_allclose(Gs2[1].T @ Gs2[1], (np.eye(3) - Q34) @ (np.eye(3) - Q34),
                               atol=1e-12)
