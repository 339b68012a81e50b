"""fp64 CPU oracle of the POET-X layer forward/backward and the Cayley-Neumann parameterization.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import or run this module; the product path (the CUDA library and
its Python binding) never does, and shares no code with it.

Plain, slow, obviously-correct numpy in float64.  Each function restates one step of the
method as the pages define it; library primitives used as steps are ``numpy.matmul`` and
fancy indexing, nothing is blocked, fused or reordered.  Sources are cited by page and
section:

* "POET-X summary" -- the summary page of *POET-X: Memory-efficient LLM Training by Scaling
  Orthogonal Transformation* (arXiv 2603.05500), sections "Background", "Core method"
  §1-§6 (§1 input-centric chain, eq. 3; §2 permutations and their merge; §3 batched
  block-diagonal multiply; §4 Cayley-Neumann parameterization, eq. 9/10; §5 fast/mem
  checkpointing; §6 POET-XQ).
* "POET skill page" -- *Poet Orthogonal LLM Training*, Step 1 (W = R W0 P) and Step 4
  (merge-then-reinitialize, ``merge_reinit``).

Conventions (readings of the pages, each also listed in the design notes):

* Row-vector batches: x is [N, m] (tokens x in-features), W0 is [n, m] (PyTorch Linear
  layout, n = out-features).  The learned factor G_R acts on the m (input) side, G_P on the
  n (output) side, and Q_R = Q_P = 0 gives y = x W0^T.
* A permutation is an int32 index vector pi used as a gather: x~[:, i] = x[:, pi[i]].
* The skew matrix of one block is Q = U - U^T with U the strict upper triangle filled
  row-major from the packed vector (order of ``numpy.triu_indices(b, 1)``); no factor 1/2.
* Neumann order k (the pages fix k = 3):  G = (I + Q)(I + Q + ... + Q^k).

Parity pins: every function is pinned in ``tests/test_oracle_pins.py`` against closed
forms, hand-derived worked examples (``tests/golden/``), finite differences, library
special cases and invariants.  ``quantize_rows_int8`` is pinned by its exact rounding
bound and brute force; no function here is "parity unpinned".
"""
from __future__ import annotations

from typing import Dict, Tuple

import numpy as np

F64 = np.float64


# ----------------------------------------------------------------------------------------
# Step S1: packed strict upper triangle <-> skew-symmetric block
# POET-X summary, "Core method" §4: only the upper triangle of Q is stored, b(b-1)/2 values.
# ----------------------------------------------------------------------------------------
def triu_unpack(q: np.ndarray, b: int) -> np.ndarray:
    """q [nblk, b(b-1)/2] -> Q [nblk, b, b] with Q[i,j] = q_k, Q[j,i] = -q_k for the k-th
    pair (i<j) in row-major order, and a zero diagonal."""
    q = np.asarray(q, dtype=F64)
    nblk = q.shape[0]
    assert q.shape[1] == b * (b - 1) // 2
    Q = np.zeros((nblk, b, b), dtype=F64)
    k = 0
    for i in range(b):
        cnt = b - 1 - i
        Q[:, i, i + 1:] = q[:, k:k + cnt]
        Q[:, i + 1:, i] = -q[:, k:k + cnt]
        k += cnt
    return Q


def triu_grad_pack(Qbar: np.ndarray) -> np.ndarray:
    """Gradient of the unpack step: d q_k = Qbar[i,j] - Qbar[j,i] for the k-th pair (i<j).

    Q[i,j] = q_k and Q[j,i] = -q_k, so by the chain rule dL/dq_k = Qbar_ij - Qbar_ji."""
    Qbar = np.asarray(Qbar, dtype=F64)
    nblk, b, _ = Qbar.shape
    out = np.zeros((nblk, b * (b - 1) // 2), dtype=F64)
    k = 0
    for i in range(b):
        cnt = b - 1 - i
        out[:, k:k + cnt] = Qbar[:, i, i + 1:] - Qbar[:, i + 1:, i]
        k += cnt
    return out


# ----------------------------------------------------------------------------------------
# Step S2: Cayley-Neumann parameterization forward
# POET-X summary, "Core method" §4: G ~ (I + Q)(I + sum_{i=1..3} Q^i), Q skew-symmetric.
# ----------------------------------------------------------------------------------------
def _neumann_factor(Q: np.ndarray, order: int) -> np.ndarray:
    """N(Q) = I + Q + Q^2 + ... + Q^order (truncated Neumann series of (I - Q)^-1)."""
    b = Q.shape[-1]
    I = np.eye(b, dtype=F64)
    Nq = np.broadcast_to(I, Q.shape).copy()
    P = np.broadcast_to(I, Q.shape).copy()
    for _ in range(order):
        P = P @ Q
        Nq = Nq + P
    return Nq


def cnp_forward(q: np.ndarray, b: int, order: int = 3) -> np.ndarray:
    """G [nblk, b, b] = (I + Q) N(Q) for every block (the definition, not the fused eq. 9)."""
    Q = triu_unpack(q, b)
    I = np.eye(b, dtype=F64)
    return (I + Q) @ _neumann_factor(Q, order)


# ----------------------------------------------------------------------------------------
# Step S14: Cayley-Neumann parameterization backward
# POET-X summary, "Core method" §4 (eq. 10 is named there but not printed): the gradient
# w.r.t. the packed triangle follows from the chain rule through G = (I+Q) N(Q).
# ----------------------------------------------------------------------------------------
def cnp_backward(q: np.ndarray, dG: np.ndarray, b: int, order: int = 3) -> np.ndarray:
    """dq [nblk, b(b-1)/2] given q and dL/dG [nblk, b, b] (or partials [S, nblk, b, b],
    which are summed first: the loss is linear in each partial).

    With A = I + Q and N = N(Q):  dL/dA = dG N^T,  dL/dN = A^T dG, and for the power term
    Q^p = Q...Q the adjoint is sum_{s+t=p-1} (Q^T)^s X (Q^T)^t.  Then dq from Qbar."""
    dG = np.asarray(dG, dtype=F64)
    if dG.ndim == 4:
        dG = dG.sum(axis=0)
    Q = triu_unpack(q, b)
    I = np.eye(b, dtype=F64)
    A = I + Q
    Nq = _neumann_factor(Q, order)
    dA = dG @ np.swapaxes(Nq, -1, -2)
    dN = np.swapaxes(A, -1, -2) @ dG
    Qt = np.swapaxes(Q, -1, -2)
    # powers of Q^T: Pt[s] = (Q^T)^s
    Pt = [np.broadcast_to(I, Q.shape).copy()]
    for _ in range(order):
        Pt.append(Pt[-1] @ Qt)
    Qbar = dA.copy()                       # d(I+Q)/dQ contributes dA directly
    for p in range(1, order + 1):          # N = I + sum_p Q^p
        for s in range(p):
            t = p - 1 - s
            Qbar = Qbar + Pt[s] @ dN @ Pt[t]
    return triu_grad_pack(Qbar)


# ----------------------------------------------------------------------------------------
# Steps S3/S7/S8/S13/S15: permutations as index remaps
# POET-X summary, "Core method" §2: permutations are applied by index remapping, and the
# two permutations around the frozen W are merged once into W' = Phi_n^T W Phi_m.
# ----------------------------------------------------------------------------------------
def perm_gather(X: np.ndarray, perm: np.ndarray) -> np.ndarray:
    """X~[:, i] = X[:, perm[i]]."""
    return np.asarray(X)[:, np.asarray(perm)]


def perm_scatter(Xt: np.ndarray, perm: np.ndarray) -> np.ndarray:
    """Y[:, perm[i]] = Xt[:, i]  (inverse of perm_gather)."""
    Xt = np.asarray(Xt)
    Y = np.empty_like(Xt)
    Y[:, np.asarray(perm)] = Xt
    return Y


def merge_perm(W0: np.ndarray, perm_n: np.ndarray, perm_m: np.ndarray) -> np.ndarray:
    """W'[r, c] = W0[perm_n[r], perm_m[c]]."""
    W0 = np.asarray(W0)
    return W0[np.asarray(perm_n)][:, np.asarray(perm_m)]


# ----------------------------------------------------------------------------------------
# Steps S4/S6/S10/S12: block-diagonal multiplies; S10/S12 weight gradients
# POET-X summary, "Core method" §3: every diagonal block is an independent batched product.
# ----------------------------------------------------------------------------------------
def blockdiag_mm(X: np.ndarray, G: np.ndarray, transpose: bool = False) -> np.ndarray:
    """Y = X . blkdiag(G) (or X . blkdiag(G)^T): Y[:, jb:(j+1)b] = X[:, jb:(j+1)b] G_j."""
    X = np.asarray(X, dtype=F64)
    G = np.asarray(G, dtype=F64)
    nblk, b, _ = G.shape
    assert X.shape[1] == nblk * b
    Y = np.empty_like(X)
    for j in range(nblk):
        Gj = G[j].T if transpose else G[j]
        Y[:, j * b:(j + 1) * b] = X[:, j * b:(j + 1) * b] @ Gj
    return Y


def blockdiag_wgrad(X: np.ndarray, dY: np.ndarray, b: int) -> np.ndarray:
    """dG_j = X_j^T dY_j summed over all tokens, for Y = X . blkdiag(G)."""
    X = np.asarray(X, dtype=F64)
    dY = np.asarray(dY, dtype=F64)
    nblk = X.shape[1] // b
    out = np.empty((nblk, b, b), dtype=F64)
    for j in range(nblk):
        out[j] = X[:, j * b:(j + 1) * b].T @ dY[:, j * b:(j + 1) * b]
    return out


# ----------------------------------------------------------------------------------------
# Step S16: per-row int8 quantisation of the frozen weight (POET-X summary, "Core method" §6
# says only "low-bit W, dequantised on the fly"; the scheme is our reading: symmetric
# absmax per output row).  The scale and the division are taken in fp32, the precision the
# stored weight has, so that both implementations decide each integer code identically.
# ----------------------------------------------------------------------------------------
def quantize_rows_int8(W: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    W32 = np.asarray(W, dtype=np.float32)
    amax = np.max(np.abs(W32), axis=1)
    s = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
    qv = np.rint(W32 / s[:, None])
    qv = np.clip(qv, -127, 127).astype(np.int8)
    return qv, s


def dequantize_rows(Wq: np.ndarray, s: np.ndarray) -> np.ndarray:
    return np.asarray(Wq, dtype=F64) * np.asarray(s, dtype=F64)[:, None]


# ----------------------------------------------------------------------------------------
# The layer: POET-X summary, "Core method" §1 (eq. 3) and §5.
#   a = G_R^T x,  b = W' a,  z = G_P^T b   (column form)  ==  in row form, per token row:
#   x~ = x[:, pi_m];  A = x~ blkdiag(G_R);  B = A W'^T;  z~ = B blkdiag(G_P);  y[:, pi_n] = z~
# ----------------------------------------------------------------------------------------
def layer_forward(x, Wp, perm_m, perm_n, G_R, G_P) -> Dict[str, np.ndarray]:
    """Forward through the merged weight Wp = W0[perm_n][:, perm_m].  Returns y and the
    intermediates (x~, A, B, z~)."""
    xt = perm_gather(np.asarray(x, dtype=F64), perm_m)
    A = blockdiag_mm(xt, G_R)
    B = A @ np.asarray(Wp, dtype=F64).T
    zt = blockdiag_mm(B, G_P)
    y = perm_scatter(zt, perm_n)
    return {"y": y, "xt": xt, "A": A, "B": B, "zt": zt}


def layer_backward(x, dy, Wp, perm_m, perm_n, G_R, G_P) -> Dict[str, np.ndarray]:
    """Gradients of L = <dy, y> w.r.t. x, G_R and G_P (derived by the chain rule from the
    forward above; the fast and mem variants compute the same values)."""
    b = G_R.shape[-1]
    f = layer_forward(x, Wp, perm_m, perm_n, G_R, G_P)
    dzt = perm_gather(np.asarray(dy, dtype=F64), perm_n)
    dG_P = blockdiag_wgrad(f["B"], dzt, b)
    dB = blockdiag_mm(dzt, G_P, transpose=True)
    dA = dB @ np.asarray(Wp, dtype=F64)
    dG_R = blockdiag_wgrad(f["xt"], dA, b)
    dxt = blockdiag_mm(dA, G_R, transpose=True)
    dx = perm_scatter(dxt, perm_m)
    return {"dx": dx, "dG_R": dG_R, "dG_P": dG_P, "dzt": dzt, "dB": dB, "dA": dA,
            "dxt": dxt, **{k: v for k, v in f.items()}}


def poetx_layer(x, dy, W0, perm_m, perm_n, q_R, q_P, b: int, order: int = 3):
    """End-to-end oracle of one POET-X layer step: CNP forward of both sides, the layer
    forward and backward, and the CNP backward.  W0 is the (possibly dequantised) frozen
    weight; the merge is applied here.  Returns y, dx, dq_R, dq_P (+ intermediates)."""
    G_R = cnp_forward(q_R, b, order)
    G_P = cnp_forward(q_P, b, order)
    Wp = merge_perm(W0, perm_n, perm_m)
    r = layer_backward(x, dy, Wp, perm_m, perm_n, G_R, G_P)
    r["dq_R"] = cnp_backward(q_R, r["dG_R"], b, order)
    r["dq_P"] = cnp_backward(q_P, r["dG_P"], b, order)
    r["G_R"], r["G_P"], r["Wp"] = G_R, G_P, Wp
    return r


def layer_forward_rows(x_rows, Wp, perm_m, perm_n, G_R, G_P) -> np.ndarray:
    """y for a subset of token rows (the forward is row-independent)."""
    return layer_forward(x_rows, Wp, perm_m, perm_n, G_R, G_P)["y"]


def dx_rows(dy_rows, Wp, perm_m, perm_n, G_R, G_P) -> np.ndarray:
    """dx for a subset of token rows (the input gradient is row-independent)."""
    dzt = perm_gather(np.asarray(dy_rows, dtype=F64), perm_n)
    dB = blockdiag_mm(dzt, G_P, transpose=True)
    dA = dB @ np.asarray(Wp, dtype=F64)
    return perm_scatter(blockdiag_mm(dA, G_R, transpose=True), perm_m)


# ----------------------------------------------------------------------------------------
# Merge-then-reinitialize (POET skill page, Step 4: the current R W0 P is written back into
# W0 and the factors are reset to the identity; the POET-X summary's "inner optimization"
# loop between merges).  In this library's form the factors are q = 0 after the reset and
# the permutations are drawn anew and merged again (merge_perm).
# ----------------------------------------------------------------------------------------
def merge_reinit(Wp, perm_m, perm_n, q_R, q_P, b: int, order: int = 3) -> np.ndarray:
    """W0_new [n, m]: the weight with which the layer at q = 0 computes the same linear map
    as the layer with the merged weight Wp, the permutations and q_R, q_P.  It is that map's
    matrix, read off as the layer's response to the identity batch (row i of the response
    is the image of the i-th unit input)."""
    G_R = cnp_forward(q_R, b, order)
    G_P = cnp_forward(q_P, b, order)
    m = np.asarray(Wp).shape[1]
    return layer_forward(np.eye(m, dtype=F64), Wp, perm_m, perm_n, G_R, G_P)["y"].T


# ----------------------------------------------------------------------------------------
# Optimizer step on the packed triangles.  The POET-X summary ("Core method" §4) counts the
# optimizer state per stored parameter, b(b-1)/2 per block, and ("Practical guidance" 3)
# scales the learning rate by gamma = 0.5 for POET-XQ; it names no optimizer.  Our reading:
# Adam (Kingma & Ba, Algorithm 1) with decoupled weight decay (AdamW), elementwise on q;
# gamma is folded into lr by the caller.
# ----------------------------------------------------------------------------------------
def adam_step(q, g, m, v, t: int, lr: float, beta1: float = 0.9, beta2: float = 0.999,
              eps: float = 1e-8, weight_decay: float = 0.0):
    """One step at step count t >= 1.  Returns (q_new, m_new, v_new)."""
    q = np.asarray(q, dtype=F64)
    g = np.asarray(g, dtype=F64)
    m_new = beta1 * np.asarray(m, dtype=F64) + (1.0 - beta1) * g
    v_new = beta2 * np.asarray(v, dtype=F64) + (1.0 - beta2) * g * g
    m_hat = m_new / (1.0 - beta1 ** t)
    v_hat = v_new / (1.0 - beta2 ** t)
    q_new = q - lr * (m_hat / (np.sqrt(v_hat) + eps) + weight_decay * q)
    return q_new, m_new, v_new


# ----------------------------------------------------------------------------------------
# Ragged last block.  The POET-X summary ("Core method" §1) splits a side of d features into
# ceil(d/b) blocks; when b does not divide d the last block has r = d - (ceil(d/b) - 1) b
# features and its own r x r factor.  Storage (our reading, the pages do not say): q keeps
# one row of b(b-1)/2 entries per block; the last block's parameters are the entries of the
# pairs (i, k), i < k < r, at their places in the b-block's row-major order, and the other
# entries of that row are not parameters (ignored on input, zero gradient).  Written out
# per block with its own size, without padding.
# ----------------------------------------------------------------------------------------
def block_sizes(d: int, b: int):
    """Sizes of the ceil(d/b) blocks of a side of d features."""
    nb = -(-d // b)
    return [min(b, d - j * b) for j in range(nb)]


def _skew_of_row(qrow: np.ndarray, b: int, r: int) -> np.ndarray:
    """The r x r skew block of one packed row (pairs i < k < r of the b-block order)."""
    Q = np.zeros((r, r), dtype=F64)
    k = 0
    for i in range(b):
        for j in range(i + 1, b):
            if j < r:
                Q[i, j] = qrow[k]
                Q[j, i] = -qrow[k]
            k += 1
    return Q


def cnp_forward_ragged(q: np.ndarray, b: int, d: int, order: int = 3):
    """[G_j] for the blocks of a side of d features, G_j = (I + Q_j) N(Q_j) of size b_j."""
    q = np.asarray(q, dtype=F64)
    out = []
    for j, r in enumerate(block_sizes(d, b)):
        Q = _skew_of_row(q[j], b, r)
        out.append((np.eye(r) + Q) @ _neumann_factor(Q, order))
    return out


def cnp_backward_ragged(q: np.ndarray, dGs, b: int, d: int, order: int = 3) -> np.ndarray:
    """dq [ceil(d/b), b(b-1)/2] from the per-block dL/dG_j (sizes b_j); entries that are
    not parameters of the last block get zero.  Per block this is cnp_backward's chain rule
    (dL/d(I+Q) = dG N^T, dL/dN = (I+Q)^T dG, the power adjoints), then dq_k = Qbar_ij -
    Qbar_ji for the parameter pairs."""
    q = np.asarray(q, dtype=F64)
    sizes = block_sizes(d, b)
    out = np.zeros((len(sizes), b * (b - 1) // 2), dtype=F64)
    for j, r in enumerate(sizes):
        Q = _skew_of_row(q[j], b, r)
        I = np.eye(r)
        A = I + Q
        Nq = _neumann_factor(Q, order)
        dG = np.asarray(dGs[j], dtype=F64)
        dA = dG @ Nq.T
        dN = A.T @ dG
        Pt = [I]
        for _ in range(order):
            Pt.append(Pt[-1] @ Q.T)
        Qbar = dA.copy()
        for p in range(1, order + 1):
            for s in range(p):
                Qbar = Qbar + Pt[s] @ dN @ Pt[p - 1 - s]
        k = 0
        for i in range(b):
            for c in range(i + 1, b):
                if c < r:
                    out[j, k] = Qbar[i, c] - Qbar[c, i]
                k += 1
    return out


def blockdiag_mm_ragged(X: np.ndarray, Gs, transpose: bool = False) -> np.ndarray:
    """Y[:, o_j:o_j+b_j] = X[:, o_j:o_j+b_j] G_j (or G_j^T), o_j = sum of earlier sizes."""
    X = np.asarray(X, dtype=F64)
    Y = np.empty_like(X)
    o = 0
    for G in Gs:
        r = G.shape[0]
        Y[:, o:o + r] = X[:, o:o + r] @ (G.T if transpose else G)
        o += r
    assert o == X.shape[1]
    return Y


def blockdiag_wgrad_ragged(X: np.ndarray, dY: np.ndarray, sizes):
    """[dG_j = X_j^T dY_j] for the column blocks of the given sizes."""
    X = np.asarray(X, dtype=F64)
    dY = np.asarray(dY, dtype=F64)
    out, o = [], 0
    for r in sizes:
        out.append(X[:, o:o + r].T @ dY[:, o:o + r])
        o += r
    return out


def poetx_layer_ragged(x, dy, W0, perm_m, perm_n, q_R, q_P, b: int, order: int = 3):
    """poetx_layer for any m, n: ceil(m/b) and ceil(n/b) blocks, the last ones ragged.
    Returns y, dx, dq_R, dq_P (dq rows of b(b-1)/2 with the non-parameters zero)."""
    x = np.asarray(x, dtype=F64)
    dy = np.asarray(dy, dtype=F64)
    m, n = x.shape[1], dy.shape[1]
    G_R = cnp_forward_ragged(q_R, b, m, order)
    G_P = cnp_forward_ragged(q_P, b, n, order)
    Wp = merge_perm(W0, perm_n, perm_m)
    xt = perm_gather(x, perm_m)
    A = blockdiag_mm_ragged(xt, G_R)
    B = A @ Wp.T
    zt = blockdiag_mm_ragged(B, G_P)
    y = perm_scatter(zt, perm_n)
    dzt = perm_gather(dy, perm_n)
    dG_P = blockdiag_wgrad_ragged(B, dzt, block_sizes(n, b))
    dB = blockdiag_mm_ragged(dzt, G_P, transpose=True)
    dA = dB @ Wp
    dG_R = blockdiag_wgrad_ragged(xt, dA, block_sizes(m, b))
    dx = perm_scatter(blockdiag_mm_ragged(dA, G_R, transpose=True), perm_m)
    return {"y": y, "dx": dx, "dq_R": cnp_backward_ragged(q_R, dG_R, b, m, order),
            "dq_P": cnp_backward_ragged(q_P, dG_P, b, n, order), "G_R": G_R, "G_P": G_P}


# ----------------------------------------------------------------------------------------
# Error metric used by every parity test: relative Frobenius error, optionally the max over
# the leading (block) axis.
# ----------------------------------------------------------------------------------------
def rel_fro(got, ref, per_block: bool = False) -> float:
    got = np.asarray(got, dtype=F64)
    ref = np.asarray(ref, dtype=F64)
    if per_block:
        num = np.sqrt(((got - ref) ** 2).reshape(ref.shape[0], -1).sum(axis=1))
        den = np.sqrt((ref ** 2).reshape(ref.shape[0], -1).sum(axis=1))
        den = np.where(den == 0, 1.0, den)
        return float(np.max(num / den)) if ref.shape[0] else 0.0
    den = np.sqrt((ref ** 2).sum())
    num = np.sqrt(((got - ref) ** 2).sum())
    return float(num / (den if den > 0 else 1.0))
