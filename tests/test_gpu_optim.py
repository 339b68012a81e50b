"""Adam on the packed triangles (poetx_adam_triu) against the fp64 oracle: fp32 state and
arithmetic, so the update and the state match to 1e-5 relative (Frobenius).  The
hyperparameters cross the C ABI as fp32, so the oracle gets the same fp32 values (0.999
in fp32 is 1 - 0.99998713e-3: a 1.3e-5 relative change of 1 - beta2)."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import DEV, P, TOL_F32, dev, host  # noqa: F401

pytestmark = pytest.mark.gpu


def _f32(**hp):
    return {k: float(np.float32(v)) for k, v in hp.items()}


def _state(count, seed):
    r = np.random.default_rng(seed)
    q = (r.standard_normal(count) * 0.02).astype(np.float32)
    m = (r.standard_normal(count) * 1e-3).astype(np.float32)
    v = (np.abs(r.standard_normal(count)) * 1e-6).astype(np.float32)
    return q, m, v


@pytest.mark.parametrize("count", [1, 7, 1001, 4096 * 255 // 2])
@pytest.mark.parametrize("step", [1, 10])
def test_adam_matches_oracle(P, count, step):
    q, m, v = _state(count, count + step)
    if step == 1:
        m[:] = 0
        v[:] = 0
    g = (np.random.default_rng(step).standard_normal(count) * 1e-2).astype(np.float32)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    qd, md, vd, gd = (dev(a, torch.float32) for a in (q, m, v, g))
    P.poetx_adam_triu(qd, gd, md, vd, step, **hp)
    torch.cuda.synchronize()
    qr, mr, vr = O.adam_step(q, g, m, v, step, **_f32(**hp))
    assert O.rel_fro(host(qd) - q, qr - q) <= TOL_F32  # the update itself
    assert O.rel_fro(host(md), mr) <= TOL_F32
    assert O.rel_fro(host(vd), vr) <= TOL_F32


def test_adam_sequence_of_steps(P):
    count = 10000
    q, _, _ = _state(count, 3)
    m = np.zeros(count, np.float32)
    v = np.zeros(count, np.float32)
    qd, md, vd = (dev(a, torch.float32) for a in (q, m, v))
    qr, mr, vr = q.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    r = np.random.default_rng(11)
    for t in range(1, 6):
        g = (r.standard_normal(count) * 1e-2).astype(np.float32)
        P.poetx_adam_triu(qd, dev(g, torch.float32), md, vd, t, lr=2e-3, beta1=0.8, beta2=0.99,
                          eps=1e-6)
        qr, mr, vr = O.adam_step(qr, g, mr, vr, t, **_f32(lr=2e-3, beta1=0.8, beta2=0.99,
                                                           eps=1e-6))
    torch.cuda.synchronize()
    assert O.rel_fro(host(qd) - q, qr - q) <= TOL_F32
    assert O.rel_fro(host(vd), vr) <= TOL_F32


@pytest.mark.parametrize("m,n,b,N,step,acc", [(1024, 512, 128, 300, 1, False),
                                              (2048, 2048, 256, 333, 5, False),
                                              (200, 328, 64, 150, 2, True)])   # ragged sides
def test_layer_bwd_adam_equals_bwd_then_adam(P, m, n, b, N, step, acc):
    """The optimizer applied by the gradient pack gives the same bits as poetx_layer_bwd
    followed by poetx_adam_triu on each side (q, m, v, dq, dx), and its update matches the
    oracle's Adam on the oracle's gradient."""
    from orthogonal_reparameterized_gb300 import inputs
    inp = inputs.small_layer_inputs(400 + m + b, m, n, b, N, act="bf16", wdt="bf16")
    m_pad, n_pad = -(-m // b) * b, -(-n // b) * b
    x = dev(inp["x"], torch.bfloat16)
    dy = dev(inp["dy"], torch.bfloat16)
    pm = dev(inp["perm_m"], torch.int32)
    pn = dev(inp["perm_n"], torch.int32)
    W0 = dev(inp["W0"], torch.bfloat16)
    Wp = torch.empty(n_pad, m_pad, dtype=torch.bfloat16, device=DEV)
    P.poetx_merge_perm_padded(W0, pn, pm, Wp)
    r = np.random.default_rng(step)
    state = {}
    for side, q in (("R", inp["q_R"]), ("P", inp["q_P"])):
        mm = np.zeros(q.shape, np.float32) if step == 1 else (r.standard_normal(q.shape) * 1e-3).astype(np.float32)
        vv = np.zeros(q.shape, np.float32) if step == 1 else (np.abs(r.standard_normal(q.shape)) * 1e-6).astype(np.float32)
        state[side] = (np.asarray(q, np.float32), mm, vv)
    dq0 = {s: (r.standard_normal(state[s][0].shape) * 1e-3).astype(np.float32) for s in "RP"}
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    outs = []
    for fused in (False, True):
        q = {s: dev(state[s][0], torch.float32) for s in "RP"}
        mo = {s: dev(state[s][1], torch.float32) for s in "RP"}
        vo = {s: dev(state[s][2], torch.float32) for s in "RP"}
        dq = {s: dev(dq0[s], torch.float32) for s in "RP"}
        L = P.make_layer(m, n, b, P.BF16, P.BF16, P.FAST, pm, pn, Wp, q["R"], q["P"], None)
        saved = P.workspace(P.poetx_layer_saved_bytes(L, N), DEV)
        wsf = P.workspace(P.poetx_layer_workspace_bytes(L, N, 0), DEV)
        wsb = P.workspace(P.poetx_layer_workspace_bytes(L, N, 1), DEV)
        y = torch.empty(N, n, dtype=torch.bfloat16, device=DEV)
        dx = torch.empty(N, m, dtype=torch.bfloat16, device=DEV)
        P.poetx_layer_fwd(L, x, y, saved, wsf)
        if fused:
            P.poetx_layer_bwd_adam(L, x, dy, saved, dx, dq["R"], dq["P"], wsb, mo["R"], vo["R"],
                                   mo["P"], vo["P"], step, accumulate=acc, **hp)
        else:
            P.poetx_layer_bwd(L, x, dy, saved, dx, dq["R"], dq["P"], wsb, accumulate=acc)
            for s in "RP":
                P.poetx_adam_triu(q[s], dq[s], mo[s], vo[s], step, **hp)
        torch.cuda.synchronize()
        assert P.poetx_get_device_error() == 0
        outs.append({"dx": host(dx), **{f"{k}{s}": host(t[s]) for k, t in
                                         (("q", q), ("m", mo), ("v", vo), ("dq", dq))
                                         for s in "RP"}})
    for k in outs[0]:
        np.testing.assert_array_equal(outs[0][k], outs[1][k], err_msg=k)
    ref = O.poetx_layer_ragged(inp["x"], inp["dy"], inp["W0"], inp["perm_m"], inp["perm_n"],
                               inp["q_R"], inp["q_P"], b)
    for s, key in (("R", "dq_R"), ("P", "dq_P")):
        # the gradient the pack wrote: the layer's (bf16 tolerance) plus the accumulated dq0
        g = outs[1][f"dq{s}"]
        assert O.rel_fro(g, ref[key] + (dq0[s] if acc else 0)) <= 2e-2
        # and the update applied to it: the oracle's Adam on that same gradient
        q0, m0, v0 = state[s]
        qr, mr, vr = O.adam_step(q0, g, m0, v0, step, **_f32(**hp))
        assert O.rel_fro(outs[1][f"q{s}"] - q0, qr - q0) <= TOL_F32
        assert O.rel_fro(outs[1][f"m{s}"], mr) <= TOL_F32
        assert O.rel_fro(outs[1][f"v{s}"], vr) <= TOL_F32
