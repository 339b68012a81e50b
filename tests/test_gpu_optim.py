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
