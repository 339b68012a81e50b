"""The data-parallel training step on CPU ranks (gloo, world size 2), through the same step
function the benchmark runs on GPU ranks (``dp.data_parallel_step``): each rank computes the
oracle gradient of its token shard into the flat gradient buffer, the exchange sums the
buffers over ranks, and the Adam update then runs on every rank.  The summed gradient must
equal the full-batch gradient, and the updated parameters those of one full-batch step
(POET-X summary page, "Practice notes": distributed data parallelism)."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O
from orthogonal_reparameterized_gb300 import dp

LR = 0.01


def _layers(ragged=False):
    r = np.random.default_rng(5)
    shapes = [(18, 10, 4, 10), (8, 12, 4, 10)] if ragged else [(16, 8, 4, 10), (8, 16, 4, 10)]
    out = []
    for m, n, b, N in shapes:
        out.append(dict(x=r.standard_normal((N, m)), dy=r.standard_normal((N, n)),
                        W0=r.standard_normal((n, m)) / 4, perm_m=r.permutation(m),
                        perm_n=r.permutation(n),
                        q_R=r.standard_normal((-(-m // b), b * (b - 1) // 2)) * 0.2,
                        q_P=r.standard_normal((-(-n // b), b * (b - 1) // 2)) * 0.2, b=b))
    return out


def _grads(L, rows, ragged):
    f = O.poetx_layer_ragged if ragged else O.poetx_layer
    return f(L["x"][rows], L["dy"][rows], L["W0"], L["perm_m"], L["perm_n"], L["q_R"],
             L["q_P"], L["b"])


def _shapes(layers):
    out = []
    for i, L in enumerate(layers):
        out += [(f"{i}R", L["q_R"].shape), (f"{i}P", L["q_P"].shape)]
    return out


def _worker(rank, world, port, out, ragged):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    layers = _layers(ragged)
    shapes = _shapes(layers)
    grads = dp.FlatBuffer(shapes, "cpu")
    q = dp.FlatBuffer(shapes, "cpu")
    for i, L in enumerate(layers):
        q.view(f"{i}R").copy_(torch.tensor(L["q_R"]))
        q.view(f"{i}P").copy_(torch.tensor(L["q_P"]))
    q_new = {}

    def compute():
        for i, L in enumerate(layers):
            sl = np.array_split(np.arange(L["x"].shape[0]), world)[rank]
            r = _grads(L, sl, ragged)
            grads.view(f"{i}R").copy_(torch.tensor(r["dq_R"]))
            grads.view(f"{i}P").copy_(torch.tensor(r["dq_P"]))

    def update():  # the oracle's Adam step (step 1, zero state) on the summed gradient
        g = grads.flat.double().numpy()
        qq = q.flat.double().numpy()
        qn, _, _ = O.adam_step(qq, g, np.zeros_like(g), np.zeros_like(g), 1, LR)
        q_new["q"] = qn

    dp.data_parallel_step(compute, grads.flat, update)
    out.put((rank, grads.flat.double().numpy(), q_new["q"]))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("ragged", [False, True])
def test_data_parallel_step_equals_full_batch(ragged):
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    qu = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, qu, ragged)) for r in range(2)]
    for p in procs:
        p.start()
    got = [qu.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    layers = _layers(ragged)
    shapes = _shapes(layers)
    ref = dp.FlatBuffer(shapes, "cpu")
    q0 = dp.FlatBuffer(shapes, "cpu")
    for i, L in enumerate(layers):
        full = _grads(L, slice(None), ragged)
        ref.view(f"{i}R").copy_(torch.tensor(full["dq_R"]))
        ref.view(f"{i}P").copy_(torch.tensor(full["dq_P"]))
        q0.view(f"{i}R").copy_(torch.tensor(L["q_R"]))
        q0.view(f"{i}P").copy_(torch.tensor(L["q_P"]))
    g_ref = ref.flat.double().numpy()
    q_ref, _, _ = O.adam_step(q0.flat.double().numpy(), g_ref, np.zeros_like(g_ref),
                              np.zeros_like(g_ref), 1, LR)
    for rank, g, qn in got:
        # fp32 buffers: the shard gradients and their sum are rounded to fp32
        np.testing.assert_allclose(g, g_ref, rtol=1e-6, atol=1e-6, err_msg=f"rank {rank}")
        np.testing.assert_allclose(qn, q_ref, rtol=1e-6, atol=1e-6, err_msg=f"rank {rank}")
    # both ranks hold the same parameters after the step
    np.testing.assert_array_equal(got[0][2], got[1][2])


def test_flat_buffer_views_are_aligned_and_disjoint():
    fb = dp.FlatBuffer([("a", (3, 5)), ("b", (7,)), ("c", (2, 2))], "cpu")
    for name in fb.names():
        assert fb.view(name).data_ptr() % 16 == 0
    fb.view("a").fill_(1.0)
    fb.view("b").fill_(2.0)
    fb.view("c").fill_(3.0)
    assert float(fb.view("a").sum()) == 15.0
    assert float(fb.view("b").sum()) == 14.0
    assert float(fb.view("c").sum()) == 12.0
