"""The data-parallel exchange on CPU ranks (gloo, world size 2): each rank computes the
oracle gradient of its token shard, a sum all-reduce gives the full-batch gradient.  The
CUDA library itself runs one replica per GPU with no collective; this pins the exchange
that a multi-GPU trainer would add (POET-X summary page, "Practice notes" §4: DDP)."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O


def _layer(ragged=False):
    r = np.random.default_rng(5)
    m, n, b, N = (18, 10, 4, 10) if ragged else (16, 8, 4, 10)
    return dict(x=r.standard_normal((N, m)), dy=r.standard_normal((N, n)),
                W0=r.standard_normal((n, m)) / 4, perm_m=r.permutation(m), perm_n=r.permutation(n),
                q_R=r.standard_normal((-(-m // b), b * (b - 1) // 2)) * 0.2,
                q_P=r.standard_normal((-(-n // b), b * (b - 1) // 2)) * 0.2, b=b)


def _grads(L, rows, ragged):
    f = O.poetx_layer_ragged if ragged else O.poetx_layer
    return f(L["x"][rows], L["dy"][rows], L["W0"], L["perm_m"], L["perm_n"], L["q_R"],
             L["q_P"], L["b"])


def _worker(rank, world, port, out, ragged):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    L = _layer(ragged)
    sl = np.array_split(np.arange(L["x"].shape[0]), world)[rank]
    r = _grads(L, sl, ragged)
    g = torch.tensor(np.concatenate([r["dq_R"].ravel(), r["dq_P"].ravel()]))
    dist.all_reduce(g)
    if rank == 0:
        out.put(g.numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("ragged", [False, True])
def test_gloo_allreduce_of_shard_gradients_equals_full_batch(ragged):
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q, ragged)) for r in range(2)]
    for p in procs:
        p.start()
    got = q.get(timeout=120)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    L = _layer(ragged)
    full = _grads(L, slice(None), ragged)
    ref = np.concatenate([full["dq_R"].ravel(), full["dq_P"].ravel()])
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
