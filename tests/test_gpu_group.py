"""Parity of the layer-group calls (one batched CNP forward and backward over every block of
every layer, the layers' chains in between) with the fp64 oracle layer by layer, and with the
single-layer calls on the same inputs (POET-X summary page, "Core method" sections 1-5)."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import DEV, P, TOL_BF16_LAYER, TOL_F32, dev, host  # noqa: F401
from orthogonal_reparameterized_gb300 import inputs

pytestmark = pytest.mark.gpu

TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _build(P, spec, b, act, N, seed):
    """Device tensors and a descriptor per layer; spec: (m, n, wdt, variant) per layer."""
    layers = []
    for k, (m, n, wdt, variant) in enumerate(spec):
        inp = inputs.small_layer_inputs(seed + 17 * k, m, n, b, N, act=act, wdt=wdt)
        m_pad, n_pad = -(-m // b) * b, -(-n // b) * b
        d = dict(inp=inp, m=m, n=n, wdt=wdt, variant=variant)
        d["x"] = dev(inp["x"], TDT[act])
        d["dy"] = dev(inp["dy"], TDT[act])
        d["pm"] = dev(inp["perm_m"], torch.int32)
        d["pn"] = dev(inp["perm_n"], torch.int32)
        d["qR"] = dev(inp["q_R"], torch.float32)
        d["qP"] = dev(inp["q_P"], torch.float32)
        d["w_scale"] = None
        if wdt == "i8":
            Wq, s = O.quantize_rows_int8(inp["W0"])
            Wq_d = torch.tensor(Wq, device=DEV)
            s_d = dev(s, torch.float32)
            d["Wp"] = torch.empty(n_pad, m_pad, dtype=torch.int8, device=DEV)
            d["w_scale"] = torch.empty(n_pad, device=DEV)
            P.poetx_merge_perm_padded(Wq_d, d["pn"], d["pm"], d["Wp"], s_d, d["w_scale"])
            d["W_eff"] = O.dequantize_rows(Wq, s)
            wcode = P.I8
        else:
            W0 = dev(inp["W0"], TDT[wdt])
            d["Wp"] = torch.empty(n_pad, m_pad, dtype=W0.dtype, device=DEV)
            P.poetx_merge_perm_padded(W0, d["pn"], d["pm"], d["Wp"])
            d["W_eff"] = inp["W0"]
            wcode = P.BF16 if wdt == "bf16" else P.F32
        acode = P.BF16 if act == "bf16" else P.F32
        vcode = P.FAST if variant == "fast" else P.MEM
        d["L"] = P.make_layer(m, n, b, acode, wcode, vcode, d["pm"], d["pn"], d["Wp"], d["qR"],
                              d["qP"], d["w_scale"])
        layers.append(d)
    return layers


def _run_group(P, layers, N, act, order=None):
    G = P.make_group([d["L"] for d in layers])
    saved = P.workspace(P.poetx_group_saved_bytes(G, N), DEV)
    ws = P.workspace(P.poetx_group_workspace_bytes(G, N), DEV)
    ys = [torch.empty(N, d["n"], dtype=TDT[act], device=DEV) for d in layers]
    dxs = [torch.empty(N, d["m"], dtype=TDT[act], device=DEV) for d in layers]
    dqR = [torch.full_like(d["qR"], float("nan")) for d in layers]
    dqP = [torch.full_like(d["qP"], float("nan")) for d in layers]
    P.poetx_group_cnp_fwd(G, N, saved)
    fwd_order = list(range(len(layers))) if order is None else order
    for i in fwd_order:
        P.poetx_group_layer_fwd(G, i, layers[i]["x"], ys[i], saved, ws)
    for i in reversed(fwd_order):
        P.poetx_group_layer_bwd(G, i, layers[i]["x"], layers[i]["dy"], saved, dxs[i], ws)
    P.poetx_group_cnp_bwd(G, N, saved, dqR, dqP, ws)
    torch.cuda.synchronize()
    assert P.poetx_get_device_error() == 0
    return [{"y": host(ys[i]), "dx": host(dxs[i]), "dq_R": host(dqR[i]), "dq_P": host(dqP[i])}
            for i in range(len(layers))]


def _run_single(P, d, N, act):
    L = d["L"]
    saved = P.workspace(P.poetx_layer_saved_bytes(L, N), DEV)
    wsf = P.workspace(P.poetx_layer_workspace_bytes(L, N, 0), DEV)
    wsb = P.workspace(P.poetx_layer_workspace_bytes(L, N, 1), DEV)
    y = torch.empty(N, d["n"], dtype=TDT[act], device=DEV)
    dx = torch.empty(N, d["m"], dtype=TDT[act], device=DEV)
    dqR = torch.empty_like(d["qR"])
    dqP = torch.empty_like(d["qP"])
    P.poetx_layer_fwd(L, d["x"], y, saved, wsf)
    P.poetx_layer_bwd(L, d["x"], d["dy"], saved, dx, dqR, dqP, wsb)
    torch.cuda.synchronize()
    assert P.poetx_get_device_error() == 0
    return {"y": host(y), "dx": host(dx), "dq_R": host(dqR), "dq_P": host(dqP)}


def _oracle(d, b):
    inp = d["inp"]
    ragged = d["m"] % b or d["n"] % b
    f = O.poetx_layer_ragged if ragged else O.poetx_layer
    return f(inp["x"], inp["dy"], d["W_eff"], inp["perm_m"], inp["perm_n"], inp["q_R"],
             inp["q_P"], b)


KEYS = ("y", "dx", "dq_R", "dq_P")

# bf16 groups: square and non-square, fast and mem, an int8 mem layer, ragged last blocks
GROUPS = {
    "mixed_b128": ([(256, 512, "bf16", "fast"), (512, 384, "bf16", "mem"),
                    (384, 256, "i8", "mem"), (384, 384, "bf16", "fast")], 128, 150),
    "ragged_b128": ([(256, 200, "bf16", "fast"), (200, 264, "bf16", "mem"),
                     (264, 256, "bf16", "fast")], 128, 97),
    "block_b256": ([(512, 512, "bf16", "fast")] * 2 + [(512, 1024, "bf16", "fast"),
                                                      (1024, 512, "bf16", "fast")], 256, 300),
    # a ragged bf16 first layer and an int8 layer, 700 tokens
    "mixed_ragged_b128": ([(200, 264, "bf16", "fast"), (256, 512, "bf16", "mem"),
                    (384, 256, "i8", "mem")], 128, 700),
}


@pytest.mark.parametrize("name", list(GROUPS))
def test_group_matches_oracle_and_single_layer_calls(P, name):
    spec, b, N = GROUPS[name]
    layers = _build(P, spec, b, "bf16", N, seed=300 + b)
    got = _run_group(P, layers, N, "bf16")
    for i, d in enumerate(layers):
        ref = _oracle(d, b)
        errs = {k: O.rel_fro(got[i][k], ref[k]) for k in KEYS}
        assert max(errs.values()) <= TOL_BF16_LAYER, (i, errs)
        single = _run_single(P, d, N, "bf16")
        for k in KEYS:  # the same kernels on the same blocks: bit for bit
            np.testing.assert_array_equal(got[i][k], single[k], err_msg=f"layer {i} {k}")
        if d["m"] % b:  # non-parameters of a ragged last block get exactly zero
            r = d["m"] % b
            iu, ju = np.triu_indices(b, 1)
            assert not np.any(got[i]["dq_R"][-1][~((iu < r) & (ju < r))])


def test_group_fp32(P):
    spec = [(256, 256, "f32", "fast"), (256, 128, "f32", "mem")]
    layers = _build(P, spec, 32, "f32", 64, seed=901)
    got = _run_group(P, layers, 64, "f32")
    for i, d in enumerate(layers):
        ref = _oracle(d, 32)
        errs = {k: O.rel_fro(got[i][k], ref[k]) for k in KEYS}
        assert max(errs.values()) <= TOL_F32, (i, errs)


def test_group_layer_order_and_zero_tokens(P):
    """Layers may run in any order between the CNP calls; N = 0 gives zero gradients."""
    spec, b, N = GROUPS["mixed_b128"]
    layers = _build(P, spec, b, "bf16", N, seed=428)
    a = _run_group(P, layers, N, "bf16")
    c = _run_group(P, layers, N, "bf16", order=[2, 0, 3, 1])
    for i in range(len(layers)):
        for k in KEYS:
            np.testing.assert_array_equal(a[i][k], c[i][k], err_msg=f"layer {i} {k}")
    empty = _build(P, spec, b, "bf16", 0, seed=429)
    z = _run_group(P, empty, 0, "bf16")
    for i in range(len(empty)):
        assert not np.any(z[i]["dq_R"]) and not np.any(z[i]["dq_P"])


def test_group_argument_errors(P):
    spec, b, N = GROUPS["mixed_b128"]
    layers = _build(P, spec, b, "bf16", 8, seed=5)
    G = P.make_group([d["L"] for d in layers])
    saved = P.workspace(P.poetx_group_saved_bytes(G, 8), DEV)
    ws = P.workspace(P.poetx_group_workspace_bytes(G, 8), DEV)
    y = torch.empty(8, layers[0]["n"], dtype=torch.bfloat16, device=DEV)
    with pytest.raises(P.PoetxError) as e:
        P.poetx_group_layer_fwd(G, len(layers), layers[0]["x"], y, saved, ws)
    assert e.value.status == 1  # i out of range
    small = P.workspace(16, DEV)
    with pytest.raises(P.PoetxError) as e:
        P.poetx_group_layer_fwd(G, 0, layers[0]["x"], y, saved, small)
    assert e.value.status == 5
    other = _build(P, [(256, 256, "bf16", "fast")], 64, "bf16", 8, seed=6)
    mixed = P.make_group([layers[0]["L"], other[0]["L"]])  # two block sizes
    assert P.poetx_group_saved_bytes(mixed, 8) == 0


@pytest.mark.parametrize("name", ["mixed_b128", "ragged_b128", "block_b256", "mixed_ragged_b128"])
def test_group_step_host_equals_device_calls(P, name):
    """The host-buffer group step (uploads and downloads beside the kernels) gives the same
    bits as the device group calls, and N = 0 gives zero gradients."""
    spec, b, N = GROUPS[name]
    layers = _build(P, spec, b, "bf16", N, seed=700 + b)
    ref = _run_group(P, layers, N, "bf16")
    G = P.make_group([d["L"] for d in layers])
    pin = lambda t: t.detach().cpu().contiguous().pin_memory()
    xs = [pin(d["x"]) for d in layers]
    dys = [pin(d["dy"]) for d in layers]
    ys = [torch.empty(N, d["n"], dtype=torch.bfloat16).pin_memory() for d in layers]
    dxs = [torch.empty(N, d["m"], dtype=torch.bfloat16).pin_memory() for d in layers]
    dqR = [torch.full(tuple(d["qR"].shape), float("nan")).pin_memory() for d in layers]
    dqP = [torch.full(tuple(d["qP"].shape), float("nan")).pin_memory() for d in layers]
    dev = P.workspace(P.poetx_group_step_host_bytes(G, N), DEV)
    for _ in range(2):  # a repeated step gives the same bits
        P.poetx_group_step_host(G, xs, dys, ys, dxs, dqR, dqP, dev)
        torch.cuda.synchronize()
        assert P.poetx_get_device_error() == 0
        for i in range(len(layers)):
            np.testing.assert_array_equal(ys[i].float().numpy(), ref[i]["y"], err_msg=f"y {i}")
            np.testing.assert_array_equal(dxs[i].float().numpy(), ref[i]["dx"], err_msg=f"dx {i}")
            np.testing.assert_array_equal(dqR[i].numpy(), ref[i]["dq_R"], err_msg=f"dq_R {i}")
            np.testing.assert_array_equal(dqP[i].numpy(), ref[i]["dq_P"], err_msg=f"dq_P {i}")
    empty = _build(P, spec, b, "bf16", 0, seed=701)
    G0 = P.make_group([d["L"] for d in empty])
    z = lambda shape, dt=torch.bfloat16: torch.empty(shape, dtype=dt).pin_memory()
    dqR0 = [torch.full(tuple(d["qR"].shape), float("nan")).pin_memory() for d in empty]
    dqP0 = [torch.full(tuple(d["qP"].shape), float("nan")).pin_memory() for d in empty]
    P.poetx_group_step_host(G0, [z((0, d["m"])) for d in empty], [z((0, d["n"])) for d in empty],
                            [z((0, d["n"])) for d in empty], [z((0, d["m"])) for d in empty],
                            dqR0, dqP0, P.workspace(P.poetx_group_step_host_bytes(G0, 0), DEV))
    torch.cuda.synchronize()
    assert all(not np.any(t.numpy()) for t in dqR0 + dqP0)
