"""Parity of the whole POET-X layer (both CNPs, forward, backward; fast and mem variants)
with the fp64 oracle on identical seeded inputs: 1e-5 for the fp32 layer, 2e-2 for bf16
(relative Frobenius error of y, dx, dq_R and dq_P)."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import DEV, P, TOL_BF16_LAYER, TOL_F32, dev, host  # noqa: F401
from orthogonal_reparameterized_gb300 import inputs

pytestmark = pytest.mark.gpu

TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


def run_layer(P, inp, b, act, wdt, variant, dy=None, q_zero=False, accumulate_init=None):
    """Runs fwd + bwd through the C ABI; returns host arrays and the effective W0 that the
    oracle must use (for int8 weights, the oracle's own quantisation of W0 dequantised: the
    library's quantiser is checked bit for bit against it on its own)."""
    m, n = inp["W0"].shape[1], inp["W0"].shape[0]
    m_pad, n_pad = -(-m // b) * b, -(-n // b) * b
    ragged = (m_pad, n_pad) != (m, n)
    adt = TDT[act]
    x = dev(inp["x"], adt)
    dyt = dev(inp["dy"] if dy is None else dy, adt)
    pm = dev(inp["perm_m"], torch.int32)
    pn = dev(inp["perm_n"], torch.int32)
    qR = dev(inp["q_R"] * (0 if q_zero else 1), torch.float32)
    qP = dev(inp["q_P"] * (0 if q_zero else 1), torch.float32)
    w_scale = None
    if wdt == "i8":
        W32 = dev(inp["W0"], torch.float32)
        Wq = torch.empty(n, m, dtype=torch.int8, device=DEV)
        s = torch.empty(n, device=DEV)
        P.poetx_quantize_rows_int8(W32, Wq, s)
        if ragged:
            Wp = torch.full((n_pad, m_pad), 7, dtype=torch.int8, device=DEV)
            w_scale = torch.full((n_pad,), float("nan"), device=DEV)
            P.poetx_merge_perm_padded(Wq, pn, pm, Wp, s, w_scale)
        else:
            Wp = torch.empty_like(Wq)
            w_scale = torch.empty_like(s)
            P.poetx_merge_perm(Wq, pn, pm, Wp, s, w_scale)
        W_eff = O.dequantize_rows(*O.quantize_rows_int8(inp["W0"]))
        wcode = P.I8
    else:
        W0 = dev(inp["W0"], TDT[wdt])
        if ragged:  # padding filled with NaN first: it must be overwritten with zeros
            Wp = torch.full((n_pad, m_pad), float("nan"), dtype=TDT[wdt], device=DEV)
            P.poetx_merge_perm_padded(W0, pn, pm, Wp)
        else:
            Wp = torch.empty_like(W0)
            P.poetx_merge_perm(W0, pn, pm, Wp)
        W_eff = inp["W0"]
        wcode = P.F32 if wdt == "f32" else P.BF16
    acode = P.F32 if act == "f32" else P.BF16
    vcode = P.FAST if variant == "fast" else P.MEM
    N = x.shape[0]
    L = P.make_layer(m, n, b, acode, wcode, vcode, pm, pn, Wp, qR, qP, w_scale)
    saved = P.workspace(P.poetx_layer_saved_bytes(L, N), DEV)
    wsf = P.workspace(P.poetx_layer_workspace_bytes(L, N, 0), DEV)
    wsb = P.workspace(P.poetx_layer_workspace_bytes(L, N, 1), DEV)
    y = torch.empty(N, n, dtype=adt, device=DEV)
    dx = torch.empty(N, m, dtype=adt, device=DEV)
    if accumulate_init is not None:
        dqR = dev(accumulate_init[0], torch.float32)
        dqP = dev(accumulate_init[1], torch.float32)
    else:
        dqR = torch.full_like(qR, float("nan"))
        dqP = torch.full_like(qP, float("nan"))
    P.poetx_layer_fwd(L, x, y, saved, wsf)
    P.poetx_layer_bwd(L, x, dyt, saved, dx, dqR, dqP, wsb, accumulate=accumulate_init is not None)
    torch.cuda.synchronize()
    assert P.poetx_get_device_error() == 0
    return {"y": host(y), "dx": host(dx), "dq_R": host(dqR), "dq_P": host(dqP), "W_eff": W_eff}


def check(got, ref, tol, keys=("y", "dx", "dq_R", "dq_P")):
    errs = {k: O.rel_fro(got[k], ref[k]) for k in keys}
    assert max(errs.values()) <= tol, errs
    return errs


def oracle_for(inp, got, b, q_zero=False, dy=None):
    s = 0 if q_zero else 1
    return O.poetx_layer(inp["x"], inp["dy"] if dy is None else dy, got["W_eff"], inp["perm_m"],
                         inp["perm_n"], inp["q_R"] * s, inp["q_P"] * s, b)


@pytest.mark.parametrize("variant", ["fast", "mem"])
def test_layer_fp32_256_b32(P, variant):
    wl = inputs.WORKLOADS["fp32_256_b32"]
    inp = inputs.layer_inputs(wl, wl.layers[0])
    got = run_layer(P, inp, wl.b, "f32", "f32", variant)
    check(got, oracle_for(inp, got, wl.b), TOL_F32)


@pytest.mark.parametrize("m,n,b,N", [(256, 512, 64, 200), (512, 256, 128, 77), (512, 512, 256, 130),
                                     (1024, 512, 512, 300),
                                     # fewer W' tiles than SMs, ragged token tail
                                     (2048, 1024, 256, 1000), (1024, 2048, 256, 520)])
@pytest.mark.parametrize("variant", ["fast", "mem"])
def test_layer_bf16_small(P, m, n, b, N, variant):
    inp = inputs.small_layer_inputs(31 + b, m, n, b, N, act="bf16", wdt="bf16")
    got = run_layer(P, inp, b, "bf16", "bf16", variant)
    check(got, oracle_for(inp, got, b), TOL_BF16_LAYER)


def test_layer_int8_small(P):
    inp = inputs.small_layer_inputs(41, 512, 768, 256, 150, act="bf16", wdt="i8")
    got = run_layer(P, inp, 256, "bf16", "i8", "mem")
    check(got, oracle_for(inp, got, 256), TOL_BF16_LAYER)


def test_layer_zero_q_is_plain_linear(P):
    inp = inputs.small_layer_inputs(43, 256, 512, 64, 100, act="bf16", wdt="bf16")
    got = run_layer(P, inp, 64, "bf16", "bf16", "fast", q_zero=True)
    assert O.rel_fro(got["y"], inp["x"] @ inp["W0"].T) <= TOL_BF16_LAYER
    assert O.rel_fro(got["dx"], inp["dy"] @ inp["W0"]) <= TOL_BF16_LAYER


def test_fast_and_mem_bitwise_equal_and_deterministic(P):
    inp = inputs.small_layer_inputs(47, 512, 512, 128, 333, act="bf16", wdt="bf16")
    a = run_layer(P, inp, 128, "bf16", "bf16", "fast")
    b2 = run_layer(P, inp, 128, "bf16", "bf16", "mem")
    c = run_layer(P, inp, 128, "bf16", "bf16", "fast")
    for k in ("y", "dx", "dq_R", "dq_P"):
        np.testing.assert_array_equal(a[k], b2[k], err_msg=k)
        np.testing.assert_array_equal(a[k], c[k], err_msg=k)


def test_layer_accumulate_and_empty(P):
    inp = inputs.small_layer_inputs(53, 256, 256, 64, 0, act="bf16", wdt="bf16")
    init = (np.full(inp["q_R"].shape, 0.5), np.full(inp["q_P"].shape, -1.0))
    got = run_layer(P, inp, 64, "bf16", "bf16", "fast", accumulate_init=init)
    np.testing.assert_array_equal(got["dq_R"], init[0])   # N = 0 adds exact zeros
    np.testing.assert_array_equal(got["dq_P"], init[1])
    inp = inputs.small_layer_inputs(54, 256, 256, 64, 90, act="bf16", wdt="bf16")
    base = run_layer(P, inp, 64, "bf16", "bf16", "fast")
    acc = run_layer(P, inp, 64, "bf16", "bf16", "fast", accumulate_init=init)
    np.testing.assert_allclose(acc["dq_R"], base["dq_R"] + 0.5, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(acc["dq_P"], base["dq_P"] - 1.0, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("variant", ["fast", "mem"])
def test_layer_llama1b_2048_full(P, variant):
    wl = inputs.WORKLOADS["llama1b_2048"]
    inp = inputs.layer_inputs(wl, wl.layers[0])
    got = run_layer(P, inp, wl.b, "bf16", "bf16", variant)
    check(got, oracle_for(inp, got, wl.b), TOL_BF16_LAYER)


@pytest.mark.parametrize("b", [64, 128, 256, 512])
def test_layer_sweep_4096_full(P, b):
    wl = inputs.WORKLOADS[f"sweep_4096_b{b}"]
    inp = inputs.layer_inputs(wl, wl.layers[0])
    got = run_layer(P, inp, b, "bf16", "bf16", "fast")
    check(got, oracle_for(inp, got, b), TOL_BF16_LAYER)


def _masked_full_size(P, wl, layer, variant, n_sample=256, n_rows=48):
    """Full token count in the benchmark's launch configuration, with the upstream gradient
    zero outside a random token subset S: then dq (a sum over tokens) equals the oracle's
    dq over S alone, and y / dx are checked on sampled rows (both are row-independent)."""
    inp = inputs.layer_inputs(wl, layer)
    N = inp["x"].shape[0]
    r = np.random.default_rng(layer.m * 7 + layer.n)
    S = np.sort(r.choice(N, n_sample, replace=False))
    dy = np.zeros_like(inp["dy"])
    dy[S] = inp["dy"][S]
    got = run_layer(P, inp, wl.b, "bf16", wl.wdt, variant, dy=dy)
    sub = {k: inp[k] for k in inp}
    sub["x"], sub["dy"] = inp["x"][S], inp["dy"][S]
    ref = O.poetx_layer(sub["x"], sub["dy"], got["W_eff"], inp["perm_m"], inp["perm_n"],
                        inp["q_R"], inp["q_P"], wl.b)
    rows = np.sort(r.choice(N, n_rows, replace=False))
    y_ref = O.layer_forward_rows(inp["x"][rows], ref["Wp"], inp["perm_m"], inp["perm_n"],
                                 ref["G_R"], ref["G_P"])
    errs = {"y": O.rel_fro(got["y"][rows], y_ref),
            "dx": O.rel_fro(got["dx"][S], ref["dx"]),
            "dq_R": O.rel_fro(got["dq_R"], ref["dq_R"]),
            "dq_P": O.rel_fro(got["dq_P"], ref["dq_P"])}
    outside = np.setdiff1d(np.arange(N), S)[:64]
    assert not np.any(got["dx"][outside]), "dx must vanish where dy does"
    assert max(errs.values()) <= TOL_BF16_LAYER, errs


@pytest.mark.parametrize("layer", ["q", "gate", "down"])
def test_layer_llama8b_block_full_size(P, layer):
    wl = inputs.WORKLOADS["llama8b_block"]
    L = [l for l in wl.layers if l.name == layer][0]
    _masked_full_size(P, wl, L, "fast")


@pytest.mark.parametrize("layer", ["up", "down"])
def test_layer_llama13b_mlp_int8_full_size(P, layer):
    wl = inputs.WORKLOADS["llama13b_mlp_int8"]
    L = [l for l in wl.layers if l.name == layer][0]
    _masked_full_size(P, wl, L, "mem")


def test_layer_bf16_split_tiles_deterministic(P):
    """Every reduction of the chain (split-K weight gradients, CNP partial sums) adds in a
    fixed order, so two runs give bit-identical outputs and gradients."""
    inp = inputs.small_layer_inputs(77, 2048, 1024, 256, 1000, act="bf16", wdt="bf16")
    a = run_layer(P, inp, 256, "bf16", "bf16", "mem")
    b = run_layer(P, inp, 256, "bf16", "bf16", "mem")
    for k in ("y", "dx", "dq_R", "dq_P"):
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("m,n,b,N", [(512, 256, 128, 77), (256, 512, 64, 200),
                                     (2048, 1024, 256, 1000)])
@pytest.mark.parametrize("variant", ["fast", "mem"])
def test_layer_fused_and_separate_products_agree(P, m, n, b, N, variant):
    """Every fusion mask (the W' contraction with the block-diagonal product after it as one
    kernel, bit 0; each backward block product with its weight gradient as one kernel, bit 1)
    matches the oracle, and the separate kernels to within accumulation-order differences."""
    inp = inputs.small_layer_inputs(61 + b, m, n, b, N, act="bf16", wdt="bf16")
    got = {}
    try:
        for mask in (0, 1, 2, 3):
            P.poetx_set_fusion(mask)
            got[mask] = run_layer(P, inp, b, "bf16", "bf16", variant)
    finally:
        P.poetx_set_fusion(True)
    ref = oracle_for(inp, got[3], b)
    for mask, r in got.items():
        check(r, ref, TOL_BF16_LAYER)
        for k in ("y", "dx", "dq_R", "dq_P"):
            assert O.rel_fro(r[k], got[0][k]) <= 1e-2, (mask, k)


def _random_shapes(count, seed=2026):
    r = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        b = int(r.choice([64, 128, 256, 512]))
        m = b * int(r.integers(1, 9))
        n = b * int(r.integers(1, 9))
        if max(m, n) > 2048:
            continue
        N = int(r.integers(1, 1500))
        out.append((m, n, b, N, str(r.choice(["fast", "mem"]))))
    return out


@pytest.mark.parametrize("m,n,b,N,variant", _random_shapes(12))
def test_layer_bf16_random_shapes(P, m, n, b, N, variant):
    """Seeded random layer shapes (block sizes 64-512, widths that may or may not fill a
    256-wide W' tile, ragged token counts): whichever kernels the shape selects (fused or
    separate products, tensor-core or CUDA-core contraction) must match the oracle."""
    inp = inputs.small_layer_inputs(1000 + m + n + N, m, n, b, N, act="bf16", wdt="bf16")
    got = run_layer(P, inp, b, "bf16", "bf16", variant)
    check(got, oracle_for(inp, got, b), TOL_BF16_LAYER)


def _step_host(P, inp, b, act, wdt, variant, pinned=True):
    """poetx_layer_step_host with host tensors; the layer descriptor is built as run_layer
    builds it (same weights, permutations and q)."""
    m, n = inp["W0"].shape[1], inp["W0"].shape[0]
    m_pad, n_pad = -(-m // b) * b, -(-n // b) * b
    adt = TDT[act]
    pm = dev(inp["perm_m"], torch.int32)
    pn = dev(inp["perm_n"], torch.int32)
    qR = dev(inp["q_R"], torch.float32)
    qP = dev(inp["q_P"], torch.float32)
    w_scale = None
    if wdt == "i8":
        Wq = torch.empty(n, m, dtype=torch.int8, device=DEV)
        s = torch.empty(n, device=DEV)
        P.poetx_quantize_rows_int8(dev(inp["W0"], torch.float32), Wq, s)
        Wp = torch.empty(n_pad, m_pad, dtype=torch.int8, device=DEV)
        w_scale = torch.empty(n_pad, device=DEV)
        P.poetx_merge_perm_padded(Wq, pn, pm, Wp, s, w_scale)
        wcode = P.I8
    else:
        W0 = dev(inp["W0"], TDT[wdt])
        Wp = torch.empty(n_pad, m_pad, dtype=W0.dtype, device=DEV)
        P.poetx_merge_perm_padded(W0, pn, pm, Wp)
        wcode = P.F32 if wdt == "f32" else P.BF16
    acode = P.F32 if act == "f32" else P.BF16
    L = P.make_layer(m, n, b, acode, wcode, P.FAST if variant == "fast" else P.MEM, pm, pn, Wp,
                     qR, qP, w_scale)
    N = inp["x"].shape[0]
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    hx = pin(torch.tensor(np.asarray(inp["x"]), dtype=adt))    # the same rounding as dev()
    hdy = pin(torch.tensor(np.asarray(inp["dy"]), dtype=adt))
    hy = pin(torch.full((N, n), float("nan"), dtype=adt))
    hdx = pin(torch.full((N, m), float("nan"), dtype=adt))
    hqR = pin(torch.full(tuple(qR.shape), float("nan")))
    hqP = pin(torch.full(tuple(qP.shape), float("nan")))
    devbuf = P.workspace(P.poetx_layer_step_host_bytes(L, N), DEV)
    s = torch.cuda.current_stream()
    P.poetx_layer_step_host(L, hx, hdy, hy, hdx, hqR, hqP, devbuf)
    s.synchronize()
    assert P.poetx_get_device_error() == 0
    f = lambda t: t.float().numpy().astype(np.float64)
    return {"y": f(hy), "dx": f(hdx), "dq_R": f(hqR), "dq_P": f(hqP)}


@pytest.mark.parametrize("act,wdt,variant,shape", [
    ("bf16", "bf16", "fast", (2048, 2048, 256, 1000)),
    ("bf16", "bf16", "mem", (512, 1024, 128, 333)),
    ("bf16", "i8", "mem", (512, 768, 256, 150)),
    ("f32", "f32", "fast", (256, 256, 32, 64)),
])
def test_step_host_equals_device_calls(P, act, wdt, variant, shape):
    """The host-buffer step runs the same kernels as poetx_layer_fwd + poetx_layer_bwd on
    device buffers: bit-identical outputs, and within the layer tolerance of the oracle."""
    m, n, b, N = shape
    inp = inputs.small_layer_inputs(61 + b, m, n, b, N, act=act, wdt=wdt)
    got = _step_host(P, inp, b, act, wdt, variant)
    ref_dev = run_layer(P, inp, b, act, wdt, variant)
    for k in ("y", "dx", "dq_R", "dq_P"):
        np.testing.assert_array_equal(got[k], ref_dev[k], err_msg=k)
    got["W_eff"] = ref_dev["W_eff"]
    check(got, oracle_for(inp, got, b), TOL_F32 if act == "f32" else TOL_BF16_LAYER)


def test_step_host_pageable_and_repeated(P):
    """Pageable host buffers give the same result (without overlap), and repeated calls
    reuse the copy stream and events."""
    inp = inputs.small_layer_inputs(71, 512, 512, 128, 200, act="bf16", wdt="bf16")
    a = _step_host(P, inp, 128, "bf16", "bf16", "fast", pinned=True)
    b2 = _step_host(P, inp, 128, "bf16", "bf16", "fast", pinned=False)
    c = _step_host(P, inp, 128, "bf16", "bf16", "fast", pinned=True)
    for k in ("y", "dx", "dq_R", "dq_P"):
        np.testing.assert_array_equal(a[k], b2[k], err_msg=k)
        np.testing.assert_array_equal(a[k], c[k], err_msg=k)


@pytest.mark.parametrize("act,wdt,variant,shape", [
    ("bf16", "bf16", "fast", (2048, 2048, 256, 1000)),
    ("bf16", "bf16", "mem", (1024, 512, 128, 333)),
    ("bf16", "i8", "mem", (512, 768, 256, 150)),
    ("f32", "f32", "fast", (256, 256, 32, 64)),
])
def test_overlap_on_and_off_bitwise_equal(P, act, wdt, variant, shape):
    """The dx scatter on the side stream (beside the CNP backward) gives the same bits as
    the serial order."""
    m, n, b, N = shape
    inp = inputs.small_layer_inputs(83 + b, m, n, b, N, act=act, wdt=wdt)
    try:
        P.poetx_set_overlap(False)
        off = run_layer(P, inp, b, act, wdt, variant)
    finally:
        P.poetx_set_overlap(True)
    on = run_layer(P, inp, b, act, wdt, variant)
    for k in ("y", "dx", "dq_R", "dq_P"):
        np.testing.assert_array_equal(on[k], off[k], err_msg=k)


def test_overlapped_step_in_a_cuda_graph(P):
    """Forward + backward with the side-stream fork and join captured into a CUDA graph and
    replayed: the same bits as the eager calls."""
    m, n, b, N = 2048, 2048, 256, 777
    inp = inputs.small_layer_inputs(89, m, n, b, N, act="bf16", wdt="bf16")
    ref = run_layer(P, inp, b, "bf16", "bf16", "fast")
    x = dev(inp["x"], torch.bfloat16)
    dyt = dev(inp["dy"], torch.bfloat16)
    pm = dev(inp["perm_m"], torch.int32)
    pn = dev(inp["perm_n"], torch.int32)
    qR = dev(inp["q_R"], torch.float32)
    qP = dev(inp["q_P"], torch.float32)
    W0 = dev(inp["W0"], torch.bfloat16)
    Wp = torch.empty_like(W0)
    P.poetx_merge_perm(W0, pn, pm, Wp)
    L = P.make_layer(m, n, b, P.BF16, P.BF16, P.FAST, pm, pn, Wp, qR, qP, None)
    saved = P.workspace(P.poetx_layer_saved_bytes(L, N), DEV)
    wsf = P.workspace(P.poetx_layer_workspace_bytes(L, N, 0), DEV)
    wsb = P.workspace(P.poetx_layer_workspace_bytes(L, N, 1), DEV)
    y = torch.empty(N, n, dtype=torch.bfloat16, device=DEV)
    dx = torch.empty(N, m, dtype=torch.bfloat16, device=DEV)
    dqR = torch.empty_like(qR)
    dqP = torch.empty_like(qP)

    def step():
        P.poetx_layer_fwd(L, x, y, saved, wsf)
        P.poetx_layer_bwd(L, x, dyt, saved, dx, dqR, dqP, wsb)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (y, dx, dqR, dqP):
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert P.poetx_get_device_error() == 0
    got = {"y": host(y), "dx": host(dx), "dq_R": host(dqR), "dq_P": host(dqP)}
    for k in got:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)


@pytest.mark.parametrize("act,wdt,variant,shape", [
    ("bf16", "bf16", "fast", (200, 328, 64, 150)),     # last blocks of 8 on both sides
    ("bf16", "bf16", "mem", (200, 328, 64, 150)),
    ("bf16", "bf16", "fast", (2000, 1000, 256, 300)),  # last blocks of 208 and 232
    ("bf16", "bf16", "mem", (1016, 2040, 128, 260)),   # 120 and 120
    ("bf16", "bf16", "fast", (512, 776, 256, 77)),     # m whole, n ragged (8)
    ("bf16", "i8", "mem", (528, 776, 256, 150)),       # int8 rows: m % 16 == 0
    ("f32", "f32", "fast", (200, 136, 32, 64)),        # fp32: last blocks of 8
    ("f32", "f32", "mem", (104, 96, 64, 33)),
])
def test_layer_ragged_last_block(P, act, wdt, variant, shape):
    """ceil(d/b) blocks with a ragged last one (padded inside the layer) against the oracle
    written per block with its own size; the non-parameter entries of dq are exactly 0."""
    m, n, b, N = shape
    inp = inputs.small_layer_inputs(97 + b + m % 97, m, n, b, N, act=act, wdt=wdt)
    got = run_layer(P, inp, b, act, wdt, variant)
    ref = O.poetx_layer_ragged(inp["x"], inp["dy"], got["W_eff"], inp["perm_m"], inp["perm_n"],
                               inp["q_R"], inp["q_P"], b)
    check(got, ref, TOL_F32 if act == "f32" else TOL_BF16_LAYER)
    for key, d in (("dq_R", m), ("dq_P", n)):
        r = d - (-(-d // b) - 1) * b
        if r < b:
            last = got[key][-1]
            mask = np.zeros(b * (b - 1) // 2, dtype=bool)
            k = 0
            for i in range(b):
                for j in range(i + 1, b):
                    mask[k] = j >= r
                    k += 1
            assert np.all(last[mask] == 0), key


def test_layer_ragged_fast_mem_equal_and_step_host(P):
    """fast and mem bit-identical on a ragged layer, and the host-buffer step too."""
    m, n, b, N = 1016, 520, 128, 200
    inp = inputs.small_layer_inputs(101, m, n, b, N, act="bf16", wdt="bf16")
    a = run_layer(P, inp, b, "bf16", "bf16", "fast")
    c = run_layer(P, inp, b, "bf16", "bf16", "mem")
    h = _step_host(P, inp, b, "bf16", "bf16", "fast")
    for k in ("y", "dx", "dq_R", "dq_P"):
        np.testing.assert_array_equal(a[k], c[k], err_msg=k)
        np.testing.assert_array_equal(a[k], h[k], err_msg=k)


@pytest.mark.parametrize("m,n,b,wdt,variant", [(640, 384, 128, "bf16", "fast"),
                                               (384, 640, 64, "bf16", "mem"),
                                               (384, 320, 64, "i8", "mem")])
def test_layer_widths_off_the_256_grid_take_tensor_cores(P, m, n, b, wdt, variant):
    """Widths that are multiples of 64 but not of 256 (the W' tile): the contraction still
    runs on the tensor cores (its last tile column is partly outside the output), which the
    engine query reports, and the layer matches the oracle; with the CUDA-core engine the
    query reports every product there and the result matches too."""
    N = 300
    inp = inputs.small_layer_inputs(880 + m + n, m, n, b, N, act="bf16", wdt=wdt)
    fake = __import__("ctypes").c_void_p(4096)
    desc = P.LayerDesc(m, n, b, 3, P.BF16, P.I8 if wdt == "i8" else P.BF16,
                       P.FAST if variant == "fast" else P.MEM, fake, fake, fake,
                       fake if wdt == "i8" else None, fake, fake)
    assert P.poetx_layer_cuda_core_steps(desc, N) == 0
    got = run_layer(P, inp, b, "bf16", wdt, variant)
    check(got, oracle_for(inp, got, b), TOL_BF16_LAYER)
    try:
        P.poetx_set_gemm_engine(1)
        assert P.poetx_layer_cuda_core_steps(desc, N) == 7
        cc = run_layer(P, inp, b, "bf16", wdt, variant)
    finally:
        P.poetx_set_gemm_engine(0)
    check(cc, oracle_for(inp, cc, b), TOL_BF16_LAYER)


def test_layer_pair_tiles_with_partial_tile_columns(P):
    """Enough tokens for the 2-CTA pair contraction, with widths (4160 = 65 x 64, 4224 = 66 x
    64) whose last 256-wide tile column is partly outside the output, at b = 64; checked on
    sampled tokens as the full-size cases are."""
    wl = inputs.Workload("pairs_partial", (inputs.LayerShape("lin", 4160, 4224),), 64, 4096,
                         "bf16", "bf16", 0.02, ("fast",), 4242)
    _masked_full_size(P, wl, wl.layers[0], "fast")
