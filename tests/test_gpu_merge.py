"""Merge-then-reinitialize on the GPU (POET skill page, Step 4): the weight written back by
poetx_merge_reinit against the fp64 oracle (fp32 arithmetic: 1e-5), and the whole
reinitialisation (merge, q = 0, new permutations, re-merge) leaving the layer's output
unchanged."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import DEV, P, TOL_BF16_LAYER, TOL_F32, dev, host  # noqa: F401
from orthogonal_reparameterized_gb300 import inputs

pytestmark = pytest.mark.gpu

TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _layer_on_gpu(P, inp, b, act, wdt, variant="fast"):
    m, n = inp["W0"].shape[1], inp["W0"].shape[0]
    m_pad, n_pad = -(-m // b) * b, -(-n // b) * b
    keep = {}
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
        W_eff = O.dequantize_rows(*O.quantize_rows_int8(inp["W0"]))
        wcode = P.I8
    else:
        W0 = dev(inp["W0"], TDT[wdt])
        Wp = torch.empty(n_pad, m_pad, dtype=W0.dtype, device=DEV)
        P.poetx_merge_perm_padded(W0, pn, pm, Wp)
        W_eff = inp["W0"]
        wcode = P.F32 if wdt == "f32" else P.BF16
    acode = P.F32 if act == "f32" else P.BF16
    L = P.make_layer(m, n, b, acode, wcode, P.FAST if variant == "fast" else P.MEM, pm, pn, Wp,
                     qR, qP, w_scale)
    keep.update(pm=pm, pn=pn, qR=qR, qP=qP, Wp=Wp, w_scale=w_scale)
    return L, keep, W_eff


def _merge(P, L, n, m):
    W0n = torch.empty(n, m, device=DEV)
    ws = P.workspace(P.poetx_merge_reinit_workspace_bytes(L), DEV)
    P.poetx_merge_reinit(L, W0n, ws)
    torch.cuda.synchronize()
    assert P.poetx_get_device_error() == 0
    return W0n


@pytest.mark.parametrize("m,n,b,act,wdt", [
    (256, 256, 32, "f32", "f32"),        # the fp32 single-layer shape
    (512, 256, 64, "bf16", "bf16"),
    (1024, 512, 256, "bf16", "bf16"),
    (512, 768, 128, "bf16", "i8"),       # int8 W': the dequantised weight is merged
    (2048, 2048, 256, "bf16", "bf16"),   # the Llama-1B-shaped layer
    (1024, 1536, 512, "bf16", "bf16"),   # b = 512
])
def test_merge_reinit_matches_oracle(P, m, n, b, act, wdt):
    inp = inputs.small_layer_inputs(500 + m + b, m, n, b, 4, act=act, wdt=wdt)
    variant = "mem" if wdt == "i8" else "fast"
    L, keep, W_eff = _layer_on_gpu(P, inp, b, act, wdt, variant)
    got = host(_merge(P, L, n, m))
    Wp_ref = O.merge_perm(W_eff, inp["perm_n"], inp["perm_m"])
    ref = O.merge_reinit(Wp_ref, inp["perm_m"], inp["perm_n"], inp["q_R"], inp["q_P"], b)
    assert O.rel_fro(got, ref) <= TOL_F32


def test_merge_reinit_zero_q_returns_w0_exactly(P):
    """q = 0: every G is the identity, the products are exact and the write-back is W0."""
    m, n, b = 512, 256, 64
    inp = inputs.small_layer_inputs(77, m, n, b, 4, act="bf16", wdt="bf16")
    inp["q_R"] = 0 * inp["q_R"]
    inp["q_P"] = 0 * inp["q_P"]
    L, keep, W_eff = _layer_on_gpu(P, inp, b, "bf16", "bf16")
    got = host(_merge(P, L, n, m))
    assert np.array_equal(got, W_eff)


def test_reinitialised_layer_computes_the_same_outputs(P):
    """Merge, then q = 0, freshly drawn permutations and a new merged weight: the layer's
    forward output is the one before (bf16 layer tolerance)."""
    m, n, b, N = 1024, 512, 128, 300
    inp = inputs.small_layer_inputs(91, m, n, b, N, act="bf16", wdt="bf16")
    L, keep, _ = _layer_on_gpu(P, inp, b, "bf16", "bf16")
    x = dev(inp["x"], torch.bfloat16)

    def fwd(Ld):
        saved = P.workspace(P.poetx_layer_saved_bytes(Ld, N), DEV)
        ws = P.workspace(P.poetx_layer_workspace_bytes(Ld, N, 0), DEV)
        y = torch.empty(N, n, dtype=torch.bfloat16, device=DEV)
        P.poetx_layer_fwd(Ld, x, y, saved, ws)
        torch.cuda.synchronize()
        return host(y)

    y_before = fwd(L)
    W0n = _merge(P, L, n, m).to(torch.bfloat16)
    r = np.random.default_rng(5)
    pm2 = dev(r.permutation(m), torch.int32)
    pn2 = dev(r.permutation(n), torch.int32)
    Wp2 = torch.empty_like(W0n)
    P.poetx_merge_perm(W0n, pn2, pm2, Wp2)
    qR0 = torch.zeros_like(keep["qR"])
    qP0 = torch.zeros_like(keep["qP"])
    L2 = P.make_layer(m, n, b, P.BF16, P.BF16, P.FAST, pm2, pn2, Wp2, qR0, qP0, None)
    y_after = fwd(L2)
    ref = O.layer_forward(inp["x"], O.merge_perm(inp["W0"], inp["perm_n"], inp["perm_m"]),
                          inp["perm_m"], inp["perm_n"], O.cnp_forward(inp["q_R"], b),
                          O.cnp_forward(inp["q_P"], b))["y"]
    assert O.rel_fro(y_before, ref) <= TOL_BF16_LAYER
    assert O.rel_fro(y_after, ref) <= TOL_BF16_LAYER
    assert O.rel_fro(y_after, y_before) <= TOL_BF16_LAYER


def test_merge_reinit_argument_errors(P):
    m, n, b = 512, 256, 64
    inp = inputs.small_layer_inputs(3, m, n, b, 4, act="bf16", wdt="bf16")
    L, keep, _ = _layer_on_gpu(P, inp, b, "bf16", "bf16")
    lib = P.lib()
    import ctypes
    W0n = torch.empty(n, m, device=DEV)
    need = P.poetx_merge_reinit_workspace_bytes(L)
    ws = P.workspace(need, DEV)
    assert lib.poetx_merge_reinit(ctypes.byref(L), ctypes.c_void_p(W0n.data_ptr()),
                                  ctypes.c_void_p(ws.data_ptr()), need - 1, None) == 5
    assert lib.poetx_merge_reinit(ctypes.byref(L), None, ctypes.c_void_p(ws.data_ptr()), need,
                                  None) == 1


@pytest.mark.parametrize("m,n,b,act,wdt", [
    (200, 136, 64, "bf16", "bf16"),     # last blocks of 8 on both sides
    (1016, 520, 128, "bf16", "bf16"),
    (528, 776, 256, "bf16", "i8"),      # int8 rows: m % 16 == 0
    (104, 96, 32, "f32", "f32"),
])
def test_merge_reinit_ragged_matches_oracle(P, m, n, b, act, wdt):
    """Ragged last blocks: W0_new is the ragged layer's map (its response to the identity,
    the oracle written per block with its own size)."""
    inp = inputs.small_layer_inputs(700 + m + b, m, n, b, 4, act=act, wdt=wdt)
    variant = "mem" if wdt == "i8" else "fast"
    L, keep, W_eff = _layer_on_gpu(P, inp, b, act, wdt, variant)
    got = host(_merge(P, L, n, m))
    ref = O.poetx_layer_ragged(np.eye(m), np.zeros((m, n)), W_eff, inp["perm_m"],
                               inp["perm_n"], inp["q_R"], inp["q_P"], b)["y"].T
    assert O.rel_fro(got, ref) <= TOL_F32
