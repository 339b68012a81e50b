"""Thin Python binding of the POET-X C ABI (``include/poetx.h``).

Argument marshalling only: every function forwards torch tensors' device pointers, sizes
and the current CUDA stream to the function of the same name in ``libpoetx.so`` and raises
``PoetxError`` on a non-OK status.  No computation happens here, and there is no fallback:
if the library is missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpoetx.so")

F32, BF16, I8 = 0, 1, 2
FAST, MEM = 0, 1
_DT = {torch.float32: F32, torch.bfloat16: BF16, torch.int8: I8}
_TORCH_DT = {F32: torch.float32, BF16: torch.bfloat16, I8: torch.int8}

_vp, _i, _sz, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float


class PoetxError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg}")
        self.status = status


class LayerDesc(ctypes.Structure):
    """Mirror of ``poetx_layer``."""
    _fields_ = [("m", _i), ("n", _i), ("b", _i), ("order", _i), ("act", _i), ("wdt", _i),
                ("variant", _i), ("perm_m", _vp), ("perm_n", _vp), ("Wp", _vp),
                ("w_scale", _vp), ("q_R", _vp), ("q_P", _vp)]


class AdamDesc(ctypes.Structure):
    """Mirror of ``poetx_adam``."""
    _fields_ = [("lr", _f), ("beta1", _f), ("beta2", _f), ("eps", _f), ("weight_decay", _f),
                ("step", _i)]


_SIGS = {
    "poetx_status_str": (ctypes.c_char_p, [_i]),
    "poetx_get_device_error": (_i, [_vp]),
    "poetx_selftest_timeout": (_i, [ctypes.c_uint, _vp]),
    "poetx_set_gemm_engine": (_i, [_i]),
    "poetx_set_fusion": (_i, [_i]),
    "poetx_set_overlap": (_i, [_i]),
    "poetx_launch_count": (ctypes.c_ulonglong, []),
    "poetx_timeout_site": (_i, []),
    "poetx_profile_enable": (_i, [_i]),
    "poetx_set_trace_buffer": (_i, [_vp, _sz]),
    "poetx_profile_collect": (_i, [ctypes.POINTER(_i), ctypes.POINTER(_f), _i]),
    "poetx_stage_name": (ctypes.c_char_p, [_i]),
    "poetx_cnp_workspace_bytes": (_sz, [_i, _i, _i]),
    "poetx_cnp_fwd": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "poetx_cnp_bwd": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _i, _vp, _sz, _vp]),
    "poetx_cnp_fwd_noalloc": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "poetx_triu_unpack": (_i, [_vp, _i, _i, _vp, _vp]),
    "poetx_triu_grad_pack": (_i, [_vp, _i, _i, _vp, _i, _vp]),
    "poetx_perm_gather": (_i, [_i, _vp, _i, _i, _vp, _vp, _vp]),
    "poetx_perm_scatter": (_i, [_i, _vp, _i, _i, _vp, _vp, _vp]),
    "poetx_merge_perm": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "poetx_merge_perm_padded": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "poetx_quantize_rows_int8": (_i, [_vp, _i, _i, _vp, _vp, _vp]),
    "poetx_blockdiag_mm": (_i, [_i, _vp, _i, _i, _i, _vp, _i, _vp, _vp, _vp, _vp]),
    "poetx_blockdiag_wgrad": (_i, [_i, _vp, _vp, _i, _i, _i, _i, _vp, _vp]),
    "poetx_wprime_gemm": (_i, [_i, _i, _vp, _i, _i, _i, _vp, _vp, _i, _vp, _vp]),
    "poetx_layer_workspace_bytes": (_sz, [ctypes.POINTER(LayerDesc), _i, _i]),
    "poetx_layer_saved_bytes": (_sz, [ctypes.POINTER(LayerDesc), _i]),
    "poetx_layer_cuda_core_steps": (_i, [ctypes.POINTER(LayerDesc), _i]),
    "poetx_layer_fwd": (_i, [ctypes.POINTER(LayerDesc), _vp, _i, _vp, _vp, _vp, _sz, _vp]),
    "poetx_layer_bwd": (_i, [ctypes.POINTER(LayerDesc), _vp, _vp, _i, _vp, _vp, _vp, _vp, _i,
                             _vp, _sz, _vp]),
    "poetx_layer_step_host_bytes": (_sz, [ctypes.POINTER(LayerDesc), _i]),
    "poetx_layer_step_host": (_i, [ctypes.POINTER(LayerDesc), _vp, _vp, _i, _vp, _vp, _vp, _vp,
                                   _vp, _sz, _vp]),
    "poetx_merge_reinit_workspace_bytes": (_sz, [ctypes.POINTER(LayerDesc)]),
    "poetx_merge_reinit": (_i, [ctypes.POINTER(LayerDesc), _vp, _vp, _sz, _vp]),
    "poetx_adam_triu": (_i, [_vp, _vp, _vp, _vp, ctypes.c_longlong, ctypes.POINTER(AdamDesc),
                             _vp]),
    "poetx_layer_bwd_adam": (_i, [ctypes.POINTER(LayerDesc), _vp, _vp, _i, _vp, _vp, _vp, _vp,
                                  _i, ctypes.POINTER(AdamDesc), _vp, _vp, _vp, _vp, _vp, _sz,
                                  _vp]),
    "poetx_group_saved_bytes": (_sz, [ctypes.POINTER(LayerDesc), _i, _i]),
    "poetx_group_workspace_bytes": (_sz, [ctypes.POINTER(LayerDesc), _i, _i]),
    "poetx_group_cnp_fwd": (_i, [ctypes.POINTER(LayerDesc), _i, _i, _vp, _vp]),
    "poetx_group_layer_fwd": (_i, [ctypes.POINTER(LayerDesc), _i, _i, _vp, _i, _vp, _vp, _vp, _sz,
                                   _vp]),
    "poetx_group_layer_bwd": (_i, [ctypes.POINTER(LayerDesc), _i, _i, _vp, _vp, _i, _vp, _vp, _vp,
                                   _sz, _vp]),
    "poetx_group_cnp_bwd": (_i, [ctypes.POINTER(LayerDesc), _i, _i, _vp,
                                 ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p),
                                 _i, _vp, _sz, _vp]),
    "poetx_group_step_host_bytes": (_sz, [ctypes.POINTER(LayerDesc), _i, _i]),
    "poetx_group_step_host": (_i, [ctypes.POINTER(LayerDesc), _i] +
                              [ctypes.POINTER(ctypes.c_void_p)] * 2 + [_i] +
                              [ctypes.POINTER(ctypes.c_void_p)] * 4 + [_vp, _sz, _vp]),
}

_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load ``libpoetx.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("poetx: tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("poetx: tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, st: int):
    if st != 0:
        raise PoetxError(fn, st, lib().poetx_status_str(st).decode())


def status_str(st: int) -> str:
    return lib().poetx_status_str(st).decode()


def poetx_get_device_error(stream=None) -> int:
    return lib().poetx_get_device_error(_stream(stream))


def poetx_selftest_timeout(timeout_us: int, stream=None):
    _check("poetx_selftest_timeout", lib().poetx_selftest_timeout(timeout_us, _stream(stream)))


def poetx_set_gemm_engine(engine: int):
    _check("poetx_set_gemm_engine", lib().poetx_set_gemm_engine(engine))


def poetx_set_fusion(on):
    """True / False: every fused kernel on / off; an int: the library's bit mask (bit 0 the
    W' contraction with the block product after it, bit 1 the backward block product with
    its weight gradient)."""
    mask = (3 if on else 0) if isinstance(on, bool) else int(on)
    _check("poetx_set_fusion", lib().poetx_set_fusion(mask))


def poetx_set_overlap(on: bool):
    _check("poetx_set_overlap", lib().poetx_set_overlap(1 if on else 0))


def poetx_launch_count() -> int:
    return lib().poetx_launch_count()


def poetx_profile_enable(on: bool):
    _check("poetx_profile_enable", lib().poetx_profile_enable(int(bool(on))))


def poetx_set_trace_buffer(buf=None):
    _check("poetx_set_trace_buffer",
           lib().poetx_set_trace_buffer(_p(buf), 0 if buf is None else buf.numel() * buf.element_size()))


def poetx_profile_collect(cap: int = 4096):
    """[(stage name, milliseconds)] for every launch timed since the last collect."""
    st = (_i * cap)()
    ms = (_f * cap)()
    n = lib().poetx_profile_collect(st, ms, cap)
    return [(lib().poetx_stage_name(st[k]).decode(), float(ms[k])) for k in range(n)]


def dtype_code(t: torch.Tensor) -> int:
    return _DT[t.dtype]


# ---------------------------------------------------------------- CNP
def poetx_cnp_workspace_bytes(nblk: int, b: int, phase: int) -> int:
    return lib().poetx_cnp_workspace_bytes(nblk, b, phase)


def workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def poetx_cnp_fwd(q, b, G_f32=None, G_bf16=None, Gt_bf16=None, ws=None, order=3, stream=None):
    nblk = q.shape[0]
    if ws is None:
        ws = workspace(poetx_cnp_workspace_bytes(nblk, b, 0), q.device)
    _check("poetx_cnp_fwd", lib().poetx_cnp_fwd(_p(q), nblk, b, order, _p(G_f32), _p(G_bf16),
                                                _p(Gt_bf16), _p(ws), ws.numel(),
                                                _stream(stream)))


CNP_NOALLOC_MAX_ELEMS = 2 * 1024 * 1024


def poetx_cnp_fwd_noalloc(q, b, G_f32=None, G_bf16=None, Gt_bf16=None, order=3, stream=None):
    """poetx_cnp_fwd without a workspace: its scratch is a fixed array inside the library
    (for callers that cannot allocate device memory; see include/poetx.h)."""
    _check("poetx_cnp_fwd_noalloc", lib().poetx_cnp_fwd_noalloc(_p(q), q.shape[0], b, order,
                                                                _p(G_f32), _p(G_bf16),
                                                                _p(Gt_bf16), _stream(stream)))


def poetx_cnp_bwd(q, dG, b, dq, accumulate=False, ws=None, order=3, stream=None):
    nblk = q.shape[0]
    splits = dG.shape[0] if dG.dim() == 4 else 1
    if ws is None:
        ws = workspace(poetx_cnp_workspace_bytes(nblk, b, 1), q.device)
    _check("poetx_cnp_bwd", lib().poetx_cnp_bwd(_p(q), _p(dG), splits, nblk, b, order, _p(dq),
                                                int(bool(accumulate)), _p(ws), ws.numel(),
                                                _stream(stream)))


def poetx_triu_unpack(q, b, Q, stream=None):
    _check("poetx_triu_unpack", lib().poetx_triu_unpack(_p(q), q.shape[0], b, _p(Q),
                                                        _stream(stream)))


def poetx_triu_grad_pack(Qbar, dq, accumulate=False, stream=None):
    nblk, b, _ = Qbar.shape
    _check("poetx_triu_grad_pack", lib().poetx_triu_grad_pack(_p(Qbar), nblk, b, _p(dq),
                                                              int(bool(accumulate)),
                                                              _stream(stream)))


# ---------------------------------------------------------------- permutations
def poetx_perm_gather(X, perm, Y, stream=None):
    N, D = X.shape
    _check("poetx_perm_gather", lib().poetx_perm_gather(dtype_code(X), _p(X), N, D, _p(perm),
                                                        _p(Y), _stream(stream)))


def poetx_perm_scatter(X, perm, Y, stream=None):
    N, D = X.shape
    _check("poetx_perm_scatter", lib().poetx_perm_scatter(dtype_code(X), _p(X), N, D, _p(perm),
                                                          _p(Y), _stream(stream)))


def poetx_merge_perm(W0, perm_n, perm_m, Wp, scale=None, scale_p=None, stream=None):
    n, m = W0.shape
    _check("poetx_merge_perm", lib().poetx_merge_perm(_p(W0), _p(scale), dtype_code(W0), n, m,
                                                      _p(perm_n), _p(perm_m), _p(Wp), _p(scale_p),
                                                      _stream(stream)))


def poetx_merge_perm_padded(W0, perm_n, perm_m, Wp, scale=None, scale_p=None, stream=None):
    """Wp [n_pad, m_pad] (its shape gives the padding) <- the merge of W0 [n, m], zero
    elsewhere; scale_p [n_pad] likewise for int8."""
    n, m = W0.shape
    n_pad, m_pad = Wp.shape
    _check("poetx_merge_perm_padded", lib().poetx_merge_perm_padded(
        _p(W0), _p(scale), dtype_code(W0), n, m, n_pad, m_pad, _p(perm_n), _p(perm_m), _p(Wp),
        _p(scale_p), _stream(stream)))


def poetx_quantize_rows_int8(W, Wq, scale, stream=None):
    n, m = W.shape
    _check("poetx_quantize_rows_int8", lib().poetx_quantize_rows_int8(_p(W), n, m, _p(Wq),
                                                                      _p(scale), _stream(stream)))


# ---------------------------------------------------------------- products
def poetx_blockdiag_mm(X, G, Y, trans=False, col_scale=None, out_perm=None, stream=None):
    N = X.shape[0]
    nblk, b, _ = G.shape
    _check("poetx_blockdiag_mm", lib().poetx_blockdiag_mm(dtype_code(X), _p(X), N, nblk, b, _p(G),
                                                          int(bool(trans)), _p(col_scale),
                                                          _p(out_perm), _p(Y), _stream(stream)))


def poetx_blockdiag_wgrad(X, dY, b, dG, stream=None):
    N, D = X.shape
    splits = dG.shape[0]
    _check("poetx_blockdiag_wgrad", lib().poetx_blockdiag_wgrad(dtype_code(X), _p(X), _p(dY), N,
                                                                D // b, b, splits, _p(dG),
                                                                _stream(stream)))


def poetx_wprime_gemm(A, W, C, trans=False, w_scale=None, stream=None):
    N = A.shape[0]
    n, m = W.shape
    _check("poetx_wprime_gemm", lib().poetx_wprime_gemm(dtype_code(A), dtype_code(W), _p(A), N, m,
                                                        n, _p(W), _p(w_scale), int(bool(trans)),
                                                        _p(C), _stream(stream)))


# ---------------------------------------------------------------- the layer
def make_layer(m, n, b, act, wdt, variant, perm_m, perm_n, Wp, q_R, q_P, w_scale=None,
               order=3) -> LayerDesc:
    """Build a ``poetx_layer`` descriptor; the tensors must outlive its use."""
    return LayerDesc(m, n, b, order, act, wdt, variant, _p(perm_m), _p(perm_n), _p(Wp),
                     _p(w_scale), _p(q_R), _p(q_P))


def poetx_layer_workspace_bytes(L: LayerDesc, N: int, phase: int) -> int:
    return lib().poetx_layer_workspace_bytes(ctypes.byref(L), N, phase)


def poetx_layer_cuda_core_steps(L: LayerDesc, N: int) -> int:
    """Bit mask of the layer's products on the CUDA cores (bit 0 CNP, bit 1 block-diagonal
    products, bit 2 W' contraction); 0: all on the tensor cores; -1: invalid descriptor."""
    return lib().poetx_layer_cuda_core_steps(ctypes.byref(L), N)


def poetx_layer_saved_bytes(L: LayerDesc, N: int) -> int:
    return lib().poetx_layer_saved_bytes(ctypes.byref(L), N)


def poetx_layer_fwd(L: LayerDesc, x, y, saved, ws, stream=None):
    N = x.shape[0]
    _check("poetx_layer_fwd", lib().poetx_layer_fwd(ctypes.byref(L), _p(x), N, _p(y), _p(saved),
                                                    _p(ws), ws.numel(), _stream(stream)))


def poetx_layer_bwd(L: LayerDesc, x, dy, saved, dx, dq_R, dq_P, ws, accumulate=False,
                    stream=None):
    N = x.shape[0]
    _check("poetx_layer_bwd", lib().poetx_layer_bwd(ctypes.byref(L), _p(x), _p(dy), N, _p(saved),
                                                    _p(dx), _p(dq_R), _p(dq_P),
                                                    int(bool(accumulate)), _p(ws), ws.numel(),
                                                    _stream(stream)))


def poetx_layer_step_host_bytes(L: LayerDesc, N: int) -> int:
    return lib().poetx_layer_step_host_bytes(ctypes.byref(L), N)


def poetx_layer_step_host(L: LayerDesc, x, dy, y, dx, dq_R, dq_P, dev, stream=None):
    """Forward + backward with host (CPU, preferably pinned) tensors x, dy in and y, dx,
    dq_R, dq_P out; dev: device scratch of poetx_layer_step_host_bytes(L, N) bytes.  The
    outputs are valid once `stream` has been synchronised."""
    for t in (x, dy, y, dx, dq_R, dq_P):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("poetx_layer_step_host takes contiguous host tensors")
    N = x.shape[0]
    h = lambda t: ctypes.c_void_p(t.data_ptr())
    _check("poetx_layer_step_host", lib().poetx_layer_step_host(
        ctypes.byref(L), h(x), h(dy), N, h(y), h(dx), h(dq_R), h(dq_P), _p(dev),
        dev.numel() * dev.element_size(), _stream(stream)))


def poetx_merge_reinit_workspace_bytes(L: LayerDesc) -> int:
    return lib().poetx_merge_reinit_workspace_bytes(ctypes.byref(L))


def poetx_merge_reinit(L: LayerDesc, W0_new, ws, stream=None):
    """W0_new [n, m] fp32 <- the layer's current map as a plain weight (q reset is the
    caller's)."""
    _check("poetx_merge_reinit", lib().poetx_merge_reinit(ctypes.byref(L), _p(W0_new), _p(ws),
                                                          ws.numel(), _stream(stream)))


def poetx_adam_triu(q, dq, m, v, step: int, lr: float, beta1: float = 0.9, beta2: float = 0.999,
                    eps: float = 1e-8, weight_decay: float = 0.0, stream=None):
    """In-place Adam step on the packed triangles q (m, v: state, zero at step 1)."""
    hp = AdamDesc(lr, beta1, beta2, eps, weight_decay, step)
    _check("poetx_adam_triu", lib().poetx_adam_triu(_p(q), _p(dq), _p(m), _p(v), q.numel(),
                                                    ctypes.byref(hp), _stream(stream)))


def poetx_timeout_site() -> int:
    """Site id of the first expired bounded wait reported by the last poetx_get_device_error
    (file id x 10000 + source line), 0 if none."""
    return lib().poetx_timeout_site()


def poetx_layer_bwd_adam(L: LayerDesc, x, dy, saved, dx, dq_R, dq_P, ws, m_R, v_R, m_P, v_P,
                         step: int, lr: float, beta1: float = 0.9, beta2: float = 0.999,
                         eps: float = 1e-8, weight_decay: float = 0.0, accumulate=False,
                         stream=None):
    """poetx_layer_bwd, then Adam on the layer's q_R and q_P in place (fused into the
    gradient pack)."""
    hp = AdamDesc(lr, beta1, beta2, eps, weight_decay, step)
    N = x.shape[0]
    _check("poetx_layer_bwd_adam", lib().poetx_layer_bwd_adam(
        ctypes.byref(L), _p(x), _p(dy), N, _p(saved), _p(dx), _p(dq_R), _p(dq_P),
        int(bool(accumulate)), ctypes.byref(hp), _p(m_R), _p(v_R), _p(m_P), _p(v_P), _p(ws),
        ws.numel(), _stream(stream)))


# ---------------------------------------------------------------- layer groups
GROUP_MAX_LAYERS = 16


def make_group(layers):
    """A ctypes array of ``poetx_layer`` descriptors (the group); the tensors the descriptors
    point to must outlive its use."""
    arr = (LayerDesc * len(layers))(*layers)
    return arr


def poetx_group_saved_bytes(G, N: int) -> int:
    return lib().poetx_group_saved_bytes(G, len(G), N)


def poetx_group_workspace_bytes(G, N: int) -> int:
    return lib().poetx_group_workspace_bytes(G, len(G), N)


def poetx_group_cnp_fwd(G, N: int, saved, stream=None):
    _check("poetx_group_cnp_fwd", lib().poetx_group_cnp_fwd(G, len(G), N, _p(saved),
                                                            _stream(stream)))


def poetx_group_layer_fwd(G, i: int, x, y, saved, ws, stream=None):
    N = x.shape[0]
    _check("poetx_group_layer_fwd", lib().poetx_group_layer_fwd(
        G, len(G), i, _p(x), N, _p(y), _p(saved), _p(ws), ws.numel(), _stream(stream)))


def poetx_group_layer_bwd(G, i: int, x, dy, saved, dx, ws, stream=None):
    N = x.shape[0]
    _check("poetx_group_layer_bwd", lib().poetx_group_layer_bwd(
        G, len(G), i, _p(x), _p(dy), N, _p(saved), _p(dx), _p(ws), ws.numel(),
        _stream(stream)))


def poetx_group_cnp_bwd(G, N: int, saved, dq_R, dq_P, ws, accumulate=False, stream=None):
    """dq_R, dq_P: one fp32 tensor per layer of the group."""
    if len(dq_R) != len(G) or len(dq_P) != len(G):
        raise ValueError("poetx_group_cnp_bwd: one dq_R and one dq_P per layer")
    pr = (ctypes.c_void_p * len(G))(*[t.data_ptr() for t in dq_R])
    pp = (ctypes.c_void_p * len(G))(*[t.data_ptr() for t in dq_P])
    for t in list(dq_R) + list(dq_P):
        _p(t)
    _check("poetx_group_cnp_bwd", lib().poetx_group_cnp_bwd(
        G, len(G), N, _p(saved), pr, pp, int(bool(accumulate)), _p(ws), ws.numel(),
        _stream(stream)))


def poetx_group_step_host_bytes(G, N: int) -> int:
    return lib().poetx_group_step_host_bytes(G, len(G), N)


def poetx_group_step_host(G, xs, dys, ys, dxs, dq_R, dq_P, dev, stream=None):
    """One training step of the group with host (CPU, preferably pinned) tensors: xs, dys in,
    ys, dxs, dq_R, dq_P out (one per layer); dev: device scratch of
    poetx_group_step_host_bytes(G, N) bytes.  The outputs are valid once `stream` has been
    synchronised."""
    k = len(G)
    lists = (xs, dys, ys, dxs, dq_R, dq_P)
    if any(len(t) != k for t in lists):
        raise ValueError("poetx_group_step_host: one tensor per layer in every list")
    for ts in lists:
        for t in ts:
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("poetx_group_step_host takes contiguous host tensors")
    N = xs[0].shape[0]
    arr = lambda ts: (ctypes.c_void_p * k)(*[t.data_ptr() for t in ts])
    _check("poetx_group_step_host", lib().poetx_group_step_host(
        G, k, arr(xs), arr(dys), N, arr(ys), arr(dxs), arr(dq_R), arr(dq_P), _p(dev),
        dev.numel() * dev.element_size(), _stream(stream)))
