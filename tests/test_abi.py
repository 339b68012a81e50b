"""CPU-only checks of the C ABI: the library builds and loads, exports every function the
header declares, and rejects bad arguments on the host before launching anything."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "poetx.h")


@pytest.fixture(scope="module")
def P():
    from orthogonal_reparameterized_gb300 import build
    build.build()
    import orthogonal_reparameterized_gb300.poetx as P
    P.lib()
    return P


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(poetx_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("poetx_cnp_fwd", "poetx_cnp_bwd", "poetx_layer_fwd", "poetx_layer_bwd",
                 "poetx_merge_perm"):
        assert must in names


def test_every_declared_symbol_is_exported(P):
    out = subprocess.run(["nm", "-D", "--defined-only", P.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (poetx_\w+)", out))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    lib = P.lib()
    for n in _declared():
        assert getattr(lib, n) is not None


def test_binding_covers_every_symbol(P):
    for n in _declared():
        assert n in P._SIGS, n


def test_status_strings(P):
    for st in range(9):
        assert P.status_str(st).startswith("POETX_")
    assert "UNKNOWN" in P.status_str(99)


def _desc(P, **kw):
    d = dict(m=256, n=512, b=64, act=P.BF16, wdt=P.BF16, variant=P.FAST, order=3)
    d.update(kw)
    fake = ctypes.c_void_p(4096)  # never dereferenced: only host-side logic runs
    return P.LayerDesc(d["m"], d["n"], d["b"], d["order"], d["act"], d["wdt"], d["variant"],
                       fake, fake, fake, fake if d["wdt"] == P.I8 else None, fake, fake)


def test_layer_sizes_host_logic(P):
    L = _desc(P)
    N = 1000
    fast = P.poetx_layer_saved_bytes(L, N)
    mem = P.poetx_layer_saved_bytes(_desc(P, variant=P.MEM), N)
    assert fast - mem >= N * (512 + 256) * 2  # B and x~
    assert mem >= (256 + 512) * 64 * (2 + 4)
    assert P.poetx_layer_workspace_bytes(L, N, 0) >= N * (256 + 512) * 2  # A, z~
    assert P.poetx_layer_workspace_bytes(_desc(P, variant=P.MEM), N, 1) > \
        P.poetx_layer_workspace_bytes(L, N, 1)
    # invalid descriptors report 0 bytes
    assert P.poetx_layer_workspace_bytes(_desc(P, b=100), N, 0) == 0        # b not supported
    # b does not divide m: a ragged last block, padded inside (m multiple of 8 needed)
    rag = P.poetx_layer_workspace_bytes(_desc(P, m=320, b=128), N, 0)
    assert rag >= N * (384 + 512) * 2                                     # A, z~ padded
    assert P.poetx_layer_workspace_bytes(_desc(P, m=324, b=128), N, 0) == 0
    assert P.poetx_layer_saved_bytes(_desc(P, m=320, b=128), N) >= N * (384 + 512) * 2
    assert P.poetx_layer_workspace_bytes(_desc(P, order=4), N, 0) == 0
    assert P.poetx_layer_workspace_bytes(_desc(P, wdt=P.I8), N, 0) == 0      # int8 needs mem
    assert P.poetx_layer_workspace_bytes(_desc(P, wdt=P.I8, variant=P.MEM), N, 0) > 0
    assert P.poetx_layer_workspace_bytes(_desc(P, act=P.F32, wdt=P.BF16), N, 0) == 0
    assert P.poetx_layer_workspace_bytes(_desc(P, act=P.F32, wdt=P.F32, b=32), N, 0) > 0


def test_merge_reinit_workspace_host_logic(P):
    L = _desc(P)
    need = P.poetx_merge_reinit_workspace_bytes(L)
    assert need >= (256 + 512) * 64 * 4 * 3 + 2 * 256 * 512 * 4  # G, Q, Q^2; T, M
    assert P.poetx_merge_reinit_workspace_bytes(_desc(P, wdt=P.I8, variant=P.MEM)) >= \
        need + 256 * 512 * 4                                      # the dequantised W'
    assert P.poetx_merge_reinit_workspace_bytes(_desc(P, b=100)) == 0
    lib = P.lib()
    fake = ctypes.c_void_p(4096)
    assert lib.poetx_merge_reinit(ctypes.byref(L), fake, fake, 16, None) == 5
    assert lib.poetx_merge_reinit(ctypes.byref(L), ctypes.c_void_p(4100), fake, 1 << 30,
                                  None) == 4
    assert lib.poetx_merge_reinit(ctypes.byref(_desc(P, order=2)), fake, fake, 1 << 30,
                                  None) == 6


def test_adam_argument_errors(P):
    lib = P.lib()
    fake = ctypes.c_void_p(4096)
    hp = P.AdamDesc(1e-3, 0.9, 0.999, 1e-8, 0.0, 0)          # step 0
    assert lib.poetx_adam_triu(fake, fake, fake, fake, 8, ctypes.byref(hp), None) == 1
    hp.step = 1
    assert lib.poetx_adam_triu(fake, fake, fake, fake, 0, ctypes.byref(hp), None) == 0
    assert lib.poetx_adam_triu(ctypes.c_void_p(4100), fake, fake, fake, 8, ctypes.byref(hp),
                               None) == 4
    hp.beta2 = 1.0
    assert lib.poetx_adam_triu(fake, fake, fake, fake, 8, ctypes.byref(hp), None) == 1
    assert lib.poetx_adam_triu(fake, fake, fake, fake, 8, None, None) == 1


def test_argument_errors_before_launch(P):
    lib = P.lib()
    fake = ctypes.c_void_p(4096)
    L = _desc(P, order=2)
    assert lib.poetx_layer_fwd(ctypes.byref(L), fake, 4, fake, fake, fake, 1 << 30, None) == 6
    L = _desc(P)
    assert lib.poetx_layer_fwd(ctypes.byref(L), fake, 4, None, fake, fake, 1 << 30, None) == 1
    assert lib.poetx_layer_fwd(ctypes.byref(L), fake, 4, fake, fake, fake, 16, None) == 5
    mis = ctypes.c_void_p(4100)
    assert lib.poetx_layer_fwd(ctypes.byref(L), mis, 4, fake, fake, fake, 1 << 30, None) == 4
    assert lib.poetx_cnp_fwd(fake, 4, 64, 2, fake, None, None, fake, 1 << 30, None) == 6
    assert lib.poetx_cnp_fwd(fake, 4, 1, 3, fake, None, None, fake, 1 << 30, None) == 2
    assert lib.poetx_cnp_fwd(fake, 4, 64, 3, None, None, None, fake, 1 << 30, None) == 1
    assert lib.poetx_cnp_fwd(fake, 4, 64, 3, fake, None, None, fake, 8, None) == 5
    assert lib.poetx_cnp_fwd(fake, 0, 64, 3, fake, None, None, fake, 8, None) == 0  # empty
    assert lib.poetx_cnp_bwd(fake, fake, 0, 4, 64, 3, fake, 0, fake, 1 << 30, None) == 1
    assert lib.poetx_perm_gather(P.BF16, fake, 0, 64, fake, fake, None) == 0     # N = 0
    assert lib.poetx_perm_gather(7, fake, 4, 64, fake, fake, None) == 3
    assert lib.poetx_perm_gather(P.BF16, mis, 4, 64, fake, fake, None) == 4
    assert lib.poetx_blockdiag_mm(P.BF16, fake, 4, 2, 100, fake, 0, None, None, fake, None) == 2
    assert lib.poetx_blockdiag_mm(P.BF16, fake, 4, 2, 64, fake, 0, None, fake, fake, None) == 1
    assert lib.poetx_blockdiag_wgrad(P.BF16, fake, fake, 4, 2, 64, 0, fake, None) == 1
    assert lib.poetx_wprime_gemm(P.F32, P.BF16, fake, 4, 64, 64, fake, None, 0, fake, None) == 3
    assert lib.poetx_wprime_gemm(P.BF16, P.I8, fake, 4, 64, 64, fake, None, 0, fake, None) == 1
    assert lib.poetx_merge_perm(fake, None, P.I8, 4, 64, fake, fake, fake, None, None) == 1
    assert lib.poetx_set_gemm_engine(5) == 1
    assert lib.poetx_cnp_workspace_bytes(4, 64, 0) == 2 * 4 * 64 * 64 * 4
    assert lib.poetx_cnp_workspace_bytes(4, 1, 0) == 0


def test_step_host_sizes_and_argument_errors(P):
    """The host-buffer step: its device scratch covers the six device arrays, the saved state
    and the larger of the two workspaces; bad arguments are refused before any CUDA call."""
    L = _desc(P)
    N = 1000
    need = P.poetx_layer_step_host_bytes(L, N)
    arrays = 2 * N * (256 + 512) * 2 + (256 // 64 + 512 // 64) * (64 * 63 // 2) * 4
    ws = max(P.poetx_layer_workspace_bytes(L, N, 0), P.poetx_layer_workspace_bytes(L, N, 1))
    assert need >= arrays + P.poetx_layer_saved_bytes(L, N) + ws
    assert P.poetx_layer_step_host_bytes(_desc(P, b=100), N) == 0
    assert P.poetx_layer_step_host_bytes(L, -1) == 0
    lib = P.lib()
    fake = ctypes.c_void_p(4096)
    args = [fake] * 6
    assert lib.poetx_layer_step_host(ctypes.byref(L), *args[:2], 4, *args[2:], fake, 16,
                                     None) == 5
    assert lib.poetx_layer_step_host(ctypes.byref(L), *args[:2], 4, *args[2:],
                                     ctypes.c_void_p(4100), 1 << 40, None) == 4
    assert lib.poetx_layer_step_host(ctypes.byref(L), None, fake, 4, *args[2:], fake, 1 << 40,
                                     None) == 1
    assert lib.poetx_layer_step_host(ctypes.byref(_desc(P, order=2)), *args[:2], 4, *args[2:],
                                     fake, 1 << 40, None) == 6
    assert lib.poetx_layer_step_host(ctypes.byref(L), *args[:2], -1, *args[2:], fake, 1 << 40,
                                     None) == 1


def test_merge_perm_padded_argument_errors(P):
    lib = P.lib()
    fake = ctypes.c_void_p(4096)
    f = lib.poetx_merge_perm_padded
    assert f(fake, None, P.BF16, 8, 8, 4, 8, fake, fake, fake, None, None) == 1   # n_pad < n
    assert f(fake, None, P.BF16, 8, 12, 8, 16, fake, fake, fake, None, None) == 2  # 24-byte rows
    assert f(fake, None, P.BF16, 8, 8, 8, 8, fake, fake, ctypes.c_void_p(4100), None,
             None) == 4                                                            # Wp unaligned
    assert f(fake, fake, P.I8, 6, 16, 8, 16, fake, fake, fake, fake, None) == 2    # int8: n % 4
    assert f(fake, None, P.I8, 8, 16, 8, 16, fake, fake, fake, fake, None) == 1    # no scale
    assert f(fake, None, 9, 8, 8, 8, 8, fake, fake, fake, None, None) == 3         # dtype


def test_layer_bwd_adam_argument_errors(P):
    lib = P.lib()
    fake = ctypes.c_void_p(4096)
    L = _desc(P)
    hp = P.AdamDesc(1e-3, 0.9, 0.999, 1e-8, 0.0, 0)           # step 0
    args = (fake, fake, 4, fake, fake, fake, fake, 0)
    assert lib.poetx_layer_bwd_adam(ctypes.byref(L), *args, ctypes.byref(hp), fake, fake, fake,
                                    fake, fake, 1 << 30, None) == 1
    hp.step = 1
    assert lib.poetx_layer_bwd_adam(ctypes.byref(L), *args, ctypes.byref(hp), None, fake, fake,
                                    fake, fake, 1 << 30, None) == 1
    assert lib.poetx_layer_bwd_adam(ctypes.byref(L), *args, None, fake, fake, fake, fake, fake,
                                    1 << 30, None) == 1
    assert lib.poetx_layer_bwd_adam(ctypes.byref(_desc(P, order=2)), *args, ctypes.byref(hp),
                                    fake, fake, fake, fake, fake, 1 << 30, None) == 6
    assert lib.poetx_layer_bwd_adam(ctypes.byref(L), *args, ctypes.byref(hp), fake, fake, fake,
                                    fake, fake, 16, None) == 5                 # workspace


def test_engine_query_host_logic(P):
    assert P.poetx_layer_cuda_core_steps(_desc(P, b=100), 64) == -1      # invalid descriptor
    assert P.poetx_layer_cuda_core_steps(_desc(P), -1) == -1
    # an fp32 layer runs its layer products on the CUDA cores by design
    f32 = P.poetx_layer_cuda_core_steps(_desc(P, act=P.F32, wdt=P.F32, b=32), 64)
    assert f32 >= 0 and f32 & 6 == 6
    assert P.poetx_layer_cuda_core_steps(_desc(P), 64) >= 0


def test_group_sizes_host_logic(P):
    a, b = _desc(P), _desc(P, m=512, n=256)
    G = P.make_group([a, b])
    N = 100
    sv = P.poetx_group_saved_bytes(G, N)
    ws = P.poetx_group_workspace_bytes(G, N)
    # the group keeps at least what the two layers keep, less N-independent duplication
    assert sv >= P.poetx_layer_saved_bytes(a, N) + P.poetx_layer_saved_bytes(b, N) - 16 * 4096
    assert ws > 0
    assert P.poetx_group_saved_bytes(P.make_group([a, _desc(P, b=128)]), N) == 0  # mixed b
    assert P.poetx_group_saved_bytes(P.make_group([a, _desc(P, act=P.F32, wdt=P.F32)]),
                                     N) == 0                                 # mixed act
    assert P.poetx_group_saved_bytes(P.make_group([a] * 17), N) == 0         # > 16 layers
    assert P.poetx_group_saved_bytes(P.make_group([a] * 16), N) > 0


def test_group_step_host_sizes_host_logic(P):
    a, b = _desc(P), _desc(P, m=512, n=256)
    G = P.make_group([a, b])
    N = 100
    host = P.poetx_group_step_host_bytes(G, N)
    # every layer's x, dy, y, dx and dq on the device, plus the group's saved state and workspace
    arrays = 0
    for d in (a, b):
        arrays += 2 * N * (d.m + d.n) * 2 + (d.m // d.b + d.n // d.b) * (d.b * (d.b - 1) // 2) * 4
    assert host >= arrays + P.poetx_group_saved_bytes(G, N) + P.poetx_group_workspace_bytes(G, N)
    assert P.poetx_group_step_host_bytes(P.make_group([a, _desc(P, b=128)]), N) == 0
    assert P.poetx_group_step_host_bytes(G, -1) == 0
