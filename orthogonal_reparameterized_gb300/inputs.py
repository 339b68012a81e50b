"""Seeded synthetic inputs for the POET-X layer and the Cayley-Neumann workloads.

This module draws random arrays and rounds them to their storage dtype; it holds none of
the method's arithmetic.  The fp64 oracle (through the tests and the CPU-baseline leg of
the benchmark) and the CUDA path both consume exactly the arrays produced here; the
benchmark's timed full-size workloads draw the same distributions on the device instead
(``device_layer_inputs``), where no oracle reads them.

Generator: numpy's Philox4x32-10 counter-based bit generator (Salmon et al., SC'11),
keyed by (seed, crc32(tensor name)) so that every tensor has its own sub-stream and the
draw of one tensor never shifts another.  Gaussians come from numpy's
``Generator.standard_normal`` and permutations from ``Generator.permutation``
(Fisher-Yates).  Values are drawn in float64, then rounded to the storage dtype
(fp32 by IEEE round-to-nearest-even; bf16 as round-to-nearest-even of that fp32), and
returned as float64 arrays holding exactly the representable stored values.

Workloads (shapes and value distributions follow the POET-X summary page's layer
profile, "Experiments": single-layer fwd+bwd at Llama hidden sizes):

* ``fp32_256_b32``   -- one fp32 layer, m=n=256, b=32, N=64, q ~ N(0, 0.01^2)
* ``llama1b_2048``   -- one bf16 layer, m=n=2048, b=256, N=4096, q ~ N(0, 0.02^2)
* ``llama8b_block``  -- the seven bf16 linears of a Llama-8B block, b=256, N=8192
* ``sweep_4096_b*``  -- one bf16 4096x4096 layer, N=4096, b in {64,128,256,512}
* ``llama13b_mlp_int8`` -- 5120->13824 and 13824->5120, int8 W0, b=512, N=4096, mem
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Dict, List, Tuple

import numpy as np

BASE_SEED = 20260305


def _rng(seed: int, name: str) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed) & 0xFFFFFFFF, zlib.crc32(name.encode())])
    return np.random.Generator(np.random.Philox(ss))


def round_to(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the storage dtype and widen them back to float64."""
    if dtype == "f64":
        return np.asarray(a, dtype=np.float64)
    f32 = np.asarray(a, dtype=np.float32)
    if dtype == "f32":
        return f32.astype(np.float64)
    if dtype == "bf16":
        # round-to-nearest-even on the 16 dropped mantissa bits, in 32-bit integers: the sum
        # stays below 2^32 for every finite value (no NaN is ever drawn)
        u = f32.view(np.uint32)
        r = (u >> 16) & np.uint32(1)
        r += np.uint32(0x7FFF)
        r += u
        r &= np.uint32(0xFFFF0000)
        return r.view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype}")


def gaussian(seed: int, name: str, shape, std: float = 1.0, dtype: str = "f32") -> np.ndarray:
    g = _rng(seed, name).standard_normal(size=shape)
    return round_to(g * std, dtype)


def permutation(seed: int, name: str, n: int) -> np.ndarray:
    return _rng(seed, name).permutation(n).astype(np.int32)


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """One linear layer: W0 is [n_out, m_in] (PyTorch Linear layout)."""
    name: str
    m: int  # in-features
    n: int  # out-features


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: Tuple[LayerShape, ...]
    b: int
    N: int
    act: str          # "f32" or "bf16"
    wdt: str          # "f32", "bf16" or "i8"
    q_std: float
    variants: Tuple[str, ...]
    seed: int


def _wl(name, layers, b, N, act, wdt, q_std, variants, idx):
    return Workload(name, tuple(LayerShape(*l) for l in layers), b, N, act, wdt, q_std,
                    tuple(variants), BASE_SEED + idx)


_LLAMA8B = [("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
            ("gate", 4096, 14336), ("up", 4096, 14336), ("down", 14336, 4096)]

WORKLOADS: Dict[str, Workload] = {
    "fp32_256_b32": _wl("fp32_256_b32", [("lin", 256, 256)], 32, 64, "f32", "f32", 0.01,
                        ["fast", "mem"], 0),
    "llama1b_2048": _wl("llama1b_2048", [("lin", 2048, 2048)], 256, 4096, "bf16", "bf16", 0.02,
                        ["fast", "mem"], 1),
    "llama8b_block": _wl("llama8b_block", _LLAMA8B, 256, 8192, "bf16", "bf16", 0.02, ["fast"], 2),
    "sweep_4096_b64": _wl("sweep_4096_b64", [("lin", 4096, 4096)], 64, 4096, "bf16", "bf16", 0.02,
                          ["fast", "mem"], 3),
    "sweep_4096_b128": _wl("sweep_4096_b128", [("lin", 4096, 4096)], 128, 4096, "bf16", "bf16",
                           0.02, ["fast", "mem"], 3),
    "sweep_4096_b256": _wl("sweep_4096_b256", [("lin", 4096, 4096)], 256, 4096, "bf16", "bf16",
                           0.02, ["fast", "mem"], 3),
    "sweep_4096_b512": _wl("sweep_4096_b512", [("lin", 4096, 4096)], 512, 4096, "bf16", "bf16",
                           0.02, ["fast", "mem"], 3),
    "llama13b_mlp_int8": _wl("llama13b_mlp_int8", [("up", 5120, 13824), ("down", 13824, 5120)],
                             512, 4096, "bf16", "i8", 0.02, ["mem"], 4),
    # ragged last blocks (b does not divide the sides): 2000 = 7 x 256 + 208, computed padded
    # to the 2048-wide layer
    "ragged_2000_b256": _wl("ragged_2000_b256", [("lin", 2000, 2000)], 256, 4096, "bf16",
                            "bf16", 0.02, ["fast", "mem"], 5),
}


def layer_inputs(wl: Workload, layer: LayerShape, N: int | None = None,
                 q_scale: float = 1.0) -> Dict[str, np.ndarray]:
    """All inputs of one layer of a workload, as float64 / int32 numpy arrays.

    x [N,m] and dy [N,n] ~ N(0,1) in the activation dtype; W0 [n,m] ~ N(0, 1/m) (fp32 when
    the layer stores int8 weights: that is the pre-quantisation weight); q_R [ceil(m/b),
    b(b-1)/2] and q_P [ceil(n/b), b(b-1)/2] ~ N(0, q_std^2) in fp32; perm_m [m], perm_n [n] uniform.
    ``N`` overrides the token count (a token prefix of the same draw is NOT implied: a
    different N gives a different draw).
    """
    N = wl.N if N is None else N
    s, tag, b = wl.seed, f"{layer.name}/", wl.b
    m, n = layer.m, layer.n
    wstore = "f32" if wl.wdt == "i8" else wl.wdt
    tri = b * (b - 1) // 2
    return {
        "x": gaussian(s, tag + f"x{N}", (N, m), 1.0, wl.act),
        "dy": gaussian(s, tag + f"dy{N}", (N, n), 1.0, wl.act),
        "W0": gaussian(s, tag + "W0", (n, m), 1.0 / np.sqrt(m), wstore),
        "q_R": gaussian(s, tag + "qR", (-(-m // b), tri), wl.q_std * q_scale, "f32"),
        "q_P": gaussian(s, tag + "qP", (-(-n // b), tri), wl.q_std * q_scale, "f32"),
        "perm_m": permutation(s, tag + "pm", m),
        "perm_n": permutation(s, tag + "pn", n),
    }


def small_layer_inputs(seed: int, m: int, n: int, b: int, N: int, act: str = "f32",
                       wdt: str = "f32", q_std: float = 0.02) -> Dict[str, np.ndarray]:
    """Inputs of an ad-hoc layer shape (tests: ragged token counts, tiny cases)."""
    wl = Workload("adhoc", (LayerShape("adhoc", m, n),), b, N, act, wdt, q_std, ("fast",), seed)
    return layer_inputs(wl, wl.layers[0])


def cnp_inputs(seed: int, nblk: int, b: int, std: float, name: str = "q") -> np.ndarray:
    """Packed strict upper triangles [nblk, b(b-1)/2] fp32 ~ N(0, std^2)."""
    return gaussian(seed, f"cnp/{name}/{nblk}x{b}", (nblk, b * (b - 1) // 2), std, "f32")


def dG_inputs(seed: int, splits: int, nblk: int, b: int, name: str = "dG") -> np.ndarray:
    """Upstream gradient partials [splits, nblk, b, b] fp32 ~ N(0, 1)."""
    return gaussian(seed, f"cnp/{name}/{splits}x{nblk}x{b}", (splits, nblk, b, b), 1.0, "f32")


def workload_names() -> List[str]:
    return list(WORKLOADS)


def device_layer_inputs(wl: Workload, layer: LayerShape, device, N: int | None = None):
    """The tensors of ``layer_inputs`` drawn on a CUDA device by torch's Philox generator,
    for the benchmark's full-size workloads (numpy draws a Llama-8B block's ~1e9 values in
    minutes).  Same names, shapes, distributions and storage dtypes, each tensor keyed by
    (seed, crc32(name)) as above; the values differ from the numpy draw, so parity tests use
    ``layer_inputs``.  Returns torch tensors on ``device``: x, dy in the activation dtype,
    W0 (fp32 for an int8-stored weight), q_R, q_P fp32, perm_m, perm_n int32."""
    import torch

    N = wl.N if N is None else N
    s, tag, b = wl.seed, f"{layer.name}/", wl.b
    m, n = layer.m, layer.n
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}
    wstore = "f32" if wl.wdt == "i8" else wl.wdt
    tri = b * (b - 1) // 2

    def gen(name):
        g = torch.Generator(device=device)
        g.manual_seed(((int(s) & 0xFFFFFFFF) << 32) | zlib.crc32((tag + name).encode()))
        return g

    def gauss(name, shape, std, dt):
        t = torch.randn(*shape, generator=gen(name), device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        return t.to(tdt[dt])

    def perm(name, d):
        return torch.randperm(d, generator=gen(name), device=device).to(torch.int32)

    return {
        "x": gauss(f"x{N}", (N, m), 1.0, wl.act),
        "dy": gauss(f"dy{N}", (N, n), 1.0, wl.act),
        "W0": gauss("W0", (n, m), 1.0 / float(np.sqrt(m)), wstore),
        "q_R": gauss("qR", (-(-m // b), tri), wl.q_std, "f32"),
        "q_P": gauss("qP", (-(-n // b), tri), wl.q_std, "f32"),
        "perm_m": perm("pm", m),
        "perm_n": perm("pn", n),
    }
