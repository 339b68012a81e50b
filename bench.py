#!/usr/bin/env python3
"""Benchmark of the POET-X layer step on GB300.

A step is one pass of the whole hot path on one batch: both Cayley-Neumann forwards, the
layer forward, the layer backward and both Cayley-Neumann backwards (poetx_layer_fwd +
poetx_layer_bwd through the C ABI), on the Llama-1B-shaped layer (m = n = 2048, b = 256,
N = 4096 bf16 tokens), fast variant.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--variant fast|mem]

N > 1 runs under torchrun: one replica per GPU on its own tokens (weak scaling, no
collective on the data path; the timing is the max over ranks).  --impl reference times
the fp64 CPU oracle on the host cores on a bounded sample of the same workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "POET-X layer fwd+bwd tokens/s; CNP blocks/s; % of BF16 TC peak / HBM BW"
L2_FLUSH_BYTES = 512 << 20  # larger than the 129 MB L2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama1b_2048")
    ap.add_argument("--variant", default="fast", choices=["fast", "mem"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fusion", default="on", choices=["on", "off"],
                    help="W' contraction + following block product in one kernel (default on)")
    ap.add_argument("--overlap", default="on", choices=["on", "off"],
                    help="dx scatter on a side stream beside the CNP backward (library switch)")
    ap.add_argument("--all-layers", action="store_true",
                    help="also time every layer of a multi-layer workload (the Llama-8B "
                         "block's 7 linears, the 13B MLP's up and down) and report their sum")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [r for t, r in self.rows if t0 <= t <= t1]
        note = "samples inside the timed region"
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = [r for t, r in self.rows if t0 - 1.0 <= t <= t1 + 1.0]
            note = "samples within 1 s of the timed region (region shorter than the period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no samples"}
        sm = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for k, nm in enumerate(names):
                if len(r) > 5 + k and r[5 + k].lower().startswith("active"):
                    reasons.add(nm)
        pw = [float(r[3]) for r in inside if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "power_w_max": max(pw) if pw else None, "samples": len(inside), "note": note}


# ------------------------------------------------------------------ CPU oracle
CPU_SNIPPET = r"""
import json, os, sys, time
sys.path.insert(0, %(root)r)
import numpy as np
import oracle as O
from orthogonal_reparameterized_gb300 import inputs
wl = inputs.WORKLOADS[%(wl)r]
layer = wl.layers[0]
inp = inputs.layer_inputs(wl, layer, N=%(ntok)d)
W = inp["W0"]
if wl.wdt == "i8":
    Wq, s = O.quantize_rows_int8(W)
    W = O.dequantize_rows(Wq, s)
# the per-block oracle when b does not divide a side (ragged last block)
f = O.poetx_layer if layer.m %% wl.b == 0 and layer.n %% wl.b == 0 else O.poetx_layer_ragged
f(inp["x"][:8], inp["dy"][:8], W, inp["perm_m"], inp["perm_n"], inp["q_R"], inp["q_P"], wl.b)
times = []
t_end = time.perf_counter() + %(budget)f
while True:
    t0 = time.perf_counter()
    f(inp["x"], inp["dy"], W, inp["perm_m"], inp["perm_n"], inp["q_R"], inp["q_P"], wl.b)
    times.append(time.perf_counter() - t0)
    if len(times) >= %(reps)d or time.perf_counter() > t_end:
        break
print(json.dumps({"times": times}))
"""


def run_oracle_sample(wl_name, ntok, reps, budget_s):
    cores = os.cpu_count() or 1
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(cores)
    code = CPU_SNIPPET % {"root": ROOT, "wl": wl_name, "ntok": ntok, "reps": reps,
                          "budget": budget_s}
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=900)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed: " + r.stderr[-2000:])
    times = json.loads(r.stdout.strip().splitlines()[-1])["times"]
    return times, cores


def cpu_baseline(wl, ntok=512):
    times, cores = run_oracle_sample(wl.name, ntok, reps=50, budget_s=15.0)
    t = statistics.median(times)
    return {"value": ntok / t, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 numpy oracle, full step (CNP fwd x2, layer fwd+bwd, CNP bwd x2) of "
                      f"the {wl.name} layer on {ntok} of its {wl.N} tokens, median of "
                      f"{len(times)} runs"}


# ------------------------------------------------------------------ reference arm
def reference_arm(args, rank, world):
    from orthogonal_reparameterized_gb300 import inputs
    if rank != 0:
        return
    wl = inputs.WORKLOADS[args.workload]
    ntok = 256
    total = max(1, args.steps) + max(0, args.warmup)
    times, cores = run_oracle_sample(wl.name, ntok, reps=total, budget_s=180.0)
    timed = times[args.warmup:] if len(times) > args.warmup else times
    t = statistics.mean(timed)
    val = ntok / t
    out = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": len(timed), "warmup": min(args.warmup, len(times)),
           "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": wl.name, "m": wl.layers[0].m, "n": wl.layers[0].n, "b": wl.b,
                      "tokens_per_step": ntok, "variant": args.variant},
           "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": f"{ntok} tokens of the {wl.name} layer per step"},
           "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    if len(timed) < args.steps:
        out["note"] = f"time budget reached after {len(times)} oracle steps"
    print(json.dumps(out))


# ------------------------------------------------------------------ our arm
def merged_weight(P, W0, pn, pm, b, scale=None):
    """The layer's merged weight (and int8 scale), zero-padded to whole blocks of b when b
    does not divide a side (a ragged last block)."""
    import torch
    n, m = W0.shape
    n_pad, m_pad = -(-n // b) * b, -(-m // b) * b
    Wp = torch.empty(n_pad, m_pad, dtype=W0.dtype, device=W0.device)
    sc = None if scale is None else torch.empty(n_pad, device=W0.device)
    if (n_pad, m_pad) == (n, m):
        P.poetx_merge_perm(W0, pn, pm, Wp, scale, sc)
    else:
        P.poetx_merge_perm_padded(W0, pn, pm, Wp, scale, sc)
    return Wp, sc


def h2d_bytes_of(*ts):
    return sum(t.numel() * t.element_size() for t in ts)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return

    import numpy as np
    import torch
    import torch.distributed as dist

    from orthogonal_reparameterized_gb300 import inputs
    import orthogonal_reparameterized_gb300.poetx as P

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    P.lib()
    P.poetx_set_fusion(args.fusion == "on")
    P.poetx_set_overlap(args.overlap == "on")

    def check_err(section):
        """Fail loudly, naming the section, if a kernel recorded an error (a bounded wait
        that expired): no number is reported from such a run."""
        st = P.poetx_get_device_error()
        if st != 0:
            raise RuntimeError(f"device error after {section}: {P.status_str(st)} "
                               f"(wait site {P.poetx_timeout_site()})")

    wl = inputs.WORKLOADS[args.workload]
    layer = wl.layers[0]
    m, n, b, N = layer.m, layer.n, wl.b, wl.N
    bf = torch.bfloat16 if wl.act == "bf16" else torch.float32
    inp = inputs.layer_inputs(wl, layer)
    t = lambda a, dt: torch.tensor(a, dtype=dt, device=dev)
    x = t(inp["x"], bf)
    dy = t(inp["dy"], bf)
    pm = t(inp["perm_m"], torch.int32)
    pn = t(inp["perm_n"], torch.int32)
    qR = t(inp["q_R"], torch.float32)
    qP = t(inp["q_P"], torch.float32)
    w_scale = None
    if wl.wdt == "i8":
        W32 = t(inp["W0"], torch.float32)
        Wq = torch.empty(n, m, dtype=torch.int8, device=dev)
        s = torch.empty(n, device=dev)
        P.poetx_quantize_rows_int8(W32, Wq, s)
        Wp, w_scale = merged_weight(P, Wq, pn, pm, b, s)
        wcode = P.I8
    else:
        W0 = t(inp["W0"], bf)
        Wp, _ = merged_weight(P, W0, pn, pm, b)
        wcode = P.BF16 if wl.wdt == "bf16" else P.F32
    acode = P.BF16 if wl.act == "bf16" else P.F32
    esz = 2 if wl.act == "bf16" else 4

    def make(variant):
        L = P.make_layer(m, n, b, acode, wcode, P.FAST if variant == "fast" else P.MEM, pm, pn,
                         Wp, qR, qP, w_scale)
        bufs = dict(L=L, saved=P.workspace(P.poetx_layer_saved_bytes(L, N), dev),
                    wsf=P.workspace(P.poetx_layer_workspace_bytes(L, N, 0), dev),
                    wsb=P.workspace(P.poetx_layer_workspace_bytes(L, N, 1), dev),
                    y=torch.empty(N, n, dtype=bf, device=dev),
                    dx=torch.empty(N, m, dtype=bf, device=dev),
                    dqR=torch.empty_like(qR), dqP=torch.empty_like(qP))
        return bufs

    def step(B, xx=None, dyy=None):
        xx = x if xx is None else xx
        dyy = dy if dyy is None else dyy
        P.poetx_layer_fwd(B["L"], xx, B["y"], B["saved"], B["wsf"])
        P.poetx_layer_bwd(B["L"], xx, dyy, B["saved"], B["dx"], B["dqR"], B["dqP"], B["wsb"])

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def capture(B):
        """CUDA graph of one step (the same C-ABI calls, replayed without host launches)."""
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                step(B)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        c0 = P.poetx_launch_count()
        with torch.cuda.graph(g):
            step(B)
        torch.cuda.synchronize()
        return g, P.poetx_launch_count() - c0

    def timed_steps(B, K, W, graph=None):
        run = (lambda: graph.replay()) if graph is not None else (lambda: step(B))
        for _ in range(W):
            run()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        w0 = time.time()
        for e0, e1 in evs:
            flush.zero_()  # untimed L2 flush between steps
            e0.record()
            run()
            e1.record()
        torch.cuda.synchronize()
        w1 = time.time()
        if world > 1:
            dist.barrier()
        ms = [e0.elapsed_time(e1) for e0, e1 in evs]
        return ms, (w0, w1)

    variant = args.variant if wl.wdt != "i8" else "mem"
    main_b = make(variant)
    graph, kernels_per_step = capture(main_b)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms, (w0, w1) = timed_steps(main_b, args.steps, max(3, args.warmup), graph)
    time.sleep(0.3)
    clocks.stop()
    launches = kernels_per_step * args.steps
    ms_step = statistics.mean(ms)
    qs = statistics.quantiles(ms, n=10) if len(ms) >= 10 else [min(ms)] * 9
    ms_pct = {"p10": qs[0], "p50": statistics.median(ms), "p90": qs[8]}
    if world > 1:
        tt = torch.tensor([ms_step], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_step = float(tt.item())
    value = world * N / (ms_step * 1e-3)
    check_err("graph-replayed steps")
    # the same step issued eagerly (host launches through the C ABI), same protocol
    ems, _ = timed_steps(main_b, max(50, args.steps // 10), 5)
    eager = {"tokens_per_s": N / (statistics.mean(ems) * 1e-3), "ms_per_step": statistics.mean(ems)}

    check_err("eager steps")
    # the other variant, same protocol, fewer steps
    other = {}
    if wl.wdt != "i8":
        ov = "mem" if variant == "fast" else "fast"
        ob = make(ov)
        og, _ = capture(ob)
        oms, _ = timed_steps(ob, max(50, args.steps // 10), 5, og)
        other[ov] = {"tokens_per_s": N / (statistics.mean(oms) * 1e-3),
                     "ms_per_step": statistics.mean(oms)}
        del ob, og

    check_err("the other variant")
    # per-stage times inside the same layer calls (library stage events), same flushes
    P.poetx_profile_enable(True)
    P.poetx_profile_collect()
    stage_ms = {}
    prof_steps = 20
    for _ in range(prof_steps):
        flush.zero_()
        torch.cuda.synchronize()
        P.poetx_profile_collect()
        step(main_b)
        for name, t_ms in P.poetx_profile_collect():
            stage_ms.setdefault(name, []).append(t_ms)
    P.poetx_profile_enable(False)
    stages = {k: {"launches_per_step": len(v) / prof_steps, "ms_per_step": sum(v) / prof_steps,
                  "ms_per_launch": sum(v) / len(v)} for k, v in stage_ms.items()}

    pk = peaks()
    # the dominant kernel: the W' contraction, or (where the layer fuses them) the W'
    # contraction with the block-diagonal product after it, whose flops count too
    fused = "wprime_gemm" not in stages and "wprime_blockdiag_fused" in stages
    w_launch_ms = stages.get("wprime_blockdiag_fused" if fused else "wprime_gemm",
                             {}).get("ms_per_launch")
    flops = 2.0 * N * m * n + (2.0 * N * n * b if fused else 0.0)  # (square layers: n = m)
    achieved = flops / (w_launch_ms * 1e-3) / 1e12 if w_launch_ms else None
    traffic = None
    prof_json = os.path.join(ROOT, "profiles", ("wprime_blockdiag_fused" if fused else
                                                 "wprime_gemm") + f"_{wl.name}.json")
    if os.path.exists(prof_json):
        try:
            pj = json.load(open(prof_json))
            import hashlib
            src = open(os.path.join(ROOT, "orthogonal_reparameterized_gb300", "csrc",
                                    "umma_gemm.cu"), "rb").read()
            if pj.get("kernel_source_sha256") == hashlib.sha256(src).hexdigest():
                traffic = pj.get("dram_bytes_per_launch")
        except (OSError, ValueError, KeyError):
            traffic = None
    roofline = {"kernel": ("wprime_blockdiag_fused (tcgen05 W' contraction with the "
                           "block-diagonal product after it: fwd z~ = (A W'^T) blkdiag(G_P), "
                           "bwd dx~ = (dB W') blkdiag(G_R)^T; 2 N m n + 2 N n b flops per "
                           "launch)") if fused else
                          "wprime_gemm (tcgen05 W' contraction, fwd B = A W'^T and bwd "
                          "dA = dB W', 2 N m n flops per launch)",
                "bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": (achieved / pk["bf16_tflops"]) if achieved else None,
                "traffic": traffic,
                "peak_source": f"{pk['source']} dense bf16 burst (MEASURED_PEAKS.json)"}

    # HBM-bound stages against the measured copy bandwidth: every launch of these reads one
    # [N, D] activation and writes one (D = m = n for the benchmarked square layers)
    hbm = {}
    for name in ("perm_gather", "perm_scatter", "blockdiag_mm"):
        if name in stages and m == n:
            by = 2.0 * N * m * esz
            gbs = by / (stages[name]["ms_per_launch"] * 1e-3) / 1e9
            hbm[name] = {"algorithmic_bytes_per_launch": by, "achieved_gbs": gbs,
                         "frac_of_hbm": gbs / pk["hbm_gbs"]}

    check_err("per-stage timing")
    # CNP blocks/s (standalone, both sides' blocks)
    qcat = torch.cat([qR, qP], 0).contiguous()
    nblk = qcat.shape[0]  # ceil(m/b) + ceil(n/b)
    Gb = torch.empty(nblk, b, b, dtype=torch.bfloat16, device=dev)
    dG = torch.randn(1, nblk, b, b, device=dev)
    dq = torch.empty_like(qcat)
    wsc = P.workspace(max(P.poetx_cnp_workspace_bytes(nblk, b, 0),
                          P.poetx_cnp_workspace_bytes(nblk, b, 1)), dev)
    for _ in range(5):
        P.poetx_cnp_fwd(qcat, b, G_bf16=Gb, ws=wsc)
        P.poetx_cnp_bwd(qcat, dG, b, dq, ws=wsc)
    cf, cb = [], []
    for _ in range(50):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        P.poetx_cnp_fwd(qcat, b, G_bf16=Gb, ws=wsc)
        e[1].record()
        P.poetx_cnp_bwd(qcat, dG, b, dq, ws=wsc)
        e[2].record()
        torch.cuda.synchronize()
        cf.append(e[0].elapsed_time(e[1]))
        cb.append(e[1].elapsed_time(e[2]))
    fwd_ms, bwd_ms = statistics.median(cf), statistics.median(cb)
    ffma_peak = 152 * 128 * 2 * pk["sm_max_mhz"] * 1e6 / 1e12  # TFLOP/s, FP32 FFMA
    cnp = {"blocks": nblk, "b": b, "fwd_blocks_per_s": nblk / (fwd_ms * 1e-3),
           "bwd_blocks_per_s": nblk / (bwd_ms * 1e-3),
           "fwd_bwd_blocks_per_s": nblk / ((fwd_ms + bwd_ms) * 1e-3),
           "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
           "roofline": {"bound": "alu", "unit": "TFLOP/s",
                        "fwd_achieved": 3 * b ** 3 * 2 * nblk / (fwd_ms * 1e-3) / 1e12,
                        "bwd_achieved": 8 * b ** 3 * 2 * nblk / (bwd_ms * 1e-3) / 1e12,
                        "peak": ffma_peak,
                        "peak_source": "152 SMs x 128 FP32 lanes x 2 flop x max SM clock"}}
    del dG, Gb, wsc

    check_err("CNP timing")
    # amortised set-up stages, timed on their own (merge once per permutation draw, the int8
    # quantiser once per weight): every launch reads and writes the whole weight
    def median_us(fn, reps=20):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)
    setup = {}
    W0s = torch.randn(n, m, device=dev).to(bf)
    Wps = torch.empty_like(W0s)
    us = median_us(lambda: P.poetx_merge_perm(W0s, pn, pm, Wps))
    by = 2.0 * n * m * esz
    setup["merge_perm"] = {"us": us, "bytes": by, "gbs": by / (us * 1e-6) / 1e9,
                           "frac_of_hbm": by / (us * 1e-6) / 1e9 / pk["hbm_gbs"]}
    W32s = torch.randn(n, m, device=dev)
    Wqs = torch.empty(n, m, dtype=torch.int8, device=dev)
    ss = torch.empty(n, device=dev)
    us = median_us(lambda: P.poetx_quantize_rows_int8(W32s, Wqs, ss))
    by = 5.0 * n * m
    setup["quantize_rows_int8"] = {"us": us, "bytes": by, "gbs": by / (us * 1e-6) / 1e9,
                                   "frac_of_hbm": by / (us * 1e-6) / 1e9 / pk["hbm_gbs"]}
    del W0s, Wps, W32s, Wqs, ss
    check_err("merge/quantise timing")
    # merge-then-reinitialize of the benchmarked layer: W0_new = R W0 P in fp32 (two batched
    # block products of 2 n m b flops each on the CUDA cores, the CNP and two index passes)
    W0n = torch.empty(n, m, device=dev)
    mws = P.workspace(P.poetx_merge_reinit_workspace_bytes(main_b["L"]), dev)
    us = median_us(lambda: P.poetx_merge_reinit(main_b["L"], W0n, mws))
    fl = 4.0 * n * m * b
    setup["merge_reinit"] = {"us": us, "flops": fl, "tflops_fp32": fl / (us * 1e-6) / 1e12,
                             "note": "fp32 FFMA products (CUDA cores) + CNP + permutation "
                                     "inverse and gather; runs once per many steps"}
    del W0n, mws
    check_err("merge_reinit timing")
    # the optimizer step on the layer's packed triangles (after the backward of every step;
    # reads q, dq, m, v and writes q, m, v: 28 bytes per parameter)
    npar = qR.numel() + qP.numel()
    oq = torch.zeros(npar, device=dev)
    og, om, ov = torch.randn_like(oq), torch.zeros_like(oq), torch.zeros_like(oq)
    us = median_us(lambda: P.poetx_adam_triu(oq, og, om, ov, 1, 1e-3))
    by = 28.0 * npar
    setup["adam_triu"] = {"us": us, "params": npar, "bytes": by,
                          "gbs": by / (us * 1e-6) / 1e9,
                          "frac_of_hbm": by / (us * 1e-6) / 1e9 / pk["hbm_gbs"],
                          "note": "per training step, not part of the timed layer step"}
    del oq, og, om, ov
    # the backward followed by the optimizer on both sides, against the backward with the
    # update applied by the gradient pack (poetx_layer_bwd_adam); on copies of q, so the
    # benchmarked layer is left as it was
    qRo, qPo = qR.clone(), qP.clone()
    Lo = P.make_layer(m, n, b, acode, wcode, P.FAST if variant == "fast" else P.MEM, pm, pn,
                      Wp, qRo, qPo, w_scale)
    st = {k: torch.zeros_like(qRo if k[1] == "R" else qPo) for k in ("mR", "vR", "mP", "vP")}
    Bo = main_b
    P.poetx_layer_fwd(Lo, x, Bo["y"], Bo["saved"], Bo["wsf"])

    def bwd_then_adam():
        P.poetx_layer_bwd(Lo, x, dy, Bo["saved"], Bo["dx"], Bo["dqR"], Bo["dqP"], Bo["wsb"])
        P.poetx_adam_triu(qRo, Bo["dqR"], st["mR"], st["vR"], 1, 1e-3)
        P.poetx_adam_triu(qPo, Bo["dqP"], st["mP"], st["vP"], 1, 1e-3)

    def bwd_adam():
        P.poetx_layer_bwd_adam(Lo, x, dy, Bo["saved"], Bo["dx"], Bo["dqR"], Bo["dqP"], Bo["wsb"],
                               st["mR"], st["vR"], st["mP"], st["vP"], 1, 1e-3)
    t_sep = median_us(bwd_then_adam)
    t_fused = median_us(bwd_adam)
    setup["bwd_with_optimizer"] = {
        "bwd_then_adam_us": t_sep, "bwd_adam_fused_us": t_fused,
        "note": "eager, L2 flushed: poetx_layer_bwd + poetx_adam_triu on each side vs "
                "poetx_layer_bwd_adam (the same bits; two launches fewer)"}
    del qRo, qPo, st, Lo

    check_err("adam timing")
    # every layer of a multi-layer workload (on request): the metric of such a workload is
    # N / (sum of the layers' step times)
    block = None
    if args.all_layers and len(wl.layers) > 1:
        per = []
        for li, ly in enumerate(wl.layers):
            li_inp = inputs.layer_inputs(wl, ly)
            lx = t(li_inp["x"], bf)
            ldy = t(li_inp["dy"], bf)
            lpm = t(li_inp["perm_m"], torch.int32)
            lpn = t(li_inp["perm_n"], torch.int32)
            lqR = t(li_inp["q_R"], torch.float32)
            lqP = t(li_inp["q_P"], torch.float32)
            lsc = None
            if wl.wdt == "i8":
                lW32 = t(li_inp["W0"], torch.float32)
                lWq = torch.empty(ly.n, ly.m, dtype=torch.int8, device=dev)
                ls = torch.empty(ly.n, device=dev)
                P.poetx_quantize_rows_int8(lW32, lWq, ls)
                lWp, lsc = merged_weight(P, lWq, lpn, lpm, b, ls)
                del lW32
            else:
                lW0 = t(li_inp["W0"], bf)
                lWp, _ = merged_weight(P, lW0, lpn, lpm, b)
                del lW0
            LL = P.make_layer(ly.m, ly.n, b, acode, wcode, P.FAST if variant == "fast" else P.MEM,
                              lpm, lpn, lWp, lqR, lqP, lsc)
            LB = dict(L=LL, saved=P.workspace(P.poetx_layer_saved_bytes(LL, N), dev),
                      wsf=P.workspace(P.poetx_layer_workspace_bytes(LL, N, 0), dev),
                      wsb=P.workspace(P.poetx_layer_workspace_bytes(LL, N, 1), dev),
                      y=torch.empty(N, ly.n, dtype=bf, device=dev),
                      dx=torch.empty(N, ly.m, dtype=bf, device=dev),
                      dqR=torch.empty_like(lqR), dqP=torch.empty_like(lqP))

            def lstep(B=LB, xx=lx, dyy=ldy):
                P.poetx_layer_fwd(B["L"], xx, B["y"], B["saved"], B["wsf"])
                P.poetx_layer_bwd(B["L"], xx, dyy, B["saved"], B["dx"], B["dqR"], B["dqP"],
                                  B["wsb"])
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for _ in range(3):
                    lstep()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            lg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(lg):
                lstep()
            torch.cuda.synchronize()
            lms, _ = timed_steps(None, max(20, args.steps // 20), 5, lg)
            per.append({"m": ly.m, "n": ly.n, "ms_per_step": statistics.mean(lms)})
            del LB, lg, lx, ldy, lWp
            torch.cuda.empty_cache()
        tot = sum(pl["ms_per_step"] for pl in per)
        block = {"layers": per, "ms_per_step": tot, "tokens_per_s": N / (tot * 1e-3),
                 "metric": "N / sum of the layers' fwd+bwd step times"}

    check_err("per-layer timing")
    # end to end through the C ABI with host buffers (pinned), copies inside the timed region:
    # one poetx_layer_step_host call per step, which uploads x and dy, runs the forward and
    # the backward and downloads y, dx, dq_R and dq_P, the copies on its own copy stream
    # beside the kernels
    hx = x.cpu().pin_memory()
    hdy = dy.cpu().pin_memory()
    hy = torch.empty(N, n, dtype=bf).pin_memory()
    hdx = torch.empty(N, m, dtype=bf).pin_memory()
    hqR = torch.empty(qR.shape).pin_memory()
    hqP = torch.empty(qP.shape).pin_memory()
    B = main_b
    step_dev = P.workspace(P.poetx_layer_step_host_bytes(B["L"], N), dev)
    e2e_ms = []
    for i in range(max(3, args.warmup // 4) + 50):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        P.poetx_layer_step_host(B["L"], hx, hdy, hy, hdx, hqR, hqP, step_dev)
        e1.record()
        torch.cuda.synchronize()
        if i >= max(3, args.warmup // 4):
            e2e_ms.append(e0.elapsed_time(e1))
    del step_dev
    # the host link's own rate, for the e2e figure: pinned copies of the step's sizes alone
    link = {}
    hbuf = torch.empty(max(h2d_bytes_of(x, dy), 1), dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(hbuf.numel(), dtype=torch.uint8, device=dev)
    for kind in ("h2d", "d2h"):
        ts = []
        for i in range(13):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record()
            if kind == "h2d":
                dbuf.copy_(hbuf, non_blocking=True)
            else:
                hbuf.copy_(dbuf, non_blocking=True)
            c1.record()
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(c0.elapsed_time(c1))
        link[kind + "_gbs"] = hbuf.numel() / (statistics.median(ts) * 1e-3) / 1e9
    del hbuf, dbuf
    e2e_t = statistics.mean(e2e_ms)
    h2d = (x.numel() + dy.numel()) * esz
    d2h = (N * n + N * m) * esz + (qR.numel() + qP.numel()) * 4
    if world > 1:
        tt = torch.tensor([e2e_t], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e2e_t = float(tt.item())
    assert P.poetx_get_device_error() == 0, "device error word set"

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline(wl)
        except Exception as ex:  # reported, not fatal
            cpu = {"error": str(ex)[:300]}

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.act, "data": "synthetic (seeded Philox inputs, shapes and "
                                     "distributions of the workload)",
            "config": {"workload": wl.name, "m": m, "n": n, "b": b, "tokens_per_gpu": N,
                       "variant": variant, "wdt": wl.wdt, "fusion": args.fusion == "on",
                       "overlap": args.overlap == "on",
                       "parallelism": f"replicas x{world} (token-sharded, no collective)",
                       "l2": "flushed between timed steps (512 MiB memset outside the events)"},
            "variants": {variant: {"tokens_per_s": N / (ms_step * 1e-3), "ms_per_step": ms_step,
                                   "ms_percentiles": ms_pct},
                         **other},
            "eager": eager,
            "timing": "CUDA-graph replay of the step's C-ABI calls (captured once); 'eager' is "
                      "the same step launched from the host each time",
            "cnp": cnp, "stages": stages, "hbm_stages": hbm, "roofline": roofline,
            "setup": setup, **({"block": block} if block else {}),
            "cpu_baseline": cpu,
            "e2e": {"value": world * N / (e2e_t * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_t,
                    "link": {**{k: round(v, 1) for k, v in link.items()},
                             "traffic_gbs": (h2d + d2h) / (e2e_t * 1e-3) / 1e9,
                             "note": "one pinned copy of the step's upload size alone, each "
                                     "direction; the step moves h2d + d2h bytes"},
                    "note": "one poetx_layer_step_host call per step (pinned host buffers): "
                            "x and dy up, forward, backward, y, dx, dq_R and dq_P down; the "
                            "library's copy stream overlaps the x upload with the CNP "
                            "forward, dy's with the forward chain, y's download with the "
                            "backward and dx's with the CNP backward"},
            "gpu_launches": launches, "gpu_launches_per_step": kernels_per_step,
            "clocks": clocks.summary(w0, w1),
        }
        print(json.dumps(out))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
