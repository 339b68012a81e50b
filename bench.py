#!/usr/bin/env python3
"""Benchmark of the POET-X layer training step on GB300.

A step is one pass of the whole hot path over one batch of synthetic tokens, for every
linear of the workload: both Cayley-Neumann forwards, the layer forward, the layer backward
and both Cayley-Neumann backwards (through the C ABI), then the data-parallel exchange of
the parameter gradients (one sum all-reduce over ranks when N > 1) and the Adam update of
the packed triangles.  The default workload is the seven linears of a Llama-8B block
(q/k/v/o 4096 x 4096, gate/up 4096 -> 14336, down 14336 -> 4096, b = 256, N = 8192 bf16
tokens per GPU, fast variant): forward of the seven layers in order, backward in reverse
order; tokens/s = N / step time.  The other workloads (the Llama-1B-shaped layer, the fp32
layer, the 4096-wide block-size sweep, the Llama-13B int8 MLP) are timed after it as short
extra lines.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--variant fast|mem] [--no-extra] [--no-cpu-baseline]

N > 1 runs under torchrun: one rank per GPU on its own N tokens (weak scaling) with the
gradient exchange in every step; the timing is the max over ranks.  --impl reference times
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
NOMINAL_TF32_PER_BF16 = 1.1 / 2.25  # dense tensor-core rates, tf32 : bf16 (nominal)
ADAM_LR = 1e-3


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b_block")
    ap.add_argument("--variant", default=None, choices=["fast", "mem"],
                    help="default: the workload's first variant (fast; mem for int8 weights)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the short lines of the other workloads")
    ap.add_argument("--fusion", default="on", choices=["on", "off", "wprime", "bwd"],
                    help="fused kernels: on (all), off, wprime (W' contraction + the block "
                         "product after it only), bwd (backward block product + weight "
                         "gradient only)")
    ap.add_argument("--overlap", default="on", choices=["on", "off"],
                    help="dx scatter on a side stream beside the CNP backward (library switch)")
    ap.add_argument("--group", default="on", choices=["on", "off"],
                    help="run the workload's layers as one layer group (one batched CNP "
                         "forward and backward per step; default) or layer by layer")
    ap.add_argument("--layers", default=None,
                    help="comma-separated names of the workload's layers to keep (profiling "
                         "cases, e.g. --layers gate)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (profiling cases)")
    ap.add_argument("--launches-only", action="store_true",
                    help="build the workload, run --warmup then --steps eager fwd+bwd steps and "
                         "exit (a short, fixed launch sequence for an ncu capture); prints the "
                         "launches before the timed steps and per step")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained") or d["bf16_tflops"],
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
# One oracle step over every layer of the workload on a sample of its tokens: both CNP
# forwards, the layer forward and backward, both CNP backwards (the fp64 oracle as it stands).
CPU_SNIPPET = r"""
import json, os, sys, time
sys.path.insert(0, %(root)r)
import numpy as np
import oracle as O
from orthogonal_reparameterized_gb300 import inputs
wl = inputs.WORKLOADS[%(wl)r]
layers = []
for layer in wl.layers:
    inp = inputs.layer_inputs(wl, layer, N=%(ntok)d)
    W = inp["W0"]
    if wl.wdt == "i8":
        W = O.dequantize_rows(*O.quantize_rows_int8(W))
    # the per-block oracle when b does not divide a side (ragged last block)
    f = O.poetx_layer if layer.m %% wl.b == 0 and layer.n %% wl.b == 0 else O.poetx_layer_ragged
    layers.append((f, inp, W))
times = []
t_end = time.perf_counter() + %(budget)f
while True:
    t0 = time.perf_counter()
    for f, inp, W in layers:
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
                       timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed: " + r.stderr[-2000:])
    times = json.loads(r.stdout.strip().splitlines()[-1])["times"]
    return times, cores


def oracle_sample_tokens(wl):
    # the oracle's cost is the CNP of every block (fixed) plus the products (per token):
    # ~10-30 s of CPU work per sampled step on a 16-core host
    return 128 if len(wl.layers) > 1 else 512


def cpu_baseline(wl):
    ntok = oracle_sample_tokens(wl)
    times, cores = run_oracle_sample(wl.name, ntok, reps=3, budget_s=30.0)
    t = statistics.median(times)
    return {"value": ntok / t, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 numpy oracle, one full step (CNP fwd of both sides, layer "
                      f"fwd+bwd, CNP bwd of both sides) of each of the {len(wl.layers)} "
                      f"layer(s) of {wl.name} on {ntok} of its {wl.N} tokens, median of "
                      f"{len(times)} runs", "seconds_per_sample": t}


# ------------------------------------------------------------------ reference arm
def reference_arm(args, rank, world):
    from orthogonal_reparameterized_gb300 import inputs
    if rank != 0:
        return
    wl = inputs.WORKLOADS[args.workload]
    ntok = oracle_sample_tokens(wl)
    total = max(1, args.steps) + max(0, args.warmup)
    times, cores = run_oracle_sample(wl.name, ntok, reps=total, budget_s=150.0)
    timed = times[args.warmup:] if len(times) > args.warmup else times
    t = statistics.mean(timed)
    val = ntok / t
    variant = args.variant or ("mem" if wl.wdt == "i8" else wl.variants[0])
    out = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": len(timed), "warmup": min(args.warmup, len(times)),
           "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": wl.name, "layers": [[l.m, l.n] for l in wl.layers],
                      "b": wl.b, "tokens_per_step": ntok, "variant": variant},
           "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": f"{ntok} tokens through every layer of {wl.name} per "
                                      f"step"},
           "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    if len(timed) < args.steps:
        out["note"] = (f"time budget reached after {len(times)} oracle steps (each step is "
                       f"one bounded sample of the workload)")
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


def padded(d, b):
    return -(-d // b) * b


def hbm_sides(direction, variant, stage):
    """The activation width ('m' or 'n') of each successive launch of an HBM-bound stage in
    one layer call, in launch order (block-diagonal products absorbed by the fused W'
    kernel are simply not launched)."""
    if direction == "fwd":
        return {"perm_gather": "m", "blockdiag_mm": "mn", "perm_scatter": "n"}.get(stage, "")
    # backward: the block products and weight gradients, fused (blockdiag_bwd_fused, P side
    # then R side) or separate, in launch order
    if variant == "fast":
        return {"perm_gather": "n", "blockdiag_wgrad": "nm", "blockdiag_mm": "nm",
                "blockdiag_bwd_fused": "nm", "perm_scatter": "m"}.get(stage, "")
    return {"perm_gather": "mn", "blockdiag_wgrad": "nm", "blockdiag_mm": "mnm",
            "blockdiag_bwd_fused": "nm", "perm_scatter": "m"}.get(stage, "")


class Rig:
    """Every tensor of one workload on the device: per layer the inputs (drawn on the device),
    the merged weight, the descriptor and the outputs; the parameters q, their gradients dq
    and the Adam state of all layers in flat buffers.  With group=True (the default) the
    layers form one layer group: one saved buffer and one workspace for the group, one CNP
    forward and one CNP backward over every block of every layer per step.  Otherwise each
    layer runs poetx_layer_fwd / poetx_layer_bwd with its own saved buffer and a shared
    forward and backward workspace."""

    def __init__(self, P, wl, variant, dev, N=None, group=True):
        import torch
        from orthogonal_reparameterized_gb300 import dp, inputs
        self.P, self.wl, self.variant, self.dev, self.group = P, wl, variant, dev, group
        self.N = N = wl.N if N is None else N
        self.bf = torch.bfloat16 if wl.act == "bf16" else torch.float32
        self.esz = 2 if wl.act == "bf16" else 4
        b = wl.b
        acode = P.BF16 if wl.act == "bf16" else P.F32
        vcode = P.FAST if variant == "fast" else P.MEM
        tri = b * (b - 1) // 2
        shapes = []
        for i, ly in enumerate(wl.layers):
            shapes += [(f"{i}R", (-(-ly.m // b), tri)), (f"{i}P", (-(-ly.n // b), tri))]
        self.q = dp.FlatBuffer(shapes, dev)
        self.dq = dp.FlatBuffer(shapes, dev)
        self.adam_m = dp.FlatBuffer(shapes, dev)
        self.adam_v = dp.FlatBuffer(shapes, dev)
        self.layers = []
        wsf = wsb = 16
        for i, ly in enumerate(wl.layers):
            inp = inputs.device_layer_inputs(wl, ly, dev, N=N)
            self.q.view(f"{i}R").copy_(inp["q_R"])
            self.q.view(f"{i}P").copy_(inp["q_P"])
            w_scale = None
            if wl.wdt == "i8":
                Wq = torch.empty(ly.n, ly.m, dtype=torch.int8, device=dev)
                s = torch.empty(ly.n, device=dev)
                P.poetx_quantize_rows_int8(inp["W0"], Wq, s)
                Wp, w_scale = merged_weight(P, Wq, inp["perm_n"], inp["perm_m"], b, s)
                wcode = P.I8
                del Wq, s
            else:
                Wp, _ = merged_weight(P, inp["W0"], inp["perm_n"], inp["perm_m"], b)
                wcode = P.BF16 if wl.wdt == "bf16" else P.F32
            del inp["W0"]
            L = P.make_layer(ly.m, ly.n, b, acode, wcode, vcode, inp["perm_m"], inp["perm_n"],
                             Wp, self.q.view(f"{i}R"), self.q.view(f"{i}P"), w_scale)
            d = dict(shape=ly, L=L, x=inp["x"], dy=inp["dy"], pm=inp["perm_m"],
                     pn=inp["perm_n"], Wp=Wp, w_scale=w_scale,
                     y=torch.empty(N, ly.n, dtype=self.bf, device=dev),
                     dx=torch.empty(N, ly.m, dtype=self.bf, device=dev),
                     dqR=self.dq.view(f"{i}R"), dqP=self.dq.view(f"{i}P"))
            if not group:
                d["saved"] = P.workspace(P.poetx_layer_saved_bytes(L, N), dev)
                wsf = max(wsf, P.poetx_layer_workspace_bytes(L, N, 0))
                wsb = max(wsb, P.poetx_layer_workspace_bytes(L, N, 1))
            self.layers.append(d)
        if group:
            self.G = P.make_group([d["L"] for d in self.layers])
            self.gsaved = P.workspace(P.poetx_group_saved_bytes(self.G, N), dev)
            self.gws = P.workspace(P.poetx_group_workspace_bytes(self.G, N), dev)
            self.dqR_list = [d["dqR"] for d in self.layers]
            self.dqP_list = [d["dqP"] for d in self.layers]
        else:
            self.wsf = P.workspace(wsf, dev)
            self.wsb = P.workspace(wsb, dev)
        self.adam_step = 1

    def calls(self):
        """The step's library calls in order: (kind, layer index)."""
        n = len(self.layers)
        c = [("fwd", i) for i in range(n)] + [("bwd", i) for i in reversed(range(n))]
        return ([("cnp_fwd", -1)] + c + [("cnp_bwd", -1)]) if self.group else c

    def run(self, kind, i):
        P = self.P
        if kind == "cnp_fwd":
            P.poetx_group_cnp_fwd(self.G, self.N, self.gsaved)
        elif kind == "cnp_bwd":
            P.poetx_group_cnp_bwd(self.G, self.N, self.gsaved, self.dqR_list, self.dqP_list,
                                  self.gws)
        elif kind == "fwd":
            d = self.layers[i]
            if self.group:
                P.poetx_group_layer_fwd(self.G, i, d["x"], d["y"], self.gsaved, self.gws)
            else:
                P.poetx_layer_fwd(d["L"], d["x"], d["y"], d["saved"], self.wsf)
        else:
            d = self.layers[i]
            if self.group:
                P.poetx_group_layer_bwd(self.G, i, d["x"], d["dy"], self.gsaved, d["dx"], self.gws)
            else:
                P.poetx_layer_bwd(d["L"], d["x"], d["dy"], d["saved"], d["dx"], d["dqR"],
                                  d["dqP"], self.wsb)

    def compute(self):
        """Forward of every layer in order, backward in reverse order (with the group: the
        CNP forward of every block first, the CNP backward of every block last)."""
        for kind, i in self.calls():
            self.run(kind, i)

    def update(self):
        """Adam on every layer's packed triangles (one launch over the flat buffers)."""
        self.P.poetx_adam_triu(self.q.flat, self.dq.flat, self.adam_m.flat, self.adam_v.flat,
                               self.adam_step, ADAM_LR)

    def nblk(self):
        b = self.wl.b
        return sum(-(-d["shape"].m // b) + -(-d["shape"].n // b) for d in self.layers)

    def wprime_flops(self):
        """Flops of the W' contractions of one step: forward, backward (and the mem
        variant's recomputation), 2 N m n each at the padded widths."""
        b, N = self.wl.b, self.N
        per = 3 if self.variant == "mem" else 2
        return sum(per * 2.0 * N * padded(d["shape"].m, b) * padded(d["shape"].n, b)
                   for d in self.layers)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return

    import torch
    import torch.distributed as dist

    from orthogonal_reparameterized_gb300 import dp, inputs
    import orthogonal_reparameterized_gb300.poetx as P

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    P.lib()
    P.poetx_set_fusion({"on": 3, "off": 0, "wprime": 1, "bwd": 2}[args.fusion])
    P.poetx_set_overlap(args.overlap == "on")
    pk = peaks()

    def check_err(section):
        """Fail loudly, naming the section, if a kernel recorded an error (a bounded wait
        that expired): no number is reported from such a run."""
        st = P.poetx_get_device_error()
        if st != 0:
            raise RuntimeError(f"device error after {section}: {P.status_str(st)} "
                               f"(wait site {P.poetx_timeout_site()})")

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def graph_of(fn):
        """CUDA graph of fn's C-ABI calls (warmed up on a side stream first)."""
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(2):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        c0 = P.poetx_launch_count()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g, P.poetx_launch_count() - c0

    def timed(run, K, W, barrier=False):
        """K timed runs after W untimed ones; the L2 is flushed (outside the events) before
        every timed run.  Returns the per-run milliseconds and the wall-clock region."""
        for _ in range(W):
            run()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        if barrier and world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        w0 = time.time()
        for e0, e1 in evs:
            flush.zero_()
            e0.record()
            run()
            e1.record()
        torch.cuda.synchronize()
        w1 = time.time()
        if barrier and world > 1:
            dist.barrier()
        return [e0.elapsed_time(e1) for e0, e1 in evs], (w0, w1)

    def max_over_ranks(v):
        if world == 1:
            return v
        tt = torch.tensor([v], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        return float(tt.item())

    # ---------------------------------------------------------------- the headline workload
    wl = inputs.WORKLOADS[args.workload]
    if args.layers:
        import dataclasses
        keep = args.layers.split(",")
        wl = dataclasses.replace(wl, layers=tuple(l for l in wl.layers if l.name in keep))
        if not wl.layers:
            raise SystemExit(f"--layers {args.layers}: no such layer in {args.workload}")
    variant = args.variant or ("mem" if wl.wdt == "i8" else wl.variants[0])
    c_setup = P.poetx_launch_count()
    rig = Rig(P, wl, variant, dev, N=args.tokens, group=args.group == "on")
    N = rig.N
    if args.launches_only:
        c0 = P.poetx_launch_count()
        for _ in range(args.warmup):
            rig.compute()
        torch.cuda.synchronize()
        c1 = P.poetx_launch_count()
        for _ in range(args.steps):
            rig.compute()
        torch.cuda.synchronize()
        check_err("eager steps")
        per = (P.poetx_launch_count() - c1) // max(1, args.steps)
        print(json.dumps({"workload": wl.name, "tokens": N, "variant": variant,
                          "launches_before_steps": c1 - c_setup, "setup_launches": c0 - c_setup,
                          "launches_per_step": per}))
        return
    g_compute, k_compute = graph_of(rig.compute)
    g_update, k_update = graph_of(rig.update)
    kernels_per_step = k_compute + k_update

    def train_step():
        dp.data_parallel_step(g_compute.replay, rig.dq.flat, g_update.replay)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms, (w0, w1) = timed(train_step, args.steps, max(3, args.warmup), barrier=True)
    time.sleep(0.3)
    clocks.stop()
    ms_step = max_over_ranks(statistics.mean(ms))
    qs = statistics.quantiles(ms, n=10) if len(ms) >= 10 else [min(ms)] * 9
    ms_pct = {"p10": qs[0], "p50": statistics.median(ms), "p90": qs[8]}
    value = world * N / (ms_step * 1e-3)
    check_err("graph-replayed steps")

    # fwd + bwd alone (the metric's own step, without the exchange and the optimizer)
    fb_ms, _ = timed(g_compute.replay, max(20, args.steps // 4), 3)
    fwd_bwd = {"tokens_per_s": N / (statistics.mean(fb_ms) * 1e-3),
               "ms_per_step": statistics.mean(fb_ms)}
    # the same fwd + bwd issued eagerly (host launches through the C ABI)
    ems, _ = timed(rig.compute, max(10, args.steps // 10), 3)
    eager = {"tokens_per_s": N / (statistics.mean(ems) * 1e-3),
             "ms_per_step": statistics.mean(ems)}
    check_err("eager steps")

    # ---------------------------------------------------------------- per-stage timing
    # library stage events inside the same layer calls (eager, L2 flushed before each step);
    # the side-stream overlap is off while stage events are on
    P.poetx_profile_enable(True)
    P.poetx_profile_collect()
    prof_steps = 5
    stage_ms, per_layer = {}, [0.0] * len(rig.layers)
    wp = {"flops": 0.0, "ms": 0.0, "launches": 0, "fused_launches": 0}
    hbm = {}
    cnp_layer_ms = 0.0
    cnp_stages = ("triu_unpack", "cnp_q2", "cnp_g", "cnp_sum_partials", "cnp_m1", "cnp_qbar",
                  "triu_grad_pack")
    for _ in range(prof_steps):
        flush.zero_()
        torch.cuda.synchronize()
        P.poetx_profile_collect()
        for direction, i in rig.calls():
            rig.run(direction, i)
            recs = P.poetx_profile_collect()
            if i < 0:  # the group's CNP calls
                for name, t_ms in recs:
                    stage_ms.setdefault(name, []).append(t_ms)
                    cnp_layer_ms += t_ms
                continue
            ly = rig.layers[i]["shape"]
            width = {"m": padded(ly.m, wl.b), "n": padded(ly.n, wl.b)}
            seen = {}
            for name, t_ms in recs:
                stage_ms.setdefault(name, []).append(t_ms)
                per_layer[i] += t_ms
                k = seen.get(name, 0)
                seen[name] = k + 1
                if name in cnp_stages:
                    cnp_layer_ms += t_ms
                if name in ("wprime_gemm", "wprime_blockdiag_fused"):
                    f = 2.0 * N * width["m"] * width["n"]
                    if name == "wprime_blockdiag_fused":
                        f += 2.0 * N * width["n" if direction == "fwd" else "m"] * wl.b
                        wp["fused_launches"] += 1
                    wp["flops"] += f
                    wp["ms"] += t_ms
                    wp["launches"] += 1
                sides = hbm_sides(direction, variant, name)
                if k < len(sides):
                    D = width[sides[k]]
                    # one [N, D] activation read, one written (the fused backward kernel
                    # reads two: the upstream gradient and the forward's activation)
                    by = (3.0 if name == "blockdiag_bwd_fused" else 2.0) * N * D * rig.esz
                    h = hbm.setdefault(name, {"bytes": 0.0, "ms": 0.0, "launches": 0})
                    h["bytes"] += by
                    h["ms"] += t_ms
                    h["launches"] += 1
    P.poetx_profile_enable(False)
    stages = {k: {"launches_per_step": len(v) / prof_steps, "ms_per_step": sum(v) / prof_steps,
                  "ms_per_launch": sum(v) / len(v)} for k, v in stage_ms.items()}
    hbm_stages = {k: {"algorithmic_bytes_per_launch": v["bytes"] / v["launches"],
                      "achieved_gbs": v["bytes"] / (v["ms"] * 1e-3) / 1e9,
                      "frac_of_hbm": v["bytes"] / (v["ms"] * 1e-3) / 1e9 / pk["hbm_gbs"],
                      "launches_per_step": v["launches"] / prof_steps}
                  for k, v in hbm.items()}
    check_err("per-stage timing")

    # the dominant kernel: the tcgen05 W' contraction (2-CTA pair tiles at these shapes, or
    # fused with the block-diagonal product after it on single-CTA tiles); achieved = its
    # algorithmic flops per launch / its average launch time, over every launch of a step
    w_ms_launch = wp["ms"] / wp["launches"] if wp["launches"] else None
    w_flops_launch = wp["flops"] / wp["launches"] if wp["launches"] else None
    achieved = (w_flops_launch / (w_ms_launch * 1e-3) / 1e12) if w_ms_launch else None
    traffic = None
    prof_json = os.path.join(ROOT, "profiles", f"wprime_traffic_{wl.name}.json")
    if os.path.exists(prof_json):
        try:
            import hashlib
            pj = json.load(open(prof_json))
            src = open(os.path.join(ROOT, "orthogonal_reparameterized_gb300", "csrc",
                                    "umma_gemm.cu"), "rb").read()
            if pj.get("kernel_source_sha256") == hashlib.sha256(src).hexdigest():
                traffic = pj.get("dram_bytes_per_launch")
        except (OSError, ValueError, KeyError):
            traffic = None
    peak_tc = pk["bf16_tflops_sustained"]
    roofline = {
        "kernel": "umma_gemm_kernel / umma_fused_kernel: the tcgen05 W' contraction "
                  "(fwd B = A W'^T, bwd dA = dB W'; 2 N m n flops per launch, + 2 N n b where "
                  "the block-diagonal product after it is fused in), every launch of a step",
        "bound": "tensor", "achieved": achieved, "peak": peak_tc, "unit": "TFLOP/s",
        "frac": (achieved / peak_tc) if achieved else None, "traffic": traffic,
        "flops_per_launch": w_flops_launch, "ms_per_launch": w_ms_launch,
        "launches_per_step": wp["launches"] / prof_steps,
        "frac_of_burst": (achieved / pk["bf16_tflops"]) if achieved else None,
        "peak_source": f"{pk['source']} dense bf16, sustained (the kernel is timed inside a "
                       f"multi-millisecond step run back to back); burst "
                       f"{pk['bf16_tflops']} TFLOP/s given as frac_of_burst"}

    # ---------------------------------------------------------------- CNP of every block
    b = wl.b
    nblk = rig.nblk()
    qcat = torch.cat([rig.q.view(k).reshape(-1, b * (b - 1) // 2) for k in rig.q.names()], 0)
    cnp = cnp_measure(P, torch, qcat, b, flush, pk, dev)
    cnp["in_step_ms"] = cnp_layer_ms / prof_steps
    check_err("CNP timing")

    # ---------------------------------------------------------------- amortised set-up stages
    setup = setup_measure(P, torch, rig, flush, pk, dev)
    check_err("set-up timing")

    # ---------------------------------------------------------------- end to end
    e2e = e2e_measure(P, torch, rig, args, world, dev, flush)
    e2e["value"] = world * N / (max_over_ranks(e2e["ms_per_step"]) * 1e-3)
    check_err("end-to-end steps")

    # ---------------------------------------------------------------- other workloads
    extra = {}
    if not args.no_extra:
        del g_compute, g_update
        keep = {"tokens_per_s": value, "ms_per_step": ms_step}
        rig_layers = len(rig.layers)
        del rig
        torch.cuda.empty_cache()
        for name in ("llama1b_2048", "fp32_256_b32", "sweep_4096_b64", "sweep_4096_b128",
                     "sweep_4096_b256", "sweep_4096_b512", "llama13b_mlp_int8",
                     "ragged_2000_b256"):
            if name == wl.name:
                continue
            try:
                extra[name] = extra_measure(P, torch, inputs.WORKLOADS[name], dev, flush, pk,
                                            graph_of, timed)
            except Exception as ex:  # reported, not fatal
                extra[name] = {"error": str(ex)[:300]}
            torch.cuda.empty_cache()
            check_err(f"extra workload {name}")
        extra[wl.name] = {"variants": {variant: keep}, "layers": rig_layers}

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
            "dtype": wl.act, "data": "synthetic (seeded Philox draws on the device, shapes and "
                                     "distributions of the workload)",
            "config": {"workload": wl.name,
                       "layers": [{"name": ly.name, "m": ly.m, "n": ly.n} for ly in wl.layers],
                       "b": wl.b, "tokens_per_gpu": N, "variant": variant, "wdt": wl.wdt,
                       "fusion": args.fusion, "overlap": args.overlap == "on",
                       "layer_group": args.group == "on",
                       "parallelism": (f"data parallel x{world}: token-sharded, one sum "
                                       f"all-reduce of dq per step") if world > 1 else
                                      "one GPU",
                       "step": "fwd of every layer, bwd in reverse order, dq exchange (N > 1), "
                               "Adam on the packed triangles",
                       "l2": "flushed between timed steps (512 MiB memset outside the events); "
                             "the step's inputs are also far larger than L2"},
            "ms_percentiles": ms_pct, "fwd_bwd": fwd_bwd, "eager": eager,
            "timing": "CUDA-graph replay of the step's C-ABI calls (captured once); "
                      "'fwd_bwd' is the layer calls alone, 'eager' the same launched from "
                      "the host each time",
            "per_layer_ms": [{"name": wl.layers[i].name, "ms": per_layer[i] / prof_steps}
                             for i in range(len(wl.layers))],
            "roofline": roofline, "cnp": cnp, "stages": stages, "hbm_stages": hbm_stages,
            "setup": setup, "workloads": extra, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": kernels_per_step * args.steps,
            "gpu_launches_per_step": kernels_per_step,
            "clocks": clocks.summary(w0, w1),
        }
        print(json.dumps(out))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def cnp_measure(P, torch, qcat, b, flush, pk, dev, reps=30):
    """Standalone CNP forward (bf16 G out) and backward over the given packed triangles; the
    tensor-core products do 4 b^3 (forward: Q^2, then Q^2 (2Q + Q^2)) and 8 b^3 (backward:
    the two two-segment products) flops per block, each as three tf32 passes."""
    nblk = qcat.shape[0]
    Gb = torch.empty(nblk, b, b, dtype=torch.bfloat16, device=dev)
    dG = torch.randn(1, nblk, b, b, device=dev)
    dq = torch.empty_like(qcat)
    wsc = P.workspace(max(P.poetx_cnp_workspace_bytes(nblk, b, 0),
                          P.poetx_cnp_workspace_bytes(nblk, b, 1)), dev)
    for _ in range(3):
        P.poetx_cnp_fwd(qcat, b, G_bf16=Gb, ws=wsc)
        P.poetx_cnp_bwd(qcat, dG, b, dq, ws=wsc)
    cf, cb = [], []
    for _ in range(reps):
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
    del Gb, dG, dq, wsc
    tf32_eff = pk["bf16_tflops"] * NOMINAL_TF32_PER_BF16 / 3.0
    f_fl, b_fl = 4.0 * b ** 3 * nblk, 8.0 * b ** 3 * nblk
    fa = f_fl / (fwd_ms * 1e-3) / 1e12
    ba = b_fl / (bwd_ms * 1e-3) / 1e12
    # HBM bytes the CNP must move: q in (b(b-1)/2 fp32), G out (bf16 b^2) and the Q, Q^2 kept
    # for the backward (fp32 2 b^2); backward: q, Q, Q^2 and one dG partial in, dq out
    tri = b * (b - 1) // 2
    fby = nblk * (4.0 * tri + 2.0 * b * b + 8.0 * b * b)
    bby = nblk * (4.0 * tri + 12.0 * b * b + 4.0 * tri)
    return {"blocks": nblk, "b": b, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "fwd_blocks_per_s": nblk / (fwd_ms * 1e-3), "bwd_blocks_per_s": nblk / (bwd_ms * 1e-3),
            "fwd_bwd_blocks_per_s": nblk / ((fwd_ms + bwd_ms) * 1e-3),
            "roofline": {
                "bound": "tensor", "unit": "TFLOP/s", "fwd_achieved": fa, "bwd_achieved": ba,
                "peak": tf32_eff, "fwd_frac": fa / tf32_eff, "bwd_frac": ba / tf32_eff,
                "flops": "4 b^3 per block forward, 8 b^3 backward (fp32 products; each runs as "
                         "three tf32 tensor-core passes)",
                "peak_source": f"{pk['source']} bf16 burst {pk['bf16_tflops']} TFLOP/s x "
                               f"nominal tf32/bf16 ratio 1.1/2.25, / 3 for the three-pass "
                               f"split"},
            "hbm": {"fwd_gbs": fby / (fwd_ms * 1e-3) / 1e9, "bwd_gbs": bby / (bwd_ms * 1e-3) / 1e9,
                    "fwd_frac_of_hbm": fby / (fwd_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                    "bwd_frac_of_hbm": bby / (bwd_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                    "bytes": "fwd: q in, bf16 G and fp32 Q, Q^2 out; bwd: q, Q, Q^2, one dG "
                             "partial in, dq out"}}


def median_us(torch, flush, fn, reps=20):
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


def setup_measure(P, torch, rig, flush, pk, dev):
    """Amortised set-up stages on the workload's first layer: the permutation merge (once per
    draw), the int8 quantiser (once per weight), merge-then-reinitialize (once per many
    steps) and the Adam step over every layer's packed triangles."""
    d = rig.layers[0]
    ly = d["shape"]
    n, m, b, esz = ly.n, ly.m, rig.wl.b, rig.esz
    setup = {"layer": {"m": m, "n": n}}
    W0s = torch.randn(n, m, device=dev).to(rig.bf)
    Wps = torch.empty_like(W0s)
    us = median_us(torch, flush, lambda: P.poetx_merge_perm(W0s, d["pn"], d["pm"], Wps))
    by = 2.0 * n * m * esz
    setup["merge_perm"] = {"us": us, "bytes": by, "gbs": by / (us * 1e-6) / 1e9,
                           "frac_of_hbm": by / (us * 1e-6) / 1e9 / pk["hbm_gbs"]}
    W32s = torch.randn(n, m, device=dev)
    Wqs = torch.empty(n, m, dtype=torch.int8, device=dev)
    ss = torch.empty(n, device=dev)
    us = median_us(torch, flush, lambda: P.poetx_quantize_rows_int8(W32s, Wqs, ss))
    by = 5.0 * n * m
    setup["quantize_rows_int8"] = {"us": us, "bytes": by, "gbs": by / (us * 1e-6) / 1e9,
                                   "frac_of_hbm": by / (us * 1e-6) / 1e9 / pk["hbm_gbs"]}
    del W0s, Wps, W32s, Wqs, ss
    W0n = torch.empty(n, m, device=dev)
    mws = P.workspace(P.poetx_merge_reinit_workspace_bytes(d["L"]), dev)
    us = median_us(torch, flush, lambda: P.poetx_merge_reinit(d["L"], W0n, mws))
    fl = 2.0 * n * m * b * 2
    setup["merge_reinit"] = {"us": us, "flops": fl, "tflops_fp32": fl / (us * 1e-6) / 1e12,
                             "engine": ("tensor cores, three-pass tf32"
                                        if P.poetx_layer_cuda_core_steps(d["L"], 0) & 1 == 0
                                        else "CUDA cores, fp32"),
                             "note": "the two block-product passes over W' (fp32 accuracy) + "
                                     "the CNP + permutation inverse and gather; once per many "
                                     "steps"}
    del W0n, mws
    npar = rig.q.flat.numel()
    oq = torch.zeros(npar, device=dev)
    og, om, ov = torch.randn_like(oq), torch.zeros_like(oq), torch.zeros_like(oq)
    us = median_us(torch, flush, lambda: P.poetx_adam_triu(oq, og, om, ov, 1, 1e-3))
    by = 28.0 * npar
    setup["adam_triu"] = {"us": us, "params": npar, "bytes": by, "gbs": by / (us * 1e-6) / 1e9,
                          "frac_of_hbm": by / (us * 1e-6) / 1e9 / pk["hbm_gbs"],
                          "note": "every layer's packed triangles, one launch; part of the "
                                  "timed step"}
    del oq, og, om, ov
    return setup


def e2e_measure(P, torch, rig, args, world, dev, flush):
    """End to end through the C ABI with pinned host buffers: every step, one
    poetx_group_step_host call over the workload's layer group (every x and dy up, the
    group's forward and backward, every y, dx, dq_R and dq_P down, the copies on the
    library's upload and download streams beside the kernels), or with --group off one
    poetx_layer_step_host call per layer."""
    from orthogonal_reparameterized_gb300 import dp
    hb = []
    dev_bytes = 16
    for d in rig.layers:
        hb.append(dict(x=d["x"].cpu().pin_memory(), dy=d["dy"].cpu().pin_memory(),
                       y=torch.empty(d["y"].shape, dtype=rig.bf).pin_memory(),
                       dx=torch.empty(d["dx"].shape, dtype=rig.bf).pin_memory(),
                       dqR=torch.empty(d["dqR"].shape).pin_memory(),
                       dqP=torch.empty(d["dqP"].shape).pin_memory()))
        dev_bytes = max(dev_bytes, P.poetx_layer_step_host_bytes(d["L"], rig.N))
    if rig.group:
        dev_bytes = P.poetx_group_step_host_bytes(rig.G, rig.N)
    step_dev = P.workspace(dev_bytes, dev)
    h2d = sum((h["x"].numel() + h["dy"].numel()) * rig.esz for h in hb)
    d2h = sum((h["y"].numel() + h["dx"].numel()) * rig.esz + (h["dqR"].numel() +
              h["dqP"].numel()) * 4 for h in hb)

    def step():
        if rig.group:
            P.poetx_group_step_host(rig.G, [h["x"] for h in hb], [h["dy"] for h in hb],
                                    [h["y"] for h in hb], [h["dx"] for h in hb],
                                    [h["dqR"] for h in hb], [h["dqP"] for h in hb], step_dev)
            return
        for d, h in zip(rig.layers, hb):
            P.poetx_layer_step_host(d["L"], h["x"], h["dy"], h["y"], h["dx"], h["dqR"],
                                    h["dqP"], step_dev)

    warm = 3
    reps = max(10, min(50, args.steps // 4))
    ms = []
    for i in range(warm + reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        step()
        e1.record()
        torch.cuda.synchronize()
        if i >= warm:
            ms.append(e0.elapsed_time(e1))
    del step_dev
    # the host link's own rate: one pinned copy of the step's upload size, each direction
    link = {}
    nb = min(max(h2d, 1), 1 << 30)
    hbuf = torch.empty(nb, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(nb, dtype=torch.uint8, device=dev)
    for kind in ("h2d", "d2h"):
        ts = []
        for i in range(8):
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
        link[kind + "_gbs"] = round(nb / (statistics.median(ts) * 1e-3) / 1e9, 1)
    # both directions at once (an upload and a download on two streams)
    hbuf2 = torch.empty(nb, dtype=torch.uint8).pin_memory()
    dbuf2 = torch.empty(nb, dtype=torch.uint8, device=dev)
    su, sd = torch.cuda.Stream(), torch.cuda.Stream()
    ts = []
    for i in range(8):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        su.wait_stream(torch.cuda.current_stream())
        sd.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(su):
            dbuf.copy_(hbuf, non_blocking=True)
        with torch.cuda.stream(sd):
            hbuf2.copy_(dbuf2, non_blocking=True)
        torch.cuda.current_stream().wait_stream(su)
        torch.cuda.current_stream().wait_stream(sd)
        c1.record()
        torch.cuda.synchronize()
        if i >= 3:
            ts.append(c0.elapsed_time(c1))
    link["both_directions_gbs"] = round(2 * nb / (statistics.median(ts) * 1e-3) / 1e9, 1)
    del hbuf, dbuf, hbuf2, dbuf2
    # the median step: a step's time is the link and the kernels; a few steps in a run take
    # 2-6x longer for host-side reasons (the mean and the 90th percentile are kept beside it)
    t = statistics.median(ms)
    qs = sorted(ms)
    return {"unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": t, "statistic": "median of the timed steps",
            "mean_ms": statistics.mean(ms), "p90_ms": qs[min(len(qs) - 1, int(0.9 * len(qs)))],
            "timed_steps": len(ms),
            "link": {**link, "traffic_gbs": (h2d + d2h) / (t * 1e-3) / 1e9,
                     "note": "one pinned copy of up to 1 GiB alone in each direction, and one "
                             "each way at once; the step moves h2d + d2h bytes"},
            "note": ("per step, one poetx_group_step_host call over the layer group"
                     if rig.group else "per step, one poetx_layer_step_host call per layer") +
                    " (pinned host buffers): x and dy up, forward, backward, y, dx, dq_R and "
                    "dq_P down; the library's upload and download streams overlap the copies "
                    "with the kernels and with each other; bound by the host link when the "
                    "step's bytes / link rate exceed the kernels' time"}


def extra_measure(P, torch, wl, dev, flush, pk, graph_of, timed, steps=30):
    """A short line for another workload: tokens/s of its fwd+bwd step (graph replay, L2
    flushed) in each of its variants, and its CNP blocks/s."""
    out = {"layers": [[l.m, l.n] for l in wl.layers], "b": wl.b, "N": wl.N, "wdt": wl.wdt,
           "variants": {}}
    for variant in (("mem",) if wl.wdt == "i8" else wl.variants):
        rig = Rig(P, wl, variant, dev)
        g, k = graph_of(rig.compute)
        ms, _ = timed(g.replay, steps, 3)
        t = statistics.mean(ms)
        out["variants"][variant] = {"tokens_per_s": rig.N / (t * 1e-3), "ms_per_step": t,
                                    "kernels_per_step": k,
                                    "wprime_tflops_if_all_time": rig.wprime_flops() /
                                    (t * 1e-3) / 1e12}
        if "cnp" not in out:
            b = wl.b
            qcat = torch.cat([rig.q.view(kk).reshape(-1, b * (b - 1) // 2)
                              for kk in rig.q.names()], 0)
            c = cnp_measure(P, torch, qcat, b, flush, pk, dev, reps=10)
            out["cnp"] = {kk: c[kk] for kk in ("blocks", "b", "fwd_ms", "bwd_ms",
                                               "fwd_blocks_per_s", "bwd_blocks_per_s",
                                               "fwd_bwd_blocks_per_s")}
            out["cnp"]["fwd_frac"] = c["roofline"]["fwd_frac"]
            out["cnp"]["bwd_frac"] = c["roofline"]["bwd_frac"]
        del g, rig
        torch.cuda.empty_cache()
    return out


if __name__ == "__main__":
    main()
