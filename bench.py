#!/usr/bin/env python3
"""Throughput of the k-quant MMQ prefill GEMM path (q8_1 quantise + q4_K/q6_K
GEMM) on GB300, printed as one JSON line.

A step is one prefill pass of a LLaMA-7B-shaped decoder stack's projection
GEMMs at T tokens: for every layer, the four q8_1 quantisations (attention
input shared by q/k/v, o input, FFN input shared by gate/up, down input)
and the seven GEMMs (q, k, o, gate, up, down in q4_K; v in q6_K).  Every
layer has its own weight buffers in HBM (32 layers = 3.8 GB), so each step
streams weights far larger than the 129 MB L2: no L2 flush is needed.
Weights and activations are seeded synthetic data (no checkpoint exists
here); all layers hold copies of one drawn layer.

Headline `value` is TMAC/s over the step (all GEMM MACs / step time, the
quantisations included in the time), measured on the device with CUDA
events around K replays of a CUDA graph of the step.  `e2e` repeats the
measurement through host buffers: each step copies its activations from
pinned host memory and reads the last layer's GEMM outputs back, the copies
on two copy streams overlapping the compute of the neighbouring steps
(device inputs and outputs double-buffered).

`--impl reference` times the CPU oracle (plain C, OpenMP over the output
columns, every host core) on a bounded sample of the same workload: full
q8_1 quantisation of the four inputs and the first rows of every GEMM's
output.  The default run also times that oracle once as `cpu_baseline`.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "q4_K×q8_1 MMQ TMAC/s and 7B-layer prefill tok/s at T=512 (fraction of int8 peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mmq", "reference"], default="mmq")
    ap.add_argument("--tokens", type=int, default=512)
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of replaying a CUDA graph")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-small-t", action="store_true", help="skip the token-sweep and decode side measurements")
    ap.add_argument("--decode-launches", action="store_true",
                    help="only run one eager decode step (T = 1) of --layers layers through the decode-shaped "
                         "kernels (for a launch list)")
    ap.add_argument("--small-t-launches", type=int, default=0, metavar="T",
                    help="only launch the small-T and the split-K GEMM of the config-4 shapes at T tokens three "
                         "times each (eager; for profiling) and exit")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def ranks_max_ms(values, device=None):
    """Per-rank durations (ms) -> their maxima over the ranks of the default
    process group (the slowest rank sets the job's time); unchanged for a
    single process."""
    import torch
    import torch.distributed as dist
    values = [float(v) for v in values]
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return values
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_tmacs(macs_per_rank_step, steps, world, ms):
    """Whole-job throughput: the MACs all ranks processed over the slowest rank's time."""
    return macs_per_rank_step * steps * world / (ms * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# Bytes per weight of each k-quant format (one super-block per 256 weights).
WEIGHT_BYTES = {"q4_K": 144 / 256, "q6_K": 210 / 256}
# f16 tensor-core MMA products per algorithmic MAC on this route: q4_K
# multiplies the exact hi and lo activation planes (2), q6_K also splits the
# weight value into hi and lo planes and forms all four products (4).
ROUTE_MMAS = {"q4_K": 2, "q6_K": 4}


def algorithmic_bytes(fmt, T, K, O):
    """Bytes one GEMM must move: the k-quant weights, the q8_1 activations
    (int8 values plus one 4-byte scale word per 32: 1.125 B per element) and
    the f32 output."""
    return WEIGHT_BYTES[fmt] * O * K + 1.125 * T * K + 4.0 * T * O


def layout_bytes(fmt, T, K, O, act_bytes_per_elem):
    """Bytes the kernel reads and writes in this library's layout: the weights,
    the activation operand planes it reads (xa: 4 B per element, xh: 2), the
    scale words (0.125 B per element) and the f32 output."""
    return WEIGHT_BYTES[fmt] * O * K + (act_bytes_per_elem + 0.125) * T * K + 4.0 * T * O


def choose_peak(peaks, clk):
    """bf16 dense peak (TFLOP/s) for the kernels timed here: the burst figure
    when the sampled SM clock stayed at its maximum with no throttle reason
    during the timed region, the sustained (power-capped) figure otherwise."""
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    sm, smax = (clk or {}).get("sm_mhz"), (clk or {}).get("sm_max_mhz")
    if sm and smax and sm >= 0.98 * smax and not (clk or {}).get("reasons"):
        return burst, "burst (median SM clock at its maximum, no throttle reason in the timed region)"
    return sustained, "sustained (SM clock below its maximum or a throttle reason in the timed region)"


def cpu_info():
    """Host CPU as seen by this process: model name, logical CPUs, affinity."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as fh:
                for line in fh:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    try:
        affinity = len(os.sched_getaffinity(0))
    except AttributeError:
        affinity = os.cpu_count()
    import platform
    return {"model": model or platform.processor() or "unknown", "arch": platform.machine(),
            "nproc": os.cpu_count(), "affinity": affinity}


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"mmq_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


def kernel_source_digest(rec):
    """sha256 over the kernel's source region and the headers it is built from."""
    import hashlib
    csrc = os.path.join(ROOT, "quantized_prefill_gemm_mmq_gb300", "csrc")
    h = hashlib.sha256()
    with open(os.path.join(csrc, rec["source"]), encoding="utf-8") as fh:
        text = fh.read()
    a = text.index(rec["region_begin"])
    b = text.index(rec["region_end"], a)
    h.update(text[a:b].encode())
    for name in rec.get("headers", []):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def traffic_bytes(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None if the kernel's source changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    try:
        if kernel_source_digest(rec) != rec["sha256"]:
            return None
    except (OSError, ValueError, KeyError):
        return None
    return rec["dram_bytes_per_launch"]


def graph_time_us(fns, n=20, reps=5):
    """Device time per call, replayed from a CUDA graph of n calls that cycles
    through the callables `fns` (best of reps)."""
    import torch
    if callable(fns):
        fns = [fns]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fns[0]()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(n):
            fns[i % len(fns)]()
    g.replay()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e3 / n)
    return best


def sweep_lines(dev, hbm_gbs, mac_peak, fast=False):
    """The token sweep (K = 4096 and 11008 into O = 4096) at T = 1, 16, 64, 256,
    1024 and 4096, device time per launch with the weights streamed from HBM
    (the timed launches cycle through copies of W larger than L2 together).
    Every kernel that takes the shape is timed: the weight-stationary small-T
    GEMM and the int8 warp-MMA form (T <= 64 / 16), the decode-shaped products
    (T <= 16, and T <= 4 with the quantisation built in: that line's time
    includes quantising the f32 tokens, the others' do not), split-K
    (T <= 256) and the one-CTA-per-tile production GEMM.
    Each line reports TMAC/s, the fraction of the f16 dense MAC peak and of
    this route's own ceiling, and algorithmic GB/s (weights + q8_1 activations
    at 1.125 B/element + f32 output) as a fraction of the HBM copy rate."""
    import torch
    from quantized_prefill_gemm_mmq_gb300 import ops, synth
    out = []
    Ts = (1, 16) if fast else (1, 16, 64, 256, 1024, 4096)
    for T in Ts:
        for g in synth.config(4, T).gemms:
            w0 = torch.from_numpy(g.weights()).to(dev)
            copies = [w0] + [w0.clone() for _ in range(int(320e6 // w0.numel()))]
            n = 2 * len(copies)
            x = torch.from_numpy(g.x()).to(dev)
            qs, ds, xh, xa = ops.quantize_q8_1(x)
            y = torch.empty((g.T, g.O), dtype=torch.float32, device=dev)
            kern = {}
            if g.T <= ops.SMALL_T_MAX:
                kern["small"] = graph_time_us([lambda w=w: ops.gemm_small(w, xa, ds, g.O, out=y) for w in copies], n=n)
            if g.T <= ops.SMALL_IMMA_T_MAX:
                kern["small_imma"] = graph_time_us([lambda w=w: ops.gemm_small_imma(w, qs, ds, g.O, out=y)
                                                    for w in copies], n=n)
            if g.T <= ops.GEMV_T_MAX:
                kern["gemv"] = graph_time_us([lambda w=w: ops.gemv(w, xh, ds, g.O, out=y) for w in copies], n=n)
            if g.T <= ops.DECODE_T_MAX:
                # f32 tokens in, the q8_1 quantisation inside the launch
                kern["gemv_f32"] = graph_time_us([lambda w=w: ops.gemv_f32(w, x, g.O, out=y) for w in copies], n=n)
            ks = None
            if g.T <= 256:
                ks = ops.choose_ksplit(g.T, g.O, g.K)
                ws = ops.SplitKWorkspace(dev, *ops.splitk_sizes(g.T, g.O, g.K, ks))
                kern["splitk"] = graph_time_us([lambda w=w: ops.gemm_splitk(w, xa, ds, g.O, ksplit=ks, workspace=ws,
                                                                            out=y) for w in copies], n=n)
            kern["production"] = graph_time_us([lambda w=w: ops.gemm("q4_K", w, xa, ds, g.O, out=y) for w in copies],
                                               n=n)
            abytes = algorithmic_bytes("q4_K", g.T, g.K, g.O)
            best = min(kern, key=kern.get)
            us = kern[best]
            line = {"T": g.T, "K": g.K, "O": g.O, "us": {k: round(v, 3) for k, v in kern.items()}, "best": best,
                    "tmacs": g.macs / (us * 1e-6) / 1e12,
                    "f16_dense_frac": g.macs / (us * 1e-6) / 1e12 / mac_peak,
                    "route_ceiling_frac": g.macs / (us * 1e-6) / 1e12 / (mac_peak / ROUTE_MMAS["q4_K"]),
                    "algorithmic_bytes": int(abytes),
                    "gbs": abytes / (us * 1e-6) / 1e9, "hbm_frac": abytes / (us * 1e-6) / 1e9 / hbm_gbs}
            if ks is not None:
                line["ksplit"] = ks
            out.append(line)
            del copies
    # the decode-shaped q6_K products on the 7B attn_v shape (K = O = 4096)
    for T in (1, 4, 16):
        w0 = torch.from_numpy(synth.make_weights("q6_K", 4096, 4096, 301)).to(dev)
        copies = [w0] + [w0.clone() for _ in range(int(320e6 // w0.numel()))]
        n = 2 * len(copies)
        x = torch.from_numpy(synth.make_x(T, 4096, 302)).to(dev)
        _, ds, xh, xa = ops.quantize_q8_1(x, want_qs=False)
        y = torch.empty((T, 4096), dtype=torch.float32, device=dev)
        kern = {"gemv": graph_time_us([lambda w=w: ops.gemv(w, xh, ds, 4096, out=y, fmt="q6_K") for w in copies], n=n),
                "production": graph_time_us([lambda w=w: ops.gemm("q6_K", w, xa, ds, 4096, out=y) for w in copies],
                                            n=n)}
        if T <= ops.DECODE_T_MAX:   # f32 token in, the q8_1 quantisation inside the launch
            kern["gemv_f32"] = graph_time_us([lambda w=w: ops.gemv_f32(w, x, 4096, out=y, fmt="q6_K")
                                              for w in copies], n=n)
        abytes = algorithmic_bytes("q6_K", T, 4096, 4096)
        us = min(kern.values())
        out.append({"fmt": "q6_K", "T": T, "K": 4096, "O": 4096, "us": {k: round(v, 3) for k, v in kern.items()},
                    "best": min(kern, key=kern.get), "algorithmic_bytes": int(abytes),
                    "gbs": abytes / (us * 1e-6) / 1e9, "hbm_frac": abytes / (us * 1e-6) / 1e9 / hbm_gbs})
        del copies
    ops.check_status(dev)
    return out


def format_lines(dev, mac_peak, T=512, K=4096, O=4096):
    """Every weight format on one 7B projection shape (T x K -> O), device time
    per launch with the weights cycled through > 320 MB of copies: the
    production super-block GEMMs (q4_K, q5_K, q6_K; activation planes xa) and
    the per-sub-block GEMMs (q4_K, q5_K, q6_K, q8_0; exact integer dots per
    sub-block, activation plane xh)."""
    import torch
    from quantized_prefill_gemm_mmq_gb300 import ops, synth
    x = torch.from_numpy(synth.make_x(T, K, 700)).to(dev)
    _, ds, xh, xa = ops.quantize_q8_1(x, want_qs=False)
    y = torch.empty((T, O), dtype=torch.float32, device=dev)
    out = []
    for fmt in ("q4_K", "q5_K", "q6_K", "q8_0"):
        w0 = torch.from_numpy(synth.make_weights(fmt, O, K, 701)).to(dev)
        copies = [w0] + [w0.clone() for _ in range(int(320e6 // w0.numel()))]
        n = 2 * len(copies)
        kern = {}
        if fmt != "q8_0":
            kern["production"] = graph_time_us([lambda w=w: ops.gemm(fmt, w, xa, ds, O, out=y) for w in copies], n=n)
        kern["subblock"] = graph_time_us([lambda w=w: ops.gemm_subblock(fmt, w, xh, ds, O, out=y) for w in copies],
                                         n=n)
        best = min(kern, key=kern.get)
        tm = T * K * O / (kern[best] * 1e-6) / 1e12
        out.append({"fmt": fmt, "T": T, "K": K, "O": O, "us": {k: round(v, 2) for k, v in kern.items()}, "best": best,
                    "tmacs": tm, "f16_dense_frac": tm / mac_peak,
                    "weight_bytes": int(w0.numel())})
        del copies
    ops.check_status(dev)
    return out


def decode_line(dev, layers, wl, xs, hbm_gbs):
    """Side measurement: one decode step (T = 1) of the whole layer stack, every
    layer's weights streamed from HBM; one CUDA graph per three steps, device
    time per step (best of 5).  Per layer the seven projections run in five
    launches (decode_groups: q and k, and gate and up, over their concatenated
    rows) as mmq_gemv_q4K_f32 / mmq_gemv_q6K_f32 on the f32 token, the q8_1
    quantisation inside each launch.  The same launches with every input
    quantised by its own launch and the products on mmq_gemv_q4K /
    mmq_gemv_q6K are timed beside it (`unfused`).  `layers` holds the prefill
    step's weights (the chained FFN's gate/up rows interleaved: the same bytes
    for a product with one token)."""
    import torch
    from quantized_prefill_gemm_mmq_gb300 import ops, synth
    groups = decode_groups(wl)
    layers = [{g.name: (torch.cat([lw[m.name] for m in g.members]) if g.name == "q+k" else lw[g.name])
               for g in groups} for lw in layers]
    kk = {s: x.shape[1] for s, x in xs.items()}
    x1 = {s: torch.from_numpy(synth.make_x(1, k, 900 + s)).to(dev) for s, k in kk.items()}
    qb = {s: (None, torch.empty((1, k // 32), dtype=torch.int32, device=dev),
              torch.empty((1, k), dtype=torch.float16, device=dev), None) for s, k in kk.items()}
    yb = {g.name: torch.empty((1, g.O), dtype=torch.float32, device=dev) for g in groups}

    def step():
        for lw in layers:
            for g in groups:
                ops.gemv_f32(lw[g.name], x1[g.x_seed], g.O, out=yb[g.name], fmt=g.fmt)

    def step_unfused():
        for lw in layers:
            for s, x in x1.items():
                ops.quantize_q8_1(x, out=qb[s])
            for g in groups:
                _, ds, xh, _ = qb[g.x_seed]
                ops.gemv(lw[g.name], xh, ds, g.O, out=yb[g.name], fmt=g.fmt)

    us = graph_time_us(step, n=3)
    us_unfused = graph_time_us(step_unfused, n=3)
    ops.check_status(dev)
    wbytes = sum(t.numel() for lw in layers for t in lw.values())
    return {"kernels": "mmq_gemv_q4K_f32 / mmq_gemv_q6K_f32 (q8_1 quantisation inside the launch)",
            "tokens": 1, "layers": len(layers),
            "us_per_step": us, "tok_s": 1e6 / us, "weight_bytes_per_step": wbytes,
            "hbm_gbs": wbytes / (us * 1e-6) / 1e9, "hbm_frac": wbytes / (us * 1e-6) / 1e9 / hbm_gbs,
            "launches_per_step": len(layers) * len(groups),
            "unfused": {"kernels": "mmq_quantize_q8_1 + mmq_gemv_q4K / mmq_gemv_q6K", "us_per_step": us_unfused,
                        "launches_per_step": len(layers) * (len(x1) + len(groups)),
                        "hbm_frac": wbytes / (us_unfused * 1e-6) / 1e9 / hbm_gbs},
            "timing": "CUDA-graph replay of 3 steps, device events, best of 5; weights from HBM (the stack "
                      "exceeds L2)"}


class LaunchGroup:
    """Projections run as one GEMM launch: members share the input and the
    format, the weight rows are concatenated and the output columns too."""

    def __init__(self, name, members):
        g0 = members[0]
        self.name, self.members = name, members
        self.fmt, self.T, self.K, self.x_seed = g0.fmt, g0.T, g0.K, g0.x_seed
        self.O = sum(m.O for m in members)
        self.macs = sum(m.macs for m in members)


def launch_groups(wl):
    """gate and up read the same input: one GEMM over their concatenated rows
    (at T = 512, 688 output tiles of 128 x 128 instead of 2 x 344, i.e. five
    waves of 152 SMs instead of six; the same MACs and, tile for tile, the
    same arithmetic).  Every other projection is its own launch."""
    byname = {g.name: g for g in wl.gemms}
    out = []
    for g in wl.gemms:
        if g.name == "up" and "gate" in byname:
            continue
        if g.name == "gate" and "up" in byname:
            out.append(LaunchGroup("gate+up", [g, byname["up"]]))
        else:
            out.append(LaunchGroup(g.name, [g]))
    return out


def decode_groups(wl):
    """The decode step's launches: as launch_groups, and q and k, which read
    the same token and are both q4_K, as one launch over their concatenated
    rows (at T = 1 every launch carries a few microseconds of fixed cost, so
    the fewer the better; v is q6_K and stays its own launch)."""
    out, qk = [], []
    for g in launch_groups(wl):
        if g.name in ("q", "k") and g.fmt == "q4_K":
            qk.extend(g.members)
        else:
            out.append(g)
    if len(qk) == 2:
        out.insert(0, LaunchGroup("q+k", qk))
    else:
        out = launch_groups(wl)
    return out


def workload_desc(T, layers):
    return (f"LLaMA-7B decoder-stack projections, prefill T={T}, {layers} layers: per layer q/k/o q4_K 4096x4096, "
            f"v q6_K 4096x4096, gate/up q4_K 4096->11008 chained into down q4_K 11008->4096 (one launch over the "
            f"interleaved gate/up rows whose epilogue writes silu(gate)*up as the down input's q8_1 planes), "
            f"3 q8_1 quantisations (attention input, o input, FFN input)")


def workload_config(args, wl, world=1):
    """The `config` object both arms print: the workload, not how it is run."""
    wbytes = sum(WEIGHT_BYTES[g.fmt] * g.O * g.K for g in wl.gemms)
    return {
        "workload": workload_desc(args.tokens, args.layers),
        "tokens": args.tokens, "layers": args.layers, "macs_per_layer": wl.macs,
        "parallelism": f"replicas x{world} (independent copies per GPU)",
        "l2": "inputs larger than L2: each layer has its own weight buffers (weights per step "
              f"{wbytes * args.layers / 1e9:.2f} GB)",
    }


def build_inputs(T):
    from quantized_prefill_gemm_mmq_gb300 import synth
    wl = synth.layer_7b(T)
    xs = {}
    for g in wl.gemms:
        if g.x_seed not in xs:
            xs[g.x_seed] = g.x()
    return wl, xs


# ------------------------------------------------------------ CPU oracle --

def run_oracle_sample(wl, xs, weights, rows_per_gemm, threads=None, split=False):
    """Quantise every input fully and compute the first rows_per_gemm output
    columns of each GEMM with the oracle (OpenMP over the output columns,
    `threads` threads, None = every core); returns (seconds, MACs), or
    (quantisation seconds, GEMM seconds, MACs) with split=True."""
    import oracle
    macs = 0
    t0 = time.perf_counter()
    q = {s: oracle.quantize_q8_1(x) for s, x in xs.items()}
    t1 = time.perf_counter()
    for g in wl.gemms:
        r = min(rows_per_gemm, g.O)
        qs, ds = q[g.x_seed]
        oracle.gemm(g.fmt, weights[g.name][:r], qs, ds, r, threads=threads)   # first r weight rows
        macs += g.T * g.K * r
    t2 = time.perf_counter()
    return (t1 - t0, t2 - t1, macs) if split else (t2 - t0, macs)


def oracle_rows_for(wl, xs, weights, seconds):
    """Rows per GEMM for an oracle sample of about `seconds` (from a short
    calibration run), at least 1 and at most the smallest O."""
    import oracle
    cal_rows = 8 * oracle.max_threads()      # enough output columns to keep every thread busy
    tq, tg, macs = run_oracle_sample(wl, xs, weights, cal_rows, split=True)
    rate = macs / max(tg, 1e-9)
    macs_per_row = sum(g.T * g.K for g in wl.gemms)
    return max(1, min(min(g.O for g in wl.gemms), int(max(seconds - tq, 0.1) * rate / macs_per_row)))


def cpu_baseline_leg(wl, xs, weights, seconds=12.0):
    import oracle
    rows = oracle_rows_for(wl, xs, weights, seconds)
    secs, macs = run_oracle_sample(wl, xs, weights, rows)
    info = cpu_info()
    return {"value": macs / secs / 1e12, "unit": "TMAC/s", "cores": oracle.max_threads(), "kind": "oracle",
            "cpu": info,
            "sample": f"q8_1 quantisation of the 4 layer inputs (one thread) and the first {rows} output rows of each "
                      f"of the 7 GEMMs of one layer ({macs} MACs, {secs:.1f} s; OpenMP over the output columns on "
                      f"{oracle.max_threads()} threads); every layer of the stack is a copy of that layer"}


def reference_arm(args):
    import oracle
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl, xs = build_inputs(args.tokens)
    weights = {g.name: g.weights() for g in wl.gemms}
    # size each step so the whole run stays within about two minutes
    budget_s = max(0.5, 120.0 / max(1, args.steps + args.warmup))
    rows = oracle_rows_for(wl, xs, weights, budget_s)
    for _ in range(args.warmup):
        run_oracle_sample(wl, xs, weights, rows)
    total_s, total_macs = 0.0, 0
    for _ in range(args.steps):
        s, m = run_oracle_sample(wl, xs, weights, rows)
        total_s += s
        total_macs += m
    value = total_macs / total_s / 1e12
    sample = (f"per step: q8_1 quantisation of the 4 layer inputs (T={args.tokens}, one thread) and the first {rows} "
              f"output rows of each of the 7 GEMMs of one layer ({total_macs // args.steps} MACs; OpenMP over the "
              f"output columns on {oracle.max_threads()} threads); every layer of the stack is a copy of that layer")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TMAC/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32 dots, f32 terms, f64 sum",
        "data": "synthetic (seeded random k-quant weights and N(0,1) activations with 1% x20 outlier channels)",
        "config": workload_config(args, wl),
        "cpu_baseline": {"value": value, "unit": "TMAC/s", "cores": oracle.max_threads(), "kind": "oracle",
                         "cpu": cpu_info(), "sample": sample},
        "e2e": {"value": value, "unit": "TMAC/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- GPU arm ---

def small_t_launches(T):
    """Three eager launches each of the small-T GEMM and of the split-K GEMM
    per config-4 shape at T tokens, and of the decode-shaped products for
    T <= 16 (q4_K on those shapes, q6_K on the attn_v shape)."""
    import torch
    from quantized_prefill_gemm_mmq_gb300 import ops, synth
    dev = torch.device("cuda", 0)
    for g in synth.config(4, T).gemms:
        w = torch.from_numpy(g.weights()).to(dev)
        _, ds, xh, xa = ops.quantize_q8_1(torch.from_numpy(g.x()).to(dev), want_qs=False)
        ks = ops.choose_ksplit(g.T, g.O, g.K)
        ws = ops.SplitKWorkspace(dev, *ops.splitk_sizes(g.T, g.O, g.K, ks))
        for _ in range(3):
            ops.gemm_small(w, xa, ds, g.O)
        for _ in range(3):
            ops.gemm_splitk(w, xa, ds, g.O, ksplit=ks, workspace=ws)
        if g.T <= ops.GEMV_T_MAX:
            for _ in range(3):
                ops.gemv(w, xh, ds, g.O)
    if T <= ops.GEMV_T_MAX:
        # the decode-shaped q6_K product on the 7B attn_v shape (K = O = 4096)
        w6 = torch.from_numpy(synth.make_weights("q6_K", 4096, 4096, 301)).to(dev)
        _, ds, xh, _ = ops.quantize_q8_1(torch.from_numpy(synth.make_x(T, 4096, 302)).to(dev), want_qs=False,
                                         want_xa=False)
        for _ in range(3):
            ops.gemv(w6, xh, ds, 4096, fmt="q6_K")
    ops.check_status(dev)
    print(json.dumps({"small_t_launches": T, "status": "ok"}))


def decode_launches(args):
    """One eager decode step (T = 1) of args.layers layers through the decode-shaped
    kernels with the q8_1 quantisation inside each launch, as timed by the
    bench's decode line (after one warm-up step)."""
    import numpy as np
    import torch
    from quantized_prefill_gemm_mmq_gb300 import ops, synth
    dev = torch.device("cuda", 0)
    wl, xs = build_inputs(args.tokens)
    groups = decode_groups(wl)
    host_w = {g.name: g.weights() for g in wl.gemms}
    w_layer = {gr.name: torch.from_numpy(np.concatenate([host_w[m.name] for m in gr.members])).to(dev)
               for gr in groups}
    layers = [w_layer] + [{n: t.clone() for n, t in w_layer.items()} for _ in range(args.layers - 1)]
    x1 = {s: torch.from_numpy(synth.make_x(1, x.shape[1], 900 + s)).to(dev) for s, x in xs.items()}
    yb = {g.name: torch.empty((1, g.O), dtype=torch.float32, device=dev) for g in groups}
    for _ in range(2):
        for lw in layers:
            for g in groups:
                ops.gemv_f32(lw[g.name], x1[g.x_seed], g.O, out=yb[g.name], fmt=g.fmt)
    torch.cuda.synchronize()
    ops.check_status(dev)
    print(json.dumps({"decode_launches": args.layers, "status": "ok"}))


def mmq_arm(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from quantized_prefill_gemm_mmq_gb300 import ops

    if args.small_t_launches:
        small_t_launches(args.small_t_launches)
        return
    if args.decode_launches:
        decode_launches(args)
        return

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    wl, xs = build_inputs(args.tokens)
    groups = launch_groups(wl)
    host_w = {g.name: g.weights() for g in wl.gemms}
    # The FFN is chained: gate and up run as one launch over their rows
    # interleaved in groups of 64 (mmq_gemm_q4K_swiglu), whose epilogue writes
    # h = silu(gate)*up as the down projection's q8_1 operand planes; the down
    # input is therefore produced on the device, not quantised from X.
    ffn = next(g for g in groups if g.name == "gate+up")
    down = next(g for g in groups if g.name == "down")
    F = ffn.O // 2

    def interleave(wg, wu):
        rb = wg.size // F
        return np.concatenate([wg.reshape(F // 64, 64, rb), wu.reshape(F // 64, 64, rb)], axis=1).reshape(-1)

    w_layer = {gr.name: torch.from_numpy(interleave(host_w["gate"], host_w["up"]) if gr is ffn else
                                         np.concatenate([host_w[m.name] for m in gr.members])).to(dev)
               for gr in groups}
    layers = [w_layer] + [{n: t.clone() for n, t in w_layer.items()} for _ in range(args.layers - 1)]
    x_dev = {s: torch.from_numpy(x).to(dev) for s, x in xs.items() if s != down.x_seed}
    # q8_1 planes per input: the production GEMMs read xa (the exact hi/lo
    # dequantised values) and ds; the down input's planes are written by the
    # fused FFN launch
    qbuf = {s: (None,
                torch.empty((x.shape[0], x.shape[1] // 32), dtype=torch.int32, device=dev),
                None,
                torch.empty((2,) + x.shape, dtype=torch.float16, device=dev))
            for s, x in xs.items()}
    ybuf = {g.name: torch.empty((g.T, g.O), dtype=torch.float32, device=dev) for g in groups if g is not ffn}
    layer_macs = wl.macs
    assert layer_macs == sum(g.macs for g in groups)
    step_macs = layer_macs * args.layers
    launches_per_step = args.layers * (len(x_dev) + len(groups))

    ext_events = None   # per-launch events of the q4_K GEMMs, recorded inside the graph
    # Events are recorded around the q4_K launches of every EV_STRIDE-th layer
    # only: each event node in the graph adds a few microseconds between its
    # neighbouring kernels, and the sampled layers are identical in shape.
    EV_STRIDE = 8

    def run_gemm(g, lw, yb=None):
        _, ds, _, xa = qbuf[g.x_seed]
        if g is ffn:
            _, hds, _, hxa = qbuf[down.x_seed]
            ops.gemm_swiglu(lw[g.name], xa, ds, F, out=(None, hds, hxa))
        else:
            ops.gemm(g.fmt, lw[g.name], xa, ds, g.O, out=(yb if yb is not None else ybuf)[g.name])

    def step(record=None, xd=None, yb=None):
        for li, lw in enumerate(layers):
            for s, x in (xd if xd is not None else x_dev).items():
                ops.quantize_q8_1(x, out=qbuf[s])
            for gi, g in enumerate(groups):
                ev = record[li][gi] if record is not None else None
                if ev is not None:
                    ev[0].record()
                run_gemm(g, lw, yb)
                if ev is not None:
                    ev[1].record()

    # warm-up (eager): builds attributes, checks status
    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    ops.check_status(dev)

    graph = None
    timing_mode = "eager"
    if not args.no_graph:
        try:
            ext_events = [[(torch.cuda.Event(enable_timing=True, external=True),
                            torch.cuda.Event(enable_timing=True, external=True))
                           if g.fmt == "q4_K" and li % EV_STRIDE == 0 else None
                           for g in groups] for li in range(len(layers))]
        except TypeError:
            ext_events = None
        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                step(ext_events)
        torch.cuda.current_stream(dev).wait_stream(s)
        timing_mode = "cuda graph"
        for _ in range(max(1, args.warmup)):
            graph.replay()
        torch.cuda.synchronize()
        ops.check_status(dev)

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step()

    # ---------------- timed region (device-resident inputs)
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)   # let the sampler start before the timed work
    cur = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(args.steps):
        run_step()
    e1.record(cur)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ops.check_status(dev)
    elapsed_ms = e0.elapsed_time(e1)

    # per-launch durations of the dominant kernel (the production q4_K GEMM),
    # by launch shape: the headline roofline is taken on its 4096 x 4096
    # launches (q, k, o; the shape of the committed ncu counters), and the
    # gate+up (4096 -> 22016) and down (11008 -> 4096) launches get their own
    shape_stats = {}     # shape key -> [ms, macs, launches, group]
    kernel_timing = None

    def shape_key(g):
        return f"T={g.T} K={g.K} O={g.O}"

    def add_time(g, ms):
        st = shape_stats.setdefault(shape_key(g), [0.0, 0, 0, g])
        st[0] += ms
        st[1] += g.macs
        st[2] += 1

    if ext_events is not None:
        for li in range(len(layers)):
            for gi, g in enumerate(groups):
                ev = ext_events[li][gi]
                if ev is not None:
                    add_time(g, ev[0].elapsed_time(ev[1]))
        kernel_timing = (f"events in the captured graph around the q4_K launches of every {EV_STRIDE}th layer "
                         "(last replay of the timed region)")
    if not shape_stats:
        pairs = []
        for lw in layers:
            for g in groups:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(cur)
                run_gemm(g, lw)
                b.record(cur)
                if g.fmt == "q4_K":
                    pairs.append((a, b, g))
        torch.cuda.synchronize()
        for a, b, g in pairs:
            add_time(g, a.elapsed_time(b))
        kernel_timing = "eager per-launch events"
    int8_peak = ops.tensor_peak_tmacs("int8", dev)

    # ---------------- end to end through host buffers
    # Every step copies its inputs from pinned host memory and its outputs back.
    # The copies run on two copy streams, pipelined with the compute stream
    # (inputs and outputs double-buffered, one captured graph per buffer set):
    # step i+1's inputs and step i-1's outputs move while step i computes.
    e2e = None
    if not args.no_e2e:
        hx = {s: torch.from_numpy(xs[s]).pin_memory() for s in x_dev}
        hy = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in ybuf.items()}
        h2d = sum(t.numel() * t.element_size() for t in hx.values())
        d2h = sum(t.numel() * t.element_size() for t in hy.values())
        x_sets = [x_dev, {s: t.clone() for s, t in x_dev.items()}]
        y_sets = [ybuf, {n: t.clone() for n, t in ybuf.items()}]
        e2e_graphs = None
        if graph is not None:
            e2e_graphs = []
            for k in range(2):
                gk = torch.cuda.CUDAGraph()
                sk = torch.cuda.Stream(device=dev)
                sk.wait_stream(torch.cuda.current_stream(dev))
                with torch.cuda.stream(sk):
                    with torch.cuda.graph(gk, stream=sk):
                        step(None, x_sets[k], y_sets[k])
                torch.cuda.current_stream(dev).wait_stream(sk)
                e2e_graphs.append(gk)
            torch.cuda.synchronize()

        def run_set(k):
            if e2e_graphs is not None:
                e2e_graphs[k].replay()
            else:
                step(None, x_sets[k], y_sets[k])

        up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()
        comp_ev, d2h_ev, h2d_ev = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        run_set(0)
        run_set(1)
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(cur)
        up.wait_stream(cur)
        down.wait_stream(cur)

        def issue_h2d(i):
            k = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(comp_ev[k])            # step i-2 has read this input set
                for s in x_sets[k]:
                    x_sets[k][s].copy_(hx[s], non_blocking=True)
                h2d_ev[k].record(up)

        issue_h2d(0)
        for i in range(args.steps):
            k = i % 2
            if i + 1 < args.steps:
                issue_h2d(i + 1)
            cur.wait_event(h2d_ev[k])
            if i >= 2:
                cur.wait_event(d2h_ev[k])                # step i-2's outputs are out
            run_set(k)
            comp_ev[k].record(cur)
            with torch.cuda.stream(down):
                down.wait_event(comp_ev[k])
                for n in y_sets[k]:
                    hy[n].copy_(y_sets[k][n], non_blocking=True)
                d2h_ev[k].record(down)
        f1.record(down)
        torch.cuda.synchronize()
        e2e_ms = f0.elapsed_time(f1)
        e2e = {"value": job_tmacs(step_macs, args.steps, world, e2e_ms), "unit": "TMAC/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.steps,
               "copies": "pinned host buffers; H2D and D2H on two copy streams pipelined with the "
                         "compute stream (double-buffered device inputs/outputs)"}
        ops.check_status(dev)

    if world > 1:
        slowest = ranks_max_ms([elapsed_ms] + ([e2e["ms_per_step"]] if e2e is not None else []), dev)
        elapsed_ms = slowest[0]
        if e2e is not None:
            e2e["ms_per_step"] = slowest[1]
            e2e["value"] = job_tmacs(step_macs, 1, world, e2e["ms_per_step"])

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    ms_step = elapsed_ms / args.steps
    value = job_tmacs(step_macs, args.steps, world, elapsed_ms)
    peak, peak_kind = choose_peak(peaks, clk)
    mac_peak = peak / 2.0                       # f16 dense TMAC/s (f16 runs at the bf16 rate)
    hbm_gbs = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))

    def shape_line(st):
        ms, macs, n, g = st
        us = 1e3 * ms / n
        tflops = 2.0 * macs / (ms * 1e-3) / 1e12
        return {"shape": shape_key(g), "launch": g.name, "launches_timed": n, "avg_launch_us": us,
                "achieved_tflops": tflops, "frac": tflops / peak,
                "route_ceiling_frac": tflops / (peak / ROUTE_MMAS[g.fmt]),
                "algorithmic_bytes_per_launch": int(algorithmic_bytes(g.fmt, g.T, g.K, g.O)),
                "layout_bytes_per_launch": int(layout_bytes(g.fmt, g.T, g.K, g.O, 4))}

    shapes = [shape_line(st) for st in shape_stats.values()]
    sq = shape_stats.get(shape_key(next(g for g in groups if g.fmt == "q4_K" and g.K == g.O == 4096)))
    sq_line = shape_line(sq) if sq else None
    roofline = {
        "bound": "tensor",
        "achieved": sq_line["achieved_tflops"] if sq_line else None,
        "peak": peak, "unit": "TFLOP/s",
        "frac": sq_line["frac"] if sq_line else None,
        "traffic": traffic_bytes("mmq_q4K_sb_kernel"),
        "kernel": f"mmq_q4K_sb_kernel (production q4_K GEMM), launches of shape T={args.tokens} K=4096 O=4096",
        "algorithmic_bytes_per_launch": sq_line["algorithmic_bytes_per_launch"] if sq_line else None,
        "layout_bytes_per_launch": sq_line["layout_bytes_per_launch"] if sq_line else None,
        "algorithmic_work": "2*T*O*K flop; bytes = 0.5625*O*K (q4_K) + 1.125*T*K (q8_1) + 4*T*O (f32 Y); the layout "
                            "reads the activations as exact f16 hi/lo planes (4 B per element) + scale words",
        "peak_source": f"{peak_src} bf16 dense, {peak_kind}; f16 runs at the bf16 rate",
        "route_ceiling_frac": sq_line["route_ceiling_frac"] if sq_line else None,
        "route_ceiling_note": "exact results take 2 f16 MMA products per useful one for q4_K (activation hi and "
                              "lo planes), 4 for q6_K (weight hi and lo planes too): the route's ceiling is 1/2 "
                              "(1/4) of the dense peak",
        "timing": kernel_timing,
        "avg_launch_us": sq_line["avg_launch_us"] if sq_line else None,
        "shapes": shapes,
    }
    # the step's ceiling on this route: every GEMM at its route's MMA count, the quantisations free
    step_ceiling = layer_macs / sum(g.macs * ROUTE_MMAS[g.fmt] / mac_peak for g in groups)
    fractions = {
        "f16_dense": value / world / mac_peak,
        "route_ceiling": value / world / step_ceiling,
        "f16_dense_mac_peak_tmacs": mac_peak,
        "route_ceiling_tmacs": step_ceiling,
    }
    cpu = None
    if not args.no_cpu and world == 1:
        cpu = cpu_baseline_leg(wl, xs, host_w)
    sweep = None
    if not args.no_small_t and world == 1:
        sweep = {"kernels": "per line every kernel that takes the shape: mmq_gemm_q4K_small (weight-stationary "
                            "tcgen05, T <= 64), mmq_gemm_q4K_small_imma (int8 warp MMA, T <= 16), mmq_gemv_q4K "
                            "(decode-shaped, T <= 16), mmq_gemm_q4K_splitk (T <= 256) and mmq_gemm_q4K (production); "
                            "q6_K lines: mmq_gemv_q6K vs the production q6_K GEMM on the attn_v shape",
                 "timing": "CUDA-graph replay cycling through >320 MB of weight copies (HBM-resident), device "
                           "events, best of 5; the line's rates are the fastest kernel's",
                 "bytes": "algorithmic: weights + q8_1 activations (1.125 B/element) + f32 Y",
                 "hbm_peak_gbs": hbm_gbs, "f16_dense_mac_peak_tmacs": mac_peak,
                 "lines": sweep_lines(dev, hbm_gbs, mac_peak)}
    decode = formats = None
    if not args.no_small_t and world == 1:
        decode = decode_line(dev, layers, wl, xs, hbm_gbs)
        formats = {"kernels": "production: mmq_gemm_q4K / _q5K / _q6K; subblock: mmq_gemm_q4K_subblock / "
                              "q5K_subblock / q6K_subblock and mmq_gemm_q8_0 (per-sub-block form)",
                   "timing": "CUDA-graph replay cycling through >320 MB of weight copies, device events, best of 5",
                   "lines": format_lines(dev, mac_peak)}
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TMAC/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 tensor-core operands holding exact int8/int4 integers, f32 accumulate and fold",
        "data": "synthetic (seeded random k-quant weights and N(0,1) activations with 1% x20 outlier channels)",
        "config": workload_config(args, wl, world),
        "launch": timing_mode,
        "fractions": fractions,
        "int8_frac": value / world / int8_peak if int8_peak else None,
        "int8_frac_note": "labelled extra: TMAC/s over the legacy warp-level int8 MMA rate (mma.sync m16n8k32 s8, "
                          "measured live); sm_103a has no int8 tcgen05 kind and this route runs on the f16 tensor "
                          "cores, so the figure can exceed 1",
        "int8_peak_tmacs": int8_peak,
        "layer_tok_s": args.tokens * args.layers * args.steps * world / (elapsed_ms * 1e-3),
        "model_tok_s_gemm_only": args.tokens * args.steps * world / (elapsed_ms * 1e-3),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clk,
        "gpu_launches": launches_per_step * args.steps,
        "sweep": sweep,
        "decode": decode,
        "formats": formats,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        reference_arm(args)
    else:
        mmq_arm(args)


if __name__ == "__main__":
    main()
