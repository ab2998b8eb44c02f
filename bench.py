#!/usr/bin/env python
"""Throughput of Fused-Softmax MX attention on one GB300 (and N replicas).

One step = the whole hot path for each of the three formats (MXFP8, MXFP6,
MXFP4) over one batch of synthetic input: MX quantization of Q, K, V
followed by the fused attention kernel.  The timed region runs its K steps'
calls format-major (K calls of MXFP8, then of MXFP6, then of MXFP4), so
each format's kernel is timed in steady state.  `value` is the aggregate attention
throughput 4*B*H*S^2*D per format-call over the device-timed region (inputs
resident in HBM); `per_format` breaks it down and gives the attention
kernel alone; `e2e` repeats the step through the public host-buffer C-ABI
call (fsa_attention_fwd_host): every format call reads Q, K, V from pinned
host memory and writes O back to it, the library streaming heads through
the device with the copies overlapping the computation.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
  python bench.py --schedule    # 20-step hybrid MXFP6/MXFP4 schedule vs all-BF16 / all-MXFP4
  python bench.py --mma-peaks   # only the tensor-core rate probe

After the timed region the default run also times the other benchmark
workloads (`configs`: B=1 H=16 S=8192, the rollback-stress shape, the
B=1 H=32 sequence sweep with the BF16 kernel) and measures the dense
block-scaled MMA rates with the library's tensor-core rate probe
(`mma_peaks`), which are the roofline denominators of every fraction.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import fsa_inputs  # noqa: E402

METRIC = "fused-softmax MX attention TFLOPS per format at 1 GB300; % of MX MMA peak"
FORMATS = ("mxfp8", "mxfp6", "mxfp4")
WORKLOADS = {
    # video-DiT self-attention: 21 x 45 x 80 latent tokens, 40 heads of 128
    "video-dit": dict(B=1, H=40, S=75600, D=128),
    "h16-s8192": dict(B=1, H=16, S=8192, D=128),
    "rollback-stress": dict(B=1, H=8, S=32768, D=128, stress_from=16384),
    "h32-s16384": dict(B=1, H=32, S=16384, D=128),
    "h32-s32768": dict(B=1, H=32, S=32768, D=128),
    "h32-s65536": dict(B=1, H=32, S=65536, D=128),
    "h32-s131072": dict(B=1, H=32, S=131072, D=128),
    # head dim 64 at scale
    "d64-h32-s32768": dict(B=1, H=32, S=32768, D=64),
    # queries and keys of different lengths (S = query rows, Sk = keys): video
    # tokens attending to a 512-token context, and a short query over a long one
    "cross-q75600-k512": dict(B=1, H=40, S=75600, Sk=512, D=128),
    "cross-q4096-k32768": dict(B=1, H=32, S=4096, Sk=32768, D=128),
}
THRESHOLD = 8.0


def keys(w):
    return w.get("Sk", w["S"])


def is_cross(w):
    return keys(w) != w["S"]


def flops(w):
    return 4.0 * w["B"] * w["H"] * w["S"] * keys(w) * w["D"]


def workload_name(name, w):
    if is_cross(w):
        return f"{name} B={w['B']} H={w['H']} Sq={w['S']} Sk={keys(w)} D={w['D']}"
    return f"{name} B={w['B']} H={w['H']} Sq=Sk={w['S']} D={w['D']}"


def make_inputs(w, seed):
    """Synthetic bf16 Q, K, V bit patterns; keys and values drawn separately
    when their length differs from the queries'."""
    B, H, S, D = w["B"], w["H"], w["S"], w["D"]
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=seed, stress_from=w.get("stress_from"))
    if is_cross(w):
        _, k, v = fsa_inputs.qkv(B, H, keys(w), D, seed=seed + 1, stress_from=w.get("stress_from"))
    return q, k, v


def peaks(mma=None):
    """Roofline denominators (TFLOP/s, GB/s).  bf16 and HBM: the measured
    figures of this machine pool (MEASURED_PEAKS.json: cuBLAS GEMM, copy).  Block-scaled MMA
    rates: the tensor-core rate probe of this run (measure_mma_peaks) when
    given -- R8 (E4M3), R6 (E2M3), R4 (packed E2M1, kind::mxf4) and the
    attention kernel's own product mix -- else the bf16 rate times the
    nominal ratios (fp8 4.5 / bf16 2.25, fp4 13.5 / 2.25)."""
    p = {"source": "fallback", "bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        p = {"source": "measured", "bf16_burst": float(m["bf16_tflops"]),
             "bf16_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
             "hbm_gbs": float(m["hbm_gbs"])}
    except (OSError, KeyError, ValueError):
        pass
    if mma:
        p["mx_source"] = "measured by the tensor-core rate probe in this run"
        p["mx8_burst"] = mma["mxf8f6f4_e4m3"]["burst_tflops"]
        p["mx8_sustained"] = mma["mxf8f6f4_e4m3"]["sustained_tflops"]
        p["mx6_sustained"] = mma["mxf8f6f4_e2m3"]["sustained_tflops"]
        p["fp4_sustained"] = mma["mxf4_e2m1"]["sustained_tflops"]
        p["attn_tile_sustained"] = mma["attention_tile_e4m3"]["sustained_tflops"]
    else:
        p["mx_source"] = f"{p['source']} bf16 rate x nominal ratios"
        ratio = 4.5 / 2.25
        p["mx8_burst"] = p["bf16_burst"] * ratio
        p["mx8_sustained"] = p["bf16_sustained"] * ratio
        p["mx6_sustained"] = p["mx8_sustained"]
        p["fp4_sustained"] = p["bf16_sustained"] * (13.5 / 2.25)
        p["attn_tile_sustained"] = None
    return p


def format_roofline(pk, fmt):
    """Dense block-scaled MMA roofline of a format: both products at the
    rate of its element type -- E4M3 (MXFP8), E2M3 (MXFP6); for MXFP4 the
    score product at the four-bit rate and the PV product on six-bit P, so
    2 / (1/R4 + 1/R6)."""
    if fmt == "mxfp8":
        return pk["mx8_sustained"]
    if fmt == "mxfp6":
        return pk["mx6_sustained"]
    return 2.0 / (1.0 / pk["fp4_sustained"] + 1.0 / pk["mx6_sustained"])


# tensor-core rate probes (fsa_mma_rate_probe), in the order they are measured
PROBES = ("mxf8f6f4_e4m3", "mxf8f6f4_e2m3", "mxf4_e2m1", "attention_tile_e4m3", "f16_bf16")


def measure_mma_peaks(fsa, dev, stream, n_sm, sustained_s=2.0, launch_s=0.02):
    """Measured tensor-core rates on this GPU (TFLOP/s): for every probe kind
    one CTA per SM issues its products back to back.  burst = the best of
    three single launches of about launch_s; sustained = back-to-back
    launches for about sustained_s, timed as a whole, with the SM clocks
    sampled meanwhile (the tensor core at full rate runs into the power cap,
    as a long attention step does)."""
    out = {}
    for kind in PROBES:
        it0 = 512
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fsa.mma_rate_probe(kind, n_sm, it0)          # warm-up (loads the kernel)
        e0.record(stream)
        fsa.mma_rate_probe(kind, n_sm, it0)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        t0 = e0.elapsed_time(e1) / 1e3
        iters = max(it0, int(it0 * launch_s / max(t0, 1e-6)))
        best = 0.0
        for _ in range(3):
            e0.record(stream)
            fl = fsa.mma_rate_probe(kind, n_sm, iters)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            best = max(best, fl / (e0.elapsed_time(e1) / 1e3) / 1e12)
        n = max(3, int(sustained_s / launch_s))
        with ClockSampler(int(dev.index or 0)) as clk:
            e0.record(stream)
            tot = 0.0
            for _ in range(n):
                tot += fsa.mma_rate_probe(kind, n_sm, iters)
            e1.record(stream)
            torch.cuda.synchronize(dev)
        sus = tot / (e0.elapsed_time(e1) / 1e3) / 1e12
        c = clk.summary()
        out[kind] = {"burst_tflops": best, "sustained_tflops": sus, "sm_mhz": c["sm_mhz"],
                     "reasons": c["reasons"]}
        if c["sm_mhz"]:
            # flops per SM per clock at the sustained rate
            out[kind]["flops_per_sm_clk"] = sus * 1e12 / (n_sm * c["sm_mhz"] * 1e6)
    st = fsa.get_device_error()
    if st != 0:
        raise RuntimeError(f"device error in the MMA rate probe: {fsa.status_string(st)}")
    return out


def traffic_from_profiles():
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary, if one exists for the current kernel."""
    path = os.path.join(ROOT, "profiles", "fsa_attn_fwd_kernel_video_dit.md")
    try:
        txt = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    return float(m.group(1)) if m else None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed
    region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def to_dev(bits, device):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device)


def sample_rows(w, n_rows):
    """Rows of an oracle sample: n_rows rows of the video-DiT key length's
    work, i.e. n_rows * 75600 / Sk rows (at most every row), evenly spaced
    over as few heads from the first on as hold them (a head's rows share
    its keys, as in a whole run)."""
    S, total = w["S"], w["B"] * w["H"] * w["S"]
    n = min(total, max(1, round(n_rows * WORKLOADS["video-dit"]["S"] / keys(w))))
    span = min(total, -(-n // S) * S)
    return np.unique(np.linspace(0, span - 1, n).astype(np.int64))


def oracle_sample(q, k, v, w, fmt, n_rows, threads):
    """Time the oracle on the rows of sample_rows(w, n_rows); returns the
    sample's FLOPs, seconds and row count."""
    import oracle
    rows = sample_rows(w, n_rows)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=THRESHOLD, rows=rows,
                     threads=threads)
    dt = time.perf_counter() - t0
    return len(rows) * 4.0 * keys(w) * w["D"], dt, len(rows)


def max_over_ranks(x, dist=None, device="cpu"):
    """The largest of every rank's x (the slowest rank sets a replica run's
    time); x itself when there is a single process."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(world, flops_per_call, n_calls, elapsed_s):
    """Whole-job throughput of weakly scaled replicas: every rank ran the
    same n_calls calls of flops_per_call, the slowest in elapsed_s."""
    return world * flops_per_call * n_calls / elapsed_s / 1e12


def cpu_affinity():
    """Cores this process may run on: their count and the affinity list as
    compact ranges ("0-15")."""
    cpus = sorted(os.sched_getaffinity(0))
    spans, start = [], cpus[0]
    for a, b in zip(cpus, cpus[1:] + [None]):
        if b != a + 1:
            spans.append(f"{start}-{a}" if a != start else f"{a}")
            start = b
    return len(cpus), ",".join(spans)


CONFIG_FORMATS = ("mxfp8", "mxfp6", "mxfp4", "mxfp4_efq")
SWEEP_S = (16384, 32768, 65536, 131072)


def host_copy_rates(h_in, h_out, dev, reps=3):
    """Pinned host <-> device copy rates (GB/s) of this box: h_in -> device
    alone, device -> h_out alone, and both at once on two streams; CUDA
    events on the copy streams, the best of `reps`."""
    d_in, d_out = torch.empty_like(h_in, device=dev), torch.empty_like(h_out, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    b_in, b_out = h_in.numel() * h_in.element_size(), h_out.numel() * h_out.element_size()
    best = {"h2d": 0.0, "d2h": 0.0, "h2d_while_d2h": 0.0, "d2h_while_h2d": 0.0}
    torch.cuda.synchronize(dev)
    def copy_in():
        with torch.cuda.stream(s_in):
            ev[0].record(s_in)
            d_in.copy_(h_in, non_blocking=True)
            ev[1].record(s_in)

    def copy_out():
        with torch.cuda.stream(s_out):
            ev[2].record(s_out)
            h_out.copy_(d_out, non_blocking=True)
            ev[3].record(s_out)

    for _ in range(reps):
        copy_in()
        torch.cuda.synchronize(dev)
        best["h2d"] = max(best["h2d"], b_in / (ev[0].elapsed_time(ev[1]) * 1e6))
        copy_out()
        torch.cuda.synchronize(dev)
        best["d2h"] = max(best["d2h"], b_out / (ev[2].elapsed_time(ev[3]) * 1e6))
        copy_in()
        copy_out()
        torch.cuda.synchronize(dev)
        best["h2d_while_d2h"] = max(best["h2d_while_d2h"], b_in / (ev[0].elapsed_time(ev[1]) * 1e6))
        best["d2h_while_h2d"] = max(best["d2h_while_h2d"], b_out / (ev[2].elapsed_time(ev[3]) * 1e6))
    del d_in, d_out
    return best


def run_configs(fsa, dev, stream, seed):
    """The other benchmark workloads, one warm-up and one timed call
    per format (quantizer and fused kernel timed apart, CUDA events on the
    launching stream): B=1 H=16 S=8192 D=128; the rollback-stress shape
    (B=1 H=8 S=32768 D=128, 1 % of the keys after 16384 scaled by 8; firings
    counted); and the sequence sweep B=1 H=32 D=128, S in SWEEP_S, every
    format plus the in-house BF16 kernel.  Inputs: N(0,1) drawn on the device
    by torch's generator (seed 1234 + seed), rounded to bf16 -- the
    distribution of the parity inputs, drawn where they are used; the shapes
    share one buffer of the largest (H=32, S=131072: 1.07 GB per tensor,
    larger than L2), each taking its leading elements."""
    g = torch.Generator(device=dev)
    g.manual_seed(1234 + seed)
    n_max = 32 * max(SWEEP_S) * 128
    base = [torch.randn(n_max, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
            for _ in range(3)]

    def view(B, H, S, D):
        return [t[:B * H * S * D].view(B, H, S, D) for t in base]

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def timed(fn_prep, fn_run):
        for rep in range(2):                 # one warm-up, one timed
            ev[0].record(stream)
            fn_prep()
            ev[1].record(stream)
            fn_run()
            ev[2].record(stream)
            torch.cuda.synchronize(dev)
        return ev[0].elapsed_time(ev[1]) / 1e3, ev[1].elapsed_time(ev[2]) / 1e3

    def one(name, B, H, S, D, qkv, with_bf16, count=False, shortcut=False):
        F = 4.0 * B * H * S * S * D
        o = torch.empty_like(qkv[0])
        ws = fsa.new_workspace(B, H, S, D, device=dev)
        r = {}
        runs = [(fmt, "fp32") for fmt in CONFIG_FORMATS]
        if shortcut:   # the shortcut rollback gate, method formats
            runs += [(fmt, "shortcut") for fmt in FORMATS]
        for fmt, gate in runs:
            cnt = torch.zeros(1, dtype=torch.int64, device=dev) if count else None

            def run():
                if cnt is not None:
                    cnt.zero_()
                fsa.attention_run(ws, o, fmt, THRESHOLD, rollback_count=cnt, gate=gate)
            tq, ta = timed(lambda: fsa.attention_prepare(*qkv, ws, fmt), run)
            key = fmt if gate == "fp32" else f"{fmt}_shortcut_gate"
            r[key] = {"attention_ms": 1e3 * ta, "quantize_ms": 1e3 * tq,
                      "attention_tflops": F / ta / 1e12}
            if cnt is not None and fmt != "mxfp4_efq":
                r[key]["rollback_count"] = int(cnt.item())
        if with_bf16:
            _, tb = timed(lambda: None, lambda: fsa.bf16_attention_fwd(*qkv, out=o))
            r["bf16"] = {"attention_ms": 1e3 * tb, "attention_tflops": F / tb / 1e12}
            for fmt in CONFIG_FORMATS:
                r[fmt]["speedup_vs_bf16_kernel"] = tb / (r[fmt]["attention_ms"] / 1e3)
        st = fsa.get_device_error()
        if st != 0:
            raise RuntimeError(f"device error in {name}: {fsa.status_string(st)}")
        del ws, o
        return r

    out = {}
    out["h16-s8192 B=1 H=16 S=8192 D=128"] = one("h16-s8192", 1, 16, 8192, 128,
                                                  view(1, 16, 8192, 128), True)
    q, k, v = view(1, 8, 32768, 128)
    k = k.clone()
    mask = torch.rand((1, 8, 32768), generator=g, device=dev) < 0.01
    mask[:, :, :16384] = False
    k[mask] = k[mask] * 8
    out["rollback-stress B=1 H=8 S=32768 D=128 (1 % of keys after 16384 x 8)"] = one(
        "rollback-stress", 1, 8, 32768, 128, (q, k, v), True, count=True, shortcut=True)
    del q, k, v, mask
    sweep = {}
    for S in SWEEP_S:
        sweep[str(S)] = one(f"sweep S={S}", 1, 32, S, 128, view(1, 32, S, 128), True)
    out["sweep B=1 H=32 D=128 (S)"] = sweep
    del base
    torch.cuda.empty_cache()
    return out


def add_config_fracs(configs, pk):
    """Each format's attention rate as a fraction of its roofline."""
    def walk(d):
        for key, val in d.items():
            base = key.replace("_shortcut_gate", "")
            if base in CONFIG_FORMATS and isinstance(val, dict):
                fmt = "mxfp4" if base == "mxfp4_efq" else base
                val["frac_of_format_roofline"] = val["attention_tflops"] / format_roofline(pk, fmt)
                val["frac_of_mx8_peak"] = val["attention_tflops"] / pk["mx8_sustained"]
            elif isinstance(val, dict):
                walk(val)
    walk(configs)


def bench_config(args, w):
    """The `config` object of both arms' JSON lines."""
    B, H, S, D = w["B"], w["H"], w["S"], w["D"]
    Sk = keys(w)
    return {"workload": workload_name(args.workload, w), "formats": list(FORMATS),
            "threshold": THRESHOLD, "non_causal": True,
            "l2": (f"inputs {2 * B * H * S * D / 1e6:.0f} MB (Q), "
                   f"{2 * B * H * Sk * D / 1e6:.0f} MB (K, V) each"),
            "step": "per format: quantize Q,K,V + fused attention"}


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    q, k, v = make_inputs(w, 0)
    threads, affinity = cpu_affinity()
    n_rows = args.ref_rows
    total_f, total_t = 0.0, 0.0
    for i in range(args.warmup + args.steps):
        f_step, t_step = 0.0, 0.0
        for fmt in FORMATS:
            f, t, n_used = oracle_sample(q, k, v, w, fmt, n_rows, threads)
            f_step += f
            t_step += t
        if i >= args.warmup:
            total_f += f_step
            total_t += t_step
    val = total_f / total_t / 1e12
    sample = (f"{n_used} query rows evenly spaced from head 0 on per format per step (all "
              f"{keys(w)} keys), 3 formats; rate extrapolates exactly since rows are independent")
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic N(0,1) bf16, seed 0",
        "config": bench_config(args, w),
        "cpu_baseline": {"kind": "oracle", "value": val, "unit": "TFLOP/s", "cores": threads,
                         "affinity": affinity, "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_schedules(args, w, fsa, tq, tk, tv, o, ws, stream, dev, rank):
    """Attention time of whole denoising schedules: every step is one library
    call on the step's format (quantization + fused kernel for MX formats,
    the BF16 kernel for bf16), timed with CUDA events around each call.  The
    inputs are the same synthetic tensors every step."""
    from matrix_core_softmax_gb300 import schedule as sch
    plans = {
        "hybrid": sch.hybrid_schedule(),
        "all-mxfp4": sch.uniform_schedule("mxfp4"),
        "all-mxfp6": sch.uniform_schedule("mxfp6"),
        "all-mxfp8": sch.uniform_schedule("mxfp8"),
        "all-bf16": sch.uniform_schedule("bf16"),
    }
    for fmt in sch.STEP_FORMATS:  # warm-up: one call of every format
        for _ in range(max(1, args.warmup)):
            sch.attention_step(tq, tk, tv, fmt, THRESHOLD, out=o, workspace=ws)
    torch.cuda.synchronize(dev)
    if fsa.get_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    res = {}
    with ClockSampler(int(dev.index or 0)) as clk:
        for name, plan in plans.items():
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(plan) + 1)]
            ev[0].record(stream)
            for i, fmt in enumerate(plan):
                sch.attention_step(tq, tk, tv, fmt, THRESHOLD, out=o, workspace=ws)
                ev[i + 1].record(stream)
            torch.cuda.synchronize(dev)
            per = [ev[i].elapsed_time(ev[i + 1]) for i in range(len(plan))]
            res[name] = {"formats": plan, "total_ms": sum(per), "per_step_ms": per}
    st = fsa.get_device_error()
    if st != 0:
        raise RuntimeError(f"device error: {fsa.status_string(st)}")
    if rank != 0:
        return
    hyb = res["hybrid"]["total_ms"]
    line = {
        "metric": "self-attention time of a 20-step video-DiT denoising schedule",
        "value": hyb, "unit": "ms", "higher_is_better": False, "n_gpus": 1,
        "data": "synthetic N(0,1) bf16, the same Q, K, V every step",
        "config": {"workload": workload_name(args.workload, w), "threshold": THRESHOLD,
                   "steps": len(plans["hybrid"]),
                   "hybrid": "MXFP6 for steps 0-2 and 17-19, MXFP4 for steps 3-16",
                   "per_step": "one library call: quantize Q,K,V + fused attention (MX), or the BF16 kernel"},
        "schedules": res,
        "speedup_hybrid_vs_all_bf16": res["all-bf16"]["total_ms"] / hyb,
        "speedup_hybrid_vs_all_mxfp4": res["all-mxfp4"]["total_ms"] / hyb,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="fsa", choices=("fsa", "reference"))
    ap.add_argument("--workload", default="video-dit", choices=sorted(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-bf16", action="store_true")
    ap.add_argument("--no-efq", action="store_true", help="skip the EFQ-Softmax format")
    ap.add_argument("--no-shortcut", action="store_true", help="skip the shortcut-gate timing")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (h16-s8192, rollback stress, the S sweep)")
    ap.add_argument("--no-mma-probe", action="store_true",
                    help="skip the tensor-core rate probe (peaks from the bf16 rate x nominal ratios)")
    ap.add_argument("--mma-peaks", action="store_true",
                    help="only measure the tensor-core rates and print them")
    ap.add_argument("--cpu-rows", type=int, default=12288)
    # rows of the reference arm's sample per format and step: every oracle
    # call also quantizes the whole Q, K and V once, so a few rows would time
    # mostly that (96 rows: 0.004 TFLOP/s against 0.043 for 12288)
    ap.add_argument("--ref-rows", type=int, default=1024)
    ap.add_argument("--schedule", action="store_true",
                    help="time the 20-step hybrid precision schedule against all-BF16 and all-MXFP4")
    args = ap.parse_args()
    w = WORKLOADS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import matrix_core_softmax_gb300 as fsa
    from matrix_core_softmax_gb300 import build as fsa_build
    if rank == 0 or world == 1:
        fsa_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
        dist.barrier()
        fsa_build.build()
    fsa.load()
    if args.mma_peaks:
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        res = measure_mma_peaks(fsa, dev, torch.cuda.current_stream(dev), n_sm)
        if rank == 0:
            print(json.dumps({"mma_peaks": res, "n_sm": n_sm,
                              "probe": "fsa_mma_rate_probe, one CTA per SM, operands resident"}),
                  flush=True)
        return

    B, H, S, D = w["B"], w["H"], w["S"], w["D"]
    Sk, cross = keys(w), is_cross(w)
    q, k, v = make_inputs(w, rank)
    tq, tk, tv = to_dev(q, dev), to_dev(k, dev), to_dev(v, dev)
    o = torch.empty_like(tq)
    ws = (fsa.new_cross_workspace(B, H, S, Sk, D, device=dev) if cross
          else fsa.new_workspace(B, H, S, D, device=dev))
    stream = torch.cuda.current_stream(dev)
    F = flops(w)
    if args.schedule and cross:
        raise SystemExit("--schedule times self-attention workloads only")
    if args.schedule:
        run_schedules(args, w, fsa, tq, tk, tv, o, ws, stream, dev, rank)
        return

    def step(ev=None):
        for i, fmt in enumerate(FORMATS):
            if ev is not None:
                ev[i][0].record(stream)
            if cross:
                fsa.cross_attention_prepare(tq, tk, tv, ws, fmt)
            else:
                fsa.attention_prepare(tq, tk, tv, ws, fmt)
            if ev is not None:
                ev[i][1].record(stream)
            if cross:
                fsa.cross_attention_run(ws, o, Sk, fmt, THRESHOLD)
            else:
                fsa.attention_run(ws, o, fmt, THRESHOLD)
            if ev is not None:
                ev[i][2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fsa.get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in FORMATS]
           for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_start.record(stream)
        # the K steps' calls in format-major order (K calls of each format in
        # turn): the same work as K interleaved steps, each format's kernel
        # timed in steady state -- a six-bit kernel launched right after an
        # MXFP8 kernel was measured 3-4 % slower than after itself or the
        # other six-bit format, whichever six-bit format it is
        for i, fmt in enumerate(FORMATS):
            for s_i in range(args.steps):
                ev = evs[s_i][i]
                ev[0].record(stream)
                if cross:
                    fsa.cross_attention_prepare(tq, tk, tv, ws, fmt)
                else:
                    fsa.attention_prepare(tq, tk, tv, ws, fmt)
                ev[1].record(stream)
                if cross:
                    fsa.cross_attention_run(ws, o, Sk, fmt, THRESHOLD)
                else:
                    fsa.attention_run(ws, o, fmt, THRESHOLD)
                ev[2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    st = fsa.get_device_error()
    if st != 0:
        raise RuntimeError(f"device error: {fsa.status_string(st)}")
    elapsed = t_start.elapsed_time(t_end) / 1e3
    if pg:
        elapsed = max_over_ranks(elapsed, pg, dev)
    n_calls = args.steps * len(FORMATS)
    value = aggregate_tflops(world, F, n_calls, elapsed)

    per_format = {}
    for i, fmt in enumerate(FORMATS):
        t_q = [evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(args.steps)]
        t_a = [evs[s][i][1].elapsed_time(evs[s][i][2]) for s in range(args.steps)]
        ka = statistics.mean(t_a) / 1e3
        kq = statistics.mean(t_q) / 1e3
        per_format[fmt] = {
            "attention_kernel_ms": 1e3 * ka,
            "quantize_ms": 1e3 * kq,
            "attention_tflops": F / ka / 1e12,
            "with_quantize_tflops": F / (ka + kq) / 1e12,
            "quantize_gbs": (B * H * (S + 2 * Sk) * D * (2 + 1 + 1 / 32)) / kq / 1e9,
        }
    # the EFQ-Softmax producer (MXFP4 Q/K/V, E2M1 P from the shifted scores,
    # running maximum): timed on its own, not part of the headline value
    efq = None
    if not args.no_efq:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        t_q, t_a = [], []
        for s_i in range(max(1, args.warmup) + args.steps):
            ev[0].record(stream)
            if cross:
                fsa.cross_attention_prepare(tq, tk, tv, ws, "mxfp4_efq")
            else:
                fsa.attention_prepare(tq, tk, tv, ws, "mxfp4_efq")
            ev[1].record(stream)
            if cross:
                fsa.cross_attention_run(ws, o, Sk, "mxfp4_efq")
            else:
                fsa.attention_run(ws, o, "mxfp4_efq")
            ev[2].record(stream)
            torch.cuda.synchronize(dev)
            if s_i >= max(1, args.warmup):
                t_q.append(ev[0].elapsed_time(ev[1]) / 1e3)
                t_a.append(ev[1].elapsed_time(ev[2]) / 1e3)
        ka = statistics.mean(t_a)
        efq = {"attention_kernel_ms": 1e3 * ka, "quantize_ms": 1e3 * statistics.mean(t_q),
               "attention_tflops": F / ka / 1e12,
               "note": "EFQ-Softmax producer: MXFP4 Q/K/V, running row maximum, E2M1 P"}
        if fsa.get_device_error() != 0:
            raise RuntimeError("device error in the EFQ format")

    # the shortcut rollback gate ("Fused-Softmax shifts ...", paragraph 12)
    # against the FP32 gate on the same workload: the attention kernel alone
    shortcut = None
    if not args.no_shortcut and not cross:
        shortcut = {}
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for fmt in FORMATS:
            fsa.attention_prepare(tq, tk, tv, ws, fmt)
            ts = []
            for s_i in range(1 + max(1, args.steps // 2)):
                ev[0].record(stream)
                fsa.attention_run(ws, o, fmt, THRESHOLD, gate="shortcut")
                ev[1].record(stream)
                torch.cuda.synchronize(dev)
                if s_i:
                    ts.append(ev[0].elapsed_time(ev[1]) / 1e3)
            ka = statistics.mean(ts)
            shortcut[fmt] = {"attention_kernel_ms": 1e3 * ka, "attention_tflops": F / ka / 1e12,
                             "vs_fp32_gate": per_format[fmt]["attention_kernel_ms"] / (1e3 * ka)}
        if fsa.get_device_error() != 0:
            raise RuntimeError("device error with the shortcut gate")

    # in-house BF16 flash-attention baseline, same inputs
    bf16 = None
    if not args.no_bf16 and not cross:  # the BF16 kernel is self-attention only
        fsa.bf16_attention_fwd(tq, tk, tv, out=o)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        nb = max(2, args.steps)
        e0.record(stream)
        for _ in range(nb):
            fsa.bf16_attention_fwd(tq, tk, tv, out=o)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        tb = e0.elapsed_time(e1) / 1e3 / nb
        bf16 = {"kernel_ms": 1e3 * tb, "tflops": F / tb / 1e12}
        for fmt in FORMATS:
            per_format[fmt]["speedup_vs_bf16_kernel"] = tb / (per_format[fmt]["attention_kernel_ms"] / 1e3)

    # end to end through the public host-buffer call: pinned host in, pinned host out
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (torch.empty_like(t, device="cpu").pin_memory() for t in (tq, tk, tv))
        for h, t in ((hq, tq), (hk, tk), (hv, tv)):
            h.copy_(t)
        ho = torch.empty_like(o, device="cpu").pin_memory()

        def e2e_call(fmt):
            # the host inputs are final: consecutive calls overlap their copies
            if cross:
                fsa.cross_attention_fwd_host(hq, hk, hv, fmt=fmt, threshold=THRESHOLD, out=ho,
                                             host_inputs_ready=True)
            else:
                fsa.attention_fwd_host(hq, hk, hv, fmt=fmt, threshold=THRESHOLD, out=ho,
                                       host_inputs_ready=True)

        for fmt in FORMATS:
            e2e_call(fmt)
        torch.cuda.synchronize(dev)
        if pg:
            pg.barrier()
        # an event after every call, so that the line also shows how evenly
        # the calls ran (each call's span on the caller's stream)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(FORMATS) * args.steps + 1)]
        evs[0].record(stream)
        n_ev = 1
        for fmt in FORMATS:            # format-major, as the device-timed region
            for _ in range(args.steps):
                e2e_call(fmt)
                evs[n_ev].record(stream)
                n_ev += 1
        torch.cuda.synchronize(dev)
        te = evs[0].elapsed_time(evs[-1]) / 1e3
        spans = [evs[i].elapsed_time(evs[i + 1]) for i in range(len(evs) - 1)]
        if pg:
            te = max_over_ranks(te, pg, dev)
        nbytes = tq.numel() * 2
        e2e = {"value": aggregate_tflops(world, F, n_calls, te), "unit": "TFLOP/s",
               "h2d_bytes_per_step": len(FORMATS) * (nbytes + 2 * tk.numel() * 2),
               "d2h_bytes_per_step": len(FORMATS) * nbytes,
               "call": "fsa_attention_fwd_host per format (pinned host buffers; chunks of heads "
                       "with copies overlapping compute)",
               "call_ms": {fmt: [round(x, 2) for x in spans[i * args.steps:(i + 1) * args.steps]]
                           for i, fmt in enumerate(FORMATS)}}
        if fsa.get_device_error() != 0:
            raise RuntimeError("device error during e2e")
        # the box's pinned host copy rates, to read the end-to-end figure by:
        # one direction alone, then both at once (the pipeline's case)
        e2e["host_copy_gbs"] = host_copy_rates(hq, ho, dev)
        e2e["copy_ms_per_step_at_these_rates"] = 1e3 * max(
            e2e["h2d_bytes_per_step"] / (1e9 * e2e["host_copy_gbs"]["h2d_while_d2h"]),
            e2e["d2h_bytes_per_step"] / (1e9 * e2e["host_copy_gbs"]["d2h_while_h2d"]))

    # the other benchmark workloads, then the tensor-core rate probe
    # (last: it runs the GPU into its power cap)
    configs = None
    if not args.no_configs and not cross:
        configs = run_configs(fsa, dev, stream, rank)
    mma = None
    if not args.no_mma_probe:
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        mma = measure_mma_peaks(fsa, dev, stream, n_sm)
    pk = peaks(mma)
    for fmt in FORMATS:
        pf = per_format[fmt]
        pf["frac_of_mx_mma_peak"] = pf["attention_tflops"] / pk["mx8_sustained"]
        pf["frac_of_format_roofline"] = pf["attention_tflops"] / format_roofline(pk, fmt)
        if pk["attn_tile_sustained"]:
            pf["frac_of_attention_tile_mma_rate"] = pf["attention_tflops"] / pk["attn_tile_sustained"]
    if efq:
        efq["frac_of_mx_mma_peak"] = efq["attention_tflops"] / pk["mx8_sustained"]
        efq["frac_of_format_roofline"] = efq["attention_tflops"] / format_roofline(pk, "mxfp4")
    if bf16:
        bf16["frac_of_bf16_peak"] = bf16["tflops"] / pk["bf16_sustained"]
    if configs:
        add_config_fracs(configs, pk)

    if rank != 0:
        return

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        threads, affinity = cpu_affinity()
        f, t, n_used = oracle_sample(q, k, v, w, "mxfp8", args.cpu_rows, threads)
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": threads, "affinity": affinity,
               "kind": "oracle",
               "sample": f"{n_used} query rows evenly spaced from head 0 on (all {Sk} keys), MXFP8, "
                         f"{t:.1f} s; rows are independent so the rate extrapolates exactly"}

    a8 = per_format["mxfp8"]
    # work items of at most 16 KV tiles run the persistent variant
    kname = "fsa_attn_fwd_persistent_kernel" if Sk <= 16 * 128 else "fsa_attn_fwd_kernel"
    roof = {"bound": "tensor", "kernel": f"{kname} (MXFP8)",
            "achieved": a8["attention_tflops"], "peak": pk["mx8_sustained"], "unit": "TFLOP/s",
            "frac": a8["attention_tflops"] / pk["mx8_sustained"],
            "peak_note": (f"dense E4M3 block-scaled MMA (kind::mxf8f6f4) rate, {pk['mx_source']}: "
                          f"sustained {pk['mx8_sustained']:.1f}, burst {pk['mx8_burst']:.1f} TFLOP/s; "
                          "one CTA per SM issuing M=128 N=256 K=32 products back to back"),
            "algorithmic_flops_per_launch": F,
            # DRAM counters exist for the default workload's kernel only
            "traffic": traffic_from_profiles() if args.workload == "video-dit" else None}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "mx (e4m3|e2m3|e2m1 x e8m0) mma, fp32 accumulate",
        "data": "synthetic N(0,1) bf16, seed = rank",
        "config": bench_config(args, w),
        "per_format": per_format,
        "bf16_baseline": bf16,
        "efq_format": efq,
        "shortcut_gate": shortcut,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "mma_peaks": mma,
        "configs": configs,
        "gpu_launches": args.steps * len(FORMATS) * 4,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
