#!/usr/bin/env python3
"""Benchmark of the gated delta rule hot path on GB300.

Default workload (the one the headline metric is quoted on): batched decode
of all 48 GDN layers of one token -- batch 32, NK = 16 key heads, NV = 48 value
heads (g = h mod 16), D = 128, fp32 state [32][48 layers][48][128][128]
(4.83 GB, larger than L2), one fused decode + gated-RMS-norm launch per layer
with its own seeded inputs, bf16 output.  One step = the 48 layer launches.

value  = token-heads/s with inputs resident in HBM (device-timed, CUDA events).
e2e    = the same through the public API with the step's token inputs copied
         host->device from pinned memory and the bf16 outputs written by the
         kernels into pinned host memory, inside the timed region (the state
         stays resident, as it does in a model).
roofline = the decode kernel's algorithmic HBM bytes per launch / its average
         launch time, against the measured HBM copy bandwidth.
cpu_baseline = the fp64 oracle, as it stands, on this host's cores over a
         bounded sample of the same workload.

Other rows of the hot path are measured under "rows" (fp16 pool decode,
h-state converters, single-layer latency, prefill).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs the per-GPU workload on its own GPU (weak
scaling, no collective in the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN state-update token-heads/s and achieved HBM GB/s (% of GB300 peak)"
UNIT = "token-heads/s"

# The workload.
B, NK, NV, D, LAYERS = 32, 16, 48, 128, 48
EPS = 1e-6
SEED = 0
REF_LAYERS_PER_STEP = 4      # oracle sample per step of the reference arm

# Per-launch DRAM traffic of a kernel from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), valid only while the kernel source is the one it was taken on.
NCU_TRAFFIC = {
    # mean of three mid-sequence launches of the full 48-layer workload, ncu --cache-control none
    # (reads 102.8 MB, writes 96.7-99.8 MB), from the ncu capture of the batch-32 48-layer decode
    "decode_norm_f32": {"bytes_per_launch": 201338539,
                        "src_sha256": "d7ef0560d8c7516145aea11e87782e28b1a70a1a80d9dd698ca3c8112066c8e8"},
    # mean of two launches of the 256-slot fp16 pool decode (reads 407.2-407.4 MB, writes 401.5-403.3 MB)
    "decode_norm_f16_pool": {"bytes_per_launch": 809747200,
                             "src_sha256": "d7ef0560d8c7516145aea11e87782e28b1a70a1a80d9dd698ca3c8112066c8e8"},
    # mean of two launches of the batch-32 fp32 decode from projections (reads 105.8-105.9 MB, writes
    # 102.8-104.3 MB), ncu --cache-control none
    "conv_norm_f32": {"bytes_per_launch": 209422848, "src": ("gdn_conv_norm.cu", "gdn_internal.cuh"),
                      "src_sha256": "991c5e322697d68f73e5a6a2a814c7162e42213e32d33b2904ca68f9be87a61e"},
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the secondary rows")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-graph", action="store_true", help="launch every kernel from Python instead of "
                    "replaying a captured CUDA graph")
    ap.add_argument("--layers", type=int, default=None,
                    help="fewer layers (a smaller case for profiling; not a bench line)")
    ap.add_argument("--prefill-tokens", type=int, default=4096,
                    help="tokens per sequence in the prefill row (smaller for profiling; not a bench line)")
    ap.add_argument("--rows-only", default=None,
                    help="comma list of secondary rows to run (profiling): fp16,conv,latency,prefill,chunk2,convnorm,q8")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "source": "measured", "sm_max_mhz": j.get("sm_max_mhz")}
    return {"hbm_gbs": 6800.0, "source": "fallback", "sm_max_mhz": 2070.0}


def tf32_peak_flops(pk):
    """Dense TF32 tensor peak: the measured bf16 burst peak times the nominal TF32 / bf16 ratio
    (1.1 / 2.25 PFLOP/s), or the fallback bf16 figure when no measured file is present."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    bf16, src = 1.9e15, "fallback 1.9 PFLOP/s bf16"
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        if j.get("bf16_tflops"):
            bf16, src = float(j["bf16_tflops"]) * 1e12, f"measured {j['bf16_tflops']} TFLOP/s bf16 burst"
    return bf16 * 1.1 / 2.25, src + " x 1.1/2.25 (nominal TF32/bf16)"


def pinned_traffic(key):
    """ncu DRAM bytes per launch for NCU_TRAFFIC[key], or None once the kernel source has changed."""
    tr = NCU_TRAFFIC[key]
    src = tr.get("src", ("gdn_decode.cu", "gdn_internal.cuh"))
    return tr["bytes_per_launch"] if tr["src_sha256"] == src_sha(*src) else None


def src_sha(*names):
    """sha256 over the named kernel sources, in order (the kernel and the header it includes)."""
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "gated_deltanet_linear_16_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 5 ms (as fast as nvidia-smi delivers) while
    running; summary() covers the samples between two marks."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        # nvidia-smi numbers GPUs physically; the process may see a remapped index, so use the UUID
        self.gpu = gpu_index
        try:
            import torch
            self.gpu = "GPU-" + str(torch.cuda.get_device_properties(gpu_index).uuid)
        except Exception:
            pass
        self.proc = None
        self.path = os.path.join("/tmp", f"gdn_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "5"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def mark(self, which):
        """Record the wall-clock start or end of the timed region."""
        setattr(self, which, datetime.datetime.now())

    def summary(self, lo_mark="start", hi_mark="end", keep=False):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons, pw = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo, hi = getattr(self, lo_mark, None), getattr(self, hi_mark, None)
        lines = [[p.strip() for p in line.split(",")] for line in open(self.path)]
        lines = [p for p in lines if len(p) >= 9]

        def when(p):
            try:
                return datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                return None

        inside = [p for p in lines if lo and hi and when(p) and lo <= when(p) <= hi]
        if not inside and lines and lo:
            # region shorter than the sampling period: the samples nearest to it
            after = [p for p in lines if when(p) and when(p) >= lo]
            inside = after[:1] or lines[-1:]
        for parts in inside:
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not keep:
            os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "window_s": (hi - lo).total_seconds() if lo and hi else None,
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons)}


# ------------------------------------------------------------------ workload buffers

def algorithmic_bytes_decode(batch, nk, nv, d, state_elem=4, norm=True):
    """Bytes one decode launch must move at minimum: the state read and written once,
    every token input read once, the output written once."""
    state = batch * nv * d * d * state_elem * 2
    qk = batch * nk * d * 4 * 2
    v = batch * nv * d * 4
    gb = batch * nv * 4 * 2
    if norm:
        z = batch * nv * d * 4
        gn = d * 4
        out = batch * nv * d * 2
    else:
        z = gn = 0
        out = batch * nv * d * 4
    return state + qk + v + gb + z + gn + out


def make_layer_inputs(torch, batch, layers, dev):
    """Seeded token inputs for every layer, resident on the device: dict of [L][...] tensors."""
    import gdn_synth as gs
    xs = [gs.decode_inputs(SEED, batch, NK, NV, D, layer=l) for l in range(layers)]
    out = {}
    for name in ("q", "k", "v", "z", "alpha", "beta"):
        out[name] = torch.from_numpy(np.stack([x[name] for x in xs])).to(dev)
    gn = np.stack([gs.norm_weight(SEED, D, layer=l) for l in range(layers)])
    out["gn"] = torch.from_numpy(gn).to(dev)
    return out


def layer_launch(gdn, state, x, outb, l, stream_ptr, batch=B, f16=False, pitch=None):
    """One fused decode + norm launch for layer l (state layout [batch][layer][NV][D][D];
    `pitch` = state elements between sequences, default all layers of the state tensor)."""
    esz = 2 if f16 else 4
    pitch = state.stride(0) if pitch is None else pitch
    gdn.gdn_decode_norm(state.data_ptr() + l * NV * D * D * esz,
                        x["q"][l], x["k"][l], x["v"][l], x["alpha"][l], x["beta"][l],
                        x["z"][l], x["gn"][l], outb[l],
                        batch=batch, nk=NK, nv=NV, d=D, eps=EPS, state_pitch=pitch,
                        state_dtype=1 if f16 else 0, stream=stream_ptr)


# ------------------------------------------------------------------ launch submission

def graphed(torch, fn, stream, enable=True):
    """Capture fn's launches once into a CUDA graph and return a replay function (the way a
    decode step is replayed in a serving loop); falls back to calling fn directly if the
    capture is not possible.  Returns (callable, used_graph)."""
    if not enable:
        return fn, False
    try:
        fn()                                   # warm (first-call set-up outside the capture)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        torch.cuda.synchronize()
        return g.replay, True
    except Exception:                          # capture unsupported here: plain launches
        torch.cuda.synchronize()
        return fn, False


# ------------------------------------------------------------------ multi-rank host logic

def max_over_ranks(ms_step, world, device):
    """Slowest rank's time per step (every rank's work counts only once all finish)."""
    if world <= 1:
        return ms_step
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_step], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms_step):
    """Whole-job units per second: every rank processes its own units (weak scaling)."""
    return world * units_per_rank / (ms_step / 1e3)


# ------------------------------------------------------------------ our arm

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import gated_deltanet_linear_16_gb300 as gdn

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    gdn.load()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    # state: [B][L][NV][D][D] fp32, N(0, 0.02), drawn on the device (values do not affect timing)
    g = torch.Generator(device=dev)
    g.manual_seed(SEED + rank)
    L = args.layers or LAYERS
    state = torch.empty((B, L, NV, D, D), dtype=torch.float32, device=dev)
    for b in range(B):
        state[b].normal_(0.0, 0.02, generator=g)
    x = make_layer_inputs(torch, B, L, dev)
    outb = torch.empty((L, B, NV * D), dtype=torch.int16, device=dev)

    def launches():
        # stream None: the binding launches on the current stream (the capture stream while
        # the graph is being captured)
        for l in range(L):
            layer_launch(gdn, state, x, outb, l, None)

    cap = torch.cuda.Stream(device=dev)
    step, used_graph = graphed(torch, launches, cap, enable=not args.no_graph)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        time.sleep(0.3)                       # let the sampler start before the timed region
        torch.cuda.synchronize()
        clk.mark("start")
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        clk.mark("end")
        # a timed region of a few tens of ms holds few clock samples: the same step replayed, untimed,
        # for a quarter second more gives the clocks under the same load a fuller record
        short = (clk.end - clk.start).total_seconds() < 0.25
        if short:
            clk.mark("after_start")
            t_end = time.time() + 0.25
            while time.time() < t_end:
                step()
                torch.cuda.synchronize()
            clk.mark("after_end")
        time.sleep(0.05)
    if world > 1:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    ms_step = max_over_ranks(ms / args.steps, world, dev)
    clocks = clk.summary(keep=short)
    if short:
        after = clk.summary("after_start", "after_end")
        if clocks is not None:
            clocks["after_timed_region"] = after

    token_heads = B * NV * L
    value = job_throughput(token_heads, world, ms_step)
    bytes_launch = algorithmic_bytes_decode(B, NK, NV, D)
    launch_s = ms_step / 1e3 / L
    pk = peaks()
    achieved = bytes_launch / launch_s / 1e9
    traffic = pinned_traffic("decode_norm_f32")

    # ---- e2e: host inputs in pinned memory -> device, 48 launches, bf16 outputs -> host
    e2e = None if args.no_e2e else run_e2e(args, torch, gdn, state, x, outb, dev, stream, not args.no_graph)
    if e2e is not None and world > 1:          # whole job: the slowest rank's step, every rank's units
        e2e["ms_per_step"] = max_over_ranks(e2e["ms_per_step"], world, dev)
        e2e["value"] = job_throughput(B * NV * L, world, e2e["ms_per_step"])
    del state, x, outb
    torch.cuda.empty_cache()

    rows = {} if args.no_rows else run_rows(torch, gdn, dev, stream, pk, args.rows_only, args.prefill_tokens,
                                            graph=not args.no_graph)
    cpu = None if (args.no_cpu or rank != 0) else cpu_baseline(sample_layers=None)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "batched decode + fused gated RMSNorm, all 48 GDN layers of one token",
                   "batch_per_gpu": B, "global_batch": B * world, "nk": NK, "nv": NV, "d": D,
                   "layers": L, "state": f"fp32 [32][{L}][48][128][128] = {B * L * NV * D * D * 4 / 1e9:.2f} GB per GPU",
                   "out": "bf16", "eps": EPS, "launches_per_step": L,
                   "l2": "inputs larger than L2 (4.83 GB state per step vs 129 MB L2)",
                   "submission": "one CUDA graph replay per step" if used_graph else "eager launches",
                   "parallelism": f"dp{world}"},
        "roofline": {"bound": "hbm", "kernel": "decode_d128<float, norm>", "achieved": achieved,
                     "peak": pk["hbm_gbs"], "peak_source": pk["source"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                     "algorithmic_bytes_per_launch": bytes_launch, "launch_us": launch_s * 1e6},
        "e2e": e2e,
        "gpu_launches": L * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "rows": rows,
    }
    return line


def run_e2e(args, torch, gdn, state, x, outb, dev, stream, graph=True):
    """Same workload through the public API with the step's inputs and outputs on the host: every
    layer's token inputs copied from pinned host memory to the device, the layer calls, every layer's
    bf16 output written by the kernel straight into pinned host memory (device-accessible over the
    host link), so the step's result is on the host when its last kernel completes.  The input copies
    run on a second stream, layer by layer, so layer l + 1's inputs travel while layer l computes; no
    copy or event sits between two layers' kernels, which keep their early launch.  The whole step is
    captured once into a CUDA graph and replayed, as a serving loop would (unless graph is False).
    (Copying the outputs back per group of 8 layers instead, each copy after an event between two
    kernels, measured 1.021 of the device-only step against 1.000-1.002 this way.)"""
    host = {k: v.cpu().pin_memory() for k, v in x.items() if k != "gn"}
    dev_in = {k: torch.empty_like(v) for k, v in host.items()}
    dev_in["gn"] = x["gn"]
    host_out = torch.empty(outb.shape, dtype=outb.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = host_out.numel() * host_out.element_size()

    L = outb.shape[0]
    copy = torch.cuda.Stream(device=dev)

    def launches():
        cur = torch.cuda.current_stream()
        copy.wait_stream(cur)                     # fork the copy stream off the step
        ready = []
        with torch.cuda.stream(copy):
            for l in range(L):
                for k, v in host.items():
                    dev_in[k][l].copy_(v[l], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy)
                ready.append(ev)
        for l in range(L):
            cur.wait_event(ready[l])
            layer_launch(gdn, state, dev_in, host_out, l, None)
        cur.wait_stream(copy)                     # join the copy stream

    step, used = graphed(torch, launches, torch.cuda.Stream(device=dev), enable=graph)
    steps = max(3, args.steps)
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": B * NV * outb.shape[0] / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "steps": steps,
            "submission": ("one CUDA graph replay per step; per-layer input copies from pinned host memory on a "
                           "second stream overlap the layers' kernels; the kernels write the bf16 outputs "
                           "straight into pinned host memory")
                          if used else "eager, per-layer input copies on a second stream, outputs written to "
                                       "pinned host memory by the kernels",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


# ------------------------------------------------------------------ secondary rows

def time_fn(torch, stream, fn, reps, warm=2):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps / 1e3     # seconds per call


# Rows on one layer at batch 32 (100 MB of fp32 state, under the 129 MB L2) cycle through this many
# layers' states, so every launch streams its state from HBM as a model's layers do.
ROW_LAYERS = 8


def cycling(fns):
    """One callable that runs fns[0], fns[1], ... in turn, one per call."""
    it = [0]

    def call():
        fns[it[0] % len(fns)]()
        it[0] += 1
    return call


def run_rows(torch, gdn, dev, stream, pk, only=None, prefill_tokens=4096, graph=True):
    want = set(only.split(",")) if only else {"fp16", "conv", "latency", "prefill", "chunk2", "convnorm", "q8"}
    rows = {}
    torch.cuda.empty_cache()
    if want & {"fp16", "conv"}:
        rows.update(row_fp16_pool(torch, gdn, dev, stream, pk, want))
    if "latency" in want:
        rows.update(row_latency(torch, gdn, dev, stream, graph))
        rows.update(row_tiny(torch, gdn, dev, stream))
    if "chunk2" in want:
        rows.update(row_chunk2(torch, gdn, dev, stream, pk))
    if "convnorm" in want:
        rows.update(row_conv_norm(torch, gdn, dev, stream, pk))
    if "q8" in want:
        rows.update(row_q8(torch, gdn, dev, stream, pk))
    if "prefill" in want:
        rows.update(row_prefill(torch, gdn, dev, stream, pk, prefill_tokens))
    return rows


def row_conv_norm(torch, gdn, dev, stream, pk, taps=4):
    """Fused decode from projections (conv ring update + silu, q/k L2 norm, gates from logits, the
    step and the gated norm in one launch): batch 32 with fp32 states, ROW_LAYERS layers' states and
    conv rings in turn (also through the allocation-free entry point), and the 256-slot fp16 pool."""
    import gdn_synth as gs
    C = (2 * NK + NV) * D
    res = {}
    for label, batch, f16 in (("fp32_b32", B, False), ("fp16_pool_b256", 256, True)):
        x = gs.conv_decode_inputs(SEED, batch, NK, NV, D, taps)
        t = {k: torch.from_numpy(v).to(dev) for k, v in x.items()}
        g = torch.Generator(device=dev)
        g.manual_seed(3)
        nl = 1 if f16 else ROW_LAYERS                  # the fp16 pool (403 MB) is larger than L2 alone
        S = torch.empty((nl, batch, NV * D * D), device=dev).normal_(0.0, 0.02, generator=g)
        if f16:
            S = S.half()
        ring = t["ring"].reshape(1, batch, taps * C).repeat(nl, 1, 1).contiguous()
        gn = torch.from_numpy(gs.norm_weight(SEED, D)).to(dev)
        out = torch.empty((batch, NV * D), dtype=torch.int16, device=dev)
        ws = torch.zeros(batch * NK, dtype=torch.int32, device=dev)
        args = [(S[l], ring[l], t["x"], t["conv_w"], t["br"], t["ar"], t["dt"], t["rate"], t["z"], gn, out)
                for l in range(nl)]
        kw = dict(batch=batch, nk=NK, nv=NV, d=D, taps=taps, stream=stream.cuda_stream)
        s = time_fn(torch, stream, cycling([lambda a=a: gdn.gdn_decode_conv_norm(*a, ws, **kw) for a in args]),
                    48 if not f16 else 20)
        es = 2 if f16 else 4
        # state read + write; ring: taps-1 entries read, all taps written; x, z read; w, dt, rate, gn
        # once; gate logits read; bf16 out written
        by = (batch * NV * D * D * es * 2 + batch * ((taps - 1) + taps + 1) * C * 4 + taps * C * 4
              + batch * NV * D * 4 + batch * NV * 2 * 4 + 2 * NV * 4 + D * 4 + batch * NV * D * 2)
        r = {"config": f"B={batch} NK=16 NV=48 D=128 {'fp16' if f16 else 'fp32'}, 4-tap conv"
                       + ("" if f16 else f", {nl} layers' states in turn"),
             "us_per_launch": s * 1e6, "token_heads_per_s": batch * NV / s, "achieved_gbs": by / s / 1e9,
             "frac_of_hbm_peak": by / s / 1e9 / pk["hbm_gbs"], "algorithmic_bytes": by}
        if not f16:
            r["traffic"] = pinned_traffic("conv_norm_f32")
        if not f16:
            s2 = time_fn(torch, stream, cycling([lambda a=a: gdn.gdn_decode_conv_norm_noalloc(*a, **kw)
                                                 for a in args]), 48)
            r["noalloc_us_per_launch"] = s2 * 1e6
        res[label] = r
        del S, ring, gn, out, t, ws, args
        torch.cuda.empty_cache()
    return {"conv_norm_from_projections": res}


def row_q8(torch, gdn, dev, stream, pk):
    """Decode + gated norm with the int8 epilogue (groups of 32, one fp32 scale each) at batch 32
    (fp32 states, ROW_LAYERS layers' states in turn), next to the bf16 epilogue on the same inputs."""
    g = torch.Generator(device=dev)
    g.manual_seed(4)
    S = torch.empty((ROW_LAYERS, B, NV, D, D), device=dev).normal_(0.0, 0.02, generator=g)
    q = torch.randn((B, NK, D), device=dev, generator=g)
    q = (q / q.norm(dim=-1, keepdim=True)).view(B, NK * D).contiguous()
    k = torch.randn((B, NK, D), device=dev, generator=g)
    k = (k / k.norm(dim=-1, keepdim=True)).view(B, NK * D).contiguous()
    v = torch.randn((B, NV * D), device=dev, generator=g)
    z = torch.randn((B, NV * D), device=dev, generator=g)
    a = torch.sigmoid(torch.randn((B, NV), device=dev, generator=g) + 2.0)
    bt = torch.sigmoid(torch.randn((B, NV), device=dev, generator=g))
    gn = torch.ones(D, device=dev)
    xq = torch.empty((B, NV * D), dtype=torch.int8, device=dev)
    xs = torch.empty((B, NV * D // 32), device=dev)
    out = torch.empty((B, NV * D), dtype=torch.int16, device=dev)
    kw = dict(batch=B, nk=NK, nv=NV, d=D, stream=stream.cuda_stream)
    s_q8 = time_fn(torch, stream, cycling([lambda l=l: gdn.gdn_decode_norm_q8(S[l], q, k, v, a, bt, z, gn, xq, xs,
                                                                            None, **kw) for l in range(ROW_LAYERS)]), 48)
    s_bf = time_fn(torch, stream, cycling([lambda l=l: gdn.gdn_decode_norm(S[l], q, k, v, a, bt, z, gn, out, **kw)
                                           for l in range(ROW_LAYERS)]), 48)
    by = B * NV * D * D * 4 * 2 + B * (2 * NK * D + 2 * NV * D + 2 * NV) * 4 + D * 4 + B * NV * D * (1 + 4 / 32)
    del S, q, k, v, z, a, bt, gn, xq, xs, out
    torch.cuda.empty_cache()
    return {"decode_norm_int8_epilogue": {
        "config": f"B=32 NK=16 NV=48 D=128 fp32, int8 codes + fp32 scale per 32 outputs, {ROW_LAYERS} layers' "
                  "states in turn", "us_per_launch": s_q8 * 1e6,
        "bf16_epilogue_us_per_launch": s_bf * 1e6, "achieved_gbs": by / s_q8 / 1e9,
        "frac_of_hbm_peak": by / s_q8 / 1e9 / pk["hbm_gbs"], "algorithmic_bytes": by}}


def row_chunk2(torch, gdn, dev, stream, pk):
    """Two-token verify step at batch 32 (fp32 states, ROW_LAYERS layers' states in turn) and on the
    256-slot fp16 pool: the state is read once and written twice (intermediate + final); both
    tokens' inputs read, both outputs written."""
    res = {}
    for label, batch, f16 in (("fp32_b32", B, False), ("fp16_pool_b256", 256, True)):
        g = torch.Generator(device=dev)
        g.manual_seed(2)
        nl = 1 if f16 else ROW_LAYERS
        S = torch.empty((nl, batch, NV, D, D), device=dev).normal_(0.0, 0.02, generator=g)
        if f16:
            S = S.half()
        M = torch.empty_like(S)
        R = 2 * batch
        q = torch.randn((R, NK * D), device=dev, generator=g)
        k = torch.randn((R, NK * D), device=dev, generator=g)
        q = (q.view(R, NK, D) / q.view(R, NK, D).norm(dim=-1, keepdim=True)).view(R, NK * D).contiguous()
        k = (k.view(R, NK, D) / k.view(R, NK, D).norm(dim=-1, keepdim=True)).view(R, NK * D).contiguous()
        v = torch.randn((R, NV * D), device=dev, generator=g)
        a = torch.sigmoid(torch.randn((R, NV), device=dev, generator=g) + 2.0)
        bt = torch.sigmoid(torch.randn((R, NV), device=dev, generator=g))
        o = torch.empty((R, NV * D), device=dev)
        s = time_fn(torch, stream, cycling([lambda l=l: gdn.gdn_decode_chunk2(S[l], M[l], q, k, v, a, bt, o, batch=batch,
                                                                             nk=NK, nv=NV, d=D,
                                                                             stream=stream.cuda_stream)
                                            for l in range(nl)]), 48 if not f16 else 20)
        es = 2 if f16 else 4
        by = batch * NV * D * D * es * 3 + R * (2 * NK * D + 2 * NV * D + 2 * NV) * 4
        res[label] = {"config": f"B={batch} NK=16 NV=48 D=128 {'fp16' if f16 else 'fp32'}, two tokens per launch"
                                + ("" if f16 else f", {nl} layers' states in turn"),
                      "us_per_launch": s * 1e6, "token_heads_per_s": R * NV / s,
                      "achieved_gbs": by / s / 1e9, "frac_of_hbm_peak": by / s / 1e9 / pk["hbm_gbs"],
                      "algorithmic_bytes": by}
        del S, M, q, k, v, a, bt, o
        torch.cuda.empty_cache()
    return {"chunk2_verify": res}


def row_fp16_pool(torch, gdn, dev, stream, pk, want):
    """fp16 h-state pool (B=256 slots, pitch 48*128*128 + 4096 halves): fused decode steps, and the
    f16 -> f32 -> f16 converter round trip over the whole pool (padding included)."""
    sp = stream.cuda_stream
    rows = {}
    PB, pitch = 256, NV * D * D + 4096
    pool = torch.zeros(PB * pitch, dtype=torch.float16, device=dev)
    pool.view(PB, pitch)[:, :NV * D * D].normal_(0.0, 0.02)
    if "conv" in want:
        n = PB * pitch
        f32 = torch.empty(n, dtype=torch.float32, device=dev)
        back = torch.empty(n, dtype=torch.float16, device=dev)
        s_up = time_fn(torch, stream, lambda: gdn.gdn_h_f16_to_f32(pool, f32, n, stream=sp), 10)
        s_dn = time_fn(torch, stream, lambda: gdn.gdn_h_f32_to_f16(f32, back, n, stream=sp), 10)
        rows["h_state_converters"] = {
            "elements": n, "f16_to_f32_us": s_up * 1e6, "f32_to_f16_us": s_dn * 1e6,
            "f16_to_f32_gbs": 6 * n / s_up / 1e9, "f32_to_f16_gbs": 6 * n / s_dn / 1e9,
            "frac_of_hbm_peak": [6 * n / s_up / 1e9 / pk["hbm_gbs"], 6 * n / s_dn / 1e9 / pk["hbm_gbs"]],
            "round_trip_identity": bool(torch.equal(back.view(torch.int16), pool.view(torch.int16)))}
        del f32, back
        torch.cuda.empty_cache()
    if "fp16" in want:
        x = make_layer_inputs(torch, PB, 1, dev)
        ob = torch.empty((1, PB, NV * D), dtype=torch.int16, device=dev)
        s = time_fn(torch, stream,
                    lambda: layer_launch(gdn, pool, x, ob, 0, sp, batch=PB, f16=True, pitch=pitch), 16)
        by = algorithmic_bytes_decode(PB, NK, NV, D, state_elem=2)
        rows["fp16_pool_decode_norm"] = {
            "config": "B=256 NK=16 NV=48 D=128, fp16 pool pitch 790528 halves, fused norm -> bf16",
            "us_per_step": s * 1e6, "token_heads_per_s": PB * NV / s, "achieved_gbs": by / s / 1e9,
            "frac_of_hbm_peak": by / s / 1e9 / pk["hbm_gbs"], "algorithmic_bytes": by,
            "traffic": pinned_traffic("decode_norm_f16_pool")}
        del x, ob
    del pool
    torch.cuda.empty_cache()
    return rows


def row_latency(torch, gdn, dev, stream, graph=True):
    """One layer, batch 1 (3 MB state, L2-resident across steps): time per fused decode step,
    256 sequential steps replayed from one CUDA graph (launch submission excluded)."""
    cap = torch.cuda.Stream(device=dev)
    st = torch.empty((1, NV, D, D), dtype=torch.float32, device=dev).normal_(0.0, 0.02)
    x1 = make_layer_inputs(torch, 1, 1, dev)
    o1 = torch.empty((1, 1, NV * D), dtype=torch.int16, device=dev)
    n = 256

    def steps():
        for _ in range(n):
            layer_launch(gdn, st, x1, o1, 0, None, batch=1, pitch=NV * D * D)

    fn, used = graphed(torch, steps, cap, enable=graph)
    s = time_fn(torch, stream, fn, 4) / n
    return {"single_layer_latency": {"config": "B=1 NK=16 NV=48 D=128 fp32, fused norm (L2-resident)",
                                     "submission": "CUDA graph of 256 steps" if used else "eager launches",
                                     "us_per_step": s * 1e6, "token_heads_per_s": NV / s}}


def row_tiny(torch, gdn, dev, stream):
    """The pages' tiny configuration (batch 1, NK 1, NV 2, D 4, fp32 state from zero): 64 sequential
    decode steps with the fused norm, captured as one CUDA graph; latency per step."""
    import gdn_synth as gs
    T, nk, nv, d = 64, 1, 2, 4
    xs = [gs.decode_inputs(SEED, 1, nk, nv, d, step=t) for t in range(T)]
    t_in = {k: torch.from_numpy(np.stack([x[k] for x in xs])).to(dev) for k in ("q", "k", "v", "alpha", "beta", "z")}
    gn = torch.from_numpy(gs.norm_weight(SEED, d)).to(dev)
    S = torch.zeros((1, nv, d, d), device=dev)
    out = torch.empty((T, nv * d), dtype=torch.int16, device=dev)

    def steps():
        for t in range(T):
            gdn.gdn_decode_norm(S, t_in["q"][t], t_in["k"][t], t_in["v"][t], t_in["alpha"][t], t_in["beta"][t],
                                t_in["z"][t], gn, out[t], batch=1, nk=nk, nv=nv, d=d, eps=EPS, stream=None)

    run, used = graphed(torch, steps, torch.cuda.Stream(device=dev))
    s = time_fn(torch, stream, run, 20)
    del S, out, t_in
    return {"tiny_config_latency": {"config": "B=1 NK=1 NV=2 D=4 fp32, 64 sequential steps, fused norm",
                                    "submission": "CUDA graph of 64 steps" if used else "eager",
                                    "us_per_step": s / T * 1e6}}


def row_prefill(torch, gdn, dev, stream, pk, T=4096):
    """Prefill: B=8, T tokens in one call, fp32 state from zero (inputs drawn on the device at the
    generator's distributions; values do not change the timing)."""
    sp = stream.cuda_stream
    PB = 8
    R = PB * T
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    q = torch.randn((R, NK * D), device=dev, generator=g)
    k = torch.randn((R, NK * D), device=dev, generator=g)
    q = (q.view(R, NK, D) / q.view(R, NK, D).norm(dim=-1, keepdim=True)).view(R, NK * D).contiguous()
    k = (k.view(R, NK, D) / k.view(R, NK, D).norm(dim=-1, keepdim=True)).view(R, NK * D).contiguous()
    v = torch.randn((R, NV * D), device=dev, generator=g)
    a = torch.sigmoid(torch.randn((R, NV), device=dev, generator=g) + 2.0)
    bt = torch.sigmoid(torch.randn((R, NV), device=dev, generator=g))
    o = torch.empty((R, NV * D), device=dev)
    S = torch.zeros((PB, NV, D, D), device=dev)

    def pf():
        gdn.gdn_prefill_seq(S, q, k, v, a, bt, o, batch=PB, seq_len=T, nk=NK, nv=NV, d=D, stream=sp)

    s = time_fn(torch, stream, pf, 3, warm=1)
    # the same recurrence in chunks of 64 tokens on the tensor cores (gdn_prefill_chunked)
    s_tc = time_fn(torch, stream, lambda: gdn.gdn_prefill_chunked(S, q, k, v, a, bt, o, batch=PB, seq_len=T, nk=NK,
                                                                  nv=NV, d=D, stream=sp), 3, warm=1)
    # the same call on an fp16 state (widened once on load, carried in fp32, rounded once on store)
    S16 = torch.zeros((PB, NV, D, D), dtype=torch.float16, device=dev)
    s16 = time_fn(torch, stream, lambda: gdn.gdn_prefill_seq(S16, q, k, v, a, bt, o, batch=PB, seq_len=T, nk=NK,
                                                             nv=NV, d=D, stream=sp), 3, warm=1)
    s16_tc = time_fn(torch, stream, lambda: gdn.gdn_prefill_chunked(S16, q, k, v, a, bt, o, batch=PB, seq_len=T,
                                                                    nk=NK, nv=NV, d=D, stream=sp), 3, warm=1)
    # the gated norm over every token's raw o (gdn_gate_norm, bf16 out): o and z read, out written
    z = torch.randn((R, NV * D), device=dev, generator=g)
    gn = torch.ones(D, device=dev)
    out = torch.empty((R, NV * D), dtype=torch.int16, device=dev)
    s_norm = time_fn(torch, stream, lambda: gdn.gdn_gate_norm(o, z, gn, out, rows=R, nv=NV, d=D, stream=sp), 5)
    norm_bytes = R * NV * D * (4 + 4 + 2) + D * 4
    # the same into int8 groups of 32 with an fp32 scale each (gdn_gate_norm_q8, no fp32 copy)
    xq = torch.empty((R, NV * D), dtype=torch.int8, device=dev)
    xs = torch.empty((R, NV * D // 32), device=dev)
    s_q8 = time_fn(torch, stream, lambda: gdn.gdn_gate_norm_q8(o, z, gn, xq, xs, rows=R, nv=NV, d=D, stream=sp), 5)
    q8_bytes = R * NV * D * (4 + 4 + 1) + R * NV * D // 32 * 4 + D * 4
    del z, gn, out, xq, xs
    th = PB * NV * T
    io = (2 * R * NK * D + R * NV * D * 2 + 2 * R * NV) * 4 + 2 * PB * NV * D * D * 4
    fma = th * D * D * 3                # per token-head: S.k, the rank-1 write, S.q (D^2 FMA each)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clk = (pk.get("sm_max_mhz") or 2070.0) * 1e6
    fma_peak = sms * 128 * clk          # FP32 FMA lanes x max clock: FMA per second
    # chunked kernel: executed TF32 MMA work per 64-token chunk and head, three split passes each:
    # G 128x64x128, Y 128x128x128, Delta 128x64x64, P Delta 128x64x64, Z 128x128x64 (multiply-adds)
    tc_flop = 2 * 3 * (128 * 64 * 128 + 128 * 128 * 128 + 128 * 64 * 64 + 128 * 64 * 64 + 128 * 128 * 64) \
        * PB * NV * ((T + 63) // 64)
    tf32_peak, tf32_basis = tf32_peak_flops(pk)
    del q, k, v, a, bt, o, S, S16
    torch.cuda.empty_cache()
    return {"prefill": {"config": f"B=8 T={T} NK=16 NV=48 D=128 fp32, state on chip",
                        "fp16_state": {"ms": s16 * 1e3, "token_heads_per_s": th / s16,
                                       "chunked_tensor_core_ms": s16_tc * 1e3},
                        "gate_norm_of_outputs": {"us": s_norm * 1e6, "achieved_gbs": norm_bytes / s_norm / 1e9,
                                                 "frac_of_hbm_peak": norm_bytes / s_norm / 1e9 / pk["hbm_gbs"],
                                                 "algorithmic_bytes": norm_bytes},
                        "gate_norm_q8_of_outputs": {"us": s_q8 * 1e6, "achieved_gbs": q8_bytes / s_q8 / 1e9,
                                                    "frac_of_hbm_peak": q8_bytes / s_q8 / 1e9 / pk["hbm_gbs"],
                                                    "algorithmic_bytes": q8_bytes},
                        "chunked_tensor_core": {
                            "ms": s_tc * 1e3, "token_heads_per_s": th / s_tc, "speedup_vs_token_loop": s / s_tc,
                            "roofline": {"bound": "tensor", "achieved": tc_flop / s_tc / 1e12,
                                         "peak": tf32_peak / 1e12, "unit": "TFLOP/s (TF32 MMA, executed)",
                                         "frac": tc_flop / s_tc / tf32_peak, "peak_basis": tf32_basis},
                            # the token-sequential work (4 D^2 FP32 instructions per token-head) over this
                            # kernel's time, against the FP32 issue peak: the rate the token loop would need
                            "token_loop_equivalent_frac_4d2": 4 / 3 * fma / s_tc / fma_peak},
                        "ms": s * 1e3, "token_heads_per_s": th / s,
                        "roofline": {"bound": "alu", "achieved": fma / s / 1e12, "peak": fma_peak / 1e12,
                                     "unit": "T FP32 FMA/s", "frac": fma / s / fma_peak,
                                     "frac_4d2_count": 4 / 3 * fma / s / fma_peak,
                                     "peak_basis": f"{sms} SMs x 128 FP32 lanes x {clk / 1e6:.0f} MHz",
                                     "count_basis": "frac: 3 D^2 FMA per token-head (S.k, the rank-1 write, S.q); "
                                                    "frac_4d2_count: 4 D^2 FP32 instructions per token-head "
                                                    "(the decay multiply counted apart)"},
                        "achieved_gbs": io / s / 1e9}}


# ------------------------------------------------------------------ oracle (CPU) timing

_ORACLE_INPUTS = {}


def _oracle_inputs(layer):
    """Seeded inputs of one layer for the oracle (drawn once, reused by later samples)."""
    import gdn_synth as gs
    if "S0" not in _ORACLE_INPUTS:
        _ORACLE_INPUTS["S0"] = gs.state_heads(SEED, range(B), range(NV), D).astype(np.float64)
    if layer not in _ORACLE_INPUTS:
        _ORACLE_INPUTS[layer] = (gs.decode_inputs(SEED, B, NK, NV, D, layer=layer),
                                 gs.norm_weight(SEED, D, layer=layer))
    return _ORACLE_INPUTS["S0"], _ORACLE_INPUTS[layer]


def cpu_baseline(sample_layers=None, budget_s=8.0):
    """Time the fp64 oracle, as it stands, on this host's cores over whole layers of the
    workload (32 sequences x 48 heads per layer, decode + gated norm): a fixed number of
    layers, or until ~budget_s of oracle time.  Only the oracle calls are timed."""
    import oracle
    threads = os.cpu_count() or 1
    step = max(1, B // threads)
    chunks = [(b0, min(B, b0 + step)) for b0 in range(0, B, step)]
    done_heads, spent, layers = 0, 0.0, 0
    limit = sample_layers or LAYERS
    while layers < limit and (sample_layers or spent < budget_s):
        S0, (x, gn) = _oracle_inputs(layers)
        S = S0.copy()

        def unit(c):
            b0, b1 = c
            # S[b0:b1] is a contiguous view: each thread updates its own sequences in place
            o = oracle.decode(S[b0:b1], x["q"][b0:b1], x["k"][b0:b1], x["v"][b0:b1],
                              x["alpha"][b0:b1], x["beta"][b0:b1], NK)
            return oracle.gated_rmsnorm(o.reshape(-1, D), x["z"][b0:b1].reshape(-1, D), gn, EPS)

        t0 = time.perf_counter()
        oracle.parallel_map(unit, chunks, threads=threads)
        spent += time.perf_counter() - t0
        done_heads += B * NV
        layers += 1
    # the same oracle on one thread, over one layer
    S0, (x, gn) = _oracle_inputs(0)
    S1 = S0.copy()
    t0 = time.perf_counter()
    o = oracle.decode(S1, x["q"], x["k"], x["v"], x["alpha"], x["beta"], NK)
    oracle.gated_rmsnorm(o.reshape(-1, D), x["z"].reshape(-1, D), gn, EPS)
    one = time.perf_counter() - t0
    return {"value": done_heads / spent, "unit": UNIT, "cores": len(chunks), "kind": "oracle",
            "seconds": spent,
            "sample": f"{layers} of 48 layers x 32 sequences x 48 heads ({done_heads} token-heads), "
                      f"decode + gated norm, fp64 C oracle on {len(chunks)} host threads",
            "single_thread": {"value": B * NV / one, "unit": UNIT, "cores": 1,
                              "sample": "1 layer x 32 sequences x 48 heads on 1 host thread"}}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is REF_LAYERS_PER_STEP whole layers of the workload."""
    if rank != 0:
        return None
    per = []
    for _ in range(args.warmup):
        cpu_baseline(sample_layers=REF_LAYERS_PER_STEP)
    t0 = time.perf_counter()
    total = 0.0
    for _ in range(args.steps):
        r = cpu_baseline(sample_layers=REF_LAYERS_PER_STEP)
        per.append(r)
        total += r["seconds"]
    wall = time.perf_counter() - t0
    heads = args.steps * B * NV * REF_LAYERS_PER_STEP
    value = heads / total
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "batched decode + fused gated RMSNorm, all 48 GDN layers of one token",
                   "batch_per_gpu": B, "nk": NK, "nv": NV, "d": D, "layers": LAYERS,
                   "step_sample": f"{REF_LAYERS_PER_STEP} of the 48 layers (32 sequences x 48 heads each) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": per[0]["cores"] if per else None,
                         "kind": "oracle",
                         "sample": f"{REF_LAYERS_PER_STEP} whole layers per step, decode + gated norm, fp64 C oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus == 1 else 1)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
