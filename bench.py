"""Benchmark of the MX quantized-training hot path on GB300.

One step = one pass of the whole path over the linear layers of one
Llama-3.1-8B decoder block at 8192 tokens (QKV 4096->6144, O 4096->4096,
gate+up 4096->28672, down 14336->4096).  Per layer:

  X  [T, in]   -> dual quantizer: row-wise E4M3 (forward A) + column-wise
                  Hadamard E2M1 (Wgrad B)
  W  [out, in] -> dual quantizer: row-wise E4M3 (forward B) + column-wise
                  E4M3 (dgrad B, i.e. W^T)
  dY [T, out]  -> dual quantizer: row-wise E4M3 (dgrad A) + column-wise
                  Hadamard E2M1 (Wgrad A)
  forward  Y  = X W^T          MXFP8 GEMM, bf16 out
  dgrad    dX = dY W           MXFP8 GEMM, bf16 out
  Wgrad    dW = (H dY)^T (H X) MXFP4 GEMM, fp32 out

The Wgrad GEMMs of the four layers need nothing from one another, so the
step issues them last, as one grouped launch (deferred weight gradients, as
a backward pass may); forward and dgrad run per layer.

Headline value: GEMM TFLOP/s of the whole step (quantizers included in the
time).  The JSON line also carries the quantizer GB/s and the MXFP8 / MXFP4
GEMM TFLOP/s, each against the measured GB300 peaks.

Multi-GPU: the path has no exchange step, so N ranks run N independent
replicas (weak scaling); rank 0 prints the aggregate.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MX quant GB/s & block-scaled MXFP8/MXFP4 GEMM TFLOPS, % of GB300 roofline"
WORKLOAD = ("llama3.1-8b decoder-block linears, T=8192: dual MX quantizers + "
            "fwd/dgrad MXFP8 (E4M3) + wgrad Hadamard-MXFP4 (E2M1) GEMMs")
L2_BYTES = 129 * 2 ** 20


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16": float(p["bf16_tflops"]),
                "bf16_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# Work description (shared by the GPU arm and the CPU oracle arm)
# ---------------------------------------------------------------------------

def layer_plan(tokens):
    from precision_mx_quantize_gb300 import synth
    out = []
    for i, (name, fin, fout) in enumerate(synth.LLAMA8B_LINEARS):
        out.append(dict(name=name, fin=fin, fout=fout, T=tokens, index=i))
    return out


def quant_bytes(rows, cols, fr, fc):
    """Algorithmic bytes of one dual quantizer pass: bf16 in + both code/scale outputs."""
    n = rows * cols
    b = 2 * n
    for f in (fr, fc):
        b += n if f == "e4m3" else n // 2
        b += n // 32
    return b


def step_work(plan):
    q, f8, f4 = 0, 0, 0
    for L in plan:
        T, fin, fout = L["T"], L["fin"], L["fout"]
        q += quant_bytes(T, fin, "e4m3", "e2m1")
        q += quant_bytes(fout, fin, "e4m3", "e4m3")
        q += quant_bytes(T, fout, "e4m3", "e2m1")
        f8 += 2 * (2 * T * fout * fin)
        f4 += 2 * T * fout * fin
    return q, f8, f4


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _smi_id(device):
    """nvidia-smi -i selector (PCI bus id) of a torch CUDA device."""
    import torch
    p = torch.cuda.get_device_properties(device)
    try:
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except AttributeError:
        return str(device.index or 0)


def build_device_state(plan, device):
    """Device inputs, preallocated outputs and workspaces for every layer."""
    import torch

    from precision_mx_quantize_gb300 import mxq, synth
    layers = []
    for L in plan:
        T, fin, fout, i = L["T"], L["fin"], L["fout"], L["index"]
        d = synth.decoder_block_layer(fin, fout, T, i)
        st = {"L": L, "host": d}
        st["x"] = d["x"].to(device)
        st["w"] = d["w"].to(device)
        st["dy"] = d["dy"].to(device)

        def codes(rows, cols, axis, fmt):
            cs, _ = mxq.code_shape(rows, cols, axis, fmt)
            lines, blocked = (rows, cols) if axis == "row" else (cols, rows)
            return (torch.empty(cs, dtype=torch.uint8, device=device),
                    torch.empty(mxq.mxq_scales_tc_bytes(lines, blocked), dtype=torch.uint8,
                                device=device))

        st["xq"] = (*codes(T, fin, "row", "e4m3"), *codes(T, fin, "col", "e2m1"))
        st["wq"] = (*codes(fout, fin, "row", "e4m3"), *codes(fout, fin, "col", "e4m3"))
        st["dyq"] = (*codes(T, fout, "row", "e4m3"), *codes(T, fout, "col", "e2m1"))
        st["y"] = torch.empty((T, fout), dtype=torch.bfloat16, device=device)
        st["dx"] = torch.empty((T, fin), dtype=torch.bfloat16, device=device)
        st["dw"] = torch.empty((fout, fin), dtype=torch.float32, device=device)
        layers.append(st)
    return layers


# The quantizers write their scales in the tensor cores' chunk layout and
# the GEMMs read them in place, so each layer launches 3 dual quantizers and
# its forward and dgrad GEMMs (no scale re-layout pass, no GEMM workspace);
# the Wgrad GEMMs of all layers depend on no other layer's result and run as
# one grouped launch at the end of the pass (deferred weight gradients).
SCALES = "tc"
LAUNCHES_PER_LAYER = 3 + 2


def launches_per_step(n_layers):
    return LAUNCHES_PER_LAYER * n_layers + 1


def run_layer(st, mark=None):
    """Enqueue one layer's dual quantizers and its forward and dgrad GEMMs on
    the current stream (its Wgrad GEMM runs in run_wgrad)."""
    import torch

    from precision_mx_quantize_gb300 import mxq
    T, fin, fout = st["L"]["T"], st["L"]["fin"], st["L"]["fout"]
    if mark:
        mark("q")
    mxq.mx_quantize_dual(st["x"], "e4m3", False, "e2m1", True, out=st["xq"], scale_layout=SCALES)
    mxq.mx_quantize_dual(st["w"], "e4m3", False, "e4m3", False, out=st["wq"], scale_layout=SCALES)
    mxq.mx_quantize_dual(st["dy"], "e4m3", False, "e2m1", True, out=st["dyq"], scale_layout=SCALES)
    if mark:
        mark("f8")
    xr, sxr, xc, sxc = st["xq"]
    wr, swr, wc, swc = st["wq"]
    dr, sdr, dc, sdc = st["dyq"]
    mxq.mx_gemm(xr, sxr, wr, swr, "e4m3", T, fout, fin, torch.bfloat16, out=st["y"],
                scale_layout=SCALES)
    mxq.mx_gemm(dr, sdr, wc, swc, "e4m3", T, fin, fout, torch.bfloat16, out=st["dx"],
                scale_layout=SCALES)


def run_wgrad(layers):
    """Enqueue the Wgrad GEMMs of all layers, dW = (H dY)^T (H X) in MXFP4
    with fp32 out, as one grouped launch."""
    import torch

    from precision_mx_quantize_gb300 import mxq
    probs = []
    for st in layers:
        T, fin, fout = st["L"]["T"], st["L"]["fin"], st["L"]["fout"]
        _, _, xc, sxc = st["xq"]
        _, _, dc, sdc = st["dyq"]
        probs.append((dc, sdc, xc, sxc, fout, fin, T, st["dw"]))
    mxq.mx_gemm_grouped(probs, "e2m1", torch.float32)


def run_step(layers, events=None):
    """Enqueue one pass of the hot path on the current stream."""
    import torch

    def mark(tag):
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        events.append((tag, e))

    for st in layers:
        run_layer(st, mark if events is not None else None)
    if events is not None:
        mark("f4")
    run_wgrad(layers)
    if events is not None:
        mark("end")


def interval_sums(events):
    """Milliseconds spent in each tagged interval of one recorded step."""
    sums = {}
    for (tag, e0), (_, e1) in zip(events[:-1], events[1:]):
        sums[tag] = sums.get(tag, 0.0) + e0.elapsed_time(e1)
    return sums


def reduce_max_ms(ms_local, device=None):
    """Slowest rank's timed-region milliseconds (identity without a process group)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    if dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(world, flops_per_step, steps, ms_max):
    """Whole-job throughput: every replica's GEMM flops over the slowest rank's time."""
    return world * flops_per_step * steps / (ms_max * 1e-3) / 1e12


def gpu_arm(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from precision_mx_quantize_gb300 import mxq

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    mxq.lib()
    plan = layer_plan(args.tokens)
    layers = build_device_state(plan, device)
    qbytes, f8, f4 = step_work(plan)
    flops = f8 + f4

    for _ in range(args.warmup):
        run_step(layers)
    mxq.check()
    torch.cuda.synchronize()

    # ---- timed region: K steps back to back, events only around them (an
    # event between two kernels keeps the second from starting early, so
    # the per-phase split is measured in a separate pass below)
    sampler = ClockSampler(_smi_id(device))
    if dist.is_initialized():
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        run_step(layers)
    t1.record()
    torch.cuda.synchronize()
    if dist.is_initialized():
        dist.barrier()
    status = mxq.mxq_check(mxq._stream())
    if status != 0:
        raise mxq.MXQError(status, "timed region")
    ms_total = t0.elapsed_time(t1)

    # ---- per-phase split (quantizers / MXFP8 / MXFP4 GEMMs): a second timed
    # pass of the same K steps with events at every phase boundary (the
    # clock samples cover both passes)
    per_step_events = []
    for _ in range(args.steps):
        ev = []
        run_step(layers, ev)
        per_step_events.append(ev)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    sums = {"q": 0.0, "f8": 0.0, "f4": 0.0}
    for ev in per_step_events:
        for k, v in interval_sums(ev).items():
            sums[k] += v

    # ---- end to end through the public API with host buffers
    e2e = e2e_measure(args, layers, flops, device)

    # ---- the other configurations, each timed on its own (after the timed
    # region, so they do not touch the headline number)
    configs = None
    if not args.no_configs and world == 1:
        del layers
        torch.cuda.empty_cache()
        configs = config_cases(_peaks())

    ms_max = reduce_max_ms(ms_total, device)
    if rank != 0:
        return None

    peaks = _peaks()
    ms_step = ms_max / args.steps
    value = aggregate_tflops(world, flops, args.steps, ms_max)
    q_gbs = qbytes * args.steps / (sums["q"] * 1e-3) / 1e9
    f8_tf = f8 * args.steps / (sums["f8"] * 1e-3) / 1e12
    f4_tf = f4 * args.steps / (sums["f4"] * 1e-3) / 1e12
    basis, bf16_peak = peak_basis(clocks, peaks)
    fp8_peak = 2.0 * bf16_peak   # nominal fp8:bf16 = 4.5 : 2.25
    fp4_peak = 6.0 * bf16_peak   # nominal fp4:bf16 = 13.5 : 2.25
    traffic = _profile_traffic()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3/e2m1 codes, e8m0 scales, fp32 accumulate",
        "data": "synthetic (seeded Student-t / normal / lognormal-scaled; no dataset or weights)",
        "config": run_config(plan, args.tokens, world),
        "breakdown": {
            "quantizers": {"GB/s": round(q_gbs, 1), "frac_of_hbm": round(q_gbs / peaks["hbm_gbs"], 3),
                            "ms_per_step": round(sums["q"] / args.steps, 4),
                            "bytes_per_step": qbytes},
            "mxfp8_gemm": {"TFLOP/s": round(f8_tf, 1), "frac_of_peak": round(f8_tf / fp8_peak, 3),
                           "ms_per_step": round(sums["f8"] / args.steps, 4), "flop_per_step": f8},
            "mxfp4_gemm": {"TFLOP/s": round(f4_tf, 1), "frac_of_peak": round(f4_tf / fp4_peak, 3),
                           "ms_per_step": round(sums["f4"] / args.steps, 4), "flop_per_step": f4},
            "peaks": {"hbm_GB/s": peaks["hbm_gbs"], "mxfp8_TFLOP/s": fp8_peak,
                      "mxfp4_TFLOP/s": fp4_peak,
                      "basis": f"{peaks['source']} (MEASURED_PEAKS.json): HBM copy; bf16 {basis} "
                               f"x nominal ratio (2x MXFP8, 6x MXFP4)"},
        },
        "roofline": {
            "kernel": "mx_gemm_kernel (MXFP8 E4M3, forward + dgrad launches)",
            "bound": "tensor",
            "achieved": round(f8_tf, 1),
            "peak": fp8_peak,
            "unit": "TFLOP/s",
            "frac": round(f8_tf / fp8_peak, 3),
            "peak_basis": basis,
            "traffic": traffic,
            "mxfp4": {"kernel": "mx_gemm_kernel (MXFP4 E2M1, Wgrad launches)", "bound": "tensor",
                      "achieved": round(f4_tf, 1), "peak": fp4_peak, "unit": "TFLOP/s",
                      "frac": round(f4_tf / fp4_peak, 3)},
            "quantizers": {"kernel": "mx_quant_kernel (dual passes)", "bound": "hbm",
                           "achieved": round(q_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": round(q_gbs / peaks["hbm_gbs"], 3)},
            "timing": "CUDA events at the phase boundaries of a second pass of the K timed "
                      "steps; the headline pass has events only around the K steps",
        },
        "e2e": e2e,
        "configs": configs,
        "gpu_launches": launches_per_step(len(plan)) * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.cpu_budget_s)
    return line


def peak_basis(clocks, peaks):
    """Which measured bf16 GEMM peak the tensor fractions are taken against.

    The burst figure (a GEMM timed alone, at full clock) applies when the
    run's own clock samples show the SM clock at its maximum and no power
    cap; otherwise the sustained figure (a seconds-long GEMM loop under the
    power cap) does.  Returns (name, bf16 TFLOP/s).
    """
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    capped = "sw_power_cap" in clocks.get("reasons", [])
    if sm and smax and not capped and sm >= 0.97 * smax:
        return "burst", peaks["bf16"]
    return "sustained", peaks["bf16_sustained"]


def _profile_traffic():
    """DRAM bytes per MXFP8 GEMM launch of this step, from the committed ncu summary.

    The summary records the sha256 of the GEMM source it was captured from;
    once the source changes the number no longer describes this kernel and
    None is returned.
    """
    import hashlib
    prof = os.path.join(ROOT, "profiles", "mx_gemm_kernel_dram_llama8b_block.md")
    src = os.path.join(ROOT, "precision_mx_quantize_gb300", "csrc", "gemm.cu")
    try:
        fields = {}
        with open(prof) as f:
            for line in f:
                if ":" in line and line.strip().startswith("- "):
                    k, _, v = line.strip()[2:].partition(":")
                    fields[k.strip().strip("`")] = v.strip().strip("`")
        with open(src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
        if fields.get("gemm_source_sha256") != digest:
            return None
        return int(fields["mxfp8_dram_bytes_per_launch"])
    except Exception:
        return None


def e2e_measure(args, layers, flops, device):
    """The same step through the public API with host buffers.

    Every step copies all of its bf16 inputs (X, W, dY of every layer) from
    pinned host memory to the device and copies the step's gradients (dW of
    every layer, fp32) back, inside the timed region.  Copies run on their own
    streams so that layer i+1's inputs and layer i-1's gradients move while
    layer i computes; events order every buffer reuse.
    """
    import torch
    host_in, host_out = [], []
    h2d = d2h = 0
    for st in layers:
        hi = {k: st["host"][k].pin_memory() for k in ("x", "w", "dy")}
        host_in.append(hi)
        h2d += sum(t.numel() * t.element_size() for t in hi.values())
        ho = torch.empty(st["dw"].shape, dtype=st["dw"].dtype, pin_memory=True)
        host_out.append(ho)
        d2h += ho.numel() * ho.element_size()
    compute = torch.cuda.current_stream(device)
    up = torch.cuda.Stream(device)
    down = torch.cuda.Stream(device)
    n = len(layers)
    # inputs of layer i may be overwritten once the previous step's layer i
    # quantized them; the dW buffers once the previous step's copies left
    done_compute = [torch.cuda.Event() for _ in range(n)]
    done_down = torch.cuda.Event()
    wgrad_done = torch.cuda.Event()
    for i in range(n):
        done_compute[i].record(compute)
    done_down.record(compute)

    def one():
        arrived = []
        for i, (st, hi) in enumerate(zip(layers, host_in)):
            with torch.cuda.stream(up):
                up.wait_event(done_compute[i])
                st["x"].copy_(hi["x"], non_blocking=True)
                st["w"].copy_(hi["w"], non_blocking=True)
                st["dy"].copy_(hi["dy"], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(up)
                arrived.append(ev)
        for i, st in enumerate(layers):
            compute.wait_event(arrived[i])
            run_layer(st)
            done_compute[i].record(compute)
        compute.wait_event(done_down)
        run_wgrad(layers)
        wgrad_done.record(compute)
        with torch.cuda.stream(down):
            down.wait_event(wgrad_done)
            for st, ho in zip(layers, host_out):
                ho.copy_(st["dw"], non_blocking=True)
            done_down.record(down)

    steps = max(1, min(args.steps, 10))
    one()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(compute)
    for _ in range(steps):
        one()
    compute.wait_event(done_down)
    t1.record(compute)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    h2d_gbs, d2h_gbs = _link_probe(host_in[0]["x"], layers[0]["x"], host_out[0], layers[0]["dw"])
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "H2D, compute and D2H on separate streams, ordered by events (inputs per "
                       "layer, gradients after the step's grouped Wgrad launch)",
            "link": {"h2d_GB/s": h2d_gbs, "d2h_GB/s": d2h_gbs,
                     "h2d_bound_ms": round(h2d / (h2d_gbs * 1e6), 3),
                     "note": "one pinned copy each way, measured on this box after the e2e steps"}}


def _link_probe(h_in, d_in, h_out, d_out, reps=5):
    """GB/s of plain pinned host->device and device->host copies on this machine."""
    import torch
    res = []
    for dst, src in ((d_in, h_in), (h_out, d_out)):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        res.append(round(reps * src.numel() * src.element_size() / (e0.elapsed_time(e1) * 1e6), 1))
    return res[0], res[1]


# ---------------------------------------------------------------------------
# CPU oracle arm (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------

def _oracle_sample_step(plan, t_s, out_s, seed=0):
    """The step's operations on a token x feature slice of every layer, in the oracle.

    Returns the GEMM flops of the sample.
    """
    import numpy as np

    from oracle import mx_oracle as O
    from precision_mx_quantize_gb300 import synth
    flops = 0
    for L in plan:
        fin = L["fin"]
        fout = min(out_s, L["fout"])
        x = synth.activation(t_s, fin, 3 * L["index"]).float().numpy()
        w = synth.weight(fout, fin, 3 * L["index"] + 1).float().numpy()
        dy = synth.out_grad(t_s, fout, 3 * L["index"] + 2).float().numpy()
        xr = O.mx_quantize(x, "row", "e4m3")
        xc = O.hadamard_mx_quantize(x, "col", "e2m1")
        wr = O.mx_quantize(w, "row", "e4m3")
        wc = O.mx_quantize(w, "col", "e4m3")
        dr = O.mx_quantize(dy, "row", "e4m3")
        dc = O.hadamard_mx_quantize(dy, "col", "e2m1")
        O.mx_gemm_f64(*xr, *wr, "e4m3")
        O.mx_gemm_f64(*dr, *wc, "e4m3")
        O.mx_gemm_f64(*dc, *xc, "e2m1")
        flops += 3 * 2 * t_s * fout * fin
        del x, w, dy, xr, xc, wr, wc, dr, dc
        _ = np
    return flops


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


def _oracle_dual_band(args):
    """Dual quantization of one row band in the oracle (a worker of the all-core leg)."""
    x, fr, hr, fc, hc = args
    from oracle import mx_oracle as O
    O.quantize_any(x, "row", fr, hr)
    O.quantize_any(x, "col", fc, hc)
    return x.shape[0]


def _oracle_quantizer_rates(rows_single=1024):
    """The oracle's dual Hadamard-E2M1 quantizer (the 8192x4096 activation
    workload) in GB/s of algorithmic bytes: on one process over a band of
    `rows_single` rows, and on every core (a spawn pool, one row band per
    process) over the whole tensor."""
    import multiprocessing

    from oracle import mx_oracle as O
    from precision_mx_quantize_gb300 import synth
    x = synth.hadamard_dual_activation()["x"].float().numpy()
    R, C = x.shape
    band = x[:rows_single]
    t0 = time.perf_counter()
    O.quantize_any(band, "row", "e2m1", True)
    O.quantize_any(band, "col", "e2m1", True)
    dt1 = time.perf_counter() - t0
    gbs1 = quant_bytes(rows_single, C, "e2m1", "e2m1") / dt1 / 1e9
    cores = os.cpu_count() or 1
    step = max(32, (R // cores) // 32 * 32)
    bands = [(x[r:r + step], "e2m1", True, "e2m1", True) for r in range(0, R, step)]
    with multiprocessing.get_context("spawn").Pool(cores) as pool:
        pool.map(_oracle_dual_band, [(x[:32], "e2m1", True, "e2m1", True)] * cores)  # warm
        t0 = time.perf_counter()
        pool.map(_oracle_dual_band, bands)
        dtn = time.perf_counter() - t0
    gbsn = quant_bytes(R, C, "e2m1", "e2m1") / dtn / 1e9
    return {"workload": f"dual Hadamard + E2M1 (rows and columns), {R}x{C} activation",
            "GB/s_one_process": round(gbs1, 4), "sample_one_process": f"{rows_single}x{C} rows band, {dt1:.2f} s",
            "GB/s_all_cores": round(gbsn, 4), "processes": cores,
            "sample_all_cores": f"the whole {R}x{C} tensor in {len(bands)} row bands, {dtn:.2f} s"}


def _oracle_gemm_rates(M=8192, N=14336, K=4096, rows=512, sample=256, fmt="e4m3"):
    """The oracle's fp64 GEMM on an M x N x K shape (default: the MLP
    up-projection, MXFP8): the sampled-element check as MAC/s, and a full
    product over a `rows`-row slice, extrapolated linearly to all M rows."""
    import numpy as np

    from oracle import mx_oracle as O
    rng = np.random.default_rng(0)
    kb = K if fmt == "e4m3" else K // 2
    hi = 0x7E if fmt == "e4m3" else 256
    A = rng.integers(0, hi, size=(rows, kb), dtype=np.uint8)
    sA = rng.integers(120, 134, size=(rows, K // 32), dtype=np.uint8)
    B = rng.integers(0, hi, size=(N, kb), dtype=np.uint8)
    sB = rng.integers(120, 134, size=(N, K // 32), dtype=np.uint8)
    ri = rng.integers(0, rows, sample)
    ci = rng.integers(0, N, sample)
    t0 = time.perf_counter()
    O.mx_gemm_f64_rows(A, sA, B, sB, fmt, ri, ci)
    dts = time.perf_counter() - t0
    t0 = time.perf_counter()
    O.mx_gemm_f64(A, sA, B, sB, fmt)
    dtf = time.perf_counter() - t0
    macs = rows * N * K
    return {"workload": f"{'MXFP8' if fmt == 'e4m3' else 'MXFP4'} GEMM {M}x{N}x{K} "
                        "(fp64 over dequantized operands, C and sum|ab|)",
            "sampled_check_MAC/s": round(sample * sample * K / dts, 1),
            "sampled_check": f"{sample} rows x {sample} columns, {dts:.2f} s",
            "slice_MAC/s": round(macs / dtf, 1),
            "slice": f"{rows} rows x {N} x {K}, {dtf:.2f} s",
            "full_ms_extrapolated": round(dtf * (M / rows) * 1e3, 1),
            "extrapolated": True}


def _oracle_round_trip_us(reps=5):
    """The oracle's 256x1024 E4M3 quantize and dequantize, microseconds per call."""
    from oracle import mx_oracle as O
    from precision_mx_quantize_gb300 import synth
    x = synth.quantize_dequantize_small()["x"].float().numpy()
    t0 = time.perf_counter()
    for _ in range(reps):
        c, s = O.mx_quantize(x, "row", "e4m3")
    tq = (time.perf_counter() - t0) / reps
    t0 = time.perf_counter()
    for _ in range(reps):
        O.mx_dequantize(c, s, "e4m3")
    td = (time.perf_counter() - t0) / reps
    return {"quantize_us": round(tq * 1e6, 1), "dequantize_us": round(td * 1e6, 1),
            "sample": f"the whole 256x1024 tensor, mean of {reps} calls, one process"}


def _oracle_dequant_rate(fmt, axis, out, rows=512, cols=4096):
    """The oracle's dequantizer GB/s (algorithmic bytes) on a rows x cols sample."""
    from oracle import mx_oracle as O
    from precision_mx_quantize_gb300 import synth
    x = synth.normal((rows, cols), 0).float().numpy()
    c, s = O.mx_quantize(x, axis, fmt)
    t0 = time.perf_counter()
    O.mx_dequantize(c, s, fmt, out)
    dt = time.perf_counter() - t0
    n = rows * cols
    b = n * ((1 if fmt == "e4m3" else 0.5) + 1 / 32 + (4 if out == "f32" else 2))
    return {"GB/s": round(b / dt / 1e9, 5), "sample": f"{rows}x{cols}, one process, {dt:.3f} s"}


def _oracle_sweep_rate(fmt, layout, had, rows=256, cols=4096):
    """The oracle's GB/s (algorithmic bytes) for one quantizer-sweep variant on
    a rows x cols N(0,1) sample, one process."""
    from oracle import mx_oracle as O
    from precision_mx_quantize_gb300 import synth
    x = synth.normal((rows, cols), 0).float().numpy()
    t0 = time.perf_counter()
    if layout in ("row", "dual"):
        O.quantize_any(x, "row", fmt, had)
    if layout in ("col", "dual"):
        O.quantize_any(x, "col", fmt, had)
    dt = time.perf_counter() - t0
    n = rows * cols
    one = (n if fmt == "e4m3" else n // 2) + n // 32
    b = 2 * n + (2 * one if layout == "dual" else one)
    return {"GB/s": round(b / dt / 1e9, 5), "sample": f"{rows}x{cols}, one process, {dt:.2f} s"}


def cpu_baseline(budget_s=15.0):
    t_s, out_s = 512, 2048
    plan = layer_plan(8192)
    t0 = time.perf_counter()
    flops = _oracle_sample_step(plan, t_s, out_s)
    dt = time.perf_counter() - t0
    line = {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle", "cpu_model": cpu_model(),
            "sample": (f"every layer of the block pass on {t_s} tokens x {out_s} output features "
                       f"(full input width): 6 quantizations + 3 fp64 GEMMs per layer; "
                       f"{dt:.1f} s, numpy (BLAS threads = cores)")}
    line["quantizer"] = _oracle_quantizer_rates()
    line["gemm"] = _oracle_gemm_rates()
    return line


def run_config(plan, tokens, world):
    """The `config` object of both arms' JSON lines (the same workload)."""
    qbytes = step_work(plan)[0]
    return {
        "workload": WORKLOAD,
        "tokens": tokens,
        "layers": [f"{L['name']} {L['fin']}->{L['fout']}" for L in plan],
        "l2": "inputs larger than L2: each step streams ~%.1f GB of distinct tensors" %
              (qbytes / 1e9),
        "parallelism": "replicas" if world > 1 else "single GPU",
    }


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    plan = layer_plan(args.tokens)
    t_s, out_s = 32, 128
    for _ in range(args.warmup):
        _oracle_sample_step(plan, t_s, out_s)
    times, flops = [], 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        flops = _oracle_sample_step(plan, t_s, out_s)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = flops * args.steps / total / 1e12
    sample = (f"each step: every layer of the block pass on {t_s} tokens x {out_s} output "
              f"features (full input width) in the CPU oracle")
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic", "config": run_config(plan, args.tokens, world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


CASES = {
    # name: (what, args) -- one small, self-contained launch sequence for ncu
    "gemm-e4m3": ("gemm", (8192, 8192, 4096, "e4m3", "f32")),
    "gemm-e2m1": ("gemm", (8192, 8192, 8192, "e2m1", "bf16")),
    "quant-dual-e4m3-he2m1": ("quant", (16384, 8192, "e4m3", False, "e2m1", True)),
    "quant-dual-he2m1-he2m1": ("quant", (16384, 8192, "e2m1", True, "e2m1", True)),
    # the epilogue writing E4M3 codes of the product, and the unfused pair it
    # replaces (bf16 product, then a row-wise E4M3 quantizer pass over it)
    "gemm-e4m3-q": ("gemmq", (8192, 8192, 4096, "e4m3", "e4m3")),
    "gemm-e4m3-bf16": ("gemm", (8192, 8192, 4096, "e4m3", "bf16")),
    "quant-row-e4m3": ("quant1", (8192, 8192, "row", "e4m3")),
    # ablation: column-wise random-sign Hadamard E2M1 with stochastic rounding
    "ablate-col-rhe2m1-sr": ("ablate", (16384, 8192, "col", "e2m1", True, 0xA5A5F00F, True)),
    "ablate-row-e4m3-sr": ("ablate", (16384, 8192, "row", "e4m3", False, 0, True)),
    # dequantizer: 16384 x 8192 codes back to bf16, column-wise (transposing) and row-wise
    "dequant-col-e4m3-bf16": ("dequant", (16384, 8192, "col", "e4m3", "bf16")),
    "dequant-row-e4m3-bf16": ("dequant", (16384, 8192, "row", "e4m3", "bf16")),
}


def _case_bytes(what, args):
    """Algorithmic HBM bytes of one launch of a case (bf16 in, codes + scales out)."""
    if what == "quant":
        R, C, fr, _, fc, _ = args
        out = sum(R * C * (0.5 if f == "e2m1" else 1.0) + R * C / 32 for f in (fr, fc))
        return 2 * R * C + out
    if what == "ablate":
        R, C, _, f, _, _, _ = args
        return 2 * R * C + R * C * (0.5 if f == "e2m1" else 1.0) + R * C / 32
    if what == "quant1":
        R, C, _, f = args
        return 2 * R * C + R * C * (0.5 if f == "e2m1" else 1.0) + R * C / 32
    if what == "dequant":
        R, C, _, f, od = args
        return R * C * (0.5 if f == "e2m1" else 1.0) + R * C / 32 + R * C * (4 if od == "f32" else 2)
    M, N, K, fmt, od = args
    eb = 1.0 if fmt != "e2m1" else 0.5
    if what == "gemmq":
        out = M * N * ((0.5 if od == "e2m1" else 1.0) + 1 / 32)
    else:
        out = M * N * (4 if od == "f32" else 2)
    return (M + N) * K * (eb + 1 / 32) + out


ABLATION_VARIANTS = [
    # name, hadamard, random sign mask, stochastic rounding
    ("no rotation, RNE", False, False, False),
    ("fixed Hadamard, RNE (the method)", True, False, False),
    ("random-sign Hadamard, RNE", True, True, False),
    ("no rotation, stochastic rounding", False, False, True),
    ("fixed Hadamard, stochastic rounding", True, False, True),
]


def ablation_error(tokens=16384, n_out=4096, n_in=4096, draws=8):
    """Error structure of the MXFP4 Wgrad under the ablation variants.

    dW = dY^T X with dY [tokens, n_out] ~ N(0, 1e-3) x per-column
    LogNormal(0, 2) and X [tokens, n_in] ~ Student-t(3) x per-channel
    LogNormal(0, 1) (the Wgrad workload's distributions), both quantized
    column-wise to E2M1 along tokens and multiplied by the MXFP4 GEMM.
    Reference: the fp32 product of the bf16 inputs (no TF32).  For each
    variant: the relative Frobenius error of one draw, and of the mean of
    `draws` draws (new random signs / seeds per draw): a deterministic
    variant's error does not shrink with averaging, an unbiased one's does.
    A quality measurement, not a parity check.
    """
    import torch

    from precision_mx_quantize_gb300 import mxq, synth
    torch.backends.cuda.matmul.allow_tf32 = False
    dy = synth.out_grad(tokens, n_out, seed=1).cuda()
    x = synth.activation(tokens, n_in, seed=2).cuda()
    ref = dy.float().t() @ x.float()
    nref = ref.norm().item()
    rng = __import__("random").Random(7)
    out = {}
    for name, had, rand_sign, sr in ABLATION_VARIANTS:
        acc = torch.zeros_like(ref)
        first = None
        for d in range(draws):
            mask = rng.getrandbits(32) if rand_sign else 0
            seed = 1000 + d
            A, sA = mxq.mx_quantize_ablation(dy, "col", "e2m1", had, mask, sr, seed)
            B, sB = mxq.mx_quantize_ablation(x, "col", "e2m1", had, mask, sr, seed + 500)
            dw = mxq.mx_gemm(A, sA, B, sB, "e2m1", n_out, n_in, tokens)
            acc += dw
            if first is None:
                first = (dw - ref).norm().item() / nref
        mxq.check()
        out[name] = {"rel_err_one_draw": round(first, 6),
                     f"rel_err_mean_of_{draws}": round((acc / draws - ref).norm().item() / nref, 6)}
    return {"case": "ablate-error", "workload": f"Wgrad dY^T X, tokens={tokens}, out={n_out}, in={n_in}, "
            "E2M1 column-wise along tokens", "variants": out}


def _time_rotating(launches, reps=20, warm=5, graph=False):
    """Average ms per launch over `reps` launches cycling through `launches`
    (one closure per buffer set; the sets together exceed 2x L2, so each
    launch reads its inputs from HBM), CUDA events on the current stream.

    graph: capture the `reps` launches in a CUDA graph and time its replay,
    which takes the host's per-call work out of the measurement."""
    import torch
    for i in range(warm):
        launches[i % len(launches)]()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph:
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(reps):
                    launches[i % len(launches)]()
        torch.cuda.current_stream().wait_stream(s)
        g.replay()
        torch.cuda.synchronize()
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps
    e0.record()
    for i in range(reps):
        launches[i % len(launches)]()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def config_cases(peaks):
    """The four configurations besides the block pass, timed on the GPU.

    * cfg1 round trip: 256x1024 N(0,1) with 1% x100 outliers, row-wise E4M3
      quantize then dequantize to fp32 (latency-bound: microseconds per call,
      launched one by one from Python, and the kernel time in a CUDA graph);
    * cfg2: dual Hadamard E2M1 of the 8192x4096 activation (GB/s);
    * cfg3: MLP up-projection forward GEMM 8192x14336x4096 MXFP8, fp32 out;
    * cfg4: MLP Wgrad GEMM 14336x4096x16384 MXFP4 on Hadamard E2M1 operands,
      fp32 out, with its two quantizers (GB/s).
    Buffers rotate so that each launch reads from HBM.  A GEMM timed alone is
    set against the burst bf16 figure times the nominal ratio.
    """
    import torch

    from precision_mx_quantize_gb300 import mxq, synth
    hbm = peaks["hbm_gbs"]
    out = {}

    x = synth.quantize_dequantize_small()["x"].cuda()
    c, sc = mxq.mx_quantize(x, "row", "e4m3")
    y = torch.empty((256, 1024), dtype=torch.float32, device="cuda")
    q1 = lambda: mxq.mx_quantize(x, "row", "e4m3", out=(c, sc))
    d1 = lambda: mxq.mx_dequantize(c, sc, 256, 1024, "row", "e4m3", out=y)
    # the C-ABI entry points called directly (pointers taken once): the
    # library's own per-call host cost, without the binding's tensor checks
    L, st = mxq.lib(), mxq._stream(x.device)
    xp, cp, sp, yp = x.data_ptr(), c.data_ptr(), sc.data_ptr(), y.data_ptr()
    q1_abi = lambda: L.mxq_quantize(xp, 256, 1024, mxq.ROWWISE, mxq.FMTS["e4m3"], cp, sp, st)
    d1_abi = lambda: L.mxq_dequantize(cp, sp, 256, 1024, mxq.ROWWISE, mxq.FMTS["e4m3"], yp,
                                      mxq.OUT_F32, st)
    out["cfg1_round_trip_256x1024_e4m3"] = {
        "config": "round trip 256x1024 E4M3",
        "quantize_us": round(_time_rotating([q1], reps=200) * 1e3, 2),
        "dequantize_us": round(_time_rotating([d1], reps=200) * 1e3, 2),
        "quantize_us_abi": round(_time_rotating([q1_abi], reps=200) * 1e3, 2),
        "dequantize_us_abi": round(_time_rotating([d1_abi], reps=200) * 1e3, 2),
        "quantize_us_graph": round(_time_rotating([q1], reps=200, graph=True) * 1e3, 2),
        "dequantize_us_graph": round(_time_rotating([d1], reps=200, graph=True) * 1e3, 2),
        "timing": "us per call launched one by one from Python through the tensor binding; "
                  "_abi: the C entry points called directly through ctypes with the pointers "
                  "taken once; _graph: the binding's calls in a CUDA graph"}
    del x, c, sc, y

    x = synth.hadamard_dual_activation()["x"].cuda()
    xs = [x] + [x.clone() for _ in range(3)]
    outs = [mxq.mx_quantize_dual(xx, "e2m1", True, "e2m1", True) for xx in xs]
    ls = [lambda i=i: mxq.mx_quantize_dual(xs[i], "e2m1", True, "e2m1", True, out=outs[i])
          for i in range(4)]
    b = quant_bytes(8192, 4096, "e2m1", "e2m1")
    ms = _time_rotating(ls)
    msg = _time_rotating(ls, graph=True)
    out["cfg2_dual_hadamard_e2m1_8192x4096"] = {
        "config": "dual Hadamard E2M1 8192x4096", "ms": round(ms, 4),
        "GB/s": round(b / ms / 1e6, 1), "frac_of_hbm": round(b / ms / 1e6 / hbm, 3),
        "ms_graph": round(msg, 4), "GB/s_graph": round(b / msg / 1e6, 1),
        "frac_of_hbm_graph": round(b / msg / 1e6 / hbm, 3),
        "bytes": b}
    del x, xs, outs, ls

    d = synth.mlp_up_forward()
    x, w = d["x"].cuda(), d["w"].cuda()
    A, sA = mxq.mx_quantize(x, "row", "e4m3", scale_layout="tc")
    B, sB = mxq.mx_quantize(w, "col", "e4m3", scale_layout="tc")
    C = torch.empty((8192, 14336), dtype=torch.float32, device="cuda")
    ms = _time_rotating([lambda: mxq.mx_gemm(A, sA, B, sB, "e4m3", 8192, 14336, 4096, out=C,
                                              scale_layout="tc")])
    f = 2 * 8192 * 14336 * 4096
    out["cfg3_mlp_up_fwd_mxfp8_8192x14336x4096"] = {
        "config": "MLP up forward 8192x14336x4096 MXFP8, fp32 out", "ms": round(ms, 4),
        "TFLOP/s": round(f / ms / 1e9, 1),
        "frac_of_peak": round(f / ms / 1e9 / (2 * peaks["bf16"]), 3), "peak_basis": "burst"}
    del d, x, w, A, B, C

    d = synth.mlp_wgrad()
    dy, x = d["dy"].cuda(), d["x"].cuda()
    A, sA = mxq.hadamard_mx_quantize(dy, "col", "e2m1", scale_layout="tc")
    B, sB = mxq.hadamard_mx_quantize(x, "col", "e2m1", scale_layout="tc")
    ms_q = _time_rotating([lambda: mxq.hadamard_mx_quantize(dy, "col", "e2m1", out=(A, sA),
                                                            scale_layout="tc"),
                           lambda: mxq.hadamard_mx_quantize(x, "col", "e2m1", out=(B, sB),
                                                            scale_layout="tc")])
    C = torch.empty((14336, 4096), dtype=torch.float32, device="cuda")
    ms = _time_rotating([lambda: mxq.mx_gemm(A, sA, B, sB, "e2m1", 14336, 4096, 16384, out=C,
                                              scale_layout="tc")])
    f = 2 * 14336 * 4096 * 16384
    qb = (16384 * 14336 + 16384 * 4096) * (2 + 0.5 + 1 / 32)
    out["cfg4_mlp_wgrad_mxfp4_14336x4096x16384"] = {
        "config": "MLP Wgrad 14336x4096x16384 MXFP4 (Hadamard E2M1), fp32 out", "ms": round(ms, 4),
        "TFLOP/s": round(f / ms / 1e9, 1),
        "frac_of_peak": round(f / ms / 1e9 / (6 * peaks["bf16"]), 3), "peak_basis": "burst",
        "quantizers_GB/s": round(qb / (2 * ms_q) / 1e6, 1),
        "quantizers_frac_of_hbm": round(qb / (2 * ms_q) / 1e6 / hbm, 3)}
    del d, dy, x, A, B, C
    mxq.check()
    torch.cuda.empty_cache()
    out["f1_mxfp8_allgather_gate_up_28672x4096"] = allgather_case()
    return out


def allgather_case(out_f=28672, in_f=4096):
    """The MXFP8 low-precision all-gather of a weight's dim-0 shards (the
    gate+up weight, 28672x4096): each rank quantizes its rows and the codes
    and scales are all-gathered, against the bf16 all-gather it replaces.
    In a world of one rank the gather is a local copy, so the figure is the
    quantize-plus-copy cost; bytes count what each rank receives."""
    import socket

    import torch
    import torch.distributed as dist

    from precision_mx_quantize_gb300 import fsdp_gather, mxq, synth
    created = False
    if not dist.is_initialized():
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                                world_size=1)
        created = True
    try:
        world, rank = dist.get_world_size(), dist.get_rank()
        lo, hi = fsdp_gather.shard_bounds(out_f, world, rank)
        shard = synth.weight(out_f, in_f, 1)[lo:hi].contiguous().cuda()
        codes = torch.empty((out_f, in_f), dtype=torch.uint8, device="cuda")
        scales = torch.empty((out_f, in_f // 32), dtype=torch.uint8, device="cuda")
        full = torch.empty((out_f, in_f), dtype=torch.bfloat16, device="cuda")
        ms_mx = _time_rotating([lambda: fsdp_gather.gather_mx_weight(shard, out=(codes, scales))])
        ms_bf = _time_rotating([lambda: dist.all_gather_into_tensor(full, shard)])
        mxq.check()
        b_mx = fsdp_gather.gathered_bytes(out_f, in_f)
        b_bf = out_f * in_f * 2
        return {"config": f"MXFP8 all-gather of dim-0 shards, weight {out_f}x{in_f}, world {world}",
                "ms_mxfp8": round(ms_mx, 4), "ms_bf16": round(ms_bf, 4),
                "bytes_mxfp8": b_mx, "bytes_bf16": b_bf,
                "volume_ratio": round(b_mx / b_bf, 4),
                "GB/s_mxfp8": round(b_mx / ms_mx / 1e6, 1), "GB/s_bf16": round(b_bf / ms_bf / 1e6, 1),
                "note": "world 1: the gather is a local copy; ms_mxfp8 includes quantizing the shard"}
    finally:
        if created:
            dist.destroy_process_group()


def sweep():
    """The measurement configurations besides the block pass, one JSON line each.

    * round trip: 256x1024 N(0,1) with 1% x100 outliers, row-wise E4M3
      quantize then dequantize to fp32 (latency-bound: reported in us);
    * dual Hadamard E2M1: 8192x4096 activation, Hadamard + E2M1 along rows
      and columns in one pass (GB/s);
    * MLP up-projection forward GEMM 8192x14336x4096 MXFP8, fp32 out, and
      the MLP Wgrad GEMM 14336x4096x16384 MXFP4 (Hadamard E2M1 operands),
      fp32 out (TFLOP/s), with their quantizers;
    * quantizer bandwidth sweep: n = 2^20 .. 2^28 elements as [n/4096][4096]
      bf16 N(0,1), {E4M3, E2M1} x {row, col, dual} x {Hadamard off, on}.
    Buffers rotate so that each launch reads from HBM.
    """
    import torch

    from precision_mx_quantize_gb300 import mxq, synth
    peaks = _peaks()
    hbm = peaks["hbm_gbs"]
    lines = []

    def emit(d):
        print(json.dumps(d), flush=True)
        lines.append(d)

    host = {"cores": os.cpu_count(), "cpu_model": cpu_model(), "kind": "oracle"}
    orates = {"cfg1_round_trip_256x1024_e4m3": _oracle_round_trip_us(),
              "cfg2_dual_hadamard_e2m1_8192x4096": _oracle_quantizer_rates(),
              "cfg3_mlp_up_fwd_mxfp8_8192x14336x4096": _oracle_gemm_rates(),
              "cfg4_mlp_wgrad_mxfp4_14336x4096x16384": _oracle_gemm_rates(
                  M=14336, N=4096, K=16384, fmt="e2m1")}
    for k, d in config_cases(peaks).items():
        if k in orates:   # the all-gather case has no oracle leg (it moves bytes, computes nothing new)
            d["cpu_oracle"] = dict(host, **orates[k])
        emit(d)
    torch.cuda.empty_cache()

    # dequantizer bandwidth (16384 x 8192 codes -> fp32 / bf16)
    for fmt in ("e4m3", "e2m1"):
        for axis in ("row", "col"):
            x = torch.randn(16384, 8192, device="cuda").to(torch.bfloat16)
            c, sc = mxq.mx_quantize(x, axis, fmt)
            for od, ob in ((torch.float32, 4), (torch.bfloat16, 2)):
                out = torch.empty((16384, 8192), dtype=od, device="cuda")
                ms = _time_rotating([lambda: mxq.mx_dequantize(c, sc, 16384, 8192, axis, fmt, od, out=out)],
                                    graph=True)
                n = 16384 * 8192
                b = n * ((1 if fmt == "e4m3" else 0.5) + 1 / 32 + ob)
                emit({"config": "dequantize 16384x8192", "fmt": fmt, "layout": axis,
                      "out": str(od).replace("torch.", ""), "us": round(ms * 1e3, 2),
                      "GB/s": round(b / ms / 1e6, 1), "frac_of_hbm": round(b / ms / 1e6 / hbm, 3),
                      "cpu_oracle": dict(host, **_oracle_dequant_rate(
                          fmt, axis, "f32" if ob == 4 else "bf16"))})
            del x, c, sc, out
    torch.cuda.empty_cache()

    # quantizer bandwidth sweep
    def qbytes_of(n, layout, fmt):
        code = n if fmt == "e4m3" else n // 2
        one = code + n // 32
        return 2 * n + (2 * one if layout == "dual" else one)

    for fmt in ("e4m3", "e2m1"):
        for layout in ("row", "col", "dual"):
            for had in (False, True):
                oracle_rate = dict(host, **_oracle_sweep_rate(fmt, layout, had))
                for e in range(20, 29):
                    n = 1 << e
                    rows = n // 4096
                    per_set = qbytes_of(n, layout, fmt)
                    sets = max(1, min(64, -(-2 * L2_BYTES // per_set)))
                    g = torch.Generator(device="cuda")
                    g.manual_seed(e)
                    xs = [torch.randn(rows, 4096, device="cuda", generator=g).to(torch.bfloat16)
                          for _ in range(sets)]
                    if layout == "dual":
                        outs = [mxq.mx_quantize_dual(xx, fmt, had, fmt, had) for xx in xs]
                        ls = [lambda i=i: mxq.mx_quantize_dual(xs[i], fmt, had, fmt, had, out=outs[i])
                              for i in range(sets)]
                    else:
                        q = mxq.hadamard_mx_quantize if had else mxq.mx_quantize
                        outs = [q(xx, layout, fmt) for xx in xs]
                        ls = [lambda i=i: q(xs[i], layout, fmt, out=outs[i]) for i in range(sets)]
                    ms_eager = _time_rotating(ls, reps=max(20, sets))
                    ms = _time_rotating(ls, reps=max(20, sets), graph=True)
                    gbs = per_set / ms / 1e6
                    emit({"config": "quantizer sweep", "fmt": fmt, "layout": layout,
                          "hadamard": had, "elements": n, "us": round(ms * 1e3, 2),
                          "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 3),
                          "us_eager": round(ms_eager * 1e3, 2),
                          "timing": "CUDA graph of the launches (us_eager: launched one by one)",
                          "cpu_oracle": oracle_rate})
                    del xs, outs, ls
                    torch.cuda.empty_cache()
    mxq.check()
    return lines


def run_case(name, timed=False):
    """Run one kernel case three times (for ncu captures of a single kernel).

    timed: instead, after 20 warm-up launches, time 100 launches each between
    CUDA events on the launching stream (inputs larger than L2) and print the
    median launch time (and the mean of 100 back-to-back launches) with the
    algorithmic GB/s or TFLOP/s against the peaks.
    """
    import torch

    from precision_mx_quantize_gb300 import mxq
    if name == "ablate-error":
        print(json.dumps(ablation_error()))
        return
    what, args = CASES[name]
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    if what in ("gemm", "gemmq"):
        M, N, K, fmt, od = args
        kb = K if fmt == "e4m3" else K // 2
        hi = 0x7E if fmt == "e4m3" else 256
        A = torch.randint(0, hi, (M, kb), dtype=torch.uint8, device="cuda", generator=g)
        B = torch.randint(0, hi, (N, kb), dtype=torch.uint8, device="cuda", generator=g)
        sA = torch.randint(120, 134, (M, K // 32), dtype=torch.uint8, device="cuda", generator=g)
        sB = torch.randint(120, 134, (N, K // 32), dtype=torch.uint8, device="cuda", generator=g)
        ws = mxq.gemm_workspace(M, N, K, fmt, "cuda")
        if what == "gemmq":
            q = mxq.mx_gemm_quantize(A, sA, B, sB, fmt, M, N, K, out_fmt=od, workspace=ws)
            launch = lambda: mxq.mx_gemm_quantize(A, sA, B, sB, fmt, M, N, K, out_fmt=od, out=q,
                                                  workspace=ws)
        else:
            dt = torch.float32 if od == "f32" else torch.bfloat16
            C = torch.empty((M, N), dtype=dt, device="cuda")
            launch = lambda: mxq.mx_gemm(A, sA, B, sB, fmt, M, N, K, out_dtype=dt, out=C,
                                         workspace=ws)
    elif what == "quant":
        R, Cc, fr, hr, fc, hc = args
        x = torch.randn(R, Cc, device="cuda", generator=g).to(torch.bfloat16)
        out = mxq.mx_quantize_dual(x, fr, hr, fc, hc)
        launch = lambda: mxq.mx_quantize_dual(x, fr, hr, fc, hc, out=out)
    elif what == "quant1":
        R, Cc, axis, f = args
        x = torch.randn(R, Cc, device="cuda", generator=g).to(torch.bfloat16)
        out = mxq.mx_quantize(x, axis, f)
        launch = lambda: mxq.mx_quantize(x, axis, f, out=out)
    elif what == "dequant":
        R, Cc, axis, f, od = args
        x = torch.randn(R, Cc, device="cuda", generator=g).to(torch.bfloat16)
        codes, sc = mxq.mx_quantize(x, axis, f)
        dt = torch.float32 if od == "f32" else torch.bfloat16
        out = torch.empty((R, Cc), dtype=dt, device="cuda")
        del x
        launch = lambda: mxq.mx_dequantize(codes, sc, R, Cc, axis, f, dt, out=out)
    else:
        R, Cc, axis, f, had, mask, sr = args
        x = torch.randn(R, Cc, device="cuda", generator=g).to(torch.bfloat16)
        out = mxq.mx_quantize_ablation(x, axis, f, had, mask, sr, 1)
        launch = lambda: mxq.mx_quantize_ablation(x, axis, f, had, mask, sr, 1, out=out)
    if not timed:
        for _ in range(3 if what in ("gemm", "gemmq") else 2):
            launch()
        mxq.check()
        print(json.dumps({"case": name, "status": "ok"}))
        return
    for _ in range(20):
        launch()
    torch.cuda.synchronize()
    n = 100
    # per-launch event pairs (median) and one back-to-back run (mean)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for a0, a1 in ev:
        a0.record()
        launch()
        a1.record()
    torch.cuda.synchronize()
    per = sorted(a0.elapsed_time(a1) for a0, a1 in ev)
    ms = per[n // 2]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        launch()
    e1.record()
    torch.cuda.synchronize()
    mxq.check()
    ms_b2b = e0.elapsed_time(e1) / n
    peaks = _peaks()
    line = {"case": name, "ms_per_launch": round(ms, 4), "timing": "median of 100 launches, "
            "each between CUDA events, after 20 warm-up launches",
            "ms_mean_back_to_back": round(ms_b2b, 4)}
    if what in ("gemm", "gemmq"):
        M, N, K, fmt, _ = args
        tf = 2 * M * N * K / ms / 1e9
        # a kernel timed alone: the burst bf16 figure times the nominal ratio
        peak = peaks["bf16"] * (6.0 if fmt == "e2m1" else 2.0)
        line.update({"TFLOP/s": round(tf, 1), "frac_of_peak": round(tf / peak, 3),
                     "peak_TFLOP/s": round(peak, 1)})
    gbs = _case_bytes(what, args) / ms / 1e6
    line.update({"algorithmic_GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 3),
                 "peak_source": peaks["source"]})
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tokens", type=int, default=8192)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the four single-kernel configurations after the block pass")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--case", choices=sorted(CASES) + ["ablate-error"],
                    help="run one kernel case (for ncu) and exit; ablate-error prints the "
                         "Wgrad error of the rotation / rounding variants")
    ap.add_argument("--timed", action="store_true", help="with --case: time the case's launches")
    ap.add_argument("--sweep", action="store_true",
                    help="time the round-trip, dual-Hadamard, MLP GEMM and quantizer-sweep "
                         "configurations (one JSON line each) and exit")
    args = ap.parse_args()
    if args.sweep:
        sweep()
        return
    if args.case:
        run_case(args.case, timed=args.timed)
        return
    args.warmup = max(3, args.warmup)

    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local_rank = _env_int("LOCAL_RANK", 0)

    if args.impl == "reference":
        line = reference_arm(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch.distributed as dist
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", rank=rank, world_size=world)
    try:
        line = gpu_arm(args, rank, world, local_rank)
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
