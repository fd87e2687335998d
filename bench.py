"""Benchmark of the WTConv layer's training step (forward + fused backward) on GB300.

One step = wtconv_forward + wtconv_backward (dx and every parameter gradient) over one batch of
the seeded synthetic workload, through the C ABI.  Default workload (the headline): four WTConv
layers back to back, bf16 activations, B = 128, k = 5: (C = 96, 64 x 64, L = 4), (192, 32 x 32,
L = 3), (384, 16 x 16, L = 2), (768, 8 x 8, L = 1).  `per_config` in the same line repeats the
device-timed measurement on every workload configuration (tiny, ConvNeXt-T stage 1 and 2 shapes,
high resolution, four layers).

Prints ONE JSON line (rank 0).  `value` is fwd+bwd throughput in Gpixel*ch/s = B*C*H*W / step
time over all ranks (replicas: each rank runs its own copy of the workload, "scaling": "weak").
Timing: W untimed warm-up steps, then K timed steps; L2 is flushed (256 MiB write) before each
timed step and each step is bracketed by CUDA events on the launching stream (the flush is not
inside the bracket).  Also reported: the roofline of the dominant kernel (FP32 packed-FMA pipe:
algorithmic FLOPs over its event-timed launches, against the peak derived from the device's SM
count and clock, against the peak measured by the library's packed-FMA probe, and at the sampled
median clock; HBM: ncu DRAM bytes per launch from the committed profiles over the same time,
beside the algorithmic bytes), an end-to-end number with host buffers (pinned host -> device
copies of x and dy and device -> host copies of y, dx and the gradients inside the timed region),
the CPU oracle baseline, and SM clocks sampled during the timed region.

`--impl reference` times the CPU oracle (the plain fp64 reference pipeline) instead, on the host
cores, on a bounded sample of the same workload.  `--impl torch-cascade` times the same reference
cascade written with PyTorch ops on the GPU (grouped convs, autograd): a comparison arm.
`--impl dwconv7` times a plain depthwise 7x7 conv at the same shapes.  `--peak` prints only the
packed-FMA probe's result.
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from memory_bound_cnn_gb300 import wtconv as W  # noqa: E402
from memory_bound_cnn_gb300.inputs import WORKLOAD_ORDER, WORKLOADS, LayerShape, make_inputs  # noqa: E402

PARAMS = ("base_w", "base_bias", "base_scale", "wavelet_w", "wavelet_scale")
GRADS = ("d_base_w", "d_base_bias", "d_base_scale", "d_wavelet_w", "d_wavelet_scale")
METRIC = "WTConv fwd+bwd Gpixel·ch/s and achieved HBM GB/s as % of GB300 peak"
UNIT = "Gpixel·ch/s"
HBM_FALLBACK_GBS = 6800.0       # the profiling recipe's fallback (MEASURED_PEAKS.json absent)
SM_MAX_MHZ_FALLBACK = 2070.0     # GB300's maximum SM clock
HEADLINE = "four_layers_bf16"


# ----------------------------------------------------------------------------- accounting

def s_levels(L: int) -> float:
    """Sum over levels of the level-input size relative to the full plane: sum_{l=1..L} 4^(1-l)."""
    return sum(4.0 ** (1 - l) for l in range(1, L + 1))


def algorithmic(shape: LayerShape) -> dict:
    """Per-layer algorithmic FLOPs and HBM bytes (conv multiply-adds x 2; one read of each input
    activation and one write of each output activation)."""
    n = shape.numel
    e = 2 if shape.dtype in ("bf16", "f16") else 4
    conv = 2.0 * shape.k * shape.k * (1.0 + s_levels(shape.L)) * n
    return {
        "fwd_flop": conv, "bwd_flop": 2.0 * conv,
        "fwd_bytes": 2.0 * n * e, "bwd_bytes": 3.0 * n * e,
    }


def source_hash() -> str:
    """Hash of the library's sources: a committed ncu traffic figure counts only while it matches."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "memory_bound_cnn_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, fn), "rb") as f:
                h.update(fn.encode() + f.read())
    with open(os.path.join(ROOT, "include", "wtconv.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str) -> dict:
    """ncu DRAM bytes per launch, {(layer, op, kernel): bytes}, from the committed profile summary of
    `workload` (profiles/traffic_<workload>.md); empty if it is missing or was taken on other sources."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.md")
    if not os.path.exists(path):
        return {}
    text = open(path).read()
    m = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    if not m or m.group(1) != source_hash():
        return {}
    out = {}
    for layer, op, kernel, b in re.findall(r"traffic: layer=(\d+) op=(\w+) kernel=(\S+) bytes=([0-9.eE+]+)", text):
        out[(int(layer), op, kernel)] = float(b)
    return out


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            return json.load(open(path))
        except ValueError:
            pass
    return {}


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,utilization.gpu,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "20", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 9:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        loaded = [r for r in rows if r[2] > 0] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in loaded for n, v in zip(names, r[3][1:]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(loaded)}


# ------------------------------------------------------------------------ distributed bits

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (identity for one process)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_throughput(elements_per_rank: int, world: int, seconds_max: float) -> float:
    """Gpixel*ch/s of the whole job: every rank processes its own copy of the workload."""
    return elements_per_rank * world / seconds_max / 1e9


# ------------------------------------------------------------------------------- CUDA arm

def dims(s: LayerShape):
    return s.B, s.C, s.H, s.W, s.L, s.k, W.DTYPE_CODE[{"f32": torch.float32, "bf16": torch.bfloat16,
                                                     "f16": torch.float16}[s.dtype]]


def setup_layers(workload: str, dev):
    """Device inputs, outputs and workspace of every layer of `workload` (seeded host inputs)."""
    layers = []
    for i, s in enumerate(WORKLOADS[workload]):
        host = make_inputs(s, seed=i)
        d = {k: v.to(dev) for k, v in host.items()}
        ws = torch.empty(max(1, W.wtconv_workspace_size(W.OP_BACKWARD, *dims(s))), dtype=torch.uint8, device=dev)
        out = {"y": torch.empty_like(d["x"]), "dx": torch.empty_like(d["x"]),
               "grads": {g: torch.empty_like(d[p]) for g, p in zip(GRADS, PARAMS)}}
        layers.append((s, host, d, ws, out))
    return layers


def make_step(layers, stream):
    def step(ev=None):
        for i, (s, _, d, ws, out) in enumerate(layers):
            p = [d[n] for n in PARAMS]
            if ev is not None:
                ev[i][0].record(stream)
            W.wtconv_forward(d["x"], *p, y=out["y"], stream=stream)
            if ev is not None:
                ev[i][1].record(stream)
            W.wtconv_backward(d["x"], d["dy"], *p, dx=out["dx"], grads=out["grads"], workspace=ws, stream=stream)
            if ev is not None:
                ev[i][2].record(stream)
    return step


def time_layers(layers, steps, warmup, stream, flush, dev, world, clk=None):
    """Per-layer fwd / bwd event times (ms, mean over the timed steps, max over ranks), L2 flushed
    before every timed step (outside the event bracket)."""
    step = make_step(layers, stream)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    nl = len(layers)
    events = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nl)] for _ in range(steps)]
    with (clk if clk is not None else contextlib.nullcontext()):
        barrier(world)
        torch.cuda.synchronize(dev)
        for k in range(steps):
            flush.zero_()
            step(events[k])
        torch.cuda.synchronize(dev)
        barrier(world)
    fwd = [max_over_ranks(sum(events[k][i][0].elapsed_time(events[k][i][1]) for k in range(steps)) / steps, world)
           for i in range(nl)]
    bwd = [max_over_ranks(sum(events[k][i][1].elapsed_time(events[k][i][2]) for k in range(steps)) / steps, world)
           for i in range(nl)]
    return fwd, bwd


def fp32_peaks(dev, clocks) -> dict:
    """FP32 packed-FMA peaks: derived from the device's SM count and maximum clock (128 FP32 lanes
    x 2 FLOP per SM per cycle), at the median SM clock sampled under load, and measured by the
    library's packed-FMA probe."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peaks = measured_peaks()
    max_mhz = float(peaks.get("sm_max_mhz") or (clocks or {}).get("sm_max_mhz") or SM_MAX_MHZ_FALLBACK)
    med_mhz = float((clocks or {}).get("sm_mhz") or max_mhz)
    derived = sms * 128 * 2 * max_mhz * 1e6 / 1e12
    with torch.cuda.device(dev):
        measured = W.wtconv_fp32_fma_peak(20000)
    return {"derived": round(derived, 2), "at_median_clock": round(sms * 256 * med_mhz * 1e6 / 1e12, 2),
            "measured": round(measured, 2), "sms": sms, "max_mhz": max_mhz, "median_mhz": med_mhz,
            "note": f"derived: {sms} SMs x 128 FP32 lanes x 2 FLOP x {max_mhz:.0f} MHz; measured: packed-FMA "
                    "chains on every SM (wtconv_fp32_fma_peak)"}


def layer_roofline(workload, i, s, fwd_ms, fp32, traffic) -> dict:
    """Roofline of layer i's forward operator kernel (it runs twice per step: y, and dx inside the
    backward); its launches in wtconv_forward are timed alone by the fwd events."""
    a = algorithmic(s)
    kname = "+".join(W.wtconv_plan_kernels(W.OP_FORWARD, *dims(s)))
    tflops = a["fwd_flop"] / (fwd_ms / 1e3) / 1e12
    peaks = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", HBM_FALLBACK_GBS))
    alg_gbs = a["fwd_bytes"] / (fwd_ms / 1e3) / 1e9
    t = traffic.get((i, "fwd", kname))
    ncu_gbs = None if t is None else t / (fwd_ms / 1e3) / 1e9
    return {
        "bound": "alu", "achieved": round(tflops, 3), "peak": fp32["derived"], "unit": "TFLOP/s",
        "frac": round(tflops / fp32["derived"], 4), "traffic": t, "kernel": kname, "layer": i,
        "launch_ms": round(fwd_ms, 5), "algorithmic_flop_per_launch": a["fwd_flop"],
        "algorithmic_bytes_per_launch": a["fwd_bytes"],
        "peak_measured": fp32["measured"], "frac_measured": round(tflops / fp32["measured"], 4),
        "peak_at_median_clock": fp32["at_median_clock"],
        "frac_at_median_clock": round(tflops / fp32["at_median_clock"], 4),
        "hbm_achieved_gbs": None if ncu_gbs is None else round(ncu_gbs, 1),
        "hbm_frac": None if ncu_gbs is None else round(ncu_gbs / hbm_peak, 4),
        "hbm_achieved_gbs_algorithmic": round(alg_gbs, 1), "hbm_frac_algorithmic": round(alg_gbs / hbm_peak, 4),
        "hbm_peak_gbs": hbm_peak,
        "peak_note": "peak: FP32 packed-FMA peak derived from the SM count and maximum clock; hbm_frac: ncu DRAM "
                     "bytes per launch (committed profile, same sources) over the event time, against the "
                     "measured copy bandwidth; hbm_frac_algorithmic: one read of x and one write of y",
    }


def workload_summary(workload, layers, fwd, bwd, fp32, world) -> dict:
    """Throughput and rooflines of one timed workload; the headline roofline is the layer whose
    forward operator (two launches per step) takes the largest share of the step."""
    traffic = profiled_traffic(workload)
    elements = sum(s.numel for s, *_ in layers)
    step_ms = sum(fwd) + sum(bwd)
    per_layer = []
    for i, (s, *_rest) in enumerate(layers):
        per_layer.append({"layer": i, "fwd_ms": round(fwd[i], 5), "bwd_ms": round(bwd[i], 5),
                          "value": round(s.numel / ((fwd[i] + bwd[i]) / 1e3) / 1e9, 3),
                          "roofline": layer_roofline(workload, i, s, fwd[i], fp32, traffic)})
    top = max(range(len(layers)), key=lambda i: fwd[i])
    return {"workload": workload, "value": round(whole_job_throughput(elements, world, step_ms / 1e3), 3),
            "ms_per_step": round(step_ms, 5), "fwd_ms": round(sum(fwd), 5), "bwd_ms": round(sum(bwd), 5),
            "roofline": per_layer[top]["roofline"], "per_layer": per_layer}


def run_gpu(args, world, rank, local):
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    shapes = WORKLOADS[args.workload]
    layers = setup_layers(args.workload, dev)
    clk = ClockSampler(local)
    fwd_ms, bwd_ms = time_layers(layers, args.steps, args.warmup, stream, flush, dev, world, clk)
    clocks = clk.summary()
    step_ms = sum(fwd_ms) + sum(bwd_ms)
    elements = sum(s.numel for s, *_ in layers)
    value = whole_job_throughput(elements, world, step_ms / 1e3)
    nl = len(layers)

    # warm: the same steps back to back without the L2 flush (small workloads stay in the 129 MB L2)
    step = make_step(layers, stream)
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    w0.record(stream)
    for k in range(args.steps):
        step()
    w1.record(stream)
    torch.cuda.synchronize(dev)
    warm_ms = max_over_ranks(w0.elapsed_time(w1) / args.steps, world)

    # end to end through the public API with host buffers (pinned), copies inside the timed region.
    # Every step copies its inputs in and its results out; the copies run on their own streams
    # (one per direction) and overlap the compute of the neighbouring steps, with two device
    # copies of every activation so that a step's uploads never overwrite what the previous
    # step still reads.
    pinned = []
    for s, host, d, ws, out in layers:
        pinned.append({"x": host["x"].pin_memory(), "dy": host["dy"].pin_memory(),
                       "y": torch.empty(host["x"].shape, dtype=host["x"].dtype).pin_memory(),
                       "dx": torch.empty(host["x"].shape, dtype=host["x"].dtype).pin_memory(),
                       "grads": {g: torch.empty(host[p].shape).pin_memory() for g, p in zip(GRADS, PARAMS)}})
    h2d = sum(p["x"].numel() * p["x"].element_size() * 2 for p in pinned)
    d2h = sum(p["y"].numel() * p["y"].element_size() * 2 + sum(v.numel() * 4 for v in p["grads"].values())
              for p in pinned)
    sets = []
    for s, host, d, ws, out in layers:
        sets.append([{"x": torch.empty_like(d["x"]), "dy": torch.empty_like(d["dy"]), "y": torch.empty_like(d["x"]),
                      "dx": torch.empty_like(d["x"]),
                      "grads": {g: torch.empty_like(d[p]) for g, p in zip(GRADS, PARAMS)}} for _ in range(2)])
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    done = [[torch.cuda.Event() for _ in range(2)] for _ in layers]  # compute of a set finished
    read = [[torch.cuda.Event() for _ in range(2)] for _ in layers]  # results of a set copied out
    for li in range(len(layers)):
        for k in range(2):
            done[li][k].record(stream)
            read[li][k].record(stream)

    def e2e_step(n):
        k = n & 1
        for li, ((s, _, d, ws, out), hp) in enumerate(zip(layers, pinned)):
            dv = sets[li][k]
            p = [d[q] for q in PARAMS]
            ex, edy, ey = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
            up.wait_event(done[li][k])              # the set's previous compute has read x and dy
            with torch.cuda.stream(up):
                dv["x"].copy_(hp["x"], non_blocking=True)
                ex.record(up)
                dv["dy"].copy_(hp["dy"], non_blocking=True)
                edy.record(up)
            stream.wait_event(ex)
            stream.wait_event(read[li][k])          # the set's previous results are out
            W.wtconv_forward(dv["x"], *p, y=dv["y"], stream=stream)
            ey.record(stream)
            stream.wait_event(edy)
            W.wtconv_backward(dv["x"], dv["dy"], *p, dx=dv["dx"], grads=dv["grads"], workspace=ws, stream=stream)
            done[li][k].record(stream)
            down.wait_event(ey)
            with torch.cuda.stream(down):
                hp["y"].copy_(dv["y"], non_blocking=True)
            down.wait_event(done[li][k])
            with torch.cuda.stream(down):
                hp["dx"].copy_(dv["dx"], non_blocking=True)
                for g in GRADS:
                    hp["grads"][g].copy_(dv["grads"][g], non_blocking=True)
                read[li][k].record(down)

    for n in range(args.warmup):
        e2e_step(n)
    torch.cuda.synchronize(dev)
    e2e_steps = max(3, min(args.steps, 50))
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_event(e0)
    down.wait_event(e0)
    for n in range(e2e_steps):
        e2e_step(n)
    for li in range(len(layers)):
        for k in range(2):
            stream.wait_event(read[li][k])  # the last results are on the host
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    barrier(world)
    # the host copies hold the last step's results: check them against the device-timed outputs
    for (s, _, d, ws, out), hp in zip(layers, pinned):
        if not torch.equal(hp["y"], out["y"].cpu()):
            raise RuntimeError("end-to-end results differ from the device-timed run")
    step_mem = int(sum(out["y"].nbytes + out["dx"].nbytes + ws.nbytes + sum(g.nbytes for g in out["grads"].values())
                       for _, _, _, ws, out in layers))
    del sets, pinned, layers
    torch.cuda.empty_cache()

    fp32 = fp32_peaks(dev, clocks)
    head = workload_summary(args.workload, [(s, None, None, None, None) for s in shapes], fwd_ms, bwd_ms, fp32,
                            world)
    # every workload configuration, device-timed the same way (fewer steps for the others)
    per_config = []
    for name in ([] if args.no_per_config else WORKLOAD_ORDER):
        if name == args.workload:
            entry = dict(head)
        else:
            lay = setup_layers(name, dev)
            f, b = time_layers(lay, max(3, min(args.steps, 100)), args.warmup, stream, flush, dev, world)
            entry = workload_summary(name, lay, f, b, fp32, world)
            del lay
            torch.cuda.empty_cache()
        entry["layers"] = [s.as_dict() for s in WORKLOADS[name]]
        per_config.append(entry)

    per_step = sum(W.wtconv_launch_count(W.OP_FORWARD, *dims(s)) + W.wtconv_launch_count(W.OP_BACKWARD, *dims(s))
                   for s in shapes)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": shapes[0].dtype, "data": "synthetic",
        "config": {"workload": args.workload, "layers": [s.as_dict() for s in shapes],
                   "l2": "flushed before every timed step (256 MiB write, outside the event bracket)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "fwd_ms": round(sum(fwd_ms), 5), "bwd_ms": round(sum(bwd_ms), 5),
        # every layer on its own (event times): fwd + bwd throughput and roofline of the layer
        "per_layer": head["per_layer"],
        "warm": {"value": round(whole_job_throughput(elements, world, warm_ms / 1e3), 3), "unit": UNIT,
                 "ms_per_step": round(warm_ms, 5), "note": "same steps back to back, L2 not flushed"},
        "roofline": head["roofline"],
        "fp32_peak": fp32,
        "e2e": {"value": round(whole_job_throughput(elements, world, e2e_ms / 1e3), 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "note": "pinned host buffers; uploads, compute and downloads on three streams, overlapping "
                        "neighbouring steps (two device copies of every activation)"},
        "gpu_launches": per_step * args.steps,
        "clocks": clocks,
        # device memory a step needs beyond the inputs and parameters: y, dx, the gradients and
        # the workspace of every layer (the autograd arms report the same quantity)
        "step_mem_bytes": step_mem,
    }
    if per_config:
        line["per_config"] = per_config
    return line


# -------------------------------------------------------------------------- oracle arm

def oracle_layers(workload: str):
    return [(s, make_inputs(s, seed=i)) for i, s in enumerate(WORKLOADS[workload])]


def oracle_run(layers, b: int, threads: int):
    """One fwd+bwd of the CPU oracle on the first b batch entries of every layer: (elements, s)."""
    import oracle
    elements, secs = 0, 0.0
    for s, inp in layers:
        bb = min(s.B, b)
        sub = dict(inp, x=inp["x"][:bb].contiguous(), dy=inp["dy"][:bb].contiguous())
        t0 = time.perf_counter()
        oracle.forward(sub["x"], sub, nthreads=threads)
        oracle.backward(sub["x"], sub["dy"], sub, nthreads=threads)
        secs += time.perf_counter() - t0
        elements += bb * s.C * s.H * s.W
    return elements, secs


def oracle_sample_size(layers, budget_s: float, threads: int) -> int:
    """Batch entries per layer whose fwd+bwd takes about budget_s (at least 1)."""
    bmax = max(s.B for s, _ in layers)
    _, t1 = oracle_run(layers, 1, threads)
    return int(max(1, min(bmax, budget_s / max(t1, 1e-6))))


def cpu_baseline(workload: str, budget_s: float) -> dict:
    import oracle
    threads = oracle.default_threads()
    layers = oracle_layers(workload)
    b = oracle_sample_size(layers, budget_s, threads)
    # repeat the sample until about budget_s of CPU work has been timed (a whole small workload
    # runs in well under a second)
    elements, secs, passes = 0, 0.0, 0
    while passes == 0 or secs < budget_s:
        e, t = oracle_run(layers, b, threads)
        elements += e
        secs += t
        passes += 1
    # and on one host thread, on a smaller sample (about a quarter of the budget)
    b1 = oracle_sample_size(layers, budget_s / 4, 1)
    e1, t1 = oracle_run(layers, b1, 1)
    return {"value": round(elements / secs / 1e9, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {b} batch entries of every layer of {workload}, fwd+bwd, fp64, "
                      f"{threads} threads, {passes} passes, {secs:.2f} s",
            "single_thread": {"value": round(e1 / t1 / 1e9, 6), "unit": UNIT, "cores": 1,
                              "sample": f"first {b1} batch entries of every layer, fwd+bwd, fp64, {t1:.2f} s"}}


def run_reference(args, world, rank):
    """The oracle as it stands on the host cores; each step is a bounded sample of the workload
    sized so that warm-up + timed steps take about two minutes in all."""
    if rank != 0:
        return None
    import oracle
    threads = oracle.default_threads()
    layers = oracle_layers(args.workload)
    per_step = min(5.0, 120.0 / (args.steps + args.warmup))
    b = oracle_sample_size(layers, per_step, threads)
    for _ in range(args.warmup):
        oracle_run(layers, b, threads)
    elements, secs = 0, 0.0
    for _ in range(args.steps):
        e, t = oracle_run(layers, b, threads)
        elements += e
        secs += t
    value = elements / secs / 1e9
    shapes = WORKLOADS[args.workload]
    desc = f"first {b} batch entries of every layer of {args.workload} per step, fwd+bwd, fp64, {threads} threads"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "layers": [s.as_dict() for s in shapes]},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------------- main

# ----------------------------------------------------------------- PyTorch-op cascade arm

def haar_filters(C: int, device, dtype) -> torch.Tensor:
    """The four orthonormal 2 x 2 Haar filters (LL, LH, HL, HH sign patterns x 1/2), repeated per
    channel as a grouped-conv weight [4C, 1, 2, 2] (subband channel 4c+s)."""
    f = torch.tensor([[[1, 1], [1, 1]], [[1, -1], [1, -1]], [[1, 1], [-1, -1]], [[1, -1], [-1, 1]]],
                     dtype=torch.float64) * 0.5
    return f.repeat(C, 1, 1).unsqueeze(1).to(device=device, dtype=dtype)


def torch_cascade(x, base_w, base_bias, base_scale, wavelet_w, wavelet_scale):
    """The reference cascade written with PyTorch ops (grouped convs, autograd for the backward):
    explicit Haar analysis per level, per-subband conv, separate scale, the synthesis cascade that
    adds each deeper reconstruction to the scaled LL conv output before the inverse transform, and
    the scaled base conv with bias.  A comparison arm only: it is not the product path."""
    import torch.nn.functional as F
    B, C, H, Wd = x.shape
    L, k = wavelet_w.shape[0], base_w.shape[-1]
    P = k // 2
    filt = haar_filters(C, x.device, x.dtype)
    ys, ll = [], x
    for l in range(L):
        y = F.conv2d(ll, filt, stride=2, groups=C)               # [B, 4C, H/2^l, W/2^l]
        ys.append(y)
        ll = y[:, 0::4]
    r = None
    for l in reversed(range(L)):
        z = F.conv2d(ys[l], wavelet_w[l].unsqueeze(1).to(x.dtype), padding=P, groups=4 * C)
        z = z * wavelet_scale[l].to(x.dtype).view(1, -1, 1, 1)
        if r is not None:
            z = torch.cat([z[:, 0::4] + r, z[:, 1::4], z[:, 2::4], z[:, 3::4]], dim=1)
            z = z.view(B, 4, C, *z.shape[2:]).transpose(1, 2).reshape(B, 4 * C, *z.shape[2:])
        r = F.conv_transpose2d(z, filt, stride=2, groups=C)
    base = F.conv2d(x, base_w.unsqueeze(1).to(x.dtype), padding=P, groups=C) + base_bias.to(x.dtype).view(1, -1, 1, 1)
    return base * base_scale.to(x.dtype).view(1, -1, 1, 1) + r


def run_torch_cascade(args, world, rank, local):
    """fwd + bwd of the PyTorch-op cascade on the GPU (fp32 convs without TF32), same workload."""
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    torch.backends.cudnn.allow_tf32 = False
    torch.backends.cuda.matmul.allow_tf32 = False
    shapes = WORKLOADS[args.workload]
    layers = []
    for i, s in enumerate(shapes):
        d = {k2: v.to(dev) for k2, v in make_inputs(s, seed=i).items()}
        for n in PARAMS:
            d[n].requires_grad_(True)
        d["x"].requires_grad_(True)
        layers.append((s, d))

    def step():
        for s, d in layers:
            for t in [d["x"]] + [d[n] for n in PARAMS]:
                t.grad = None
            y = torch_cascade(d["x"], *[d[n] for n in PARAMS])
            y.backward(d["dy"])

    leaves = [t for _, d in layers for t in [d["x"]] + [d[n] for n in PARAMS]]
    line = time_autograd_arm(args, world, dev, layers, step, leaves)
    # one more step with its forward and backward inside NVTX ranges, so that a profiler can
    # attribute the DRAM traffic of each (the backward runs on autograd's own thread: a
    # process-wide start/end range)
    for s, d in layers:
        torch.cuda.synchronize(dev)
        torch.cuda.nvtx.range_push("cascade_fwd")
        y = torch_cascade(d["x"], *[d[n] for n in PARAMS])
        torch.cuda.synchronize(dev)
        torch.cuda.nvtx.range_pop()
        rid = torch.cuda.nvtx.range_start("cascade_bwd")
        y.backward(d["dy"])
        torch.cuda.synchronize(dev)
        torch.cuda.nvtx.range_end(rid)
    line.update({"impl": "torch-cascade",
                 "note": "PyTorch grouped convs (PyTorch's depthwise kernels or cuDNN, as PyTorch picks; no TF32) + "
                         "autograd of the reference cascade; comparison arm"})
    return line


def time_autograd_arm(args, world, dev, layers, step, leaves):
    """Warm-up, the device memory one step allocates at its peak beyond what exists before it
    (activations saved for the backward, outputs, the gradients of `leaves`), then event-timed
    steps."""
    shapes = WORKLOADS[args.workload]
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    for t in leaves:
        t.grad = None
    torch.cuda.synchronize(dev)
    before = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    step()
    torch.cuda.synchronize(dev)
    step_mem = torch.cuda.max_memory_allocated(dev) - before
    steps = max(3, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    elements = sum(s.numel for s, _ in layers)
    value = whole_job_throughput(elements, world, ms / 1e3)
    return {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": shapes[0].dtype, "data": "synthetic",
        "config": {"workload": args.workload, "layers": [s.as_dict() for s in shapes]},
        "step_mem_bytes": int(step_mem),
    }


def run_dwconv(args, world, rank, local, k=7):
    """fwd + bwd of a plain depthwise k x k conv with bias (torch conv2d, groups=C: PyTorch's
    depthwise kernels or cuDNN, as PyTorch picks; no TF32) at the workload's shapes: the layer
    WTConv replaces, timed for context."""
    import torch.nn.functional as F
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    torch.backends.cudnn.allow_tf32 = False
    torch.backends.cuda.matmul.allow_tf32 = False
    g = torch.Generator().manual_seed(0)
    layers = []
    for i, s in enumerate(WORKLOADS[args.workload]):
        d = {k2: v.to(dev) for k2, v in make_inputs(s, seed=i).items() if k2 in ("x", "dy")}
        act = d["x"].dtype
        d["w"] = (torch.randn(s.C, 1, k, k, generator=g) / k).to(dev, act).requires_grad_(True)
        d["b"] = (torch.randn(s.C, generator=g) * 0.1).to(dev, act).requires_grad_(True)
        d["x"].requires_grad_(True)
        layers.append((s, d))

    def step():
        for s, d in layers:
            for t in (d["x"], d["w"], d["b"]):
                t.grad = None
            y = F.conv2d(d["x"], d["w"], d["b"], padding=k // 2, groups=s.C)
            y.backward(d["dy"])

    leaves = [t for _, d in layers for t in (d["x"], d["w"], d["b"])]
    line = time_autograd_arm(args, world, dev, layers, step, leaves)
    line.update({"impl": f"dwconv{k}",
                 "note": f"plain depthwise {k}x{k} conv + bias (torch conv2d groups=C, no TF32), "
                         "fwd+bwd at the same shapes; context, not the product"})
    return line


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("cuda", "reference", "torch-cascade", "dwconv7"), default="cuda")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--peak", action="store_true", help="print only the packed-FMA peak probe's result")
    ap.add_argument("--no-per-config", action="store_true", help="time the chosen workload only")
    ap.add_argument("--shape", help="one custom layer B,C,H,W,L,k,dtype instead of a named workload "
                                    "(e.g. 32,96,64,64,4,5,bf16)")
    args = ap.parse_args(argv)
    if args.shape:
        f = args.shape.split(",")
        if len(f) != 7:
            ap.error("--shape wants B,C,H,W,L,k,dtype")
        WORKLOADS["custom"] = [LayerShape(*(int(v) for v in f[:6]), f[6])]
        args.workload = "custom"
        args.no_per_config = True
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "cuda" else "gloo"
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            line = run_reference(args, world, rank)
        elif args.impl == "torch-cascade":
            line = run_torch_cascade(args, world, rank, local)
        elif args.impl == "dwconv7":
            line = run_dwconv(args, world, rank, local, k=7)
        elif args.peak:
            W.load()
            torch.cuda.set_device(local)
            line = {"fp32_peak": fp32_peaks(torch.device("cuda", local), None)}
        else:
            W.load()
            line = run_gpu(args, world, rank, local)
            if rank == 0 and not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=10.0)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
