"""Benchmark of the conv + BN + activation backward on GB300.

One step = one backward of the darknet residual block (batch 32 at 26x26:
the 3x3 conv 256 -> 512 + BN + leaky with delta D, then the 1x1 conv
512 -> 256 + BN + leaky with the shortcut D added into the block-input
gradient), the largest of the five workloads, through the C ABI: per layer
reduction pass -> dz -> wgrad -> dgrad, captured once into a CUDA graph and
replayed (the per-phase split and the direct-call time come from traced calls
without the graph).  ``per_config`` repeats the measurement, with fewer steps,
for each of the five workloads.  Inputs are resident in HBM
when the timed region starts; L2 is flushed before every timed step, outside
the per-step CUDA-event window: a 512 MiB write (evicts everything), then a
256 MiB read sweep, so that the flush's own dirty lines are written back
before the step instead of inside it.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead, on bounded samples of the same workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "conv+BN+act backward TFLOP/s and fraction of TF32 roofline per layer, 1×GB300"
UNIT = "TFLOP/s"
# nominal dense tensor rates, PFLOP/s: tf32 1.1, bf16 2.25 -> tf32 = bf16 * 1.1/2.25
TF32_PER_BF16 = 1.1 / 2.25
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# the phases a traced call's events bound: reduction pass, GEMM operand
# layout pass, weight gradient, input gradient
PHASES = ("reduce", "layout", "wgrad", "dgrad")
SPIN_CYCLES = 2_000_000  # about 1 ms at the SM clock
PATH_NAMES = {0: "ffma", 1: "tc_rows", 2: "tc_batch_inner", 3: "tc_gemm_1x1"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=5,
                    help="workload 1-5 (default 5, the residual block, the largest)")
    ap.add_argument("--math", default="tf32", choices=["tf32", "ffma"])
    ap.add_argument("--act", default=None,
                    choices=["linear", "leaky", "logistic", "relu", "relie", "ramp", "tanh",
                             "plse", "elu", "selu", "lhtan", "hardtan", "loggy", "stair"],
                    help="replace the workload's activation (outputs recomputed)")
    ap.add_argument("--layer", default="conv", choices=["conv", "maxpool", "route", "yolo"],
                    help="conv (default): the convolution layer backward; the others time "
                         "the data-movement layers' backward in GB/s")
    ap.add_argument("--groups", type=int, default=1,
                    help="run the workload (configs 1-4) as a grouped convolution")
    ap.add_argument("--z-free", action="store_true",
                    help="BN layers without z: the library recomputes z = conv(x, W)")
    ap.add_argument("--bn", default="batch", choices=["batch", "frozen"],
                    help="BN statistics of the workload's BN layers: the batch's own "
                         "(training mode, default) or frozen ones (batch_normalize = 2)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config entries (configs 1-5, 1 GPU only)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (a smaller case for profiling)")
    ap.add_argument("--layer-index", type=int, default=None,
                    help="time only this layer call of the workload (config 5 has two: "
                         "0 = the 3x3 conv, 1 = the 1x1 conv); for profiling")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target seconds of oracle work for cpu_baseline")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, ws, device):
    """The largest of every rank's `value` (each rank is one replica; the job
    takes as long as its slowest rank).  Collective only when ws > 1."""
    if ws <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ws, flops_per_replica_step, ms_per_step):
    """Whole-job throughput in TFLOP/s: every rank runs one replica's step,
    all ranks' work divided by the slowest rank's step time."""
    return ws * flops_per_replica_step / (ms_per_step * 1e-3) / 1e12


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((float(parts[2]), float(parts[3]), float(parts[4]), parts[5:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[3][1:5]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [r[0] for r in rows if r[2] > 150.0] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r[2] for r in rows)}


# ---------------------------------------------------------- oracle timing

def oracle_sample_run(layer, n_img, k_sub):
    """The oracle's full chain on a bounded sample of one layer call: the
    first n_img images and the first k_sub output channels.  Returns
    (seconds, GEMM FLOPs of the sample)."""
    import numpy as np

    import oracle
    from activation_backward_gb300 import inputs
    g = layer["geom"]
    sub = dict(layer)
    sl = slice(0, n_img)
    for key in ("x", "residual"):
        if sub.get(key) is not None:
            sub[key] = np.ascontiguousarray(sub[key][sl])
    for key in ("output", "z", "delta"):
        if sub.get(key) is not None:
            sub[key] = np.ascontiguousarray(sub[key][sl, :k_sub])
    for key in ("gamma", "mean", "var"):
        if sub.get(key) is not None:
            sub[key] = np.ascontiguousarray(sub[key][:k_sub])
    sub["W"] = np.ascontiguousarray(sub["W"][:k_sub])
    gs = inputs.Geometry(n_img, g.C, g.H, g.W, k_sub, g.R, g.S, g.stride, g.pad)
    t0 = time.perf_counter()
    oracle.conv_bn_act_backward(sub["x"], sub["output"], sub["z"], sub["delta"], sub["W"],
                                sub["gamma"], sub["mean"], sub["var"], sub["residual"],
                                stride=g.stride, pad=g.pad, act=sub["act"],
                                batch_normalize=sub["bn"], accumulate=sub["accumulate"],
                                eps=sub["eps"])
    return time.perf_counter() - t0, 2 * gs.gemm_flops()


def pick_sample(layers, seconds):
    """Choose (n_img, k_sub) so that one oracle run takes about `seconds`."""
    layer = layers[0]
    g = layer["geom"]
    k1 = max(1, min(g.K, 16))
    t, _ = oracle_sample_run(layer, 1, k1)
    per = t / k1  # seconds per (image, channel)
    units = max(1, int(seconds / max(per, 1e-9)))
    n_img = max(1, min(g.N, units // g.K))
    k_sub = g.K if n_img > 1 else max(1, min(g.K, units))
    return n_img, k_sub


def cpu_baseline(layers, seconds):
    """The oracle on a bounded sample of the workload, run repeatedly until
    about `seconds` of CPU time have accumulated (at most 64 runs)."""
    import oracle
    n_img, k_sub = pick_sample(layers, seconds)
    t_tot, flops_tot, runs = 0.0, 0, 0
    while runs < 64 and (runs == 0 or t_tot < seconds):
        t, flops = oracle_sample_run(layers[0], n_img, k_sub)
        t_tot += t
        flops_tot += flops
        runs += 1
    g = layers[0]["geom"]
    return {"value": flops_tot / t_tot / 1e12, "unit": UNIT, "cores": oracle.get_threads(),
            "kind": "oracle",
            "sample": f"{layers[0]['name']}: {n_img} of {g.N} images x {k_sub} of {g.K} output "
                      f"channels, full chain (fp64 direct loops), {runs} run(s) in "
                      f"{t_tot:.1f} s"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from activation_backward_gb300 import inputs
    layers = workload_layers(args)
    total = args.steps + args.warmup
    budget = 150.0 / max(total, 1)  # ~2.5 minutes for the whole run
    n_img, k_sub = pick_sample(layers, budget)
    for _ in range(args.warmup):
        oracle_sample_run(layers[0], n_img, k_sub)
    times, flops = [], 0
    for _ in range(args.steps):
        t, flops = oracle_sample_run(layers[0], n_img, k_sub)
        times.append(t)
    tot = sum(times)
    value = flops * args.steps / tot / 1e12
    g = layers[0]["geom"]
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": config_dict(args, layers, 1),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.get_threads(),
                             "kind": "oracle",
                             "sample": f"per step {n_img} of {g.N} images x {k_sub} of {g.K} "
                                       f"output channels"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def profiled_traffic(phase, workload, layer):
    """DRAM bytes per launch of a phase's kernels from a committed ncu summary
    (a line "traffic: workload=W layer=L phase=P bytes=B source=F sha1=H" in
    profiles/*.md; workload darknet_3x3 and layer 0 when absent), or None when
    there is none or the kernel source has changed since that capture."""
    import glob
    import hashlib
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for line in open(path):
            if not line.startswith("traffic: "):
                continue
            f = dict(kv.split("=", 1) for kv in line.split()[1:])
            if (f.get("phase") != phase or f.get("workload", "darknet_3x3") != workload
                    or int(f.get("layer", 0)) != layer):
                continue
            src = os.path.join(ROOT, f["source"])
            if not os.path.exists(src):
                return None
            if hashlib.sha1(open(src, "rb").read()).hexdigest() != f["sha1"]:
                return None
            return int(f["bytes"])
    return None


def workload_layers(args, cid=None, groups=None):
    """The layer calls of workload `cid` (default: --config) as a convolution
    of `groups` groups (default: --groups); with --bn frozen, every BN layer
    gets frozen statistics (inputs.with_frozen_stats)."""
    from activation_backward_gb300 import ACT_NAMES, inputs
    cid = args.config if cid is None else cid
    groups = getattr(args, "groups", 1) if groups is None else groups
    batch = getattr(args, "batch", None)
    layers = (inputs.make_config(cid, batch=batch) if groups == 1
              else [inputs.make_grouped_config(cid, groups, batch=batch)])
    if getattr(args, "act", None):
        code = {v: k for k, v in ACT_NAMES.items()}[args.act]
        layers = [inputs.with_activation(l, code) for l in layers]
    if args.bn == "frozen":
        layers = [inputs.with_frozen_stats(l, 700 + i) if l["bn"] else l
                  for i, l in enumerate(layers)]
    if getattr(args, "layer_index", None) is not None:
        layers = [layers[args.layer_index]]
    return layers


def config_dict(args, layers, ws):
    from activation_backward_gb300 import ACT_NAMES
    g = layers[0]["geom"]
    flops = sum(2 * l["geom"].gemm_flops() // l.get("groups", 1) for l in layers)
    return {"workload": workload_name(layers),
            "N": g.N, "C": g.C, "H": g.H, "W": g.W, "K": g.K, "R": g.R, "S": g.S,
            "stride": g.stride, "pad": g.pad,
            "bn": {0: False, 1: "batch statistics", 2: "frozen statistics"}[int(layers[0]["bn"])],
            "act": ACT_NAMES[int(layers[0]["act"])],
            "z": "recomputed by the library (conv forward)" if getattr(args, "z_free", False)
                 else "given",
            "groups": int(layers[0].get("groups", 1)),
            "gemm_gflop_per_step": flops / 1e9,
            "l2": "flushed before every step, outside the timing: 512 MiB write, then a 256 MiB "
                  "read sweep so no dirty flush lines are written back inside the step",
            "launch": "the step's library calls captured into one CUDA graph, replayed; a ~1 ms "
                      "GPU spin precedes each timed step so that it is enqueued before the GPU "
                      "reaches it (the events time the GPU, not the host's launch)",
            "parallelism": "replicas only" if ws > 1 else "single GPU"}


# ------------------------------------------------------------- GPU timing

def tf32_cublas_peak(dev):
    """Dense TF32 tensor-core rate of this GPU as cuBLAS reaches it: fp32
    8192^3 matmuls with TF32 allowed, best of 10, CUDA events (2 * 8192^3
    FLOPs each).  TFLOP/s."""
    import torch
    n = 8192
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        g = torch.Generator(device=dev).manual_seed(3)
        a = torch.randn(n, n, device=dev, generator=g)
        b = torch.randn(n, n, device=dev, generator=g)
        c = torch.empty(n, n, device=dev)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = float("inf")
        for _ in range(10):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            torch.matmul(a, b, out=c)
            e.record()
            e.synchronize()
            best = min(best, s.elapsed_time(e))
        del a, b, c
        torch.cuda.empty_cache()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    return 2 * n ** 3 / (best * 1e-3) / 1e12


def tf32_peak(peaks, peak_src, measured_tf32):
    """The TF32 denominator of every GEMM fraction: the larger of the measured
    bf16 rate times the nominal tf32/bf16 ratio and the live cuBLAS TF32
    measurement (the larger one gives the smaller, conservative fraction)."""
    ratio = peaks["bf16_tflops"] * TF32_PER_BF16
    src = (f"max of {peak_src} bf16 {peaks['bf16_tflops']} x nominal tf32/bf16 1.1/2.25 "
           f"(= {ratio:.1f}) and cuBLAS TF32 fp32 8192^3 measured in this run")
    if measured_tf32 is None:
        return ratio, src.replace(" and cuBLAS TF32 fp32 8192^3 measured in this run", "")
    return max(ratio, measured_tf32), src + f" (= {measured_tf32:.1f})"


def time_workload(cid, args, dev, math, steps, warmup, stream, flush, phases=True,
                  clocks=None, ws=1, groups=None):
    """Time one workload: its library call(s) captured into a CUDA graph and
    replayed `steps` times, L2 flushed before each (outside the events); then
    (if `phases`) traced direct calls with events between the phases of every
    layer.  Returns a dict with the layers, device layers, ms per step, the
    kernels per step and the per-layer phase times."""
    import torch

    import activation_backward_gb300 as cba
    from activation_backward_gb300.layer import DeviceLayer, capture_graph

    layers = workload_layers(args, cid, groups)
    dls = [DeviceLayer(l, math=math, device=dev, z_free=args.z_free) for l in layers]

    def step(events_per_layer=None):
        n = 0
        for i, dl in enumerate(dls):
            if i > 0 and cid == 5 and len(dls) == 2:
                dl.delta.copy_(dls[0].prev)  # conv1's delta is conv2's prev_delta
            n += dl.run_traced(events_per_layer[i] if events_per_layer else None)
        return n

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    for dl in dls:
        assert dl.status() == cba.CBA_OK, "device status after warm-up"

    # The timed step: the library call(s) captured once into a CUDA graph and
    # replayed (the calls only enqueue stream-ordered work on fixed buffers, so
    # a replay is the same step without per-launch host cost).
    launches_per_step = step()
    torch.cuda.synchronize()
    graph = capture_graph(step, warmup=1)
    torch.cuda.synchronize()

    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    starts = [mk() for _ in range(steps)]
    ends = [mk() for _ in range(steps)]
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    if clocks is not None:
        clocks.start()
    torch.cuda.synchronize()
    for i in range(steps):
        flush()
        torch.cuda._sleep(SPIN_CYCLES)  # the replay is enqueued before the GPU reaches it
        starts[i].record(stream)
        graph.replay()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    clk = clocks.stop() if clocks is not None else None
    for dl in dls:
        assert dl.status() == cba.CBA_OK, "device status after the timed region"
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # what each call runs, and the bytes of its GEMM operand layout pass
    plans = [cba.cba_plan_info(dl.desc, dl.groups, dl.prev is not None) for dl in dls]
    out = dict(layers=layers, dls=dls, step_ms=step_ms, clocks=clk,
               launches_per_step=launches_per_step, phases=None, direct_ms=None,
               paths=[PATH_NAMES[p[0]] for p in plans],
               layout_bytes=[p[1] + p[2] for p in plans])
    if phases:
        nph = min(steps, 50)
        ev = [[[mk() for _ in range(cba.CBA_PHASE_EVENTS)] for _ in dls] for _ in range(nph)]
        d_starts = [mk() for _ in range(nph)]
        d_ends = [mk() for _ in range(nph)]
        for i in range(nph):
            flush()
            # a ~1 ms spin first, so that the host has enqueued the whole step
            # before the GPU reaches it: the phase events then time the
            # kernels, not the host's launch calls
            torch.cuda._sleep(SPIN_CYCLES)
            d_starts[i].record(stream)
            step(ev[i])
            d_ends[i].record(stream)
        torch.cuda.synchronize()
        out["direct_ms"] = sum(s.elapsed_time(e) for s, e in zip(d_starts, d_ends)) / nph
        per_layer = []
        for li in range(len(dls)):
            ph = {k: 0.0 for k in PHASES}
            for i in range(nph):
                e = ev[i][li]
                for j, k in enumerate(PHASES):
                    ph[k] += e[j].elapsed_time(e[j + 1])
            per_layer.append({k: v / nph for k, v in ph.items()})
        out["phases"] = per_layer
        # a plain read of the reduction's bytes, one launch per layer (torch's
        # sum over one buffer of that size, same L2 flush): what a single
        # streaming-read kernel of this size achieves on this part
        from activation_backward_gb300 import inputs
        floor = []
        for l in layers:
            buf = torch.empty(inputs.layer_bytes_reduce(l) // 4, dtype=torch.float32, device=dev)
            buf.fill_(1.0)
            tot = 0.0
            for i in range(nph + 3):
                flush()
                torch.cuda._sleep(SPIN_CYCLES)
                a, b = mk(), mk()
                a.record(stream)
                buf.sum()
                b.record(stream)
                torch.cuda.synchronize()
                if i >= 3:
                    tot += a.elapsed_time(b)
            floor.append(tot / nph)
            del buf
        out["read_floor_ms"] = floor
    return out


def summarize(t, tf32, hbm):
    """Per-workload figures from time_workload's result: the step, the phases
    summed over the layers, the GEMM and reduction fractions, and per layer."""
    from activation_backward_gb300 import inputs
    layers = t["layers"]
    flops = sum(2 * l["geom"].gemm_flops() // l.get("groups", 1) for l in layers)
    ms = sum(t["step_ms"]) / len(t["step_ms"])
    d = {"workload": workload_name(layers), "ms_per_step": ms,
         "tflops": flops / (ms * 1e-3) / 1e12, "gemm_gflop_per_step": flops / 1e9}
    if t["phases"] is None:
        return d
    red_bytes = sum(inputs.layer_bytes_reduce(l) for l in layers)
    lay_bytes = sum(t["layout_bytes"])
    tot = {k: sum(p[k] for p in t["phases"]) for k in PHASES}
    gemm_ms = tot["wgrad"] + tot["dgrad"]

    def gbs(nbytes, ms):
        return nbytes / (ms * 1e-3) / 1e9 if ms > 0 else None

    floor = sum(t["read_floor_ms"]) if t.get("read_floor_ms") else None
    d.update({"paths": t["paths"],
              "reduce_read_floor_ms": floor,
              "reduce_vs_read_floor": floor / tot["reduce"] if floor else None,
              "reduce_ms": tot["reduce"], "layout_ms": tot["layout"], "wgrad_ms": tot["wgrad"],
              "dgrad_ms": tot["dgrad"],
              "gemm_tflops": flops / (gemm_ms * 1e-3) / 1e12,
              "gemm_frac_tf32": flops / (gemm_ms * 1e-3) / 1e12 / tf32,
              "reduce_gbs": gbs(red_bytes, tot["reduce"]),
              "reduce_frac_hbm": gbs(red_bytes, tot["reduce"]) / hbm,
              "reduce_bytes": red_bytes,
              "layout_gbs": gbs(lay_bytes, tot["layout"]) if lay_bytes else None,
              "layout_frac_hbm": gbs(lay_bytes, tot["layout"]) / hbm if lay_bytes else None,
              "layout_bytes": lay_bytes, "direct_call_ms_per_step": t["direct_ms"]})
    if len(layers) > 1:
        d["layers"] = []
        for l, p, lb in zip(layers, t["phases"], t["layout_bytes"]):
            g = l["geom"]
            half = g.gemm_flops() // l.get("groups", 1)
            d["layers"].append({
                "conv": f"{g.R}x{g.S} {g.C}->{g.K}", "reduce_ms": p["reduce"],
                "layout_ms": p["layout"], "wgrad_ms": p["wgrad"], "dgrad_ms": p["dgrad"],
                "wgrad_frac_tf32": half / (p["wgrad"] * 1e-3) / 1e12 / tf32,
                "dgrad_frac_tf32": half / (p["dgrad"] * 1e-3) / 1e12 / tf32,
                "reduce_frac_hbm": gbs(inputs.layer_bytes_reduce(l), p["reduce"]) / hbm,
                "layout_frac_hbm": gbs(lb, p["layout"]) / hbm if lb else None})
    return d


def workload_name(layers):
    return "residual_block" if len(layers) == 2 else layers[0]["name"]


def run_ours(args):
    import torch
    import torch.distributed as dist

    import activation_backward_gb300 as cba

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    math = cba.CBA_MATH_TF32 if args.math == "tf32" else cba.CBA_MATH_FFMA
    cba.load()

    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_rd = flush_buf[: 256 << 20].view(torch.int32)

    def flush():
        flush_buf.zero_()
        flush_rd.max()  # read sweep: L2 ends with clean lines

    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()
    measured_tf32 = tf32_cublas_peak(dev) if ws == 1 else None
    tf32, tf32_src = tf32_peak(peaks, peak_src, measured_tf32)
    hbm = peaks["hbm_gbs"]

    t = time_workload(args.config, args, dev, math, args.steps, args.warmup, stream, flush,
                      clocks=ClockSampler(local), ws=ws)
    layers, dls = t["layers"], t["dls"]
    flops = sum(2 * l["geom"].gemm_flops() // l.get("groups", 1) for l in layers)
    total_ms = max_over_ranks(sum(t["step_ms"]), ws, dev)
    ms_per_step = total_ms / args.steps
    value = job_value(ws, flops, ms_per_step)
    launches = t["launches_per_step"] * args.steps

    # the dominant kernel phase: the (layer, GEMM) pair that takes longest
    best = None
    for li, (l, p) in enumerate(zip(layers, t["phases"])):
        for ph in ("wgrad", "dgrad"):
            if best is None or p[ph] > best[2]:
                best = (li, ph, p[ph])
    li, dom, dom_ms = best
    g = layers[li]["geom"]
    achieved = g.gemm_flops() // layers[li].get("groups", 1) / (dom_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor",
                "kernel": f"{dom} phase ({args.math}) of the {g.R}x{g.S} {g.C}->{g.K} conv",
                "achieved": achieved, "peak": tf32, "unit": "TFLOP/s",
                "frac": achieved / tf32,
                "traffic": profiled_traffic(dom, workload_name(layers), li)
                if args.math == "tf32" else None,
                "peak_source": tf32_src,
                "frac_of_bf16_ratio": achieved / (peaks["bf16_tflops"] * TF32_PER_BF16)}
    phases = summarize(t, tf32, hbm)

    per_config = None
    if (ws == 1 and not args.no_per_config and args.layer == "conv" and args.groups == 1
            and args.layer_index is None and args.batch is None):
        per_config = {}
        for cid in range(1, 6):
            if cid == args.config:
                per_config[str(cid)] = phases
                continue
            tc = time_workload(cid, args, dev, math, min(args.steps, 50), max(3, args.warmup),
                               stream, flush)
            per_config[str(cid)] = summarize(tc, tf32, hbm)
            del tc
        # config 2 as a convolution of 4 groups (one call, the same kernels)
        tc = time_workload(2, args, dev, math, min(args.steps, 50), max(3, args.warmup), stream,
                           flush, groups=4)
        per_config["2_groups4"] = summarize(tc, tf32, hbm)
        per_config["2_groups4"]["step_vs_ungrouped"] = (per_config["2_groups4"]["ms_per_step"] /
                                                        per_config["2"]["ms_per_step"])
        del tc

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(dls, layers, flops, args, stream, dev, math)

    cpu = None
    grouped = any(l.get("groups", 1) > 1 for l in layers)
    if rank == 0 and not args.no_cpu_baseline and ws == 1 and not grouped:
        cpu = cpu_baseline(layers, args.cpu_seconds)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "tf32" if math == cba.CBA_MATH_TF32 else "f32", "data": "synthetic",
            "config": config_dict(args, layers, ws),
            "roofline": roofline, "phases": phases, "per_config": per_config,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": t["clocks"],
            "tf32_cublas_tflops": measured_tf32}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def measure_e2e(dls, layers, flops, args, stream, dev, math):
    """The same metric through the public call with HOST buffers: every step
    copies the step's inputs from pinned host memory to the device, runs the
    backward and reads the results back.

    The steps are pipelined as a data loader would run them: two sets of device
    buffers, the inputs of step i + 1 copied on one stream while step i
    computes on another, the results of step i read back on a third.  Events
    keep each set's reuse in order (a set's inputs are overwritten only after
    the step that read them has finished, its outputs only after they were
    read back).  Every step's copies stay inside the timed region."""
    import torch
    from activation_backward_gb300.layer import DeviceLayer
    names_in = ("x", "output", "z", "delta", "W", "gamma", "mean", "var", "residual")
    names_out = ("dW", "db", "dgamma", "prev")
    sets = [dls, [DeviceLayer(l, math=math, device=dev, z_free=args.z_free) for l in layers]]
    hin = [{n: getattr(dl, n).cpu().pin_memory() for n in names_in
            if getattr(dl, n) is not None} for dl in dls]
    hout = [[{n: torch.empty_like(getattr(dl, n), device="cpu").pin_memory()
              for n in names_out if getattr(dl, n) is not None} for dl in dset]
            for dset in sets]
    h2d = sum(t.numel() * 4 for h in hin for t in h.values())
    d2h = sum(t.numel() * 4 for h in hout[0] for t in h.values())
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    mk = lambda: torch.cuda.Event()  # noqa: E731

    def pipeline(nsteps):
        ev_in = [mk() for _ in range(nsteps)]
        ev_done = [mk() for _ in range(nsteps)]
        ev_out = [mk() for _ in range(nsteps)]
        for i in range(nsteps):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[i - 2])  # step i - 2 has read this set's inputs
                for dl, h in zip(sets[b], hin):
                    for n, t in h.items():
                        getattr(dl, n).copy_(t, non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # this set's outputs were read back
            for dl in sets[b]:
                dl.run(stream=stream)
            ev_done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[i])
                for dl, h in zip(sets[b], hout[b]):
                    for n, t in h.items():
                        t.copy_(getattr(dl, n), non_blocking=True)
                ev_out[i].record(s_out)
        stream.wait_event(ev_out[nsteps - 1])

    steps = max(3, min(args.steps, 50))
    pipeline(3)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    s_in.wait_event(s)
    pipeline(steps)
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    return {"value": flops / (ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
            "overlap": "inputs of step i+1 copied while step i computes; two device "
                       "buffer sets, three streams"}


LAYER_WORKLOADS = {
    # LeNet pool1 geometry (20 x 24 x 24, 2 x 2 stride 2) at a batch past the L2
    "maxpool": dict(workload="lenet_pool1", N=4096, C=20, H=24, W=24, k=2, stride=2, pad=0),
    # a YOLOv3 route at 26 x 26: 128 upsampled channels + 512, batch 16
    "route": dict(workload="yolov3_route_26", batch=16, sizes=[128 * 26 * 26, 512 * 26 * 26]),
    # a YOLOv3 detection head's delta at 52 x 52: 255 channels, batch 16
    "yolo": dict(workload="yolov3_yolo_52", n=16 * 255 * 52 * 52),
}


def run_layer(args):
    """GB/s of one data-movement layer's backward: algorithmic bytes (each
    input read once, each output written once) over the device time, L2
    flushed before every step.  N = 1 only (each call is one GPU's work)."""
    import torch

    import activation_backward_gb300 as cba
    from activation_backward_gb300 import inputs
    cba.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = LAYER_WORKLOADS[args.layer]
    if args.layer == "maxpool":
        c = inputs.make_pool_case(w["N"], w["C"], w["H"], w["W"], w["k"], w["stride"], w["pad"],
                                  seed=1)
        desc = cba.make_pool_desc(w["N"], w["C"], w["H"], w["W"], w["k"], w["stride"], w["pad"])
        top, mask = torch.from_numpy(c["top_diff"]).to(dev), torch.from_numpy(c["mask"]).to(dev)
        bottom = torch.empty((w["N"], w["C"], w["H"], w["W"]), device=dev)
        nbytes = (top.numel() + mask.numel() + bottom.numel()) * 4
        call = lambda: cba.cba_maxpool_backward(desc, top, mask, bottom)  # noqa: E731
    elif args.layer == "route":
        c = inputs.make_route_case(w["batch"], w["sizes"], seed=1)
        route = torch.from_numpy(c["route_delta"]).to(dev)
        deltas = [torch.from_numpy(a).to(dev) for a in c["input_deltas"]]
        nbytes = (route.numel() + 2 * sum(d.numel() for d in deltas)) * 4
        call = lambda: cba.cba_route_backward(route, deltas)  # noqa: E731
    else:
        g = torch.Generator(device=dev).manual_seed(1)
        l_delta = torch.randn(w["n"], device=dev, generator=g)
        net = torch.randn(w["n"], device=dev, generator=g)
        nbytes = 3 * w["n"] * 4
        call = lambda: cba.cba_yolo_backward(l_delta, net)  # noqa: E731
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_rd = flush_buf[: 256 << 20].view(torch.int32)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(0)
    clocks.start()
    for a, b in ev:
        flush_buf.zero_()
        flush_rd.max()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in ev) / len(ev)
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks, src = load_peaks()
    line = {"metric": f"{args.layer} backward bandwidth", "value": gbs, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": dict({k: v for k, v in w.items()},
                           l2="flushed before every step, outside the timing"),
            "roofline": {"bound": "hbm", "kernel": f"{args.layer}_backward_kernel",
                         "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                         "peak_source": f"{src} copy bandwidth"},
            "algorithmic_bytes": nbytes, "cpu_baseline": None, "e2e": None,
            "gpu_launches": args.steps, "clocks": clk}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.layer != "conv":
        run_layer(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
