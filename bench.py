"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the whole path over one batch: fa_forward (S = QK^T,
online softmax, O = PV, L) followed by fa_backward (D = rowsum(dO o O), the
dK/dV/dQ kernel, dQ finalise), on the causal training workload
B=2, H=8, N=4096, d=64 (bf16 in, fp32 accumulate).  FLOPs follow the usual
convention: forward 4 B H N^2 d, backward 10 B H N^2 d (five products, the
recompute included), both halved under the causal mask.

Prints ONE JSON line (rank 0).  With --impl reference the same workload is
timed on the host cores with the double-precision CPU oracle instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "attention TFLOP/s (causal bf16 fwd/bwd) and % of GB300 dense BF16 peak"
STEP_WORKLOAD = "causal_train_n4096_d64"
FWD_WORKLOADS = ["causal_n4096_d64", "causal_n8192_d128", "causal_gqa_n16384_d128",
                 "causal_n8192_d96", "causal_n8192_d256", "causal_gqa_n16384_d256"]
FALLBACK_TFLOPS = 1900.0
FALLBACK_GBS = 6800.0
L2_BYTES = 129 * 10**6


# ------------------------------------------------------------------ helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_TFLOPS, FALLBACK_GBS, "fallback"


# The source file of each kernel named in profiles/traffic.txt.
KERNEL_SOURCES = {"fa_bwd64_kernel": "fa_bwd_d64.cu", "fa_fwd_kernel": "fa_fwd.cu",
                  "fa_fwd1_kernel": "fa_fwd_tile1.cu", "fa_bwd_kernel": "fa_bwd.cu",
                  "fa_bwd_dq_kernel": "fa_bwd_dq.cu", "fa_bwd256_kv_kernel": "fa_bwd_d256.cu"}


def kernel_traffic(kernel):
    """Bytes per launch from the committed ncu summary, if the kernel's source
    is unchanged since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src_hash = source_hash(kernel)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel:
            if parts[3] == src_hash:
                return float(parts[2])
    return None


def workload_traffic(workload):
    """{kernel: DRAM bytes per launch} for every kernel of a workload named in
    the committed ncu summary whose source is unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    out = {}
    if not os.path.exists(path):
        return out
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[1] == workload:
            if parts[3] == source_hash(parts[0]):
                out[parts[0]] = int(parts[2])
    return out


def source_hash(kernel):
    """Hash of the kernel's own source file and the headers it includes."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_27_gb300", "csrc")
    base = kernel.split("<")[0]
    for f in (KERNEL_SOURCES[base], "fa_ptx.cuh", "fa_internal.h"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.15)
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


# ------------------------------------------------------------------ our arm

def _rotation(bytes_per_set):
    """Number of input sets to cycle through so that a step's inputs were
    evicted from the 129 MB L2 by the steps before it (at least 3x L2)."""
    return max(1, math.ceil(3 * L2_BYTES / bytes_per_set))


def step_set_bytes(w):
    """Device bytes of one step's buffers: q, k, v, dO in; o, L, dq, dk, dv out."""
    q = w.B * w.Hq * w.N * w.d * 2    # q, dO, o, dq
    kv = w.B * w.Hkv * w.N * w.d * 2  # k, v, dk, dv
    return 4 * q + 4 * kv + w.B * w.Hq * w.N * 4


def bench_config(w, world):
    """The benchmark configuration, the same dict in both arms' lines: the
    workload, how it runs across GPUs, and how the device arm keeps a step's
    inputs out of L2 (the reference arm runs on the host and times the
    same workload)."""
    set_bytes = step_set_bytes(w)
    return {"workload": w.describe(), "B": w.B, "H_q": w.Hq, "H_kv": w.Hkv, "N": w.N,
            "d": w.d, "causal": True,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": f"inputs larger than L2: {_rotation(set_bytes)} rotating input sets of "
                  f"{set_bytes / 2**20:.0f} MiB, steps back to back"}


def run_ours(args, rank, world):
    import torch
    import exact_attention_27_gb300 as fa
    from exact_attention_27_gb300 import _build

    dev = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev)
    if rank == 0 or not os.path.exists(_build.LIB_PATH):
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    w = WORKLOADS[STEP_WORKLOAD]
    stream = torch.cuda.current_stream()
    inp = make_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, seed=rank * 100, with_grad=True)
    base = {n: inp[n].cuda() for n in ("q", "k", "v", "do")}

    def new_set():
        t = {n: x.clone() for n, x in base.items()}
        t["o"] = torch.empty_like(t["q"])
        t["lse"] = torch.empty(t["q"].shape[:-1], dtype=torch.float32, device="cuda")
        t["dq"], t["dk"], t["dv"] = (torch.empty_like(t["q"]), torch.empty_like(t["k"]),
                                     torch.empty_like(t["v"]))
        return t

    first = new_set()
    set_bytes = sum(x.numel() * x.element_size() for x in first.values())
    assert set_bytes == step_set_bytes(w)
    R = _rotation(set_bytes)
    sets = [first] + [new_set() for _ in range(R - 1)]
    flops_fwd, flops_bwd = w.fwd_flops(), w.bwd_flops()

    # An event recorded between two kernels stops the second from being
    # scheduled while the first finishes (each kernel here is launched as a
    # programmatic dependent of the one before), so per-kernel events go on
    # every EVENT_EVERY-th timed step only: before and after the forward and
    # around the backward main kernel.  The other steps run unobserved.
    EVENT_EVERY = 10

    def step(t, ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fa_forward(t["q"], t["k"], t["v"], t["o"], t["lse"], w.scale, True)
        if ev is not None:
            ev[1].record(stream)
        fa.fa_set_backward_events(ev[2] if ev else None, ev[3] if ev else None)
        fa.fa_backward(t["q"], t["k"], t["v"], t["o"], t["lse"], t["do"], t["dq"], t["dk"],
                       t["dv"], w.scale, True)

    for i in range(args.warmup):
        step(sets[i % R])
    torch.cuda.synchronize()
    if fa.fa_last_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    K = args.steps
    n_obs = (K + EVENT_EVERY - 1) // EVENT_EVERY  # observed steps: 0, 10, 20, ...
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_obs)]
    for e in ev:  # create the events (torch creates them on first record)
        for x in e:
            x.record(stream)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clocks:
        t_wall = time.perf_counter()
        t_start.record(stream)
        for i in range(K):
            obs = ev[i // EVENT_EVERY] if i % EVENT_EVERY == 0 else None
            step(sets[(args.warmup + i) % R], obs)
        t_end.record(stream)
        fa.fa_set_backward_events(None, None)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    if fa.fa_last_device_error() != 0:
        raise RuntimeError("device error during the timed steps")
    total_ms = t_start.elapsed_time(t_end)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_main_ms = [e[2].elapsed_time(e[3]) for e in ev]
    # per-step time over blocks of EVENT_EVERY steps (one observed step each)
    step_ms = [ev[j][0].elapsed_time(ev[j + 1][0]) / EVENT_EVERY for j in range(n_obs - 1)]
    step_ms.append(ev[n_obs - 1][0].elapsed_time(t_end) / (K - (n_obs - 1) * EVENT_EVERY))
    if world > 1:
        t = torch.tensor([total_ms], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / K
    value = world * (flops_fwd + flops_bwd) * K / (total_ms * 1e-3) / 1e12

    tflops_peak, hbm_peak, peak_src = peaks()
    fwd_avg = statistics.mean(fwd_ms)
    bwd_main_avg = statistics.mean(bwd_main_ms)
    if bwd_main_avg >= fwd_avg:
        kname, kflops, kms = "fa_bwd64_kernel<causal>", flops_bwd, bwd_main_avg
    else:
        kname, kflops, kms = "fa_fwd_kernel<64,causal>", flops_fwd, fwd_avg
    achieved = kflops / (kms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": kname, "achieved": round(achieved, 1),
                "peak": tflops_peak, "unit": "TFLOP/s", "frac": round(achieved / tflops_peak, 4),
                "peak_source": f"{peak_src} bf16 burst", "traffic": kernel_traffic(kname)}

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": bench_config(w, world),
        "step": "fa_forward + fa_backward",
        "frac_of_peak": round(value / world / tflops_peak, 4),
        "fwd_ms": round(fwd_avg, 5),
        "bwd_ms": round(ms_per_step - fwd_avg, 5),
        "bwd_main_kernel_ms": round(bwd_main_avg, 5),
        "per_step_ms": {"step": _med_min(step_ms), "fwd": _med_min(fwd_ms),
                        "bwd_main_kernel": _med_min(bwd_main_ms),
                        "events": f"forward and backward main kernel timed on every "
                                  f"{EVENT_EVERY}th step ({n_obs} steps); step over "
                                  f"{EVENT_EVERY}-step blocks"},
        "roofline": roofline,
        "gpu_launches": 4 * K,
        "wall_s_timed_region": round(t_wall, 4),
    }
    gpu_out = None
    if rank == 0 and not args.only_step:
        result["graph"] = graph_steps(fa, torch, step, sets, flops_fwd + flops_bwd)
        if world == 1:  # rank 0's inputs are the oracle sample's (seed 0)
            torch.cuda.synchronize()
            gpu_out = {n: first[n].double().cpu().numpy() for n in ("o", "lse", "dq", "dk", "dv")}
    del sets, first, base
    torch.cuda.empty_cache()
    if rank == 0:
        result["clocks"] = clocks.summary()
        if not args.only_step:
            result["fwd_workloads"] = forward_workloads(fa, torch, tflops_peak, peak_src)
            result["fwd_workloads"].append(forward_fp8_workload(fa, torch, tflops_peak, peak_src))
            result["bwd_workloads"] = backward_workloads(fa, torch, tflops_peak, peak_src)
            result["preprocess"] = [preprocess_workload(fa, torch, w, hbm_peak, peak_src),
                                    preprocess_workload(fa, torch, WORKLOADS["causal_n8192_d128"],
                                                        hbm_peak, peak_src)]
            result["e2e"] = end_to_end(fa, torch, w, min(K, 50))
            if world == 1:
                result["cpu_baseline"] = cpu_baseline(w, gpu_out)
            result["summary"] = summary(result)
    return result


def summary(result):
    """The per-workload results in a few hundred characters, printed as the
    last key of the line so that a reader that keeps only the end of the
    output still sees them: [workload, ms, TFLOP/s, fraction of peak]."""
    rows = [["step: " + result["config"]["workload"], result["ms_per_step"], result["value"],
             result["frac_of_peak"]],
            ["bwd main kernel (roofline)", result["bwd_main_kernel_ms"],
             result["roofline"]["achieved"], result["roofline"]["frac"]]]
    for key in ("fwd_workloads", "bwd_workloads"):
        for x in result.get(key, []):
            name = x["workload"].replace(" bf16", "").replace("e4m3 (O bf16)", "fp8")
            rows.append([name, x["ms"], x["tflops"], x["frac"]])
    return {"columns": ["workload", "ms", "TFLOP/s", "frac of measured peak"], "rows": rows}


def _med_min(xs):
    return {"median": round(statistics.median(xs), 5), "min": round(min(xs), 5)}


def per_launch_ms(torch, launch, reps=10):
    """Median and min of `reps` launches, each bracketed by its own events
    (which also keeps it from overlapping its neighbours)."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for i in range(reps):
        ev[i][0].record()
        launch(i)
        ev[i][1].record()
    torch.cuda.synchronize()
    return _med_min([a.elapsed_time(b) for a, b in ev])


def graph_launches(torch, launch, n=100, replays=5):
    """`n` launches captured into one CUDA graph and replayed: ms per launch."""
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            launch(0)
            side.synchronize()
            with torch.cuda.graph(g, stream=side):
                for i in range(n):
                    launch(i)
        torch.cuda.current_stream().wait_stream(side)
        g.replay()
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s_ev.record()
        for _ in range(replays):
            g.replay()
        e_ev.record()
        torch.cuda.synchronize()
        ms = s_ev.elapsed_time(e_ev) / (replays * n)
        del g
        return {"launches_per_graph": n, "ms": round(ms, 5)}
    except Exception as exc:  # reported, not fatal
        return {"error": f"{type(exc).__name__}: {exc}"[:200]}


def graph_steps(fa, torch, step, sets, flops, n=100, replays=5):
    """The benchmark step captured n times into one CUDA graph (cycling
    through the same rotating input sets) and replayed: device time per step
    with no host launch overhead between kernels."""
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step(sets[0])
            side.synchronize()
            with torch.cuda.graph(g, stream=side):
                for i in range(n):
                    step(sets[i % len(sets)])
        torch.cuda.current_stream().wait_stream(side)
        g.replay()
        g.replay()
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s_ev.record()
        for _ in range(replays):
            g.replay()
        e_ev.record()
        torch.cuda.synchronize()
        if fa.fa_last_device_error() != 0:
            raise RuntimeError("device error during the graph replays")
        ms = s_ev.elapsed_time(e_ev) / (replays * n)
        del g
        return {"steps_per_graph": n, "replays": replays, "ms_per_step": round(ms, 5),
                "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s"}
    except Exception as exc:  # reported, not fatal: the eager numbers stand
        return {"error": f"{type(exc).__name__}: {exc}"[:200]}


def run_backward_only(args):
    """fa_backward (or the deterministic one) alone on one backward workload,
    after one forward for O and L (used for kernel profiles).  Its time (one
    input set, calls back to back, part of it left in L2) is for orientation
    only; the benchmark line's `bwd_workloads` are the measured figures."""
    import torch
    import exact_attention_27_gb300 as fa
    from exact_attention_27_gb300 import _build
    _build.build()
    name, (B, Hq, Hkv, N, d), det = BWD_WORKLOADS[BWD_NAMES[args.backward_only]]
    inp = make_inputs(B, Hq, Hkv, N, d, seed=11, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_forward(q, k, v, causal=True, scale=scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    call = fa.fa_backward_deterministic if det else fa.fa_backward
    for _ in range(args.warmup):
        call(q, k, v, o, lse, do, dq, dk, dv, scale, True)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.steps):
        call(q, k, v, o, lse, do, dq, dk, dv, scale, True)
    e.record()
    torch.cuda.synchronize()
    if fa.fa_last_device_error() != 0:
        raise RuntimeError("device error")
    ms = s.elapsed_time(e) / args.steps
    return {"workload": name, "launches": args.warmup + args.steps, "ms": round(ms, 4),
            "tflops": round(10.0 * B * Hq * N * N * d / 2 / (ms * 1e-3) / 1e12, 1)}


def run_forward_only(args):
    """fa_forward alone on one workload (used for kernel profiles)."""
    import torch
    import exact_attention_27_gb300 as fa
    from exact_attention_27_gb300 import _build
    _build.build()
    w = WORKLOADS[args.forward_only]
    inp = make_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, seed=7)
    if args.fp8:  # the e4m3 forward on the same shape (d = 128), unit descales
        if w.d != 128:
            raise SystemExit("--fp8 needs a d = 128 workload")
        q = inp["q"].to(torch.float8_e4m3fn).cuda()
        k = inp["k"].to(torch.float8_e4m3fn).cuda()
        v = inp["v"].to(torch.float8_e4m3fn).transpose(-1, -2).contiguous().cuda()
        o = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")

        def launch():
            fa.fa_forward_fp8(q, k, v, o, lse, w.scale, w.causal)
    else:
        q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
        o = torch.empty_like(q)

        def launch():
            fa.fa_forward(q, k, v, o, lse, w.scale, w.causal)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
    for _ in range(args.warmup):
        launch()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.steps):
        launch()
    e.record()
    torch.cuda.synchronize()
    if fa.fa_last_device_error() != 0:
        raise RuntimeError("device error")
    ms = s.elapsed_time(e) / args.steps
    return {"workload": w.describe() + (" e4m3" if args.fp8 else ""),
            "launches": args.warmup + args.steps, "ms": round(ms, 4),
            "tflops": round(w.fwd_flops() / (ms * 1e-3) / 1e12, 1)}


TILE_SWEEP_SHAPES = (
    # (B, H_q, H_kv, N): the shapes the per-shape tile choice was fitted on ...
    [(1, h, h, n) for h in (2, 4, 8, 16, 32, 64) for n in (1024, 2048, 4096, 8192)
     if h * n <= 64 * 8192]
    # ... and shapes held out of the fit (other head counts, GQA, other N).
    + [(b, h, g, n) for (b, h, g) in ((1, 12, 12), (1, 24, 24), (1, 48, 48), (2, 20, 20),
                                       (1, 32, 8), (1, 40, 5)) for n in (1536, 3072, 6144)])


def run_tile_rows_sweep(args):
    """fa_forward at 128 and 256 query rows per CTA and at the per-shape
    choice, on every shape of TILE_SWEEP_SHAPES, d = 64, 96 and 128, causal and
    not: one JSON line per shape, then the time the choice lost against the
    faster size, summed over the shapes.  Each size runs as 20 launches
    captured in one CUDA graph and replayed 5 times, timed with CUDA events,
    so that small shapes measure the kernels rather than the host calls."""
    import torch
    import exact_attention_27_gb300 as fa
    from exact_attention_27_gb300 import _build
    _build.build()
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def timed(f):
        r = graph_launches(torch, lambda i: f(), n=20, replays=5)
        if "ms" not in r:
            raise RuntimeError(r["error"])
        return r["ms"]

    lost, n_shapes = 0.0, 0
    try:
        for d in (64, 96, 128):
            for causal in (True, False):
                for B, Hq, Hkv, N in TILE_SWEEP_SHAPES:
                    inp = make_inputs(B, Hq, Hkv, N, d, seed=1)
                    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
                    o = torch.empty_like(q)
                    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
                    ms = {}
                    for rows in (128, 256, 0):
                        fa.fa_set_forward_tile_rows(rows)
                        ms[rows] = timed(lambda: fa.fa_forward(q, k, v, o, lse, d ** -0.5, causal))
                    fa.fa_set_forward_tile_rows(0)
                    pick = fa.fa_forward_tile_rows_for(B, Hq, Hkv, N, N, d, causal, 0, sms)
                    best = min(ms[128], ms[256])
                    lost += ms[pick] / best - 1.0
                    n_shapes += 1
                    print(json.dumps({"d": d, "causal": causal, "B": B, "H_q": Hq, "H_kv": Hkv,
                                      "N": N, "ms_128": round(ms[128], 4),
                                      "ms_256": round(ms[256], 4), "ms_chosen": round(ms[0], 4),
                                      "chosen": pick}), flush=True)
                    del q, k, v, o, lse, inp
        if fa.fa_last_device_error() != 0:
            raise RuntimeError("device error")
    finally:
        fa.fa_set_forward_tile_rows(0)
    return {"sweep": "forward tile rows", "shapes": n_shapes, "sms": sms,
            "summed_loss_vs_faster": round(lost, 3)}


def preprocess_workload(fa, torch, w, hbm_peak, peak_src):
    """The row-dot pass D = rowsum(dO o O) (fa_backward_preprocess) alone on
    the step's shapes: memory-bound, reported in GB/s against the copy
    bandwidth.  Algorithmic bytes: O and dO read once, D written.  Each launch
    reads a different input set, enough sets that together they exceed L2 by
    3x, so every launch reads from HBM; per-launch CUDA events."""
    rows = w.B * w.Hq * w.N
    nbytes = 2 * rows * w.d * 2 + rows * 4
    nset = _rotation(2 * rows * w.d * 2)
    gen = torch.Generator(device="cuda").manual_seed(5)
    sets = []
    for _ in range(nset):
        o = torch.randn(w.B, w.Hq, w.N, w.d, device="cuda", generator=gen).to(torch.bfloat16)
        do = torch.randn(w.B, w.Hq, w.N, w.d, device="cuda", generator=gen).to(torch.bfloat16)
        D = torch.empty(w.B, w.Hq, w.N, device="cuda", dtype=torch.float32)
        sets.append((o, do, D))
    for i in range(3):
        fa.fa_backward_preprocess(*sets[i % nset])
    t = per_launch_ms(torch, lambda i: fa.fa_backward_preprocess(*sets[i % nset]),
                      reps=max(20, nset))
    gbs = nbytes / (t["median"] * 1e-3) / 1e9
    del sets
    return {"kernel": "preprocess_kernel<%d>" % w.d, "workload": w.describe(),
            "bytes_per_launch": nbytes, "input_sets": nset, "per_launch_ms": t,
            "achieved_gbs": round(gbs, 1), "peak_gbs": hbm_peak, "frac": round(gbs / hbm_peak, 4),
            "peak_source": f"{peak_src} copy"}


def forward_workloads(fa, torch, tflops_peak, peak_src):
    """Forward-only throughput on the larger workloads: back-to-back launches,
    cycling through enough input sets that each launch's inputs come from HBM."""
    out = []
    for name in FWD_WORKLOADS:
        w = WORKLOADS[name]
        inp = make_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, seed=7)
        per_set = sum(t.numel() * t.element_size() for t in inp.values()) * 4 // 3
        R = _rotation(per_set)
        sets = []
        for _ in range(R):
            t = {n: x.cuda() for n, x in inp.items()}
            t["o"] = torch.empty_like(t["q"])
            t["lse"] = torch.empty(t["q"].shape[:-1], dtype=torch.float32, device="cuda")
            sets.append(t)
        for i in range(3):
            t = sets[i % R]
            fa.fa_forward(t["q"], t["k"], t["v"], t["o"], t["lse"], w.scale, w.causal)
        reps = 30
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s_ev.record()
        for i in range(reps):
            t = sets[i % R]
            fa.fa_forward(t["q"], t["k"], t["v"], t["o"], t["lse"], w.scale, w.causal)
        e_ev.record()
        torch.cuda.synchronize()
        ms = s_ev.elapsed_time(e_ev) / reps

        def launch(i, sets=sets, w=w, R=R):
            t = sets[i % R]
            fa.fa_forward(t["q"], t["k"], t["v"], t["o"], t["lse"], w.scale, w.causal)

        tf = w.fwd_flops() / (ms * 1e-3) / 1e12
        line = {"workload": w.describe(), "ms": round(ms, 4), "tflops": round(tf, 1),
                "frac": round(tf / tflops_peak, 4), "peak": f"{peak_src} bf16 burst",
                "input_sets": R, "per_launch_ms": per_launch_ms(torch, launch),
                "dram_bytes_per_launch": workload_traffic(name) or None}
        if name == GRAPH_FWD_WORKLOAD:
            line["graph"] = graph_launches(torch, launch)
        out.append(line)
        del sets, inp
        torch.cuda.empty_cache()
    return out


# The forward workload also timed as a 100-launch CUDA graph.
GRAPH_FWD_WORKLOAD = "causal_n4096_d64"


# Backward beside the benchmark step: the d = 128 and d = 96 kernel on the
# causal d = 128 shape's heads (B2 H16 N4096), and the deterministic
# two-kernel backward on the training shape.
BWD_WORKLOADS = [
    ("causal bwd B2 H16 N4096 d128 bf16", (2, 16, 16, 4096, 128), False),
    ("causal bwd B2 H16 N4096 d96 bf16", (2, 16, 16, 4096, 96), False),
    ("causal bwd B2 H16 N4096 d256 bf16", (2, 16, 16, 4096, 256), False),
    ("causal bwd B2 H8 N4096 d64 bf16, deterministic", (2, 8, 8, 4096, 64), True),
]
# Short names for --backward-only.
BWD_NAMES = {"causal_bwd_n4096_d128": 0, "causal_bwd_n4096_d96": 1,
             "causal_bwd_n4096_d256": 2, "causal_bwd_det_n4096_d64": 3}


def backward_workloads(fa, torch, tflops_peak, peak_src):
    """fa_backward (or fa_backward_deterministic) alone, inputs resident,
    back-to-back calls; FLOPs 10 B H N^2 d / 2 (causal)."""
    out = []
    short = {i: n for n, i in BWD_NAMES.items()}
    for idx, (name, (B, Hq, Hkv, N, d), det) in enumerate(BWD_WORKLOADS):
        inp = make_inputs(B, Hq, Hkv, N, d, seed=11, with_grad=True)
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
        scale = 1.0 / math.sqrt(d)
        o, lse = fa.attention_forward(q, k, v, causal=True, scale=scale)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        call = fa.fa_backward_deterministic if det else fa.fa_backward
        for _ in range(3):
            call(q, k, v, o, lse, do, dq, dk, dv, scale, True)
        reps = 20
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s_ev.record()
        for _ in range(reps):
            call(q, k, v, o, lse, do, dq, dk, dv, scale, True)
        e_ev.record()
        torch.cuda.synchronize()
        ms = s_ev.elapsed_time(e_ev) / reps
        tf = 10.0 * B * Hq * N * N * d / 2 / (ms * 1e-3) / 1e12
        pl = per_launch_ms(torch, lambda i: call(q, k, v, o, lse, do, dq, dk, dv, scale, True))
        out.append({"workload": name, "ms": round(ms, 4), "tflops": round(tf, 1),
                    "frac": round(tf / tflops_peak, 4), "peak": f"{peak_src} bf16 burst",
                    "per_launch_ms": pl, "dram_bytes_per_launch": workload_traffic(short[idx]) or None})
        del q, k, v, do, o, lse, dq, dk, dv
        torch.cuda.empty_cache()
    return out


def forward_fp8_workload(fa, torch, tflops_peak, peak_src):
    """The FP8 forward (e4m3 Q, K, V^T; unit descales) on the shape of the
    causal d = 128 workload, against twice the measured bf16 peak (the
    nominal FP8 : bf16 dense tensor ratio)."""
    w = WORKLOADS["causal_n8192_d128"]
    inp = make_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, seed=7)
    q = inp["q"].to(torch.float8_e4m3fn).cuda()
    k = inp["k"].to(torch.float8_e4m3fn).cuda()
    vt = inp["v"].to(torch.float8_e4m3fn).transpose(-1, -2).contiguous().cuda()
    o = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
    for _ in range(3):
        fa.fa_forward_fp8(q, k, vt, o, lse, w.scale, w.causal)
    reps = 20
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s_ev.record()
    for _ in range(reps):
        fa.fa_forward_fp8(q, k, vt, o, lse, w.scale, w.causal)
    e_ev.record()
    torch.cuda.synchronize()
    ms = s_ev.elapsed_time(e_ev) / reps
    tf = w.fwd_flops() / (ms * 1e-3) / 1e12
    peak = 2.0 * tflops_peak
    pl = per_launch_ms(torch, lambda i: fa.fa_forward_fp8(q, k, vt, o, lse, w.scale, w.causal))
    out = {"workload": w.describe().replace("bf16", "e4m3 (O bf16)"), "dtype": "e4m3",
           "ms": round(ms, 4), "tflops": round(tf, 1), "frac": round(tf / peak, 4),
           "peak": f"2 x {peak_src} bf16 burst (nominal fp8/bf16 ratio)",
           "input_sets": 1, "per_launch_ms": pl}
    del q, k, vt, o, lse
    torch.cuda.empty_cache()
    return out


def end_to_end(fa, torch, w, K):
    """Same step through the public API with the inputs in pinned host memory:
    every step copies its q, k, v, dO host->device and reads its o, lse, dq,
    dk, dv back device->host, all inside the timed region.  The inputs sit
    in one pinned host buffer and the outputs in one device buffer (views of
    each), so a step makes one copy in each direction.  The loop is
    pipelined as a training or serving loop would be: three sets of device
    buffers and three streams, so that step i+1's inputs go up and step
    i-1's results come down while step i computes (each copy waits only for
    the step that last used its buffers)."""
    inp = make_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, seed=1, with_grad=True)
    names = ("q", "k", "v", "do")

    def carve(buf, specs):
        """Views of a flat byte buffer: (name, shape, dtype) in order."""
        out, off = {}, 0
        for n, shape, dt in specs:
            nb = math.prod(shape) * torch.tensor([], dtype=dt).element_size()
            out[n] = buf[off:off + nb].view(dt).view(shape)
            off += nb
        return out

    in_specs = [(n, tuple(inp[n].shape), inp[n].dtype) for n in names]
    q_shape, kv_shape = tuple(inp["q"].shape), tuple(inp["k"].shape)
    out_specs = [("o", q_shape, torch.bfloat16), ("dq", q_shape, torch.bfloat16),
                 ("dk", kv_shape, torch.bfloat16), ("dv", kv_shape, torch.bfloat16),
                 ("lse", q_shape[:-1], torch.float32)]
    nb_in = sum(math.prod(sh) * 2 for _, sh, _ in in_specs)
    nb_out = sum(math.prod(sh) * (4 if dt == torch.float32 else 2) for _, sh, dt in out_specs)
    h_in = torch.empty(nb_in, dtype=torch.uint8).pin_memory()
    hv = carve(h_in, in_specs)
    for n in names:
        hv[n].copy_(inp[n])

    def buffers():
        d_in = torch.empty(nb_in, dtype=torch.uint8, device="cuda")
        d_out = torch.empty(nb_out, dtype=torch.uint8, device="cuda")
        return {"d_in": d_in, "d_out": d_out, "i": carve(d_in, in_specs),
                "o": carve(d_out, out_specs),
                "h_out": torch.empty(nb_out, dtype=torch.uint8).pin_memory(),
                "ev": {k: torch.cuda.Event() for k in ("in", "cmp", "out")}}

    NSET = 3
    sets = [buffers() for _ in range(NSET)]
    s_cmp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def step(i):
        S = sets[i % NSET]
        d, o, ev = S["i"], S["o"], S["ev"]
        with torch.cuda.stream(s_in):
            if i >= NSET:
                s_in.wait_event(ev["cmp"])  # step i-NSET is done with these inputs
            S["d_in"].copy_(h_in, non_blocking=True)
            ev["in"].record(s_in)
        s_cmp.wait_event(ev["in"])
        if i >= NSET:
            s_cmp.wait_event(ev["out"])  # step i-NSET's results have been read
        fa.fa_forward(d["q"], d["k"], d["v"], o["o"], o["lse"], w.scale, True)
        fa.fa_backward(d["q"], d["k"], d["v"], o["o"], o["lse"], d["do"], o["dq"], o["dk"],
                       o["dv"], w.scale, True)
        ev["cmp"].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["cmp"])
            S["h_out"].copy_(S["d_out"], non_blocking=True)
            ev["out"].record(s_out)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    t_host = time.perf_counter()
    for i in range(K):
        step(i)
    t_host = time.perf_counter() - t_host
    stop.record(s_out)
    stop.synchronize()  # the host holds every step's results
    torch.cuda.synchronize()
    ms = start.elapsed_time(stop) / K
    return {"value": round((w.fwd_flops() + w.bwd_flops()) / (ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "ms_per_step": round(ms, 4), "h2d_bytes_per_step": nb_in,
            "d2h_bytes_per_step": nb_out, "host_enqueue_ms_per_step": round(t_host * 1e3 / K, 4),
            "pipelined": f"{NSET} buffer sets, 3 streams, one copy each way per step"}


# ------------------------------------------------------------------ oracle arms

def oracle_sample(w, q_block, step_index, keep=None):
    """Oracle forward + backward for one block of `q_block` query rows in every
    head of the workload (full keys, causal), and the algorithmic FLOPs of the
    rows processed.  Rows rotate through the sequence from step to step,
    starting with the last block.  If `keep` is a list, the block's first row
    and the oracle's outputs are appended to it."""
    import oracle

    inp = _oracle_inputs(w)
    nblk = w.N // q_block
    r0 = ((nblk - 1 + step_index * 7919) % nblk) * q_block
    q = inp["q"][:, :, r0:r0 + q_block]
    do = inp["do"][:, :, r0:r0 + q_block]
    t0 = time.perf_counter()
    fwd = oracle.attention_forward(q, inp["k"], inp["v"], w.scale, True, q_offset=r0)
    bwd = oracle.attention_backward(q, inp["k"], inp["v"], do, w.scale, True, q_offset=r0)
    dt = time.perf_counter() - t0
    if keep is not None:
        keep.append((r0, fwd, bwd))
    keys_seen = sum(i + 1 for i in range(r0, r0 + q_block))  # per head
    heads = w.B * w.Hq
    flops = heads * keys_seen * w.d * (4 + 10)
    return flops, dt


# Tolerances of the comparison against the oracle (bf16 inputs, fp32
# accumulation): O max and mean absolute error, L max absolute error, and
# each gradient's max absolute error relative to its largest reference value.
TOL = {"o_max_abs": 2e-2, "o_mean_abs": 2e-3, "lse_max_abs": 1e-3, "grad_rel": 5e-2}


def sampled_errors(w, samples, gpu, q_block):
    """Errors of the GPU outputs `gpu` (o, lse, dq, dk, dv as float arrays)
    on the oracle's sampled blocks.  Under the causal mask the last block's
    keys are seen only by that block's queries, so its dK and dV rows are
    complete and are compared too."""
    import numpy as np
    o_err, o_sum, o_n, l_err = 0.0, 0.0, 0, 0.0
    g_err = {"dq": 0.0, "dk": 0.0, "dv": 0.0}
    g_ref = {"dq": 0.0, "dk": 0.0, "dv": 0.0}
    for r0, (o_ref, l_ref), (dq_ref, dk_ref, dv_ref) in samples:
        rows = slice(r0, r0 + q_block)
        e = np.abs(gpu["o"][:, :, rows] - o_ref)
        o_err, o_sum, o_n = max(o_err, e.max()), o_sum + e.sum(), o_n + e.size
        l_err = max(l_err, np.abs(gpu["lse"][:, :, rows] - l_ref).max())
        pairs = [("dq", gpu["dq"][:, :, rows], dq_ref)]
        if r0 + q_block == w.N:
            pairs += [("dk", gpu["dk"][:, :, rows], dk_ref[:, :, rows]),
                      ("dv", gpu["dv"][:, :, rows], dv_ref[:, :, rows])]
        for n, g, r in pairs:
            g_err[n] = max(g_err[n], np.abs(g - r).max())
            g_ref[n] = max(g_ref[n], np.abs(r).max())
    out = {"o_max_abs": float(o_err), "o_mean_abs": float(o_sum / max(o_n, 1)),
           "lse_max_abs": float(l_err)}
    for n in g_err:
        out[f"{n}_rel"] = float(g_err[n] / g_ref[n]) if g_ref[n] > 0 else None
    ok = (out["o_max_abs"] <= TOL["o_max_abs"] and out["o_mean_abs"] <= TOL["o_mean_abs"]
          and out["lse_max_abs"] <= TOL["lse_max_abs"]
          and all(out[f"{n}_rel"] is None or out[f"{n}_rel"] <= TOL["grad_rel"] for n in g_err))
    out = {k: (round(v, 7) if isinstance(v, float) else v) for k, v in out.items()}
    out["rows"] = (f"{len(samples)} blocks of {q_block} query rows x {w.B * w.Hq} heads "
                   f"(dq, o, lse); dk, dv: the last {q_block} keys")
    out["tolerance"] = TOL
    out["within_tolerance"] = bool(ok)
    return out


_INPUT_CACHE = {}


def _oracle_inputs(w):
    if w.name not in _INPUT_CACHE:
        from workloads import as_f64
        inp = make_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, seed=0, with_grad=True)
        _INPUT_CACHE[w.name] = {n: as_f64(t) for n, t in inp.items()}
    return _INPUT_CACHE[w.name]


def cpu_baseline(w, gpu=None):
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload: forward + backward of 256-row query blocks in all 16 heads.
    With the GPU's outputs for the same inputs (`gpu`), the errors on the
    sampled rows are reported beside the timing."""
    import oracle
    q_block, flops, secs, steps = 256, 0.0, 0.0, 0
    samples = [] if gpu is not None else None
    while secs < 10.0 and steps < 64:
        f, dt = oracle_sample(w, q_block, steps, samples)
        flops += f
        secs += dt
        steps += 1
    out = {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s",
           "cores": min(oracle.num_threads(), w.B * w.Hq), "kind": "oracle",
           "sample": f"{steps} blocks of {q_block} query rows x {w.B * w.Hq} heads, "
                     f"fwd+bwd against all {w.N} keys (causal), {secs:.1f} s"}
    if gpu is not None:
        out["gpu_errors_on_sample"] = sampled_errors(w, samples, gpu, q_block)
    return out


def run_reference(args, rank, world):
    """The double-precision CPU oracle timed on the host cores, on the same
    workload, metric and unit; each step a bounded sample of query rows."""
    import oracle
    w = WORKLOADS[STEP_WORKLOAD]
    oracle.load()
    # size the per-step sample so that warm-up + steps stay within ~2 minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    q_block = 256
    f, dt = oracle_sample(w, q_block, 0)
    while dt > budget and q_block > 16:
        q_block //= 2
        f, dt = oracle_sample(w, q_block, 0)
    for i in range(args.warmup):
        oracle_sample(w, q_block, i + 1)
    flops, secs = 0.0, 0.0
    for i in range(args.steps):
        f, dt = oracle_sample(w, q_block, args.warmup + 1 + i)
        flops += f
        secs += dt
    value = flops / secs / 1e12
    sample = (f"per step: {q_block} query rows x {w.B * w.Hq} heads, fwd+bwd against all "
              f"{w.N} keys (causal)")
    cores = min(oracle.num_threads(), w.B * w.Hq)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, world),
        "step": "oracle forward + backward",
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only-step", action="store_true",
                    help="time the step only (no extra workloads, e2e or CPU baseline)")
    ap.add_argument("--forward-only", choices=sorted(WORKLOADS), default=None,
                    help="run fa_forward alone on one workload (for kernel profiles)")
    ap.add_argument("--fp8", action="store_true",
                    help="with --forward-only: the e4m3 forward (d = 128 workloads)")
    ap.add_argument("--backward-only", choices=sorted(BWD_NAMES), default=None,
                    help="run fa_backward alone on one backward workload (for kernel profiles)")
    ap.add_argument("--sweep-tile-rows", action="store_true",
                    help="time both forward tile sizes and the per-shape choice on a shape grid")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus != world and world > 1:
        ap.error("--gpus must match the launcher's WORLD_SIZE")
    if args.forward_only:
        print(json.dumps(run_forward_only(args)), flush=True)
        return
    if args.backward_only:
        print(json.dumps(run_backward_only(args)), flush=True)
        return
    if args.sweep_tile_rows:
        print(json.dumps(run_tile_rows_sweep(args)), flush=True)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
