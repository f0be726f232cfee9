"""Throughput of the FP4 routed-MoE layer on GB300.

One step = one pass of the whole layer (routing, expert sort, W13 + SwiGLU,
W2, combine) over one batch of synthetic inputs resident in HBM.  The
default workload is the decode-shaped layer (T=32, d=4096, I=2048, E=256,
k=8); the prefill-shaped layer (T=4608) is measured the same way and
reported in the "prefill" object of the same line, the skewed-routing
(T=2048) and large (T=16384, d=7168) layers under "other_workloads", the
layer with MXFP8 activations on block-scaled tensor cores (prefill shape)
under "mx_layer", and the MXFP8 activation quantiser under "mxfp8_quantize".  Every expert weight
set touched per step (~2.2 GB decode, 3.4 GB prefill) is far larger than
L2 (129 MB), so no L2 flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun: every rank runs its own replica of the same
workload (the layer has no data-path exchange here), timed between
barriers; the max over ranks is taken and rank 0 prints one JSON line.
``--impl reference`` times the CPU oracle on a bounded sample of the same
workload on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_inputs import CONFIGS, make_config  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
STAGES = ["route", "gather", "w13_swiglu", "w2", "combine"]
# flags of every exact-layer call (bench --deterministic: the slot-order combine pass)
LAYER_FLAGS = 0


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def ncu_traffic(key):
    """DRAM bytes per launch (read + write) of one kernel on one workload, from the
    committed ncu capture, or None when the kernel's source changed since then."""
    import hashlib
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)[key]
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha1(f.read()).hexdigest() != rec["source_sha1"]:
                return None
        return int(rec["dram_read_bytes"]) + int(rec["dram_write_bytes"])
    except (OSError, ValueError, KeyError):
        return None


def decode_config(world):
    """The `config` object of both arms' JSON lines: the decode workload, the
    same keys and values for the CUDA path and the oracle's reference arm
    (the touched experts counted from the workload's router logits: the top-8
    of each token, ties to the lower index, as the layer routes)."""
    L = make_config("decode")
    order = np.lexsort((np.broadcast_to(np.arange(L.E), L.router_logits.shape), -L.router_logits), axis=1)
    touched = int(np.unique(order[:, :L.k]).size)
    return {"workload": "decode-shaped MoE layer T=32 d=4096 I=2048 E=256 k=8 (seed 0)",
            "global_batch": world * L.T, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (touched weights %.2f GB)" % (touched * sum(expert_bytes(L.d, L.I)) / 1e9),
            "touched_experts": touched}


def expert_bytes(d, I):
    """packed codes + E8M0 scales of one expert: W13 [2I, d] and W2 [d, I]"""
    w13 = 2 * I * d // 2 + 2 * I * d // 32
    w2 = d * I // 2 + d * I // 32
    return w13, w2


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, windows):
        """clocks over the samples taken inside the timed regions `windows`
        [(t0, t1), ...]; if none landed inside (short regions), the samples
        within 0.3 s of them"""
        rows = []
        for ts, ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
            except ValueError:
                continue
        inside = [r for r in rows if any(t0 <= r[0] <= t1 for t0, t1 in windows)]
        window = inside if inside else [r for r in rows if any(t0 - 0.3 <= r[0] <= t1 + 0.3 for t0, t1 in windows)]
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in window:
            for name, v in zip(names, r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median([r[1] for r in window])), "sm_max_mhz": max(r[2] for r in window),
                "reasons": sorted(reasons), "samples": len(inside),
                "window": "inside the timed regions of all workloads" if inside else "within 0.3 s of them"}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def dist_setup(n_gpus):
    import torch
    if n_gpus <= 1:
        return 0, 1, 0, None
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    world = int(os.environ["WORLD_SIZE"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local, dist


def barrier(dist, device="cuda"):
    import torch
    if device == "cuda":
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
        if device == "cuda":
            torch.cuda.synchronize()


def _reduce(dist, v, op, device):
    import torch
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(dist, v, device="cuda"):
    """the slowest rank's time (the whole job waits for it)"""
    return v if dist is None else _reduce(dist, v, dist.ReduceOp.MAX, device)


def sum_over_ranks(dist, v, device="cuda"):
    return v if dist is None else _reduce(dist, v, dist.ReduceOp.SUM, device)


def measure_workload(name, steps, warmup, dist, local, sampler=None):
    """Time `steps` forward passes of one workload; returns a dict of results."""
    import torch

    import fp4_mixture_experts_gb300 as moe

    L = make_config(name)
    dev = torch.device("cuda", local)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    x = t(L.x_bf16.view(np.int16)).view(torch.bfloat16)
    logits, w13, w13s, w2, w2s = t(L.router_logits), t(L.w13), t(L.w13_scale), t(L.w2), t(L.w2_scale)
    ws = torch.empty(moe.workspace_bytes(L.T, L.d, L.I, L.E, L.k), dtype=torch.uint8, device=dev)
    out = torch.empty(L.T, L.d, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # per-step stage events; record each once so the handles exist
    n_ev = 6
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(steps)]
    for row in evs:
        for ev in row:
            ev.record(stream)
    r = moe.forward(x, logits, w13, w13s, w2, w2s, L.k, out=out, workspace=ws, return_routing=True,
                    flags=LAYER_FLAGS)
    torch.cuda.synchronize()
    ids = r["topk_ids"].cpu().numpy()
    touched = int(np.unique(ids).size)
    for _ in range(warmup):
        moe.forward(x, logits, w13, w13s, w2, w2s, L.k, out=out, workspace=ws, flags=LAYER_FLAGS)
    barrier(dist)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    start.record(stream)
    for s in range(steps):
        moe.forward(x, logits, w13, w13s, w2, w2s, L.k, out=out, workspace=ws, stage_events=evs[s],
                    flags=LAYER_FLAGS)
    end.record(stream)
    barrier(dist)
    t_wall1 = time.time()
    ms_stream = start.elapsed_time(end)
    windows = [(t_wall0, t_wall1)]
    stage_ms = {name_: float(np.mean([evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps)]))
                for i, name_ in enumerate(STAGES)}
    # the same layer call captured once in a CUDA graph and replayed: the
    # launches of a step go to the GPU together (how a decode loop runs it)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        moe.forward(x, logits, w13, w13s, w2, w2s, L.k, out=out, workspace=ws, flags=LAYER_FLAGS)
    stream.wait_stream(side)
    with torch.cuda.graph(graph):
        moe.forward(x, logits, w13, w13s, w2, w2s, L.k, out=out, workspace=ws, flags=LAYER_FLAGS)
    for _ in range(warmup):
        graph.replay()
    barrier(dist)
    t_wall0 = time.time()
    start.record(stream)
    for s in range(steps):
        graph.replay()
    end.record(stream)
    barrier(dist)
    t_wall1 = time.time()
    ms_graph = start.elapsed_time(end)
    windows.append((t_wall0, t_wall1))
    res = dict(L=L, touched=touched, ms_total=max_over_ranks(dist, ms_graph),
               ms_stream=max_over_ranks(dist, ms_stream), stage_ms=stage_ms,
               windows=windows, tensors=(x, logits, w13, w13s, w2, w2s, ws), graph=graph)
    return res


def measure_e2e(res, steps, warmup, dist, local):
    """Same metric through the host-buffer entry point: H2D of x and logits,
    the layer, D2H of out, every step (pinned host memory)."""
    import torch

    import fp4_mixture_experts_gb300 as moe
    L = res["L"]
    _, _, w13, w13s, w2, w2s, _ = res["tensors"]
    xh = torch.from_numpy(L.x_bf16.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    lh = torch.from_numpy(L.router_logits.copy()).pin_memory()
    oh = torch.empty(L.T, L.d, dtype=torch.float32).pin_memory()
    dev = torch.device("cuda", local)
    wsh = torch.empty(moe.host_workspace_bytes(L.T, L.d, L.I, L.E, L.k), dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        moe.forward_host(xh, lh, w13, w13s, w2, w2s, L.k, out_host=oh, workspace=wsh, flags=LAYER_FLAGS)
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(steps):
        moe.forward_host(xh, lh, w13, w13s, w2, w2s, L.k, out_host=oh, workspace=wsh, flags=LAYER_FLAGS)
    barrier(dist)
    dt = max_over_ranks(dist, time.perf_counter() - t0)
    h2d = L.x_bf16.nbytes + L.router_logits.nbytes
    d2h = L.T * L.d * 4
    return dt, h2d, d2h


def roofline_decode(res, pk, src):
    """Dominant kernel of the streaming path: W13 + SwiGLU (2/3 of the weight bytes)."""
    L = res["L"]
    w13b, w2b = expert_bytes(L.d, L.I)
    st = res["stage_ms"]
    w13_bytes = res["touched"] * w13b + L.T * L.d * 2
    w2_bytes = res["touched"] * w2b
    ach = w13_bytes / (st["w13_swiglu"] * 1e-3) / 1e9
    step_bytes = w13_bytes + w2_bytes
    return {"bound": "hbm", "kernel": "w13_swiglu", "achieved": round(ach, 1), "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4),
            "traffic": ncu_traffic("stream_kernel<W13>@decode"),
            "peak_source": f"{src} hbm_gbs (copy, burst)",
            "bytes_per_launch": w13_bytes,
            "step_bytes": step_bytes,
            "step_frac": round(step_bytes / (res["ms_total"] / res["steps"] * 1e-3) / 1e9 / pk["hbm_gbs"], 4)}


def roofline_prefill(res, pk, src):
    """Dominant kernel of the tensor-core path: W13 + SwiGLU (2/3 of the FLOPs).
    The timed region lasts tens of milliseconds at full clock, so the peak is
    the burst figure (cuBLAS bf16, best of 10); the sustained figure (a 4 s
    loop under the power cap) is reported beside it."""
    L = res["L"]
    st = res["stage_ms"]
    flops_w13 = 4.0 * L.T * L.k * L.d * L.I
    ach = flops_w13 / (st["w13_swiglu"] * 1e-3) / 1e12
    peak = pk["bf16_tflops"]
    step_flops = 6.0 * L.T * L.k * L.d * L.I
    step_ach = step_flops / (res["ms_total"] / res["steps"] * 1e-3) / 1e12
    out = {"bound": "tensor", "kernel": "w13_swiglu", "achieved": round(ach, 1), "peak": peak,
           "unit": "TFLOP/s", "frac": round(ach / peak, 4),
           "traffic": None,
           "peak_source": f"{src} bf16_tflops (cuBLAS bf16 burst, the kernel is timed in a short run)",
           "flops_per_launch": flops_w13,
           "step_frac": round(step_ach / peak, 4)}
    if "bf16_tflops_sustained" in pk:
        out["frac_of_sustained"] = round(ach / pk["bf16_tflops_sustained"], 4)
    return out


def measure_mx_layer(name, steps, warmup, dist, local, pk, src):
    """The layer with MXFP8 activations (moe_fp4_forward_mx: both projections
    on block-scaled kind::mxf8f6f4 tensor cores) on one workload, stage events
    per step.  Stages: route, quantising gather, W13 (+ SwiGLU), h quantiser +
    W2, combine.  The dominant kernel (W13) is reported against the dense fp8
    peak, taken as the measured bf16 peak times 2 (the nominal fp8:bf16 ratio,
    4.5 : 2.25 PFLOP/s)."""
    import torch

    import fp4_mixture_experts_gb300 as moe
    L = make_config(name)
    dev = torch.device("cuda", local)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    x = t(L.x_bf16.view(np.int16)).view(torch.bfloat16)
    args = (x, t(L.router_logits), t(L.w13), t(L.w13_scale), t(L.w2), t(L.w2_scale), L.k)
    ws = torch.empty(moe.mx_workspace_bytes(L.T, L.d, L.I, L.E, L.k), dtype=torch.uint8, device=dev)
    out = torch.empty(L.T, L.d, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    for row in evs:
        for ev in row:
            ev.record(stream)
    for _ in range(warmup):
        moe.forward_mx(*args, out=out, workspace=ws)
    barrier(dist)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record(stream)
    for k in range(steps):
        moe.forward_mx(*args, out=out, workspace=ws, stage_events=evs[k])
    end.record(stream)
    barrier(dist)
    t1 = time.time()
    moe.check(ws)
    ms = max_over_ranks(dist, start.elapsed_time(end)) / steps
    names = ["route", "gather_quantise", "w13_swiglu", "quantise_h_w2", "combine"]
    stage_ms = {n: float(np.mean([evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(steps)]))
                for i, n in enumerate(names)}
    S = L.T * L.k
    flops_w13 = 4.0 * S * L.d * L.I
    ach = flops_w13 / (stage_ms["w13_swiglu"] * 1e-3) / 1e12
    peak = 2.0 * pk["bf16_tflops"]
    world = 1 if dist is None else dist.get_world_size()
    res = {"workload": f"{name} MoE layer T={L.T} d={L.d} I={L.I} E={L.E} k={L.k} (seed 0), MXFP8 activations",
           "value": round(world * L.T / (ms * 1e-3), 1), "unit": "tokens/s", "steps": steps,
           "ms_per_step": round(ms, 4), "dtype": "fp4(e2m1) x fp8(e4m3), e8m0 block scales -> f32",
           "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
           "roofline": {"bound": "tensor", "kernel": "mx_kernel<W13>", "achieved": round(ach, 1), "peak": peak,
                        "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                        "traffic": ncu_traffic("mx_kernel<W13>@prefill"),
                        "peak_source": f"{src} bf16_tflops x 2 (nominal fp8:bf16 ratio; fp8 not measured)",
                        "flops_per_launch": flops_w13}}
    del ws, out, args, x
    return res, (t0, t1)


def measure_mxfp8(local, warmup=5, iters=50):
    """The MXFP8 activation quantiser on the prefill layer's permuted-activation
    shape (36,864 x 4096 bf16, 302 MB: larger than L2), CUDA events over
    `iters` back-to-back calls; bytes = 2 read + 1 + 1/32 written per element."""
    import torch

    import fp4_mixture_experts_gb300 as moe
    R, K = 36864, 4096
    dev = torch.device("cuda", local)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    x = torch.randn(R, K, device=dev, generator=g).to(torch.bfloat16)
    codes = torch.empty(R, K, dtype=torch.uint8, device=dev)
    scales = torch.empty(R, K // 32, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        moe.mxfp8_quantize(x, codes, scales)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record()
    for _ in range(iters):
        moe.mxfp8_quantize(x, codes, scales)
    end.record()
    torch.cuda.synchronize()
    t1 = time.time()
    ms = start.elapsed_time(end) / iters
    nbytes = R * K * 2 + R * K + R * K // 32
    del x, codes, scales
    return {"shape": [R, K], "us_per_call": round(ms * 1e3, 2), "bytes_per_call": nbytes,
            "achieved_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}, (t0, t1)


def cpu_baseline_sample(name, seconds_target=15.0, gpu=None):
    """The oracle, as it stands, on a bounded sample of the workload: whole
    tokens through oracle.forward_tokens until ~seconds_target elapse.  With
    `gpu` (numpy out [T, d] and topk_ids [T, k] of the CUDA path on the same
    layer), the sampled tokens' oracle results are compared with it after the
    timed loop and reported as "parity"."""
    import oracle
    L = make_config(name)
    toks, outs, ids = [], [], []
    t0 = time.perf_counter()
    for t in range(L.T):
        i, _, o = oracle.forward_tokens(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k, [t])
        toks.append(t)
        ids.append(i[0])
        outs.append(o[0])
        if time.perf_counter() - t0 >= seconds_target:
            break
    dt = time.perf_counter() - t0
    res = {"value": round(len(toks) / dt, 4), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
           "sample": f"{len(toks)} of {L.T} tokens of the {name} layer, one token per oracle call "
                     f"(numpy fp64, BLAS threads = host cores), {dt:.1f} s"}
    if gpu is not None:
        got = np.asarray(gpu["out"], dtype=np.float64)[toks]
        want = np.stack(outs)
        res["parity"] = {"tokens": len(toks),
                         "topk_ids_equal": bool(np.array_equal(np.asarray(gpu["topk_ids"])[toks], np.stack(ids))),
                         "rel_l2": float(np.linalg.norm(got - want) / np.linalg.norm(want)),
                         "max_abs": float(np.abs(got - want).max())}
    return res


def run_ours(args):
    import torch
    rank, world, local, dist = dist_setup(args.gpus)
    pk, src = peaks()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    windows = []
    dec = measure_workload("decode", args.steps, args.warmup, dist, local)
    dec["steps"] = args.steps
    windows += dec["windows"]
    e2e_dt, h2d, d2h = measure_e2e(dec, args.steps, args.warmup, dist, local)
    pre = None
    if not args.no_prefill:
        pre_steps = max(3, min(args.steps, 50))
        pre = measure_workload("prefill", pre_steps, max(3, min(args.warmup, 5)), dist, local)
        pre["steps"] = pre_steps
        windows += pre["windows"]
    others = {}
    for name in [n for n in args.also.split(",") if n]:
        # further workloads (tensor-core path), timed like the prefill workload
        o_steps = max(3, min(args.steps, 50))
        res = measure_workload(name, o_steps, max(3, min(args.warmup, 5)), dist, local)
        res["steps"] = o_steps
        windows += res["windows"]
        Lo = res["L"]
        ms_o = res["ms_total"] / o_steps
        rf = roofline_prefill(res, pk, src)
        others[name] = {"workload": f"{name} MoE layer T={Lo.T} d={Lo.d} I={Lo.I} E={Lo.E} k={Lo.k} (seed 0)",
                        "value": round(world * Lo.T / (ms_o * 1e-3), 1), "unit": "tokens/s", "steps": o_steps,
                        "ms_per_step": round(ms_o, 4), "touched_experts": res["touched"],
                        "stage_ms": {k: round(v, 4) for k, v in res["stage_ms"].items()},
                        "roofline": rf}
        del res
        torch.cuda.empty_cache()
    mxl = None
    if not args.no_mx_layer:
        mx_steps = max(3, min(args.steps, 50))
        mxl, win = measure_mx_layer("prefill", mx_steps, max(3, min(args.warmup, 5)), dist, local, pk, src)
        windows.append(win)
        torch.cuda.empty_cache()
    mxq = None
    if rank == 0 and not args.no_mxfp8:
        mxq, win = measure_mxfp8(local)
        windows.append(win)
        mxq["frac"] = round(mxq["achieved_gbs"] / pk["hbm_gbs"], 4)
        mxq["peak_gbs"] = pk["hbm_gbs"]
    clocks = sampler.summary(windows) if sampler else None
    if sampler:
        sampler.stop()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    L = dec["L"]
    ms_step = dec["ms_total"] / args.steps
    value = world * L.T * args.steps / (dec["ms_total"] * 1e-3)
    # decode path: route_small (routing + sort in one cluster launch), W13 + SwiGLU (which also
    # zeroes out), W2 with the weighted combine in its epilogue; --deterministic: W2 writes y
    # and the combine pass is a fourth launch
    launches_per_step = 4 if LAYER_FLAGS else 3
    line = {
        "metric": "routed-MoE tokens/s (decode T=32, prefill T=4608); % of HBM/tensor roofline",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "ms_per_step_stream_launch": round(dec["ms_stream"] / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp4(e2m1)xbf16->f32", "data": "synthetic",
        "config": decode_config(world),
        "launch": "one layer call captured in a CUDA graph, replayed per step",
        "combine": ("slot-order pass (deterministic)" if LAYER_FLAGS
                    else "in the W2 epilogue (fp32 atomic adds, summation order not fixed)"),
        "stage_ms": {k: round(v, 5) for k, v in dec["stage_ms"].items()},
        "roofline": roofline_decode(dec, pk, src),
        "gpu_launches": launches_per_step * args.steps,
        "e2e": {"value": round(world * L.T * args.steps / e2e_dt, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "clocks": clocks,
    }
    if pre is not None:
        P = pre["L"]
        ms_pre = pre["ms_total"] / pre["steps"]
        rf = roofline_prefill(pre, pk, src)
        rf["traffic"] = ncu_traffic("tc_kernel<W13>@prefill")
        line["prefill"] = {
            "workload": "prefill-shaped MoE layer T=4608 d=4096 I=2048 E=256 k=8 (seed 0)",
            "value": round(world * P.T / (ms_pre * 1e-3), 1), "unit": "tokens/s", "steps": pre["steps"],
            "ms_per_step": round(ms_pre, 4), "ms_per_step_stream_launch": round(pre["ms_stream"] / pre["steps"], 4),
            "stage_ms": {k: round(v, 4) for k, v in pre["stage_ms"].items()},
            "roofline": rf}
    if others:
        line["other_workloads"] = others
    if mxl is not None:
        line["mx_layer"] = mxl
    if mxq is not None:
        line["mxfp8_quantize"] = mxq
    if not args.no_cpu_baseline:
        # one more layer call on the measured decode tensors, checked against the oracle's sample
        x, logits, w13, w13s, w2, w2s, _ = dec["tensors"]
        import fp4_mixture_experts_gb300 as moe
        r = moe.forward(x, logits, w13, w13s, w2, w2s, L.k, return_routing=True, flags=LAYER_FLAGS)
        torch.cuda.synchronize()
        gpu = {"out": r["out"].cpu().numpy(), "topk_ids": r["topk_ids"].cpu().numpy()}
        line["cpu_baseline"] = cpu_baseline_sample("decode", args.cpu_seconds, gpu)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# reference arm: the CPU oracle on the host cores
# ----------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    L = make_config("decode")
    # one step = one token of the decode layer through the oracle
    for s in range(args.warmup):
        oracle.forward_tokens(L.x_bf16, L.router_logits, L.w13, L.w13_scale, L.w2, L.w2_scale, L.k, [s % L.T])
    per_step_cap = max(0.05, 150.0 / max(1, args.steps))
    t0 = time.perf_counter()
    units = 0.0
    for s in range(args.steps):
        ts = time.perf_counter()
        t = s % L.T
        ids, _ = oracle.route(L.router_logits[t:t + 1], L.k)
        # experts of this token, one oracle expert evaluation at a time, until the per-step cap
        done = 0
        x = oracle.bf16_bits_to_f64(L.x_bf16[t:t + 1])
        for e in ids[0]:
            oracle.expert_ffn(x, L.w13[e], L.w13_scale[e], L.w2[e], L.w2_scale[e])
            done += 1
            if time.perf_counter() - ts > per_step_cap:
                break
        units += done / L.k
    dt = time.perf_counter() - t0
    value = units / dt
    line = {"impl": "reference", "metric": "routed-MoE tokens/s (decode T=32, prefill T=4608); % of HBM/tensor roofline",
            "value": round(value, 4), "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": decode_config(args.gpus),
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{units:.3f} tokens (one token, or part of its {L.k} experts, per step)"},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


PROFILE_CASES = {
    # name: (workload, experts override, tokens override, MXFP8 layer) -- smaller expert
    # counts keep ncu captures to about a GB on the device while the weights stay larger than L2
    "decode": ("decode", None, None, False),
    "prefill": ("prefill", None, None, False),
    "decode-e64": ("decode", 64, 32, False),
    "prefill-e64": ("prefill", 64, 1152, False),
    "prefill-mx": ("prefill", None, None, True),
    "prefill-mx-e64": ("prefill", 64, 1152, True),
}


def run_profile_case(args):
    """Run `--steps` forward passes of one case with no timing or JSON output:
    the command that ncu captures."""
    import torch

    import fp4_mixture_experts_gb300 as moe
    from moe_inputs import make_layer
    name, E, T, mx = PROFILE_CASES[args.profile_case]
    c = dict(CONFIGS[name])
    if E is not None:
        c["E"], c["T"] = E, T
    L = make_layer(**c)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    x = t(L.x_bf16.view(np.int16)).view(torch.bfloat16)
    args_ = (x, t(L.router_logits), t(L.w13), t(L.w13_scale), t(L.w2), t(L.w2_scale), L.k)
    nbytes = (moe.mx_workspace_bytes if mx else moe.workspace_bytes)(L.T, L.d, L.I, L.E, L.k)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty(L.T, L.d, dtype=torch.float32, device="cuda")
    for _ in range(args.warmup + args.steps):
        if mx:
            moe.forward_mx(*args_, out=out, workspace=ws)
        else:
            moe.forward(*args_, out=out, workspace=ws, flags=LAYER_FLAGS)
    torch.cuda.synchronize()
    moe.check(ws)
    print(f"profile case {args.profile_case}: T={L.T} d={L.d} I={L.I} E={L.E} k={L.k}, "
          f"{args.warmup + args.steps} forward passes, out rms {out.float().pow(2).mean().sqrt().item():.3f}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--also", default="skewed,large", help="comma list of further workloads to time after "
                    "decode and prefill (skewed, large; '' for none); reported under other_workloads")
    ap.add_argument("--no-mxfp8", action="store_true", help="skip timing the MXFP8 activation quantiser")
    ap.add_argument("--no-mx-layer", action="store_true",
                    help="skip timing the layer with MXFP8 activations (block-scaled tensor cores) at prefill")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="run the exact layer with the slot-order combine pass (bitwise reproducible) instead "
                         "of the combine in the W2 epilogue")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES), default=None,
                    help="only run forward passes of one case (for ncu), no measurement")
    args = ap.parse_args()
    global LAYER_FLAGS
    LAYER_FLAGS = 0x10 if args.deterministic else 0  # MOE_FP4_FLAG_DETERMINISTIC
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    for n in [n for n in args.also.split(",") if n]:
        if n not in CONFIGS or n in ("decode", "prefill"):
            ap.error(f"--also takes workloads other than decode and prefill: {sorted(set(CONFIGS) - {'decode', 'prefill'})}")
    if args.profile_case:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
