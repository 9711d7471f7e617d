"""Benchmark of the Flint MoE decode step on GB300: us per MoE sublayer and effective HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Workloads (weights drawn on the GPU by the seeded generator, 47 distinct sublayers):
  stack47_b1_nvfp4   47 chained NVFP4 sublayers, batch 1     (default)
  stack47_b8_nvfp4   same weights, batch 8
  stack47_b8_bf16    47 chained BF16-expert sublayers, batch 8 (~76 GB)
  prefill8192_nvfp4  one NVFP4 sublayer over 8,192 tokens (tensor-core grouped GEMMs)
A step is one pass of the 47-sublayer stack (one CUDA-graph launch of 141
kernels) over one batch; inputs cycle through 16 seeded batches so routing,
and hence the experts touched, changes every step.  The resident weights
(21.4 GB NVFP4 / 76 GB BF16) and the bytes touched per step (>= 631 MB) are far
larger than the 129 MB L2, so weights stream from HBM.

The JSON line reports `value` = us per sublayer (lower is better) measured with
CUDA events over K steps, the algorithmic HBM bytes of the step (router +
shared + distinct selected experts, counted from the actual routing), the
roofline fraction of the decode sublayer against the measured HBM copy
bandwidth, the end-to-end number through the C ABI with host buffers, SM
clocks sampled during the timed region, and the CPU oracle timed on a bounded
sample (`cpu_baseline`).  `--impl reference` times only the oracle.
"""

from __future__ import annotations

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

N_LAYERS = 47
NVFP4_EXPERT_BYTES = 1_769_472
BF16_EXPERT_BYTES = 6_291_456
ROUTER_BYTES = 256 * 2048 * 2
N_INPUTS = 16

WORKLOADS = {
    "stack47_b1_nvfp4": dict(cfg=1, batch=1, fmt="nvfp4"),
    "stack47_b8_nvfp4": dict(cfg=2, batch=8, fmt="nvfp4"),
    "stack47_b8_bf16": dict(cfg=3, batch=8, fmt="bf16"),
    "prefill8192_nvfp4": dict(cfg=4, batch=8192, fmt="nvfp4", prefill=True),
}
METRIC = "MoE decode µs/layer & effective HBM GB/s (% of roofline) at batch 1 and 8"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--layers", type=int, default=N_LAYERS,
                    help="sublayers in the stack (47 for the benchmark; fewer only for profiling captures)")
    ap.add_argument("--workload", default="stack47_b1_nvfp4", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------- CPU oracle timing

_ORACLE_CHILD = r"""
import json, sys, time, os
sys.path.insert(0, os.environ["FLINT_ROOT"])
import numpy as np, torch
torch.set_num_threads(1)
import oracle as O, synth
cfg, batch, budget, fmt = int(sys.argv[1]), int(sys.argv[2]), float(sys.argv[3]), sys.argv[4]
layers = [synth.gen_layer(cfg, i, device="cpu") for i in (1, 2)]
lws = [O.layer_from_tensors(d) for d in layers]
del layers
x = synth.gen_x(cfg, batch, index=0)
y = O.bf16_bits_to_f64(x.view(torch.int16).numpy().view(np.uint16))
n = 0
t0 = time.perf_counter()
while True:
    lw = lws[n % 2]
    lw.drop_cache()
    y = O.moe_layer(y, lw)["y"]
    n += 1
    if time.perf_counter() - t0 >= budget and n >= 2:
        break
dt = time.perf_counter() - t0
print(json.dumps({"layers": n, "seconds": dt}))
"""


_ORACLE_PREFILL_CHILD = r"""
import json, sys, time, os
sys.path.insert(0, os.environ["FLINT_ROOT"])
import numpy as np, torch
torch.set_num_threads(1)
import oracle as O, synth
cfg, t_small, t_large = int(sys.argv[1]), int(sys.argv[2]), int(sys.argv[3])
lw = O.layer_from_tensors(synth.gen_layer(cfg, 0, device="cpu"))
x = synth.gen_x(cfg, t_large, index=0)
x64 = O.bf16_bits_to_f64(x.view(torch.int16).numpy().view(np.uint16))
out = {}
for T in (t_small, t_large):
    lw.drop_cache()
    t0 = time.perf_counter()
    O.moe_prefill(x64[:T], lw)
    out[str(T)] = time.perf_counter() - t0
print(json.dumps(out))
"""


def time_oracle_prefill(cfg: int, tokens: int, small: int = 64, large: int = 256) -> dict:
    """The oracle's expert-grouped prefill on two bounded token counts (single
    thread); its cost is a per-layer part (every expert dequantised once) plus
    a per-token part, fitted on the two samples and evaluated at `tokens`."""
    env = dict(os.environ)
    env.update(FLINT_ROOT=ROOT, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _ORACLE_PREFILL_CHILD, str(cfg), str(small), str(large)],
                       capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        raise RuntimeError(f"oracle child failed: {r.stderr[-2000:]}")
    res = json.loads(r.stdout.strip().splitlines()[-1])
    ts, tl = res[str(small)], res[str(large)]
    per_token = max(0.0, (tl - ts) / (large - small))
    fixed = max(0.0, ts - per_token * small)
    us = (fixed + per_token * tokens) * 1e6
    return dict(value=us, unit="us/layer", cores=1, kind="oracle",
                sample=f"oracle prefill of {small} and {large} tokens ({ts:.1f} s, {tl:.1f} s single-threaded "
                       f"numpy fp64); per-layer {fixed:.1f} s + {per_token * 1e3:.2f} ms/token, "
                       f"evaluated at {tokens} tokens")


def time_oracle(cfg: int, batch: int, fmt: str, budget_s: float) -> dict:
    """Runs the oracle single-threaded in a fresh process on a bounded sample:
    consecutive sublayers (drawn on the CPU with the same distributions) until
    `budget_s` seconds of work; returns us per sublayer."""
    env = dict(os.environ)
    env.update(FLINT_ROOT=ROOT, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _ORACLE_CHILD, str(cfg), str(batch), str(budget_s), fmt],
                       capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        raise RuntimeError(f"oracle child failed: {r.stderr[-2000:]}")
    res = json.loads(r.stdout.strip().splitlines()[-1])
    us = res["seconds"] / res["layers"] * 1e6
    return dict(value=us, unit="us/layer", cores=1, kind="oracle",
                sample=f"{res['layers']} sublayers of the {fmt} stack at batch {batch}, "
                       f"{res['seconds']:.1f} s single-threaded numpy fp64 on the host")


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="flint_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- ncu traffic

def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("moe_decode_router_gb300/csrc/decode.cu", "moe_decode_router_gb300/csrc/flint_common.cuh"):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def prefill_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("moe_decode_router_gb300/csrc/prefill.cu", "moe_decode_router_gb300/csrc/tc05.cuh",
              "moe_decode_router_gb300/csrc/flint_common.cuh"):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_prefill_traffic(workload: str):
    """DRAM bytes (read + write) of one prefill sublayer, summed over its kernels, from
    the committed ncu summary; None if there is none or the kernels changed since."""
    path = os.path.join(ROOT, "profiles", "prefill8192_nvfp4_kernels.md")
    if not os.path.exists(path):
        return None, None
    src = prefill_source_hash()
    for line in open(path):
        if line.startswith("flint-traffic "):
            kv = dict(t.split("=", 1) for t in line.split()[1:])
            if kv.get("workload") == workload and kv.get("source") == src:
                return int(kv["bytes"]), os.path.relpath(path, ROOT)
    return None, None


def profiled_traffic_ratio(workload: str):
    """DRAM traffic / algorithmic bytes of one sublayer from the committed ncu summary,
    or None if there is none for this workload or the kernels changed since."""
    path = os.path.join(ROOT, "profiles", "decode_kernels_full_b1_b8.md")
    if not os.path.exists(path):
        return None, None
    src = kernel_source_hash()
    for line in open(path):
        if line.startswith("flint-traffic "):
            kv = dict(t.split("=", 1) for t in line.split()[1:])
            if kv.get("workload") == workload and kv.get("source") == src:
                return float(kv["ratio"]), os.path.relpath(path, ROOT)
    return None, None


# ----------------------------------------------------------------------------- our arm

def build_stack(F, synth, torch, wl, dev, n_layers):
    fmt = wl["fmt"]
    cfg = 1 if fmt == "nvfp4" else 3  # the NVFP4 stacks share one weight set (config-1 seeds)
    layers = []
    for i in range(n_layers):
        p = synth.gen_layer(cfg, i, device=dev)
        L = F.pack_layer(p, device=dev)
        torch.cuda.synchronize()
        L._keepalive = None
        layers.append(L)
        del p
    torch.cuda.empty_cache()
    return layers


def prefill_flops(T: int) -> float:
    """Algorithmic FLOPs of one prefill sublayer: router GEMM plus gate/up and
    down GEMMs over the 6 T routed and T shared token-expert pairs."""
    H, E, I = 2048, 256, 512
    return 2.0 * T * E * H + 2.0 * 7 * T * (2 * I * H + H * I)


def run_prefill(args, wl):
    import torch
    import torch.distributed as tdist

    import synth
    from moe_decode_router_gb300 import flint_moe as F

    world, rank, local = dist_env()
    if world > 1:
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    F.load_library()
    T = wl["batch"]
    plain = synth.gen_layer(wl["cfg"], 0, device=dev)
    L = F.pack_layer(plain, device=dev)
    torch.cuda.synchronize()
    del plain
    torch.cuda.empty_cache()
    n_in = 4
    xs = [synth.gen_x(wl["cfg"], T, index=i, device=dev) for i in range(n_in)]
    ys = [torch.empty_like(x) for x in xs]
    ws = F.alloc_workspace(F.W_NVFP4, T, device=dev)
    for s in range(max(3, args.warmup)):
        F.prefill_layer(L, xs[s % n_in], ys[s % n_in], ws)
    torch.cuda.synchronize()
    assert F.device_error() == 0
    steps = args.steps
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        tdist.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for s in range(steps):
        F.prefill_layer(L, xs[s % n_in], ys[s % n_in], ws)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        tdist.barrier()
    clk = clocks.stop()
    err = F.device_error()

    # End to end through the C ABI: pinned host tokens -> device, sublayer, device -> pinned host.
    hx = [x.cpu().pin_memory() for x in xs]
    hy = torch.empty_like(hx[0]).pin_memory()
    xin = torch.empty_like(xs[0])
    yout = torch.empty_like(xs[0])
    for s in range(3):
        xin.copy_(hx[s % n_in], non_blocking=True)
        F.prefill_layer(L, xin, yout, ws)
        hy.copy_(yout, non_blocking=True)
    torch.cuda.synchronize()
    e2e_steps = max(10, steps // 4)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(e2e_steps):
        xin.copy_(hx[s % n_in], non_blocking=True)
        F.prefill_layer(L, xin, yout, ws)
        hy.copy_(yout, non_blocking=True)
    t1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = t0.elapsed_time(t1) / e2e_steps

    ms_t = torch.tensor([ms], device=dev)
    if world > 1:
        tdist.all_reduce(ms_t, op=tdist.ReduceOp.MAX)
    ms_per_step = float(ms_t.item()) / steps
    flops = prefill_flops(T)
    tflops = flops / (ms_per_step / 1000.0) / 1e12
    peaks = {}
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk_path):
        peaks = json.load(open(pk_path))
    peak = peaks.get("bf16_tflops_sustained")
    peak_src = "measured (sustained bf16 cuBLAS)" if peak else "fallback"
    peak = peak or 1700.0
    ptraffic, _ = profiled_prefill_traffic(args.workload)
    out = {
        "metric": METRIC,
        "value": round(ms_per_step * 1000.0, 2),
        "unit": "us/layer",
        "n_gpus": world,
        "steps": steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4-w/bf16-a (f16/bf16 tensor-core operands, f32 accumulate)",
        "data": "synthetic (seeded generator, random-init weights of the Flint MoE shapes)",
        "config": {
            "workload": args.workload, "tokens": T, "hidden": 2048, "experts": "256+1", "inter": 512,
            "top_k": 6, "weights": "nvfp4", "parallelism": f"replicas x{world}",
            "l2": "every step streams all 257 experts' packed weights (455 MB) and 4 rotating 32 MB token "
                  "batches: far larger than L2",
        },
        "tflops": round(tflops, 1),
        "roofline": {
            "kernel": "prefill sublayer (router GEMM, routing, grouped gate/up and down GEMMs, combine)",
            "bound": "tensor", "achieved": round(tflops, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(tflops / peak, 4), "peak_source": peak_src,
            "flops_per_layer": flops, "traffic": ptraffic,
        },
        "e2e": {"value": round(e2e_ms * 1000.0, 2), "unit": "us/layer",
                "h2d_bytes_per_step": T * 2048 * 2, "d2h_bytes_per_step": T * 2048 * 2},
        "gpu_launches": steps * 7,
        "clocks": clk,
        "device_error_word": err,
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        try:
            out["cpu_baseline"] = time_oracle_prefill(wl["cfg"], T)
        except Exception as e:  # report, do not hide
            out["cpu_baseline"] = {"value": None, "error": str(e)[:300]}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        tdist.destroy_process_group()


def run_ours(args):
    if WORKLOADS[args.workload].get("prefill"):
        return run_prefill(args, WORKLOADS[args.workload])
    import torch
    import torch.distributed as tdist

    import synth
    from moe_decode_router_gb300 import flint_moe as F

    world, rank, local = dist_env()
    if world > 1:
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    F.load_library()
    wl = WORKLOADS[args.workload]
    B = wl["batch"]
    fmt = F.W_NVFP4 if wl["fmt"] == "nvfp4" else F.W_BF16
    NL = args.layers
    layers = build_stack(F, synth, torch, wl, dev, NL)
    xs = [synth.gen_x(wl["cfg"], B, index=i, device=dev) for i in range(N_INPUTS)]
    ys = [torch.empty_like(x) for x in xs]
    ws = F.alloc_workspace(fmt, B, device=dev)

    # Algorithmic bytes per input: router + (distinct routed + shared) experts per sublayer.
    expert_bytes = NVFP4_EXPERT_BYTES if fmt == F.W_NVFP4 else BF16_EXPERT_BYTES
    ids = torch.empty((NL, B, 6), dtype=torch.int32, device=dev)
    bytes_per_input = []
    uniq = []
    for i, x in enumerate(xs):
        F.decode_stack(layers, x, ys[i], ws, ids_per_layer=ids)
        torch.cuda.synchronize()
        idc = ids.cpu()
        u = [len(set(idc[l].flatten().tolist())) for l in range(NL)]
        uniq.extend(u)
        bytes_per_input.append(sum(ROUTER_BYTES + (n + 1) * expert_bytes for n in u))
    # Prime one cached graph per input buffer (the graph bakes in pointers).
    for i, x in enumerate(xs):
        F.decode_stack(layers, x, ys[i], ws)
    torch.cuda.synchronize()
    assert F.device_error() == 0

    stream = torch.cuda.current_stream()
    for s in range(args.warmup):
        F.decode_stack(layers, xs[s % N_INPUTS], ys[s % N_INPUTS], ws)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        tdist.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for s in range(args.steps):
        F.decode_stack(layers, xs[s % N_INPUTS], ys[s % N_INPUTS], ws)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        tdist.barrier()
    clk = clocks.stop()
    err = F.device_error()

    # End to end through the C ABI: pinned host input -> device, stack, device -> pinned host.
    hx = [x.cpu().pin_memory() for x in xs]
    hy = torch.empty_like(hx[0]).pin_memory()
    xin = torch.empty_like(xs[0])
    yout = torch.empty_like(xs[0])
    for s in range(max(3, args.warmup)):
        xin.copy_(hx[s % N_INPUTS], non_blocking=True)
        F.decode_stack(layers, xin, yout, ws)
        hy.copy_(yout, non_blocking=True)
    torch.cuda.synchronize()
    e2e_steps = max(10, args.steps // 2)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(e2e_steps):
        xin.copy_(hx[s % N_INPUTS], non_blocking=True)
        F.decode_stack(layers, xin, yout, ws)
        hy.copy_(yout, non_blocking=True)
    t1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = t0.elapsed_time(t1) / e2e_steps

    ms_t = torch.tensor([ms], device=dev)
    if world > 1:
        tdist.all_reduce(ms_t, op=tdist.ReduceOp.MAX)
    ms = float(ms_t.item())
    ms_per_step = ms / args.steps
    us_per_layer = ms_per_step * 1000.0 / NL
    total_bytes = sum(bytes_per_input[s % N_INPUTS] for s in range(args.steps))
    gbs = total_bytes / (ms / 1000.0) / 1e9
    peaks = {}
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk_path):
        peaks = json.load(open(pk_path))
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    bytes_per_layer = total_bytes / args.steps / NL
    traffic_ratio, traffic_src = profiled_traffic_ratio(args.workload)
    out = {
        "metric": METRIC,
        "value": round(us_per_layer, 3),
        "unit": "us/layer",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4-w/bf16-a (f32 accumulate)" if fmt == F.W_NVFP4 else "bf16 (f32 accumulate)",
        "data": "synthetic (seeded generator, random-init weights of the Flint MoE shapes)",
        "config": {
            "workload": args.workload, "layers": NL, "batch": B, "hidden": 2048, "experts": "256+1",
            "inter": 512, "top_k": 6, "weights": wl["fmt"], "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2: 16 rotating batches, >=631 MB touched per step, weights resident "
                  f"{len(layers) * F.packed_bytes(fmt) / 1e9:.1f} GB",
            "mean_unique_experts_per_layer": round(sum(uniq) / len(uniq), 2),
        },
        "effective_hbm_gbs": round(gbs, 1),
        "roofline": {
            "kernel": "decode sublayer (router + gate/up + down, chained by programmatic dependent launch)",
            "bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(gbs / peak, 4), "peak_source": peak_src,
            "bytes_per_layer": round(bytes_per_layer),
            "traffic": round(traffic_ratio * bytes_per_layer) if traffic_ratio else None,
            "traffic_source": traffic_src,
        },
        "e2e": {"value": round(e2e_ms * 1000.0 / NL, 3), "unit": "us/layer",
                "h2d_bytes_per_step": B * 2048 * 2, "d2h_bytes_per_step": B * 2048 * 2},
        "gpu_launches": args.steps * NL * 3,
        "clocks": clk,
        "device_error_word": err,
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        try:
            out["cpu_baseline"] = time_oracle(wl["cfg"], B, wl["fmt"], args.cpu_seconds)
        except Exception as e:  # report, do not hide
            out["cpu_baseline"] = {"value": None, "error": str(e)[:300]}
    elif rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = {"value": None, "note": "timed at N=1 only"}
    if rank == 0:
        print(json.dumps(out), flush=True)
    F.release()
    if world > 1:
        tdist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm (oracle)

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    if wl.get("prefill"):
        r = time_oracle_prefill(wl["cfg"], wl["batch"])
        us = r["value"]
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/layer", "n_gpus": world,
            "steps": 1, "warmup": 0, "ms_per_step": round(us / 1000.0, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded generator)",
            "config": {"workload": args.workload, "tokens": wl["batch"], "weights": wl["fmt"]},
            "cpu_baseline": r,
            "e2e": {"value": round(us, 1), "unit": "us/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return
    per_step_budget = max(0.5, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(wl["cfg"], wl["batch"], wl["fmt"], per_step_budget / 4)
    vals = []
    samples = []
    for _ in range(args.steps):
        r = time_oracle(wl["cfg"], wl["batch"], wl["fmt"], per_step_budget)
        vals.append(r["value"])
        samples.append(r["sample"])
    us = statistics.mean(vals)
    out = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/layer", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us * N_LAYERS / 1000.0, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded generator)",
        "config": {"workload": args.workload, "layers": N_LAYERS, "batch": wl["batch"], "weights": wl["fmt"]},
        "cpu_baseline": {"value": round(us, 1), "unit": "us/layer", "cores": 1, "kind": "oracle",
                         "sample": samples[-1] if samples else ""},
        "e2e": {"value": round(us, 1), "unit": "us/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
