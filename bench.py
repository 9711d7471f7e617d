"""Benchmark of the Flint MoE decode step on GB300: us per MoE sublayer and effective HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--no-extras] [--no-cpu-baseline]

Workloads (weights drawn on the GPU by the seeded generator, 47 distinct sublayers):
  stack47_b1_nvfp4   47 chained NVFP4 sublayers, batch 1     (default)
  stack47_b8_nvfp4   same weights, batch 8
  stack47_b8_bf16    47 chained BF16-expert sublayers, batch 8 (~76 GB)
  prefill8192_nvfp4  one NVFP4 sublayer over 8,192 tokens (tensor-core grouped GEMMs)
A step is one pass of the 47-sublayer stack over one batch (one CUDA-graph
launch of 141 chained kernels; with the persistent NVFP4 kernel, one launch); inputs cycle through 16 seeded batches so routing, and hence the
experts touched, changes every step.  The resident weights (21.4 GB NVFP4 /
76 GB BF16) and the bytes touched per step (>= 631 MB) are far larger than the
129 MB L2, so weights stream from HBM.

The JSON line reports `value` = us per sublayer (lower is better) measured with
CUDA events over K steps, the algorithmic HBM bytes of the step (router +
shared + distinct selected experts, counted from the actual routing), the
roofline fraction against the measured HBM copy bandwidth, the end-to-end
number through the C ABI with host buffers, SM clocks sampled during the timed
region, and the CPU oracle timed on a bounded sample (`cpu_baseline`: all host
cores, one independent oracle process per core; `single_core` inside it).
The default run also measures batch 8, both batches on the persistent NVFP4
decode kernel, the small-batch dense NVFP4 GEMV (8192 x 2048, batch 1 and 8),
the prefill sublayer and the BF16 batch-8 stack, and reports each under its
own key of the same line (`--no-extras` skips them).  `--impl reference` times only the oracle, on the
same workload and with the same `config`.
"""

from __future__ import annotations

import argparse
import json
import math
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
FUSED_MAX_LAYERS = 64  # sublayers per launch of the persistent NVFP4 decode kernel

WORKLOADS = {
    "stack47_b1_nvfp4": dict(cfg=1, batch=1, fmt="nvfp4"),
    "stack47_b8_nvfp4": dict(cfg=2, batch=8, fmt="nvfp4"),
    "stack47_b8_bf16": dict(cfg=3, batch=8, fmt="bf16"),
    "stack47_b16_nvfp4": dict(cfg=2, batch=16, fmt="nvfp4"),  # medium-batch path (9..64 tokens)
    "stack47_b64_nvfp4": dict(cfg=2, batch=64, fmt="nvfp4"),
    "prefill8192_nvfp4": dict(cfg=4, batch=8192, fmt="nvfp4", prefill=True),
    "dense_gemv_b1_nvfp4": dict(dense=True, batch=1, fmt="nvfp4"),  # 8192 x 2048 packed NVFP4 GEMV
    "dense_gemv_b8_nvfp4": dict(dense=True, batch=8, fmt="nvfp4"),
}
METRIC = "MoE decode µs/layer & effective HBM GB/s (% of roofline) at batch 1 and 8"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--layers", type=int, default=N_LAYERS,
                    help="sublayers in the stack (47 for the benchmark; fewer only for profiling captures)")
    ap.add_argument("--workload", default="stack47_b1_nvfp4", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="measure only --workload")
    ap.add_argument("--decode-kernel", default="chained", choices=["chained", "persistent"],
                    help="NVFP4 decode kernels of a 1..8-token --workload")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def workload_config(name: str, world: int, layers: int = N_LAYERS) -> dict:
    """The `config` object of a workload; both arms print exactly this."""
    wl = WORKLOADS[name]
    if wl.get("dense"):
        return {"workload": name, "batch": wl["batch"], "N": DENSE_N, "K": DENSE_K, "matrices": DENSE_MATS,
                "weights": "nvfp4", "parallelism": f"replicas x{world}",
                "l2": f"{DENSE_MATS} distinct matrices cycled (444 MB): larger than L2"}
    if wl.get("prefill"):
        return {"workload": name, "tokens": wl["batch"], "hidden": 2048, "experts": "256+1", "inter": 512,
                "top_k": 6, "weights": wl["fmt"], "parallelism": f"replicas x{world}",
                "l2": "every step streams all 257 experts' packed weights (455 MB) and 4 rotating 32 MB token "
                      "batches: far larger than L2"}
    return {"workload": name, "layers": layers, "batch": wl["batch"], "hidden": 2048, "experts": "256+1",
            "inter": 512, "top_k": 6, "weights": wl["fmt"], "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2: 16 rotating batches, >= 631 MB of weights touched per step out of "
                  f"{'21.4' if wl['fmt'] == 'nvfp4' else '76'} GB resident"}


def read_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    return json.load(open(path)) if os.path.exists(path) else {}


# ----------------------------------------------------------------------------- CPU oracle timing

_ORACLE_CHILD = r"""
import json, sys, time, os
sys.path.insert(0, os.environ["FLINT_ROOT"])
import numpy as np, torch
torch.set_num_threads(1)
import oracle as O, synth
cfg, batch, budget, seed_index = int(sys.argv[1]), int(sys.argv[2]), float(sys.argv[3]), int(sys.argv[4])
lw = O.layer_from_tensors(synth.gen_layer(cfg, 1, device="cpu"))
x = synth.gen_x(cfg, batch, index=seed_index)
y = O.bf16_bits_to_f64(x.view(torch.int16).numpy().view(np.uint16))
print("ready", flush=True)
sys.stdin.readline()
n = 0
t0 = time.perf_counter()
while True:
    lw.drop_cache()
    y = O.moe_layer(y, lw)["y"]
    n += 1
    if time.perf_counter() - t0 >= budget and n >= 2:
        break
dt = time.perf_counter() - t0
print(json.dumps({"layers": n, "seconds": dt}), flush=True)
"""


_DENSE_CHILD = r"""
import json, sys, time, os
sys.path.insert(0, os.environ["FLINT_ROOT"])
import numpy as np, torch
torch.set_num_threads(1)
import oracle as O, synth
N, K, batch, budget = int(sys.argv[1]), int(sys.argv[2]), int(sys.argv[3]), float(sys.argv[4])
d = synth.gen_dense(N, K, index=0, device="cpu")
codes, scales = d["codes"].numpy(), d["scales"].numpy()
x = O.bf16_bits_to_f64(synth.gen_dense_x(batch, K, index=0).view(torch.int16).numpy().view(np.uint16))
n = 0
t0 = time.perf_counter()
while True:
    O.dense_gemv(x, codes, scales, d["tensor_scale"])
    n += 1
    if time.perf_counter() - t0 >= budget and n >= 2:
        break
print(json.dumps({"calls": n, "seconds": time.perf_counter() - t0}), flush=True)
"""


def time_oracle_dense(batch: int, budget_s: float) -> dict:
    """The oracle's dense GEMV (dequantise the whole matrix, fp64 product) on one
    8192 x 2048 matrix, single-threaded, for about budget_s seconds: us per call."""
    env = dict(os.environ)
    env.update(FLINT_ROOT=ROOT, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _DENSE_CHILD, str(DENSE_N), str(DENSE_K), str(batch), str(budget_s)],
                       capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        raise RuntimeError(f"oracle child failed: {r.stderr[-2000:]}")
    res = json.loads(r.stdout.strip().splitlines()[-1])
    return dict(value=1e6 * res["seconds"] / res["calls"], unit="us/call", cores=1, kind="oracle",
                sample=f"{res['calls']} calls of the {DENSE_N}x{DENSE_K} dense GEMV at batch {batch}, one "
                       f"single-threaded numpy fp64 process, {res['seconds']:.1f} s")


def time_oracle(cfg: int, batch: int, fmt: str, budget_s: float, procs: int = 1) -> dict:
    """The oracle on a bounded sample: `procs` independent single-threaded processes, each
    chaining sublayers (the same seeded weights, its own input) for `budget_s` seconds after
    all are ready.  Returns the aggregate throughput as us per sublayer."""
    env = dict(os.environ)
    env.update(FLINT_ROOT=ROOT, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    kids = [subprocess.Popen([sys.executable, "-c", _ORACLE_CHILD, str(cfg), str(batch), str(budget_s), str(i)],
                             stdin=subprocess.PIPE, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                             env=env) for i in range(procs)]
    try:
        for k in kids:
            line = k.stdout.readline()
            if line.strip() != "ready":
                raise RuntimeError(f"oracle child failed: {k.stderr.read()[-2000:]}")
        for k in kids:  # start together
            k.stdin.write("go\n")
            k.stdin.flush()
        res = []
        for k in kids:
            out, err = k.communicate(timeout=900)
            if k.returncode != 0:
                raise RuntimeError(f"oracle child failed: {err[-2000:]}")
            res.append(json.loads(out.strip().splitlines()[-1]))
    finally:
        for k in kids:
            if k.poll() is None:
                k.kill()
    rate = sum(r["layers"] / r["seconds"] for r in res)  # sublayers per second, all processes together
    n = sum(r["layers"] for r in res)
    secs = max(r["seconds"] for r in res)
    return dict(value=1e6 / rate, unit="us/layer", cores=procs, kind="oracle",
                sample=f"{n} sublayers of the {fmt} stack at batch {batch} in {procs} independent "
                       f"single-threaded numpy fp64 process{'es' if procs > 1 else ''} over {secs:.1f} s")


def time_oracle_all(cfg: int, batch: int, fmt: str, budget_s: float) -> dict:
    """All host cores (one oracle process per core), with the single-core figure inside."""
    one = time_oracle(cfg, batch, fmt, budget_s, 1)
    cores = max(1, min(os.cpu_count() or 1, 64))
    if cores == 1:
        return one
    allc = time_oracle(cfg, batch, fmt, budget_s, cores)
    allc["single_core"] = {k: one[k] for k in ("value", "unit", "cores", "sample")}
    return allc


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
        time.sleep(0.3)

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

def _hash_files(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


CSRC = "moe_decode_router_gb300/csrc/"
SOURCES = {
    "fused": [CSRC + "decode_fused.cu", CSRC + "decode_common.cuh", CSRC + "flint_common.cuh"],
    "chain": [CSRC + "decode.cu", CSRC + "decode_common.cuh", CSRC + "flint_common.cuh"],
    "prefill": [CSRC + "prefill.cu", CSRC + "tc05.cuh", CSRC + "flint_common.cuh"],
    "medium": [CSRC + "medium.cu", CSRC + "decode_common.cuh", CSRC + "flint_common.cuh"],
    "dense": [CSRC + "dense.cu", CSRC + "decode_common.cuh", CSRC + "flint_common.cuh"],
}
TRAFFIC_FILES = {
    "fused": "profiles/decode_fused_dram.md",
    "chain": "profiles/decode_chain_dram.md",
    "medium": "profiles/decode_medium_dram.md",
    "dense": "profiles/dense_gemv_8192x2048.md",
    "prefill": "profiles/prefill8192_nvfp4_kernels.md",
}


def profiled_traffic(kind: str, workload: str):
    """DRAM bytes per sublayer (read + write) from the committed ncu summary of this
    path, as a ratio to the algorithmic bytes (decode) or as bytes (prefill); None if
    there is none for this workload or the kernel sources changed since."""
    path = os.path.join(ROOT, TRAFFIC_FILES[kind])
    if not os.path.exists(path):
        return None, None
    src = _hash_files(SOURCES[kind])
    for line in open(path):
        if line.startswith("flint-traffic "):
            kv = dict(t.split("=", 1) for t in line.split()[1:])
            if kv.get("workload") == workload and kv.get("source") == src:
                return kv, TRAFFIC_FILES[kind]
    return None, None


# ----------------------------------------------------------------------------- our arm

def build_stack(F, synth, torch, fmt: str, dev, n_layers: int):
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


def timed(torch, stream, fn, steps: int) -> float:
    """Device milliseconds of `steps` calls of fn(s), CUDA events on `stream`."""
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(steps):
        fn(s)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def max_over_ranks(torch, ms: float, world: int, dev) -> float:
    if world == 1:
        return ms
    import torch.distributed as tdist
    t = torch.tensor([ms], device=dev)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()


def measure_stack(F, synth, torch, name: str, layers, steps: int, warmup: int, world: int, dev, local: int,
                  persistent: bool = False) -> dict:
    """One decode-stack workload: device time, algorithmic bytes, roofline, e2e, clocks.
    persistent: NVFP4 weights on the persistent decode kernel instead of the chained kernels."""
    wl = WORKLOADS[name]
    F.set_decode_kernel(F.DECODE_PERSISTENT if persistent else F.DECODE_CHAINED)
    B = wl["batch"]
    fmt = F.W_NVFP4 if wl["fmt"] == "nvfp4" else F.W_BF16
    NL = len(layers)
    xs = [synth.gen_x(wl["cfg"], B, index=i, device=dev) for i in range(N_INPUTS)]
    ys = [torch.empty_like(x) for x in xs]
    ws = F.alloc_workspace(fmt, B, device=dev)

    # Algorithmic bytes per input: router + (distinct routed + shared) experts per sublayer.
    expert_bytes = NVFP4_EXPERT_BYTES if fmt == F.W_NVFP4 else BF16_EXPERT_BYTES
    ids = torch.empty((NL, B, 6), dtype=torch.int32, device=dev)
    bytes_per_input, uniq = [], []
    for i, x in enumerate(xs):
        F.decode_stack(layers, x, ys[i], ws, ids_per_layer=ids)
        torch.cuda.synchronize()
        idc = ids.cpu()
        u = [len(set(idc[l].flatten().tolist())) for l in range(NL)]
        uniq.extend(u)
        bytes_per_input.append(sum(ROUTER_BYTES + (n + 1) * expert_bytes for n in u))
    for i, x in enumerate(xs):  # BF16: one cached graph per input buffer (graphs bake in pointers)
        F.decode_stack(layers, x, ys[i], ws)
    torch.cuda.synchronize()
    assert F.device_error() == 0

    stream = torch.cuda.current_stream()
    for s in range(max(3, warmup)):
        F.decode_stack(layers, xs[s % N_INPUTS], ys[s % N_INPUTS], ws)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    ms = timed(torch, stream, lambda s: F.decode_stack(layers, xs[s % N_INPUTS], ys[s % N_INPUTS], ws), steps)
    barrier(world)
    clk = clocks.stop()
    err = F.device_error()

    # End to end through the C ABI: pinned host input -> device, stack, device -> pinned host.
    hx = [x.cpu().pin_memory() for x in xs]
    hy = torch.empty_like(hx[0]).pin_memory()
    xin = torch.empty_like(xs[0])
    yout = torch.empty_like(xs[0])

    def e2e_step(s):
        xin.copy_(hx[s % N_INPUTS], non_blocking=True)
        F.decode_stack(layers, xin, yout, ws)
        hy.copy_(yout, non_blocking=True)

    for s in range(max(3, warmup)):
        e2e_step(s)
    e2e_steps = max(10, steps // 2)
    e2e_ms = timed(torch, stream, e2e_step, e2e_steps) / e2e_steps

    ms = max_over_ranks(torch, ms, world, dev)
    ms_per_step = ms / steps
    total_bytes = sum(bytes_per_input[s % N_INPUTS] for s in range(steps))
    gbs = total_bytes * world / (ms / 1000.0) / 1e9
    peaks = read_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured (MEASURED_PEAKS.json hbm_gbs)" if peak else "fallback"
    peak = peak or 6800.0
    bytes_per_layer = total_bytes / steps / NL
    F.set_decode_kernel(F.DECODE_CHAINED)
    persistent = persistent and fmt == F.W_NVFP4
    kind = "fused" if persistent else ("medium" if B > 8 else "chain")
    prof, prof_src = profiled_traffic(kind, name)
    traffic = round(float(prof["ratio"]) * bytes_per_layer * NL) if prof else None
    # medium: 5 kernels per sublayer, plus the first sublayer's RMSNorm step
    launches = math.ceil(NL / FUSED_MAX_LAYERS) if persistent else (5 * NL + 1 if B > 8 else 3 * NL)
    return {
        "value": round(ms_per_step * 1000.0 / NL, 3),
        "unit": "us/layer",
        "ms_per_step": round(ms_per_step, 4),
        "effective_hbm_gbs": round(gbs, 1),
        "decode_kernel": "persistent" if persistent else ("medium" if B > 8 else "chained"),
        "roofline": {
            "kernel": ("decode_fused_kernel: one persistent launch = the whole 47-sublayer step"
                       if persistent else
                       "medium-batch step (logits over (8-token chunk, expert) units, routing tables, "
                       "expert-grouped gate/up and down, combine that also normalises the next sublayer's input: "
                       "5 kernels per sublayer plus the first sublayer's RMSNorm, PDL-chained, one CUDA graph)"
                       if B > 8 else
                       "decode step (router + gate/up + down per sublayer, PDL-chained, one CUDA graph)"),
            "bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(gbs / peak, 4), "peak_source": peak_src,
            "bytes_per_step": round(total_bytes / steps), "bytes_per_layer": round(bytes_per_layer),
            "traffic": traffic, "traffic_source": prof_src,
        },
        "e2e": {"value": round(e2e_ms * 1000.0 / NL, 3), "unit": "us/layer",
                "h2d_bytes_per_step": B * 2048 * 2, "d2h_bytes_per_step": B * 2048 * 2},
        "gpu_launches": steps * launches,
        "mean_unique_experts_per_layer": round(sum(uniq) / len(uniq), 2),
        "clocks": clk,
        "device_error_word": err,
    }


def prefill_flops(T: int) -> float:
    """Algorithmic FLOPs of one prefill sublayer: router GEMM plus gate/up and
    down GEMMs over the 6 T routed and T shared token-expert pairs."""
    H, E, I = 2048, 256, 512
    return 2.0 * T * E * H + 2.0 * 7 * T * (2 * I * H + H * I)


def measure_prefill(F, synth, torch, name: str, steps: int, warmup: int, world: int, dev, local: int) -> dict:
    wl = WORKLOADS[name]
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
    for s in range(max(3, warmup)):
        F.prefill_layer(L, xs[s % n_in], ys[s % n_in], ws)
    torch.cuda.synchronize()
    assert F.device_error() == 0
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    ms = timed(torch, stream, lambda s: F.prefill_layer(L, xs[s % n_in], ys[s % n_in], ws), steps)
    barrier(world)
    clk = clocks.stop()
    err = F.device_error()

    hx = [x.cpu().pin_memory() for x in xs]
    hy = torch.empty_like(hx[0]).pin_memory()
    xin = torch.empty_like(xs[0])
    yout = torch.empty_like(xs[0])

    def e2e_step(s):
        xin.copy_(hx[s % n_in], non_blocking=True)
        F.prefill_layer(L, xin, yout, ws)
        hy.copy_(yout, non_blocking=True)

    for s in range(3):
        e2e_step(s)
    e2e_steps = max(10, steps // 4)
    e2e_ms = timed(torch, stream, e2e_step, e2e_steps) / e2e_steps

    ms_per_step = max_over_ranks(torch, ms, world, dev) / steps
    flops = prefill_flops(T)
    tflops = flops * world / (ms_per_step / 1000.0) / 1e12
    peak = read_peaks().get("bf16_tflops_sustained")
    peak_src = "measured (MEASURED_PEAKS.json bf16_tflops_sustained)" if peak else "fallback"
    peak = peak or 1700.0
    prof, prof_src = profiled_traffic("prefill", name)
    return {
        "value": round(ms_per_step * 1000.0, 2),
        "unit": "us/layer",
        "ms_per_step": round(ms_per_step, 4),
        "tflops": round(tflops, 1),
        "roofline": {
            "kernel": "prefill sublayer (router GEMM, routing, grouped gate/up and down GEMMs, combine)",
            "bound": "tensor", "achieved": round(tflops, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(tflops / peak, 4), "peak_source": peak_src,
            "flops_per_layer": flops, "traffic": int(prof["bytes"]) if prof else None, "traffic_source": prof_src,
        },
        "e2e": {"value": round(e2e_ms * 1000.0, 2), "unit": "us/layer",
                "h2d_bytes_per_step": T * 2048 * 2, "d2h_bytes_per_step": T * 2048 * 2},
        "gpu_launches": steps * 7,
        "clocks": clk,
        "device_error_word": err,
    }


DENSE_N, DENSE_K, DENSE_MATS = 8192, 2048, 47


def measure_dense(F, synth, torch, B: int, steps: int, warmup: int, world: int, dev, local: int) -> dict:
    """The small-batch dense GEMV on packed NVFP4: an 8192 x 2048 matrix (the
    shape of a 4x-wide dense MLP projection of the 2048-wide model), 47 distinct
    matrices cycled so that the weights stream from HBM (444 MB > L2)."""
    mats = []
    for i in range(DENSE_MATS):
        d = synth.gen_dense(DENSE_N, DENSE_K, index=i, device=dev)
        mats.append(F.pack_dense(d["codes"], d["scales"], d["tensor_scale"], device=dev))
        torch.cuda.synchronize()
        mats[-1]._keepalive = None
    x = synth.gen_dense_x(B, DENSE_K, index=0, device=dev)
    y = torch.empty((B, DENSE_N), dtype=torch.bfloat16, device=dev)
    for s in range(max(3, warmup)):
        F.dense_gemv(mats[s % DENSE_MATS], x, y)
    torch.cuda.synchronize()
    assert F.device_error() == 0
    # One CUDA graph of 47 calls (one per matrix), as a model's forward would run
    # them: the time is the GPU's, not the host's launch rate.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(DENSE_MATS):
            F.dense_gemv(mats[i], x, y)
    graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    reps = max(3, steps // DENSE_MATS)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    ms = timed(torch, stream, lambda s: graph.replay(), reps)
    barrier(world)
    clk = clocks.stop()
    calls = reps * DENSE_MATS
    hx = x.cpu().pin_memory()
    hy = torch.empty((B, DENSE_N), dtype=torch.bfloat16).pin_memory()
    xin = torch.empty_like(x)

    def e2e_step(s):
        xin.copy_(hx, non_blocking=True)
        F.dense_gemv(mats[s % DENSE_MATS], xin, y)
        hy.copy_(y, non_blocking=True)

    for s in range(3):
        e2e_step(s)
    e2e_ms = timed(torch, stream, e2e_step, steps) / steps
    us = max_over_ranks(torch, ms, world, dev) / calls * 1000.0
    nbytes = DENSE_N * DENSE_K * 9 // 16
    gbs = nbytes * world / (us * 1e-6) / 1e9
    peak = read_peaks().get("hbm_gbs") or 6800.0
    prof, prof_src = profiled_traffic("dense", f"dense_gemv_b{B}_nvfp4")
    return {
        "workload": f"dense_gemv_{DENSE_N}x{DENSE_K}_b{B}_nvfp4", "value": round(us, 3), "unit": "us/call",
        "effective_hbm_gbs": round(gbs, 1),
        "roofline": {"kernel": "dense_gemv_kernel", "bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(gbs / peak, 4), "bytes_per_call": nbytes,
                     "traffic": int(prof["bytes"]) if prof else None, "traffic_source": prof_src},
        "e2e": {"value": round(e2e_ms * 1000.0, 3), "unit": "us/call", "h2d_bytes_per_step": B * DENSE_K * 2,
                "d2h_bytes_per_step": B * DENSE_N * 2},
        "gpu_launches": calls, "timing": "CUDA graph of 47 calls (one per distinct matrix), replayed",
        "clocks": clk, "device_error_word": F.device_error(),
    }


def dtype_of(fmt: str) -> str:
    return {"nvfp4": "nvfp4-w/bf16-a (f16 operands, f32 accumulate)", "bf16": "bf16 (f32 accumulate)"}[fmt]


def run_ours(args):
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
    name = args.workload
    wl = WORKLOADS[name]
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline

    extras = {}
    if wl.get("dense"):
        res = measure_dense(F, synth, torch, wl["batch"], args.steps, args.warmup, world, dev, local)
        res["ms_per_step"] = round(res["value"] / 1000.0, 6)
    elif wl.get("prefill"):
        res = measure_prefill(F, synth, torch, name, args.steps, args.warmup, world, dev, local)
    else:
        layers = build_stack(F, synth, torch, wl["fmt"], dev, args.layers)
        res = measure_stack(F, synth, torch, name, layers, args.steps, args.warmup, world, dev, local,
                            persistent=args.decode_kernel == "persistent" and wl["batch"] <= 8)
        if name == "stack47_b1_nvfp4" and not args.no_extras:
            # batch 8 on the same resident weights, and both batches on the persistent kernel
            extras["batch8"] = dict(workload="stack47_b8_nvfp4", **measure_stack(
                F, synth, torch, "stack47_b8_nvfp4", layers, max(10, args.steps // 4), args.warmup, world, dev,
                local))
            extras["persistent_b1"] = dict(workload="stack47_b1_nvfp4", **measure_stack(
                F, synth, torch, "stack47_b1_nvfp4", layers, args.steps, args.warmup, world, dev, local,
                persistent=True))
            extras["persistent_b8"] = dict(workload="stack47_b8_nvfp4", **measure_stack(
                F, synth, torch, "stack47_b8_nvfp4", layers, max(10, args.steps // 4), args.warmup, world, dev,
                local, persistent=True))
            # past the low-latency cap: the expert-grouped medium-batch kernels
            for b, div in ((16, 20), (64, 40)):
                extras[f"medium_b{b}"] = dict(workload=f"stack47_b{b}_nvfp4", **measure_stack(
                    F, synth, torch, f"stack47_b{b}_nvfp4", layers, max(10, args.steps // div), args.warmup, world,
                    dev, local))
        del layers
        F.release()
        torch.cuda.empty_cache()
        if name == "stack47_b1_nvfp4" and not args.no_extras:
            for b in (1, 8):
                extras[f"dense_gemv_b{b}"] = measure_dense(F, synth, torch, b, max(50, args.steps), args.warmup,
                                                          world, dev, local)
                torch.cuda.empty_cache()
            extras["prefill"] = dict(workload="prefill8192_nvfp4", **measure_prefill(
                F, synth, torch, "prefill8192_nvfp4", max(5, args.steps // 40), 3, world, dev, local))
            torch.cuda.empty_cache()
            layers = build_stack(F, synth, torch, "bf16", dev, args.layers)
            extras["bf16_batch8"] = dict(workload="stack47_b8_bf16", **measure_stack(
                F, synth, torch, "stack47_b8_bf16", layers, max(10, args.steps // 8), args.warmup, world, dev,
                local))
            del layers
            F.release()
            torch.cuda.empty_cache()

    out = {
        "metric": METRIC,
        "value": res["value"],
        "unit": res.get("unit", "us/layer"),
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": res["ms_per_step"],
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_of(wl["fmt"]),
        "data": "synthetic (seeded generator, random-init weights of the Flint MoE shapes)",
        "config": workload_config(name, world, args.layers),
    }
    out.update({k: v for k, v in res.items() if k not in ("value", "unit", "ms_per_step")})
    if want_cpu:
        try:
            if wl.get("dense"):
                out["cpu_baseline"] = time_oracle_dense(wl["batch"], args.cpu_seconds)
            elif wl.get("prefill"):
                out["cpu_baseline"] = time_oracle_prefill(wl["cfg"], wl["batch"])
            else:
                out["cpu_baseline"] = time_oracle_all(wl["cfg"], wl["batch"], wl["fmt"], args.cpu_seconds)
        except Exception as e:  # report, do not hide
            out["cpu_baseline"] = {"value": None, "error": str(e)[:300]}
        for key, ex in extras.items():
            if key.startswith("persistent") or key.startswith("dense") or key.startswith("medium"):
                continue  # the oracle is timed once per decode workload of the headline metric
            try:
                w2 = WORKLOADS[ex["workload"]]
                if w2.get("prefill"):
                    ex["cpu_baseline"] = time_oracle_prefill(w2["cfg"], w2["batch"])
                else:
                    ex["cpu_baseline"] = time_oracle(w2["cfg"], w2["batch"], w2["fmt"], args.cpu_seconds / 3)
            except Exception as e:
                ex["cpu_baseline"] = {"value": None, "error": str(e)[:300]}
    elif rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = {"value": None, "note": "timed at N=1 only"}
    out.update(extras)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        tdist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm (oracle)

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    name = args.workload
    wl = WORKLOADS[name]
    common = {
        "impl": "reference", "metric": METRIC, "unit": "us/layer", "n_gpus": world, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded generator, random-init weights of the Flint MoE shapes)",
        "config": workload_config(name, world, args.layers),
    }
    if wl.get("dense"):
        r = time_oracle_dense(wl["batch"], max(1.0, min(60.0, 2.0 * max(1, args.steps))))
        us = r["value"]
        common["unit"] = "us/call"
        print(json.dumps(dict(common, value=round(us, 1), steps=args.steps, warmup=0,
                              ms_per_step=round(us / 1000.0, 3), cpu_baseline=r,
                              e2e={"value": round(us, 1), "unit": "us/call", "h2d_bytes_per_step": 0,
                                   "d2h_bytes_per_step": 0})), flush=True)
        return
    if wl.get("prefill"):
        r = time_oracle_prefill(wl["cfg"], wl["batch"])
        us = r["value"]
        print(json.dumps(dict(common, value=round(us, 1), steps=1, warmup=0, ms_per_step=round(us / 1000.0, 3),
                              cpu_baseline=r,
                              e2e={"value": round(us, 1), "unit": "us/layer", "h2d_bytes_per_step": 0,
                                   "d2h_bytes_per_step": 0})), flush=True)
        return
    per_step_budget = max(0.5, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(wl["cfg"], wl["batch"], wl["fmt"], per_step_budget / 4)
    vals, samples = [], []
    for _ in range(args.steps):
        r = time_oracle(wl["cfg"], wl["batch"], wl["fmt"], per_step_budget)
        vals.append(r["value"])
        samples.append(r["sample"])
    us = statistics.mean(vals)
    print(json.dumps(dict(common, value=round(us, 1), steps=args.steps, warmup=args.warmup,
                          ms_per_step=round(us * args.layers / 1000.0, 3),
                          cpu_baseline={"value": round(us, 1), "unit": "us/layer", "cores": 1, "kind": "oracle",
                                        "sample": samples[-1] if samples else ""},
                          e2e={"value": round(us, 1), "unit": "us/layer", "h2d_bytes_per_step": 0,
                               "d2h_bytes_per_step": 0})), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
