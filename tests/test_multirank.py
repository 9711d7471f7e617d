"""The benchmark's multi-process path on CPU (gloo, world size 2).

The path does not shard: `bench.py --gpus N` runs N independent replicas
(one process per GPU), joined only by a barrier and the maximum of the ranks'
device times, and rank 0 alone prints the JSON line.  These tests run that
host logic as two gloo ranks on 127.0.0.1, without a GPU.
"""

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_env(rank, world, port):
    env = dict(os.environ)
    env.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), LOCAL_RANK=str(rank),
               WORLD_SIZE=str(world), CUDA_VISIBLE_DEVICES="")
    return env


RANK_SCRIPT = r"""
import torch, torch.distributed as tdist
import bench
world, rank, local = bench.dist_env()
tdist.init_process_group("gloo")
# each replica timed a different device time; the job's time is the slowest
ms = bench.max_over_ranks(torch, 1.5 + rank, world, torch.device("cpu"))
bench.barrier(world)
print("RESULT", rank, ms, flush=True)
tdist.destroy_process_group()
"""


def test_max_over_ranks_and_barrier_on_two_gloo_ranks():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", RANK_SCRIPT], cwd=ROOT, env=_rank_env(r, 2, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    got = sorted(tuple(line.split()[1:]) for o in outs for line in o.splitlines() if line.startswith("RESULT"))
    assert got == [("0", "2.5"), ("1", "2.5")]


def test_reference_arm_prints_only_on_rank_0():
    # rank 1 of a 2-process run exits at once without output
    env = _rank_env(1, 2, _free_port())
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "0", "--workload", "dense_gemv_b1_nvfp4"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=180)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_arm_under_torchrun_two_ranks():
    # launched as the driver launches a 2-GPU run: one JSON line, from rank 0, with n_gpus = 2
    port = _free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
                        "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload",
                        "dense_gemv_b1_nvfp4"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["config"]["parallelism"] == "replicas x2"
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
