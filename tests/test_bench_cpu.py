"""Host-side logic of bench.py on CPU: the reference (oracle) arm prints one
JSON line with the contract's keys, and under torchrun with two gloo ranks
only rank 0 prints while both ranks exit 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _env():
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""
    env["MASTER_ADDR"] = "127.0.0.1"
    return env


def test_reference_arm_single_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=_env())
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "config", "cpu_baseline", "e2e", "impl"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_two_gloo_ranks():
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node=2", "--master-addr=127.0.0.1", "--master-port=29731",
                        "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                        "--gpus", "2"], cwd=ROOT, capture_output=True, text=True, timeout=900,
                       env=_env())
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert json.loads(lines[0])["n_gpus"] == 2


def test_max_over_ranks_with_gloo():
    code = r"""
import os, sys, torch, torch.distributed as dist
sys.path.insert(0, os.getcwd())
import bench
dist.init_process_group("gloo")
r = dist.get_rank()
v = bench.reduce_max(float(r + 1) * 1.5, dist.get_world_size())
bench.barrier(dist.get_world_size())
assert v == 3.0, v
dist.destroy_process_group()
"""
    path = os.path.join(ROOT, "_build", "maxranks.py")
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w") as f:
        f.write(code)
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node=2", "--master-addr=127.0.0.1", "--master-port=29733",
                        path], cwd=ROOT, capture_output=True, text=True, timeout=300, env=_env())
    assert r.returncode == 0, r.stderr[-3000:]


def test_gpus_flag_spawns_ranks_without_torchrun():
    # --gpus 2 outside torchrun relaunches itself with two ranks
    env = _env()
    env["MASTER_PORT"] = "29737"
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--gpus", "2", "--format", "3"], cwd=ROOT,
                       capture_output=True, text=True, timeout=900, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["config"]["format"] == "UE5M3-b32"
    assert d["ms_per_step_extrapolated"] is True
