"""The benchmark's multi-rank host logic on two CPU ranks (gloo, world size 2):
every rank runs its own batch (its own seed and inputs), the step time is the
slowest rank's, the whole-job value counts every rank's tokens, and under
torchrun only rank 0 runs and prints the reference arm. No GPU is used."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        b = _bench()
        from fixed_state_recurrence_phi_b300.inputs import torch_qkv
        # each rank's own batch
        seed = b.rank_seed(2, rank)
        q, _, _ = torch_qkv(1, 2, 64, 16, 64, "f32", seed, 0, "cpu")
        sums = [torch.zeros(1, dtype=torch.float64) for _ in range(ws)]
        dist.all_gather(sums, q.double().sum().reshape(1))
        # the slowest rank's time, seen by every rank
        local_ms = [3.0, 5.0][rank]
        slowest = b.max_over_ranks(local_ms, ws, "cpu")
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"seed": seed, "slowest": slowest, "sums": [float(x) for x in sums]}, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    r = [json.load(open(tmp_path / f"rank{k}.json")) for k in range(2)]
    assert r[0]["seed"] != r[1]["seed"]
    assert r[0]["sums"][0] != r[0]["sums"][1]           # different batches
    assert r[0]["sums"] == r[1]["sums"]
    assert r[0]["slowest"] == r[1]["slowest"] == 5.0    # max over ranks
    b = _bench()
    assert b.weak_scaling_value(2, 8192, 5.0) == pytest.approx(2 * 8192 / 5e-3)
    assert b.weak_scaling_value(1, 8192, 5.0) == pytest.approx(8192 / 5e-3)


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r1 = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                         "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    env0 = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r0 = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                         "--warmup", "0"], env=env0, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r0.returncode == 0
    lines = [l for l in r0.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
