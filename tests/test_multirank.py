"""World-size-2 runs of the bench's multi-rank path on CPU (gloo).

The decode path shards by sequence with no exchange between ranks, so the
multi-rank logic is the bench's own: every rank builds its own seeded units,
the step time is the slowest rank's (all-reduce MAX after a barrier), and the
whole-job value is the units of all ranks over that time (weak scaling).
Under torchrun the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    from compressed_kv_cache_vector_gb300 import synth
    dist.barrier()
    ms = bench.max_over_ranks([3.0, 5.0][rank], dist, "cpu")
    value = bench.weak_value(1000.0, world, ms)
    seed = synth.seed_for("c3-llama8b-128k-32layers", rank, 0, 0, 0)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": value, "seed": int(seed)}, f)
    dist.destroy_process_group()


def test_slowest_rank_time_and_weak_scaling_value(tmp_path):
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    r = [json.load(open(tmp_path / f"r{i}.json")) for i in range(2)]
    assert r[0]["ms"] == r[1]["ms"] == 5.0          # both ranks report the slowest rank's time
    assert r[0]["value"] == pytest.approx(1000.0 * 2 / 5e-3)
    assert r[0]["seed"] != r[1]["seed"]              # each rank builds its own units


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, None, "cpu") == 2.5
    assert bench.weak_value(10.0, 1, 1.0) == pytest.approx(1e4)


def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--config", "c1", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT, env=env)
    assert p.returncode == 0, p.stderr[-3000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_gpus_flag_outside_a_launcher_starts_the_ranks_itself():
    # `bench.py --gpus 2` with no WORLD_SIZE in the environment runs itself as
    # two ranks under torch.distributed.run (here the CPU reference arm).
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
           "--config", "c1", "--steps", "1", "--warmup", "0"]
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env["OMP_NUM_THREADS"] = "1"
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT, env=env)
    assert p.returncode == 0, p.stderr[-3000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["cpu_baseline"]["cores"] >= 1 and "processes" in d["cpu_baseline"]["sample"]
