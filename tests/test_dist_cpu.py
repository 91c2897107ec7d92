"""The bench's multi-rank path on the CPU (gloo, world size 2).

The path does not shard across GPUs ("replicas only"): with N ranks every
rank runs the whole workload on its own GPU, the slowest rank's time counts,
and rank 0 alone prints the line.  What runs without a GPU is checked here:
the max-over-ranks reduction and the weak-scaling throughput with two gloo
ranks, and the CPU reference arm launched the way the driver launches N > 1
(torch.distributed.run), where rank 0 alone prints and the others exit 0.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    # rank r reports step times (ms) 10 + r and 20 - r: the maxima are 11 and 20
    got = bench.max_over_ranks([10.0 + rank, 20.0 - rank])
    value = bench.weak_scaling_value(world, 4.4e12, got[0] * 1e-3)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got, "value": value}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_with_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        d = json.load(open(tmp_path / f"rank{r}.json"))
        assert d["max"] == [11.0, 20.0]
        assert d["value"] == pytest.approx(2 * 4.4e12 / 11e-3 / 1e12)


def test_max_over_ranks_without_a_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(port), "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
