"""The benchmark's multi-rank logic on the CPU: two gloo ranks (the GPU runs use NCCL with one rank per GPU)."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks(1.5 + 3.0 * rank)  # the slowest rank's time wins
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"rank": rank, "max": got}, f)


def test_max_over_ranks_with_two_gloo_ranks(tmp_path):
    port = 29500 + (os.getpid() % 1000)
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    assert [r["max"] for r in res] == [4.5, 4.5]


def test_max_over_ranks_is_identity_without_a_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.25) == 2.25


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "w4a16_sym",
                        "--steps", "2", "--warmup", "0"], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if rank == 0:
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    else:
        assert lines == []
