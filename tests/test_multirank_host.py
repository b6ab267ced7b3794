"""Host logic of the multi-GPU bench path, run as gloo ranks on the CPU: the
path shards by (sequence, kv head) with no exchange, so `bench.py --gpus N`
runs N independent replicas and only its timing is collective (barrier, then
the largest time over ranks). The reference arm runs on rank 0 alone."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.5], dist)
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(",".join(repr(x) for x in got))


def test_max_over_ranks_gloo_two_ranks(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        vals = [float(x) for x in (tmp_path / f"rank{r}.txt").read_text().split(",")]
        assert vals == [2.0, 10.0, 3.5]   # every rank sees the slowest replica's times


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1, 2.5]) == [1.0, 2.5]


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert res.returncode == 0
    assert res.stdout.strip() == ""


def test_gpus_flag_starts_that_many_ranks():
    # Without WORLD_SIZE, `bench.py --gpus 2` starts two ranks itself
    # (torch.distributed.run on 127.0.0.1). On this host neither rank finds a
    # GPU, so each reports its rank and the world size and the run fails.
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1",
                          "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode != 0
    assert "rank 0 of 2: no CUDA device" in res.stderr and "rank 1 of 2: no CUDA device" in res.stderr


def test_gpus_flag_must_match_world_size():
    env = dict(os.environ, RANK="0", WORLD_SIZE="2", LOCAL_RANK="0")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "4", "--steps", "1"],
                         env=env, capture_output=True, text=True, timeout=120)
    assert res.returncode == 2 and "WORLD_SIZE=2" in res.stderr
