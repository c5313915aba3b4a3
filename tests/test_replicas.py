"""The N > 1 host logic of bench.py, on CPU with world-size-2 gloo process
groups: each rank runs an independent replica (the product needs no
collective), the job's step time is the largest over the ranks, the job's
throughput counts every replica's bytes, and rank 0 alone prints."""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # rank r timed its replica at (1 + r) ms per step and its end-to-end
        # step at (5 - r) ms: the job takes the slowest of each
        ms, e2e = bench.max_over_ranks(dist, [1.0 + rank, 5.0 - rank])
        dist.barrier()
        gbs = bench.job_gbs(world, 2.0e9, ms)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "e2e": e2e, "gbs": gbs}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_world2(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for g in got:  # every rank sees the same job figures
        assert g["ms"] == 2.0 and g["e2e"] == 5.0
        # two replicas of 2 GB each in 2 ms: 2000 GB/s for the job
        assert abs(g["gbs"] - 2000.0) < 1e-9


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, [3, 4.5]) == [3.0, 4.5]
    assert abs(bench.job_gbs(1, 1.0e9, 1.0) - 1000.0) < 1e-9


def test_reference_arm_prints_on_rank_0_only():
    """Under torchrun only rank 0 times the oracle; other ranks exit 0 silent."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == ""
