"""The bench's N > 1 host logic on the CPU: two ranks over gloo (127.0.0.1), the barrier, the
max-over-ranks timing and the whole-job GB/s of independent replicas (weak scaling), and the
reference arm's rule that only rank 0 works and prints."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier()
        local_ms = 10.0 + 5.0 * rank           # rank 1 is the slower one
        total = bench.max_over_ranks(local_ms)
        value = bench.whole_job_gbs(world, 6 << 20, 260, total)
        bench.rank_barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"total_ms": total, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_replicas(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn",
                       join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert res[0] == res[1]                              # every rank agrees
    assert res[0]["total_ms"] == 15.0                    # the slower rank's timed region
    # both replicas' bytes over the slowest rank's time
    assert res[0]["value"] == pytest.approx(2 * (6 << 20) * 260 / 15e-3 / 1e9)


def test_single_process_helpers_are_identities():
    sys.path.insert(0, ROOT)
    import bench

    bench.rank_barrier()
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_gbs(1, 1000, 10, 1.0) == pytest.approx(1000 * 10 / 1e-3 / 1e9)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
