"""The N > 1 frame of the benchmark on CPU: world-size-2 ``gloo`` ranks go
through bench.py's timed region (barrier + synchronize on both sides) and its
max-over-ranks reduction; the whole-job figure sums every replica's bytes over
the slowest rank's time. The attention path itself has no exchange step, so
each rank is an independent replica and nothing else crosses ranks. No GPU."""
import json
import os
import socket
import subprocess
import sys
import time

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir, delays):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    entered = time.time()
    time.sleep(delays["enter"][rank])         # ranks reach the region at different times
    record = {"entered": entered}

    def run():
        record["run_start"] = time.time()
        time.sleep(delays["work"][rank])
        record["run_end"] = time.time()
        return 1e3 * delays["work"][rank]      # this rank's "timed milliseconds"

    own_ms = bench.timed_region(dist, lambda: None, run)
    record["left"] = time.time()
    record["own_ms"] = own_ms
    record["max_ms"] = bench.max_over_ranks(dist, own_ms)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(record, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time(tmp_path):
    world = 2
    delays = {"enter": [0.0, 0.4], "work": [0.05, 0.25]}
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path), delays), nprocs=world,
             join=True)
    recs = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    # both ranks get the slower replica's time
    assert [r["own_ms"] for r in recs] == pytest.approx([50.0, 250.0])
    assert all(r["max_ms"] == pytest.approx(250.0) for r in recs)
    # the barrier in front: no rank starts its timed work before the late rank arrives
    late_arrival = recs[1]["entered"] + delays["enter"][1]
    assert all(r["run_start"] >= late_arrival - 0.02 for r in recs)
    # the barrier behind: no rank leaves before the slowest one has finished
    assert all(r["left"] >= recs[1]["run_end"] - 0.02 for r in recs)


def test_whole_job_value_is_weak_scaling_sum():
    sys.path.insert(0, ROOT)
    import bench
    per_step, ms = 150e6, 0.05
    one = bench.whole_job_gbs(1, per_step, ms)
    assert one == pytest.approx(3000.0)
    assert bench.whole_job_gbs(4, per_step, ms) == pytest.approx(4 * one)
    assert bench.max_over_ranks(None, 1.25) == 1.25   # one rank: its own time


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    t0 = time.time()
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""                   # only rank 0 prints
    assert time.time() - t0 < 60                    # and rank 1 times nothing
