"""The multi-process (N > 1) host logic of bench.py, run as two gloo ranks on CPU.

Attention shards by batch with no data exchange: every rank runs the same
workload shape on its own seeded batch, and the only collective is the
timing reduction (maximum over ranks) before rank 0 reports the units of all
ranks over that time.  These tests run the same helpers bench.py uses, in two
real processes joined by a gloo process group on 127.0.0.1.
"""
import hashlib
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    import seeded_inputs as si

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # each rank's own prefill and decode batch (small shapes of the bench's recipes)
        xp = si.prefill_inputs(1, 2, 64, 64, bench.rank_seed(1002, rank), qk_std=3.0)
        xd = si.decode_inputs(2, 2, 64, bench.rank_seed(1004, rank), 16, 64)
        digest = [hashlib.sha256(xp.Q.bits.tobytes()).hexdigest(),
                  hashlib.sha256(xd.seqlens.tobytes()).hexdigest()]
        digests = [None] * world
        dist.all_gather_object(digests, digest)
        # per-rank timings: rank r is slowest on entry r % 3
        times = [1.0, 1.0, 1.0]
        times[rank % 3] = 2.0 + rank
        reduced = bench.max_over_ranks(times, dist, torch.device("cpu"))
        rate = bench.whole_job_rate(world, 100.0, reduced[0])
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"digests": digests, "reduced": reduced, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_reduce(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    # both ranks saw the same gathered digests, and the two batches differ
    assert res[0]["digests"] == res[1]["digests"]
    assert res[0]["digests"][0] != res[0]["digests"][1]
    # the timing reduction is the element-wise maximum, identical on every rank
    expected = [2.0, 3.0, 1.0]
    assert res[0]["reduced"] == expected and res[1]["reduced"] == expected
    # whole-job rate: units of all ranks over the slowest rank's time
    assert res[0]["rate"] == pytest.approx(world * 100.0 / 2.0)


def test_rank_seed_is_distinct_and_rank0_keeps_base_seed():
    sys.path.insert(0, ROOT)
    import bench
    seeds = [bench.rank_seed(1002, r) for r in range(8)]
    assert seeds[0] == 1002
    assert len(set(seeds)) == 8
    # no rank's seed collides with another workload's base seed (1001..1005)
    assert not (set(seeds[1:]) & set(range(1001, 1006)))


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([0.5, 2.0], None, torch.device("cpu")) == [0.5, 2.0]
    assert bench.whole_job_rate(1, 10.0, 2.0) == 5.0


def test_launch_percentiles_nearest_rank():
    import bench
    p = bench.launch_percentiles([0.4, 0.1, 0.3, 0.2] + [0.25] * 16)
    assert p["us_p50"] == pytest.approx(250.0)
    assert p["us_p95"] == pytest.approx(300.0)
    one = bench.launch_percentiles([0.5])
    assert one == {"us_p50": 500.0, "us_p95": 500.0}


def test_bench_gpus_2_starts_two_ranks_itself():
    """`bench.py --gpus 2` with no launcher in the environment starts two ranks
    (torch.distributed.run on 127.0.0.1); --dry-run stops before any CUDA call.
    Each rank reports its own seed and input digest, and the timing reduction
    is the maximum over both ranks."""
    import subprocess
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--dry-run"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["dry_run"] is True and d["n_gpus"] == 2
    ranks = sorted(d["ranks"], key=lambda x: x["rank"])
    assert [x["rank"] for x in ranks] == [0, 1]
    assert ranks[0]["seed"] != ranks[1]["seed"]
    assert ranks[0]["q_sha256"] != ranks[1]["q_sha256"]
    assert d["max_time_over_ranks"] == 2.0


def test_bench_gpus_must_match_the_launcher():
    import subprocess
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--dry-run"],
                       capture_output=True, text=True, timeout=120, cwd=ROOT, env=env)
    assert r.returncode != 0 and "does not match WORLD_SIZE" in r.stderr
