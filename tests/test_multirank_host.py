"""The N > 1 host logic of bench.py on CPU with world_size-2 gloo ranks:
the step time is the max over ranks, the throughput counts every rank's
bytes, every rank draws its own inputs, and the reference arm under
torchrun prints exactly one line (rank 0) while the other rank exits 0."""
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


def _rank_main(rank, world, port, q):
    import torch
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    local = [3.25, 7.5][rank]
    got = bench.reduce_max_over_ranks(local, world, torch.device("cpu"))
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()
    q.put((rank, got, bench.rank_seed_offset(rank)))


def test_max_over_ranks_and_seeds_with_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [7.5, 7.5]            # both ranks see the slowest rank's time
    assert res[0][2] == 0 and res[1][2] != res[0][2]    # rank 0 keeps the seeds, rank 1 its own batch


def test_whole_job_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_gbs(2.0e9, 1.0, 1)
    assert bench.whole_job_gbs(2.0e9, 1.0, 2) == pytest.approx(2 * one)
    assert bench.reduce_max_over_ranks(4.0, 1, None) == 4.0


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
                        "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_all_cores_oracle_baseline_spawns_independent_processes():
    """The all-cores CPU baseline: spawned processes, each on its own slice;
    its bytes per second add up over the processes."""
    sys.path.insert(0, ROOT)
    import bench
    d = bench.cpu_baseline_all_cores(min_seconds=0.3, processes=2)
    assert d["kind"] == "oracle" and d["cores"] == 2 and d["value"] > 0
    assert "2 processes" in d["sample"]
