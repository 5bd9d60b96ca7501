"""bench.py's multi-rank plumbing (barrier, max over ranks) on two gloo ranks, CPU only."""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, lr = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    got = bench.max_over_ranks(dist, 10.0 + 5.0 * r)
    bench.barrier(dist)
    q.put((r, got))
    dist.destroy_process_group()


def test_max_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 15.0, 1: 15.0}


def test_single_rank_needs_no_process_group():
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5


def test_reference_arm_prints_the_contract_line():
    """``bench.py --impl reference`` (the float64 oracle on the host cores) prints one JSON line
    with the keys the driver reads."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    p = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, env={**os.environ, "RANK": "0", "WORLD_SIZE": "1"})
    assert p.returncode == 0, p.stderr[-2000:]
    line = json.loads(p.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["higher_is_better"] is False
    assert line["steps"] == 2 and line["warmup"] == 3 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"] and "workload" in line["config"]


def test_reference_arm_other_ranks_do_no_work():
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    p = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True,
                       timeout=120, env={**os.environ, "RANK": "1", "WORLD_SIZE": "2"})
    assert p.returncode == 0 and p.stdout.strip() == ""
