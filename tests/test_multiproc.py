"""The multi-process host logic of bench.py, on CPU: two gloo ranks (world
size 2, rendezvous on 127.0.0.1).

The attention path shards by (batch, head) with no exchange, so a run on N
GPUs is N replicas: each rank times its own copy of the workload, the ranks
meet at barriers around the timed region, the reported time is the maximum
over ranks and the reported rate counts all ranks' work.  These tests check
that machinery without a GPU: rank and world from the environment, the
max-over-ranks reduction, the barrier, and that only rank 0 would print.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    r, w = bench.dist_init("gloo")
    import time

    # ranks reach the barrier at different times; both leave it together
    time.sleep(0.2 * r)
    bench.barrier()
    t_after = time.time()
    ms = 10.0 + 5.0 * r            # each rank's own timing
    worst = bench.reduce_max(ms)   # the bench reports the slowest rank
    out.put((r, w, worst, t_after))
    import torch.distributed as dist

    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_reduce_and_barrier():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [r for r, *_ in res] == [0, 1]
    assert all(w == 2 for _, w, _, _ in res)
    assert all(worst == 15.0 for _, _, worst, _ in res)     # max over ranks, seen by both
    # the barrier released both ranks after the later one (0.2 s) arrived
    assert abs(res[0][3] - res[1][3]) < 0.15


def test_single_process_defaults():
    import bench

    os.environ.pop("WORLD_SIZE", None)
    assert bench.dist_init("gloo") == (0, 1)
    assert bench.reduce_max(3.5) == 3.5
    bench.barrier()   # a no-op without a process group


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched the way N > 1 runs are (torchrun,
    two ranks, gloo on CPU): rank 0 alone times the oracle and prints one JSON
    line; the other rank exits 0 without work."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(root, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "bf16_b4_h12_n512_d64_causal", "--steps", "1",
           "--warmup", "3"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=240, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
