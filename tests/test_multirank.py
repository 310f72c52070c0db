"""The N > 1 bench path on CPU: two gloo ranks, each a full replica with its
own tokens; the whole-job value is all ranks' units over the slowest rank's
time, and the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist = bench.init_dist(world, "gloo")
    secs = [2.0, 3.0][rank]
    value, t = bench.aggregate(100.0, secs, dist)
    mx = bench.reduce_max(float(rank), dist)
    # the reference arm: rank 1 returns at once without touching the oracle
    ref_rc = bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])) \
        if rank == 1 else 0
    q.put((rank, value, t, mx, ref_rc))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, t, mx, ref_rc in out:
        assert t == 3.0                       # slowest rank
        assert value == pytest.approx(200.0 / 3.0)
        assert mx == 1.0
        assert ref_rc == 0
