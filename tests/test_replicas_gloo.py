"""The multi-GPU path is replicas: each process runs its own copy of the
workload on its own GPU and the processes only agree on timing.  These
world_size-2 tests run that host logic over gloo on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.cpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _child(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    d = bench.Dist()
    d.init("gloo")
    # rank r: 10*(r+1) ms for (r+1) GB
    t, b, gbs = bench.aggregate(d, 10.0 * (rank + 1), 1e9 * (rank + 1))
    d.barrier()
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    ref = bench.run_reference(args, d) if rank != 0 else "skipped"
    d.close()
    q.put((rank, t, b, gbs, ref))


def test_replica_aggregation_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_child, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    for rank, t, b, gbs, ref in res:
        assert t == 20.0                     # slowest replica's time
        assert b == 3e9                      # all replicas' bytes
        assert gbs == pytest.approx(3e9 / 20e-3 / 1e9)
        if rank != 0:
            assert ref is None               # only rank 0 runs the reference arm


def test_single_process_aggregation_is_identity():
    import bench
    d = bench.Dist()
    assert d.world == 1 or os.environ.get("WORLD_SIZE")
    t, b, gbs = bench.aggregate(bench.Dist(), 4.0, 8e9)
    assert (t, b) == (4.0, 8e9) and gbs == pytest.approx(2000.0)
