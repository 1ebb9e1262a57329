"""The benchmark's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.  Each rank runs
its own batch; the only cross-rank traffic is the reduction of timings (max) and work (sum)."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = {"step_ms": 10.0 + rank, "fwd_ms": 2.0 * (rank + 1), "flops": 1e12 * (rank + 1)}
    out = bench.reduce_over_ranks(local, world)
    q.put((rank, out))
    dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        assert results[rank]["step_ms"] == 11.0     # slowest rank
        assert results[rank]["fwd_ms"] == 4.0
        assert results[rank]["flops"] == 3e12       # total work


def test_reference_arm_other_ranks_do_nothing():
    import bench
    args = bench.parse_args(["--impl", "reference"])
    assert bench.run_reference(args, world=2, rank=1) == 0
