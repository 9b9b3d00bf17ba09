"""The N > 1 path of bench.py on CPU: two gloo ranks run independent
replicas (their own seeds, no exchange of data) and meet only to take the
slowest rank's time and the sum of the units they processed."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from paged_attention_int8_gb300 import inputs
        spec = bench.replica_spec(inputs.TINY_DECODE, rank)
        w = inputs.make_workload(spec)
        units = bench.step_work(w)["step_bytes"]
        ms, total = bench.reduce_over_ranks(1.0 + rank, units, torch.device("cpu"))
        q.put((rank, spec.seed, units, ms, total, w.q.sum().item()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_are_independent_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=180) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    (r0, seed0, u0, ms0, tot0, qs0), (r1, seed1, u1, ms1, tot1, qs1) = out
    assert (r0, r1) == (0, 1)
    assert seed0 != seed1 and qs0 != qs1          # different data on each rank
    assert ms0 == ms1 == pytest.approx(2.0)        # the slowest rank's time
    assert tot0 == tot1 == pytest.approx(u0 + u1)  # units of all ranks
