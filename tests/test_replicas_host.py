"""The multi-GPU path is independent replicas (no data exchange): the host side that combines ranks, run as
two gloo processes on the CPU."""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import contextlib
    import io

    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup()
        step = 1.0 + 0.25 * r                       # each rank's own step time
        worst = bench.max_over_ranks(step, dist, device="cpu")
        value = bench.replica_throughput(w, 1024, worst)
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.emit({"value": value, "rank": r}, r)
        q.put((r, w, local, worst, value, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_print_once():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, local, worst, value, printed) in enumerate(out):
        assert (rank, world, local) == (r, 2, r)
        assert worst == 1.25                       # the slower rank's step time, on both ranks
        assert value == pytest.approx(2 * 1024 / 1.25)
        if rank == 0:
            assert json.loads(printed)["value"] == pytest.approx(value)
        else:
            assert printed == ""
