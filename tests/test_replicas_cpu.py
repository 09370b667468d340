"""bench.py's multi-process host logic at world size 2, on CPU with gloo.

The hot path shards into independent replicas (no data-path collective), so
what runs across ranks is bookkeeping: each rank reads its place from the
launcher's environment, the whole-job figure sums the units of all ranks and
divides by the slowest rank's time, and the reference arm runs on rank 0
only (the other ranks exit 0 without work)."""
import io
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, l = bench.dist_env()
        # rank i: 0.5 + i seconds for 10 (i + 1) units
        t, u = bench.aggregate(0.5 + rank, 10.0 * (rank + 1), w)
        res = {"env": (w, r, l), "time": t, "units": u}
        if rank == 1:
            class A:
                gpus, steps, warmup = world, 3, 3
            buf = io.StringIO()
            with redirect_stdout(buf):
                res["ref_rc"] = bench.run_reference(A())
            res["ref_out"] = buf.getvalue()
        dist.barrier()
        out.put((rank, res))
    finally:
        dist.destroy_process_group()


def test_two_replicas_aggregate_and_reference_rank_gate():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert got[r]["env"] == (2, r, r)
        assert got[r]["time"] == 1.5     # the slowest rank
        assert got[r]["units"] == 30.0   # all ranks' units
    assert got[1]["ref_rc"] == 0 and got[1]["ref_out"] == ""
