"""bench.py's multi-GPU path is N independent replicas (the round does not
shard): each rank decodes its own region and the job rate is every rank's
tokens over the slowest rank's timed seconds.  The aggregation runs here as
two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import datetime
    import sys
    import torch.distributed as dist
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    try:
        # rank r: 1.5 + r seconds, 100 * (r + 1) tokens
        secs, toks = bench.replica_totals(1.5 + rank, 100 * (rank + 1), torch.device("cpu"))
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{secs} {toks}\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replica_totals_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
        assert p.exitcode == 0
    for r in range(world):
        secs, toks = open(tmp_path / f"rank{r}.txt").read().split()
        assert float(secs) == 2.5          # the slowest rank's time
        assert int(toks) == 100 + 200      # every rank's tokens
