"""The multi-rank path of bench.py on the CPU: two gloo ranks (processes
started with spawn), each a replica of the path with its own sequences.  The
only collective is the end-of-run reduction: tokens are summed over ranks
and the elapsed time is the maximum over ranks.  No GPU is touched."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    ws, r, _ = bench.dist_setup()
    assert (ws, r) == (world, rank) and dist.get_backend() == "gloo"
    # each replica drafted its own sequences: rank r, 100*(r+1) tokens in (10 + r) ms
    tokens, ms = bench.aggregate(100.0 * (rank + 1), 10.0 + rank, ws)
    bench.barrier(ws)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{tokens} {ms}\n")
    dist.destroy_process_group()


def test_two_rank_reduction(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for rank in range(world):
        tokens, ms = map(float, open(tmp_path / f"rank{rank}.txt").read().split())
        assert tokens == 300.0        # 100 + 200: whole-job tokens
        assert ms == 11.0             # the slowest rank's time


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate(123.0, 4.5, 1) == (123.0, 4.5)
