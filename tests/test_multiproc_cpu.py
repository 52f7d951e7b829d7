"""Host logic of the multi-replica bench path, on CPU with gloo, world size 2.

The attention path shards into independent units, so ``bench.py --gpus N``
runs N replicas with no collective on the data path.  What remains on the
host is the rendezvous, the barrier around the timed region and the
max-over-ranks reduction of the step time; this test runs exactly those
helpers in two gloo processes.
"""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    ws, r, local = bench.dist_setup()
    assert dist.get_backend() == "gloo"
    bench.barrier(ws)
    # Rank r "measured" 10 + r ms; every rank must see the slowest one.
    t = bench.max_over_ranks(10.0 + r, ws)
    bench.barrier(ws)
    out.put((r, ws, local, t))
    dist.destroy_process_group()


def test_two_rank_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2, 0, 11.0), (1, 2, 1, 11.0)]


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)  # no-op without a process group


@pytest.mark.parametrize("ws", [1, 2, 4])
def test_reference_arm_only_rank0_prints(ws, capsys, monkeypatch):
    """Under torchrun every rank but 0 exits without work in the reference arm."""
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup, gpus = 1, 3, ws

    for rank in range(1, ws):
        bench.run_reference(A, ws, rank)
    assert capsys.readouterr().out == ""
