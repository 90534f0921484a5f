"""The N > 1 benchmark path on CPU: two gloo ranks, each timing its own replica,
agree on the max over ranks (no GPU, no collective on the data path)."""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.0])
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, out))


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 10.0, 3.0]


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]


def test_reference_arm_other_ranks_print_nothing(capsys):
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    args = argparse.Namespace(gpus=2, steps=1, warmup=3, impl="reference")
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""
