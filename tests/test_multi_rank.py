"""The multi-GPU path of bench.py runs replicas (one independent batch per
rank, no collective on the data path).  Its host logic -- the job time is the
slowest rank's, the aggregate counts every rank's sequences, only rank 0
reports -- runs here on CPU as two gloo ranks."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(2.0 + rank, world, "cpu")   # rank 1 is the slow one
    el = bench.max_over_ranks(0.5 * (rank + 1), world, "cpu")
    dist.barrier()
    out.put((rank, ms, el, bench.aggregate_tok_s(4, world, ms)))
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank_and_every_sequence():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, el, tok_s in res:
        assert ms == 3.0 and el == 1.0
        assert tok_s == pytest.approx(4 * 2 * 1000.0 / 3.0)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert bench.aggregate_tok_s(8, 1, 4.0) == 2000.0


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import argparse
    import bench
    a = argparse.Namespace(layers=None, B=1, L=8, kv="f16", seed=1, steps=1, warmup=1, gpus=2)
    assert bench.run_reference(a, rank=1, world=2) is None
    assert capsys.readouterr().out == ""
