"""The benchmark's multi-rank host logic on CPU with gloo, world size 2: every
rank learns the slowest replica's time and the whole-job throughput counts the
tokens of all replicas (replicas only: no collective on the data path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import importlib.util

    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    ms = [12.5, 20.0][rank]
    worst = bench.reduce_max(ms, dist, "cpu")
    q.put((rank, worst, bench.whole_job_tokens_per_s(world, 8192, worst)))
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_and_throughput_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, tps in out:
        assert worst == 20.0
        assert tps == pytest.approx(2 * 8192 / 0.020)


def test_single_rank_needs_no_process_group():
    import importlib.util

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert bench.reduce_max(3.5, None, "cpu") == 3.5
    assert bench.whole_job_tokens_per_s(1, 8192, 25.0) == pytest.approx(327680.0)
