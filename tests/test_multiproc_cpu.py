"""The N > 1 path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Every (sequence, head) is independent, so N GPUs run N replicas with no data-path collective; the
only cross-rank steps are the barrier around the timed region and the max over ranks of the step
time, from which rank 0 reports the whole-job throughput.  The reference arm runs on rank 0 only.
"""
import importlib.util
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import types

    import torch.distributed as dist
    bench = _load_bench()
    args = types.SimpleNamespace(impl="reference", steps=1, warmup=3, cpu_seconds=1.0)
    w, r, local = bench.dist_setup(args)
    try:
        assert dist.get_backend() == "gloo"
        # each rank measured a different step time; every rank must see the slowest
        ms = 10.0 + 5.0 * r
        worst = bench.max_over_ranks(ms, w)
        bench.barrier(w)
        tokens_per_rank = 8192
        value = tokens_per_rank * w / (worst / 1e3)
        # the reference arm prints on rank 0 only; rank 1 returns at once without work
        out = io.StringIO()
        if r != 0:
            args.rank, args.world = r, w
            with redirect_stdout(out):
                bench.run_reference(args)
        q.put((r, w, worst, value, out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_aggregate():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    assert [r[0] for r in results] == [0, 1]
    assert all(r[1] == 2 for r in results)
    assert all(r[2] == 15.0 for r in results)                 # max over ranks
    assert all(abs(r[3] - 2 * 8192 / 0.015) < 1e-6 for r in results)
    assert results[1][4] == ""                                 # rank 1 printed nothing
