"""The N > 1 path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Every (sequence, head) is independent, so N GPUs run N replicas with no data-path collective; the
only cross-rank steps are the barrier around the timed region and the max over ranks of the step
time, from which rank 0 reports the whole-job throughput.  The reference arm runs on rank 0 only.

Each rank here runs a replica step for real: the tiny workload (one sequence of 256 tokens, H = 2,
d = 64, fp32) through the CPU path that exists without a GPU, the oracle's gates and token
recurrence, between the bench's barriers.  The replicas share no data, so each must reproduce, bit for
bit, the same step run in a single process; the test gathers the outputs only to check that.
"""
import importlib.util
import io
import os
import socket
import sys
import time
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


def _replica_step():
    """One replica's step on the tiny workload, by the oracle: gates from the logits, then the
    token recurrence with the raw output.  Returns (out, final state) as float64 tensors."""
    import torch

    from gated_deltanet_recurrence_gb300 import synthetic
    from tests._util import oracle_gates, oracle_prefill
    inp = synthetic.prefill_inputs("tiny")
    g32, b32 = oracle_gates(inp)
    y, S = oracle_prefill(inp, g32, b32, threads=1)
    return torch.as_tensor(y, dtype=torch.float64), torch.as_tensor(S, dtype=torch.float64), inp["total_T"]


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import types

    import torch
    import torch.distributed as dist
    bench = _load_bench()
    args = types.SimpleNamespace(impl="reference", steps=1, warmup=3, cpu_seconds=1.0)
    w, r, local = bench.dist_setup(args)
    try:
        assert dist.get_backend() == "gloo"
        # the timed region as the bench brackets it: barrier, K replica steps, barrier
        bench.barrier(w)
        t0 = time.perf_counter()
        y, S, tokens_per_rank = _replica_step()
        ms = (time.perf_counter() - t0) * 1e3
        bench.barrier(w)
        worst = bench.max_over_ranks(ms, w)
        value = tokens_per_rank * w / (worst / 1e3)
        # for the check only: every rank's outputs to every rank
        ys = [torch.empty_like(y) for _ in range(w)]
        Ss = [torch.empty_like(S) for _ in range(w)]
        dist.all_gather(ys, y)
        dist.all_gather(Ss, S)
        replicas_equal = all(torch.equal(ys[0], t) for t in ys) and all(torch.equal(Ss[0], t) for t in Ss)
        # the reference arm prints on rank 0 only; rank 1 returns at once without work
        out = io.StringIO()
        if r != 0:
            args.rank, args.world = r, w
            with redirect_stdout(out):
                bench.run_reference(args)
        q.put((r, w, ms, worst, value, tokens_per_rank, replicas_equal, y.numpy(), S.numpy(), out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_run_replicas_take_the_max_and_aggregate():
    mp = pytest.importorskip("torch.multiprocessing")
    import numpy as np
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=300) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort(key=lambda t: t[0])
    assert [r[0] for r in results] == [0, 1]
    assert all(r[1] == 2 for r in results)
    worst = max(r[2] for r in results)
    assert all(r[3] == worst for r in results)                 # every rank sees the slowest rank
    tokens = results[0][5]
    assert tokens == 256
    assert all(abs(r[4] - 2 * tokens / (worst / 1e3)) <= 1e-9 * r[4] for r in results)
    assert all(r[6] for r in results)                          # the replicas agree bit for bit
    # and each equals the same step run in this single process
    y1, S1, _ = _replica_step()
    np.testing.assert_array_equal(results[0][7], y1.numpy())
    np.testing.assert_array_equal(results[0][8], S1.numpy())
    assert results[1][9] == ""                                 # rank 1 printed nothing
