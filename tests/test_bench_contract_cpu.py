"""The benchmark's reference arm on the CPU: `bench.py --impl reference` times the fp64 oracle on
the host cores and prints one JSON line with the benchmark's keys, alone or under torchrun with
two ranks (rank 0 prints, the other rank exits 0 without work).  No GPU is involved."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _json_lines(text):
    return [json.loads(x) for x in text.splitlines() if x.startswith("{")]


def _check_line(line, n_gpus):
    assert line["impl"] == "reference"
    assert line["metric"] == "prefill tokens/s" and line["unit"] == "tokens/s"
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["n_gpus"] == n_gpus and line["steps"] == 1 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["vs_baseline"] is None and line["data"] == "synthetic" and line["dtype"] == "f64"
    assert line["config"]["workload"] == "prefill"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert cb["unit"] == "tokens/s" and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_under_torchrun_two_ranks():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(_free_port()), "bench.py", "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 2)


def test_roofline_numerators_follow_the_stated_formulas():
    """The algorithmic bytes and FLOPs behind the roofline fractions: per (sequence, head) and token,
    the decode step reads and writes the fp32 state once and moves q, k, v (bf16), g, beta (fp32)
    and y (bf16); the prefill call moves q, k, v, g, beta, z (fp32) and out once per token-head and
    the final state once; the chunk products cost 10 C d + 6 d^2 + C^2 / 3 FLOP per token-head."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    # decode workload: 256 sequences x 32 heads x (2 * 128^2 * 4 + 3 * 128 * 2 + 8 + 128 * 2) bytes
    assert bench.decode_bytes(256, 32, 128) == 256 * 32 * 132_104 == 1_082_195_968
    # prefill workload: 2 x 4096 tokens, 16 heads, fused gate, final state only
    assert bench.prefill_bytes(8192, 16, 128, 2) == 8192 * 16 * 1_544 + 2 * 16 * 128 * 128 * 4 == 204_472_320
    # with an initial state read as well (varlen workload), and without the gate
    assert bench.prefill_bytes(100, 2, 64, 3, gated=False, init_state=True) == \
        100 * 2 * (3 * 64 * 2 + 8 + 64 * 2) + 3 * 2 * 64 * 64 * 4 * 2
    assert abs(bench.prefill_flops_per_token_head(128) - (10 * 64 * 128 + 6 * 128 ** 2 + 64 ** 2 / 3)) < 1e-9
