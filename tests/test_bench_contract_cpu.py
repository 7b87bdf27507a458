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
