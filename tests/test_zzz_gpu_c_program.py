"""The C ABI without Python on the data path: tests/c_decode_gpu.c allocates device memory with the
CUDA runtime, runs gdn_recurrent_step through libgdn.so and checks it against the oracle's C entry
point.  The CPU test only compiles and links the program; the GPU test runs it.  The file name
makes pytest run it after the kernel parity tests."""
import glob
import os
import shutil
import subprocess

import pytest

import gated_deltanet_recurrence_gb300 as gdn
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCE = os.path.join(ROOT, "tests", "c_decode_gpu.c")


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime.h")):
            return cand
    return None


def _cudart_dir(home):
    for d in [os.path.join(home, "lib64")] + glob.glob(os.path.join(home, "targets", "*", "lib")):
        if glob.glob(os.path.join(d, "libcudart.so*")):
            return d
    return None


def _build(tmp_path):
    home = _cuda_home()
    if home is None or shutil.which("gcc") is None:
        pytest.skip("needs gcc and the CUDA toolkit headers")
    cudart = _cudart_dir(home)
    if cudart is None:
        pytest.skip("libcudart not found")
    gdn.lib()
    gdn_dir = os.path.dirname(gdn._binding.LIB_PATH)
    oracle_dir = os.path.dirname(oracle.build())
    exe = str(tmp_path / "c_decode_gpu")
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(home, "include"), SOURCE, "-o", exe,
           "-L", gdn_dir, "-lgdn", "-L", oracle_dir, "-lgdn_oracle", "-L", cudart, "-lcudart", "-lm",
           "-Wl,-rpath," + ":".join([gdn_dir, oracle_dir, cudart])]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
def test_c_program_decodes_on_the_gpu(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("max_rel_y")
