"""The ABI as a C program sees it (no GPU): gdn.h compiles as strict C99 and as C++, a C program
links against libgdn.so with nothing but the header, and the host-side behaviour it checks
(status codes, workspace sizing, argument errors before any launch) holds."""
import os
import shutil
import subprocess

import pytest

import gated_deltanet_recurrence_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
SOURCE = os.path.join(ROOT, "tests", "c_consumer.c")


def _lib_dir():
    gdn.lib()                                   # builds the library if it is missing
    return os.path.dirname(os.path.abspath(gdn._binding.LIB_PATH))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_uses_the_abi(tmp_path):
    exe = str(tmp_path / "c_consumer")
    libdir = _lib_dir()
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-O1",
                    "-I", INCLUDE, SOURCE, "-o", exe, "-L", libdir, "-lgdn",
                    "-Wl,-rpath," + libdir], check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "c consumer ok" in r.stdout


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_header_compiles_as_cxx(tmp_path):
    src = tmp_path / "h.cc"
    src.write_text('#include "gdn.h"\nint main() { return gdn_status_string(0) ? 0 : 1; }\n')
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                    "-I", INCLUDE, str(src)], check=True, capture_output=True, text=True)
