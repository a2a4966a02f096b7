"""The boundary from C and C++ (no GPU): include/gemm.h compiles as strict C99
and as C++17, and a C program linked against libgemm_gb300.so runs the
host-side part of the API (tests/c_consumer.c)."""

import os
import shutil
import subprocess

import pytest

import dense_matrix_multiply_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
SRC = os.path.join(ROOT, "tests", "c_consumer.c")


@pytest.fixture(scope="module")
def lib_dir():
    g.ensure_built()
    return os.path.dirname(g.LIB_PATH)


def _need(tool):
    if shutil.which(tool) is None:
        pytest.skip(f"{tool} not installed")


def test_header_is_strict_c99_and_cxx17(tmp_path):
    _need("gcc")
    _need("g++")
    src = tmp_path / "only_header.c"
    src.write_text('#include "gemm.h"\nint main(void) { return GEMM_OK; }\n')
    for cmd in (["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic"],
                ["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-pedantic", "-x", "c++"]):
        r = subprocess.run(cmd + ["-fsyntax-only", "-I", INCLUDE, str(src)], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_c_program_links_and_runs_the_host_side(tmp_path, lib_dir):
    _need("gcc")
    exe = tmp_path / "c_consumer"
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, SRC,
                        "-o", str(exe), "-L", lib_dir, "-lgemm_gb300", f"-Wl,-rpath,{lib_dir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
