"""The paged KV cache's host bookkeeping (llama_decode_kv_gb300/csrc/kv_pages.h) on the
CPU: a C++ harness drives the page manager through prefills, appends, forks and resets
against a simulated device memory and checks that every sequence reads back what was
written at its positions, that reference counts match the tables, and that an append the
pool cannot hold changes nothing."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "llama_decode_kv_gb300", "csrc")


def test_kv_page_manager(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path / "kv_pages_test")
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-I", CSRC, os.path.join(HERE, "native", "kv_pages_test.cpp"),
                    "-o", exe], check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
