"""The C ABI from plain C: tests/c/abi_host_example.c is compiled with gcc as C11 against
include/quail.h alone, linked against libquail.so alone, and run (host-side entry points
only, so no GPU is needed)."""
import os
import shutil
import subprocess

import pytest

import prefill_only_cascade_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not installed")
def test_plain_c_program_uses_the_abi(tmp_path):
    lib_dir = os.path.dirname(q.LIB_PATH)
    exe = tmp_path / "abi_host_example"
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c",
                                                             "abi_host_example.c"),
           "-L", lib_dir, "-l:libquail.so", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)]
    build = subprocess.run(cmd, capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "FAILED" not in run.stdout and run.stdout.count("ok ") == 14
