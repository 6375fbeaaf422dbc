"""The C ABI from C: tests/c/abi_check.c includes only include/bkv.h, is
compiled with gcc, links libbkv.so and checks the host-decided behaviour of
the entry points (status text, version, argument validation, workspace
sizing).  No GPU and no Python binding involved."""
import os
import shutil
import subprocess

import pytest

from paged_kv_cache_slot_gb300 import build as bkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc is needed to build the C caller")
def test_c_caller_links_and_passes(tmp_path):
    lib = bkv_build.build()
    exe = tmp_path / "abi_check"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_check.c"), "-o", str(exe),
                    "-L", os.path.dirname(lib), "-lbkv", "-Wl,-rpath," + os.path.dirname(lib)], check=True)
    p = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert p.returncode == 0, p.stdout + p.stderr
    assert p.stdout.strip() == "ok"
