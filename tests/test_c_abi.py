"""The C ABI from plain C (no GPU): tests/c/abi_smoke.c compiles as C99 against
include/splitkv.h with warnings as errors, links against the built library and its
host-only calls answer as the header documents."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

from split_kv_attention_flash_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_against_the_header_and_library(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = _build.build()
    exe = tmp_path / "abi_smoke"
    src = os.path.join(ROOT, "tests", "c", "abi_smoke.c")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        src, lib, f"-Wl,-rpath,{os.path.dirname(lib)}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
