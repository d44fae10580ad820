"""The boundary is a C ABI: a plain C99 program compiles against include/dllm_cache.h
(warnings as errors, pedantic), links libdllmcache.so and runs the calls that need no
GPU.  No Python binding is involved."""
import os
import shutil
import subprocess

import pytest

from denoising_step_attention_qkv_b300 import capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
def test_plain_c_caller(tmp_path):
    capi.lib()  # the library must exist (built in tree)
    libdir = os.path.dirname(capi.LIB_PATH)
    exe = tmp_path / "abi_check"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi_check.c"), "-L", libdir, "-ldllmcache", f"-Wl,-rpath,{libdir}",
           "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
