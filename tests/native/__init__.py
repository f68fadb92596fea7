"""Test-only native code: built here for the tests, never part of the library."""
from __future__ import annotations

import os
import subprocess
from pathlib import Path

HERE = Path(__file__).resolve().parent
BUILD = HERE / "_build"


def build_wait_probe() -> Path:
    """Compile wait_probe.cu (sm_103a, -DPA_TEST_HOOKS) into its own shared library."""
    from paged_kv_cache_83_gb300 import build as lib_build

    src = HERE / "wait_probe.cu"
    out = BUILD / "libwait_probe.so"
    deps = [src, lib_build.CSRC / "pa_common.cuh", lib_build.ROOT / "include" / "pa.h"]
    if out.exists() and all(d.stat().st_mtime <= out.stat().st_mtime for d in deps):
        return out
    BUILD.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(f".{os.getpid()}.tmp")
    cmd = [lib_build.nvcc(), *lib_build.ARCH, "-O3", "-std=c++17", "-DPA_TEST_HOOKS", "-shared",
           "-Xcompiler", "-fPIC", "-cudart", "shared", f"-I{lib_build.ROOT / 'include'}", str(src),
           "-o", str(tmp)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src.name}:\n{r.stderr}")
    os.replace(tmp, out)
    return out
