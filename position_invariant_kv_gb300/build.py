"""Builds libkvrp.so (the C-ABI library and its sm_103a kernel) in place.

    python -m position_invariant_kv_gb300.build [-v]

One nvcc invocation, four translation units compiled in parallel, one
-gencode (sm_103a).  The shared object lands next to this file and is
git-ignored.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libkvrp.so")
SOURCES = [os.path.join(HERE, "csrc", "kvrp_kernel.cu"), os.path.join(HERE, "csrc", "kvrp_patch_form.cu"),
           os.path.join(HERE, "csrc", "kvrp_attend.cu"), os.path.join(HERE, "csrc", "kvrp_host.cpp")]
HEADERS = [os.path.join(ROOT, "include", "kvrp.h"), os.path.join(HERE, "csrc", "kvrp_plan.h"),
           os.path.join(HERE, "csrc", "kvrp_ptx.h")]


def nvcc_command(out: str = LIB, ptxas_verbose: bool = False) -> list:
    cmd = [
        "nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
        "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2", "--threads", "4",
        "-I", os.path.join(ROOT, "include"), "-I", os.path.join(HERE, "csrc"),
        "-o", out,
    ]
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    return cmd + SOURCES


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False) -> str:
    if force or not up_to_date():
        tmp = LIB + ".tmp"
        cmd = nvcc_command(tmp, ptxas_verbose=verbose)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
        if verbose:
            sys.stdout.write(res.stdout + res.stderr)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
