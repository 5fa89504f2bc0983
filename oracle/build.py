"""Compile the CPU oracle (``gpt2_ref.c``) into two shared libraries.

Test infrastructure only: the oracle is built and loaded by the tests, by
``__graft_entry__`` and by bench.py's CPU-baseline leg.

* ``libgpt2ref_f32_<isa>.so`` -- REAL=float, the fp32 reference.
* ``libgpt2ref_f64_<isa>.so`` -- REAL=double, for finite differences and
  library-routine checks.

``<isa>`` is ``v3`` (AVX2+FMA code generation) when the host CPU has those
extensions and ``v1`` otherwise, so a library built on one machine is never
run on a CPU that lacks its instructions.  ``-ffp-contract=off`` keeps every
expression rounded exactly as written.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gpt2_ref.c")
OUT_DIR = os.path.join(HERE, "_build")


def host_isa() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            flags = set()
            for line in f:
                if line.startswith("flags"):
                    flags = set(line.split(":", 1)[1].split())
                    break
        if {"avx2", "fma", "bmi2"} <= flags:
            return "v3"
    except OSError:
        pass
    return "v1"


def lib_path(real: str, isa: str | None = None) -> str:
    isa = isa or host_isa()
    return os.path.join(OUT_DIR, f"libgpt2ref_{real}_{isa}.so")


def build(force: bool = False, verbose: bool = False) -> dict:
    os.makedirs(OUT_DIR, exist_ok=True)
    isa = host_isa()
    march = ["-march=x86-64-v3"] if isa == "v3" else []
    out = {}
    for real, ctype in (("f32", "float"), ("f64", "double")):
        dst = lib_path(real, isa)
        fresh = os.path.exists(dst) and os.path.getmtime(dst) >= os.path.getmtime(SRC)
        if force or not fresh:
            cmd = ["gcc", "-O3", *march, "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                   f"-DREAL={ctype}", "-o", dst + ".tmp", SRC, "-lm"]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            subprocess.check_call(cmd)
            os.replace(dst + ".tmp", dst)
        out[real] = dst
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
