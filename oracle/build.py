"""Compile the CPU oracle (test infrastructure) into oracle/_build/libpa_oracle.so.

Plain C99 with gcc; OpenMP when the compiler has it. No fast-math and no FMA
contraction, so the oracle gives the same bits on x86-64 and aarch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpa_oracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    base = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-Wno-unknown-pragmas", SRC]
    tmp = LIB + f".tmp{os.getpid()}"
    for extra in (["-fopenmp"], []):
        cmd = base + extra + ["-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode == 0:
            os.replace(tmp, LIB)
            return LIB
    raise RuntimeError("oracle build failed: " + " ".join(base))


if __name__ == "__main__":
    print(build(force=True, verbose=True))
