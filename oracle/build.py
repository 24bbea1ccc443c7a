"""Compile the C oracle into ``oracle/liboracle_attn.so`` with the host gcc.

Test infrastructure: the library built here is loaded only by the tests, the
smoke check and the benchmark's CPU-baseline leg.  OpenMP is used when the
compiler supports it (rows are independent); otherwise the build is serial.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
LIB = os.path.join(HERE, "liboracle_attn.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    cc = os.environ.get("CC", "gcc")
    base = [cc, "-O2", "-std=c11", "-shared", "-fPIC", "-fvisibility=hidden",
            SRC, "-o", LIB + ".tmp", "-lm"]
    # -ffp-contract=off: no fused multiply-add, so every product and sum is
    # rounded exactly as the binary64 source says, on x86 and on Arm alike.
    flags = ["-ffp-contract=off"]
    r = subprocess.run(base[:1] + flags + ["-fopenmp"] + base[1:],
                       capture_output=True, text=True)
    if r.returncode != 0:
        r = subprocess.run(base[:1] + flags + base[1:], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
