"""Compile the C oracle (test infrastructure; never used by the product path).

The shared object goes to ``oracle/_build/libqs_oracle.so``.  Flags keep IEEE
fp32 semantics exactly as written: no FMA contraction, no fast-math.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qs_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libqs_oracle.so")

_BASE = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
         "-fPIC", "-shared", SRC, "-o", LIB, "-lm"]


def build(force: bool = False) -> str:
    """Build the oracle library if missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [a if a != LIB else tmp for a in _BASE]
    # OpenMP over (sequence, head) when the compiler has it, plain C otherwise
    r = subprocess.run(cmd[:1] + ["-fopenmp"] + cmd[1:], capture_output=True, text=True)
    if r.returncode != 0:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
