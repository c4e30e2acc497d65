"""Compile the plain-C oracle into oracle/_build/libbsoracle.so with gcc.

Test infrastructure: the library never links or loads the result.
-ffp-contract=off keeps every multiply and add a separate rounding, so the
oracle's summation is exactly the one its source spells out.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "bs_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
OUT = os.path.join(OUT_DIR, "libbsoracle.so")


def build(src: str = SRC, out: str = OUT, extra=()) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src) and not extra:
        return out
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11", "-Wall", "-Wextra",
           *extra, "-o", out + ".tmp", src]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build())
    sys.exit(0)
