"""Compile the C oracle into ``oracle/liboracle.so`` with the host C compiler.

Test infrastructure: the product library never links this.  The flags keep
binary64/binary32 arithmetic exactly as written (no contraction into fused
multiply-adds, no fast-math reassociation, no flush-to-zero).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-frounding-math", "-fvisibility=hidden"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source.

    ``EW_ORACLE_LIB`` names a prebuilt library to use instead; the mutation
    tests point it at deliberately broken builds to show the pins catch them.
    """
    override = os.environ.get("EW_ORACLE_LIB")
    if override:
        return override
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    cc = os.environ.get("CC", "cc")
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [cc, *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
