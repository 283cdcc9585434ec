"""Compile the CPU oracle (test infrastructure) into oracle/_w4_oracle.so.

Plain C, no target-specific flags, so the same source builds on x86_64 and
aarch64 hosts.  Building the checker is not using it: the package build
calls this so that tests on a fresh machine find the oracle ready.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "w4_oracle.c")
LIB = os.path.join(HERE, "_w4_oracle.so")


def build_oracle(force: bool = False) -> str:
    """Build the oracle shared object if missing or stale; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    compile_oracle(SRC, tmp)
    os.replace(tmp, LIB)
    return LIB


def compile_oracle(src: str, out: str) -> None:
    """Compile one C source with the oracle's flags into the shared object
    `out` (no fast-math, no FMA contraction: the source's own rounding)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)


if __name__ == "__main__":
    print(build_oracle(force=True))
