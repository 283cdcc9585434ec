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
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
