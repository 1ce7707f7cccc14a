"""Builds liboracle.so from smoe_oracle.c with the host C compiler.

Test infrastructure only: the library it makes is loaded by the tests, the
smoke check and the benchmark's CPU-baseline leg, never by the product path.
The build uses no target-specific flags, so the same source gives the same
results on x86_64 and aarch64 hosts (-ffp-contract=off keeps gcc from fusing
multiply-adds on one host and not on the other).
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "smoe_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compiles the oracle if the library is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + ".tmp"
    cmd = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
