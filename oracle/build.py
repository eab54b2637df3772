"""Compile the fp64 CPU oracle (test infrastructure) into a shared library.

Plain gcc, OpenMP, no fast-math, no machine-specific flags, so the same source
builds on x86-64 and aarch64 hosts and keeps IEEE semantics.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "lmhead_oracle.c")
LIBRARY = os.path.join(HERE, "liblmhead_oracle.so")


def build(force: bool = False, source: str = SOURCE, output: str = LIBRARY) -> str:
    """Build `output` from `source` unless it is newer than the source."""
    if (not force and os.path.exists(output)
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    tmp = output + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-Wall", "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, output)
    return output


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
