"""Build the CPU oracle shared library (liboracle.so) with gcc.

Test infrastructure: the oracle is the checker of the CUDA library and is
never on its product path.  ``-ffp-contract=off`` keeps every a*b+c as two
roundings on both x86-64 and aarch64, so the oracle gives identical bits on
either host.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build_cmd():
    return ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC", "-shared",
            "-pthread", SRC, "-o", LIB, "-lm"]


def needs_build():
    return (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


def build(force=False):
    """Compile liboracle.so next to its source (no-op if up to date)."""
    if force or needs_build():
        subprocess.check_call(build_cmd())
    return LIB


def start_build():
    """Start the compile in the background; returns a Popen or None if up to date."""
    if not needs_build():
        return None
    return subprocess.Popen(build_cmd())


if __name__ == "__main__":
    build(force="--force" in sys.argv)
    print(LIB)
