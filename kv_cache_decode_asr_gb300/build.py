"""Build libasrkv.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in its own nvcc process (in parallel), then
one nvcc call links the shared library.  Only the CUDA runtime is linked.
"""
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libasrkv.so")
ROOT = os.path.dirname(HERE)
HEADERS = [os.path.join(ROOT, "include", "asrkv.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# per-file flags (none at present: each kernel's __launch_bounds__ sets its
# register budget)
EXTRA = {}
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v"]


def nvcc():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libasrkv.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return sources() + HEADERS + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                                  if f.endswith(".cuh")]


def needs_build():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force=False, verbose=False):
    """Compile every .cu under csrc/ and link libasrkv.so (no-op if up to date)."""
    if not force and not needs_build():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        log = obj + ".log"
        objs.append(obj)
        fh = open(log, "w")
        extra = EXTRA.get(os.path.basename(src), [])
        p = subprocess.Popen([cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj], stdout=fh,
                             stderr=subprocess.STDOUT)
        procs.append((p, fh, log, src))
    failed = []
    for p, fh, log, src in procs:
        rc = p.wait()
        fh.close()
        if verbose or rc != 0:
            with open(log) as f:
                sys.stderr.write(f.read())
        if rc != 0:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    tmp = LIB + ".tmp"
    subprocess.check_call([cc, *ARCH, "-shared", "--cudart", "static", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
