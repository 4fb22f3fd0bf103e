"""Build libglance.so in-tree with nvcc (sm_103a only).

Each CUDA translation unit is compiled in parallel, then linked into one
shared library under ``tree_verified_block_gb300/_lib/``. The same units are
also compiled with -DGLANCE_CHECK into ``libglance_check.so`` (objects under
``_lib/check/``): the bounds-checked build, in which every computed global
index is tested and an out-of-range one reports GLANCE_DEV_OUT_OF_BOUNDS
instead of being accessed. A unit is rebuilt
unless the sha256 digest stored beside its object matches the digest of its
source, the internal header, the public header and the compiler flags; the
library is relinked unless its stored digest matches those of its objects.
Timestamps are not trusted: a copied tree can carry objects newer than an
edited source.
"""
import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT, "libglance.so")
CHECK_OUT = os.path.join(OUT, "check")
LIB_CHECK = os.path.join(OUT, "libglance_check.so")
UNITS = ["api", "build_tree", "tree_attention", "lmhead", "commit", "dense"]
HEADERS = [os.path.join(CSRC, "glance_internal.cuh"), os.path.join(ROOT, "include", "glance.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-I" + os.path.join(ROOT, "include")]


def nvcc():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the GLANCE CUDA library cannot be built")


def _digest(paths, extra=()):
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
        h.update(b"\0")
    for e in extra:
        h.update(e.encode())
        h.update(b"\0")
    return h.hexdigest()


def _stored(path):
    try:
        with open(path + ".sha256") as f:
            return f.read().strip()
    except OSError:
        return None


def _store(path, digest):
    with open(path + ".sha256", "w") as f:
        f.write(digest + "\n")


def _compile(unit, force, checked=False):
    src = os.path.join(CSRC, unit + ".cu")
    obj = os.path.join(CHECK_OUT if checked else OUT, unit + ".o")
    flags = FLAGS + (["-DGLANCE_CHECK"] if checked else [])
    cmd = [nvcc()] + ARCH + flags + ["-c", src, "-o", obj]
    want = _digest([src] + HEADERS, ARCH + flags)
    if not force and os.path.exists(obj) and _stored(obj) == want:
        return obj, False
    if os.path.exists(obj + ".sha256"):
        os.remove(obj + ".sha256")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {unit}.cu:\n{r.stdout}\n{r.stderr}")
    _store(obj, want)
    return obj, True


def _link(objs, lib, force, verbose):
    want = _digest(objs)
    if force or not os.path.exists(lib) or _stored(lib) != want:
        tmp = lib + ".tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
        _store(lib, want)
        if verbose:
            print("built", lib)


def build(force=False, verbose=False, checked=True):
    """Compile and link libglance.so (and, with checked, libglance_check.so);
    returns the path of libglance.so."""
    os.makedirs(OUT, exist_ok=True)
    os.makedirs(CHECK_OUT, exist_ok=True)
    jobs = [(u, False) for u in UNITS] + ([(u, True) for u in UNITS] if checked else [])
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(lambda j: _compile(j[0], force, j[1]), jobs))
    objs = [o for (o, _), (_, c) in zip(results, jobs) if not c]
    _link(objs, LIB, force, verbose)
    if checked:
        _link([o for (o, _), (_, c) in zip(results, jobs) if c], LIB_CHECK, force, verbose)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
