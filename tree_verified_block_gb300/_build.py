"""Build libglance.so in-tree with nvcc (sm_103a only).

Each CUDA translation unit is compiled in parallel, then linked into one
shared library under ``tree_verified_block_gb300/_lib/``. A unit is rebuilt
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


def _compile(unit, force):
    src = os.path.join(CSRC, unit + ".cu")
    obj = os.path.join(OUT, unit + ".o")
    cmd = [nvcc()] + ARCH + FLAGS + ["-c", src, "-o", obj]
    want = _digest([src] + HEADERS, ARCH + FLAGS)
    if not force and os.path.exists(obj) and _stored(obj) == want:
        return obj, False
    if os.path.exists(obj + ".sha256"):
        os.remove(obj + ".sha256")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {unit}.cu:\n{r.stdout}\n{r.stderr}")
    _store(obj, want)
    return obj, True


def build(force=False, verbose=False):
    """Compile and link; returns the library path."""
    os.makedirs(OUT, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(lambda u: _compile(u, force), UNITS))
    objs = [o for o, _ in results]
    want = _digest(objs)
    if force or not os.path.exists(LIB) or _stored(LIB) != want:
        tmp = LIB + ".tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
        _store(LIB, want)
        if verbose:
            print("built", LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
