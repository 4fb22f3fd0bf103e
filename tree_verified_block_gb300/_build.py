"""Build libglance.so in-tree with nvcc (sm_103a only).

Each CUDA translation unit is compiled in parallel, then linked into one
shared library under ``tree_verified_block_gb300/_lib/``. A unit is rebuilt
when it, the internal header or the public header is newer than its object.
"""
import concurrent.futures as cf
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


def _mtime(p):
    return os.path.getmtime(p) if os.path.exists(p) else -1.0


def _compile(unit, force):
    src = os.path.join(CSRC, unit + ".cu")
    obj = os.path.join(OUT, unit + ".o")
    newest = max([_mtime(src)] + [_mtime(h) for h in HEADERS])
    if not force and _mtime(obj) >= newest:
        return obj, False
    cmd = [nvcc()] + ARCH + FLAGS + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {unit}.cu:\n{r.stdout}\n{r.stderr}")
    return obj, True


def build(force=False, verbose=False):
    """Compile and link; returns the library path."""
    os.makedirs(OUT, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(lambda u: _compile(u, force), UNITS))
    objs = [o for o, _ in results]
    rebuilt = any(b for _, b in results)
    if rebuilt or not os.path.exists(LIB) or _mtime(LIB) < max(_mtime(o) for o in objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
        if verbose:
            print("built", LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
