"""Shared helpers for the tests: building the library, host<->device views."""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "glance.h")


def ensure_built():
    from tree_verified_block_gb300 import _build
    return _build.build()


def header_functions():
    """Names of the functions include/glance.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(glance_[a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def bf16_tensor(bits, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def boundary_gap(x, N):
    """Score gap between the N-th and (N+1)-th best prefix (oracle, fp64)."""
    from oracle.marginals import candidate_lists
    from oracle.tree import top_n_best_first
    L, V = x.shape
    total = sum(V ** d for d in range(1, L + 1)) if V ** 1 < 10 ** 6 else N + 2
    if N + 1 > total:
        return np.inf
    _, logq, _ = candidate_lists(x, min(N + 1, V))
    best = top_n_best_first(logq, N + 1)
    return best[N - 1][1] - best[N][1]
