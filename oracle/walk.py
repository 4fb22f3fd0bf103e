"""Acceptance walk, A(S) and commit (oracle step O6).

Follows "Vision Is Not Overhead ..." (arXiv 2609.00355):
  * Section 3.1: each round commits a + 1 tokens, the a accepted nonroot tokens
    plus one token read off the last verified distribution.
  * Definition 1: A(S) = max{k >= 0 : Y_{1:j} in S for all j <= k}; the walk
    commits Y_{1:A(S)} and emits the next target-greedy token of the last
    verified row as the new root.
  * Appendix B.1, proof of Theorem 1: at a verified node the walk descends if
    the node extended by the target's greedy token is in S, otherwise it stops
    and emits that token as the next root.

Commit: the verified rows' K/V already sit in cache slots T..T+N (row r at
slot T + r). The root row and the a accepted rows, path_0 = 0, path_1..path_a,
are moved to slots T..T+a, and T becomes T + a + 1. The new root is pending:
its K/V are produced by the next round's verify pass.
"""
import numpy as np


def walk(tree, argmax, L=None):
    """Traversal form. Returns (a, path rows [a+1], accepted tokens [a], new_root)."""
    token, parent, depth = tree["token"], tree["parent"], tree["depth"]
    rows = len(token)
    u = 0
    path = [0]
    while True:
        if L is not None and depth[u] >= L:
            break
        target = int(argmax[u])
        nxt = None
        for c in range(rows):
            if parent[c] == u and token[c] == target:
                nxt = c
                break
        if nxt is None:
            break
        u = nxt
        path.append(u)
    a = len(path) - 1
    acc = [int(token[r]) for r in path[1:]]
    return a, path, acc, int(argmax[u])


def walk_gated(tree, argmax, gap, L, threshold):
    """Walk with the tie-aware gate ("Vision Is Not Overhead ...", Section 4.2
    and the end of the proof of Theorem 1 in Appendix B.1): a visited row whose
    top-2 logit margin is below `threshold` is a near-tie, where reduced
    precision may reorder the target's top two tokens, so the round defers to
    the target's own token there. The walk stops at the first such row and
    reports gated = True; that row's packed argmax is then not trusted as the
    next token (the caller recomputes it). Returns (a, path, accepted tokens,
    new_root, gated); without a near-tie on the path this is walk().
    """
    token, parent, depth = tree["token"], tree["parent"], tree["depth"]
    rows = len(token)
    u = 0
    path = [0]
    gated = False
    while True:
        if gap[u] < threshold:
            gated = True
            break
        if depth[u] >= L:
            break
        target = int(argmax[u])
        nxt = None
        for c in range(rows):
            if parent[c] == u and token[c] == target:
                nxt = c
                break
        if nxt is None:
            break
        u = nxt
        path.append(u)
    a = len(path) - 1
    return a, path, [int(token[r]) for r in path[1:]], int(argmax[u]), gated


def tree_strings(tree):
    """The set S as token tuples (root excluded)."""
    token, parent = tree["token"], tree["parent"]
    out = set()
    for i in range(1, len(token)):
        s = []
        u = i
        while u != 0:
            s.append(int(token[u]))
            u = parent[u]
        out.add(tuple(reversed(s)))
    return out


def accepted_length_set_form(S, Y):
    """A(S) = max{k >= 0 : Y_{1:j} in S for all j <= k} for a token sequence Y."""
    a = 0
    for k in range(1, len(Y) + 1):
        if tuple(Y[:k]) in S:
            a = k
        else:
            break
    return a


def commit(k_cache, v_cache, T, path):
    """Move tree slots T + path[i] to T + i for i = 0..a. Returns new T.

    k_cache, v_cache: arrays (..., T_cap, D) with the slot axis second to last;
    modified in place. All sources are read before any destination is written.
    """
    src = [T + p for p in path]
    ks = k_cache[..., src, :].copy()
    vs = v_cache[..., src, :].copy()
    for i in range(len(path)):
        k_cache[..., T + i, :] = ks[..., i, :]
        v_cache[..., T + i, :] = vs[..., i, :]
    return T + len(path)
