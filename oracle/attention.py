"""Ancestor-masked tree attention (oracle step O4).

Follows "Vision Is Not Overhead ..." (arXiv 2609.00355), Definition 1 and the
proof of Theorem 1 (Appendix B.1): the tree is packed into one ancestor-masked
target pass, and the row of a depth-d node sees exactly what the unpacked
sequence x . b . y_{1:d} would see: the whole cached prefix x (positions
0..T-1), the root b and the node's ancestors, and itself. The layout changes,
the conditioning does not.

Per query head h and packed row i, with kv head g = h // (Hq / Hkv) (grouped
query attention), the visible keys are the prefix slots 0..T-1 and the tree
slots T + k for every row k with anc(i, k). Scores are (q . k) * scale, the
softmax is taken over the visible keys only, and the output is the weighted sum
of their values. Computed directly in float64.
"""
import numpy as np


def visible_tree_rows(anc, i):
    """Rows k whose bit is set in row i's ancestor mask, ascending."""
    rows = []
    for w in range(anc.shape[1]):
        word = int(anc[i, w])
        for b in range(64):
            if (word >> b) & 1:
                rows.append(64 * w + b)
    return rows


def tree_attention(q, k_cache, v_cache, T, anc, scale):
    """q: (R, Hq, D); k_cache, v_cache: (Hkv, T_cap, D); tree keys at T..T+R-1.

    Returns out (R, Hq, D) float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    R, Hq, D = q.shape
    Hkv = k_cache.shape[0]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    out = np.empty((R, Hq, D), dtype=np.float64)
    for i in range(R):
        keys = np.concatenate([np.arange(T), T + np.asarray(visible_tree_rows(anc, i), dtype=np.int64)])
        for h in range(Hq):
            g = h // group
            s = (k_cache[g, keys] @ q[i, h]) * scale
            s = s - s.max()
            p = np.exp(s)
            p /= p.sum()
            out[i, h] = p @ v_cache[g, keys]
    return out


def causal_attention(q, k, v, scale):
    """Plain causal GQA attention over one sequence: q (S, Hq, D), k/v (S, Hkv, D).

    Written separately from tree_attention (no mask words) so that a chain
    shaped tree can be checked against it.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S, Hq, D = q.shape
    group = Hq // k.shape[1]
    out = np.empty_like(q)
    for t in range(S):
        for h in range(Hq):
            g = h // group
            s = (k[: t + 1, g] @ q[t, h]) * scale
            p = np.exp(s - s.max())
            out[t, h] = (p / p.sum()) @ v[: t + 1, g]
    return out
