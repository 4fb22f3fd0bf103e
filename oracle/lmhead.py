"""LM-head projection, greedy argmax and top-2 gap (oracle step O5).

Follows "Vision Is Not Overhead ..." (arXiv 2609.00355): greedy decoding emits
argmax_w p(w | prefix) (Section 3.1); Theorem 1's full statement (Appendix B.1)
defines the top logit gap gamma_k = l_(1) - l_(2) at a visited prefix, the
margin the tie-aware gate reads (Section 4.2).

logits[i, v] = sum_k h[i, k] * W[k, v] (no bias; h already final-normed).
argmax is the lowest token id among equal maxima, and gap = l_(1) minus the
largest logit of any other token, so an exact tie gives gap 0. Computed in
float64, in column chunks to bound memory.
"""
import numpy as np


def lmhead_argmax(h, W, chunk=8192):
    """h: (M, d), W: (d, V). Returns (argmax int64[M], gap f64[M], maxlogit f64[M])."""
    h = np.asarray(h, dtype=np.float64)
    M = h.shape[0]
    V = W.shape[1]
    best = np.full(M, -np.inf)
    arg = np.zeros(M, dtype=np.int64)
    second = np.full(M, -np.inf)
    for c0 in range(0, V, chunk):
        c1 = min(V, c0 + chunk)
        lg = h @ np.asarray(W[:, c0:c1], dtype=np.float64)
        for i in range(M):
            row = lg[i]
            j = int(np.argmax(row))  # first index of the maximum
            m = row[j]
            rest = np.delete(row, j)
            m2 = rest.max() if rest.size else -np.inf
            if m > best[i]:
                second[i] = max(best[i], m2)
                best[i], arg[i] = m, c0 + j
            else:
                # equal maximum in a later chunk keeps the lower id
                second[i] = max(second[i], m)
    return arg, best - second, best


def logits(h, W):
    return np.asarray(h, dtype=np.float64) @ np.asarray(W, dtype=np.float64)


def next_token_entropy(h, W, chunk=8192):
    """Entropy in nats of softmax(logits[i]) for each row i.

    The target's next-token entropy H at the round root ("Vision Is Not
    Overhead ...", Section 6 and Equation 2; Proposition 1 in Appendix B):
    the packed root row of a round carries the target's distribution
    p(. | x, b), and H = -sum_w p(w) log p(w) = logsumexp(l) - sum_w p(w) l_w.
    Two passes in float64: the row maxima, then sum exp(l - m) and
    sum exp(l - m) l over column chunks.
    """
    h = np.asarray(h, dtype=np.float64)
    M = h.shape[0]
    V = W.shape[1]
    m = np.full(M, -np.inf)
    for c0 in range(0, V, chunk):
        lg = h @ np.asarray(W[:, c0:c0 + chunk], dtype=np.float64)
        m = np.maximum(m, lg.max(axis=1))
    s = np.zeros(M)
    el = np.zeros(M)
    for c0 in range(0, V, chunk):
        lg = h @ np.asarray(W[:, c0:c0 + chunk], dtype=np.float64)
        e = np.exp(lg - m[:, None])
        s += e.sum(axis=1)
        el += (e * lg).sum(axis=1)
    lse = m + np.log(s)
    return lse - el / s
