"""Per-offset marginals and candidate lists (oracle step O1).

Follows "Vision Is Not Overhead: One-Pass Block Drafting ..." (arXiv 2609.00355),
Section 3.2, Assumption 1: the drafter returns one marginal q_j(. | x, b) over
the vocabulary at each offset j = 1..L in a single pass, and a prefix y_{1:l} is
ranked by the plug-in score pi_hat(y_{1:l}) = prod_{j<=l} q_j(y_j | x, b). The
project page (js-lee-ai.github.io/GLANCE, "Draft pass") states the same with
L = B - 1 = 15.

The drafter's output is taken to be logits x_{j,v}; q_j = softmax(x_j). The
oracle works in log space: log q_j(v) = x_{j,v} - logsumexp_v x_{j,v}, so that
log pi_hat is a sum.

Candidate lists: at offset j only the K = min(N, V) best tokens can appear in a
top-N prefix set, since a token of rank >= N at offset j has N siblings that
beat every string passing through it. Tokens are ranked by logit descending,
equal logits by token id ascending (a total order; both sides see the same
input bits, so exact ties break the same way).
"""
import numpy as np


def log_marginals(x):
    """log q_j(v) for logits x of shape (L, V); float64, exact definition."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("draft logits must be finite")
    m = x.max(axis=1, keepdims=True)
    lse = m + np.log(np.exp(x - m).sum(axis=1, keepdims=True))
    return x - lse


def logsumexp_rows(x):
    x = np.asarray(x, dtype=np.float64)
    m = x.max(axis=1)
    return m + np.log(np.exp(x - m[:, None]).sum(axis=1))


def token_order(x_row):
    """Token ids of one offset sorted by (logit desc, id asc)."""
    x_row = np.asarray(x_row, dtype=np.float64)
    ids = np.arange(x_row.shape[0])
    return np.lexsort((ids, -x_row))


def candidate_lists(x, K):
    """Top-K candidate tokens per offset and their log q.

    Returns (tok[L, K] int64, logq[L, K] float64, rank_of[L, V] int64) where
    rank_of[j, v] is the position of token v in offset j's full ordering.
    """
    x = np.asarray(x, dtype=np.float64)
    L, V = x.shape
    if not 1 <= K <= V:
        raise ValueError("K must be in [1, V]")
    lq = log_marginals(x)
    tok = np.empty((L, K), dtype=np.int64)
    logq = np.empty((L, K), dtype=np.float64)
    rank_of = np.empty((L, V), dtype=np.int64)
    for j in range(L):
        order = token_order(x[j])
        rank_of[j, order] = np.arange(V)
        tok[j] = order[:K]
        logq[j] = lq[j, order[:K]]
    return tok, logq, rank_of
