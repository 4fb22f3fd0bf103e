"""Shared verifier budget across a batch of rounds, with entropy-keyed node
masses (oracle; test infrastructure only).

"Vision Is Not Overhead ..." (arXiv 2609.00355), Appendix B.5 and
Propositions 4-6: under a shared verifier budget the allocation maximising the
total expected committed length is global best-first over all rounds' nodes
(the node-sum value of a tree and top-prefix optimality are cited machinery),
and the law keys a round's node masses by its root entropy H through

    V(H) proportional to E[a | H] (1 - p_m(H))           (Equation 5)

with logit p_m(H) = b0 - b1 H and E[a | H] the geometric mean
p_m / (1 - p_m) truncated at the block horizon L (Equation 2), i.e.
E[a | H] = sum_{k=1..L} p_m^k, so V(H) = p_m (1 - p_m^L).

Reading taken here: node s of round r has mass w_r * pi_hat_r(s) with
w_r = V(H_r) (w_r = 1 when no entropies are given); the budget N_total goes
to the N_total globally highest-mass nodes, each round holding at most N_max
(its tree capacity). Because w_r is one factor per round, round r's share is
the best n_r nodes of its own best-first order, a prefix-closed set. Ties in
mass go to the lower round index, then to the round's own order.

Trees keep N_max + 1 rows; rows n_r + 1 .. N_max are inactive: token -1,
parent -1 (no row's child, so the walk never reaches them), depth 0,
pos_id = T, score -inf, ancestor mask = the row itself.
"""
import numpy as np

from .marginals import candidate_lists
from .tree import pack_tree, top_n_best_first


def entropy_keyed_log_weight(H, b0, b1, L):
    """log V(H) = log(p_m (1 - p_m^L)), logit p_m = b0 - b1 H."""
    pm = 1.0 / (1.0 + np.exp(-(b0 - b1 * np.asarray(H, dtype=np.float64))))
    return np.log(pm) + np.log1p(-pm ** L)


def _n_strings(V, L):
    total, pw = 0, 1
    for _ in range(L):
        pw *= V
        total += pw
    return total


def shared_budget_trees(xs, N_total, N_max, roots, Ts, log_w=None):
    """xs: B draft logit arrays (L, V). Returns (trees [B] with N_max + 1 rows,
    n_active [B], the sorted global keys (for tie-gap checks))."""
    B = len(xs)
    log_w = np.zeros(B) if log_w is None else np.asarray(log_w, dtype=np.float64)
    pops, lists = [], []
    for r, x in enumerate(xs):
        x = np.asarray(x, dtype=np.float64)
        L, V = x.shape
        n_r = min(N_max, _n_strings(V, L))
        tok, logq, _ = candidate_lists(x, min(N_max, V))
        pr = top_n_best_first(logq, n_r)
        pops.append(pr)
        lists.append((tok, logq))
    entries = sorted(((-(log_w[r] + sc), r, i) for r in range(B) for i, (_, sc) in enumerate(pops[r])))
    take = entries[:N_total]
    n_active = np.zeros(B, dtype=np.int64)
    for _, r, _ in take:
        n_active[r] += 1
    trees = []
    for r in range(B):
        tok, logq = lists[r]
        nodes = [rk for rk, _ in pops[r][:n_active[r]]]
        t = pack_tree(nodes, tok, logq, roots[r], Ts[r])
        rows, n = N_max + 1, n_active[r] + 1
        W = (rows + 63) // 64
        out = dict(token=np.full(rows, -1, np.int64), parent=np.full(rows, -1, np.int64),
                   depth=np.zeros(rows, np.int64), pos_id=np.full(rows, Ts[r], np.int64),
                   score=np.full(rows, -np.inf), anc=np.zeros((rows, W), np.uint64))
        for k in ("token", "parent", "depth", "pos_id", "score"):
            out[k][:n] = t[k]
        out["anc"][:n, :t["anc"].shape[1]] = t["anc"]
        for i in range(n, rows):
            out["anc"][i, i // 64] = np.uint64(1) << np.uint64(i % 64)
        trees.append(out)
    keys = np.array([-e[0] for e in entries])
    return trees, n_active, keys
