"""Candidate tree: the top-N prefix set and its packing (oracle steps O2, O3).

Follows "Vision Is Not Overhead ..." (arXiv 2609.00355):
  * Definition 1 (Section 3.2): a candidate tree S is a prefix-closed set of
    nonempty strings after the root b, of depth at most L, with budget N = |S|.
  * Section 4.2 and the project page ("Verify pass"): the builder keeps the N
    prefixes of highest plug-in score pi_hat; that set is prefix-closed.
  * Appendix B.5: node-sum value and top-prefix optimality are taken from prior
    work; the tests use them as a pin (the top-N set maximises the node-sum).

A node is identified by its rank vector (r_1, ..., r_d): r_j is the position of
y_j in offset j's token ordering (logit desc, id asc). Its score is
sum_{j<=d} log q_j(y_j), summed in order j = 1..d. Nodes are totally ordered,
best first, by (score desc, depth asc, rank vector lexicographic asc). The depth
and rank keys only decide exact score ties; a parent is never worse than its
child because log q <= 0.

Packing (canonical order): row 0 is the root b; rows 1..N are the nodes sorted
by (depth asc, rank vector lexicographic asc). Within one depth that is the
order (parent row asc, own rank asc), i.e. breadth-first, so every parent row
precedes its children's rows. pos_id = T + depth, where T is the number of
cached prefix tokens (the root sits at position T). The ancestor mask of row i
has bit k set iff row k is row i itself, the root, or an ancestor of row i.
"""
import heapq
import itertools

import numpy as np

from .marginals import candidate_lists, log_marginals, token_order


def node_key(score, ranks):
    """Sort key (ascending = better) of a node under the total order."""
    return (-score, len(ranks), tuple(ranks))


def top_n_bruteforce(x, N):
    """Top-N strings by enumerating every string of length 1..L (tiny V, L only).

    Returns a list of rank tuples, best first.
    """
    x = np.asarray(x, dtype=np.float64)
    L, V = x.shape
    total = sum(V ** d for d in range(1, L + 1))
    if N > total:
        raise ValueError("N exceeds the number of strings")
    lq = log_marginals(x)
    rank_of = np.empty((L, V), dtype=np.int64)
    for j in range(L):
        rank_of[j, token_order(x[j])] = np.arange(V)
    keyed = []
    for d in range(1, L + 1):
        for ys in itertools.product(range(V), repeat=d):
            s = 0.0
            for j, y in enumerate(ys):
                s += lq[j, y]
            ranks = tuple(int(rank_of[j, y]) for j, y in enumerate(ys))
            keyed.append((node_key(s, ranks), ranks))
    keyed.sort()
    return [r for _, r in keyed[:N]]


def top_n_best_first(logq, N):
    """Top-N nodes by lazy best-first search over the candidate lists.

    logq[j, r] is log q of the rank-r candidate at offset j+1 (rows sorted by
    rank). Every node other than (0,) has a predecessor that is strictly better
    under the total order: its previous sibling (last rank - 1) when the last
    rank is > 0, else its parent. Popping nodes in order and pushing, for each
    popped node, its first child (rank 0 at the next offset) and its next
    sibling (last rank + 1) therefore pops nodes in exactly the total order.
    Returns a list of (rank tuple, score), best first.
    """
    logq = np.asarray(logq, dtype=np.float64)
    L, K = logq.shape
    heap = [(node_key(logq[0, 0], (0,)), (0,), float(logq[0, 0]))]
    out = []
    while len(out) < N:
        if not heap:
            raise ValueError("N exceeds the number of strings")
        _, ranks, score = heapq.heappop(heap)
        out.append((ranks, score))
        d = len(ranks)
        if d < L:
            child = ranks + (0,)
            cs = score + logq[d, 0]
            heapq.heappush(heap, (node_key(cs, child), child, cs))
        r = ranks[-1]
        if r + 1 < K:
            sib = ranks[:-1] + (r + 1,)
            # the sibling's score is summed along its own path, in order
            ss = 0.0
            for j, rj in enumerate(sib):
                ss += logq[j, rj]
            heapq.heappush(heap, (node_key(ss, sib), sib, ss))
    return out


def pack_tree(nodes, tok, logq, root_token, T):
    """Pack a prefix-closed node set into the canonical row order.

    nodes: iterable of rank tuples (any order). tok/logq: candidate lists.
    Returns a dict of numpy arrays with N+1 rows: token, parent, depth, pos_id,
    score (float64, sum of log q along the path, 0 at the root) and anc
    (uint64, shape (N+1, ceil((N+1)/64))).
    """
    nodes = sorted(set(tuple(n) for n in nodes), key=lambda r: (len(r), r))
    n = len(nodes)
    index = {(): 0}
    for i, r in enumerate(nodes):
        index[r] = i + 1
    for r in nodes:
        if r[:-1] not in index:
            raise ValueError("node set is not prefix-closed")
    rows = n + 1
    W = (rows + 63) // 64
    token = np.empty(rows, dtype=np.int64)
    parent = np.empty(rows, dtype=np.int64)
    depth = np.empty(rows, dtype=np.int64)
    score = np.empty(rows, dtype=np.float64)
    anc = np.zeros((rows, W), dtype=np.uint64)
    token[0], parent[0], depth[0], score[0] = root_token, -1, 0, 0.0
    anc[0, 0] = np.uint64(1)
    for i, r in enumerate(nodes, start=1):
        d = len(r)
        token[i] = tok[d - 1, r[-1]]
        parent[i] = index[r[:-1]]
        depth[i] = d
        s = 0.0
        for j, rj in enumerate(r):
            s += logq[j, rj]
        score[i] = s
        anc[i] = anc[parent[i]]
        anc[i, i // 64] |= np.uint64(1) << np.uint64(i % 64)
    pos_id = T + depth
    return dict(token=token, parent=parent, depth=depth, pos_id=pos_id,
                score=score, anc=anc, ranks=[()] + nodes)


def build_tree(x, N, root_token, T):
    """The whole draft-to-tree stage: candidate lists, top-N, packing."""
    x = np.asarray(x, dtype=np.float64)
    L, V = x.shape
    K = min(N, V)
    tok, logq, _ = candidate_lists(x, K)
    nodes = [r for r, _ in top_n_best_first(logq, N)]
    return pack_tree(nodes, tok, logq, root_token, T)


def is_ancestor(tree, i, k):
    """True iff packed row k is row i, the root, or an ancestor of row i."""
    w = tree["anc"][i, k // 64]
    return bool((int(w) >> (k % 64)) & 1)


def all_prefix_closed_sets(V, L, N):
    """Every prefix-closed set of N nonempty strings over V tokens, depth <= L.

    Strings are token tuples. Enumerated by walking the full V-ary tree in
    breadth-first order and deciding, for each node whose parent is in the set,
    whether it is in the set. Tiny V, L, N only.
    """
    full = [ys for d in range(1, L + 1) for ys in itertools.product(range(V), repeat=d)]
    out = []

    def rec(pos, chosen, chosen_set):
        if len(chosen) == N:
            out.append(list(chosen))
            return
        if pos == len(full):
            return
        ys = full[pos]
        if len(ys) == 1 or ys[:-1] in chosen_set:
            chosen.append(ys)
            chosen_set.add(ys)
            rec(pos + 1, chosen, chosen_set)
            chosen.pop()
            chosen_set.discard(ys)
        rec(pos + 1, chosen, chosen_set)

    rec(0, [], set())
    return out
