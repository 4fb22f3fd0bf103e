"""Pins for the oracle's tree builder and packing (CPU).

What fixes the builder independently of its own code:
* brute-force enumeration of every string (tiny V, L) sorted by plug-in score;
* brute-force enumeration of every prefix-closed set: the top-N set is the
  unique maximiser of the node-sum value sum_{s in S} pi_hat(s) (top-prefix
  optimality, cited in Appendix B.5);
* special cases: L = 1 is a plain top-N; point-mass marginals give a chain;
  N = 1 is the single best token of q_1;
* a hand-derived example (tests/golden/tree_tiny.txt).
"""
import itertools
import os

import numpy as np
import pytest

from oracle.marginals import candidate_lists, log_marginals
from oracle.tree import (all_prefix_closed_sets, build_tree, is_ancestor, pack_tree,
                         top_n_best_first, top_n_bruteforce)
from oracle.walk import tree_strings

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_tiny.txt")


def _tokens_of(x, ranks_list):
    L, V = x.shape
    tok, _, _ = candidate_lists(x, V)
    return [tuple(int(tok[j, r]) for j, r in enumerate(rk)) for rk in ranks_list]


@pytest.mark.parametrize("V,L", [(2, 1), (2, 3), (3, 2), (3, 3), (4, 2), (4, 3)])
def test_best_first_equals_bruteforce(V, L):
    g = np.random.default_rng(10 * V + L)
    total = sum(V ** d for d in range(1, L + 1))
    for trial in range(6):
        x = g.standard_normal((L, V)) * (0.5 + trial)
        for N in range(1, min(12, total) + 1):
            bf = top_n_bruteforce(x, N)
            K = min(N, V)
            _, logq, _ = candidate_lists(x, K)
            bfs = [r for r, _ in top_n_best_first(logq, N)]
            assert bfs == bf, (V, L, N, trial)


def test_best_first_equals_bruteforce_with_exact_ties():
    # equal logits inside an offset: the rank tie-break must agree
    x = np.array([[0.0, 1.0, 1.0], [2.0, 2.0, 0.0], [1.0, 1.0, 1.0]])
    for N in range(1, 20):
        bf = top_n_bruteforce(x, N)
        _, logq, _ = candidate_lists(x, min(N, 3))
        assert [r for r, _ in top_n_best_first(logq, N)] == bf


def _node_sum(x, S):
    q = np.exp(log_marginals(x))
    return sum(np.prod([q[j, y] for j, y in enumerate(s)]) for s in S)


@pytest.mark.parametrize("V,L,N", [(2, 2, 3), (3, 2, 4), (3, 2, 6), (2, 3, 5), (3, 3, 4)])
def test_top_n_set_uniquely_maximises_node_sum(V, L, N):
    g = np.random.default_rng(100 + V * 10 + L + N)
    x = g.standard_normal((L, V)) * 1.5
    tree = build_tree(x, N, root_token=0, T=0)
    S_built = tree_strings(tree)
    best = _node_sum(x, S_built)
    sets = all_prefix_closed_sets(V, L, N)
    assert len(sets) > 1
    n_best = 0
    for S in sets:
        v = _node_sum(x, S)
        assert v <= best + 1e-12
        if abs(v - best) <= 1e-12:
            n_best += 1
            assert set(S) == S_built
    assert n_best == 1


def test_prefix_closed_enumeration_counts():
    # binary tree of depth 2: closed sets of size 1..3 are easy to count by hand
    # size 1: {0},{1}; size 2: {0,1},{0,00},{0,01},{1,10},{1,11}
    assert len(all_prefix_closed_sets(2, 2, 1)) == 2
    assert len(all_prefix_closed_sets(2, 2, 2)) == 5
    for S in all_prefix_closed_sets(3, 3, 4):
        for s in S:
            assert len(s) == 1 or s[:-1] in S


def test_special_case_L1_is_top_n():
    g = np.random.default_rng(5)
    x = g.standard_normal((1, 50))
    tree = build_tree(x, 10, root_token=7, T=3)
    assert np.array_equal(tree["token"][1:], np.argsort(-x[0], kind="stable")[:10])
    assert np.all(tree["parent"][1:] == 0) and np.all(tree["depth"][1:] == 1)


def test_special_case_point_mass_gives_chain():
    L, V = 6, 40
    g = np.random.default_rng(6)
    want = g.integers(0, V, size=L)
    x = np.full((L, V), -80.0)
    x[np.arange(L), want] = 0.0
    tree = build_tree(x, 4, root_token=1, T=0)
    assert tree["token"][1:].tolist() == want[:4].tolist()
    assert tree["parent"].tolist() == [-1, 0, 1, 2, 3]


def test_special_case_n1():
    g = np.random.default_rng(7)
    x = g.standard_normal((5, 30))
    tree = build_tree(x, 1, root_token=2, T=11)
    assert tree["token"].tolist() == [2, int(np.argmax(x[0]))]


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = [p.split() for p in line.split("|")]
            rows.append(dict(N=int(parts[0][0]), token=list(map(int, parts[1])),
                             parent=list(map(int, parts[2])), depth=list(map(int, parts[3])),
                             anc=list(map(int, parts[4]))))
    return rows


@pytest.mark.parametrize("case", _golden_rows(), ids=lambda c: f"N{c['N']}")
def test_golden_hand_derived_tree(case):
    x = np.log(np.array([[0.2, 0.5, 0.3], [0.1, 0.7, 0.2]]))
    tree = build_tree(x, case["N"], root_token=9, T=100)
    assert tree["token"].tolist() == case["token"]
    assert tree["parent"].tolist() == case["parent"]
    assert tree["depth"].tolist() == case["depth"]
    assert [int(a) for a in tree["anc"][:, 0]] == case["anc"]
    assert tree["pos_id"].tolist() == [100 + d for d in case["depth"]]
    # scores are log pi_hat of each row's string
    want = {1: .5, 2: .3, 3: .2}
    for i in range(1, 4):
        assert abs(tree["score"][i] - np.log(want[i])) < 1e-12


def check_tree_invariants(tree, N, L, T):
    token, parent, depth, anc = tree["token"], tree["parent"], tree["depth"], tree["anc"]
    rows = N + 1
    assert len(token) == rows and parent[0] == -1 and depth[0] == 0
    strings = set()
    for i in range(1, rows):
        p = parent[i]
        assert 0 <= p < i                      # topological: parent first
        assert depth[i] == depth[p] + 1 <= L
        assert tree["score"][i] <= tree["score"][p]
        for k in range(rows):                  # anc = self + ancestors + root
            chain = set()
            u = i
            while u != -1:
                chain.add(u)
                u = parent[u]
            assert is_ancestor(tree, i, k) == (k in chain)
        s, u = [], i
        while u != 0:
            s.append(int(token[u]))
            u = parent[u]
        strings.add(tuple(reversed(s)))
    assert len(strings) == N                   # distinct strings: |S| = N
    for s in strings:                          # prefix-closed
        assert len(s) == 1 or s[:-1] in strings
    assert np.array_equal(tree["pos_id"], T + depth)
    # canonical order: depth asc, then parent row asc, then own rank asc
    keys = [(int(depth[i]), int(parent[i]), tree["ranks"][i][-1]) for i in range(1, rows)]
    assert keys == sorted(keys)


@pytest.mark.parametrize("N", [15, 31, 63, 127, 255])
def test_invariants_full_vocab_shape(N):
    g = np.random.default_rng(N)
    x = g.standard_normal((15, 2000)).astype(np.float32)
    tree = build_tree(x, N, root_token=5, T=4096)
    check_tree_invariants(tree, N, 15, 4096)


def test_pack_rejects_non_prefix_closed():
    _, logq, _ = candidate_lists(np.zeros((2, 3)), 3)
    tok = np.array([[0, 1, 2], [0, 1, 2]])
    with pytest.raises(ValueError):
        pack_tree([(0,), (1, 0)], tok, logq, 0, 0)


def test_mutation_wrong_successor_rule_is_caught():
    # A plausible mistake: pushing the next sibling only for rank-0 nodes.
    def broken(logq, N):
        import heapq
        from oracle.tree import node_key
        L, K = logq.shape
        heap = [(node_key(logq[0, 0], (0,)), (0,), float(logq[0, 0]))]
        out = []
        while len(out) < N and heap:
            _, r, s = heapq.heappop(heap)
            out.append((r, s))
            if len(r) < L:
                heapq.heappush(heap, (node_key(s + logq[len(r), 0], r + (0,)), r + (0,), s + logq[len(r), 0]))
            if r[-1] == 0 and K > 1:
                sib = r[:-1] + (1,)
                ss = sum(logq[j, k] for j, k in enumerate(sib))
                heapq.heappush(heap, (node_key(ss, sib), sib, ss))
        return out
    g = np.random.default_rng(11)
    caught = False
    for _ in range(20):
        x = g.standard_normal((3, 4))
        _, logq, _ = candidate_lists(x, 4)
        if [r for r, _ in broken(logq, 8)] != top_n_bruteforce(x, 8):
            caught = True
            break
    assert caught
