"""Pins for the oracle's acceptance walk, A(S) and commit (CPU)."""
import numpy as np
import pytest

from oracle.tree import build_tree
from oracle.walk import accepted_length_set_form, commit, tree_strings, walk


def _greedy_stream_from_argmax(tree, argmax, L):
    """Y as the walk sees it: follow argmax from the root while in the tree."""
    token, parent = tree["token"], tree["parent"]
    u, Y = 0, []
    while True:
        t = int(argmax[u])
        Y.append(t)
        kids = [c for c in range(len(token)) if parent[c] == u and token[c] == t]
        if not kids or tree["depth"][u] >= L:
            return Y
        u = kids[0]


@pytest.mark.parametrize("seed", range(8))
def test_set_form_equals_traversal(seed):
    g = np.random.default_rng(seed)
    L, V, N = 5, 6, 20
    x = g.standard_normal((L, V)) * 2
    tree = build_tree(x, N, root_token=0, T=0)
    # argmax per row: mostly the row's best child, sometimes a random token
    argmax = g.integers(0, V, size=N + 1)
    for i in range(N + 1):
        kids = [c for c in range(N + 1) if tree["parent"][c] == i]
        if kids and g.random() < 0.7:
            argmax[i] = tree["token"][kids[0]]
    a, path, acc, new_root = walk(tree, argmax, L)
    Y = _greedy_stream_from_argmax(tree, argmax, L)
    S = tree_strings(tree)
    assert a == accepted_length_set_form(S, Y)
    assert acc == Y[:a] and new_root == Y[a]
    assert path[0] == 0 and len(path) == a + 1


def test_planted_path_depth():
    L, V, N = 7, 50, 31
    g = np.random.default_rng(9)
    x = g.standard_normal((L, V))
    tree = build_tree(x, N, root_token=0, T=0)
    # plant the highest-score child chain down to the deepest row on it
    u, chain = 0, []
    while True:
        kids = [c for c in range(N + 1) if tree["parent"][c] == u]
        if not kids:
            break
        u = max(kids, key=lambda c: tree["score"][c])
        chain.append(u)
    argmax = np.full(N + 1, V + 1)   # a token no row has
    u = 0
    for c in chain:
        argmax[u] = tree["token"][c]
        u = c
    a, path, acc, new_root = walk(tree, argmax, L)
    assert a == len(chain) and path[1:] == chain and new_root == V + 1


def test_depth_L_leaf_stops():
    # a chain of depth L: the walk stops at depth L even if argmax "matches"
    L = 3
    x = np.full((L, 4), -50.0)
    x[:, 1] = 0
    tree = build_tree(x, 3, root_token=2, T=0)
    argmax = np.array([1, 1, 1, 1])
    a, path, acc, new_root = walk(tree, argmax, L)
    assert a == 3 and acc == [1, 1, 1] and new_root == 1


def test_commit_overlapping_rows():
    g = np.random.default_rng(3)
    T, R, D = 5, 8, 4
    k = g.standard_normal((2, 3, T + R + 2, D))
    v = g.standard_normal((2, 3, T + R + 2, D))
    k0, v0 = k.copy(), v.copy()
    path = [0, 2, 3, 7]              # dest T+2 is the source of path[1]
    newT = commit(k, v, T, path)
    assert newT == T + 4
    assert np.array_equal(k[..., :T, :], k0[..., :T, :])
    for i, p in enumerate(path):
        assert np.array_equal(k[..., T + i, :], k0[..., T + p, :])
        assert np.array_equal(v[..., T + i, :], v0[..., T + p, :])
    # slots past the committed rows are untouched
    assert np.array_equal(k[..., T + 4:, :], k0[..., T + 4:, :])


def test_mutation_commit_without_read_first_is_caught():
    # writing each destination before reading later sources corrupts path [0,2,3]
    T, D = 0, 2
    k = np.arange(5 * D, dtype=float).reshape(1, 5, D)
    k0 = k.copy()
    path = [0, 2, 3]
    for i, p in enumerate(path):
        k[..., T + i, :] = k[..., T + p, :]
    # the in-order version happens to work here: move 2->1, 3->2 reads 3 first;
    # the reverse order overwrites slot 2 before it is read
    k2 = k0.copy()
    for i, p in reversed(list(enumerate(path))):
        k2[..., T + i, :] = k2[..., T + p, :]
    assert not np.array_equal(k2[..., 1, :], k0[..., 2, :])
    kk, vv = k0.copy(), k0.copy()
    commit(kk, vv, T, path)
    assert np.array_equal(kk[..., 1, :], k0[..., 2, :]) and np.array_equal(kk[..., 2, :], k0[..., 3, :])
