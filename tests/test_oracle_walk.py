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


# ---------------------------------------------------------- tie-aware gate

def _chain_setup(seed=9, L=7, V=50, N=31):
    from oracle.walk import walk_gated  # noqa: F401
    g = np.random.default_rng(seed)
    tree = build_tree(g.standard_normal((L, V)), N, root_token=0, T=0)
    u, chain = 0, []
    while True:
        kids = [c for c in range(N + 1) if tree["parent"][c] == u]
        if not kids:
            break
        u = max(kids, key=lambda c: tree["score"][c])
        chain.append(u)
    argmax = np.full(N + 1, V + 1)
    u = 0
    for c in chain:
        argmax[u] = tree["token"][c]
        u = c
    return tree, argmax, chain, L


@pytest.mark.parametrize("seed", range(6))
def test_gate_off_is_the_plain_walk(seed):
    from oracle.walk import walk_gated
    g = np.random.default_rng(100 + seed)
    L, V, N = 5, 6, 20
    tree = build_tree(g.standard_normal((L, V)) * 2, N, root_token=0, T=0)
    argmax = g.integers(0, V, size=N + 1)
    for i in range(N + 1):
        kids = [c for c in range(N + 1) if tree["parent"][c] == i]
        if kids and g.random() < 0.7:
            argmax[i] = tree["token"][kids[0]]
    gap = g.uniform(0.0, 3.0, size=N + 1)
    want = walk(tree, argmax, L)
    for thr in (0.0, -1.0, -np.inf):
        a, path, acc, nr, gated = walk_gated(tree, argmax, gap, L, thr)
        assert (a, path, acc, nr) == want and not gated


def test_gate_stops_at_the_first_near_tie_on_the_path():
    from oracle.walk import walk_gated
    tree, argmax, chain, L = _chain_setup()
    rows = len(tree["token"])
    gap = np.full(rows, 5.0)
    k = 2                                   # the row reached after 2 steps is a near-tie
    gap[chain[k - 1]] = 1e-4
    gap[[r for r in range(rows) if r not in chain and r != 0][:5]] = 0.0   # off the path: ignored
    a, path, acc, nr, gated = walk_gated(tree, argmax, gap, L, 1e-3)
    assert gated and a == k and path[1:] == chain[:k]
    assert nr == argmax[chain[k - 1]]
    # a threshold below the margin lets the walk through to the end
    a2, path2, _, nr2, gated2 = walk_gated(tree, argmax, gap, L, 1e-5)
    assert not gated2 and path2[1:] == chain and a2 == len(chain)


def test_gate_at_the_root_and_infinite_threshold():
    from oracle.walk import walk_gated
    tree, argmax, chain, L = _chain_setup(seed=3)
    gap = np.full(len(tree["token"]), 2.0)
    a, path, acc, nr, gated = walk_gated(tree, argmax, gap, L, np.inf)
    assert gated and a == 0 and path == [0] and acc == [] and nr == argmax[0]


def test_gate_matches_set_form_cut_at_the_first_near_tie():
    # gated a = min(A(S), depth of the first visited row with a small margin)
    from oracle.walk import walk_gated
    g = np.random.default_rng(77)
    L, V, N = 6, 5, 30
    for trial in range(20):
        tree = build_tree(g.standard_normal((L, V)) * 2, N, root_token=0, T=0)
        argmax = np.array([tree["token"][[c for c in range(N + 1) if tree["parent"][c] == i][0]]
                           if any(tree["parent"][c] == i for c in range(N + 1)) else 0
                           for i in range(N + 1)])
        gap = g.uniform(0, 1, size=N + 1)
        thr = 0.2
        a_plain, path, _, _ = walk(tree, argmax, L)
        cut = next((d for d, r in enumerate(path) if gap[r] < thr), None)
        a, _, _, _, gated = walk_gated(tree, argmax, gap, L, thr)
        assert a == (a_plain if cut is None else min(a_plain, cut))
        assert gated == (cut is not None)
