"""Pins for the shared-budget, entropy-keyed builder oracle (CPU)."""
import itertools

import numpy as np
import pytest

from oracle.marginals import log_marginals
from oracle.shared_budget import entropy_keyed_log_weight, shared_budget_trees
from oracle.tree import all_prefix_closed_sets, build_tree


def _node_sum(x, S):
    lq = log_marginals(np.asarray(x, dtype=np.float64))
    return sum(np.exp(sum(lq[j, t] for j, t in enumerate(s))) for s in S)


def _strings(tree):
    out = []
    for i in range(1, len(tree["token"])):
        if tree["parent"][i] < 0:
            continue
        s, u = [], i
        while u != 0:
            s.append(int(tree["token"][u]))
            u = int(tree["parent"][u])
        out.append(tuple(reversed(s)))
    return out


def test_one_request_is_the_plain_builder():
    g = np.random.default_rng(1)
    x = g.standard_normal((4, 9))
    trees, n, _ = shared_budget_trees([x], 12, 20, [5], [30])
    ref = build_tree(x, 12, 5, 30)
    assert n.tolist() == [12]
    for k in ("token", "parent", "depth", "pos_id"):
        assert np.array_equal(trees[0][k][:13], ref[k])
    assert np.all(trees[0]["parent"][13:] == -1) and np.all(trees[0]["token"][13:] == -1)


@pytest.mark.parametrize("seed", range(6))
def test_global_best_first_maximises_weighted_node_sum(seed):
    # brute force over every split of the budget and every prefix-closed set
    g = np.random.default_rng(seed)
    V, L, N_max, N_total = 3, 2, 4, 5
    xs = [g.standard_normal((L, V)) * 1.5 for _ in range(2)]
    log_w = g.uniform(-1.0, 1.0, size=2)
    trees, n, keys = shared_budget_trees(xs, N_total, N_max, [0, 0], [0, 0], log_w)
    got = sum(np.exp(log_w[r]) * _node_sum(xs[r], _strings(trees[r])) for r in range(2))
    best = -np.inf
    for n0 in range(0, N_max + 1):
        n1 = N_total - n0
        if not 0 <= n1 <= N_max:
            continue
        v0 = max((_node_sum(xs[0], S) for S in all_prefix_closed_sets(V, L, n0)), default=0.0) if n0 else 0.0
        v1 = max((_node_sum(xs[1], S) for S in all_prefix_closed_sets(V, L, n1)), default=0.0) if n1 else 0.0
        best = max(best, np.exp(log_w[0]) * v0 + np.exp(log_w[1]) * v1)
    assert abs(got - best) < 1e-12
    assert n.sum() == N_total


def test_equal_weights_and_drafts_split_evenly_and_weight_dominates():
    x = np.random.default_rng(2).standard_normal((5, 40))
    _, n, _ = shared_budget_trees([x, x, x], 30, 20, [1, 2, 3], [0, 0, 0])
    assert n.tolist() == [10, 10, 10]
    _, n, _ = shared_budget_trees([x, x, x], 30, 20, [1, 2, 3], [0, 0, 0], log_w=[0.0, 50.0, 0.0])
    assert n.tolist() == [5, 20, 5]
    _, n, _ = shared_budget_trees([x, x], 100, 20, [1, 2], [0, 0])
    assert n.tolist() == [20, 20]  # capacity caps each round
    _, n, _ = shared_budget_trees([x, x], 1, 20, [1, 2], [0, 0])
    assert n.tolist() == [1, 0]    # ties go to the lower round


def test_entropy_keyed_weight_closed_form_and_shape():
    # V(H) = p_m (1 - p_m^L), logit p_m = b0 - b1 H (Equations 2 and 5)
    b0, b1, L = 0.96, 0.63, 15
    H = np.linspace(0.0, 8.0, 81)
    lw = entropy_keyed_log_weight(H, b0, b1, L)
    pm = 1 / (1 + np.exp(-(b0 - b1 * H)))
    assert np.allclose(np.exp(lw), pm * (1 - pm ** L), rtol=1e-12)
    # small when acceptance is hopeless (high H) or already deep (p_m -> 1)
    assert np.exp(entropy_keyed_log_weight(-40.0, b0, b1, L)) < 1e-9
    assert np.exp(entropy_keyed_log_weight(40.0, b0, b1, L)) < 1e-9
    # the peak sits where d/dp (p - p^(L+1)) = 0: p* = (L + 1)^(-1/L)
    b0, b1 = 3.0, 1.0
    Hs = np.linspace(-5.0, 10.0, 150001)
    peak = Hs[np.argmax(entropy_keyed_log_weight(Hs, b0, b1, L))]
    p_star = (L + 1.0) ** (-1.0 / L)
    assert abs(peak - (b0 - np.log(p_star / (1 - p_star))) / b1) < 1e-3
