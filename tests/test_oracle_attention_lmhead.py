"""Pins for the oracle's tree attention and LM head (CPU)."""
import numpy as np
import pytest

from oracle.attention import causal_attention, tree_attention
from oracle.lmhead import lmhead_argmax
from oracle.tree import pack_tree


def chain_tree(n_rows):
    """A chain: row i's ancestors are rows 0..i."""
    nodes = [tuple([0] * d) for d in range(1, n_rows)]
    tok = np.zeros((max(1, n_rows - 1), 1), dtype=np.int64)
    logq = np.zeros((max(1, n_rows - 1), 1))
    return pack_tree(nodes, tok, logq, 0, 0)


@pytest.mark.parametrize("T,R", [(0, 5), (7, 9), (3, 70)])
def test_chain_tree_is_causal_attention(T, R):
    g = np.random.default_rng(T + R)
    Hq, Hkv, D = 4, 2, 16
    k_seq = g.standard_normal((T + R, Hkv, D))
    v_seq = g.standard_normal((T + R, Hkv, D))
    q_seq = g.standard_normal((T + R, Hq, D))
    tree = chain_tree(R)
    kc = k_seq.transpose(1, 0, 2).copy()
    vc = v_seq.transpose(1, 0, 2).copy()
    out = tree_attention(q_seq[T:], kc, vc, T, tree["anc"], 1 / np.sqrt(D))
    ref = causal_attention(q_seq, k_seq, v_seq, 1 / np.sqrt(D))[T:]
    assert np.allclose(out, ref, atol=1e-13, rtol=0)


def test_single_root_row_sees_only_itself():
    g = np.random.default_rng(1)
    kc, vc = g.standard_normal((2, 1, 4, 8)), g.standard_normal((2, 1, 4, 8))
    tree = chain_tree(1)
    out = tree_attention(g.standard_normal((1, 2, 8)), kc[0], vc[0], 0, tree["anc"], 0.3)
    assert np.array_equal(out[0, 0], vc[0][0, 0]) and np.array_equal(out[0, 1], vc[0][0, 0])


def test_identical_keys_average_visible_values():
    g = np.random.default_rng(2)
    T, D = 6, 8
    nodes = [(0,), (1,), (0, 0)]
    tree = pack_tree(nodes, np.array([[3, 4], [5, 6]]), np.zeros((2, 2)), 1, T)
    R = 4
    kc = np.tile(g.standard_normal(D), (1, T + R, 1))
    vc = g.standard_normal((1, T + R, D))
    out = tree_attention(g.standard_normal((R, 1, D)), kc, vc, T, tree["anc"], 1.0)
    # row order: root, (0,), (1,), (0,0); row 3 sees prefix + rows {0, 1, 3}
    vis = list(range(T)) + [T + 0, T + 1, T + 3]
    assert np.allclose(out[3, 0], vc[0, vis].mean(axis=0), atol=1e-14)
    vis2 = list(range(T)) + [T + 0, T + 2]
    assert np.allclose(out[2, 0], vc[0, vis2].mean(axis=0), atol=1e-14)


def test_two_key_closed_form():
    # one prefix key with score a, the root with score b: p = sigmoid(a - b)
    q = np.array([[[1.0, 0.0]]])
    kc = np.array([[[2.0, 0.0], [0.5, 0.0]]])
    vc = np.array([[[1.0, 0.0], [0.0, 1.0]]])
    tree = chain_tree(1)
    out = tree_attention(q, kc, vc, 1, tree["anc"], 1.0)
    p = 1 / (1 + np.exp(-(2.0 - 0.5)))
    assert np.allclose(out[0, 0], [p, 1 - p], atol=1e-15)


def test_gqa_head_mapping():
    # q heads 0,1 read kv head 0, heads 2,3 read kv head 1
    g = np.random.default_rng(3)
    kc = g.standard_normal((2, 5, 4))
    vc = np.stack([np.zeros((5, 4)), np.ones((5, 4))])
    tree = chain_tree(1)
    out = tree_attention(g.standard_normal((1, 4, 4)), kc, vc, 4, tree["anc"], 1.0)
    assert np.allclose(out[0, :2], 0) and np.allclose(out[0, 2:], 1)


def test_dense_mask_formulation_agrees():
    # the same attention written as a dense -inf mask over all slots
    g = np.random.default_rng(4)
    T, Hq, Hkv, D = 10, 4, 2, 8
    nodes = [(0,), (1,), (0, 0), (0, 1), (1, 0), (0, 0, 0)]
    tree = pack_tree(nodes, g.integers(0, 9, (3, 2)), np.zeros((3, 2)), 1, T)
    R = 7
    q = g.standard_normal((R, Hq, D))
    kc, vc = g.standard_normal((Hkv, T + R + 3, D)), g.standard_normal((Hkv, T + R + 3, D))
    out = tree_attention(q, kc, vc, T, tree["anc"], 0.5)
    parent = tree["parent"]
    for i in range(R):
        mask = np.full(T + R + 3, -np.inf)
        mask[:T] = 0
        u = i
        while u != -1:
            mask[T + u] = 0
            u = parent[u]
        for h in range(Hq):
            s = kc[h // 2] @ q[i, h] * 0.5 + mask
            p = np.exp(s - s.max())
            assert np.allclose(out[i, h], (p / p.sum()) @ vc[h // 2], atol=1e-13)


def test_lmhead_matches_library_argmax():
    g = np.random.default_rng(5)
    h = g.standard_normal((6, 32))
    W = g.standard_normal((32, 20000))
    arg, gap, mx = lmhead_argmax(h, W, chunk=777)
    lg = h @ W
    assert np.array_equal(arg, np.argmax(lg, axis=1))
    srt = np.sort(lg, axis=1)
    assert np.allclose(gap, srt[:, -1] - srt[:, -2], atol=1e-12)
    assert np.allclose(mx, srt[:, -1], atol=1e-12)


def test_lmhead_planted_margins():
    g = np.random.default_rng(6)
    d, V = 64, 5000
    W = g.standard_normal((d, V)) * 0.02
    want = g.integers(0, V, 8)
    h = g.standard_normal((8, d))
    for i, t in enumerate(want):
        col = W[:, t]
        h[i] += 10 * col / (col @ col)
    arg, gap, _ = lmhead_argmax(h, W)
    assert np.array_equal(arg, want)
    assert np.all(gap > 1e-3)


def test_lmhead_exact_ties_lowest_id_gap_zero():
    W = np.zeros((2, 10))
    W[0, [3, 7]] = 1.0          # tie between 3 and 7 across chunk boundaries
    W[0, 5] = 0.5
    h = np.array([[1.0, 0.0]])
    for chunk in (2, 4, 10):
        arg, gap, mx = lmhead_argmax(h, W, chunk=chunk)
        assert arg[0] == 3 and gap[0] == 0.0 and mx[0] == 1.0


# ------------------------------------------------------- next-token entropy

def test_entropy_uniform_logits_is_log_V():
    from oracle.lmhead import next_token_entropy
    d, V = 16, 1000
    H = next_token_entropy(np.ones((3, d)), np.zeros((d, V)), chunk=300)
    assert np.allclose(H, np.log(V), atol=1e-12)


def test_entropy_one_raised_logit_closed_form():
    # logits c on one token and 0 on the other V - 1: p = e^c / (e^c + V - 1),
    # H = -p ln p - (1 - p) ln((1 - p) / (V - 1))
    from oracle.lmhead import next_token_entropy
    V = 513
    for c in (0.5, 4.0, 20.0):
        W = np.zeros((1, V))
        W[0, 77] = c
        H = next_token_entropy(np.ones((1, 1)), W, chunk=100)[0]
        p = np.exp(c) / (np.exp(c) + V - 1)
        want = -p * np.log(p) - (1 - p) * np.log((1 - p) / (V - 1))
        assert abs(H - want) < 1e-12


def test_entropy_matches_scipy_and_is_shift_invariant():
    from scipy.special import softmax
    from scipy.stats import entropy
    from oracle.lmhead import next_token_entropy
    g = np.random.default_rng(5)
    h = g.standard_normal((6, 24))
    W = g.standard_normal((24, 700)) * 0.7
    H = next_token_entropy(h, W, chunk=128)
    lg = h @ W
    assert np.allclose(H, entropy(softmax(lg, axis=1), axis=1), atol=1e-10)
    # an extra input column of ones with a constant W row shifts every logit
    h2 = np.concatenate([h, np.ones((6, 1))], axis=1)
    W2 = np.concatenate([W, np.full((1, 700), 9.0)], axis=0)
    assert np.allclose(next_token_entropy(h2, W2, chunk=50), H, atol=1e-10)
