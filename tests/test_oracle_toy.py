"""Theorem 1 and Definition 1's packing identity on the toy target (CPU).

Theorem 1 (Section 4.2; Appendix B.1): for any candidate tree, GLANCE rounds
emit exactly the target's greedy autoregressive sequence. Definition 1: the
packed row of a depth-d node yields p(. | x . b . y_{1:d}), the same as the
unpacked causal evaluation of that sequence.
"""
import numpy as np
import pytest

import workloads as W
from oracle.lmhead import lmhead_argmax
from oracle.tree import build_tree, pack_tree
from oracle.toy import ToyTarget, glance_decode, greedy_ar

CFG = W.TOY


@pytest.fixture(scope="module")
def toy():
    w = W.toy_weights(0)
    return w, ToyTarget(w, CFG)


@pytest.fixture(scope="module")
def ar_stream(toy):
    w, tgt = toy
    Y, gap = greedy_ar(tgt, w["prompt"], CFG["n_tokens"] + CFG["L"])
    return Y, gap


def test_theorem1_planted_drafts(toy, ar_stream):
    w, tgt = toy
    Y, _ = ar_stream
    out, acc, gap = glance_decode(tgt, w["prompt"], 64, CFG["N"], CFG["L"],
                                  lambda r: W.toy_draft_logits(Y, r, CFG["L"], CFG["V"]))
    assert out == Y[:64]
    assert max(acc) >= 3          # the drafts are useful: some rounds accept deep
    assert gap > 1e-5


def test_theorem1_flat_drafts(toy, ar_stream):
    w, tgt = toy
    Y, _ = ar_stream
    out, acc, _ = glance_decode(tgt, w["prompt"], 24, CFG["N"], CFG["L"],
                                lambda r: np.zeros((CFG["L"], CFG["V"]), np.float32))
    assert out == Y[:24]


def test_theorem1_arbitrary_trees(toy, ar_stream):
    # random prefix-closed trees, unrelated to any draft
    w, tgt = toy
    Y, _ = ar_stream
    g = np.random.default_rng(42)

    def random_tree(r, root, T):
        nodes = set()
        while len(nodes) < 12:
            d = int(g.integers(1, CFG["L"] + 1))
            s = tuple(int(v) for v in g.integers(0, 3, size=d))
            for k in range(1, d + 1):
                nodes.add(s[:k])
        nodes = sorted(nodes, key=lambda s: (len(s), s))
        # rank r at offset j is token Y[r+j] for rank 0 (so some paths match)
        tok = np.empty((CFG["L"], 3), dtype=np.int64)
        for j in range(CFG["L"]):
            base = Y[r + j + 1] if r + j + 1 < len(Y) else 0
            tok[j] = [base, (base + 1) % CFG["V"], (base + 2) % CFG["V"]]
        return pack_tree(nodes, tok, np.zeros((CFG["L"], 3)), root, T)

    out, acc, _ = glance_decode(tgt, w["prompt"], 40, 12, CFG["L"], None, tree_override=random_tree)
    assert out == Y[:40]
    assert max(acc) >= 2


def test_theorem1_fp32(toy):
    w, _ = toy
    tgt32 = ToyTarget(w, CFG, dtype=np.float32)
    Y32, _ = greedy_ar(tgt32, w["prompt"], 40 + CFG["L"])
    out, _, _ = glance_decode(tgt32, w["prompt"], 40, CFG["N"], CFG["L"],
                              lambda r: W.toy_draft_logits(Y32, r, CFG["L"], CFG["V"]))
    assert out == Y32[:40]


def test_packed_equals_unpacked(toy, ar_stream):
    w, tgt = toy
    prompt = w["prompt"]
    P = len(prompt)
    root = ar_stream[0][0]
    x = np.random.default_rng(3).standard_normal((CFG["L"], CFG["V"])) * 2
    tree = build_tree(x, 15, root, P)
    rows = len(tree["token"])
    cache = tgt.new_cache(P + rows)
    tgt.forward(prompt, np.arange(P), np.arange(P), [np.arange(i + 1) for i in range(P)], cache)
    visible = []
    for i in range(rows):
        anc = [k for k in range(rows) if (int(tree["anc"][i, 0]) >> k) & 1]
        visible.append(np.concatenate([np.arange(P), P + np.asarray(anc)]))
    h_packed = tgt.forward(tree["token"], tree["pos_id"], P + np.arange(rows), visible, cache)
    lg_packed = tgt.logits(h_packed)
    for i in range(rows):
        # the unpacked sequence prompt . b . y_{1:d}, evaluated causally from scratch
        seq = [int(tree["token"][i])]
        u = tree["parent"][i]
        while u != -1:
            seq.append(int(tree["token"][u]))
            u = tree["parent"][u]
        seq = list(prompt) + seq[::-1]
        c2 = tgt.new_cache(len(seq))
        h = tgt.forward(seq, np.arange(len(seq)), np.arange(len(seq)),
                        [np.arange(t + 1) for t in range(len(seq))], c2)
        lg = tgt.logits(h[-1])
        assert np.allclose(lg, lg_packed[i], atol=1e-12, rtol=0)
        assert np.argmax(lg) == np.argmax(lg_packed[i])


def test_mutation_unmasked_tree_is_caught(toy, ar_stream):
    # Plant a mistake in the oracle: tree rows see every tree row, not only
    # their ancestors. The packing identity must then fail for some row.
    w, tgt = toy
    prompt = w["prompt"]
    P = len(prompt)
    x = np.random.default_rng(3).standard_normal((CFG["L"], CFG["V"])) * 2
    tree = build_tree(x, 15, ar_stream[0][0], P)
    rows = len(tree["token"])
    cache = tgt.new_cache(P + rows)
    tgt.forward(prompt, np.arange(P), np.arange(P), [np.arange(i + 1) for i in range(P)], cache)
    vis_all = [np.arange(P + rows)] * rows
    h_bad = tgt.forward(tree["token"], tree["pos_id"], P + np.arange(rows), vis_all, cache)
    seq = list(prompt) + [int(tree["token"][0])]
    c2 = tgt.new_cache(len(seq))
    h = tgt.forward(seq, np.arange(len(seq)), np.arange(len(seq)),
                    [np.arange(t + 1) for t in range(len(seq))], c2)
    assert not np.allclose(tgt.logits(h[-1]), tgt.logits(h_bad[0]), atol=1e-9)
