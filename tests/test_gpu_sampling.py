"""Sampling-mode LM head on the GPU vs the oracle (same Philox4x32-10 noise,
fp64 logits and logs there): drawn tokens bit-exact where the oracle's top-2
margin of the perturbed values exceeds 1e-3, margins within 2e-2 (bf16) /
1e-3 (fp32); the draws follow softmax(l / T) (chi-square); and GLANCE rounds
on the toy target with position-keyed sampling emit the oracle's sampled
autoregressive tokens of the same seed."""
import numpy as np
import pytest
import torch
from scipy import stats

import workloads as W
from _util import bf16_tensor
from oracle.bf16 import bf16_bits_to_f64
from oracle.sampling import lmhead_sample as o_sample
from oracle.toy import ToyTarget, greedy_ar, sample_pick

pytestmark = pytest.mark.gpu


def gpu_sample(h, Wt, inv_t, seed, pos, seq, dev):
    import tree_verified_block_gb300 as g
    M, d = h.shape
    V = Wt.shape[1]
    tok = torch.full((M,), -1, dtype=torch.int32, device=dev)
    gap = torch.full((M,), float("nan"), dtype=torch.float32, device=dev)
    ws = g.workspace(g.lmhead_argmax_workspace_bytes(M, d, V, h.dtype), dev)
    p = torch.tensor(pos, dtype=torch.int32, device=dev)
    s = None if seq is None else torch.tensor(seq, dtype=torch.int32, device=dev)
    g.lmhead_sample(h, Wt, inv_t, seed, p, s, tok, gap, ws)
    return tok.cpu().numpy(), gap.cpu().numpy()


@pytest.mark.parametrize("M,d,V,inv_t", [(16, 128, 1000, 1.0), (200, 256, 3000, 0.7),
                                         (512, 128, 2048, 1.5), (64, 4096, 151936, 1.0)])
def test_bf16_sample_matches_oracle(dev, clean_status, M, d, V, inv_t):
    gen = W.rng(M, d, V, 9)
    hb = W.normal_bf16(gen, (M, d))
    Wb = W.normal_bf16(gen, (d, V), std=0.03)
    pos = (1000 + np.arange(M) * 3).tolist()
    seq = (np.arange(M) % 5).tolist()
    tok, gap = gpu_sample(bf16_tensor(hb, dev), bf16_tensor(Wb, dev), inv_t, 0xABCDEF0123, pos, seq, dev)
    want, wgap = o_sample(bf16_bits_to_f64(hb), bf16_bits_to_f64(Wb), inv_t, 0xABCDEF0123, pos, seq)
    sure = wgap > 1e-3
    assert sure.mean() > 0.9
    assert np.array_equal(tok[sure], want[sure])
    assert np.abs(gap - wgap).max() < 2e-2


def test_f32_sample_matches_oracle(dev, clean_status):
    gen = np.random.default_rng(4)
    M, d, V = 16, 128, 512
    h = gen.standard_normal((M, d)).astype(np.float32)
    Wm = (gen.standard_normal((d, V)) * 0.1).astype(np.float32)
    pos = list(range(64, 64 + M))
    tok, gap = gpu_sample(torch.from_numpy(h).to(dev), torch.from_numpy(Wm).to(dev), 1.0, 77, pos, None, dev)
    want, wgap = o_sample(h.astype(np.float64), Wm.astype(np.float64), 1.0, 77, pos)
    sure = wgap > 1e-3
    assert np.array_equal(tok[sure], want[sure])
    assert np.abs(gap - wgap).max() < 1e-3


@pytest.mark.parametrize("inv_t", [1.0, 0.5])
def test_bf16_draws_follow_softmax(dev, clean_status, inv_t):
    # one-hot rows pick row 0 of W, so every row's logits are W[0]
    M, d, V = 512, 64, 16
    logits = np.array([0.5, -1.0, 1.75, 0.0, 1.0, -0.5, 0.75, -2.0,
                       0.25, 1.5, -0.25, 0.0, -1.5, 0.5, 1.25, -0.75], dtype=np.float32)
    Wb = np.zeros((d, V), dtype=np.float32)
    Wb[0] = logits
    hb = np.zeros((M, d), dtype=np.float32)
    hb[:, 0] = 1.0
    h = bf16_tensor(W.to_bf16_bits(hb), dev)
    Wt = bf16_tensor(W.to_bf16_bits(Wb), dev)
    counts = np.zeros(V, dtype=np.int64)
    for k in range(30):
        tok, _ = gpu_sample(h, Wt, inv_t, 31337, (np.arange(M) + k * M).tolist(), None, dev)
        counts += np.bincount(tok, minlength=V)
    p = np.exp(logits.astype(np.float64) * inv_t)
    p /= p.sum()
    assert stats.chisquare(counts, counts.sum() * p).pvalue > 1e-4


def test_sampled_glance_rounds_equal_sampled_autoregression(dev, clean_status):
    import tree_verified_block_gb300 as g
    from test_gpu_theorem1 import CFG, GpuToy, chain_tree
    weights = W.toy_weights(0)
    target = ToyTarget(weights, CFG)
    seed, inv_t = 4242, 1.0
    n_tokens = 48
    Y, _ = greedy_ar(target, weights["prompt"], n_tokens + CFG["L"], pick=sample_pick(target, inv_t, seed))
    L, V, N = CFG["L"], CFG["V"], CFG["N"]
    prompt = weights["prompt"]
    P = len(prompt)
    toy = GpuToy(weights, dev, cap=P + n_tokens + N + 4)
    pre = chain_tree(g, P, dev)
    toks = torch.tensor(prompt, dtype=torch.int32, device=dev)
    h = toy.forward(toks, torch.arange(P, device=dev, dtype=torch.int32), pre, 0)
    tok = torch.empty(N + 1, dtype=torch.int32, device=dev)
    gap = torch.empty(N + 1, dtype=torch.float32, device=dev)
    ws_lm = g.workspace(g.lmhead_argmax_workspace_bytes(N + 1, CFG["d"], V, torch.float32), dev)
    g.lmhead_sample(h[P - 1:P], toy.Wlm, inv_t, seed, torch.tensor([P], dtype=torch.int32, device=dev),
                    None, tok[:1], gap[:1], ws_lm)
    root = tok[:1].clone()
    toy.t_len.fill_(P)
    emitted = [int(root.item())]
    tree = g.Tree(N, L, dev)
    ws_tree = g.workspace(g.build_tree_workspace_bytes(L, V, N), dev)
    ws_c = g.workspace(g.accept_commit_workspace_bytes(len(toy.kv)), dev)
    n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
    acc = torch.zeros(L, dtype=torch.int32, device=dev)
    T, accepted = P, []
    while len(emitted) < n_tokens:
        r = len(emitted) - 1
        x = torch.from_numpy(W.toy_draft_logits(Y, r, L, V)).to(dev)
        g.build_tree(x, N, root, toy.t_len, tree, ws_tree)
        h = toy.forward(tree.token, tree.pos_id, tree, T)
        g.lmhead_sample(h, toy.Wlm, inv_t, seed, tree.pos_id + 1, None, tok, gap, ws_lm)
        g.accept_commit(tree, tok, toy.kv, n_acc, acc, root, ws_c)
        a = int(n_acc.item())
        emitted += acc[:a].cpu().tolist() + [int(root.item())]
        T += a + 1
        accepted.append(a)
    assert emitted[:n_tokens] == Y[:n_tokens]
    assert max(accepted) >= 2
