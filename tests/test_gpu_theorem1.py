"""Theorem 1 on the GPU: GLANCE rounds run through the C ABI on the fp32 toy
target emit exactly the oracle's greedy autoregressive tokens.

The verify path (tree build, ancestor-masked attention, LM head argmax,
walk + commit) runs in the library; the toy target's dense layers (embedding,
RMSNorm, projections, RoPE, SwiGLU) are test-harness torch ops in fp32 on the
GPU, since they are not part of the verify path.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle.toy import ToyTarget, greedy_ar

pytestmark = pytest.mark.gpu
CFG = W.TOY


class GpuToy:
    def __init__(self, weights, dev, cap):
        import tree_verified_block_gb300 as g
        self.g = g
        f = lambda a: torch.tensor(np.asarray(a), dtype=torch.float32, device=dev)
        self.dev = dev
        self.emb = f(weights["emb"])
        self.layers = [{k: f(v) for k, v in lw.items()} for lw in weights["layers"]]
        self.Wlm = f(weights["Wlm"]).contiguous()
        D = CFG["D"]
        self.inv_freq = torch.tensor(CFG["theta"] ** (-np.arange(0, D, 2, dtype=np.float64) / D),
                                     dtype=torch.float64, device=dev)
        self.t_len = torch.zeros(1, dtype=torch.int32, device=dev)
        self.kv = [g.KVLayer(torch.zeros((CFG["Hkv"], cap, D), device=dev),
                             torch.zeros((CFG["Hkv"], cap, D), device=dev), self.t_len)
                   for _ in self.layers]
        self.ws_attn = g.workspace(1 << 20, dev)

    def _rms(self, x):
        return x / torch.sqrt((x * x).mean(dim=-1, keepdim=True) + CFG["eps"])

    def _rope(self, x, pos):
        ang = pos.to(torch.float64)[:, None] * self.inv_freq[None, :]
        cos = torch.cat([torch.cos(ang), torch.cos(ang)], -1).float()[:, None, :]
        sin = torch.cat([torch.sin(ang), torch.sin(ang)], -1).float()[:, None, :]
        half = x.shape[-1] // 2
        rot = torch.cat([-x[..., half:], x[..., :half]], -1)
        return x * cos + rot * sin

    def forward(self, tokens, pos, tree, T):
        Hq, Hkv, D = CFG["Hq"], CFG["Hkv"], CFG["D"]
        R = tokens.shape[0]
        x = self.emb[tokens.long()]
        for lw, kv in zip(self.layers, self.kv):
            hn = self._rms(x)
            q = self._rope((hn @ lw["Wq"]).view(R, Hq, D), pos).contiguous()
            k = self._rope((hn @ lw["Wk"]).view(R, Hkv, D), pos)
            v = (hn @ lw["Wv"]).view(R, Hkv, D)
            kv.k[:, T:T + R] = k.transpose(0, 1)
            kv.v[:, T:T + R] = v.transpose(0, 1)
            out = torch.empty_like(q)
            self.g.tree_attention(q, kv, tree, D ** -0.5, out, self.ws_attn)
            x = x + out.view(R, Hq * D) @ lw["Wo"]
            hn = self._rms(x)
            gate = hn @ lw["Wg"]
            x = x + (gate * torch.sigmoid(gate) * (hn @ lw["Wu"])) @ lw["Wd"]
        return self._rms(x).contiguous()


def chain_tree(g, rows, dev):
    tree = g.Tree(rows - 1, 16, dev)
    anc = np.zeros((rows, tree.mask_words), dtype=np.uint64)
    for i in range(rows):
        for k in range(i + 1):
            anc[i, k // 64] |= np.uint64(1) << np.uint64(k % 64)
    tree.anc.copy_(torch.from_numpy(anc.view(np.int64)))
    return tree


def glance_on_gpu(weights, Y, dev, n_tokens=64):
    import tree_verified_block_gb300 as g
    L, V, N = CFG["L"], CFG["V"], CFG["N"]
    prompt = weights["prompt"]
    P = len(prompt)
    toy = GpuToy(weights, dev, cap=P + n_tokens + N + 4)
    # prefill: the prompt as a chain "tree" at T = 0 (causal attention)
    pre = chain_tree(g, P, dev)
    toks = torch.tensor(prompt, dtype=torch.int32, device=dev)
    h = toy.forward(toks, torch.arange(P, device=dev, dtype=torch.int32), pre, 0)
    am = torch.empty(N + 1, dtype=torch.int32, device=dev)
    gap = torch.empty(N + 1, dtype=torch.float32, device=dev)
    ws_lm = g.workspace(g.lmhead_argmax_workspace_bytes(N + 1, CFG["d"], V, torch.float32), dev)
    g.lmhead_argmax(h[P - 1:P], toy.Wlm, am[:1], gap[:1], None, ws_lm)
    root = am[:1].clone()
    toy.t_len.fill_(P)
    emitted = [int(root.item())]
    tree = g.Tree(N, L, dev)
    ws_tree = g.workspace(g.build_tree_workspace_bytes(L, V, N), dev)
    ws_c = g.workspace(g.accept_commit_workspace_bytes(len(toy.kv)), dev)
    n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
    acc = torch.zeros(L, dtype=torch.int32, device=dev)
    T = P
    accepted = []
    while len(emitted) < n_tokens:
        r = len(emitted) - 1
        x = torch.from_numpy(W.toy_draft_logits(Y, r, L, V)).to(dev)
        g.build_tree(x, N, root, toy.t_len, tree, ws_tree)
        h = toy.forward(tree.token, tree.pos_id, tree, T)
        g.lmhead_argmax(h, toy.Wlm, am, gap, None, ws_lm)
        g.accept_commit(tree, am, toy.kv, n_acc, acc, root, ws_c)
        a = int(n_acc.item())
        emitted += acc[:a].cpu().tolist() + [int(root.item())]
        T += a + 1
        assert int(toy.t_len.item()) == T
        accepted.append(a)
    return emitted[:n_tokens], accepted


def test_theorem1_toy_gpu(dev, clean_status):
    weights = W.toy_weights(0)
    Y, min_gap = greedy_ar(ToyTarget(weights, CFG), weights["prompt"], CFG["n_tokens"] + CFG["L"])
    out, accepted = glance_on_gpu(weights, Y, dev)
    assert out == Y[:CFG["n_tokens"]]
    assert max(accepted) >= 3
    assert min_gap > 1e-5


def test_theorem1_toy_gpu_flat_drafts(dev, clean_status, monkeypatch):
    # uninformative drafts: the output is still greedy AR, one or two tokens a round
    weights = W.toy_weights(0)
    Y, _ = greedy_ar(ToyTarget(weights, CFG), weights["prompt"], 40)
    monkeypatch.setattr(W, "toy_draft_logits",
                        lambda Y, r, L, V, **k: np.zeros((L, V), np.float32))
    out, _ = glance_on_gpu(weights, Y, dev, n_tokens=24)
    assert out == Y[:24]
