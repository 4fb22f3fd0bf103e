"""Toy decoder target, greedy autoregression and GLANCE rounds (oracle step O7).

Follows "Vision Is Not Overhead ..." (arXiv 2609.00355):
  * Section 3.1: greedy autoregression emits argmax_w p(w | x), one token per
    target forward; a speculative round commits a + 1 tokens.
  * Definition 1 and Section 4.2: one round = candidate tree from the draft
    marginals, one ancestor-masked pass over root + tree rows, greedy walk,
    commit, bonus token as the next root.
  * Theorem 1 (Section 4.2; full statement and proof in Appendix B.1): for any
    tree the rounds emit exactly the greedy autoregressive sequence.
  * Section 5.4: under sampling every committed token is a draw from the
    target's own verified row. With `pick` = a sampler whose noise is keyed by
    the predicted token's absolute position (oracle.sampling), the rounds emit
    exactly the sampled autoregressive sequence of the same seed.

The pages do not describe the toy target; it is a plain pre-norm decoder:
token embedding; per layer RMSNorm -> GQA attention with rotate-half RoPE
(theta 10000) -> residual -> RMSNorm -> SwiGLU MLP -> residual; final RMSNorm;
untied LM head; no biases; RMSNorm weight 1, eps 1e-6. Its weights come from
``workloads.toy_weights``. Arithmetic runs in the dtype given (float64 by
default, float32 for the fp32 form of Theorem 1).
"""
import numpy as np

from .lmhead import lmhead_argmax
from .sampling import lmhead_sample
from .tree import build_tree
from .walk import walk


class ToyTarget:
    def __init__(self, weights, cfg, dtype=np.float64):
        self.cfg = cfg
        self.dt = dtype
        c = lambda a: np.asarray(a, dtype=dtype)
        self.emb = c(weights["emb"])
        self.layers = [{k: c(v) for k, v in lw.items()} for lw in weights["layers"]]
        self.Wlm = c(weights["Wlm"])
        D = cfg["D"]
        self.inv_freq = (cfg["theta"] ** (-np.arange(0, D, 2, dtype=np.float64) / D))

    def new_cache(self, T_cap):
        c = self.cfg
        return [(np.zeros((c["Hkv"], T_cap, c["D"]), self.dt),
                 np.zeros((c["Hkv"], T_cap, c["D"]), self.dt)) for _ in self.layers]

    def _rmsnorm(self, x):
        ms = (x * x).mean(axis=-1, keepdims=True)
        return x / np.sqrt(ms + self.dt(self.cfg["eps"]))

    def _rope(self, x, pos):
        # x: (R, H, D); rotate-half convention
        ang = np.asarray(pos, dtype=np.float64)[:, None] * self.inv_freq[None, :]
        cos = np.concatenate([np.cos(ang), np.cos(ang)], axis=-1).astype(self.dt)[:, None, :]
        sin = np.concatenate([np.sin(ang), np.sin(ang)], axis=-1).astype(self.dt)[:, None, :]
        half = x.shape[-1] // 2
        rot = np.concatenate([-x[..., half:], x[..., :half]], axis=-1)
        return x * cos + rot * sin

    def forward(self, tokens, pos, slots, visible, cache):
        """Run rows through the target.

        tokens, pos, slots: (R,) ints; the rows' K/V are stored at cache slots
        `slots`; visible[i] lists the cache slots row i attends to (its own slot
        included). Returns the final-normed hidden states h (R, d).
        """
        c = self.cfg
        R = len(tokens)
        Hq, Hkv, D = c["Hq"], c["Hkv"], c["D"]
        group = Hq // Hkv
        scale = self.dt(1.0 / np.sqrt(D))
        x = self.emb[np.asarray(tokens)]
        for lw, (Kc, Vc) in zip(self.layers, cache):
            hn = self._rmsnorm(x)
            q = self._rope((hn @ lw["Wq"]).reshape(R, Hq, D), pos)
            k = self._rope((hn @ lw["Wk"]).reshape(R, Hkv, D), pos)
            v = (hn @ lw["Wv"]).reshape(R, Hkv, D)
            Kc[:, slots] = k.transpose(1, 0, 2)
            Vc[:, slots] = v.transpose(1, 0, 2)
            att = np.empty((R, Hq, D), self.dt)
            for i in range(R):
                vis = np.asarray(visible[i])
                for hh in range(Hq):
                    g = hh // group
                    s = (Kc[g, vis] @ q[i, hh]) * scale
                    p = np.exp(s - s.max())
                    att[i, hh] = (p / p.sum()) @ Vc[g, vis]
            x = x + att.reshape(R, Hq * D) @ lw["Wo"]
            hn = self._rmsnorm(x)
            gate = hn @ lw["Wg"]
            x = x + ((gate / (1 + np.exp(-gate))) * (hn @ lw["Wu"])) @ lw["Wd"]
        return self._rmsnorm(x)

    def logits(self, h):
        return h @ self.Wlm


def greedy_pick(target):
    """Token choice of greedy decoding: (argmax, top-2 gap) of each row."""
    def pick(h, pos):
        arg, gap, _ = lmhead_argmax(h, target.Wlm)
        return arg, gap
    return pick


def sample_pick(target, inv_temp, seed, seq=0):
    """Token choice of sampled decoding: a Gumbel-max draw from softmax(l / T)
    keyed by the absolute position of the predicted token."""
    def pick(h, pos):
        return lmhead_sample(h, target.Wlm, inv_temp, seed, pos, np.full(len(pos), seq))
    return pick


def greedy_ar(target, prompt, n_tokens, pick=None):
    """Plain autoregression (greedy unless `pick` says otherwise): returns
    (tokens, min top-2 gap seen). pick(h, pos) returns (tokens, gaps) for rows
    h whose predicted tokens sit at absolute positions pos."""
    pick = pick or greedy_pick(target)
    P = len(prompt)
    cache = target.new_cache(P + n_tokens + 1)
    slots = np.arange(P)
    h = target.forward(prompt, np.arange(P), slots, [np.arange(i + 1) for i in range(P)], cache)
    arg, gap = pick(h[-1:], np.array([P]))
    out = [int(arg[0])]
    min_gap = float(gap[0])
    t = P
    while len(out) < n_tokens:
        h = target.forward([out[-1]], [t], [t], [np.arange(t + 1)], cache)
        arg, gap = pick(h, np.array([t + 1]))
        out.append(int(arg[0]))
        min_gap = min(min_gap, float(gap[0]))
        t += 1
    return out, min_gap


def glance_decode(target, prompt, n_tokens, N, L, draft_fn, tree_override=None, pick=None):
    """GLANCE rounds on the toy target.

    draft_fn(r) returns the (L, V) draft logits of the round whose root is
    emitted token r. tree_override(r, root, T) may return a tree dict to use in
    place of the built one (Theorem 1 holds for any tree). Returns (tokens,
    per-round accepted lengths, min top-2 gap over visited rows). pick as in
    greedy_ar (greedy by default).
    """
    pick = pick or greedy_pick(target)
    P = len(prompt)
    cap = P + n_tokens + N + 2
    cache = target.new_cache(cap)
    h = target.forward(prompt, np.arange(P), np.arange(P), [np.arange(i + 1) for i in range(P)], cache)
    arg, gap = pick(h[-1:], np.array([P]))
    out = [int(arg[0])]
    min_gap = float(gap[0])
    T = P
    accepted = []
    while len(out) < n_tokens:
        r = len(out) - 1
        root = out[-1]
        tree = tree_override(r, root, T) if tree_override else build_tree(draft_fn(r), N, root, T)
        rows = len(tree["token"])
        slots = T + np.arange(rows)
        visible = []
        for i in range(rows):
            anc_rows = [k for k in range(rows) if (int(tree["anc"][i, k // 64]) >> (k % 64)) & 1]
            visible.append(np.concatenate([np.arange(T), T + np.asarray(anc_rows)]))
        h = target.forward(tree["token"], tree["pos_id"], slots, visible, cache)
        arg, gap = pick(h, np.asarray(tree["pos_id"]) + 1)
        a, path, acc, new_root = walk(tree, arg, L)
        min_gap = min([min_gap] + [float(gap[p]) for p in path])
        for Kc, Vc in cache:
            src = [T + p for p in path]
            ks, vs = Kc[:, src].copy(), Vc[:, src].copy()
            Kc[:, T:T + a + 1] = ks
            Vc[:, T:T + a + 1] = vs
        T += a + 1
        out.extend(acc)
        out.append(new_root)
        accepted.append(a)
    return out[:n_tokens], accepted, min_gap
