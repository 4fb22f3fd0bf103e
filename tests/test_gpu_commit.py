"""Acceptance walk + KV commit on the GPU vs the oracle: A(S), accepted
tokens, new root, T and every cache byte bit-exact."""
import numpy as np
import pytest
import torch

import workloads as W
from _util import bf16_tensor
from oracle.tree import build_tree as o_build
from oracle.walk import commit as o_commit
from oracle.walk import walk as o_walk
from test_gpu_attention import upload_tree

pytestmark = pytest.mark.gpu


def planted_argmax(ref, depth_target, V, gen):
    """argmax that follows the highest-score child chain for depth_target
    steps, then a token that is no child of the last row."""
    rows = len(ref["token"])
    am = gen.integers(0, V, size=rows).astype(np.int64)
    u, reached = 0, 0
    for _ in range(depth_target):
        kids = [c for c in range(rows) if ref["parent"][c] == u]
        if not kids:
            break
        c = max(kids, key=lambda k: (ref["score"][k], -k))
        am[u] = ref["token"][c]
        u = c
        reached += 1
    kid_tokens = {int(ref["token"][c]) for c in range(rows) if ref["parent"][c] == u}
    free = [t for t in range(V) if t not in kid_tokens][:1] if len(kid_tokens) < V else []
    if free:                       # stop the walk here
        t = int(am[u])
        while t in kid_tokens:
            t = (t + 1) % V
        am[u] = t
    else:                          # every token is a child: the walk goes on
        reached = None
    return am, reached


def run(ref, am, L, n_layers, Hkv, D, T, t_cap, dtype, dev, seed):
    import tree_verified_block_gb300 as g
    gen = W.rng(seed)
    if dtype == torch.bfloat16:
        ks = [W.normal_bf16(gen, (Hkv, t_cap, D)) for _ in range(n_layers)]
        vs = [W.normal_bf16(gen, (Hkv, t_cap, D)) for _ in range(n_layers)]
        kt = [bf16_tensor(k, dev) for k in ks]
        vt = [bf16_tensor(v, dev) for v in vs]
        host_k = [k.copy() for k in ks]
        host_v = [v.copy() for v in vs]
    else:
        host_k = [gen.standard_normal((Hkv, t_cap, D)).astype(np.float32) for _ in range(n_layers)]
        host_v = [gen.standard_normal((Hkv, t_cap, D)).astype(np.float32) for _ in range(n_layers)]
        kt = [torch.from_numpy(k.copy()).to(dev) for k in host_k]
        vt = [torch.from_numpy(v.copy()).to(dev) for v in host_v]
    t_len = torch.tensor([T], dtype=torch.int32, device=dev)
    layers = [g.KVLayer(k, v, t_len) for k, v in zip(kt, vt)]
    tree = upload_tree(ref, L, dev)
    amt = torch.from_numpy(am.astype(np.int32)).to(dev)
    n_acc = torch.full((1,), -1, dtype=torch.int32, device=dev)
    acc = torch.full((L,), -1, dtype=torch.int32, device=dev)
    nr = torch.full((1,), -1, dtype=torch.int32, device=dev)
    ws = g.workspace(g.accept_commit_workspace_bytes(n_layers), dev)
    g.accept_commit(tree, amt, layers, n_acc, acc, nr, ws)
    a, path, toks, new_root = o_walk(ref, am, L)
    assert int(n_acc.item()) == a
    assert acc.cpu().numpy()[:a].tolist() == toks
    assert int(nr.item()) == new_root
    for l in range(n_layers):
        newT = o_commit(host_k[l], host_v[l], T, path)
        gk = kt[l].view(torch.int16).cpu().numpy().view(np.uint16) if dtype == torch.bfloat16 else kt[l].cpu().numpy()
        gv = vt[l].view(torch.int16).cpu().numpy().view(np.uint16) if dtype == torch.bfloat16 else vt[l].cpu().numpy()
        assert np.array_equal(gk, host_k[l]) and np.array_equal(gv, host_v[l])
    assert int(t_len.item()) == newT
    return a, path


@pytest.mark.parametrize("depth", [0, 1, 3, 7, 15])
def test_bf16_qwen_shaped(dev, clean_status, depth):
    L, N, V = 15, 63, 151936
    x = W.draft_logits_planted(L, V, seed=300 + depth).astype(np.float64)
    ref = o_build(x, N, 5, 4096)
    am, reached = planted_argmax(ref, depth, V, np.random.default_rng(depth))
    a, path = run(ref, am, L, 4, 8, 128, 4096, 4096 + 70, torch.bfloat16, dev, seed=depth)
    assert a == reached


def test_overlapping_rows_and_wide_tree(dev, clean_status):
    # a bushy tree puts path rows far apart and lets destinations overlap sources
    L, N, V = 4, 255, 6
    x = np.random.default_rng(2).standard_normal((L, V)) * 0.3
    ref = o_build(x, N, 0, 100)
    for depth in (2, 3, 4):
        am, reached = planted_argmax(ref, depth, V, np.random.default_rng(depth))
        a, path = run(ref, am, L, 2, 2, 128, 100, 100 + 256 + 3, torch.bfloat16, dev, seed=depth)
        assert a >= 2 and (reached is None or a == reached)
        assert any(p > i for i, p in enumerate(path))


def test_depth_L_stops(dev, clean_status):
    L, V = 3, 10
    x = np.full((L, V), -30.0)
    x[:, 4] = 0.0
    ref = o_build(x, 3, 1, 20)      # a chain 4-4-4
    am = np.array([4, 4, 4, 4])
    a, _ = run(ref, am, L, 1, 2, 128, 20, 40, torch.bfloat16, dev, seed=1)
    assert a == 3


def test_fp32_cache(dev, clean_status):
    L, N, V = 7, 15, 512
    x = np.random.default_rng(9).standard_normal((L, V)) * 2
    ref = o_build(x, N, 3, 64)
    am, _ = planted_argmax(ref, 4, V, np.random.default_rng(4))
    run(ref, am, L, 2, 2, 32, 64, 64 + 20, torch.float32, dev, seed=4)


def test_capacity_error_leaves_T(dev):
    import tree_verified_block_gb300 as g
    g.reset_device_status()
    L, N = 3, 7
    x = np.random.default_rng(1).standard_normal((L, 5))
    ref = o_build(x, N, 0, 30)
    K = torch.zeros((2, 32, 128), dtype=torch.bfloat16, device=dev)
    t_len = torch.tensor([30], dtype=torch.int32, device=dev)   # 30 + 8 > 32
    layer = g.KVLayer(K, K.clone(), t_len)
    tree = upload_tree(ref, L, dev)
    am = torch.zeros(N + 1, dtype=torch.int32, device=dev)
    out = [torch.zeros(k, dtype=torch.int32, device=dev) for k in (1, L, 1)]
    g.accept_commit(tree, am, [layer], out[0], out[1], out[2], g.workspace(256, dev))
    code, _ = g.device_status()
    g.reset_device_status()
    assert code == 2 and int(t_len.item()) == 30


# ---------------------------------------------------------- tie-aware gate

def _gated_case(seed, near_tie_depth, L=15, N=63, V=40):
    from test_gpu_attention import random_tree
    ref = random_tree(N, L, 1000, seed)
    gen = W.rng(seed, 5)
    am, _ = planted_argmax(ref, 15, V, gen)
    gap = gen.uniform(0.5, 3.0, size=N + 1).astype(np.float32)
    # walk the planted chain to place a near-tie at the requested depth
    u, chain = 0, [0]
    while True:
        kids = [c for c in range(N + 1) if ref["parent"][c] == u and ref["token"][c] == am[u]]
        if not kids or ref["depth"][u] >= L:
            break
        u = kids[0]
        chain.append(u)
    if near_tie_depth is not None and near_tie_depth < len(chain):
        gap[chain[near_tie_depth]] = 1e-4
    off_path = [r for r in range(N + 1) if r not in chain][:4]
    gap[off_path] = 0.0
    return ref, am, gap, chain


@pytest.mark.parametrize("near_tie_depth,thr", [(None, 1e-3), (0, 1e-3), (2, 1e-3), (2, 1e-5),
                                                (3, 0.0)])
def test_gated_commit_matches_oracle(dev, clean_status, near_tie_depth, thr):
    import tree_verified_block_gb300 as g
    from oracle.walk import walk_gated
    L, n_layers, Hkv, D, T = 15, 2, 8, 128, 1000
    ref, am, gap, chain = _gated_case(11, near_tie_depth)
    t_cap = T + len(ref["token"]) + 8
    gen = W.rng(12)
    ks = [W.normal_bf16(gen, (Hkv, t_cap, D)) for _ in range(n_layers)]
    vs = [W.normal_bf16(gen, (Hkv, t_cap, D)) for _ in range(n_layers)]
    t_len = torch.tensor([T], dtype=torch.int32, device=dev)
    layers = [g.KVLayer(bf16_tensor(k, dev), bf16_tensor(v, dev), t_len) for k, v in zip(ks, vs)]
    tree = upload_tree(ref, L, dev)
    n_acc = torch.full((1,), -1, dtype=torch.int32, device=dev)
    acc = torch.full((L,), -1, dtype=torch.int32, device=dev)
    nr = torch.full((1,), -1, dtype=torch.int32, device=dev)
    gated = torch.full((1,), -1, dtype=torch.int32, device=dev)
    ws = g.workspace(g.accept_commit_workspace_bytes(n_layers), dev)
    g.accept_commit_gated(tree, torch.from_numpy(am.astype(np.int32)).to(dev),
                          torch.from_numpy(gap).to(dev), thr, layers, n_acc, acc, nr, gated, ws)
    a, path, toks, new_root, want_gated = walk_gated(ref, am, gap, L, thr)
    assert int(n_acc.item()) == a and acc.cpu().numpy()[:a].tolist() == toks
    assert int(nr.item()) == new_root and int(gated.item()) == int(want_gated)
    if near_tie_depth is not None and thr > 1e-4 and near_tie_depth < len(chain):
        assert want_gated and a == near_tie_depth
    assert int(t_len.item()) == T + a + 1
    for l in range(n_layers):
        kk, vv = ks[l].copy(), vs[l].copy()
        o_commit(kk, vv, T, path)
        assert np.array_equal(layers[l].k.view(torch.int16).cpu().numpy().view(np.uint16), kk)
        assert np.array_equal(layers[l].v.view(torch.int16).cpu().numpy().view(np.uint16), vv)


def test_gated_batched_matches_oracle(dev, clean_status):
    import tree_verified_block_gb300 as g
    from oracle.walk import walk_gated
    L, n_layers, Hkv, D, B = 15, 2, 2, 128, 3
    cases = [_gated_case(20 + r, [None, 1, 0][r]) for r in range(B)]
    Ts = [700, 64, 3000]
    t_lens = torch.tensor(Ts, dtype=torch.int32, device=dev)
    gen = W.rng(13)
    trees, layers, host = [], [], []
    for r, (ref, am, gap, chain) in enumerate(cases):
        t_cap = Ts[r] + len(ref["token"]) + 3
        ks = [W.normal_bf16(gen, (Hkv, t_cap, D)) for _ in range(n_layers)]
        vs = [W.normal_bf16(gen, (Hkv, t_cap, D)) for _ in range(n_layers)]
        host.append((ks, vs))
        trees.append(upload_tree(ref, L, dev))
        layers.append([g.KVLayer(bf16_tensor(k, dev), bf16_tensor(v, dev), t_lens[r:r + 1])
                       for k, v in zip(ks, vs)])
    amt = torch.from_numpy(np.stack([c[1] for c in cases]).astype(np.int32)).to(dev)
    gapt = torch.from_numpy(np.stack([c[2] for c in cases])).to(dev)
    n_acc = torch.full((B,), -1, dtype=torch.int32, device=dev)
    acc = torch.full((B, L), -1, dtype=torch.int32, device=dev)
    nr = torch.full((B,), -1, dtype=torch.int32, device=dev)
    gated = torch.full((B,), -1, dtype=torch.int32, device=dev)
    ws = g.workspace(g.accept_commit_batched_workspace_bytes(B, n_layers), dev)
    g.accept_commit_gated_batched(trees, amt, gapt, 1e-3, layers, n_acc, acc, nr, gated, ws)
    n_acc, acc, nr, gated, newT = (t.cpu().numpy() for t in (n_acc, acc, nr, gated, t_lens))
    for r, (ref, am, gap, chain) in enumerate(cases):
        a, path, toks, new_root, want_gated = walk_gated(ref, am, gap, L, 1e-3)
        assert n_acc[r] == a and acc[r][:a].tolist() == toks and nr[r] == new_root
        assert gated[r] == int(want_gated) and newT[r] == Ts[r] + a + 1
        for l in range(n_layers):
            kk, vv = host[r][0][l].copy(), host[r][1][l].copy()
            o_commit(kk, vv, Ts[r], path)
            assert np.array_equal(layers[r][l].k.view(torch.int16).cpu().numpy().view(np.uint16), kk)
    assert [bool(x) for x in gated] == [False, True, True]
