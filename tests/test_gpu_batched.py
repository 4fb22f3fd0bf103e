"""Batched rounds (B independent requests, one launch per step) on the GPU vs
the oracle run on each request alone: a batch is B separate rounds
(Definition 1 defines one round per request), so every request must match
its own single-request oracle result: trees bit-exact (boundary gap > 1e-3,
else a valid top-N), attention within 2e-2 absolute, LM-head argmax
bit-exact where the gap exceeds 1e-3, walk and commit bit-exact.

Workload shape: 8 requests, prefix lengths T ~ U{512..8192}, draft
marginals at mixed entropy (0.3 / 1.5 / 4.0 nats cycled) over V = 151936,
N = 63, Qwen3-VL-8B heads (32 / 8 x 128); LM head over the 8 x 64 stacked
rows."""
import numpy as np
import pytest
import torch

import workloads as W
from _util import bf16_tensor, boundary_gap
from oracle.attention import tree_attention as o_attn
from oracle.bf16 import bf16_bits_to_f64
from oracle.lmhead import lmhead_argmax as o_lmhead
from oracle.tree import build_tree as o_build
from oracle.walk import commit as o_commit
from oracle.walk import walk as o_walk
from test_gpu_attention import random_tree, upload_tree
from test_gpu_build_tree import assert_same_tree, assert_valid_top_n
from test_gpu_commit import planted_argmax

pytestmark = pytest.mark.gpu

ENTROPY = (0.3, 1.5, 4.0)


def ragged_T(B, seed, lo=512, hi=8192):
    return [int(t) for t in W.rng(seed, 55).integers(lo, hi + 1, size=B)]


# ------------------------------------------------------------------ build

@pytest.mark.parametrize("B,V,N", [(8, 151936, 63), (3, 5000, 255), (16, 700, 31)])
def test_build_tree_batched_matches_each_request(dev, clean_status, B, V, N):
    import tree_verified_block_gb300 as g
    L = 15
    xs = [W.draft_logits_entropy(L, V, ENTROPY[r % 3], seed=9000 + r) for r in range(B)]
    Ts = ragged_T(B, B)
    roots = [11 * r + 1 for r in range(B)]
    x = torch.from_numpy(np.stack(xs).astype(np.float32)).to(dev)
    trees = [g.Tree(N, L, dev) for _ in range(B)]
    ws = g.workspace(g.build_tree_batched_workspace_bytes(B, L, V, N), dev)
    t_len = torch.tensor(Ts, dtype=torch.int32, device=dev)
    rt = torch.tensor(roots, dtype=torch.int32, device=dev)
    for _ in range(2):  # the workspace's tickets are reusable
        g.build_tree_batched(x, N, rt, t_len, trees, ws)
        for r in range(B):
            got = trees[r].to_host()
            xv = xs[r].astype(np.float64)
            ref = o_build(xv, N, roots[r], Ts[r])
            if boundary_gap(xv, N) > 1e-3:
                assert_same_tree(got, ref)
            else:
                assert_valid_top_n(got, xv, N, Ts[r], roots[r])


# -------------------------------------------------------------- attention

def _attention_batch(B, Ts, N, Hq, Hkv, dev, seed, pad=7):
    import tree_verified_block_gb300 as g
    D, L, rows = 128, 15, N + 1
    refs, kbs, vbs, layers, trees = [], [], [], [], []
    t_lens = torch.tensor(Ts, dtype=torch.int32, device=dev)
    for r in range(B):
        t_cap = Ts[r] + rows + pad + 64 * r
        ref = random_tree(N, L, Ts[r], seed + r)
        gen = W.rng(seed, r, 3)
        kb = W.normal_bf16(gen, (Hkv, t_cap, D))
        vb = W.normal_bf16(gen, (Hkv, t_cap, D))
        refs.append(ref)
        kbs.append(kb)
        vbs.append(vb)
        layers.append(g.KVLayer(bf16_tensor(kb, dev), bf16_tensor(vb, dev), t_lens[r:r + 1]))
        trees.append(upload_tree(ref, L, dev))
    qb = W.normal_bf16(W.rng(seed, 99), (B, rows, Hq, D))
    q = bf16_tensor(qb, dev)
    out = torch.full_like(q, float("nan"))
    ws = g.workspace(g.tree_attention_batched_workspace_bytes(rows, Hq, layers), dev)
    g.tree_attention_batched(q, layers, trees, D ** -0.5, out, ws)
    return refs, kbs, vbs, qb, out.float().cpu().numpy().astype(np.float64), ws


def _check_groups(refs, kbs, vbs, qb, got, Ts, Hq, Hkv, groups):
    D = 128
    G = Hq // Hkv
    for r, gs in groups.items():
        for gk in gs:
            qs = bf16_bits_to_f64(qb[r][:, gk * G:(gk + 1) * G])
            ks = bf16_bits_to_f64(kbs[r][gk:gk + 1])
            vs = bf16_bits_to_f64(vbs[r][gk:gk + 1])
            want = o_attn(qs, ks, vs, Ts[r], refs[r]["anc"], D ** -0.5)
            part = got[r][:, gk * G:(gk + 1) * G]
            err = np.abs(part - want).max()
            assert err <= 2e-2, (r, gk, err)


def test_attention_batched_ragged_qwen(dev, clean_status):
    B, N, Hq, Hkv = 8, 63, 32, 8
    Ts = ragged_T(B, 5)
    refs, kbs, vbs, qb, got, _ = _attention_batch(B, Ts, N, Hq, Hkv, dev, seed=700)
    assert np.isfinite(got).all()
    # two kv-head groups per request (every group of the first request)
    groups = {r: [r % Hkv, (r + 3) % Hkv] for r in range(B)}
    groups[0] = list(range(Hkv))
    _check_groups(refs, kbs, vbs, qb, got, Ts, Hq, Hkv, groups)


@pytest.mark.parametrize("Ts,N,Hq,Hkv", [([0, 300, 1], 31, 8, 2), ([900, 129, 2048, 64], 255, 4, 1),
                                         ([5, 6], 63, 16, 2)])
def test_attention_batched_edges(dev, clean_status, Ts, N, Hq, Hkv):
    B = len(Ts)
    refs, kbs, vbs, qb, got, ws = _attention_batch(B, Ts, N, Hq, Hkv, dev, seed=800 + N)
    _check_groups(refs, kbs, vbs, qb, got, Ts, Hq, Hkv, {r: list(range(Hkv)) for r in range(B)})
    # counters left at zero: the workspace's first 256 bytes hold them
    assert int(ws[:256].sum().item()) == 0


def test_attention_batched_one_request_equals_single_call(dev, clean_status):
    # B = 1 through the batched entry point takes the single-request plan
    import tree_verified_block_gb300 as g
    Ts, N, Hq, Hkv = [3000], 63, 32, 8
    refs, kbs, vbs, qb, got, _ = _attention_batch(1, Ts, N, Hq, Hkv, dev, seed=901)
    t_len = torch.tensor(Ts, dtype=torch.int32, device=dev)
    layer = g.KVLayer(bf16_tensor(kbs[0], dev), bf16_tensor(vbs[0], dev), t_len)
    tree = upload_tree(refs[0], 15, dev)
    q = bf16_tensor(qb[0], dev)
    out = torch.empty_like(q)
    ws = g.workspace(g.tree_attention_workspace_bytes(N + 1, Hq, layer), dev)
    g.tree_attention(q, layer, tree, 128 ** -0.5, out, ws)
    assert np.array_equal(out.float().cpu().numpy(), got[0].astype(np.float32))


# ---------------------------------------------------------------- LM head

def test_lmhead_stacked_rows_m512_planted(dev, clean_status):
    # the 8 requests' 64 rows stacked: [512, 4096] x [4096, 151936], one launch
    import tree_verified_block_gb300 as g
    M, d, V = 512, 4096, 151936
    gen = W.rng(77)
    Wf = W.bf16_bits_to_f32(W.normal_bf16(gen, (d, V), std=0.02))
    h = gen.standard_normal((M, d), dtype=np.float32)
    rows = np.arange(1, M, 3)
    toks = gen.integers(0, V, size=rows.size)
    h = W.plant_greedy_path(h, Wf, rows, toks)
    hb, Wb = W.to_bf16_bits(h), W.to_bf16_bits(Wf)
    am = torch.full((M,), -1, dtype=torch.int32, device=dev)
    gap = torch.empty(M, dtype=torch.float32, device=dev)
    mx = torch.empty(M, dtype=torch.float32, device=dev)
    ws = g.workspace(g.lmhead_argmax_workspace_bytes(M, d, V, torch.bfloat16), dev)
    g.lmhead_argmax(bf16_tensor(hb, dev), bf16_tensor(Wb, dev), am, gap, mx, ws)
    am, gap, mx = am.cpu().numpy(), gap.cpu().numpy(), mx.cpu().numpy()
    assert np.array_equal(am[rows], toks)
    # rows are independent: the oracle on sampled rows from every 128-row block
    sample = np.array([0, 1, 127, 128, 200, 255, 256, 383, 384, 450, 510, 511])
    ra, rg, rm = o_lmhead(bf16_bits_to_f64(hb[sample]), bf16_bits_to_f64(Wb))
    sure = rg > 1e-3
    assert np.array_equal(am[sample][sure], ra[sure])
    assert np.all(np.abs(mx[sample] - rm) <= 2e-2)
    assert np.all(np.abs(gap[sample] - rg) <= 2e-2)


# ----------------------------------------------------------------- commit

def test_commit_batched_ragged(dev, clean_status):
    import tree_verified_block_gb300 as g
    B, N, L, n_layers, Hkv, D = 8, 63, 15, 3, 8, 128
    rows = N + 1
    Ts = ragged_T(B, 21)
    depths = [0, 1, 3, 7, 15, 2, 5, 11]
    gen = W.rng(4242)
    refs, ams, trees, host_k, host_v, layers = [], [], [], [], [], []
    t_lens = torch.tensor(Ts, dtype=torch.int32, device=dev)
    for r in range(B):
        t_cap = Ts[r] + rows + 16 * r + 3
        ref = random_tree(N, L, Ts[r], 300 + r)
        am, _ = planted_argmax(ref, depths[r], 40, gen)
        refs.append(ref)
        ams.append(am)
        trees.append(upload_tree(ref, L, dev))
        ks = [W.normal_bf16(gen, (Hkv, t_cap, D)) for _ in range(n_layers)]
        vs = [W.normal_bf16(gen, (Hkv, t_cap, D)) for _ in range(n_layers)]
        host_k.append(ks)
        host_v.append(vs)
        layers.append([g.KVLayer(bf16_tensor(k, dev), bf16_tensor(v, dev), t_lens[r:r + 1])
                       for k, v in zip(ks, vs)])
    amt = torch.from_numpy(np.stack(ams).astype(np.int32)).to(dev)
    n_acc = torch.full((B,), -1, dtype=torch.int32, device=dev)
    acc = torch.full((B, L), -1, dtype=torch.int32, device=dev)
    nr = torch.full((B,), -1, dtype=torch.int32, device=dev)
    ws = g.workspace(g.accept_commit_batched_workspace_bytes(B, n_layers), dev)
    g.accept_commit_batched(trees, amt, layers, n_acc, acc, nr, ws)
    n_acc, acc, nr, newT = n_acc.cpu().numpy(), acc.cpu().numpy(), nr.cpu().numpy(), t_lens.cpu().numpy()
    for r in range(B):
        a, path, toks, new_root = o_walk(refs[r], ams[r], L)
        assert n_acc[r] == a and acc[r][:a].tolist() == toks and nr[r] == new_root
        for l in range(n_layers):
            want_T = o_commit(host_k[r][l], host_v[r][l], Ts[r], path)
            gk = layers[r][l].k.view(torch.int16).cpu().numpy().view(np.uint16)
            gv = layers[r][l].v.view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(gk, host_k[r][l]) and np.array_equal(gv, host_v[r][l])
        assert newT[r] == want_T
    assert int(ws[:256].sum().item()) == 0


def test_batched_argument_errors(dev):
    import tree_verified_block_gb300 as g
    N, L, V = 63, 15, 1000
    trees = [g.Tree(N, L, dev) for _ in range(17)]
    x = torch.zeros((17, L, V), dtype=torch.float32, device=dev)
    rt = torch.zeros(17, dtype=torch.int32, device=dev)
    ws = g.workspace(1 << 20, dev)
    with pytest.raises(g.GlanceError):  # B > 16
        g.build_tree_batched(x, N, rt, rt, trees, ws)
    bad = [g.Tree(N, L, dev), g.Tree(31, L, dev)]
    with pytest.raises(g.GlanceError):  # trees of different N
        g.build_tree_batched(x[:2], N, rt[:2], rt[:2], bad, ws)
