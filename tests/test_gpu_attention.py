"""Tree attention on the GPU vs the oracle (fp64 on the same bf16 / fp32
inputs): bf16 within 2e-2 absolute, fp32 within 1e-5 absolute."""
import numpy as np
import pytest
import torch

import workloads as W
from _util import bf16_tensor
from oracle.attention import tree_attention as o_attn
from oracle.bf16 import bf16_bits_to_f64
from oracle.tree import build_tree as o_build
from oracle.tree import pack_tree

pytestmark = pytest.mark.gpu


def upload_tree(ref, L, dev):
    import tree_verified_block_gb300 as g
    N = len(ref["token"]) - 1
    tree = g.Tree(N, L, dev)
    tree.token.copy_(torch.from_numpy(ref["token"].astype(np.int32)))
    tree.parent.copy_(torch.from_numpy(ref["parent"].astype(np.int32)))
    tree.depth.copy_(torch.from_numpy(ref["depth"].astype(np.int32)))
    tree.pos_id.copy_(torch.from_numpy(ref["pos_id"].astype(np.int32)))
    tree.score.copy_(torch.from_numpy(ref["score"].astype(np.float32)))
    tree.anc.copy_(torch.from_numpy(ref["anc"].view(np.int64)))
    return tree


def random_tree(N, L, T, seed):
    g = np.random.default_rng(seed)
    x = g.standard_normal((L, max(2, min(40, N + 1)))) * 1.5
    return o_build(x, N, 0, T)


def run_bf16(T, N, Hq, Hkv, dev, seed=0, t_cap=None, head_pad=0, L=15):
    import tree_verified_block_gb300 as g
    D = 128
    rows = N + 1
    t_cap = t_cap or T + rows + 5
    ref = random_tree(N, L, T, seed) if N > 0 else pack_tree([], np.zeros((1, 1), int), np.zeros((1, 1)), 0, T)
    gen = W.rng(seed, 7)
    kb = W.normal_bf16(gen, (Hkv, t_cap + head_pad, D))
    vb = W.normal_bf16(gen, (Hkv, t_cap + head_pad, D))
    qb = W.normal_bf16(gen, (rows, Hq, D))
    K = bf16_tensor(kb, dev)[:, :t_cap]
    V = bf16_tensor(vb, dev)[:, :t_cap]
    t_len = torch.tensor([T], dtype=torch.int32, device=dev)
    layer = g.KVLayer(K, V, t_len)
    tree = upload_tree(ref, L, dev)
    q = bf16_tensor(qb, dev)
    out = torch.full_like(q, float("nan"))
    ws = g.workspace(g.tree_attention_workspace_bytes(rows, Hq, layer), dev)
    scale = D ** -0.5
    g.tree_attention(q, layer, tree, scale, out, ws)
    want = o_attn(bf16_bits_to_f64(qb), bf16_bits_to_f64(kb[:, :t_cap]), bf16_bits_to_f64(vb[:, :t_cap]),
                  T, ref["anc"], scale)
    got = out.float().cpu().numpy().astype(np.float64)
    return got, want


@pytest.mark.parametrize("T,N,Hq,Hkv", [
    (100, 15, 4, 1),      # G=4, 16 rows -> one q tile
    (300, 40, 8, 8),      # G=1, padded rows
    (1000, 31, 16, 2),    # G=8, two q tiles
    (5, 0, 4, 2),         # root row only
    (1, 63, 8, 2),        # prefix of one slot
    (127, 20, 4, 4),
    (129, 20, 4, 4),
    (1024, 31, 32, 8),    # one Qwen3-VL-8B layer, N=31
    (0, 63, 32, 8),       # no prefix: tree rows only (nothing fetched before the wait)
    (128, 63, 32, 8),     # the prefix is exactly the first key tile
    (256, 255, 4, 1),     # 256 rows
])
def test_bf16_small(dev, clean_status, T, N, Hq, Hkv):
    got, want = run_bf16(T, N, Hq, Hkv, dev, seed=T + N)
    assert np.isfinite(got).all()
    err = np.abs(got - want).max()
    assert err < 2e-2, err


@pytest.mark.parametrize("T,N", [(4096, 63), (2048, 127), (2048, 255), (4097, 63)])
def test_bf16_qwen_geometry(dev, clean_status, T, N):
    got, want = run_bf16(T, N, 32, 8, dev, seed=N)
    err = np.abs(got - want).max()
    assert err < 2e-2, err


def test_bf16_strided_cache(dev, clean_status):
    # heads padded apart in memory: head_stride > t_cap * head_dim
    got, want = run_bf16(500, 31, 8, 2, dev, seed=3, head_pad=64)
    assert np.abs(got - want).max() < 2e-2


def test_bf16_chain_tree_is_causal(dev, clean_status):
    import tree_verified_block_gb300 as g
    from oracle.attention import causal_attention
    T, R, Hq, Hkv, D = 50, 16, 8, 2, 128
    nodes = [tuple([0] * d) for d in range(1, R)]
    ref = pack_tree(nodes, np.zeros((R, 1), int), np.zeros((R, 1)), 0, T)
    gen = W.rng(11)
    kb = W.normal_bf16(gen, (Hkv, T + R, D))
    vb = W.normal_bf16(gen, (Hkv, T + R, D))
    qb = W.normal_bf16(gen, (R, Hq, D))
    t_len = torch.tensor([T], dtype=torch.int32, device=dev)
    layer = g.KVLayer(bf16_tensor(kb, dev), bf16_tensor(vb, dev), t_len)
    tree = upload_tree(ref, R, dev)
    out = torch.empty((R, Hq, D), dtype=torch.bfloat16, device=dev)
    ws = g.workspace(g.tree_attention_workspace_bytes(R, Hq, layer), dev)
    g.tree_attention(bf16_tensor(qb, dev), layer, tree, D ** -0.5, out, ws)
    k_seq = bf16_bits_to_f64(kb).transpose(1, 0, 2)
    v_seq = bf16_bits_to_f64(vb).transpose(1, 0, 2)
    q_full = np.concatenate([np.zeros((T, Hq, D)), bf16_bits_to_f64(qb)])
    want = causal_attention(q_full, k_seq, v_seq, D ** -0.5)[T:]
    assert np.abs(out.float().cpu().numpy() - want).max() < 2e-2


@pytest.mark.parametrize("T,N,Hq,Hkv,D", [(70, 15, 4, 2, 32), (0, 63, 4, 2, 32), (200, 31, 8, 8, 128)])
def test_fp32(dev, clean_status, T, N, Hq, Hkv, D):
    import tree_verified_block_gb300 as g
    rows = N + 1
    ref = random_tree(N, 7, T, seed=N)
    gen = np.random.default_rng(T + N)
    kc = gen.standard_normal((Hkv, T + rows, D)).astype(np.float32)
    vc = gen.standard_normal((Hkv, T + rows, D)).astype(np.float32)
    q = gen.standard_normal((rows, Hq, D)).astype(np.float32)
    t_len = torch.tensor([T], dtype=torch.int32, device=dev)
    layer = g.KVLayer(torch.from_numpy(kc).to(dev), torch.from_numpy(vc).to(dev), t_len)
    tree = upload_tree(ref, 7, dev)
    out = torch.empty((rows, Hq, D), dtype=torch.float32, device=dev)
    ws = g.workspace(g.tree_attention_workspace_bytes(rows, Hq, layer), dev)
    g.tree_attention(torch.from_numpy(q).to(dev), layer, tree, D ** -0.5, out, ws)
    want = o_attn(q, kc, vc, T, ref["anc"], D ** -0.5)
    assert np.abs(out.cpu().numpy() - want).max() < 1e-5


def test_capacity_error_on_device(dev):
    import tree_verified_block_gb300 as g
    g.reset_device_status()
    rows, Hq, Hkv, D = 16, 4, 1, 128
    K = torch.zeros((Hkv, 40, D), dtype=torch.bfloat16, device=dev)
    t_len = torch.tensor([30], dtype=torch.int32, device=dev)   # 30 + 16 > 40
    layer = g.KVLayer(K, K.clone(), t_len)
    ref = random_tree(15, 7, 30, 1)
    tree = upload_tree(ref, 7, dev)
    q = torch.zeros((rows, Hq, D), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    ws = g.workspace(g.tree_attention_workspace_bytes(rows, Hq, layer), dev)
    g.tree_attention(q, layer, tree, 0.1, out, ws)
    code, _ = g.device_status()
    g.reset_device_status()
    assert code == 2


@pytest.mark.parametrize("T,N", [(1000, 63), (4096, 63), (130, 15)])
def test_bf16_cache_slots_past_the_tree_may_hold_nan(dev, clean_status, T, N):
    """Slots T + N + 1 .. t_cap - 1 of the cache are not part of the call
    (Definition 1: a row sees the prefix and its ancestors only). They may
    hold anything, NaN included: the output must not change."""
    import tree_verified_block_gb300 as g
    D, Hq, Hkv, L = 128, 32, 8, 15
    rows = N + 1
    t_cap = T + rows + 200
    ref = random_tree(N, L, T, 11)
    gen = W.rng(11, 7)
    kb = W.normal_bf16(gen, (Hkv, t_cap, D))
    vb = W.normal_bf16(gen, (Hkv, t_cap, D))
    qb = W.normal_bf16(gen, (rows, Hq, D))
    kb[:, T + rows:] = 0x7FC0  # bf16 quiet NaN
    vb[:, T + rows:] = 0x7FC0
    t_len = torch.tensor([T], dtype=torch.int32, device=dev)
    layer = g.KVLayer(bf16_tensor(kb, dev), bf16_tensor(vb, dev), t_len)
    tree = upload_tree(ref, L, dev)
    q = bf16_tensor(qb, dev)
    out = torch.full_like(q, float("nan"))
    ws = g.workspace(g.tree_attention_workspace_bytes(rows, Hq, layer), dev)
    g.tree_attention(q, layer, tree, D ** -0.5, out, ws)
    want = o_attn(bf16_bits_to_f64(qb), bf16_bits_to_f64(kb[:, :T + rows]), bf16_bits_to_f64(vb[:, :T + rows]),
                  T, ref["anc"], D ** -0.5)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    assert np.abs(got - want).max() < 2e-2
