"""Dense verify layers on the GPU vs the oracle (fp64 on the same bf16
inputs): RMSNorm row scales from the library's row sums of squares within
1e-5 relative (row_sumsq, and the residual projections' per-tile sums of
their own outputs); projections, SwiGLU,
q/k with RoPE and the cache rows within 2e-2 * max(1, |ref|); the whole
layer (with tree attention between) call by call on each call's own bf16
inputs, and end to end against the fp64 oracle layer within 6e-2 (the bf16
stores between the calls); cache slots outside the rows'
untouched."""
import numpy as np
import pytest
import torch

import workloads as W
from _util import bf16_tensor
from oracle.attention import tree_attention as o_attn
from oracle.bf16 import bf16_bits_to_f64
from oracle.dense import dense_layer, qkv as o_qkv, residual as o_residual, rms_scale as o_rms
from oracle.dense import round_bf16, swiglu as o_swiglu
from test_gpu_attention import random_tree, upload_tree

pytestmark = pytest.mark.gpu


def close(got, want):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - want) / np.maximum(1.0, np.abs(want))
    assert err.max() < 2e-2, err.max()


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def scale_from_sumsq(parts, d, eps):
    """1 / rms per row from [n][M] partial sums of squares."""
    return 1.0 / np.sqrt(parts.reshape(-1, parts.shape[-1]).astype(np.float64).sum(axis=0) / d + eps)


def tile_sumsq(xb, width=256):
    """[d / width][M] fp32 partial row sums of squares of bf16 bits xb [M][d] (test input)."""
    x = bf16_bits_to_f64(xb)
    M, d = x.shape
    return torch.from_numpy(np.ascontiguousarray(
        (x * x).reshape(M, d // width, width).sum(axis=2).T.astype(np.float32)))


@pytest.mark.parametrize("M,d", [(64, 4096), (7, 512), (128, 12288)])
def test_row_sumsq(dev, clean_status, M, d):
    import tree_verified_block_gb300 as g
    xb = W.normal_bf16(W.rng(M, d), (M, d))
    ss = torch.empty(M, dtype=torch.float32, device=dev)
    g.row_sumsq(bf16_tensor(xb, dev), ss)
    got = scale_from_sumsq(ss.cpu().numpy()[None], d, 1e-6)
    want = o_rms(bf16_bits_to_f64(xb), 1e-6)
    assert np.all(np.abs(got - want) <= 1e-5 * want)


@pytest.mark.parametrize("M,K,N", [(64, 4096, 4096), (17, 12288, 4096), (64, 12288, 4096), (128, 512, 768),
                                   (1, 64, 256), (8, 128, 40960)])
def test_residual_projection(dev, clean_status, M, K, N):
    # (1, 64, 256): one CTA; (8, 128, 40960): 160 tiles, more clusters than fit at once
    import tree_verified_block_gb300 as g
    gen = W.rng(M, K, N)
    xb = W.normal_bf16(gen, (M, K))
    Wb = W.normal_bf16(gen, (K, N), std=0.02)
    rb = W.normal_bf16(gen, (M, N))
    res = bf16_tensor(rb, dev)
    out = torch.full_like(res, float("nan"))
    x, Wt = bf16_tensor(xb, dev), bf16_tensor(Wb, dev)
    want = o_residual(bf16_bits_to_f64(rb), bf16_bits_to_f64(xb), bf16_bits_to_f64(Wb))
    ss = torch.full((N // 256, M), float("nan"), dtype=torch.float32, device=dev)
    g.dense_residual(x, Wt, res, out, ss)
    close(f64(out), want)
    # the per-tile sums of squares are those of the stored outputs
    ob = out.view(torch.int16).cpu().numpy().view(np.uint16)
    got_r = scale_from_sumsq(ss.cpu().numpy(), N, 1e-6)
    assert np.all(np.abs(got_r - o_rms(bf16_bits_to_f64(ob), 1e-6)) <= 1e-5 * got_r)
    assert np.allclose(ss.cpu().numpy(), tile_sumsq(ob).numpy(), rtol=1e-5, atol=0)
    g.dense_residual(x, Wt, res, res)  # in place: out aliases the residual
    close(f64(res), want)
    assert np.array_equal(res.view(torch.int16).cpu().numpy(), out.view(torch.int16).cpu().numpy())


@pytest.mark.parametrize("M,d,inter", [(64, 4096, 12288), (5, 256, 384), (128, 1024, 256)])
def test_swiglu(dev, clean_status, M, d, inter):
    import tree_verified_block_gb300 as g
    gen = W.rng(M, d, inter)
    hb = W.normal_bf16(gen, (M, d))
    Gb = W.normal_bf16(gen, (d, inter), std=0.02)
    Ub = W.normal_bf16(gen, (d, inter), std=0.02)
    h = bf16_tensor(hb, dev)
    act = torch.full((M, inter), float("nan"), dtype=torch.bfloat16, device=dev)
    # the input's sums of squares in 256-column parts, as a residual projection leaves them
    g.dense_swiglu(h, bf16_tensor(Gb, dev), bf16_tensor(Ub, dev), tile_sumsq(hb).to(dev), 1e-6, act)
    want = o_swiglu(bf16_bits_to_f64(hb), None, bf16_bits_to_f64(Gb), bf16_bits_to_f64(Ub), 1e-6)
    close(f64(act), want)


@pytest.mark.parametrize("qk_norm,norm_input", [(False, True), (True, True), (False, False)])
def test_qkv_rope_into_cache(dev, clean_status, qk_norm, norm_input):
    import tree_verified_block_gb300 as g
    M, d, Hq, Hkv, D, T = 64, 4096, 32, 8, 128, 3000
    t_cap = T + M + 16
    gen = W.rng(77, int(qk_norm), int(norm_input))
    hb = W.normal_bf16(gen, (M, d))
    Wb = W.normal_bf16(gen, (d, (Hq + 2 * Hkv) * D), std=0.02)
    qn = gen.uniform(0.5, 1.5, size=D).astype(np.float32) if qk_norm else None
    kn = gen.uniform(0.5, 1.5, size=D).astype(np.float32) if qk_norm else None
    pos = (T + gen.integers(0, 16, size=M)).astype(np.int32)
    kb = W.normal_bf16(gen, (Hkv, t_cap, D))
    vb = W.normal_bf16(gen, (Hkv, t_cap, D))
    t_len = torch.tensor([T], dtype=torch.int32, device=dev)
    kv = g.KVLayer(bf16_tensor(kb, dev), bf16_tensor(vb, dev), t_len)
    h = bf16_tensor(hb, dev)
    q = torch.full((M, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    tt = lambda a: None if a is None else torch.from_numpy(a).to(dev)
    ss = None
    if norm_input:
        ss = torch.empty(M, dtype=torch.float32, device=dev)
        g.row_sumsq(h, ss)
    g.dense_qkv(h, bf16_tensor(Wb, dev), Hq, ss, tt(qn), tt(kn), 1e-6, torch.from_numpy(pos).to(dev),
                1e6, q, kv)
    wq, wk, wv = o_qkv(bf16_bits_to_f64(hb), None, bf16_bits_to_f64(Wb), Hq, Hkv, D, pos, 1e6, 1e-6,
                       None if qn is None else qn.astype(np.float64),
                       None if kn is None else kn.astype(np.float64))
    if not norm_input:  # RoPE is linear: without the row norm every output is 1 / r times larger
        r = o_rms(bf16_bits_to_f64(hb), 1e-6)[:, None, None]
        wq, wk, wv = wq / r, wk / r, wv / r
    close(f64(q), wq)
    K = f64(kv.k)
    V = f64(kv.v)
    close(K[:, T:T + M], wk.transpose(1, 0, 2))
    close(V[:, T:T + M], wv.transpose(1, 0, 2))
    # slots outside the rows' are untouched
    keep = np.r_[0:T, T + M:t_cap]
    assert np.array_equal(kv.k.view(torch.int16).cpu().numpy().view(np.uint16)[:, keep], kb[:, keep])
    assert np.array_equal(kv.v.view(torch.int16).cpu().numpy().view(np.uint16)[:, keep], vb[:, keep])


def test_full_layer_with_tree_attention(dev, clean_status):
    import tree_verified_block_gb300 as g
    M, d, Hq, Hkv, D, I, T = 64, 4096, 32, 8, 128, 12288, 512
    t_cap = T + M + 8
    gen = W.rng(2025)
    ref = random_tree(M - 1, 15, T, 9)
    xb = W.normal_bf16(gen, (M, d))
    Wqkv = W.normal_bf16(gen, (d, (Hq + 2 * Hkv) * D), std=0.02)
    Wo = W.normal_bf16(gen, (Hq * D, d), std=0.02)
    Wg = W.normal_bf16(gen, (d, I), std=0.02)
    Wu = W.normal_bf16(gen, (d, I), std=0.02)
    Wd = W.normal_bf16(gen, (I, d), std=0.02)
    qn = gen.uniform(0.5, 1.5, size=D).astype(np.float32)
    kn = gen.uniform(0.5, 1.5, size=D).astype(np.float32)
    kb = W.normal_bf16(gen, (Hkv, t_cap, D))
    vb = W.normal_bf16(gen, (Hkv, t_cap, D))
    pos = ref["pos_id"].astype(np.int32)
    # GPU layer
    t_len = torch.tensor([T], dtype=torch.int32, device=dev)
    kv = g.KVLayer(bf16_tensor(kb, dev), bf16_tensor(vb, dev), t_len)
    tree = upload_tree(ref, 15, dev)
    x = bf16_tensor(xb, dev)
    q = torch.empty((M, Hq, D), dtype=torch.bfloat16, device=dev)
    att = torch.empty_like(q)
    x1 = torch.empty_like(x)
    act = torch.empty((M, I), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(x)
    ws_a = g.workspace(g.tree_attention_workspace_bytes(M, Hq, kv), dev)
    ss0 = torch.empty(M, dtype=torch.float32, device=dev)
    ss1 = torch.empty((d // 256, M), dtype=torch.float32, device=dev)
    ss2 = torch.empty_like(ss1)
    g.row_sumsq(x, ss0)
    g.dense_qkv(x, bf16_tensor(Wqkv, dev), Hq, ss0, torch.from_numpy(qn).to(dev), torch.from_numpy(kn).to(dev),
                1e-6, torch.from_numpy(pos).to(dev), 1e6, q, kv)
    g.tree_attention(q, kv, tree, D ** -0.5, att, ws_a)
    g.dense_residual(att.view(M, Hq * D), bf16_tensor(Wo, dev), x, x1, ss1)
    g.dense_swiglu(x1, bf16_tensor(Wg, dev), bf16_tensor(Wu, dev), ss1, 1e-6, act)
    g.dense_residual(act, bf16_tensor(Wd, dev), x1, out, ss2)  # ss2: the next layer's norm input
    # every call against the oracle's step on that call's own bf16 inputs (the
    # previous call's stored output); fp64 inside every step
    Kc, Vc = bf16_bits_to_f64(kb), bf16_bits_to_f64(vb)
    x0 = bf16_bits_to_f64(xb)
    wq, wk, wv = o_qkv(x0, None, bf16_bits_to_f64(Wqkv), Hq, Hkv, D, pos, 1e6, 1e-6,
                       qn.astype(np.float64), kn.astype(np.float64))
    close(f64(q), wq)
    K, V = f64(kv.k), f64(kv.v)
    close(K[:, T:T + M], wk.transpose(1, 0, 2))
    close(V[:, T:T + M], wv.transpose(1, 0, 2))
    close(f64(att), o_attn(f64(q), K[:, :T + M], V[:, :T + M], T, ref["anc"], D ** -0.5))
    close(f64(x1), o_residual(x0, f64(att).reshape(M, Hq * D), bf16_bits_to_f64(Wo)))
    close(f64(act), o_swiglu(f64(x1), None, bf16_bits_to_f64(Wg), bf16_bits_to_f64(Wu), 1e-6))
    close(f64(out), o_residual(f64(x1), f64(act), bf16_bits_to_f64(Wd)))
    got_r = scale_from_sumsq(ss2.cpu().numpy(), d, 1e-6)
    assert np.all(np.abs(got_r - o_rms(f64(out), 1e-6)) <= 1e-5 * got_r)
    # and the whole layer, against the oracle layer that rounds the five values
    # the calls store in bf16 (q, K/V rows, att, x1, act) at the same points.
    # Each call above is within 2e-2 of the oracle on its own inputs, but a
    # chain of bf16 stores is sensitive to where each value falls against a
    # rounding boundary: a difference far below a bf16 step flips some stored
    # values by one step, and the 12288-term down projection sums the flips.
    # The bound is taken from the oracle itself: oracle chains whose stored
    # values carry the noise the kernels' own arithmetic brings (one bf16 step,
    # 2^-9 relative, on the attention output, whose probabilities enter the PV
    # product as bf16; float32-level, 2^-20, on the other stores) spread by D
    # around the rounded chain; the GPU chain must stay within 2 D of it.
    lw = dict(W_qkv=bf16_bits_to_f64(Wqkv), W_o=bf16_bits_to_f64(Wo), W_gate=bf16_bits_to_f64(Wg),
              W_up=bf16_bits_to_f64(Wu), W_down=bf16_bits_to_f64(Wd), q_norm=qn.astype(np.float64),
              k_norm=kn.astype(np.float64))
    layer = lambda store: dense_layer(x0, lw, pos, T, bf16_bits_to_f64(kb), bf16_bits_to_f64(vb), ref["anc"],
                                      Hq, Hkv, D, 1e6, 1e-6, store=store)
    rel = lambda a, b: np.abs(a - b) / np.maximum(1.0, np.abs(b))
    want = layer(round_bf16)
    spread_max, spread_mean = 0.0, 0.0
    for seed in (0, 1):
        noise = np.random.default_rng(seed)
        n_store = [0]

        def noisy(a):  # stores in the layer's order: q, k, v, att, x1, act
            n_store[0] += 1
            level = 2.0 ** -9 if n_store[0] == 4 else 2.0 ** -20
            return round_bf16(a * (1 + level * noise.standard_normal(a.shape)))
        alt = layer(noisy)
        spread_max = max(spread_max, rel(alt, want).max())
        spread_mean = max(spread_mean, rel(alt, want).mean())
    err = rel(f64(out), want)
    assert err.max() <= 2 * spread_max and err.mean() <= 2 * spread_mean, (err.max(), err.mean(),
                                                                          spread_max, spread_mean)


def test_qkv_cache_capacity_and_arguments(dev, clean_status):
    """Rows whose K/V slots T + row would pass t_cap set device status 2 and
    leave the cache alone; misaligned or mis-shaped arguments are refused on
    the host before any launch."""
    import tree_verified_block_gb300 as g
    M, d, Hq, Hkv, D = 16, 256, 4, 2, 128
    t_cap = 40
    gen = W.rng(99)
    h = bf16_tensor(W.normal_bf16(gen, (M, d)), dev)
    Wq = bf16_tensor(W.normal_bf16(gen, (d, (Hq + 2 * Hkv) * D), std=0.02), dev)
    kb = W.normal_bf16(gen, (Hkv, t_cap, D))
    kv = g.KVLayer(bf16_tensor(kb, dev), bf16_tensor(kb, dev), torch.tensor([t_cap - M + 1], dtype=torch.int32,
                                                                             device=dev))
    q = torch.empty((M, Hq, D), dtype=torch.bfloat16, device=dev)
    pos = torch.arange(M, dtype=torch.int32, device=dev)
    g.dense_qkv(h, Wq, Hq, None, None, None, 1e-6, pos, 1e6, q, kv)
    code, _ = g.device_status()
    assert code == 2
    g.reset_device_status()
    assert np.array_equal(kv.k.view(torch.int16).cpu().numpy().view(np.uint16), kb)
    # host-side refusals: x not 16-byte aligned, N not a multiple of 256, M > 128
    x_bad = torch.empty(M * d + 1, dtype=torch.bfloat16, device=dev)[1:].view(M, d)
    res = torch.zeros((M, 256), dtype=torch.bfloat16, device=dev)
    W256 = torch.zeros((d, 256), dtype=torch.bfloat16, device=dev)
    with pytest.raises(g.GlanceError):
        g.dense_residual(x_bad, W256, res, torch.empty_like(res))
    with pytest.raises(g.GlanceError):
        g.dense_residual(h, torch.zeros((d, 320), dtype=torch.bfloat16, device=dev), torch.zeros((M, 320),
                         dtype=torch.bfloat16, device=dev), torch.zeros((M, 320), dtype=torch.bfloat16, device=dev))
    big = torch.zeros((129, d), dtype=torch.bfloat16, device=dev)
    with pytest.raises(g.GlanceError):
        g.dense_residual(big, W256, torch.zeros((129, 256), dtype=torch.bfloat16, device=dev),
                         torch.zeros((129, 256), dtype=torch.bfloat16, device=dev))
