"""Pins for the dense-layer oracle (CPU): RMSNorm, rotate-half RoPE, SwiGLU
and the whole layer against independent forms (torch ops, closed forms,
rotation invariants, the toy target's layer)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle.dense import dense_layer, qkv, rms_scale, rmsnorm, rope, round_bf16, swiglu
from oracle.toy import ToyTarget


def test_rmsnorm_matches_torch_and_has_unit_rms():
    g = np.random.default_rng(0)
    x = g.standard_normal((5, 96)) * 3
    w = g.uniform(0.5, 1.5, size=96)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(w), eps=1e-6).numpy()
    assert np.allclose(rmsnorm(x, w, 1e-6), ref, atol=1e-12)
    assert np.allclose(np.sqrt((rmsnorm(x, None, 0.0) ** 2).mean(axis=1)), 1.0)
    assert np.allclose(rms_scale(np.full((2, 8), 2.0), 0.0), 0.5)


def test_rope_preserves_norms_and_depends_on_relative_position():
    g = np.random.default_rng(1)
    D = 64
    q = g.standard_normal((1, 1, D))
    k = g.standard_normal((1, 1, D))
    theta = 1e6
    for p in (0, 3, 1000):
        assert np.allclose(np.linalg.norm(rope(q, [p], theta)), np.linalg.norm(q))
    dots = [float(rope(q, [m], theta)[0, 0] @ rope(k, [m - 7], theta)[0, 0]) for m in (7, 50, 12345)]
    assert np.allclose(dots, dots[0], rtol=1e-9)
    assert np.allclose(rope(q, [0], theta), q)


def test_rope_pairs_dimension_j_with_j_plus_half():
    D = 8
    x = np.zeros((1, 1, D))
    x[0, 0, 1] = 1.0
    ang = 5 * 10000.0 ** (-2 / D)  # pair j = 1
    out = rope(x, [5], 10000.0)[0, 0]
    assert np.isclose(out[1], np.cos(ang)) and np.isclose(out[1 + D // 2], np.sin(ang))
    assert np.count_nonzero(np.abs(out) > 1e-15) == 2


def test_swiglu_closed_form_and_gamma_folds_into_the_weights():
    g = np.random.default_rng(2)
    x = g.standard_normal((3, 16))
    Wg, Wu = g.standard_normal((16, 24)), g.standard_normal((16, 24))
    gam = g.uniform(0.5, 2.0, size=16)
    hn = x / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-6) * gam
    a, b = hn @ Wg, hn @ Wu
    assert np.allclose(swiglu(x, gam, Wg, Wu, 1e-6), a * b / (1 + np.exp(-a)))
    # the norm weight can be folded into the projection's rows (the kernels' form)
    r = rms_scale(x, 1e-6)[:, None]
    assert np.allclose(swiglu(x, gam, Wg, Wu, 1e-6),
                       swiglu(x, None, gam[:, None] * Wg, gam[:, None] * Wu, 1e-6))
    assert np.allclose(r * (x @ (gam[:, None] * Wg)), a)


def test_layer_equals_the_toy_targets_layer():
    # the toy decoder (oracle.toy) is the same layer with unit norm weights,
    # no q/k norm, separate q/k/v weights
    cfg = W.TOY
    w = W.toy_weights(0)
    tgt = ToyTarget(w, cfg)
    lw0 = w["layers"][0]
    P = 10
    tokens = np.asarray(w["prompt"][:P])
    x = tgt.emb[tokens]
    cache = tgt.new_cache(P + 4)
    # toy forward through layer 0 only
    tgt1 = ToyTarget(dict(w, layers=[lw0]), cfg)
    want = tgt1.forward(tokens, np.arange(P), np.arange(P), [np.arange(i + 1) for i in range(P)],
                        tgt1.new_cache(P + 4))
    lw = dict(W_qkv=np.concatenate([lw0["Wq"], lw0["Wk"], lw0["Wv"]], axis=1), W_o=lw0["Wo"],
              W_gate=lw0["Wg"], W_up=lw0["Wu"], W_down=lw0["Wd"])
    anc = np.zeros((P, 1), np.uint64)
    for i in range(P):
        for k in range(i + 1):
            anc[i, 0] |= np.uint64(1) << np.uint64(k)
    K = np.zeros((cfg["Hkv"], P + 4, cfg["D"]))
    V = np.zeros_like(K)
    out = dense_layer(x, lw, np.arange(P), 0, K, V, anc, cfg["Hq"], cfg["Hkv"], cfg["D"],
                      cfg["theta"], cfg["eps"])
    assert np.allclose(tgt1._rmsnorm(out), want, atol=1e-10)


def test_qk_norm_normalises_each_head():
    g = np.random.default_rng(3)
    x = g.standard_normal((4, 32))
    Wqkv = g.standard_normal((32, (2 + 2) * 8))
    q, k, v = qkv(x, None, Wqkv, 2, 1, 8, [0, 0, 0, 0], 1e4, 1e-6, np.ones(8), np.ones(8))
    assert np.allclose(np.sqrt((q ** 2).mean(axis=-1)), 1.0, atol=1e-5)
    assert np.allclose(np.sqrt((k ** 2).mean(axis=-1)), 1.0, atol=1e-5)


def test_round_bf16_is_torchs_bfloat16_conversion():
    """The store rounding of the layer's bf16 path is round-to-nearest-even
    to bfloat16, as torch converts float32 (an independent implementation)."""
    g = np.random.default_rng(5)
    x = np.concatenate([g.standard_normal(4000) * 10 ** g.uniform(-6, 6, 4000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, 3.0e38]])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(round_bf16(x), want)


def test_layer_with_bf16_stores_keeps_only_the_store_rounding():
    """store=round_bf16 changes the layer only through the five stores: an
    identity store gives the float64 layer bit for bit, and the rounded layer
    stays within the rounding's propagated size of it (a store that skipped
    the activation or the residual would move the tails far more)."""
    g = np.random.default_rng(6)
    R, d, Hq, Hkv, D, I, T = 8, 64, 4, 2, 16, 96, 5
    x = g.standard_normal((R, d))
    lw = dict(W_qkv=g.standard_normal((d, (Hq + 2 * Hkv) * D)) * 0.1, W_o=g.standard_normal((Hq * D, d)) * 0.1,
              W_gate=g.standard_normal((d, I)) * 0.1, W_up=g.standard_normal((d, I)) * 0.1,
              W_down=g.standard_normal((I, d)) * 0.1)
    Kc = g.standard_normal((Hkv, T + R, D))
    Vc = g.standard_normal((Hkv, T + R, D))
    anc = np.zeros((R, 1), dtype=np.uint64)
    for i in range(R):  # a chain: row i sees rows 0..i
        anc[i, 0] = np.uint64((1 << (i + 1)) - 1)
    pos = T + np.arange(R)
    base = dense_layer(x, lw, pos, T, Kc.copy(), Vc.copy(), anc, Hq, Hkv, D, 1e4, 1e-6)
    same = dense_layer(x, lw, pos, T, Kc.copy(), Vc.copy(), anc, Hq, Hkv, D, 1e4, 1e-6, store=lambda a: a)
    assert np.array_equal(base, same)
    rounded = dense_layer(x, lw, pos, T, Kc.copy(), Vc.copy(), anc, Hq, Hkv, D, 1e4, 1e-6, store=round_bf16)
    rel = np.abs(rounded - base) / np.maximum(1.0, np.abs(base))
    assert 0 < rel.max() < 3e-2
