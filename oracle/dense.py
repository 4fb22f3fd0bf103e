"""The target's dense verify layers around tree attention (oracle; test
infrastructure only), for a Qwen3-shaped decoder layer.

"Vision Is Not Overhead ..." (arXiv 2609.00355): the verify pass runs the
frozen target once over the packed tree rows (Definition 1; Section 4.2),
and its forward at the verify width dominates a round's cost (Table 11, the
round-cost regression of Appendix E). The pages do not describe the layer
itself. Reading taken here: a pre-norm decoder layer,

  x  -> RMSNorm(g1) -> [q | k | v] = . W_qkv -> per-head RMSNorm of q and k
     (when q_norm / k_norm weights are given) -> rotate-half RoPE at the
     rows' position ids (theta) -> K, V into the cache at the rows' slots
     -> ancestor-masked attention -> + x W_o ... residual
  x' -> RMSNorm(g2) -> SiLU(. W_gate) * (. W_up) -> . W_down -> + x' residual

RMSNorm(x) = x / sqrt(mean(x^2) + eps) * g. Everything in float64 here.

The layer can also round the five values that a bf16 implementation stores
between its steps (q, the K/V rows, the attention output, the residual
output x', the SwiGLU activation) to bf16, nearest-even: `store=round_bf16`.
That is the same function with those stores made explicit (reading R27 of
the design notes: each call normalises exactly the bf16 rows the previous
call stored), so a bf16 implementation can be held to the per-step
tolerance over a whole layer.
"""
import numpy as np

from .attention import tree_attention
from .bf16 import bf16_bits_to_f64, f32_to_bf16_bits


def round_bf16(x):
    """x rounded to the nearest bf16 value (ties to even), via float32."""
    x = np.asarray(x, dtype=np.float64)
    return bf16_bits_to_f64(f32_to_bf16_bits(x.astype(np.float32))).reshape(x.shape)


def rms_scale(x, eps):
    """1 / sqrt(mean(x^2) + eps) per row."""
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / np.sqrt((x * x).mean(axis=-1) + eps)


def rmsnorm(x, g, eps):
    x = np.asarray(x, dtype=np.float64)
    out = x * rms_scale(x, eps)[..., None]
    return out if g is None else out * np.asarray(g, dtype=np.float64)


def rope(x, pos, theta):
    """Rotate-half rotary embedding of x (R, H, D) at positions pos (R,)."""
    D = x.shape[-1]
    inv = theta ** (-np.arange(0, D, 2, dtype=np.float64) / D)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    cos = np.concatenate([np.cos(ang), np.cos(ang)], axis=-1)[:, None, :]
    sin = np.concatenate([np.sin(ang), np.sin(ang)], axis=-1)[:, None, :]
    half = D // 2
    rot = np.concatenate([-x[..., half:], x[..., :half]], axis=-1)
    return x * cos + rot * sin


def qkv(x, g1, W_qkv, Hq, Hkv, D, pos, theta, eps, q_norm=None, k_norm=None):
    """q (R, Hq, D), k and v (R, Hkv, D) of the rows x (R, d)."""
    R = x.shape[0]
    y = rmsnorm(x, g1, eps) @ np.asarray(W_qkv, dtype=np.float64)
    q = y[:, :Hq * D].reshape(R, Hq, D)
    k = y[:, Hq * D:(Hq + Hkv) * D].reshape(R, Hkv, D)
    v = y[:, (Hq + Hkv) * D:].reshape(R, Hkv, D)
    if q_norm is not None:
        q = rmsnorm(q, q_norm, eps)
    if k_norm is not None:
        k = rmsnorm(k, k_norm, eps)
    return rope(q, pos, theta), rope(k, pos, theta), v


def swiglu(x, g2, W_gate, W_up, eps):
    hn = rmsnorm(x, g2, eps)
    gate = hn @ np.asarray(W_gate, dtype=np.float64)
    up = hn @ np.asarray(W_up, dtype=np.float64)
    return gate / (1.0 + np.exp(-gate)) * up


def residual(res, a, W):
    return np.asarray(res, dtype=np.float64) + np.asarray(a, dtype=np.float64) @ np.asarray(W, dtype=np.float64)


def dense_layer(x, lw, pos, T, K_cache, V_cache, anc, Hq, Hkv, D, theta, eps, store=None):
    """One decoder layer over the packed rows x (R, d); the rows' K/V go to
    cache slots T..T+R-1 (row i at T + i) of K_cache/V_cache (Hkv, t_cap, D),
    which are updated in place. lw: g1, W_qkv, q_norm, k_norm, W_o, g2, W_gate,
    W_up, W_down. store: applied to each value the layer keeps between its
    steps (q, K/V rows, attention output, x', activation); None keeps float64.
    Returns the layer's output rows (before any store)."""
    keep = (lambda a: a) if store is None else store
    R = x.shape[0]
    q, k, v = qkv(x, lw.get("g1"), lw["W_qkv"], Hq, Hkv, D, pos, theta, eps,
                  lw.get("q_norm"), lw.get("k_norm"))
    q, k, v = keep(q), keep(k), keep(v)
    K_cache[:, T:T + R] = k.transpose(1, 0, 2)
    V_cache[:, T:T + R] = v.transpose(1, 0, 2)
    att = keep(tree_attention(q, K_cache[:, :T + R], V_cache[:, :T + R], T, anc, 1.0 / np.sqrt(D)))
    x1 = keep(residual(x, att.reshape(R, Hq * D), lw["W_o"]))
    act = keep(swiglu(x1, lw.get("g2"), lw["W_gate"], lw["W_up"], eps))
    return residual(x1, act, lw["W_down"])
