"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This package holds input generation only: random draws (numpy PCG64), the
encoding of float32 draws as bf16 bit patterns, and the shaping of inputs
(planted peaks in draft logits, temperature calibration to a target entropy,
planted greedy paths in LM-head inputs). It holds none of the method's
arithmetic: no log-softmax, no tree search, no attention, no walk.

Workloads (Qwen3-VL-8B verify geometry: hidden 4096, 36 layers, 32 query
heads, 8 KV heads, head_dim 128, vocabulary 151936, block 16 so L = 15):

* toy      2-layer random-init fp32 decoder (hidden 128, 4/2 heads, head_dim
           32, V 512, weights N(0, 0.02), seed 0), 64-token uniform prompt,
           L = 7, N = 15.
* verify1  1 layer, T = 1024, bf16 q/K/V ~ N(0,1), N = 31, draft logits over
           V = 151936 at L = 15 offsets with a planted peak of margin U(2, 8).
* full36   36 layers, T = 4096, N = 63, LM head W ~ N(0, 0.02) [4096, 151936].
* entropy  T = 2048, 36 layers, draft marginals calibrated to 0.3 / 1.5 / 4.0
           nats, N in {31, 63, 127, 255}.
* ragged   8 requests, T ~ U{512..8192}, N = 63 each.
"""
import numpy as np

QWEN3VL8B = dict(d=4096, n_layers=36, Hq=32, Hkv=8, D=128, V=151936, L=15)
TOY = dict(d=128, n_layers=2, Hq=4, Hkv=2, D=32, V=512, L=7, inter=384,
           eps=1e-6, theta=10000.0, prompt_len=64, n_tokens=64, N=15)


def rng(*seed):
    """numpy Generator on PCG64 keyed by one or more integers."""
    return np.random.Generator(np.random.PCG64(list(seed) if len(seed) > 1 else seed[0]))


def to_bf16_bits(x):
    """float32 -> bf16 bit patterns, round to nearest even (input encoding)."""
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)
    u = u.astype(np.uint64)
    out = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return out.astype(np.uint16)


def bf16_bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(g, shape, std=1.0, chunk=1 << 24):
    """bf16 bit patterns of N(0, std^2) draws, generated in chunks of `chunk`
    elements (same values as one draw of the whole array)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        x = g.standard_normal(size=c1 - c0, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        u = x.view(np.uint32)
        out[c0:c1] = ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)
    return out.reshape(shape)


# ---------------------------------------------------------------- draft logits

def draft_logits_planted(L, V, seed, margin=(2.0, 8.0)):
    """Gaussian logits per offset with one planted peak: x_t = max(x) + U(margin)."""
    g = rng(seed)
    x = g.standard_normal(size=(L, V), dtype=np.float32)
    for j in range(L):
        t = int(g.integers(0, V))
        x[j, t] = x[j].max() + np.float32(g.uniform(*margin))
    return x


def _entropy_nats(z):
    z = z.astype(np.float64)
    z = z - z.max()
    p = np.exp(z)
    p /= p.sum()
    nz = p > 0
    return float(-(p[nz] * np.log(p[nz])).sum())


def draft_logits_entropy(L, V, H, seed, margin=(2.0, 8.0), tol=0.01):
    """Planted-peak Gaussian logits scaled by a temperature found by bisection
    so that the entropy of softmax(row) is H nats within tol (relative)."""
    base = draft_logits_planted(L, V, seed, margin)
    out = np.empty_like(base)
    for j in range(L):
        lo, hi = 1e-3, 1e3  # inverse temperature bracket
        for _ in range(200):
            mid = np.sqrt(lo * hi)
            e = _entropy_nats(base[j] * mid)
            if abs(e - H) <= tol * H:
                break
            if e > H:
                lo = mid
            else:
                hi = mid
        out[j] = (base[j] * np.float32(mid)).astype(np.float32)
    return out


def toy_draft_logits(Y, r, L, V, seed=0, plant=6.0, p_plant=0.7):
    """Toy round draft: N(0,1) logits, +plant at Y[r+j] with probability p_plant.

    Y is the target's greedy token stream after the prompt (Y[0] is the first
    emitted token); r is the stream index of this round's root.
    """
    g = rng(seed, 1, r)
    x = g.standard_normal(size=(L, V), dtype=np.float32)
    coins = g.uniform(size=L)
    for j in range(1, L + 1):
        if r + j < len(Y) and coins[j - 1] < p_plant:
            x[j - 1, int(Y[r + j])] += np.float32(plant)
    return x


# ---------------------------------------------------------------- toy target

def toy_weights(seed=0, cfg=TOY):
    """Random-init toy decoder weights, N(0, 0.02), drawn in a fixed order, and
    the uniform 64-token prompt drawn after them from the same generator."""
    g = rng(seed)
    d, V, Hq, Hkv, D, I = cfg["d"], cfg["V"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["inter"]

    def w(*shape):
        return g.normal(0.0, 0.02, size=shape)

    out = {"emb": w(V, d), "layers": []}
    for _ in range(cfg["n_layers"]):
        out["layers"].append(dict(Wq=w(d, Hq * D), Wk=w(d, Hkv * D), Wv=w(d, Hkv * D),
                                  Wo=w(Hq * D, d), Wg=w(d, I), Wu=w(d, I), Wd=w(I, d)))
    out["Wlm"] = w(d, V)
    out["prompt"] = g.integers(0, V, size=cfg["prompt_len"])
    return out


# ---------------------------------------------------------------- verify rows

def kv_cache_bf16(n_layers, Hkv, T_cap, D, T_fill, seed):
    """Per-layer K and V caches [Hkv][T_cap][D] as bf16 bits; slots >= T_fill
    that the caller does not overwrite hold N(0,1) draws as well."""
    g = rng(seed)
    ks, vs = [], []
    for _ in range(n_layers):
        ks.append(normal_bf16(g, (Hkv, T_cap, D)))
        vs.append(normal_bf16(g, (Hkv, T_cap, D)))
    return ks, vs


def q_rows_bf16(n_layers, R, Hq, D, seed):
    g = rng(seed)
    return [normal_bf16(g, (R, Hq, D)) for _ in range(n_layers)]


def plant_greedy_path(h, W, path_rows, path_tokens, wrong_row=None, wrong_token=None, s=10.0):
    """Add s * W[:, t] / ||W[:, t]||^2 to h[row] so that token t wins that row.

    h: float32 (M, d), W: float32 (d, V). Used to make the target's greedy path
    follow a chosen chain of tree rows; optionally a last row gets a token that
    is not one of its children.
    """
    h = h.copy()
    for r, t in zip(path_rows, path_tokens):
        col = W[:, t].astype(np.float64)
        h[r] += (s * col / (col @ col)).astype(np.float32)
    if wrong_row is not None:
        col = W[:, wrong_token].astype(np.float64)
        h[wrong_row] += (s * col / (col @ col)).astype(np.float32)
    return h
