"""Sampling-mode verification: each visited row's token is a draw from the
target's own distribution (oracle; test infrastructure only).

"Vision Is Not Overhead ..." (arXiv 2609.00355), Section 5.4 and its
limitations paragraph: under sampling the committed token is drawn from the
target's own verified row, so the output distribution is the target's, and
the walk of Definition 1 runs unchanged on the drawn tokens.

A draw at temperature T from softmax(l / T) is taken as the Gumbel-max
argmax_v (l_v / T + g_v), g_v = -ln(-ln u_v) with u_v uniform on (0, 1). The
uniforms come from the counter-based generator Philox4x32-10 (Salmon, Moraes,
Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011): for
the row that predicts the token at absolute sequence position `pos` of stream
`seq`, column v uses counter (v // 4, pos, seq, 0), key (seed mod 2^32,
seed div 2^32), output word v mod 4, and u = (floor(word / 2^9) + 1/2) / 2^23
(the top 23 bits, centred: exact in float32, never 0 or 1).
Keying the noise by the predicted token's position (not by the round) makes
speculative sampling reproduce autoregressive sampling with the same seed
token for token, by the argument of Theorem 1 applied to the perturbed
logits.
"""
import numpy as np

# Philox4x32 constants from the SC 2011 paper: round multipliers and the Weyl
# key increments (the 32-bit golden ratio and sqrt(3) - 1).
_M0, _M1 = 0xD2511F53, 0xCD9E8D57
_W0, _W1 = 0x9E3779B9, 0xBB67AE85
_MASK = (1 << 32) - 1


def philox4x32_10(ctr, key):
    """ctr: uint array (..., 4), key: (k0, k1). Returns uint64 array (..., 4)
    of the ten-round Philox4x32 output words."""
    x = [np.asarray(ctr[..., i], dtype=np.uint64) for i in range(4)]
    k0, k1 = np.uint64(int(key[0]) & _MASK), np.uint64(int(key[1]) & _MASK)
    m0, m1 = np.uint64(_M0), np.uint64(_M1)
    mask, sh = np.uint64(_MASK), np.uint64(32)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + np.uint64(_W0)) & mask
            k1 = (k1 + np.uint64(_W1)) & mask
        p0 = x[0] * m0           # 64-bit product of 32-bit values: no overflow
        p1 = x[2] * m1
        hi0, lo0 = p0 >> sh, p0 & mask
        hi1, lo1 = p1 >> sh, p1 & mask
        x = [hi1 ^ x[1] ^ k0, lo1, hi0 ^ x[3] ^ k1, lo0]
    return np.stack(x, axis=-1)


def uniforms(words):
    """(0, 1) uniforms from 32-bit words: the top 23 bits, centred."""
    w = np.asarray(words, dtype=np.uint64) >> np.uint64(9)
    return (w.astype(np.float64) + 0.5) / float(1 << 23)


def gumbel_noise(seed, seq, pos, V):
    """g_v = -ln(-ln u_v) for columns 0..V-1 of the row predicting position pos."""
    groups = (V + 3) // 4
    ctr = np.zeros((groups, 4), dtype=np.uint64)
    ctr[:, 0] = np.arange(groups, dtype=np.uint64)
    ctr[:, 1] = np.uint64(int(pos) & _MASK)
    ctr[:, 2] = np.uint64(int(seq) & _MASK)
    words = philox4x32_10(ctr, (seed & _MASK, (seed >> 32) & _MASK)).reshape(-1)[:V]
    return -np.log(-np.log(uniforms(words)))


def lmhead_sample(h, W, inv_temp, seed, pos, seq=None, chunk=8192):
    """Per row i: token = argmax_v (l_iv * inv_temp + g_iv) (lowest id on ties)
    and gap = best - second best of those perturbed values, in float64.
    pos[i]: absolute position of the token row i predicts; seq[i]: its stream."""
    h = np.asarray(h, dtype=np.float64)
    M = h.shape[0]
    V = W.shape[1]
    seq = np.zeros(M, dtype=np.int64) if seq is None else np.asarray(seq)
    noise = np.stack([gumbel_noise(seed, seq[i], pos[i], V) for i in range(M)])
    best = np.full(M, -np.inf)
    second = np.full(M, -np.inf)
    arg = np.zeros(M, dtype=np.int64)
    for c0 in range(0, V, chunk):
        z = (h @ np.asarray(W[:, c0:c0 + chunk], dtype=np.float64)) * inv_temp + noise[:, c0:c0 + chunk]
        for i in range(M):
            row = z[i]
            j = int(np.argmax(row))
            m = row[j]
            rest = np.delete(row, j)
            m2 = rest.max() if rest.size else -np.inf
            if m > best[i]:
                second[i] = max(best[i], m2)
                best[i], arg[i] = m, c0 + j
            else:
                second[i] = max(second[i], m)
    return arg, best - second
