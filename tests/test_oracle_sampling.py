"""Pins for the sampling-mode oracle (CPU): the Philox4x32-10 stream is
uniform, distinct per counter and sensitive to every counter bit; the
Gumbel-max draw follows softmax(l / T); T -> 0 is greedy; and speculative
sampling with position-keyed noise reproduces sampled autoregression token
for token on the toy target (Theorem 1's argument on perturbed logits)."""
import numpy as np
import pytest
from scipy import stats

import workloads as W
from oracle.sampling import gumbel_noise, lmhead_sample, philox4x32_10, uniforms
from oracle.toy import ToyTarget, glance_decode, greedy_ar, sample_pick


def _words(n, key=(7, 11)):
    ctr = np.zeros((n, 4), dtype=np.uint64)
    ctr[:, 0] = np.arange(n, dtype=np.uint64)
    ctr[:, 1] = 3
    return philox4x32_10(ctr, key).reshape(-1)


def test_philox_bytes_and_bits_are_uniform():
    w = _words(1 << 14)
    for b in range(4):
        byte = ((w >> np.uint64(8 * b)) & np.uint64(255)).astype(np.int64)
        counts = np.bincount(byte, minlength=256)
        assert stats.chisquare(counts).pvalue > 1e-4
    bits = np.array([((w >> np.uint64(i)) & np.uint64(1)).mean() for i in range(32)])
    assert np.all(np.abs(bits - 0.5) < 0.01)


def test_philox_counters_give_distinct_blocks_and_avalanche():
    ctr = np.zeros((20000, 4), dtype=np.uint64)
    ctr[:, 0] = np.arange(20000)
    out = philox4x32_10(ctr, (1, 2))
    blocks = {tuple(int(v) for v in r) for r in out}
    assert len(blocks) == 20000
    g = np.random.default_rng(0)
    flips = []
    for _ in range(300):
        c = g.integers(0, 1 << 32, size=4, dtype=np.uint64)
        bit = int(g.integers(0, 128))
        c2 = c.copy()
        c2[bit // 32] ^= np.uint64(1 << (bit % 32))
        a, b = philox4x32_10(c[None], (5, 6))[0], philox4x32_10(c2[None], (5, 6))[0]
        flips.append(sum(bin(int(x) ^ int(y)).count("1") for x, y in zip(a, b)))
    assert abs(np.mean(flips) - 64) < 2.0
    # the key matters too
    assert not np.array_equal(philox4x32_10(ctr[:10], (1, 2)), philox4x32_10(ctr[:10], (1, 3)))


def test_uniform_range_and_gumbel_moments():
    u = uniforms(np.array([0, 511, (1 << 32) - 1], dtype=np.uint64))
    assert u[0] > 0 and u[-1] < 1 and u[0] == u[1]
    g = np.concatenate([gumbel_noise(99, 0, p, 4096) for p in range(40)])
    assert abs(g.mean() - np.euler_gamma) < 0.02
    assert abs(g.var() - np.pi ** 2 / 6) < 0.05


@pytest.mark.parametrize("inv_temp", [0.5, 1.0, 2.0])
def test_draws_follow_softmax(inv_temp):
    logits = np.array([0.3, -1.0, 2.0, 0.0, 1.1, -0.4, 0.7])
    V = logits.size
    n = 30000
    h = np.ones((n, 1))
    Wm = logits[None, :]
    tok, _ = lmhead_sample(h, Wm, inv_temp, seed=2024, pos=np.arange(n), seq=np.zeros(n, int))
    counts = np.bincount(tok, minlength=V)
    p = np.exp(logits * inv_temp)
    p /= p.sum()
    assert stats.chisquare(counts, n * p).pvalue > 1e-4


def test_low_temperature_is_greedy():
    g = np.random.default_rng(3)
    h = g.standard_normal((20, 8))
    Wm = g.standard_normal((8, 300))
    lg = h @ Wm
    top2 = np.sort(lg, axis=1)[:, -2:]
    sure = top2[:, 1] - top2[:, 0] > 0.05
    tok, _ = lmhead_sample(h, Wm, 1e4, seed=1, pos=np.arange(20))
    assert np.array_equal(tok[sure], lg.argmax(axis=1)[sure])


def test_noise_is_keyed_by_position_and_stream_only():
    a = gumbel_noise(5, 2, 100, 64)
    assert np.array_equal(a, gumbel_noise(5, 2, 100, 64))
    assert not np.array_equal(a, gumbel_noise(5, 2, 101, 64))
    assert not np.array_equal(a, gumbel_noise(5, 3, 100, 64))
    assert not np.array_equal(a, gumbel_noise(6, 2, 100, 64))


def test_speculative_sampling_reproduces_sampled_autoregression():
    cfg = W.TOY
    weights = W.toy_weights(0)
    target = ToyTarget(weights, cfg)
    pick = sample_pick(target, 1.0, seed=77)
    n = 40
    Y, _ = greedy_ar(target, weights["prompt"], n + cfg["L"], pick=pick)
    out, acc, _ = glance_decode(target, weights["prompt"], n, cfg["N"], cfg["L"],
                                lambda r: W.toy_draft_logits(Y, r, cfg["L"], cfg["V"]), pick=pick)
    assert out == Y[:n]
    assert max(acc) >= 2
    # a sampled stream differs from the greedy one
    G, _ = greedy_ar(target, weights["prompt"], n)
    assert G != Y[:n]


def test_round_keyed_noise_would_break_the_equality():
    # plant a mistake: key the noise by the row's index within the forward
    # instead of the predicted token's absolute position
    cfg = W.TOY
    weights = W.toy_weights(0)
    target = ToyTarget(weights, cfg)
    good = sample_pick(target, 1.0, seed=77)

    def bad(h, pos):
        return lmhead_sample(h, target.Wlm, 1.0, 77, np.arange(len(pos)))
    n = 30
    Y, _ = greedy_ar(target, weights["prompt"], n + cfg["L"], pick=good)
    out, _, _ = glance_decode(target, weights["prompt"], n, cfg["N"], cfg["L"],
                              lambda r: W.toy_draft_logits(Y, r, cfg["L"], cfg["V"]), pick=bad)
    assert out != Y[:n]
