"""Pins for the oracle's marginals, candidate lists and bf16 helpers (CPU)."""
import numpy as np
import pytest

from oracle.bf16 import bf16_bits_to_f64, f32_to_bf16_bits
from oracle.marginals import candidate_lists, log_marginals, logsumexp_rows


def test_log_marginals_normalise():
    g = np.random.default_rng(1)
    x = g.standard_normal((5, 1000)) * 3
    lq = log_marginals(x)
    assert np.allclose(np.exp(lq).sum(axis=1), 1.0, atol=1e-12, rtol=0)


def test_log_marginals_constant_rows_closed_form():
    # softmax of a constant row is uniform: log q = -ln V
    x = np.full((3, 777), 2.5)
    assert np.allclose(log_marginals(x), -np.log(777), atol=1e-13, rtol=0)


def test_log_marginals_of_log_probs_closed_form():
    # logits that are log-probabilities are their own log-softmax
    q = np.array([[0.1, 0.2, 0.3, 0.4], [0.25, 0.25, 0.25, 0.25]])
    assert np.allclose(log_marginals(np.log(q)), np.log(q), atol=1e-14, rtol=0)


def test_logsumexp_large_shift():
    x = np.array([[1000.0, 1000.0], [-1000.0, -1001.0]])
    assert np.allclose(logsumexp_rows(x), [1000 + np.log(2), -1000 + np.log1p(np.exp(-1))])


def test_log_marginals_rejects_non_finite():
    with pytest.raises(ValueError):
        log_marginals(np.array([[0.0, np.nan]]))


@pytest.mark.parametrize("K", [1, 7, 64])
def test_candidate_lists_match_library_sort(K):
    g = np.random.default_rng(2)
    x = np.round(g.standard_normal((4, 300)) * 4) / 4  # many exact ties
    tok, logq, rank_of = candidate_lists(x, K)
    lq = log_marginals(x)
    for j in range(4):
        # stable argsort of -x keeps equal logits in id order
        ref = np.argsort(-x[j], kind="stable")
        assert np.array_equal(tok[j], ref[:K])
        assert np.array_equal(logq[j], lq[j, ref[:K]])
        assert np.array_equal(rank_of[j, ref], np.arange(300))


def test_candidate_ties_lowest_id_first():
    x = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]])
    tok, _, _ = candidate_lists(x, 4)
    assert tok[0].tolist() == [1, 2, 4, 3]


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(3)
    x = np.concatenate([g.standard_normal(10000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 65504.0,
                                  3.3895314e38, 1e-40, -1e-40, np.inf, -np.inf], np.float32)])
    ours = f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # widening is exact
    assert np.array_equal(bf16_bits_to_f64(ours).astype(np.float32),
                          torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_bf16_ties_to_even():
    # 1 + 2^-8 is halfway between bf16 1.0 and 1 + 2^-7: rounds to even (1.0)
    assert f32_to_bf16_bits(np.float32(1 + 2 ** -8)).item() == 0x3F80
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: rounds to even (1 + 2^-6)
    assert f32_to_bf16_bits(np.float32(1 + 3 * 2 ** -8)).item() == 0x3F82
