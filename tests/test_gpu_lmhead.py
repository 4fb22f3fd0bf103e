"""LM head + argmax + top-2 gap on the GPU vs the oracle (fp64 on the same
bf16 inputs): argmax bit-exact where the oracle gap exceeds 1e-3, gap and max
logit within 2e-2 (bf16) / 1e-5 (fp32)."""
import numpy as np
import pytest
import torch

import workloads as W
from _util import bf16_tensor
from oracle.bf16 import bf16_bits_to_f64
from oracle.lmhead import lmhead_argmax as o_lmhead

pytestmark = pytest.mark.gpu


def run_bf16(hb, Wb, dev):
    import tree_verified_block_gb300 as g
    M, d = hb.shape
    V = Wb.shape[1]
    am = torch.full((M,), -1, dtype=torch.int32, device=dev)
    gap = torch.empty(M, dtype=torch.float32, device=dev)
    mx = torch.empty(M, dtype=torch.float32, device=dev)
    ws = g.workspace(g.lmhead_argmax_workspace_bytes(M, d, V, torch.bfloat16), dev)
    g.lmhead_argmax(bf16_tensor(hb, dev), bf16_tensor(Wb, dev), am, gap, mx, ws)
    return am.cpu().numpy(), gap.cpu().numpy(), mx.cpu().numpy()


def compare(got, ref, tol):
    am, gap, mx = got
    ra, rg, rm = ref
    sure = rg > 1e-3
    assert np.array_equal(am[sure], ra[sure])
    assert np.all(np.abs(mx - rm) <= tol)
    assert np.all(np.abs(gap - rg) <= tol)


@pytest.mark.parametrize("M,d,V", [(1, 64, 8), (16, 128, 1000), (64, 256, 5000),
                                   (128, 512, 4104), (200, 256, 3000), (64, 192, 136), (384, 256, 4104), (129, 64, 520),
                                   (512, 128, 2048)])
def test_bf16_shapes(dev, clean_status, M, d, V):
    gen = W.rng(M, d, V)
    hb = W.normal_bf16(gen, (M, d))
    Wb = W.normal_bf16(gen, (d, V), std=0.02)
    got = run_bf16(hb, Wb, dev)
    ref = o_lmhead(bf16_bits_to_f64(hb), bf16_bits_to_f64(Wb))
    compare(got, ref, 2e-2)


def test_bf16_qwen_lm_head_planted(dev, clean_status):
    # [64, 4096] x [4096, 151936] with planted greedy tokens on half the rows
    M, d, V = 64, 4096, 151936
    gen = W.rng(31)
    Wf = W.bf16_bits_to_f32(W.normal_bf16(gen, (d, V), std=0.02))
    h = gen.standard_normal((M, d), dtype=np.float32)
    rows = np.arange(0, M, 2)
    toks = gen.integers(0, V, size=rows.size)
    h = W.plant_greedy_path(h, Wf, rows, toks)
    hb = W.to_bf16_bits(h)
    Wb = W.to_bf16_bits(Wf)
    got = run_bf16(hb, Wb, dev)
    ref = o_lmhead(bf16_bits_to_f64(hb), bf16_bits_to_f64(Wb))
    compare(got, ref, 2e-2)
    assert np.array_equal(got[0][rows], toks)


def test_bf16_exact_ties_lowest_id(dev, clean_status):
    M, d, V = 4, 64, 4096
    gen = W.rng(5)
    Wb = W.normal_bf16(gen, (d, V), std=0.02)
    for dst, src in ((3000, 17), (2049, 17), (4095, 100)):
        Wb[:, dst] = Wb[:, src]        # duplicate columns: exact logit ties
    hb = np.zeros((M, d), np.uint16)
    hb[:] = W.to_bf16_bits(np.ones(d, np.float32))
    h = bf16_bits_to_f64(hb)
    col17 = bf16_bits_to_f64(Wb[:, 17])
    Wbig = Wb.copy()
    # make column 17 (and its copies) the clear winner for every row
    Wbig[:, 17] = W.to_bf16_bits((col17 + 0.5).astype(np.float32))
    for dst in (3000, 2049):
        Wbig[:, dst] = Wbig[:, 17]
    am, gap, mx = run_bf16(hb, Wbig, dev)
    ref = o_lmhead(h, bf16_bits_to_f64(Wbig))
    assert np.all(am == 17) and np.all(ref[0] == 17)
    assert np.all(gap == 0.0) and np.all(ref[1] == 0.0)


@pytest.mark.parametrize("M,d,V", [(16, 128, 512), (3, 100, 777), (64, 256, 300)])
def test_fp32(dev, clean_status, M, d, V):
    import tree_verified_block_gb300 as g
    gen = np.random.default_rng(M + d + V)
    h = gen.standard_normal((M, d)).astype(np.float32)
    Wm = (gen.standard_normal((d, V)) * 0.02).astype(np.float32)
    am = torch.empty(M, dtype=torch.int32, device=dev)
    gap = torch.empty(M, dtype=torch.float32, device=dev)
    mx = torch.empty(M, dtype=torch.float32, device=dev)
    ws = g.workspace(g.lmhead_argmax_workspace_bytes(M, d, V, torch.float32), dev)
    g.lmhead_argmax(torch.from_numpy(h).to(dev), torch.from_numpy(Wm).to(dev), am, gap, mx, ws)
    ref = o_lmhead(h, Wm)
    compare((am.cpu().numpy(), gap.cpu().numpy(), mx.cpu().numpy()), ref, 1e-5)


# ------------------------------------------------------- next-token entropy
# Tolerance: |dH| <= max|dl| * E_p|l - E_p l| for a logit perturbation dl;
# bf16-input logits agree with fp64 to ~1e-3 and fp32 sums over V terms add
# ~1e-4 relative, so 1e-2 absolute bounds the difference with margin.

def run_entropy(hb, Wb, dev):
    import tree_verified_block_gb300 as g
    M, d = hb.shape
    V = Wb.shape[1]
    h, Wt = bf16_tensor(hb, dev), bf16_tensor(Wb, dev)
    out = [torch.full((M,), -1, dtype=torch.int32, device=dev)] + \
          [torch.full((M,), float("nan"), dtype=torch.float32, device=dev) for _ in range(3)]
    ws = g.workspace(g.lmhead_argmax_workspace_bytes(M, d, V, torch.bfloat16), dev)
    g.lmhead_argmax_entropy(h, Wt, out[0], out[1], out[2], out[3], ws)
    plain = [torch.empty_like(t) for t in out[:3]]
    g.lmhead_argmax(h, Wt, plain[0], plain[1], plain[2], ws)
    got = [t.cpu().numpy() for t in out]
    for a, b in zip(got[:3], plain):
        assert np.array_equal(a, b.cpu().numpy())  # same fold, same answer
    return got


@pytest.mark.parametrize("M,d,V", [(16, 128, 1000), (64, 256, 5000), (129, 64, 520),
                                   (200, 256, 3000), (512, 128, 2048)])
def test_bf16_entropy_shapes(dev, clean_status, M, d, V):
    from oracle.lmhead import next_token_entropy
    gen = W.rng(M, d, V, 5)
    hb = W.normal_bf16(gen, (M, d))
    Wb = W.normal_bf16(gen, (d, V), std=0.05)
    am, gap, mx, H = run_entropy(hb, Wb, dev)
    compare((am, gap, mx), o_lmhead(bf16_bits_to_f64(hb), bf16_bits_to_f64(Wb)), 2e-2)
    want = next_token_entropy(bf16_bits_to_f64(hb), bf16_bits_to_f64(Wb))
    assert np.abs(H - want).max() < 1e-2


def test_bf16_entropy_qwen_vocab_across_temperatures(dev, clean_status):
    # rows scaled from near-uniform to near-deterministic next-token distributions
    from oracle.lmhead import next_token_entropy
    M, d, V = 64, 4096, 151936
    gen = W.rng(41)
    Wb = W.normal_bf16(gen, (d, V), std=0.02)
    h = gen.standard_normal((M, d), dtype=np.float32)
    h *= np.geomspace(0.05, 40.0, M, dtype=np.float32)[:, None]
    hb = W.to_bf16_bits(h)
    am, gap, mx, H = run_entropy(hb, Wb, dev)
    want = next_token_entropy(bf16_bits_to_f64(hb), bf16_bits_to_f64(Wb))
    assert want.max() > 11.0 and want.min() < 0.5   # the sweep spans the range
    assert np.abs(H - want).max() < 1e-2


def test_entropy_rejects_f32(dev):
    import tree_verified_block_gb300 as g
    h = torch.zeros((4, 32), device=dev)
    Wt = torch.zeros((32, 64), device=dev)
    out = torch.zeros(4, dtype=torch.int32, device=dev)
    f = torch.zeros(4, device=dev)
    ws = g.workspace(1 << 16, dev)
    with pytest.raises(g.GlanceError):
        g.lmhead_argmax_entropy(h, Wt, out, f, f, f, ws)


def run_bf16_packed(hb, Wb, dev):
    """The same call with W packed once (glance_lmhead_pack_w) and read through
    glance_lmhead_argmax_packed."""
    import tree_verified_block_gb300 as g
    M, d = hb.shape
    V = Wb.shape[1]
    Wt = bf16_tensor(Wb, dev)
    Wp = torch.empty(g.lmhead_packed_w_bytes(d, V), dtype=torch.uint8, device=dev)
    g.lmhead_pack_w(Wt, Wp)
    am = torch.full((M,), -1, dtype=torch.int32, device=dev)
    gap = torch.empty(M, dtype=torch.float32, device=dev)
    mx = torch.empty(M, dtype=torch.float32, device=dev)
    ws = g.workspace(g.lmhead_argmax_workspace_bytes(M, d, V, torch.bfloat16), dev)
    g.lmhead_argmax_packed(bf16_tensor(hb, dev), Wp, V, am, gap, mx, ws)
    return am.cpu().numpy(), gap.cpu().numpy(), mx.cpu().numpy()


@pytest.mark.parametrize("M,d,V", [(1, 64, 8), (16, 128, 1000), (64, 256, 5000), (128, 512, 4104),
                                   (64, 4096, 151936)])
def test_bf16_packed_w_is_bit_identical(dev, clean_status, M, d, V):
    # same MMA inputs in the same order: argmax, gap and max equal the unpacked
    # call's bit for bit, and the unpacked call is held to the oracle above;
    # V not a multiple of 256 leaves a partial last tile (zero columns)
    gen = W.rng(M, d, V, 7)
    hb = W.normal_bf16(gen, (M, d))
    Wb = W.normal_bf16(gen, (d, V), std=0.02)
    got = run_bf16_packed(hb, Wb, dev)
    ref = run_bf16(hb, Wb, dev)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)
    if V <= 5000:
        compare(got, o_lmhead(bf16_bits_to_f64(hb), bf16_bits_to_f64(Wb)), 2e-2)
