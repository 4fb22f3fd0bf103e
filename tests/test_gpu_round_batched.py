"""One ragged8 batched round (8 requests, T ~ U{512..8192}, mixed-entropy
drafts, N = 63; 3 layers here, 36 in the bench) in the launch sequence
bench.py times, replayed from a CUDA graph and checked per request against
the oracle: trees bit-exact, attention of sampled (layer, kv head) pairs
within 2e-2, LM-head argmax / gap / max of sampled rows (every planted path
row among them), the walk on the library's argmax, commit and T bit-exact."""
import os
import sys

import numpy as np
import pytest
import torch

from _util import boundary_gap
from oracle.attention import tree_attention as o_attn
from oracle.bf16 import bf16_bits_to_f64
from oracle.lmhead import lmhead_argmax as o_lmhead
from oracle.tree import build_tree as o_build
from oracle.walk import commit as o_commit
from oracle.walk import walk as o_walk
from test_gpu_build_tree import assert_same_tree, assert_valid_top_n

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_ragged8_round_graph_replay(dev, clean_status):
    sys.path.insert(0, ROOT)
    import bench
    bw = bench.BatchedWorkload(bench.RAGGED8, dev, seed=5000, host=True, n_layers=3)
    c = bw.cfg
    B, R, N, L, n_layers = bw.B, bw.R, c["N"], c["L"], c["n_layers"]

    def restore():
        for l in range(n_layers):
            for r in range(B):
                bw.k[l][r].copy_(torch.from_numpy(bw.k_bits[l][r].view(np.int16)).view(torch.bfloat16))
                bw.v[l][r].copy_(torch.from_numpy(bw.v_bits[l][r].view(np.int16)).view(torch.bfloat16))

    bw.step()
    torch.cuda.synchronize()
    restore()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        bw.step()
    restore()
    graph.replay()
    torch.cuda.synchronize()

    refs = []
    roots = bw.root.cpu().numpy()
    for r in range(B):
        x = bw.x[r].astype(np.float64)
        ref = o_build(x, N, int(roots[r]), bw.T[r])
        got = bw.trees[r].to_host()
        if boundary_gap(x, N) > 1e-3:
            assert_same_tree(got, ref)
        else:
            assert_valid_top_n(got, x, N, bw.T[r], int(roots[r]))
            ref = got  # the library's tree is one valid top-N set: check the rest on it
        refs.append(ref)

    G = c["Hq"] // c["Hkv"]
    for l in (0, n_layers - 1):
        out = bw.out[l].float().cpu().numpy()
        for r in range(B):
            gk = (r + l) % c["Hkv"]
            want = o_attn(bf16_bits_to_f64(bw.q_bits[l][r][:, gk * G:(gk + 1) * G]),
                          bf16_bits_to_f64(bw.k_bits[l][r][gk:gk + 1]),
                          bf16_bits_to_f64(bw.v_bits[l][r][gk:gk + 1]), bw.T[r], refs[r]["anc"],
                          c["D"] ** -0.5)
            err = np.abs(out[r][:, gk * G:(gk + 1) * G] - want).max()
            assert err < 2e-2, (l, r, err)

    am = bw.argmax.cpu().numpy()
    gap = bw.gap.cpu().numpy()
    mx = bw.maxlogit.cpu().numpy()
    planted = sorted({r * R + u for r in range(B) for u in bw.path_rows[r]})
    sample = np.array(sorted(set(planted) | {0, 63, 64, 200, 300, 511}))
    ra, rg, rm = o_lmhead(bf16_bits_to_f64(bw.h_bits[sample]), bf16_bits_to_f64(bw.W_bits))
    sure = rg > 1e-3
    assert np.array_equal(am[sample][sure], ra[sure])
    assert np.abs(mx[sample] - rm).max() < 2e-2 and np.abs(gap[sample] - rg).max() < 2e-2
    for r in range(B):
        for u, t in zip(bw.path_rows[r], bw.path_tokens[r]):
            assert am[r * R + u] == t

    n_acc = bw.n_acc.cpu().numpy()
    acc = bw.acc_tok.cpu().numpy()
    nr = bw.new_root.cpu().numpy()
    t_now = bw.t_len.cpu().numpy()
    for r in range(B):
        a, path, toks, new_root = o_walk(refs[r], am[r * R:(r + 1) * R], L)
        assert a == len(bw.path_rows[r]) - 1
        assert n_acc[r] == a and acc[r][:a].tolist() == toks and nr[r] == new_root
        assert t_now[r] == bw.T[r] + a + 1
        for l in (0, n_layers - 1):
            kk, vv = bw.k_bits[l][r].copy(), bw.v_bits[l][r].copy()
            o_commit(kk, vv, bw.T[r], path)
            assert np.array_equal(bw.k[l][r].view(torch.int16).cpu().numpy().view(np.uint16), kk)
            assert np.array_equal(bw.v[l][r].view(torch.int16).cpu().numpy().view(np.uint16), vv)
