"""The LM-head entry point that allocates nothing.

Some callers cannot allocate device memory or pass a workspace on this path:
for example code running while a stream is captured in a mode that forbids
cudaMalloc, or an engine that has reserved all device memory for its own pool.
For them the library exports glance_lmhead_argmax_noalloc, whose scratch is a
device array inside the library. This test calls it through the C ABI twice in
a row, on different inputs, and checks each result against
glance_lmhead_argmax (the workspace entry point) within the LM-head tolerance
of the other tests, and its argmax against the CPU oracle. The file name makes
pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from _util import bf16_tensor
from oracle.bf16 import bf16_bits_to_f64
from oracle.lmhead import lmhead_argmax as o_lmhead

pytestmark = pytest.mark.gpu


def _with_workspace(g, h, Wt, dev):
    M, d = h.shape
    V = Wt.shape[1]
    out = (torch.empty(M, dtype=torch.int32, device=dev), torch.empty(M, device=dev),
           torch.empty(M, device=dev))
    ws = g.workspace(g.lmhead_argmax_workspace_bytes(M, d, V, torch.bfloat16), dev)
    g.lmhead_argmax(h, Wt, out[0], out[1], out[2], ws)
    return out


def _no_alloc(lib, h, Wt, dev, am, gap, mx):
    M, d = h.shape
    V = Wt.shape[1]
    st = lib.glance_lmhead_argmax_noalloc(
        ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(Wt.data_ptr()), 1, M, d, V,
        ctypes.c_void_p(am.data_ptr()), ctypes.c_void_p(gap.data_ptr()),
        ctypes.c_void_p(mx.data_ptr()) if mx is not None else None,
        ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    assert st == 0, lib.glance_last_error()


def test_no_alloc_lmhead_matches_workspace_entry_point(dev):
    import tree_verified_block_gb300 as g
    lib = g.lib()
    g.reset_device_status()
    # call 1: one 128-row block over the full vocabulary; call 2: 200 rows (two
    # blocks) on other inputs, reusing the scratch that call 1 left behind
    for seed, (M, d, V) in ((1, (64, 512, 151936)), (2, (200, 256, 20000))):
        gen = W.rng(seed, 99)
        hb = W.normal_bf16(gen, (M, d))
        Wb = W.normal_bf16(gen, (d, V), std=0.02)
        h, Wt = bf16_tensor(hb, dev), bf16_tensor(Wb, dev)
        ref = _with_workspace(g, h, Wt, dev)
        # outputs allocated before the call: the call itself allocates nothing
        am = torch.full((M,), -1, dtype=torch.int32, device=dev)
        gap = torch.full((M,), -1.0, device=dev)
        mx = torch.full((M,), -1.0, device=dev)
        am2 = torch.full((M,), -1, dtype=torch.int32, device=dev)
        gap2 = torch.full((M,), -1.0, device=dev)
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated(dev)
        _no_alloc(lib, h, Wt, dev, am, gap, mx)
        _no_alloc(lib, h, Wt, dev, am2, gap2, None)   # maxlogit is optional
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated(dev) == before
        ra, rg, rm = (t.cpu().numpy() for t in ref)
        ga, gg, gm = (t.cpu().numpy() for t in (am, gap, mx))
        sure = rg > 1e-3
        assert np.array_equal(ga[sure], ra[sure])
        assert np.abs(gm - rm).max() <= 2e-2
        assert np.abs(gg - rg).max() <= 2e-2
        assert np.array_equal(am2.cpu().numpy(), ga) and np.array_equal(gap2.cpu().numpy(), gg)
        # the oracle (fp64 on the same bf16 inputs) agrees where its gap is > 1e-3
        oa, og, om = o_lmhead(bf16_bits_to_f64(hb), bf16_bits_to_f64(Wb))
        sure = og > 1e-3
        assert np.array_equal(ga[sure], oa[sure])
        assert np.abs(gm - om).max() <= 2e-2
    code, text = g.device_status()
    assert code == 0, text


def test_no_alloc_rejects_what_it_cannot_hold(dev):
    import tree_verified_block_gb300 as g
    lib = g.lib()
    one = ctypes.c_void_p(256)
    assert lib.glance_lmhead_argmax_noalloc(one, one, 0, 16, 64, 64, one, one, None, None) == 2
    assert lib.glance_lmhead_argmax_noalloc(one, one, 1, 513, 64, 64, one, one, None, None) == 1
