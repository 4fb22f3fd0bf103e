"""The verify forward with the dense layers (the bench's forward36 round, cut
to 3 layers): it runs through the library's calls in one CUDA graph without
a device status, its rows stay finite, and a replay from the same state
gives bit-identical rows, argmax and commit."""
import os
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_forward_round_graph_replay(dev, clean_status):
    sys.path.insert(0, ROOT)
    import bench
    cfg = dict(bench.FORWARD36, n_layers=3)
    fw = bench.ForwardWorkload(cfg, dev, seed=7100)
    k0 = [k.clone() for k in fw.k]
    fw.step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fw.step()
    outs = []
    for _ in range(2):
        for k, k_init in zip(fw.k, k0):
            k.copy_(k_init)
        graph.replay()
        torch.cuda.synchronize()
        outs.append((fw.xa.clone(), fw.argmax.clone(), fw.n_acc.clone(), fw.t_len.clone()))
    xa, am, na, tl = outs[0]
    assert torch.isfinite(xa.float()).all()
    assert 0 <= int(na.item()) <= cfg["L"] and int(tl.item()) == cfg["T"] + int(na.item()) + 1
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    assert np.all((am.cpu().numpy() >= 0) & (am.cpu().numpy() < cfg["V"]))
