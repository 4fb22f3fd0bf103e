"""glance_kv_write_rows: the tree rows' K/V land at slots T..T+rows-1 of every
layer's cache, bit for bit, and nothing else moves; a prefix that leaves no
room sets device status 2 and writes nothing."""
import numpy as np
import pytest
import torch

import workloads as W
from _util import bf16_tensor

pytestmark = pytest.mark.gpu


def _caches(n_layers, Hkv, t_cap, D, dev, gen):
    ks = [W.normal_bf16(gen, (Hkv, t_cap, D)) for _ in range(n_layers)]
    vs = [W.normal_bf16(gen, (Hkv, t_cap, D)) for _ in range(n_layers)]
    return ks, vs


@pytest.mark.parametrize("n_layers,rows,T", [(36, 64, 4096), (3, 16, 0), (2, 256, 100)])
def test_rows_land_at_T(dev, clean_status, n_layers, rows, T):
    import tree_verified_block_gb300 as g
    Hkv, D = 8, 128
    t_cap = T + rows + 7
    gen = W.rng(n_layers, rows)
    ks, vs = _caches(n_layers, Hkv, t_cap, D, dev, gen)
    src = W.normal_bf16(gen, (n_layers, 2, Hkv, rows, D))
    t_len = torch.tensor([T], dtype=torch.int32, device=dev)
    layers = [g.KVLayer(bf16_tensor(k, dev), bf16_tensor(v, dev), t_len) for k, v in zip(ks, vs)]
    g.kv_write_rows(bf16_tensor(src, dev), layers, rows)
    torch.cuda.synchronize()
    for l in range(n_layers):
        wk, wv = ks[l].copy(), vs[l].copy()
        wk[:, T:T + rows] = src[l, 0]
        wv[:, T:T + rows] = src[l, 1]
        gk = layers[l].k.view(torch.int16).cpu().numpy().view(np.uint16)
        gv = layers[l].v.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(gk, wk) and np.array_equal(gv, wv), l
    assert int(t_len.item()) == T


def test_no_room_sets_status_2_and_writes_nothing(dev):
    import tree_verified_block_gb300 as g
    g.reset_device_status()
    Hkv, D, rows, t_cap = 2, 128, 16, 40
    gen = W.rng(5)
    ks, vs = _caches(2, Hkv, t_cap, D, dev, gen)
    t_len = torch.tensor([t_cap - rows + 1], dtype=torch.int32, device=dev)
    layers = [g.KVLayer(bf16_tensor(k, dev), bf16_tensor(v, dev), t_len) for k, v in zip(ks, vs)]
    g.kv_write_rows(bf16_tensor(W.normal_bf16(gen, (2, 2, Hkv, rows, D)), dev), layers, rows)
    code, _ = g.device_status()
    g.reset_device_status()
    assert code == 2
    for l in range(2):
        assert np.array_equal(layers[l].k.view(torch.int16).cpu().numpy().view(np.uint16), ks[l])
