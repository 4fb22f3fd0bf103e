"""Stream-ordered status read (glance_get_status / glance_clear_status): the
words reach a device and a pinned host buffer from inside a captured CUDA
graph, without a device synchronisation in the graph, and are cleared in
stream order."""
import numpy as np
import pytest
import torch

from test_gpu_attention import random_tree, upload_tree

pytestmark = pytest.mark.gpu


def capacity_call(dev):
    """A tree attention call whose prefix leaves no room for its tree rows
    (T + rows > t_cap): the kernel sets status 2 and writes nothing."""
    import tree_verified_block_gb300 as g
    rows, Hq, Hkv, D = 16, 4, 1, 128
    K = torch.zeros((Hkv, 40, D), dtype=torch.bfloat16, device=dev)
    t_len = torch.tensor([30], dtype=torch.int32, device=dev)
    layer = g.KVLayer(K, K.clone(), t_len)
    tree = upload_tree(random_tree(15, 7, 30, 1), 7, dev)
    q = torch.zeros((rows, Hq, D), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    ws = g.workspace(g.tree_attention_workspace_bytes(rows, Hq, layer), dev)
    return lambda: g.tree_attention(q, layer, tree, 0.1, out, ws)


def test_status_words_reach_host_and_device_from_a_graph(dev):
    import tree_verified_block_gb300 as g
    g.reset_device_status()
    call = capacity_call(dev)
    on_dev = torch.full((g.STATUS_WORDS,), -1, dtype=torch.int32, device=dev)
    pinned = torch.full((g.STATUS_WORDS,), -1, dtype=torch.int32).pin_memory()
    call()
    g.clear_status()           # first calls outside the capture
    g.get_status(on_dev)
    torch.cuda.synchronize()
    assert on_dev.cpu().tolist() == [0] * g.STATUS_WORDS
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.clear_status()
        call()
        g.get_status(on_dev)
        g.get_status(pinned)
    graph.replay()
    torch.cuda.current_stream().synchronize()
    # word 0 = first non-zero; word 2 = the attention kernels' word
    assert on_dev.cpu().tolist() == [2, 0, 2, 0, 0, 0]
    assert pinned.tolist() == [2, 0, 2, 0, 0, 0]
    # the synchronous read agrees; then a stream-ordered clear empties every word
    code, _ = g.device_status()
    assert code == 2
    g.clear_status()
    g.get_status(pinned)
    torch.cuda.current_stream().synchronize()
    assert pinned.tolist() == [0] * g.STATUS_WORDS
    code, _ = g.device_status()
    assert code == 0


def test_get_status_refuses_pageable_host_memory(dev):
    import tree_verified_block_gb300 as g
    with pytest.raises(ValueError):
        g.get_status(torch.zeros(g.STATUS_WORDS, dtype=torch.int32))
