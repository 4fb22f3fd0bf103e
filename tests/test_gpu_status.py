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


def test_a_pipeline_wait_that_runs_out_sets_status_4_and_returns(dev):
    """The kernel's bounded waits: with one V copy withheld per CTA and a
    1 ms limit, the MMA warp's wait runs out; the CTA reports status 4 and
    leaves (the other roles see its abort flag), the launch ends normally, the
    context stays usable and the next ordinary call is correct."""
    import time

    import tree_verified_block_gb300 as g
    from test_gpu_attention import run_bf16
    from _util import bf16_tensor
    import workloads as W
    T, N, Hq, Hkv, D = 1000, 63, 32, 8, 128
    rows = N + 1
    ref = random_tree(N, 15, T, 3)
    gen = W.rng(3, 7)
    t_cap = T + rows + 5
    K = bf16_tensor(W.normal_bf16(gen, (Hkv, t_cap, D)), dev)
    V = bf16_tensor(W.normal_bf16(gen, (Hkv, t_cap, D)), dev)
    q = bf16_tensor(W.normal_bf16(gen, (rows, Hq, D)), dev)
    t_len = torch.tensor([T], dtype=torch.int32, device=dev)
    layer = g.KVLayer(K, V, t_len)
    tree = upload_tree(ref, 15, dev)
    out = torch.empty_like(q)
    ws = g.workspace(g.tree_attention_workspace_bytes(rows, Hq, layer), dev)
    g.reset_device_status()
    status = torch.full((g.STATUS_WORDS,), -1, dtype=torch.int32, device=dev)
    t0 = time.perf_counter()
    g.tree_attention_timeout_check(q, layer, tree, D ** -0.5, out, ws, 1_000_000)
    g.get_status(status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert status.cpu().tolist() == [4, 0, 4, 0, 0, 0]
    assert elapsed < 1.5   # 1 ms waits, not the 2 s default
    g.clear_status()
    torch.cuda.synchronize()
    # the context is usable and the ordinary call is right again
    got, want = run_bf16(T, N, Hq, Hkv, dev, seed=3)
    assert np.abs(got - want).max() < 2e-2
    code, _ = g.device_status()
    assert code == 0
