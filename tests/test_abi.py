"""The C ABI library loads and exports every declared symbol; host-side
argument checks reject bad calls before any launch (CPU only, no compute)."""
import ctypes

import pytest

from _util import ensure_built, header_functions


@pytest.fixture(scope="module")
def glib():
    ensure_built()
    import tree_verified_block_gb300 as g
    return g.lib()


def test_header_declares_the_four_path_calls():
    names = header_functions()
    for n in ("glance_build_tree", "glance_tree_attention", "glance_lmhead_argmax",
              "glance_accept_commit"):
        assert n in names
    assert len(names) >= 13


def test_every_declared_symbol_is_exported(glib):
    for name in header_functions():
        assert hasattr(glib, name), name
    import tree_verified_block_gb300 as g
    assert sorted(g.EXPORTS) == header_functions()


def test_version_and_status_strings(glib):
    assert glib.glance_version() == 300
    assert glib.glance_status_string(0) == b"GLANCE_OK"
    assert glib.glance_status_string(3) == b"GLANCE_ERR_CAPACITY"


def test_build_tree_workspace_sizes(glib):
    assert glib.glance_build_tree_workspace_bytes(15, 151936, 63) > 0
    assert glib.glance_build_tree_workspace_bytes(0, 100, 5) == 0       # L out of range
    assert glib.glance_build_tree_workspace_bytes(17, 100, 5) == 0
    assert glib.glance_build_tree_workspace_bytes(15, 100, 256) == 0    # N > 255
    assert glib.glance_build_tree_workspace_bytes(1, 3, 4) == 0         # N > #strings
    assert glib.glance_build_tree_workspace_bytes(2, 3, 12) > 0         # 3 + 9 strings
    assert glib.glance_build_tree_workspace_bytes(15, 1 << 19, 5) == 0  # V too large


def test_build_tree_rejects_bad_arguments(glib):
    import tree_verified_block_gb300._binding as b
    tree = b.TreeC(15, 7, 1, 1, 1, 1, 1, 1, 1)
    one = ctypes.c_void_p(16)
    # null logits
    assert glib.glance_build_tree(None, 0, 7, 512, 15, one, one, ctypes.byref(tree), one, 1 << 20, None) == 1
    # tree struct sized for another N
    assert glib.glance_build_tree(one, 0, 7, 512, 14, one, one, ctypes.byref(tree), one, 1 << 20, None) == 1
    assert b"sized for n=15" in glib.glance_last_error()
    # bad dtype
    assert glib.glance_build_tree(one, 7, 7, 512, 15, one, one, ctypes.byref(tree), one, 1 << 20, None) == 1
    # workspace too small
    assert glib.glance_build_tree(one, 0, 7, 512, 15, one, one, ctypes.byref(tree), ctypes.c_void_p(256), 8, None) == 3


def test_attention_rejects_bad_arguments(glib):
    import tree_verified_block_gb300._binding as b
    tree = b.TreeC(15, 7, 1, 1, 1, 1, 1, 1, 1)
    kv = b.KVC(16, 16, 1, 8, 128, 4096, 4096 * 128, 128, 16)
    one = ctypes.c_void_p(16)
    # q heads not a multiple of kv heads
    assert glib.glance_tree_attention(one, 12, ctypes.byref(kv), ctypes.byref(tree), 0.1, one, one, 1 << 20, None) == 1
    # mask_words inconsistent with N
    bad = b.TreeC(100, 7, 1, 1, 1, 1, 1, 1, 1)
    assert glib.glance_tree_attention(one, 32, ctypes.byref(kv), ctypes.byref(bad), 0.1, one, one, 1 << 20, None) == 1
    # bf16 needs head_dim 128
    kv64 = b.KVC(16, 16, 1, 8, 64, 4096, 4096 * 64, 64, 16)
    assert glib.glance_tree_attention(one, 32, ctypes.byref(kv64), ctypes.byref(tree), 0.1, one, one, 1 << 20, None) == 2
    # null output
    assert glib.glance_tree_attention(one, 32, ctypes.byref(kv), ctypes.byref(tree), 0.1, None, one, 1 << 20, None) == 1


def test_lmhead_rejects_bad_arguments(glib):
    one = ctypes.c_void_p(256)
    assert glib.glance_lmhead_argmax(one, one, 1, 0, 4096, 1000, one, one, None, one, 1 << 20, None) == 1
    assert glib.glance_lmhead_argmax(one, one, 1, 600, 4096, 1000, one, one, None, one, 1 << 20, None) == 1
    # bf16 needs d % 64 == 0 and V % 8 == 0
    assert glib.glance_lmhead_argmax(one, one, 1, 64, 100, 1000, one, one, None, one, 1 << 20, None) == 2
    assert glib.glance_lmhead_argmax(one, one, 1, 64, 128, 1001, one, one, None, one, 1 << 20, None) == 2
    assert glib.glance_lmhead_argmax_workspace_bytes(0, 10, 10, 1) == 0


def test_packed_lmhead_sizes_and_bad_arguments(glib):
    # ceil(V / 256) x (d / 64) blocks of 32 KB; 0 for shapes the kernel has no layout for
    assert glib.glance_lmhead_packed_w_bytes(4096, 151936) == 594 * 64 * 32768
    assert glib.glance_lmhead_packed_w_bytes(64, 8) == 32768
    assert glib.glance_lmhead_packed_w_bytes(4096, 151937) == 0
    assert glib.glance_lmhead_packed_w_bytes(100, 1024) == 0
    assert glib.glance_lmhead_packed_w_bytes(0, 1024) == 0
    one = ctypes.c_void_p(256)
    need = 4 * 2 * 32768  # d = 128, V = 1000: 4 tiles x 2 row slices
    assert glib.glance_lmhead_pack_w(None, 128, 1000, one, need, None) == 1
    assert glib.glance_lmhead_pack_w(one, 100, 1000, one, need, None) == 2
    assert glib.glance_lmhead_pack_w(one, 128, 1000, one, need - 16, None) == 3
    assert glib.glance_lmhead_pack_w(ctypes.c_void_p(264), 128, 1000, one, need, None) == 1
    # M <= 128 only; the same workspace as glance_lmhead_argmax
    assert glib.glance_lmhead_argmax_packed(one, one, 129, 128, 1000, one, one, None, one, 1 << 20, None) == 1
    assert glib.glance_lmhead_argmax_packed(one, one, 0, 128, 1000, one, one, None, one, 1 << 20, None) == 1
    assert glib.glance_lmhead_argmax_packed(one, None, 64, 128, 1000, one, one, None, one, 1 << 20, None) == 1
    assert glib.glance_lmhead_argmax_packed(one, one, 64, 100, 1000, one, one, None, one, 1 << 20, None) == 2
    assert glib.glance_lmhead_argmax_packed(one, one, 64, 128, 1000, one, one, None, one, 16, None) == 3


def test_commit_rejects_bad_arguments(glib):
    import tree_verified_block_gb300._binding as b
    tree = b.TreeC(15, 7, 1, 16, 16, 16, 16, 16, 16)
    kv = (b.KVC * 2)(b.KVC(256, 256, 1, 8, 128, 4096, 4096 * 128, 128, 16),
                     b.KVC(256, 256, 1, 8, 128, 2048, 2048 * 128, 128, 16))
    one = ctypes.c_void_p(256)
    # layers disagree on t_cap
    assert glib.glance_accept_commit(ctypes.byref(tree), one, kv, 2, one, one, one, one, 256, None) == 1
    assert b"share geometry" in glib.glance_last_error()
    assert glib.glance_accept_commit(ctypes.byref(tree), one, kv, 0, one, one, one, one, 256, None) == 1
    assert glib.glance_accept_commit(ctypes.byref(tree), one, kv, 1, one, one, one, one, 8, None) == 3
    assert glib.glance_accept_commit_workspace_bytes(1) == 256
    assert glib.glance_accept_commit_workspace_bytes(129) == 0


def test_binding_refuses_to_run_without_library(monkeypatch, tmp_path):
    import tree_verified_block_gb300._binding as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        b.lib()


def test_host_tensors_are_refused_before_any_call():
    """A CPU tensor would reach a kernel as an address it cannot read: the
    binding refuses it (no GPU needed to check)."""
    import torch
    import tree_verified_block_gb300 as g
    with pytest.raises(ValueError):
        g.Tree(15, 7, "cpu")
    z = torch.zeros((2, 4, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        g.KVLayer(z, z, torch.zeros(1, dtype=torch.int32))
