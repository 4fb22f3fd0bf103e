"""GLANCE verify-round hot path for GB300 (sm_103a).

The compute lives in ``libglance.so`` (CUDA kernels behind a C ABI declared in
``include/glance.h``); this package is its Python binding. Calls:

* ``build_tree``      draft logits [L, V] -> packed top-N candidate tree
* ``tree_attention``  ancestor-masked GQA attention of the packed rows
* ``lmhead_argmax``   LM head with fused per-row argmax and top-2 gap
* ``accept_commit``   acceptance walk A(S), KV commit, new root

``*_batched`` forms run B independent requests (ragged prefix lengths) in one
launch per step; the LM head takes the B requests' rows stacked.
"""
from ._binding import (STATUS_WORDS, BF16, EXPORTS, F32, LIB_PATH, GlanceError, KVLayer, Tree, accept_commit,
                       accept_commit_batched, accept_commit_batched_workspace_bytes,
                       accept_commit_gated, accept_commit_gated_batched, lmhead_argmax_entropy,
                       lmhead_sample,
                       accept_commit_workspace_bytes, build_tree, build_tree_batched, clear_status,
                       get_status, kv_write_rows,
                       build_tree_batched_workspace_bytes, build_tree_shared,
                       build_tree_shared_workspace_bytes, build_tree_workspace_bytes,
                       dense_qkv, dense_residual, dense_swiglu,
                       device_status, lib, lmhead_argmax, lmhead_argmax_noalloc, row_sumsq,
                       lmhead_argmax_packed, lmhead_pack_w, lmhead_packed_w_bytes,
                       lmhead_argmax_workspace_bytes, reset_device_status, tree_attention,
                       tree_attention_timeout_check, tree_attention_batched, tree_attention_batched_workspace_bytes,
                       tree_attention_workspace_bytes, version, workspace)

__all__ = ["STATUS_WORDS", "BF16", "EXPORTS", "F32", "LIB_PATH", "GlanceError", "KVLayer", "Tree",
           "accept_commit", "accept_commit_batched", "accept_commit_batched_workspace_bytes",
           "accept_commit_gated", "accept_commit_gated_batched", "lmhead_argmax_entropy",
           "lmhead_sample",
           "accept_commit_workspace_bytes", "build_tree", "build_tree_batched", "clear_status", "get_status", "kv_write_rows",
           "build_tree_batched_workspace_bytes", "build_tree_shared",
           "build_tree_shared_workspace_bytes", "build_tree_workspace_bytes", "dense_qkv",
           "dense_residual", "dense_swiglu", "device_status", "row_sumsq",
           "lib", "lmhead_argmax", "lmhead_argmax_noalloc", "lmhead_argmax_workspace_bytes",
           "lmhead_argmax_packed", "lmhead_pack_w", "lmhead_packed_w_bytes",
           "reset_device_status", "tree_attention", "tree_attention_timeout_check", "tree_attention_batched",
           "tree_attention_batched_workspace_bytes", "tree_attention_workspace_bytes", "version",
           "workspace"]
