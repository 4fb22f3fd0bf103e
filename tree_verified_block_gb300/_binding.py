"""ctypes binding of libglance.so: argument marshalling only.

Every step runs in the library's CUDA kernels. PyTorch provides device memory
and streams; tensors are passed as raw pointers. There is no fallback: if the
library is not built, every call raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libglance.so")

F32, BF16 = 0, 1
STATUS = {0: "GLANCE_OK", 1: "GLANCE_ERR_INVALID_ARG", 2: "GLANCE_ERR_UNSUPPORTED",
          3: "GLANCE_ERR_CAPACITY", 4: "GLANCE_ERR_CUDA", 5: "GLANCE_ERR_DEVICE"}
DEV_STATUS = {0: "ok", 1: "non-finite draft logits", 2: "tree does not fit the cache",
              3: "inconsistent tree", 4: "pipeline wait timed out",
              5: "index out of bounds (bounds-checked build)"}

EXPORTS = [
    "glance_build_tree_workspace_bytes", "glance_build_tree",
    "glance_tree_attention_workspace_bytes", "glance_tree_attention",
    "glance_tree_attention_timeout_check",
    "glance_lmhead_argmax_workspace_bytes", "glance_lmhead_argmax", "glance_lmhead_argmax_noalloc",
    "glance_lmhead_packed_w_bytes", "glance_lmhead_pack_w", "glance_lmhead_argmax_packed",
    "glance_accept_commit_workspace_bytes", "glance_accept_commit",
    "glance_build_tree_batched_workspace_bytes", "glance_build_tree_batched",
    "glance_tree_attention_batched_workspace_bytes", "glance_tree_attention_batched",
    "glance_accept_commit_batched_workspace_bytes", "glance_accept_commit_batched",
    "glance_lmhead_argmax_entropy", "glance_lmhead_sample", "glance_accept_commit_gated",
    "glance_build_tree_shared_workspace_bytes", "glance_build_tree_shared",
    "glance_row_sumsq", "glance_dense_qkv",
    "glance_dense_residual", "glance_dense_swiglu",
    "glance_accept_commit_gated_batched",
    "glance_last_error", "glance_status_string", "glance_device_status",
    "glance_reset_device_status", "glance_get_status", "glance_kv_write_rows", "glance_clear_status", "glance_version",
]


class GlanceError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class TreeC(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("L", ctypes.c_int32), ("mask_words", ctypes.c_int32),
                ("token", ctypes.c_void_p), ("parent", ctypes.c_void_p),
                ("depth", ctypes.c_void_p), ("pos_id", ctypes.c_void_p),
                ("score", ctypes.c_void_p), ("anc", ctypes.c_void_p)]


class KVC(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("t_cap", ctypes.c_int32), ("head_stride", ctypes.c_int64),
                ("row_stride", ctypes.c_int64), ("t_len", ctypes.c_void_p)]


_lib = None


def lib():
    """Load libglance.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; build it with "
                           "tree_verified_block_gb300._build.build() (nvcc, sm_103a)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    st = ctypes.c_int
    L.glance_build_tree_workspace_bytes.argtypes = [i32, i32, i32]
    L.glance_build_tree_workspace_bytes.restype = sz
    L.glance_build_tree.argtypes = [vp, i32, i32, i32, i32, vp, vp, ctypes.POINTER(TreeC), vp, sz, vp]
    L.glance_build_tree.restype = st
    L.glance_tree_attention_workspace_bytes.argtypes = [i32, i32, ctypes.POINTER(KVC)]
    L.glance_tree_attention_workspace_bytes.restype = sz
    L.glance_tree_attention.argtypes = [vp, i32, ctypes.POINTER(KVC), ctypes.POINTER(TreeC),
                                        ctypes.c_float, vp, vp, sz, vp]
    L.glance_tree_attention.restype = st
    L.glance_tree_attention_timeout_check.argtypes = [vp, i32, ctypes.POINTER(KVC), ctypes.POINTER(TreeC),
                                                      ctypes.c_float, vp, vp, sz, ctypes.c_ulonglong, vp]
    L.glance_tree_attention_timeout_check.restype = st
    L.glance_lmhead_argmax_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.glance_lmhead_argmax_workspace_bytes.restype = sz
    L.glance_lmhead_argmax.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    L.glance_lmhead_argmax.restype = st
    L.glance_lmhead_argmax_noalloc.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
    L.glance_lmhead_argmax_noalloc.restype = st
    L.glance_lmhead_packed_w_bytes.argtypes = [i32, i32]
    L.glance_lmhead_packed_w_bytes.restype = sz
    L.glance_lmhead_pack_w.argtypes = [vp, i32, i32, vp, sz, vp]
    L.glance_lmhead_pack_w.restype = st
    L.glance_lmhead_argmax_packed.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    L.glance_lmhead_argmax_packed.restype = st
    L.glance_accept_commit_workspace_bytes.argtypes = [i32]
    L.glance_accept_commit_workspace_bytes.restype = sz
    L.glance_accept_commit.argtypes = [ctypes.POINTER(TreeC), vp, ctypes.POINTER(KVC), i32, vp, vp,
                                       vp, vp, sz, vp]
    L.glance_accept_commit.restype = st
    L.glance_build_tree_batched_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.glance_build_tree_batched_workspace_bytes.restype = sz
    L.glance_build_tree_batched.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp,
                                            ctypes.POINTER(TreeC), vp, sz, vp]
    L.glance_build_tree_batched.restype = st
    L.glance_tree_attention_batched_workspace_bytes.argtypes = [i32, i32, i32, ctypes.POINTER(KVC)]
    L.glance_tree_attention_batched_workspace_bytes.restype = sz
    L.glance_tree_attention_batched.argtypes = [vp, i32, ctypes.POINTER(KVC), ctypes.POINTER(TreeC),
                                                i32, ctypes.c_float, vp, vp, sz, vp]
    L.glance_tree_attention_batched.restype = st
    L.glance_accept_commit_batched_workspace_bytes.argtypes = [i32, i32]
    L.glance_accept_commit_batched_workspace_bytes.restype = sz
    L.glance_accept_commit_batched.argtypes = [ctypes.POINTER(TreeC), i32, vp, ctypes.POINTER(KVC),
                                               i32, vp, vp, vp, vp, sz, vp]
    L.glance_accept_commit_batched.restype = st
    L.glance_lmhead_argmax_entropy.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    L.glance_lmhead_argmax_entropy.restype = st
    L.glance_build_tree_shared_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.glance_build_tree_shared_workspace_bytes.restype = sz
    L.glance_build_tree_shared.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp, vp, vp,
                                           ctypes.c_float, ctypes.c_float, ctypes.POINTER(TreeC),
                                           vp, vp, sz, vp]
    L.glance_build_tree_shared.restype = st
    L.glance_row_sumsq.argtypes = [vp, i32, i32, vp, vp]
    L.glance_row_sumsq.restype = st
    L.glance_dense_qkv.argtypes = [vp, vp, i32, i32, i32, vp, i32, vp, vp, ctypes.c_float, vp,
                                   ctypes.c_float, vp, vp, vp]
    L.glance_dense_qkv.restype = st
    L.glance_dense_residual.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp]
    L.glance_dense_residual.restype = st
    L.glance_dense_swiglu.argtypes = [vp, vp, vp, i32, i32, i32, vp, i32, ctypes.c_float, vp, vp]
    L.glance_dense_swiglu.restype = st
    L.glance_lmhead_sample.argtypes = [vp, vp, i32, i32, i32, i32, ctypes.c_float, ctypes.c_uint64,
                                       vp, vp, vp, vp, vp, sz, vp]
    L.glance_lmhead_sample.restype = st
    L.glance_accept_commit_gated.argtypes = [ctypes.POINTER(TreeC), vp, vp, ctypes.c_float,
                                             ctypes.POINTER(KVC), i32, vp, vp, vp, vp, vp, sz, vp]
    L.glance_accept_commit_gated.restype = st
    L.glance_accept_commit_gated_batched.argtypes = [ctypes.POINTER(TreeC), i32, vp, vp,
                                                     ctypes.c_float, ctypes.POINTER(KVC), i32, vp,
                                                     vp, vp, vp, vp, sz, vp]
    L.glance_accept_commit_gated_batched.restype = st
    L.glance_last_error.argtypes = []
    L.glance_last_error.restype = ctypes.c_char_p
    L.glance_status_string.argtypes = [st]
    L.glance_status_string.restype = ctypes.c_char_p
    L.glance_device_status.argtypes = [ctypes.POINTER(ctypes.c_int32)]
    L.glance_device_status.restype = st
    L.glance_reset_device_status.argtypes = []
    L.glance_reset_device_status.restype = st
    L.glance_kv_write_rows.argtypes = [vp, ctypes.POINTER(KVC), i32, i32, vp]
    L.glance_kv_write_rows.restype = st
    L.glance_get_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    L.glance_get_status.restype = st
    L.glance_clear_status.argtypes = [ctypes.c_void_p]
    L.glance_clear_status.restype = st
    L.glance_version.argtypes = []
    L.glance_version.restype = ctypes.c_int
    _lib = L
    return L


def _check(status):
    if status != 0:
        raise GlanceError(status, lib().glance_last_error().decode())


def _ptr(t):
    """Device pointer of a CUDA tensor (None for None). A host tensor would
    reach a kernel as an address it cannot read, so it is refused here."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("glance: every array argument must be a CUDA tensor (got one on %s)" % t.device)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}: float32 or bfloat16")


def workspace(nbytes, device="cuda"):
    """A zero-filled device workspace (the library leaves its counters at zero)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class Tree:
    """Device arrays of one packed tree (N + 1 rows) and the C view of them."""

    def __init__(self, N, L, device="cuda"):
        rows = N + 1
        self.N, self.L, self.rows = N, L, rows
        self.mask_words = (rows + 63) // 64
        i32 = dict(dtype=torch.int32, device=device)
        self.token = torch.zeros(rows, **i32)
        self.parent = torch.zeros(rows, **i32)
        self.depth = torch.zeros(rows, **i32)
        self.pos_id = torch.zeros(rows, **i32)
        self.score = torch.zeros(rows, dtype=torch.float32, device=device)
        self.anc = torch.zeros((rows, self.mask_words), dtype=torch.int64, device=device)
        self.c = TreeC(N, L, self.mask_words, *(_ptr(t).value for t in (self.token, self.parent, self.depth,
                                                                            self.pos_id, self.score, self.anc)))

    def to_host(self):
        return dict(token=self.token.cpu().numpy(), parent=self.parent.cpu().numpy(),
                    depth=self.depth.cpu().numpy(), pos_id=self.pos_id.cpu().numpy(),
                    score=self.score.cpu().numpy(),
                    anc=self.anc.cpu().numpy().view("uint64"))


class KVLayer:
    """One layer's cache view: k, v tensors [n_kv_heads][t_cap][head_dim]."""

    def __init__(self, k, v, t_len):
        assert k.shape == v.shape and k.dim() == 3 and k.stride() == v.stride()
        assert k.stride(2) == 1, "head_dim must be contiguous"
        self.k, self.v, self.t_len = k, v, t_len
        Hkv, t_cap, D = k.shape
        self.c = KVC(_ptr(k).value, _ptr(v).value, _dtype_code(k), Hkv, D, t_cap,
                     k.stride(0), k.stride(1), _ptr(t_len).value)


# ------------------------------------------------------------------- calls

def build_tree_workspace_bytes(L, V, N):
    return lib().glance_build_tree_workspace_bytes(L, V, N)


def build_tree(draft_logits, N, root_token, t_len, tree, ws, stream=None):
    L, V = draft_logits.shape
    assert draft_logits.is_contiguous()
    _check(lib().glance_build_tree(_ptr(draft_logits), _dtype_code(draft_logits), L, V, N,
                                   _ptr(root_token), _ptr(t_len), ctypes.byref(tree.c),
                                   _ptr(ws), ws.numel(), _stream(stream, draft_logits.device)))


def tree_attention_workspace_bytes(rows, n_q_heads, kv):
    return lib().glance_tree_attention_workspace_bytes(rows, n_q_heads, ctypes.byref(kv.c))


def tree_attention(q, kv, tree, scale, out, ws, stream=None):
    assert q.is_contiguous() and out.is_contiguous() and q.shape == out.shape
    _check(lib().glance_tree_attention(_ptr(q), q.shape[1], ctypes.byref(kv.c),
                                       ctypes.byref(tree.c), float(scale), _ptr(out), _ptr(ws),
                                       ws.numel(), _stream(stream, q.device)))


def tree_attention_timeout_check(q, kv, tree, scale, out, ws, wait_ns, stream=None):
    """The bf16 attention call with every pipeline wait limited to wait_ns and
    one key tile's V copy withheld: the kernel must set device status 4 and
    return (include/glance.h)."""
    assert q.is_contiguous() and out.is_contiguous() and q.shape == out.shape
    _check(lib().glance_tree_attention_timeout_check(_ptr(q), q.shape[1], ctypes.byref(kv.c),
                                                     ctypes.byref(tree.c), float(scale), _ptr(out),
                                                     _ptr(ws), ws.numel(), int(wait_ns),
                                                     _stream(stream, q.device)))


def lmhead_argmax_workspace_bytes(M, d, V, dtype):
    code = BF16 if dtype == torch.bfloat16 else F32
    return lib().glance_lmhead_argmax_workspace_bytes(M, d, V, code)


def lmhead_argmax(h, W, argmax, gap, maxlogit, ws, stream=None):
    M, d = h.shape
    assert W.shape[0] == d and h.is_contiguous() and W.is_contiguous() and h.dtype == W.dtype
    _check(lib().glance_lmhead_argmax(_ptr(h), _ptr(W), _dtype_code(h), M, d, W.shape[1],
                                      _ptr(argmax), _ptr(gap), _ptr(maxlogit), _ptr(ws),
                                      ws.numel(), _stream(stream, h.device)))


def lmhead_argmax_noalloc(h, W, argmax, gap, maxlogit, stream=None):
    """LM head + argmax for callers that cannot allocate: no workspace, the
    scratch lives in the library (calls on one device must not overlap)."""
    M, d = h.shape
    assert W.shape[0] == d and h.is_contiguous() and W.is_contiguous() and h.dtype == W.dtype
    _check(lib().glance_lmhead_argmax_noalloc(_ptr(h), _ptr(W), _dtype_code(h), M, d, W.shape[1],
                                              _ptr(argmax), _ptr(gap), _ptr(maxlogit),
                                              _stream(stream, h.device)))


def lmhead_packed_w_bytes(d, V):
    return lib().glance_lmhead_packed_w_bytes(d, V)


def lmhead_pack_w(W, W_packed, stream=None):
    """W (bf16 [d][V]) -> W_packed (any contiguous device tensor of at least
    lmhead_packed_w_bytes(d, V) bytes), the layout lmhead_argmax_packed reads."""
    d, V = W.shape
    assert W.is_contiguous() and W.dtype == torch.bfloat16 and W_packed.is_contiguous()
    _check(lib().glance_lmhead_pack_w(_ptr(W), d, V, _ptr(W_packed), W_packed.numel() * W_packed.element_size(),
                                      _stream(stream, W.device)))


def lmhead_argmax_packed(h, W_packed, V, argmax, gap, maxlogit, ws, stream=None):
    """lmhead_argmax (bf16, M <= 128) with W given as lmhead_pack_w wrote it."""
    M, d = h.shape
    assert h.is_contiguous() and h.dtype == torch.bfloat16 and W_packed.is_contiguous()
    _check(lib().glance_lmhead_argmax_packed(_ptr(h), _ptr(W_packed), M, d, V, _ptr(argmax), _ptr(gap),
                                             _ptr(maxlogit), _ptr(ws), ws.numel(), _stream(stream, h.device)))


def lmhead_argmax_entropy(h, W, argmax, gap, maxlogit, entropy, ws, stream=None):
    """lmhead_argmax plus each row's next-token entropy (nats), bf16."""
    M, d = h.shape
    assert W.shape[0] == d and h.is_contiguous() and W.is_contiguous() and h.dtype == W.dtype
    _check(lib().glance_lmhead_argmax_entropy(_ptr(h), _ptr(W), _dtype_code(h), M, d, W.shape[1],
                                              _ptr(argmax), _ptr(gap), _ptr(maxlogit),
                                              _ptr(entropy), _ptr(ws), ws.numel(),
                                              _stream(stream, h.device)))


def lmhead_sample(h, W, inv_temperature, seed, position, seq, tokens, gap, ws, stream=None):
    """Sampling-mode LM head: tokens[i] is a Gumbel-max draw from
    softmax(l_i / T), the noise keyed by (seed, position[i], seq[i])."""
    M, d = h.shape
    assert W.shape[0] == d and h.is_contiguous() and W.is_contiguous() and h.dtype == W.dtype
    _check(lib().glance_lmhead_sample(_ptr(h), _ptr(W), _dtype_code(h), M, d, W.shape[1],
                                      float(inv_temperature), int(seed) & ((1 << 64) - 1),
                                      _ptr(position), _ptr(seq), _ptr(tokens), _ptr(gap), _ptr(ws),
                                      ws.numel(), _stream(stream, h.device)))


def accept_commit_workspace_bytes(n_layers):
    return lib().glance_accept_commit_workspace_bytes(n_layers)


def accept_commit(tree, argmax, layers, n_accepted, accepted_tok, new_root, ws, stream=None):
    arr = (KVC * len(layers))(*[l.c for l in layers])
    _check(lib().glance_accept_commit(ctypes.byref(tree.c), _ptr(argmax), arr, len(layers),
                                      _ptr(n_accepted), _ptr(accepted_tok), _ptr(new_root),
                                      _ptr(ws), ws.numel(), _stream(stream, argmax.device)))


def accept_commit_gated(tree, argmax, gap, threshold, layers, n_accepted, accepted_tok, new_root,
                        gated, ws, stream=None):
    """accept_commit with the tie-aware gate on the rows' top-2 margins."""
    arr = (KVC * len(layers))(*[l.c for l in layers])
    _check(lib().glance_accept_commit_gated(ctypes.byref(tree.c), _ptr(argmax), _ptr(gap),
                                            float(threshold), arr, len(layers), _ptr(n_accepted),
                                            _ptr(accepted_tok), _ptr(new_root), _ptr(gated),
                                            _ptr(ws), ws.numel(), _stream(stream, argmax.device)))


# ------------------------------------------------------------ batched calls

def _trees(trees):
    return (TreeC * len(trees))(*[t.c for t in trees])


def _kvs(kvs):
    return (KVC * len(kvs))(*[k.c for k in kvs])


def build_tree_batched_workspace_bytes(B, L, V, N):
    return lib().glance_build_tree_batched_workspace_bytes(B, L, V, N)


def build_tree_batched(draft_logits, N, root_token, t_len, trees, ws, stream=None):
    """draft_logits [B][L][V]; root_token, t_len int32 [B]; trees: B Tree objects."""
    B, L, V = draft_logits.shape
    assert draft_logits.is_contiguous() and len(trees) == B
    _check(lib().glance_build_tree_batched(_ptr(draft_logits), _dtype_code(draft_logits), B, L, V,
                                           N, _ptr(root_token), _ptr(t_len), _trees(trees),
                                           _ptr(ws), ws.numel(),
                                           _stream(stream, draft_logits.device)))


def build_tree_shared_workspace_bytes(B, L, V, N_max):
    return lib().glance_build_tree_shared_workspace_bytes(B, L, V, N_max)


def build_tree_shared(draft_logits, N_max, N_total, root_token, t_len, trees, n_active, ws,
                      root_entropy=None, law_b0=0.0, law_b1=0.0, stream=None):
    """B trees under a shared budget of N_total nodes (at most N_max each); with
    root_entropy [B], node masses are keyed by the entropy law."""
    B, L, V = draft_logits.shape
    assert draft_logits.is_contiguous() and len(trees) == B
    _check(lib().glance_build_tree_shared(_ptr(draft_logits), _dtype_code(draft_logits), B, L, V,
                                          N_max, N_total, _ptr(root_token), _ptr(t_len),
                                          _ptr(root_entropy), float(law_b0), float(law_b1),
                                          _trees(trees), _ptr(n_active), _ptr(ws), ws.numel(),
                                          _stream(stream, draft_logits.device)))


def tree_attention_batched_workspace_bytes(rows, n_q_heads, kvs):
    return lib().glance_tree_attention_batched_workspace_bytes(len(kvs), rows, n_q_heads, _kvs(kvs))


def tree_attention_batched(q, kvs, trees, scale, out, ws, stream=None):
    """q, out [B][N+1][Hq][128] bf16; kvs: B KVLayer views of this layer."""
    B = q.shape[0]
    assert q.is_contiguous() and out.is_contiguous() and q.shape == out.shape
    assert len(kvs) == B and len(trees) == B
    _check(lib().glance_tree_attention_batched(_ptr(q), q.shape[2], _kvs(kvs), _trees(trees), B,
                                               float(scale), _ptr(out), _ptr(ws), ws.numel(),
                                               _stream(stream, q.device)))


def accept_commit_batched_workspace_bytes(B, n_layers):
    return lib().glance_accept_commit_batched_workspace_bytes(B, n_layers)


def accept_commit_batched(trees, argmax, layers, n_accepted, accepted_tok, new_root, ws,
                          stream=None):
    """layers[r][l]: KVLayer of request r, layer l; argmax [B][N+1]; outputs [B], [B][L], [B]."""
    B = len(trees)
    n_layers = len(layers[0])
    flat = [layers[r][l] for r in range(B) for l in range(n_layers)]
    _check(lib().glance_accept_commit_batched(_trees(trees), B, _ptr(argmax), _kvs(flat), n_layers,
                                              _ptr(n_accepted), _ptr(accepted_tok),
                                              _ptr(new_root), _ptr(ws), ws.numel(),
                                              _stream(stream, argmax.device)))


def accept_commit_gated_batched(trees, argmax, gap, threshold, layers, n_accepted, accepted_tok,
                                new_root, gated, ws, stream=None):
    B = len(trees)
    n_layers = len(layers[0])
    flat = [layers[r][l] for r in range(B) for l in range(n_layers)]
    _check(lib().glance_accept_commit_gated_batched(_trees(trees), B, _ptr(argmax), _ptr(gap),
                                                    float(threshold), _kvs(flat), n_layers,
                                                    _ptr(n_accepted), _ptr(accepted_tok),
                                                    _ptr(new_root), _ptr(gated), _ptr(ws),
                                                    ws.numel(), _stream(stream, argmax.device)))


# -------------------------------------------------------------- dense layers

def row_sumsq(x, sumsq, stream=None):
    """sumsq [M] (float32) = row sums of squares of x [M][d] (bf16)."""
    M, d = x.shape
    assert x.is_contiguous()
    _check(lib().glance_row_sumsq(_ptr(x), M, d, _ptr(sumsq), _stream(stream, x.device)))


def _n_parts(in_sumsq, M):
    if in_sumsq is None:
        return 0
    assert in_sumsq.dtype == torch.float32 and in_sumsq.is_contiguous() and in_sumsq.numel() % M == 0
    return in_sumsq.numel() // M


def dense_qkv(h, W_qkv, n_q_heads, in_sumsq, q_norm, k_norm, eps, pos_id, rope_theta, q_out, kv,
              stream=None):
    """in_sumsq: [n][M] partial row sums of squares of h (None: no input norm)."""
    M, d = h.shape
    assert h.is_contiguous() and W_qkv.is_contiguous() and q_out.is_contiguous()
    _check(lib().glance_dense_qkv(_ptr(h), _ptr(W_qkv), M, d, n_q_heads, _ptr(in_sumsq),
                                  _n_parts(in_sumsq, M), _ptr(q_norm), _ptr(k_norm), float(eps),
                                  _ptr(pos_id), float(rope_theta), _ptr(q_out), ctypes.byref(kv.c),
                                  _stream(stream, h.device)))


def dense_residual(x, W, residual, out, out_sumsq=None, stream=None):
    """out_sumsq: [N / 256][M] float32 to receive the output rows' sums of squares, or None."""
    M, K = x.shape
    N = W.shape[1]
    assert x.is_contiguous() and W.is_contiguous() and residual.is_contiguous() and out.is_contiguous()
    if out_sumsq is not None:
        assert out_sumsq.dtype == torch.float32 and out_sumsq.numel() >= (N // 256) * M
    _check(lib().glance_dense_residual(_ptr(x), _ptr(W), M, K, N, _ptr(residual), _ptr(out),
                                       _ptr(out_sumsq), _stream(stream, x.device)))


def dense_swiglu(h, W_gate, W_up, in_sumsq, eps, act, stream=None):
    M, d = h.shape
    inter = W_gate.shape[1]
    assert h.is_contiguous() and W_gate.is_contiguous() and W_up.is_contiguous() and act.is_contiguous()
    _check(lib().glance_dense_swiglu(_ptr(h), _ptr(W_gate), _ptr(W_up), M, d, inter, _ptr(in_sumsq),
                                     _n_parts(in_sumsq, M), float(eps), _ptr(act),
                                     _stream(stream, h.device)))


def device_status():
    """(code, text) of the device status word; synchronises the device."""
    code = ctypes.c_int32(0)
    lib().glance_device_status(ctypes.byref(code))
    return code.value, DEV_STATUS.get(code.value, "unknown")


def reset_device_status():
    _check(lib().glance_reset_device_status())


def kv_write_rows(src, layers, rows, stream=None):
    """Scatter src [n_layers, 2, n_kv_heads, rows, head_dim] (K before V) into
    every layer's cache at slots T..T+rows-1 (T read on the device)."""
    assert src.is_contiguous()
    arr = (KVC * len(layers))(*[l.c for l in layers])
    _check(lib().glance_kv_write_rows(_ptr(src), arr, len(layers), int(rows), _stream(stream, src.device)))


STATUS_WORDS = 6


def get_status(out, stream=None):
    """Enqueue the stream-ordered status read: out (int32 [6], CUDA or pinned
    host tensor) gets the first non-zero word in out[0] and the words of the
    tree build, attention, LM head, commit and dense kernels in out[1..5]."""
    assert out.dtype == torch.int32 and out.numel() >= STATUS_WORDS and out.is_contiguous()
    if not (out.is_cuda or out.is_pinned()):
        raise ValueError("glance: get_status needs a CUDA or pinned host tensor")
    dev = out.device if out.is_cuda else torch.device("cuda", torch.cuda.current_device())
    _check(lib().glance_get_status(ctypes.c_void_p(out.data_ptr()), _stream(stream, dev)))


def clear_status(stream=None, device=None):
    """Enqueue a clear of every device status word on the stream."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    _check(lib().glance_clear_status(_stream(stream, dev)))


def version():
    return lib().glance_version()
