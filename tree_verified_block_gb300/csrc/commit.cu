// Acceptance walk A(S) and KV commit. One launch.
//
// Paper: "Vision Is Not Overhead ..." (arXiv 2609.00355), Definition 1
// (A(S) = max{k : Y_{1:j} in S for all j <= k}; commit Y_{1:A(S)} and emit
// the next greedy token of the last verified row as the new root), Section
// 3.1 (a round commits a + 1 tokens) and the proof of Theorem 1 in Appendix
// B.1 (descend while the target's greedy token is a child, else stop).
//
// Grid: one CTA per (layer, K or V, kv head). Every CTA repeats the walk in
// its first warp (at most L steps, each a warp ballot over the rows looking
// for the child of the current row whose token is the row's argmax; siblings
// have distinct tokens, so at most one matches), then moves its slice of the
// path rows: slot T + path_i -> slot T + i for i = 0..a. A destination slot
// can be the source of a later path row (path = [0, 2, 3] moves 2 -> 1 and
// 3 -> 2), so every source row is staged in shared memory before any
// destination is written. The last CTA to finish (atomic ticket; all others
// have read T by then) writes a, the accepted tokens and the new root, and
// advances T by a + 1.
#include "glance_internal.cuh"

GLANCE_DEFINE_STATUS_WORD(status_commit)

using namespace glance_dev;

namespace {

constexpr int kMaxLayers = 128;
constexpr int kMaxRowBytes = 512;  // head_dim * element size
constexpr int kMaxPath = 17;       // root + L <= 16 accepted rows
constexpr int kThreads = 128;

struct LayerPtrs {
  char* k;
  char* v;
};

struct CommitParams {
  const int32_t* token;
  const int32_t* parent;
  const int32_t* depth;
  const int32_t* argmax;
  int rows, L;
  int n_layers, n_kv_heads, row_bytes, t_cap;
  long long head_stride_bytes, row_stride_bytes;
  int32_t* t_len;
  int32_t* n_accepted;
  int32_t* accepted_tok;
  int32_t* new_root;
  uint32_t* ticket;
  LayerPtrs layer[kMaxLayers];
};

__global__ void __launch_bounds__(kThreads) accept_commit_kernel(const CommitParams p) {
  __shared__ int s_path[kMaxPath];
  __shared__ int s_a, s_newroot, s_T;
  __shared__ __align__(16) unsigned char stage[kMaxPath * kMaxRowBytes];
  __shared__ uint32_t s_ticket;
  __shared__ int s_tok[256], s_par[256], s_dep[256], s_arg[256];

  // stage the tree and the argmax row tokens (coalesced), then walk in smem
  for (int i = threadIdx.x; i < p.rows; i += kThreads) {
    s_tok[i] = __ldg(p.token + i);
    s_par[i] = __ldg(p.parent + i);
    s_dep[i] = __ldg(p.depth + i);
    s_arg[i] = __ldg(p.argmax + i);
  }
  if (threadIdx.x == 0) s_T = *p.t_len;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int u = 0, a = 0;
    if (lane == 0) s_path[0] = 0;
    for (int step = 0; step < p.L; ++step) {
      if (s_dep[u] >= p.L) break;
      const int target = s_arg[u];
      int found = -1;
      for (int base = 0; base < p.rows; base += 32) {
        const int c = base + lane;
        const bool hit = c < p.rows && c > 0 && s_par[c] == u && s_tok[c] == target;
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (m) {
          found = base + __ffs(m) - 1;
          break;
        }
      }
      if (found < 0) break;
      u = found;
      ++a;
      if (lane == 0) s_path[a] = u;
    }
    if (lane == 0) {
      s_a = a;
      s_newroot = s_arg[u];
    }
  }
  __syncthreads();
  const int a = s_a, T = s_T;
  const int n_rows = a + 1;

  // slice: blockIdx.x = (layer * 2 + kv) * n_kv_heads + head
  const int head = blockIdx.x % p.n_kv_heads;
  const int lk = blockIdx.x / p.n_kv_heads;
  const int layer = lk >> 1;
  char* base = (lk & 1) ? p.layer[layer].v : p.layer[layer].k;
  base += head * p.head_stride_bytes;
  const bool room = T >= 0 && T + p.rows <= p.t_cap;
  if (!room && blockIdx.x == 0 && threadIdx.x == 0) report(GLANCE_DEV_TREE_CAPACITY);
  if (room && a > 0) {
    const int vec_per_row = p.row_bytes / 16;
    const int total = n_rows * vec_per_row;
    for (int i = threadIdx.x; i < total; i += kThreads) {
      const int r = i / vec_per_row, c = i - r * vec_per_row;
      const char* src = base + static_cast<long long>(T + s_path[r]) * p.row_stride_bytes + 16 * c;
      *reinterpret_cast<uint4*>(stage + r * p.row_bytes + 16 * c) =
          *reinterpret_cast<const uint4*>(src);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < total; i += kThreads) {
      const int r = i / vec_per_row, c = i - r * vec_per_row;
      char* dst = base + static_cast<long long>(T + r) * p.row_stride_bytes + 16 * c;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(stage + r * p.row_bytes + 16 * c);
    }
  }

  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_ticket = atomicAdd(p.ticket, 1u);
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;
  if (threadIdx.x == 0) {
    *p.ticket = 0;
    *p.n_accepted = a;
    *p.new_root = s_newroot;
    if (room) *p.t_len = T + a + 1;
  }
  if (threadIdx.x >= 1 && threadIdx.x <= a) p.accepted_tok[threadIdx.x - 1] = s_tok[s_path[threadIdx.x]];
}

}  // namespace

extern "C" size_t glance_accept_commit_workspace_bytes(int n_layers) {
  return (n_layers >= 1 && n_layers <= kMaxLayers) ? 256 : 0;
}

extern "C" glance_status glance_accept_commit(const glance_tree* tree, const int32_t* argmax,
                                              const glance_kv* layers, int n_layers,
                                              int32_t* n_accepted, int32_t* accepted_tok,
                                              int32_t* new_root, void* workspace,
                                              size_t workspace_bytes, void* stream) {
  using glance::fail;
  if (!tree || !argmax || !layers || !n_accepted || !accepted_tok || !new_root || !workspace)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_accept_commit: null pointer argument");
  if (n_layers < 1 || n_layers > kMaxLayers)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_accept_commit: n_layers must be in [1, %d]",
                kMaxLayers);
  if (tree->n < 1 || tree->n > 255 || tree->L < 1 || tree->L > 16 || !tree->token ||
      !tree->parent || !tree->depth)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_accept_commit: bad tree struct");
  if (workspace_bytes < 256)
    return fail(GLANCE_ERR_CAPACITY, "glance_accept_commit: workspace must be >= 256 bytes");
  const glance_kv& l0 = layers[0];
  const int esize = l0.dtype == GLANCE_BF16 ? 2 : 4;
  if (l0.dtype != GLANCE_BF16 && l0.dtype != GLANCE_F32)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_accept_commit: kv dtype must be F32 or BF16");
  const int row_bytes = l0.head_dim * esize;
  if (l0.head_dim < 1 || row_bytes % 16 != 0 || row_bytes > kMaxRowBytes)
    return fail(GLANCE_ERR_UNSUPPORTED,
                "glance_accept_commit: head_dim * element size must be a multiple of 16 and "
                "<= %d bytes",
                kMaxRowBytes);
  if (l0.n_kv_heads < 1 || l0.t_cap < tree->n + 1 || !l0.t_len)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_accept_commit: bad kv geometry");
  if ((l0.row_stride * esize) % 16 != 0 || (l0.head_stride * esize) % 16 != 0 ||
      l0.row_stride < l0.head_dim || l0.head_stride < static_cast<int64_t>(l0.t_cap) * l0.row_stride)
    return fail(GLANCE_ERR_INVALID_ARG,
                "glance_accept_commit: strides must be 16-byte multiples covering the rows");
  CommitParams p;
  for (int l = 0; l < n_layers; ++l) {
    const glance_kv& x = layers[l];
    if (x.dtype != l0.dtype || x.head_dim != l0.head_dim || x.n_kv_heads != l0.n_kv_heads ||
        x.t_cap != l0.t_cap || x.head_stride != l0.head_stride ||
        x.row_stride != l0.row_stride || x.t_len != l0.t_len)
      return fail(GLANCE_ERR_INVALID_ARG,
                  "glance_accept_commit: every layer must share geometry and t_len (layer %d)",
                  l);
    if (!x.k || !x.v || !glance::aligned16(x.k) || !glance::aligned16(x.v))
      return fail(GLANCE_ERR_INVALID_ARG,
                  "glance_accept_commit: layer %d K/V must be non-null, 16-byte aligned", l);
    p.layer[l].k = static_cast<char*>(x.k);
    p.layer[l].v = static_cast<char*>(x.v);
  }
  p.token = tree->token;
  p.parent = tree->parent;
  p.depth = tree->depth;
  p.argmax = argmax;
  p.rows = tree->n + 1;
  p.L = tree->L;
  p.n_layers = n_layers;
  p.n_kv_heads = l0.n_kv_heads;
  p.row_bytes = row_bytes;
  p.t_cap = l0.t_cap;
  p.head_stride_bytes = l0.head_stride * esize;
  p.row_stride_bytes = l0.row_stride * esize;
  p.t_len = l0.t_len;
  p.n_accepted = n_accepted;
  p.accepted_tok = accepted_tok;
  p.new_root = new_root;
  p.ticket = static_cast<uint32_t*>(workspace);
  const int grid = n_layers * 2 * l0.n_kv_heads;
  accept_commit_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return glance::cuda_fail(e, "glance_accept_commit: launch");
  return GLANCE_OK;
}
