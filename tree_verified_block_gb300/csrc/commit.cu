// Acceptance walk A(S) and KV commit. One launch.
//
// Paper: "Vision Is Not Overhead ..." (arXiv 2609.00355), Definition 1
// (A(S) = max{k : Y_{1:j} in S for all j <= k}; commit Y_{1:A(S)} and emit
// the next greedy token of the last verified row as the new root), Section
// 3.1 (a round commits a + 1 tokens) and the proof of Theorem 1 in Appendix
// B.1 (descend while the target's greedy token is a child, else stop).
//
// Grid: one CTA per (request, layer, K or V, kv head). Every CTA repeats the
// walk of its request in
// its first warp (at most L steps, each a warp ballot over the rows looking
// for the child of the current row whose token is the row's argmax; siblings
// have distinct tokens, so at most one matches), then moves its slice of the
// path rows: slot T + path_i -> slot T + i for i = 0..a. A destination slot
// can be the source of a later path row (path = [0, 2, 3] moves 2 -> 1 and
// 3 -> 2), so every source row is staged in shared memory before any
// destination is written. The last CTA of a request to finish (atomic ticket;
// all others have read T by then) writes a, the accepted tokens and the new
// root of that request, and advances its T by a + 1.
//
// Tie-aware gate (Section 4.2; the end of the proof of Theorem 1 in Appendix
// B.1), when the rows' top-2 margins are given: the walk stops at the first
// visited row whose margin is below the threshold (a near-tie, where reduced
// precision may reorder the target's top two tokens) and flags the request;
// its new root is then the caller's to recompute.
#include "glance_internal.cuh"

GLANCE_DEFINE_STATUS_WORD(status_commit)

using namespace glance_dev;

namespace {

constexpr int kMaxLayers = 128;
constexpr int kMaxB = 16;
constexpr int kMaxEntries = 1024;  // requests x layers of one call
constexpr int kSmallEntries = 128;  // parameter block of the common small calls
constexpr int kMaxRowBytes = 512;  // head_dim * element size
constexpr int kMaxPath = 17;       // root + L <= 16 accepted rows
constexpr int kThreads = 128;

struct LayerPtrs {
  char* k;
  char* v;
};

struct ReqInfo {
  const int32_t* token;
  const int32_t* parent;
  const int32_t* depth;
  int32_t* t_len;
  long long head_stride_bytes, row_stride_bytes;
  int t_cap;
};

template <int kEntries>
struct CommitParams {
  const int32_t* argmax;      // [B][rows]
  const float* gap;           // [B][rows] top-2 margins, or null (no gate)
  float gate;                 // margin threshold of the gate
  int32_t* gated;             // [B], or null
  int rows, L, B;
  int n_layers, n_kv_heads, row_bytes;
  int32_t* n_accepted;        // [B]
  int32_t* accepted_tok;      // [B][L]
  int32_t* new_root;          // [B]
  uint32_t* ticket;           // [B]
  ReqInfo req[kMaxB];
  LayerPtrs layer[kEntries];  // [B][n_layers]
};

template <int kEntries>
__global__ void __launch_bounds__(kThreads)
    accept_commit_kernel(const __grid_constant__ CommitParams<kEntries> p) {
  __shared__ int s_path[kMaxPath];
  __shared__ int s_a, s_newroot, s_T;
  __shared__ __align__(16) unsigned char stage[kMaxPath * kMaxRowBytes];
  __shared__ uint32_t s_ticket;
  __shared__ int s_tok[256], s_par[256], s_dep[256], s_arg[256];
  __shared__ float s_gap[256];
  __shared__ int s_gated;

  // slice: blockIdx.x = ((request * n_layers + layer) * 2 + kv) * n_kv_heads + head
  // launched as a programmatic dependent of the LM head: nothing is read
  // before its writes are visible
  pdl_wait_prior();
  const int per_req = p.n_layers * 2 * p.n_kv_heads;
  const int req = blockIdx.x / per_req;
  const ReqInfo& rq = p.req[req];
  // stage the tree and the argmax row tokens (coalesced), then walk in smem
  for (int i = threadIdx.x; i < p.rows; i += kThreads) {
    s_tok[i] = __ldg(rq.token + i);
    s_par[i] = __ldg(rq.parent + i);
    s_dep[i] = __ldg(rq.depth + i);
    s_arg[i] = __ldg(p.argmax + req * p.rows + i);
    s_gap[i] = p.gap ? __ldg(p.gap + req * p.rows + i) : INFINITY;
  }
  if (threadIdx.x == 0) s_T = *rq.t_len;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int u = 0, a = 0;
    bool gated = false;
    if (lane == 0) s_path[0] = 0;
    for (int step = 0; step <= p.L; ++step) {
      if (s_gap[u] < p.gate) {  // near-tie on the path: defer (never true without margins)
        gated = true;
        break;
      }
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
      s_gated = gated ? 1 : 0;
    }
  }
  __syncthreads();
  const int a = s_a, T = s_T;
  const int n_rows = a + 1;

  const int slice = blockIdx.x - req * per_req;
  const int head = slice % p.n_kv_heads;
  const int lk = slice / p.n_kv_heads;
  const int layer = lk >> 1;
  const LayerPtrs& lp = p.layer[req * p.n_layers + layer];
  char* base = (lk & 1) ? lp.v : lp.k;
  base += head * rq.head_stride_bytes;
  const bool room = T >= 0 && T + p.rows <= rq.t_cap;
  if (!room && slice == 0 && threadIdx.x == 0) report(GLANCE_DEV_TREE_CAPACITY);
  if (room && a > 0) {
    const int vec_per_row = p.row_bytes / 16;
    const int total = n_rows * vec_per_row;
    for (int i = threadIdx.x; i < total; i += kThreads) {
      const int r = i / vec_per_row, c = i - r * vec_per_row;
      const char* src = base + static_cast<long long>(T + s_path[r]) * rq.row_stride_bytes + 16 * c;
      if (GLANCE_IN_BOUNDS(T + s_path[r], rq.t_cap))
        *reinterpret_cast<uint4*>(stage + r * p.row_bytes + 16 * c) = *reinterpret_cast<const uint4*>(src);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < total; i += kThreads) {
      const int r = i / vec_per_row, c = i - r * vec_per_row;
      char* dst = base + static_cast<long long>(T + r) * rq.row_stride_bytes + 16 * c;
      if (GLANCE_IN_BOUNDS(T + r, rq.t_cap))
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(stage + r * p.row_bytes + 16 * c);
    }
  }

  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_ticket = atomicAdd(p.ticket + req, 1u);
  __syncthreads();
  if (s_ticket != static_cast<uint32_t>(per_req - 1)) return;
  if (threadIdx.x == 0) {
    p.ticket[req] = 0;
    p.n_accepted[req] = a;
    p.new_root[req] = s_newroot;
    if (p.gated) p.gated[req] = s_gated;
    if (room) *rq.t_len = T + a + 1;
  }
  if (threadIdx.x >= 1 && threadIdx.x <= a && GLANCE_IN_BOUNDS(s_path[threadIdx.x], p.rows))
    p.accepted_tok[req * p.L + threadIdx.x - 1] = s_tok[s_path[threadIdx.x]];
}

template <int kEntries>
glance_status fill_and_launch(const char* who, const glance_tree* trees, int B,
                              const int32_t* argmax, const float* gap, float gate, int32_t* gated,
                              const glance_kv* layers, int n_layers, int32_t* n_accepted,
                              int32_t* accepted_tok, int32_t* new_root, void* workspace,
                              int row_bytes, int esize, void* stream);

// layers: [B][n_layers] cache views, argmax [B][rows]; outputs per request.
glance_status launch_commit(const char* who, const glance_tree* trees, int B,
                            const int32_t* argmax, const float* gap, float gate,
                            int32_t* gated, const glance_kv* layers, int n_layers,
                            int32_t* n_accepted, int32_t* accepted_tok, int32_t* new_root,
                            void* workspace, size_t workspace_bytes, void* stream) {
  using glance::fail;
  if (!trees || !argmax || !layers || !n_accepted || !accepted_tok || !new_root || !workspace)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: null pointer argument", who);
  if (B < 1 || B > kMaxB) return fail(GLANCE_ERR_INVALID_ARG, "%s: need 1 <= B <= %d", who, kMaxB);
  if (n_layers < 1 || n_layers > kMaxLayers || B * n_layers > kMaxEntries)
    return fail(GLANCE_ERR_INVALID_ARG,
                "%s: need 1 <= n_layers <= %d and B * n_layers <= %d", who, kMaxLayers,
                kMaxEntries);
  if (workspace_bytes < 256)
    return fail(GLANCE_ERR_CAPACITY, "%s: workspace must be >= 256 bytes", who);
  const glance_kv& l0 = layers[0];
  if (l0.dtype != GLANCE_BF16 && l0.dtype != GLANCE_F32)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: kv dtype must be F32 or BF16", who);
  const int esize = l0.dtype == GLANCE_BF16 ? 2 : 4;
  const int row_bytes = l0.head_dim * esize;
  if (l0.head_dim < 1 || row_bytes % 16 != 0 || row_bytes > kMaxRowBytes)
    return fail(GLANCE_ERR_UNSUPPORTED,
                "%s: head_dim * element size must be a multiple of 16 and <= %d bytes", who,
                kMaxRowBytes);
  if (B * n_layers <= kSmallEntries)
    return fill_and_launch<kSmallEntries>(who, trees, B, argmax, gap, gate, gated, layers,
                                          n_layers, n_accepted, accepted_tok, new_root, workspace,
                                          row_bytes, esize, stream);
  return fill_and_launch<kMaxEntries>(who, trees, B, argmax, gap, gate, gated, layers, n_layers,
                                      n_accepted, accepted_tok, new_root, workspace, row_bytes,
                                      esize, stream);
}

template <int kEntries>
glance_status fill_and_launch(const char* who, const glance_tree* trees, int B,
                              const int32_t* argmax, const float* gap, float gate, int32_t* gated,
                              const glance_kv* layers, int n_layers, int32_t* n_accepted,
                              int32_t* accepted_tok, int32_t* new_root, void* workspace,
                              int row_bytes, int esize, void* stream) {
  using glance::fail;
  const glance_kv& l0 = layers[0];
  CommitParams<kEntries> p;
  const int n = trees[0].n, L = trees[0].L;
  for (int r = 0; r < B; ++r) {
    const glance_tree& t = trees[r];
    if (t.n != n || t.L != L || t.n < 1 || t.n > 255 || t.L < 1 || t.L > 16 || !t.token ||
        !t.parent || !t.depth)
      return fail(GLANCE_ERR_INVALID_ARG, "%s: bad tree struct (request %d)", who, r);
    const glance_kv& f = layers[r * n_layers];
    if (f.dtype != l0.dtype || f.head_dim != l0.head_dim || f.n_kv_heads != l0.n_kv_heads)
      return fail(GLANCE_ERR_INVALID_ARG,
                  "%s: every request must share dtype, head_dim and n_kv_heads (request %d)", who,
                  r);
    if (f.n_kv_heads < 1 || f.t_cap < n + 1 || !f.t_len)
      return fail(GLANCE_ERR_INVALID_ARG, "%s: bad kv geometry (request %d)", who, r);
    if ((f.row_stride * esize) % 16 != 0 || (f.head_stride * esize) % 16 != 0 ||
        f.row_stride < f.head_dim || f.head_stride < static_cast<int64_t>(f.t_cap) * f.row_stride)
      return fail(GLANCE_ERR_INVALID_ARG,
                  "%s: strides must be 16-byte multiples covering the rows (request %d)", who, r);
    for (int l = 0; l < n_layers; ++l) {
      const glance_kv& x = layers[r * n_layers + l];
      if (x.dtype != f.dtype || x.head_dim != f.head_dim || x.n_kv_heads != f.n_kv_heads ||
          x.t_cap != f.t_cap || x.head_stride != f.head_stride || x.row_stride != f.row_stride ||
          x.t_len != f.t_len)
        return fail(GLANCE_ERR_INVALID_ARG,
                    "%s: every layer of a request must share geometry and t_len (request %d, "
                    "layer %d)", who, r, l);
      if (!x.k || !x.v || !glance::aligned16(x.k) || !glance::aligned16(x.v))
        return fail(GLANCE_ERR_INVALID_ARG,
                    "%s: K/V of request %d layer %d must be non-null, 16-byte aligned", who, r, l);
      p.layer[r * n_layers + l].k = static_cast<char*>(x.k);
      p.layer[r * n_layers + l].v = static_cast<char*>(x.v);
    }
    for (int q = 0; q < r; ++q)
      if (layers[q * n_layers].t_len == f.t_len)
        return fail(GLANCE_ERR_INVALID_ARG, "%s: requests %d and %d share t_len", who, q, r);
    ReqInfo& ri = p.req[r];
    ri.token = t.token;
    ri.parent = t.parent;
    ri.depth = t.depth;
    ri.t_len = f.t_len;
    ri.head_stride_bytes = f.head_stride * esize;
    ri.row_stride_bytes = f.row_stride * esize;
    ri.t_cap = f.t_cap;
  }
  for (int r = B; r < kMaxB; ++r) p.req[r] = p.req[0];
  p.argmax = argmax;
  p.gap = gap;
  p.gate = gate;
  p.gated = gated;
  p.rows = n + 1;
  p.L = L;
  p.B = B;
  p.n_layers = n_layers;
  p.n_kv_heads = l0.n_kv_heads;
  p.row_bytes = row_bytes;
  p.n_accepted = n_accepted;
  p.accepted_tok = accepted_tok;
  p.new_root = new_root;
  p.ticket = static_cast<uint32_t*>(workspace);
  const int grid = B * n_layers * 2 * l0.n_kv_heads;
  // a programmatic dependent of the previous kernel (the LM head lets it
  // launch once every CTA has written its partial; the kernel waits at its
  // first instruction). It lets no kernel after it start early: the cache
  // prefix and T it writes are read before the dependency wait by the next
  // attention call.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, accept_commit_kernel<kEntries>, p);
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  e = cudaGetLastError();
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  return GLANCE_OK;
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
  return launch_commit("glance_accept_commit", tree, 1, argmax, nullptr, 0.f, nullptr, layers,
                       n_layers, n_accepted, accepted_tok, new_root, workspace, workspace_bytes,
                       stream);
}

extern "C" size_t glance_accept_commit_batched_workspace_bytes(int B, int n_layers) {
  return (B >= 1 && B <= kMaxB && n_layers >= 1 && n_layers <= kMaxLayers &&
          B * n_layers <= kMaxEntries)
             ? 256
             : 0;
}

extern "C" glance_status glance_accept_commit_batched(const glance_tree* trees, int B,
                                                      const int32_t* argmax,
                                                      const glance_kv* layers, int n_layers,
                                                      int32_t* n_accepted, int32_t* accepted_tok,
                                                      int32_t* new_root, void* workspace,
                                                      size_t workspace_bytes, void* stream) {
  return launch_commit("glance_accept_commit_batched", trees, B, argmax, nullptr, 0.f, nullptr,
                       layers, n_layers, n_accepted, accepted_tok, new_root, workspace,
                       workspace_bytes, stream);
}

extern "C" glance_status glance_accept_commit_gated(const glance_tree* tree, const int32_t* argmax,
                                                    const float* gap, float gate_threshold,
                                                    const glance_kv* layers, int n_layers,
                                                    int32_t* n_accepted, int32_t* accepted_tok,
                                                    int32_t* new_root, int32_t* gated,
                                                    void* workspace, size_t workspace_bytes,
                                                    void* stream) {
  if (!gap || !gated)
    return glance::fail(GLANCE_ERR_INVALID_ARG, "glance_accept_commit_gated: null gap or gated");
  return launch_commit("glance_accept_commit_gated", tree, 1, argmax, gap, gate_threshold, gated,
                       layers, n_layers, n_accepted, accepted_tok, new_root, workspace,
                       workspace_bytes, stream);
}

extern "C" glance_status glance_accept_commit_gated_batched(
    const glance_tree* trees, int B, const int32_t* argmax, const float* gap, float gate_threshold,
    const glance_kv* layers, int n_layers, int32_t* n_accepted, int32_t* accepted_tok,
    int32_t* new_root, int32_t* gated, void* workspace, size_t workspace_bytes, void* stream) {
  if (!gap || !gated)
    return glance::fail(GLANCE_ERR_INVALID_ARG,
                        "glance_accept_commit_gated_batched: null gap or gated");
  return launch_commit("glance_accept_commit_gated_batched", trees, B, argmax, gap,
                       gate_threshold, gated, layers, n_layers, n_accepted, accepted_tok, new_root,
                       workspace, workspace_bytes, stream);
}

// ------------------------------------------------------ tree rows into caches
//
// The verify pass writes the K/V of the packed tree rows into every layer's
// cache at slots T..T+rows-1 (row r at T + r) before tree attention reads them
// (Definition 1: the rows are evaluated in the same pass as the prefix). This
// call does that for K/V rows computed elsewhere (e.g. uploaded from the
// host): one CTA per (layer, K or V, kv head) copies that head's rows with
// 16-byte loads and stores.

namespace {

constexpr int kRowsThreads = 256;

struct RowsParams {
  const char* src;            // [n_layers][2][n_kv_heads][rows][row_bytes]
  char* dst[2 * kMaxLayers];  // per (layer, K/V): the cache
  const int32_t* t_len;
  long long head_stride_bytes, row_stride_bytes;
  int n_kv_heads, rows, row_bytes, t_cap;
};

__global__ void __launch_bounds__(kRowsThreads) kv_write_rows_kernel(const __grid_constant__ RowsParams p) {
  const int head = blockIdx.x % p.n_kv_heads;
  const int lkv = blockIdx.x / p.n_kv_heads;  // layer * 2 + (0: K, 1: V)
  const int T = *p.t_len;
  if (T < 0 || T + p.rows > p.t_cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(GLANCE_DEV_TREE_CAPACITY);
    return;
  }
  const int per_row = p.row_bytes / 16;
  const uint4* src = reinterpret_cast<const uint4*>(
      p.src + (static_cast<size_t>(lkv) * p.n_kv_heads + head) * p.rows * p.row_bytes);
  char* dst = p.dst[lkv] + head * p.head_stride_bytes + static_cast<long long>(T) * p.row_stride_bytes;
  for (int i = threadIdx.x; i < p.rows * per_row; i += kRowsThreads) {
    const int r = i / per_row, c = i - r * per_row;
    if (GLANCE_IN_BOUNDS(T + r, p.t_cap)) reinterpret_cast<uint4*>(dst + r * p.row_stride_bytes)[c] = __ldg(src + i);
  }
}

}  // namespace

extern "C" glance_status glance_kv_write_rows(const void* src, const glance_kv* layers, int n_layers,
                                              int rows, void* stream) {
  using glance::fail;
  const char* who = "glance_kv_write_rows";
  if (!src || !layers) return fail(GLANCE_ERR_INVALID_ARG, "%s: null pointer argument", who);
  if (n_layers < 1 || n_layers > kMaxLayers || rows < 1 || rows > 256)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: need 1 <= n_layers <= %d and 1 <= rows <= 256", who,
                kMaxLayers);
  const glance_kv& l0 = layers[0];
  const int esize = l0.dtype == GLANCE_BF16 ? 2 : 4;
  RowsParams p;
  p.src = static_cast<const char*>(src);
  p.t_len = l0.t_len;
  p.head_stride_bytes = l0.head_stride * esize;
  p.row_stride_bytes = l0.row_stride * esize;
  p.n_kv_heads = l0.n_kv_heads;
  p.rows = rows;
  p.row_bytes = l0.head_dim * esize;
  p.t_cap = l0.t_cap;
  if (!glance::aligned16(src) || p.row_bytes % 16 || p.row_stride_bytes % 16 || p.head_stride_bytes % 16)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: src, rows and strides must be 16-byte aligned", who);
  for (int l = 0; l < n_layers; ++l) {
    const glance_kv& x = layers[l];
    if (!x.k || !x.v || x.t_len != l0.t_len || x.dtype != l0.dtype || x.n_kv_heads != l0.n_kv_heads ||
        x.head_dim != l0.head_dim || x.t_cap != l0.t_cap || x.head_stride != l0.head_stride ||
        x.row_stride != l0.row_stride || x.n_kv_heads < 1 || x.t_cap < rows ||
        x.row_stride < x.head_dim || x.head_stride < static_cast<int64_t>(x.t_cap) * x.row_stride)
      return fail(GLANCE_ERR_INVALID_ARG,
                  "%s: every layer needs k, v, the same t_len, dtype and geometry (layer %d)", who, l);
    if (!glance::aligned16(x.k) || !glance::aligned16(x.v))
      return fail(GLANCE_ERR_INVALID_ARG, "%s: k and v must be 16-byte aligned (layer %d)", who, l);
    p.dst[2 * l] = static_cast<char*>(x.k);
    p.dst[2 * l + 1] = static_cast<char*>(x.v);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  kv_write_rows_kernel<<<n_layers * 2 * l0.n_kv_heads, kRowsThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  return GLANCE_OK;
}
