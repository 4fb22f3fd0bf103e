// Draft-to-tree: per-offset log-softmax + top-K, best-first top-N builder,
// canonical packing. One launch.
//
// Paper: "Vision Is Not Overhead ..." (arXiv 2609.00355), Assumption 1 (one
// marginal q_j per offset, plug-in score pi_hat = prod_j q_j(y_j)),
// Definition 1 (prefix-closed candidate tree, budget N, packed into one
// ancestor-masked pass) and Section 4.2 (keep the N prefixes of highest
// plug-in score).
//
// Layout of the work (grid = L rows x C chunks of 8192 logits, 256 threads):
//  1. every CTA streams its chunk into registers (vectorised, coalesced),
//     computes the chunk max and sum of exp, and selects the chunk's K best
//     tokens. Selection first histograms the gap to the chunk max in 2048
//     buckets of 1/64 nat (exact: the bucket is monotone in the logit), then,
//     only inside the boundary bucket, runs a radix select on unique 64-bit
//     keys (order-preserving logit bits << 32 | ~token id), so that equal
//     logits rank by ascending id;
//  2. the last CTA of each row (atomic ticket, no spinning) selects the K best
//     of the row's chunk candidates the same way, ranks them by counting and
//     writes (token, log q) using the row's log-sum-exp (fp32: each chunk's
//     sum is relative to its own max, so every term is at most 8192);
//  3. the last row-merger overall runs the best-first search in one warp
//     (frontier nodes in registers, 2 / 4 / 8 slots per lane by N, one warp
//     max-reduction per pop; exact score ties take a slow path that compares
//     depth and rank vectors) and the whole CTA packs the N popped nodes into
//     canonical order.
#include "glance_internal.cuh"

#include <cstddef>

GLANCE_DEFINE_STATUS_WORD(status_build_tree)

using namespace glance_dev;

namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 32;
constexpr int kChunk = kThreads * kPerThread;  // logits per CTA
constexpr int kMaxL = 16;
constexpr int kMaxN = 255;
constexpr int kMaxB = 16;       // requests of one batched call
constexpr int kTicketsPerReq = 32;  // [0, L): row tickets, [kMaxL]: request ticket

// B requests (blockIdx.y); "global row" = request * L + offset row.
struct BuildParams {
  const void* logits;           // [B][L][V]
  int is_bf16;
  int B, L, V, N, K, C;
  const int32_t* root_token;    // [B]
  const int32_t* t_len;         // [B]
  uint32_t* tickets;            // [B][kTicketsPerReq]
  float* chunk_m;               // [B * L][C] chunk max
  float* chunk_s;               // [B * L][C] chunk sum exp(x - m)
  unsigned long long* cand;     // [B * L][C][K]
  int32_t* top_tok;             // [B * L][K]
  float* top_logq;              // [B * L][K]
  glance_tree tree[kMaxB];
  // shared budget (two launches): the search writes its pops here instead of
  // packing; the pack kernel allocates the budget and packs
  int search_only;
  void* pops_out;               // [B][kMaxN] PopRec
};

constexpr int kBuckets = 2048;      // first-pass buckets of the gap to the max
constexpr float kBucketsPerNat = 64.f;

constexpr int kBoundary = 512;  // boundary-bucket items resolved by counting

struct SelectSmem {
  uint32_t hist[kBuckets];
  uint32_t warp_tot[kThreads / 32];
  int bstar;
  uint32_t above, cnt;
  uint32_t digit, above2, cnt2;
  uint32_t nb;
  uint32_t pos;  // pass-2 output count
  unsigned long long bnd[kBoundary];
};

__device__ __forceinline__ float inv_ord_key(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

__device__ __forceinline__ unsigned long long make_key(float x, uint32_t id) {
  return (static_cast<unsigned long long>(ord_key(x)) << 32) | (0xFFFFFFFFu - id);
}

// Bucket of a logit x given the maximum m (x <= m): floor((m - x) * 64),
// clamped. Non-increasing in x, equal for equal x, so lower buckets hold
// strictly larger logits.
__device__ __forceinline__ int bucket_of(float m, float x) {
  const float dd = (m - x) * kBucketsPerNat;
  return dd < static_cast<float>(kBuckets - 1) ? static_cast<int>(dd) : kBuckets - 1;
}

// Inclusive block scan (sum) of one value per thread; 256 threads.
__device__ uint32_t block_incl_scan(uint32_t v, uint32_t* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  uint32_t add = 0;
  for (int w = 0; w < warp; ++w) add += warp_tot[w];
  __syncthreads();
  return v + add;
}

// Selects the `want` best items (by unique 64-bit key) of n_per items per
// thread and writes their keys, in any order, to out[0..want). item(e, v, x, k)
// gives item e's validity, logit and key; m is the maximum valid logit.
// Pass 1 histograms the gap to m in 1/64-nat buckets; the buckets above the
// boundary bucket are taken whole in pass 2, which also collects the boundary
// bucket's items; those (normally a handful) are ranked by counting. Only a
// boundary bucket of more than kBoundary items (massive exact ties) falls back
// to a radix select over the items.
template <typename Item>
__device__ void select_top(Item item, const int n_per, uint32_t want, float m, unsigned long long* out,
                           SelectSmem& sm) {
  if (want == 0) return;  // uniform across the block
  for (int i = threadIdx.x; i < kBuckets; i += kThreads) sm.hist[i] = 0;
  if (threadIdx.x == 0) {
    sm.nb = 0;
    sm.pos = 0;
  }
  __syncthreads();
#pragma unroll 4
  for (int e = 0; e < n_per; ++e) {
    bool v;
    float x;
    unsigned long long k;
    item(e, v, x, k);
    if (v) atomicAdd(&sm.hist[bucket_of(m, x)], 1u);
  }
  __syncthreads();
  // boundary bucket: the first b whose cumulative count reaches `want`
  constexpr int kPer = kBuckets / kThreads;
  uint32_t loc = 0;
#pragma unroll
  for (int b = 0; b < kPer; ++b) loc += sm.hist[kPer * threadIdx.x + b];
  const uint32_t incl = block_incl_scan(loc, sm.warp_tot);
  uint32_t c = incl - loc;
  if (c < want && incl >= want) {
    for (int b = 0; b < kPer; ++b) {
      const uint32_t h = sm.hist[kPer * threadIdx.x + b];
      if (c + h >= want) {
        sm.bstar = kPer * threadIdx.x + b;
        sm.above = c;
        sm.cnt = h;
        break;
      }
      c += h;
    }
  }
  __syncthreads();
  const int bstar = sm.bstar;
  const uint32_t above = sm.above;
  const uint32_t need = want - above;
  const bool whole = sm.cnt == need;
  const bool small = sm.cnt <= static_cast<uint32_t>(kBoundary);
  // pass 2: buckets above the boundary (and the boundary when it is taken
  // whole) go straight to out, compacted per warp by ballot (any order);
  // boundary items go to the shared list
  const int lane = threadIdx.x & 31;
#pragma unroll 4
  for (int e = 0; e < n_per; ++e) {
    bool v;
    float x;
    unsigned long long k;
    item(e, v, x, k);
    const int b = v ? bucket_of(m, x) : kBuckets;
    const bool sel = b < bstar || (whole && b == bstar);
    const unsigned bal = __ballot_sync(0xffffffffu, sel);
    if (bal != 0u) {
      const int leader = __ffs(bal) - 1;
      uint32_t base = 0;
      if (lane == leader) base = atomicAdd(&sm.pos, static_cast<uint32_t>(__popc(bal)));
      base = __shfl_sync(0xffffffffu, base, leader);
      const uint32_t at = base + __popc(bal & ((1u << lane) - 1u));
      if (sel && GLANCE_IN_BOUNDS(at, want)) out[at] = k;
    }
    if (!sel && b == bstar && small) sm.bnd[atomicAdd(&sm.nb, 1u)] = k;
  }
  if (whole) return;  // uniform: `whole` is read from shared memory
  __syncthreads();
  if (small) {
    // rank of each boundary item among the boundary items (unique keys)
    const uint32_t nb = sm.nb;
    for (uint32_t i = threadIdx.x; i < nb; i += kThreads) {
      const unsigned long long k = sm.bnd[i];
      uint32_t rank = 0;
      for (uint32_t j = 0; j < nb; ++j) rank += sm.bnd[j] > k;
      if (rank < need) out[above + rank] = k;
    }
    return;
  }
  // fallback: radix select on the full keys inside the boundary bucket
  unsigned long long prefix = 0, mask = 0;
  uint32_t krem = need;
  for (int shift = 56; shift >= 0; shift -= 8) {
    sm.hist[threadIdx.x] = 0;
    __syncthreads();
#pragma unroll 2
    for (int e = 0; e < n_per; ++e) {
      bool v;
      float x;
      unsigned long long k;
      item(e, v, x, k);
      if (v && bucket_of(m, x) == bstar && (k & mask) == prefix)
        atomicAdd(&sm.hist[static_cast<uint32_t>(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    // thread t holds digit d = 255 - t; the scan gives the count of digits >= d
    const uint32_t d = 255u - threadIdx.x;
    const uint32_t hv = sm.hist[d];
    const uint32_t in2 = block_incl_scan(hv, sm.warp_tot);
    const uint32_t ex2 = in2 - hv;
    if (ex2 < krem && in2 >= krem) {
      sm.digit = d;
      sm.above2 = ex2;
      sm.cnt2 = hv;
    }
    __syncthreads();
    prefix |= static_cast<unsigned long long>(sm.digit) << shift;
    mask |= 0xFFull << shift;
    krem -= sm.above2;
    const bool done = sm.cnt2 == krem;
    __syncthreads();
    if (done) break;
  }
  uint32_t c2 = 0;
#pragma unroll 2
  for (int e = 0; e < n_per; ++e) {
    bool v;
    float x;
    unsigned long long k;
    item(e, v, x, k);
    c2 += v && bucket_of(m, x) == bstar && (k & mask) >= prefix;
  }
  uint32_t pos2 = above + block_incl_scan(c2, sm.warp_tot) - c2;
#pragma unroll 2
  for (int e = 0; e < n_per; ++e) {
    bool v;
    float x;
    unsigned long long k;
    item(e, v, x, k);
    if (v && bucket_of(m, x) == bstar && (k & mask) >= prefix) {
      if (GLANCE_IN_BOUNDS(pos2, want)) out[pos2] = k;
      ++pos2;
    }
  }
}

// -------------------------------------------------------------- tree search

__device__ __forceinline__ void set_rank(unsigned long long& hi, unsigned long long& lo, int j,
                                         uint32_t r) {
  if (j < 8) {
    const int sh = (7 - j) * 8;
    hi = (hi & ~(0xFFull << sh)) | (static_cast<unsigned long long>(r) << sh);
  } else {
    const int sh = (15 - j) * 8;
    lo = (lo & ~(0xFFull << sh)) | (static_cast<unsigned long long>(r) << sh);
  }
}
__device__ __forceinline__ uint32_t get_rank(unsigned long long hi, unsigned long long lo, int j) {
  return j < 8 ? static_cast<uint32_t>(hi >> ((7 - j) * 8)) & 0xFFu
               : static_cast<uint32_t>(lo >> ((15 - j) * 8)) & 0xFFu;
}

// (depth, hi, lo) lexicographic: the order among nodes of equal score
__device__ __forceinline__ bool tie_less(uint32_t da, unsigned long long ha, unsigned long long la,
                                         uint32_t db, unsigned long long hb, unsigned long long lb) {
  if (da != db) return da < db;
  if (ha != hb) return ha < hb;
  return la < lb;
}

// One popped node: 32 bytes, written with two 16-byte stores.
struct __align__(16) PopRec {
  float score;   // log plug-in score
  float pscore;  // parent's score (0 at depth 1)
  int dep;       // depth
  int par;       // parent's pop index, -1 at depth 1
  unsigned long long hi, lo;  // rank bytes of the path
};

struct TreeSmem {  // sizeof is a multiple of 16 (PopRec alignment)
  PopRec pop[kMaxN];
  int16_t p_pos[kMaxN];
  uint8_t rank[kMaxN];  // a pop's rank at its own depth (the search's record)
};

template <int kSlots>
__device__ __forceinline__ uint32_t get_reg(const uint32_t (&a)[kSlots], int i) {
  uint32_t v = 0;
#pragma unroll
  for (int t = 0; t < kSlots; ++t)
    if (t == i) v = a[t];
  return v;
}

// Packs the first n pops of request req (a prefix of the best-first order, so
// a prefix-closed set) into canonical rows 0..n; rows n+1..N are inactive:
// token -1, parent -1 (never a child, so the walk never reaches them), depth
// 0, pos_id T, score -inf, ancestor mask = the row itself.
__device__ void pack_rows(const BuildParams& p, const int* s_tok, TreeSmem& ts, const int req,
                          const int n, const bool have_pos) {
  const int N = p.N, K = p.K;
  // canonical position: 1 + number of nodes before it in (depth, rank vector)
  // (given in ts.p_pos when have_pos)
  const int T = p.t_len[req];
  const glance_tree& tree = p.tree[req];
  const int W = tree.mask_words;
  for (int kk = have_pos ? n : threadIdx.x; kk < n; kk += kThreads) {
    const uint32_t dk = ts.pop[kk].dep;
    const unsigned long long hk = ts.pop[kk].hi, lk = ts.pop[kk].lo;
    int pos = 1;
#pragma unroll 4
    for (int j = 0; j < n; ++j)
      pos += tie_less(ts.pop[j].dep, ts.pop[j].hi, ts.pop[j].lo, dk, hk, lk);
    ts.p_pos[kk] = static_cast<int16_t>(pos);
  }
  __syncthreads();
  for (int kk = threadIdx.x; kk <= N; kk += kThreads) {
    if (kk == N) {  // root row
      tree.token[0] = p.root_token[req];
      tree.parent[0] = -1;
      tree.depth[0] = 0;
      tree.pos_id[0] = T;
      tree.score[0] = 0.f;
      for (int w = 0; w < W; ++w) tree.anc[w] = (w == 0) ? 1ull : 0ull;
      continue;
    }
    if (kk >= n) {  // inactive row n + 1 + (kk - n)
      const int row = kk + 1;
      tree.token[row] = -1;
      tree.parent[row] = -1;
      tree.depth[row] = 0;
      tree.pos_id[row] = T;
      tree.score[row] = -INFINITY;
      for (int w = 0; w < W; ++w) tree.anc[row * W + w] = (w == (row >> 6)) ? (1ull << (row & 63)) : 0ull;
      continue;
    }
    const int row = ts.p_pos[kk];
    if (!GLANCE_IN_BOUNDS(row, N + 1)) continue;
    const int d = ts.pop[kk].dep;
    const uint32_t r = get_rank(ts.pop[kk].hi, ts.pop[kk].lo, d - 1);
    const int par = ts.pop[kk].par;
    tree.token[row] = s_tok[(d - 1) * K + r];
    tree.parent[row] = par < 0 ? 0 : ts.p_pos[par];
    tree.depth[row] = d;
    tree.pos_id[row] = T + d;
    tree.score[row] = ts.pop[kk].score;
    unsigned long long words[4] = {1ull, 0ull, 0ull, 0ull};
    words[row >> 6] |= 1ull << (row & 63);
    for (int u = par; u >= 0; u = ts.pop[u].par) {
      const int pr = ts.p_pos[u];
      words[pr >> 6] |= 1ull << (pr & 63);
    }
    for (int w = 0; w < W; ++w) tree.anc[row * W + w] = words[w];
  }
}

// Best-first search in one warp (the calling lanes are 0..31): pops N nodes
// into ts.pop / ts.rank in best-first order, then rebuilds their rank vectors.
template <int kSlots>
__device__ __noinline__ void search_warp(TreeSmem& ts, const float* s_logq, const int N, const int L,
                                         const int K) {
    // Lane-owned frontier slots (slot s = lane + 32 i), each a node held in
    // registers: its 32-bit score key (0 = empty), its parent's score, and
    // depth | rank << 8 | (parent pop + 1) << 16. A pop then needs no shared
    // memory: successor scores come from the node's own fields, and the
    // popped record (score, parent score, depth, parent, rank) is written for
    // later; the rank vectors are rebuilt from the parent links after the
    // search (and walked up on the rare exact-tie path).
    const int lane = threadIdx.x;
    uint32_t ko[kSlots], ki[kSlots];
    float kp[kSlots];
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      ko[i] = 0;
      ki[i] = 0;
      kp[i] = 0.f;
    }
    if (lane == 0) {
      ko[0] = ord_key(s_logq[0]);
      ki[0] = 1u;  // depth 1, rank 0, no parent
    }
    auto get_f = [&](const float (&a)[kSlots], int i) {
      float v = 0.f;
#pragma unroll
      for (int t2 = 0; t2 < kSlots; ++t2)
        if (t2 == i) v = a[t2];
      return v;
    };
    // rank vector of a node (depth d, rank r, parent pop par) from the records
    auto path_of = [&](int d, uint32_t r, int par, unsigned long long& hi, unsigned long long& lo) {
      hi = lo = 0ull;
      set_rank(hi, lo, d - 1, r);
      for (int v = par; v >= 0; v = ts.pop[v].par) set_rank(hi, lo, ts.pop[v].dep - 1, ts.rank[v]);
    };
    int cnt = 1;
    for (int k = 0; k < N; ++k) {
      uint32_t bo = 0;
      int bi = 0;
      bool dup = false;
#pragma unroll
      for (int i = 0; i < kSlots; ++i) {
        const uint32_t v = ko[i];
        if (v > bo) {
          bo = v;
          bi = i;
          dup = false;
        } else if (v == bo && v != 0) {
          dup = true;
        }
      }
      const uint32_t mmax = __reduce_max_sync(0xffffffffu, bo);
      // every lane prepares its best slot's successors while the maximum is in flight
      uint32_t info = get_reg<kSlots>(ki, bi);
      float ps = get_f(kp, bi);
      float c_score = 0.f, s_score = 0.f;
      {
        const int d = static_cast<int>(info & 0xFFu);
        const int r = static_cast<int>((info >> 8) & 0xFFu);
        const float sc = inv_ord_key(bo);
        if (bo != 0 && d < L) c_score = sc + s_logq[d * K];
        if (bo != 0 && r + 1 < K) s_score = ps + s_logq[(d - 1) * K + r + 1];
      }
      if (mmax == 0) {  // frontier exhausted: the host checks make this unreachable
        if (lane == 0) report(GLANCE_DEV_BAD_TREE);
        break;
      }
      const unsigned cand = __ballot_sync(0xffffffffu, bo == mmax);
      const bool slow = __popc(cand) > 1 || __ballot_sync(0xffffffffu, bo == mmax && dup) != 0;
      int ws;  // winning slot
      if (!slow) {
        const int win = __ffs(cand) - 1;
        ws = __shfl_sync(0xffffffffu, bi * 32 + lane, win);
        info = __shfl_sync(0xffffffffu, info, win);
        ps = __shfl_sync(0xffffffffu, ps, win);
        c_score = __shfl_sync(0xffffffffu, c_score, win);
        s_score = __shfl_sync(0xffffffffu, s_score, win);
      } else {
        // exact score tie: least (depth, rank vector) among slots with key mmax
        __syncwarp();  // the records written so far are visible to every lane
        int my = -1;
        uint32_t md = 0, mi = 0;
        float mp = 0.f;
        unsigned long long mh = 0, ml = 0;
#pragma unroll
        for (int i = 0; i < kSlots; ++i) {
          if (ko[i] == mmax) {
            const int d = static_cast<int>(ki[i] & 0xFFu);
            unsigned long long h, l;
            path_of(d, (ki[i] >> 8) & 0xFFu, static_cast<int>(ki[i] >> 16) - 1, h, l);
            if (my < 0 || tie_less(d, h, l, md, mh, ml)) {
              my = i * 32 + lane;
              md = d;
              mh = h;
              ml = l;
              mi = ki[i];
              mp = kp[i];
            }
          }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const int oy = __shfl_xor_sync(0xffffffffu, my, o);
          const uint32_t od = __shfl_xor_sync(0xffffffffu, md, o);
          const unsigned long long oh = __shfl_xor_sync(0xffffffffu, mh, o);
          const unsigned long long ol = __shfl_xor_sync(0xffffffffu, ml, o);
          const uint32_t oi = __shfl_xor_sync(0xffffffffu, mi, o);
          const float op = __shfl_xor_sync(0xffffffffu, mp, o);
          if (oy >= 0 && (my < 0 || tie_less(od, oh, ol, md, mh, ml))) {
            my = oy;
            md = od;
            mh = oh;
            ml = ol;
            mi = oi;
            mp = op;
          }
        }
        ws = my;
        info = mi;
        ps = mp;
        const int d = static_cast<int>(info & 0xFFu);
        const int r = static_cast<int>((info >> 8) & 0xFFu);
        const float sc = inv_ord_key(mmax);
        c_score = d < L ? sc + s_logq[d * K] : 0.f;
        s_score = r + 1 < K ? ps + s_logq[(d - 1) * K + r + 1] : 0.f;
      }
      const float score = inv_ord_key(mmax);
      const int d = static_cast<int>(info & 0xFFu);
      const uint32_t r = (info >> 8) & 0xFFu;
      const uint32_t par1 = info >> 16;  // parent pop + 1
      const bool has_child = d < L;
      const bool has_sib = static_cast<int>(r) + 1 < K;
      if (lane == 0) {
        uint4* dst = reinterpret_cast<uint4*>(&ts.pop[k]);
        dst[0] = make_uint4(__float_as_uint(score), __float_as_uint(ps), static_cast<uint32_t>(d),
                            static_cast<uint32_t>(static_cast<int>(par1) - 1));
        ts.rank[k] = static_cast<uint8_t>(r);
      }
      // the popped slot takes the child (else the sibling); a new slot takes
      // the sibling when both exist (predicated, no divergence)
      const uint32_t child_info = static_cast<uint32_t>(d + 1) | (static_cast<uint32_t>(k + 1) << 16);
      const uint32_t sib_info = static_cast<uint32_t>(d) | ((r + 1) << 8) | (par1 << 16);
      const uint32_t k_ws = has_child ? ord_key(c_score) : (has_sib ? ord_key(s_score) : 0u);
      const uint32_t i_ws = has_child ? child_info : sib_info;
      const float p_ws = has_child ? score : ps;
      const bool both = has_child && has_sib;
      const int ns = both ? cnt : -1;
      cnt += both ? 1 : 0;
      const uint32_t k_ns = ord_key(s_score);
#pragma unroll
      for (int i = 0; i < kSlots; ++i) {
        const int slot = i * 32 + lane;
        ko[i] = slot == ws ? k_ws : (slot == ns ? k_ns : ko[i]);
        ki[i] = slot == ws ? i_ws : (slot == ns ? sib_info : ki[i]);
        kp[i] = slot == ws ? p_ws : (slot == ns ? ps : kp[i]);
      }
    }
    __syncwarp();
    // rank vectors of the pops from their parent links (depth <= 16 steps)
    for (int kk = lane; kk < N; kk += 32) {
      unsigned long long h, l;
      path_of(ts.pop[kk].dep, ts.rank[kk], ts.pop[kk].par, h, l);
      ts.pop[kk].hi = h;
      ts.pop[kk].lo = l;
    }
}

// ------------------------------------------------- threshold level expansion
//
// The best-first order pops the nodes in the total order (score desc, then
// depth, then rank vector): a node's parent and its left sibling both precede
// it, so the N pops are exactly the N first nodes of that order, and every
// one of them scores at least the N-th score tau. The expansion below builds
// a superset of them without popping one node at a time:
//  - t starts as a lower bound on tau: the N-th score of the one-deviation
//    nodes (0, .., 0, r), which are N real nodes;
//  - depth by depth, every node with score >= t gets all its children with
//    score >= t (a prefix of its rank list: the log q rows are sorted), so
//    after the last depth the set holds every node scoring >= t;
//  - t is raised during the expansion to the score below which fewer than N
//    generated nodes lie (a score histogram; the value stays a lower bound
//    on tau because it counts real nodes);
//  - the nodes scoring >= the final t are ranked by the total order and the
//    N first become the pops, in best-first order.
// Scores are computed exactly as the search adds them (parent score plus the
// child's log q, fp32), so the pops are identical. If the set would outgrow
// its capacity the expansion gives up and the one-warp search runs instead.
constexpr int kLvCap = 2048;  // generated nodes
constexpr int kLvBuckets = 256;
constexpr int kLvDirect = 8;  // children a parent writes itself
constexpr int kLvMaxCand = 512;  // nodes ranked at the end

struct LevelSmem {
  float sc[kLvCap];        // score
  uint32_t meta[kLvCap];   // depth | rank << 5 | (parent + 1) << 13
  float csc[kLvCap];       // candidates' scores (read as float4)
  uint32_t off[kLvCap + 1];
  uint16_t cand[kLvCap];
  uint16_t pop_of[kLvCap];
  unsigned long long chi[kLvMaxCand], clo[kLvMaxCand];  // candidates' rank vectors
  uint8_t cdep[kLvMaxCand];
  uint32_t hcnt[kLvBuckets];
  float P[kMaxL + 1];      // chain scores: P[d] = score of 0^d
  uint32_t warp_tot[kThreads / 32];
  float t;
  int m;
};
static_assert(offsetof(LevelSmem, csc) % 16 == 0, "candidate scores are read as float4");
static_assert(sizeof(TreeSmem) % 16 == 0, "LevelSmem follows TreeSmem 16-byte aligned");

__device__ __forceinline__ int lv_dep(uint32_t m) { return static_cast<int>(m & 31u); }
__device__ __forceinline__ uint32_t lv_rank(uint32_t m) { return (m >> 5) & 0xFFu; }
__device__ __forceinline__ int lv_par(uint32_t m) { return static_cast<int>(m >> 13) - 1; }

// Score histogram from the best score s_max down: bucket b holds scores in
// (s_max - (b+1) w, s_max - b w]; monotone in the score.
struct LvBuckets {
  float s_max, inv_w, w;
  __device__ int operator()(float s) const {
    const float x = (s_max - s) * inv_w;
    if (!(x < static_cast<float>(kLvBuckets - 1))) return kLvBuckets - 1;
    return x > 0.f ? static_cast<int>(x) : 0;
  }
};

// Threads 0..31: the bucket b* where the count from the top reaches N. Every
// counted node scores above s_max - (b* + 1) w up to rounding, which the
// bucket width (at least 2^-18 of the largest magnitude) keeps far below one
// bucket, so t = s_max - (b* + 2) w has N real nodes at or above it. Writes
// max(t_cur, t) to S.t; the caller syncs before reading it.
__device__ void lv_propose(LevelSmem& S, const LvBuckets& bk, int N, float t_cur) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  constexpr int per = kLvBuckets / 32;
  uint32_t c[per], local = 0;
#pragma unroll
  for (int i = 0; i < per; ++i) {
    c[i] = S.hcnt[lane * per + i];
    local += c[i];
  }
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  uint32_t run = incl - local;
  int bs = -1;
#pragma unroll
  for (int i = 0; i < per; ++i) {
    if (bs < 0 && run + c[i] >= static_cast<uint32_t>(N)) bs = lane * per + i;
    run += c[i];
  }
  const unsigned hit = __ballot_sync(0xffffffffu, bs >= 0);
  const int b = __shfl_sync(0xffffffffu, bs, hit ? __ffs(hit) - 1 : 0);
  if (lane == 0) {
    float t = t_cur;
    if (hit && b < kLvBuckets - 2) t = fmaxf(t_cur, bk.s_max - static_cast<float>(b + 2) * bk.w);
    S.t = t;
  }
}

// Number of ranks r < K with s + row[r] >= t (a prefix: the row is sorted
// descending and fp32 addition is monotone): galloping, then bisection.
__device__ __forceinline__ int lv_prefix_count(float s, const float* row, int K, float t) {
  if (!(s + row[0] >= t)) return 0;
  int lo = 1, step = 1;  // ranks below lo pass
  while (lo < K && s + row[min(lo + step - 1, K - 1)] >= t) {
    lo = min(lo + step, K);
    step <<= 1;
  }
  int hi = min(lo + step - 1, K);  // the first failing rank is in [lo, hi]
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s + row[mid] >= t) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// (depth, rank vector) of a generated node, from its parent links
__device__ __forceinline__ void lv_path(const LevelSmem& S, int u, uint32_t& dep,
                                        unsigned long long& hi, unsigned long long& lo) {
  hi = lo = 0ull;
  const uint32_t m0 = S.meta[u];
  dep = static_cast<uint32_t>(lv_dep(m0));
  for (int v = u; v >= 0;) {
    const uint32_t m = S.meta[v];
    set_rank(hi, lo, lv_dep(m) - 1, lv_rank(m));
    v = lv_par(m);
  }
}

// All threads of the CTA. Returns false (uniformly) when the node set would
// outgrow kLvCap or more than kLvMaxCand nodes tie into the final bound;
// ts.pop is then untouched.
__device__ bool expand_levels(TreeSmem& ts, LevelSmem& S, const float* s_logq, const int N,
                              const int L, const int K) {
  const int tid = threadIdx.x;
  if (K < N) return false;  // V < N: the depth-1 row cannot seed the bound
  const float t_lo = s_logq[N - 1], s_max = s_logq[0];
  LvBuckets bk;
  bk.s_max = s_max;
  bk.w = fmaxf((s_max - t_lo) / static_cast<float>(kLvBuckets), fabsf(t_lo) * 0x1p-18f);
  bk.inv_w = bk.w > 0.f ? 1.f / bk.w : 0.f;
  for (int i = tid; i < kLvBuckets; i += kThreads) S.hcnt[i] = 0u;
  if (tid == 0) {
    float v[kMaxL];
#pragma unroll
    for (int d = 0; d < kMaxL; ++d) v[d] = d < L ? s_logq[d * K] : 0.f;
    float pd = 0.f;
    int deep = 0;  // deepest rank-0 chain scoring >= t_lo
    S.P[0] = 0.f;
#pragma unroll
    for (int d = 0; d < kMaxL; ++d) {
      pd = pd + v[d];
      S.P[d + 1] = pd;
      if (d < L && pd >= t_lo) deep = d + 1;
    }
    S.m = deep;
  }
  __syncthreads();
  // The one-deviation bound pays for its histogram only on deep trees: with
  // the rank-0 chain at most 3 deep above t_lo, t_lo itself leaves few nodes
  // past the N best.
  float t = t_lo;
  if (S.m > 3) {
    // one-deviation nodes (0^(d-1), r); consecutive threads take different rows
    for (int i = tid; i < L * K; i += kThreads) {
      const int d = i % L, r = i / L;
      const float f = S.P[d] + s_logq[d * K + r];
      if (f >= t_lo) atomicAdd(&S.hcnt[bk(f)], 1u);
    }
    __syncthreads();
    lv_propose(S, bk, N, t_lo);
    __syncthreads();
    t = S.t;
    for (int i = tid; i < kLvBuckets; i += kThreads) S.hcnt[i] = 0u;
  }
  // depth 1: the ranks with log q >= t
  int total;
  {
    int a = 0, b = K;
    while (a < b) {
      const int mid = (a + b) >> 1;
      if (s_logq[mid] >= t) a = mid + 1;
      else b = mid;
    }
    total = a;
  }
  __syncthreads();
  for (int r = tid; r < total; r += kThreads) {
    const float s = s_logq[r];
    S.sc[r] = s;
    S.meta[r] = 1u | (static_cast<uint32_t>(r) << 5);
    atomicAdd(&S.hcnt[bk(s)], 1u);
  }
  __syncthreads();
  int lb = 0, le = total, last_raise = 0;
  for (int d = 2; d <= L && le > lb; ++d) {
    if (total > 2 * N && total - last_raise >= N / 2) {
      lv_propose(S, bk, N, t);
      __syncthreads();
      t = S.t;
      last_raise = total;
    }
    const float* row = s_logq + (d - 1) * K;
    const int n = le - lb;
    const int q = (n + kThreads - 1) / kThreads;  // nodes per thread, <= kLvCap / kThreads
    const int u0 = lb + tid * q, u1 = min(u0 + q, le);
    uint32_t excl = 0, tot_new = 0;
    for (int attempt = 0;; ++attempt) {
      // child counts, kept in off[] until the offsets replace them
      uint32_t local = 0;
#pragma unroll 1
      for (int u = u0; u < u1; ++u) {
        const float s = S.sc[u];
        const uint32_t c = s >= t ? static_cast<uint32_t>(lv_prefix_count(s, row, K, t)) : 0u;
        S.off[u - lb] = c;
        local += c;
      }
      const uint32_t incl = block_incl_scan(local, S.warp_tot);
      excl = incl - local;
      if (tid == kThreads - 1) S.off[kLvCap] = incl;
      __syncthreads();
      tot_new = S.off[kLvCap];
      if (total + static_cast<int>(tot_new) <= kLvCap) break;
      if (attempt > 0 || total < N) return false;
      lv_propose(S, bk, N, t);
      __syncthreads();
      t = S.t;
      last_raise = total;
    }
    // children: each parent writes its first kLvDirect itself
    bool big = false;
    {
      uint32_t o = excl;
#pragma unroll 1
      for (int u = u0; u < u1; ++u) {
        const int nc = static_cast<int>(S.off[u - lb]);
        S.off[u - lb] = o;
        big |= nc > kLvDirect;
        const float s = S.sc[u];
#pragma unroll 1
        for (int c = 0; c < min(nc, kLvDirect); ++c) {
          const int idx = total + static_cast<int>(o) + c;
          const float sc = s + row[c];
          S.sc[idx] = sc;
          S.meta[idx] = static_cast<uint32_t>(d) | (static_cast<uint32_t>(c) << 5) |
                        (static_cast<uint32_t>(u + 1) << 13);
          atomicAdd(&S.hcnt[bk(sc)], 1u);
        }
        o += static_cast<uint32_t>(nc);
      }
    }
    if (__syncthreads_or(big)) {
      // the remaining children, spread over the CTA; a child's parent is the
      // last node of the depth whose offset is <= the child's slot
      for (int c = tid; c < static_cast<int>(tot_new); c += kThreads) {
        int a = 0, b = n - 1;
        while (a < b) {
          const int mid = (a + b + 1) >> 1;
          if (S.off[mid] <= static_cast<uint32_t>(c)) a = mid;
          else b = mid - 1;
        }
        const int j = c - static_cast<int>(S.off[a]);
        if (j < kLvDirect) continue;
        const int u = lb + a;
        const float sc = S.sc[u] + row[j];
        const int idx = total + c;
        S.sc[idx] = sc;
        S.meta[idx] = static_cast<uint32_t>(d) | (static_cast<uint32_t>(j) << 5) |
                      (static_cast<uint32_t>(u + 1) << 13);
        atomicAdd(&S.hcnt[bk(sc)], 1u);
      }
      __syncthreads();
    }
    lb = total;
    total += static_cast<int>(tot_new);
    le = total;
  }
  // candidates: the nodes scoring >= the final bound
  lv_propose(S, bk, N, t);
  __syncthreads();
  t = S.t;
  {
    const int q = (total + kThreads - 1) / kThreads;
    uint32_t local = 0;
    for (int j = 0; j < q; ++j) {
      const int u = tid * q + j;
      if (u < total && S.sc[u] >= t) ++local;
    }
    const uint32_t incl = block_incl_scan(local, S.warp_tot);
    uint32_t o = incl - local;
    for (int j = 0; j < q; ++j) {
      const int u = tid * q + j;
      if (u < total && S.sc[u] >= t) {
        S.cand[o] = static_cast<uint16_t>(u);
        S.csc[o] = S.sc[u];
        ++o;
      }
    }
    if (tid == kThreads - 1) S.m = static_cast<int>(incl);
  }
  __syncthreads();
  const int M = S.m;
  if (M > kLvMaxCand) return false;
  for (int i = tid; i < M; i += kThreads) {
    uint32_t dep;
    lv_path(S, S.cand[i], dep, S.chi[i], S.clo[i]);
    S.cdep[i] = static_cast<uint8_t>(dep);
  }
  for (int u = tid; u < total; u += kThreads) S.pop_of[u] = 0xFFFFu;  // not a pop
  __syncthreads();
  // rank of every candidate in the total order, by counting: the scores
  // first (four at a time), the (depth, rank vector) keys only among equal
  // scores
  for (int i = tid; i < M; i += kThreads) {
    const float su = S.csc[i];
    int above = 0, eq = 0, j = 0;
#pragma unroll 4
    for (; j + 4 <= M; j += 4) {
      const float4 v = *reinterpret_cast<const float4*>(&S.csc[j]);
      above += (v.x > su) + (v.y > su) + (v.z > su) + (v.w > su);
      eq += (v.x == su) + (v.y == su) + (v.z == su) + (v.w == su);
    }
    for (; j < M; ++j) {
      const float v = S.csc[j];
      above += v > su;
      eq += v == su;
    }
    int rank = above;
    const int u = S.cand[i];
    if (eq > 1) {
      const uint32_t du = S.cdep[i];
      const unsigned long long hu = S.chi[i], lu = S.clo[i];
      for (int k = 0; k < M; ++k) {
        if (S.csc[k] != su || k == i) continue;
        rank += tie_less(S.cdep[k], S.chi[k], S.clo[k], du, hu, lu);
      }
    }
    if (rank < N) {
      S.off[rank] = static_cast<uint32_t>(i);  // pop rank -> candidate
      S.pop_of[u] = static_cast<uint16_t>(rank);
    }
  }
  __syncthreads();
  // the pops, in best-first order; a pop's parent pops before it
  for (int k = tid; k < N; k += kThreads) {
    const int i = static_cast<int>(S.off[k]);
    const int u = S.cand[i];
    const int par = lv_par(S.meta[u]);
    PopRec pr;
    pr.score = S.sc[u];
    pr.pscore = par >= 0 ? S.sc[par] : 0.f;
    pr.dep = static_cast<int>(S.cdep[i]);
    pr.par = par >= 0 ? static_cast<int>(S.pop_of[par]) : -1;
    pr.hi = S.chi[i];
    pr.lo = S.clo[i];
    ts.pop[k] = pr;
  }
  // Canonical positions. Nodes are stored depth by depth, and a depth's nodes
  // follow their parents' order and then their own rank, so the storage order
  // is the (depth, rank vector) order; a pop's row is 1 + the pops stored
  // before it.
  {
    const int q = (total + kThreads - 1) / kThreads;
    const int u0 = tid * q, u1 = min(u0 + q, total);
    uint32_t local = 0;
    for (int u = u0; u < u1; ++u) local += S.pop_of[u] != 0xFFFFu;
    uint32_t at = block_incl_scan(local, S.warp_tot) - local;
    for (int u = u0; u < u1; ++u) {
      const uint32_t k = S.pop_of[u];
      if (k != 0xFFFFu) ts.p_pos[k] = static_cast<int16_t>(1 + at++);
    }
  }
  __syncthreads();
  return true;
}

// Which search is cheaper, packing included. The expansion costs about
// 8000 + 2000 D cycles for D depths and hands the canonical rows over
// (~1400 cycles); the one-warp search costs about 600 cycles per pop and its
// packing about 4000 + 100 N (all measured on GB300). D is bounded by the
// deepest chain 0^d scoring at least the N-th depth-1 score, the expansion's
// loosest bound. All threads; uniform result.
__device__ bool use_levels(LevelSmem& S, const float* s_logq, const int N, const int L,
                           const int K) {
  if (K < N) return false;
  if (threadIdx.x == 0) {
    const float t_lo = s_logq[N - 1];
    float pd = 0.f;
    int D = 0;
    for (int d = 0; d < L; ++d) {
      pd = pd + s_logq[d * K];
      if (pd >= t_lo) D = d + 1;
    }
    S.m = 8000 + 2000 * D + 1400 < 600 * N + 4000 + 100 * N ? 1 : 0;
  }
  __syncthreads();
  const bool r = S.m != 0;
  __syncthreads();
  return r;
}

__device__ void tree_phase(const BuildParams& p, unsigned char* dyn, const int req) {
  // dynamic smem: logq [L][K] floats, tok [L][K] ints, TreeSmem, LevelSmem
  float* s_logq = reinterpret_cast<float*>(dyn);
  int* s_tok = reinterpret_cast<int*>(dyn + sizeof(float) * p.L * p.K);
  TreeSmem& ts = *reinterpret_cast<TreeSmem*>(
      dyn + 16 * ((sizeof(float) * 2 * p.L * p.K + 15) / 16));
  const int LK = p.L * p.K;
  const size_t lk0 = static_cast<size_t>(req) * LK;
  for (int i = threadIdx.x; i < LK; i += kThreads) {
    s_logq[i] = __ldcg(p.top_logq + lk0 + i);
    s_tok[i] = __ldcg(p.top_tok + lk0 + i);
  }
  __syncthreads();
  const int N = p.N, L = p.L, K = p.K;

  LevelSmem& ls = *reinterpret_cast<LevelSmem*>(reinterpret_cast<unsigned char*>(&ts) + sizeof(TreeSmem));
  bool have_pos = use_levels(ls, s_logq, N, L, K) && expand_levels(ts, ls, s_logq, N, L, K);
  if (!have_pos) {
    if (threadIdx.x < 32) {
      // frontier capacity 32 x slots per lane >= N + 1: fewer slots, shorter pops
      if (N < 64)
        search_warp<2>(ts, s_logq, N, L, K);
      else if (N < 128)
        search_warp<4>(ts, s_logq, N, L, K);
      else
        search_warp<8>(ts, s_logq, N, L, K);
    }
    __syncthreads();
  }

  if (p.search_only) {
    // shared budget: hand the pops (in best-first order) to the pack kernel
    PopRec* dst = static_cast<PopRec*>(p.pops_out) + static_cast<size_t>(req) * kMaxN;
    for (int kk = threadIdx.x; kk < N; kk += kThreads) dst[kk] = ts.pop[kk];
    return;
  }
  pack_rows(p, s_tok, ts, req, N, have_pos);
}

// ------------------------------------------------------------------- kernel

template <bool kBF16, bool kVec>
__global__ void __launch_bounds__(kThreads, 2) build_tree_kernel(const __grid_constant__ BuildParams p) {
  extern __shared__ __align__(16) unsigned char dyn[];
  __shared__ SelectSmem sm;
  __shared__ float red_d[kThreads / 32];
  __shared__ float red_f[kThreads / 32];
  __shared__ uint32_t s_ticket;
  __shared__ unsigned long long sel[256];
  __shared__ float s_lse;

  const int req = blockIdx.y;
  const int row = req * p.L + blockIdx.x / p.C;  // global row
  const int chunk = blockIdx.x % p.C;
  uint32_t* const tickets = p.tickets + req * kTicketsPerReq;
  const int orow = blockIdx.x / p.C;               // offset row within the request
  const int base = chunk * kChunk;
  const int n_valid = min(kChunk, p.V - base);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // The next kernel (tree attention) may start its prologue on SMs this grid
  // frees: it reads nothing this kernel writes before its own dependency wait.
  pdl_launch_dependents();

  // ---- 1. load the chunk into registers (ids: see id_of below)
  float x[kPerThread];
  if (kVec) {
    // vector v = t + 256 * q holds ids base + 4v .. 4v+3
#pragma unroll
    for (int q = 0; q < kPerThread / 4; ++q) {
      const int v = threadIdx.x + kThreads * q;
      const int id0 = base + 4 * v;
      if (4 * v < n_valid &&  // n_valid % 4 == 0 when vectorised
          GLANCE_IN_BOUNDS(static_cast<size_t>(row) * p.V + id0 + 3, static_cast<size_t>(p.B) * p.L * p.V)) {
        if (kBF16) {
          const uint2 raw = *reinterpret_cast<const uint2*>(
              static_cast<const uint16_t*>(p.logits) + static_cast<size_t>(row) * p.V + id0);
          x[4 * q + 0] = bf16_to_f32(raw.x & 0xFFFFu);
          x[4 * q + 1] = bf16_to_f32(raw.x >> 16);
          x[4 * q + 2] = bf16_to_f32(raw.y & 0xFFFFu);
          x[4 * q + 3] = bf16_to_f32(raw.y >> 16);
        } else {
          const float4 f = *reinterpret_cast<const float4*>(
              static_cast<const float*>(p.logits) + static_cast<size_t>(row) * p.V + id0);
          x[4 * q + 0] = f.x;
          x[4 * q + 1] = f.y;
          x[4 * q + 2] = f.z;
          x[4 * q + 3] = f.w;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) x[4 * q + c] = -INFINITY;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int local = threadIdx.x + kThreads * e;
      const size_t gi = static_cast<size_t>(row) * p.V + base + local;
      if (local < n_valid && GLANCE_IN_BOUNDS(gi, static_cast<size_t>(p.B) * p.L * p.V)) {
        x[e] = kBF16 ? bf16_to_f32(static_cast<const uint16_t*>(p.logits)[gi])
                     : static_cast<const float*>(p.logits)[gi];
      } else {
        x[e] = -INFINITY;
      }
    }
  }
  auto id_of = [&](int e) -> int {
    if (kVec) return base + 4 * (threadIdx.x + kThreads * (e / 4)) + (e % 4);
    return base + threadIdx.x + kThreads * e;
  };
  auto valid_of = [&](int e) -> bool { return id_of(e) - base < n_valid; };

  // ---- chunk max and sum of exp
  float m = -INFINITY;
  bool bad = false;
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    if (valid_of(e)) {
      bad |= !isfinite(x[e]);
      m = fmaxf(m, x[e]);
    }
  }
  if (bad) report(GLANCE_DEV_NONFINITE_LOGITS);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red_f[warp] = m;
  __syncthreads();
  m = red_f[0];
  for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, red_f[w]);
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < kPerThread; ++e)
    if (valid_of(e)) s += expf(x[e] - m);
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) red_d[warp] = s;

  // ---- chunk top-K. The logits move to shared memory (item e of thread t at
  // e * 256 + t, conflict-free) so the selection passes re-read them instead
  // of holding 32 values, keys and buckets live in registers.
  float* xs = reinterpret_cast<float*>(dyn);
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) xs[e * kThreads + threadIdx.x] = x[e];
  const int kc = min(p.K, n_valid);
  unsigned long long* my_cand = p.cand + (static_cast<size_t>(row) * p.C + chunk) * p.K;
  select_top(
      [&](int e, bool& v, float& xv, unsigned long long& k) {
        v = valid_of(e);
        xv = xs[e * kThreads + threadIdx.x];
        k = make_key(xv, static_cast<uint32_t>(id_of(e)));
      },
      kPerThread, static_cast<uint32_t>(kc), m, my_cand, sm);
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) tot += red_d[w];
    if (GLANCE_IN_BOUNDS(row * p.C + chunk, p.B * p.L * p.C)) {
      p.chunk_m[row * p.C + chunk] = m;
      p.chunk_s[row * p.C + chunk] = tot;
    }
  }

  // ---- 2. last CTA of this row merges
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_ticket = atomicAdd(&tickets[orow], 1u);
  __syncthreads();
  if (s_ticket != static_cast<uint32_t>(p.C - 1)) return;
  __threadfence();
  if (threadIdx.x == 0) tickets[orow] = 0;  // ready for the next call

  // The row's candidate keys move to shared memory first (one coalesced
  // pass; the selection passes then read them there): flat index f = c * K
  // + i, zero where i >= min(K, chunk size).
  unsigned long long* s_cand = reinterpret_cast<unsigned long long*>(dyn);
  const unsigned long long* row_cand = p.cand + static_cast<size_t>(row) * p.C * p.K;
  const int n_cand = p.C * p.K;
  for (int f = threadIdx.x; f < n_cand; f += kThreads) {
    const int c = f / p.K, i = f - c * p.K;
    s_cand[f] = i < min(p.K, min(kChunk, p.V - c * kChunk)) ? __ldcg(row_cand + f) : 0ull;
  }
  // row log-sum-exp and max from the chunks' (max, sum) pairs: every sum is
  // relative to its chunk's max, so the fp32 terms are at most 8192 each
  if (warp == 0) {
    float cm[2], cs[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {  // C <= 64
      const int c = lane + 32 * q;
      cm[q] = c < p.C ? __ldcg(p.chunk_m + row * p.C + c) : -INFINITY;
      cs[q] = c < p.C ? __ldcg(p.chunk_s + row * p.C + c) : 0.f;
    }
    float M = fmaxf(cm[0], cm[1]);
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float S = cs[0] * expf(cm[0] - M) + cs[1] * expf(cm[1] - M);
#pragma unroll
    for (int o = 16; o; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    if (lane == 0) {
      s_lse = M + logf(S);
      red_f[0] = M;
    }
  }
  __syncthreads();
  const float row_max = red_f[0];
  select_top(
      [&](int e, bool& v, float& xv, unsigned long long& k) {
        const int f = threadIdx.x + kThreads * e;
        k = f < n_cand ? s_cand[f] : 0ull;
        v = k != 0ull;
        xv = inv_ord_key(static_cast<uint32_t>(k >> 32));
      },
      (n_cand + kThreads - 1) / kThreads, static_cast<uint32_t>(p.K), row_max, sel, sm);
  __syncthreads();
  // rank of each selected key among the K (keys are unique), by counting
  if (threadIdx.x < p.K) {
    const unsigned long long k = sel[threadIdx.x];
    int rank = 0;
#pragma unroll 4
    for (int j = 0; j < p.K; ++j) rank += sel[j] > k;
    const float xv = inv_ord_key(static_cast<uint32_t>(k >> 32));
    const uint32_t id = 0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull);
    if (GLANCE_IN_BOUNDS(row * p.K + rank, p.B * p.L * p.K)) {
      p.top_tok[row * p.K + rank] = static_cast<int32_t>(id);
      p.top_logq[row * p.K + rank] = xv - s_lse;
    }
  }

  // ---- 3. last row-merger builds the tree
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_ticket = atomicAdd(&tickets[kMaxL], 1u);
  __syncthreads();
  if (s_ticket != static_cast<uint32_t>(p.L - 1)) return;
  __threadfence();
  if (threadIdx.x == 0) tickets[kMaxL] = 0;
  tree_phase(p, dyn, req);
}

// Shared budget, second launch: one CTA per request. Every CTA ranks its own
// request's pops (best-first order) among all B x N pops by weighted key
// log w_r + score (desc; ties to the lower request, then the request's own
// order), keeps those ranked below N_total (a prefix of its order), and packs
// them. log w_r = log(p_m (1 - p_m^L)), logit p_m = b0 - b1 H_r, from the
// root entropies when given, else 0.
struct SharedArgs {
  int n_total;
  const float* root_entropy;  // [B] or null
  float b0, b1;
  int32_t* n_active;          // [B]
};

__global__ void __launch_bounds__(kThreads) shared_pack_kernel(const __grid_constant__ BuildParams p,
                                                                const SharedArgs sa) {
  extern __shared__ __align__(16) unsigned char dyn[];
  TreeSmem& ts = *reinterpret_cast<TreeSmem*>(dyn);
  int* s_tok = reinterpret_cast<int*>(dyn + sizeof(TreeSmem));
  float* keys = reinterpret_cast<float*>(s_tok + p.L * p.K);  // [B][N]
  __shared__ float s_logw[kMaxB];
  __shared__ int s_cnt;
  const int req = blockIdx.x;
  const int N = p.N, B = p.B;
  if (threadIdx.x < B) {
    float lw = 0.f;
    if (sa.root_entropy) {
      const float H = sa.root_entropy[threadIdx.x];
      const float pm = 1.f / (1.f + expf(-(sa.b0 - sa.b1 * H)));
      lw = logf(pm) + log1pf(-powf(pm, static_cast<float>(p.L)));
    }
    s_logw[threadIdx.x] = lw;
  }
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  const PopRec* pops = static_cast<const PopRec*>(p.pops_out);
  for (int f = threadIdx.x; f < B * N; f += kThreads) {
    const int r = f / N, i = f - r * N;
    keys[f] = s_logw[r] + pops[static_cast<size_t>(r) * kMaxN + i].score;
  }
  for (int i = threadIdx.x; i < N; i += kThreads) ts.pop[i] = pops[static_cast<size_t>(req) * kMaxN + i];
  for (int i = threadIdx.x; i < p.L * p.K; i += kThreads)
    s_tok[i] = p.top_tok[static_cast<size_t>(req) * p.L * p.K + i];
  __syncthreads();
  int mine = 0;
  for (int i = threadIdx.x; i < N; i += kThreads) {
    const float k = keys[req * N + i];
    int rank = i;
    for (int r = 0; r < B; ++r) {
      if (r == req) continue;
      // entries of list r ahead of k form a prefix (the list is non-increasing)
      const float* lst = keys + r * N;
      int lo = 0, hi = N;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const bool ahead = r < req ? lst[mid] >= k : lst[mid] > k;
        if (ahead)
          lo = mid + 1;
        else
          hi = mid;
      }
      rank += lo;
    }
    mine += rank < sa.n_total ? 1 : 0;
  }
  atomicAdd(&s_cnt, mine);
  __syncthreads();
  const int n = s_cnt;
  if (threadIdx.x == 0) sa.n_active[req] = n;
  pack_rows(p, s_tok, ts, req, n, false);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t tickets, chunk_m, chunk_s, cand, top_tok, top_logq, total;
};

WsLayout ws_layout(int B, int L, int V, int N) {
  const int K = N < V ? N : V;
  const int C = (V + kChunk - 1) / kChunk;
  const size_t rows = static_cast<size_t>(B) * L;
  WsLayout w;
  size_t o = 0;
  w.tickets = o;
  o = align_up(o + sizeof(uint32_t) * kTicketsPerReq * B, 256);
  w.chunk_m = o;
  o = align_up(o + sizeof(float) * rows * C, 256);
  w.chunk_s = o;
  o = align_up(o + sizeof(float) * rows * C, 256);
  w.cand = o;
  o = align_up(o + sizeof(unsigned long long) * rows * C * K, 256);
  w.top_tok = o;
  o = align_up(o + sizeof(int32_t) * rows * K, 256);
  w.top_logq = o;
  o = align_up(o + sizeof(float) * rows * K, 256);
  w.total = o;
  return w;
}

bool sizes_ok(int L, int V, int N) {
  if (L < 1 || L > kMaxL || V < 2 || N < 1 || N > kMaxN) return false;
  if (V > (1 << 18)) return false;
  const int K = N < V ? N : V;
  const int C = (V + kChunk - 1) / kChunk;
  if (static_cast<long long>(C) * K > kChunk) return false;
  // N must not exceed the number of strings of length <= L over V tokens
  long long total = 0, pw = 1;
  for (int d = 1; d <= L && total < N; ++d) {
    pw *= V;
    total += pw;
    if (pw > (1ll << 40)) total = 1ll << 40;
  }
  return total >= N;
}

glance_status launch_build(const char* who, const void* draft_logits, glance_dtype dtype, int B,
                           int L, int V, int N, const int32_t* root_token, const int32_t* t_len,
                           const glance_tree* trees, void* workspace, size_t workspace_bytes,
                           void* stream, const SharedArgs* shared = nullptr) {
  using glance::fail;
  if (!draft_logits || !root_token || !t_len || !trees || !workspace)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: null pointer argument", who);
  if (B < 1 || B > kMaxB)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: need 1 <= B <= %d (got %d)", who, kMaxB, B);
  if (dtype != GLANCE_F32 && dtype != GLANCE_BF16)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: dtype must be F32 or BF16", who);
  if (!sizes_ok(L, V, N))
    return fail(GLANCE_ERR_INVALID_ARG,
                "%s: need 1<=L<=16, 2<=V<=262144, 1<=N<=255, N <= #strings, "
                "ceil(V/8192)*min(N,V) <= 8192 (got L=%d V=%d N=%d)",
                who, L, V, N);
  for (int r = 0; r < B; ++r) {
    const glance_tree* tree = trees + r;
    if (tree->n != N || tree->L != L || tree->mask_words != (N + 1 + 63) / 64)
      return fail(GLANCE_ERR_INVALID_ARG,
                  "%s: tree %d sized for n=%d L=%d mask_words=%d, call has N=%d L=%d "
                  "(mask_words must be %d)",
                  who, r, tree->n, tree->L, tree->mask_words, N, L, (N + 64) / 64);
    if (!tree->token || !tree->parent || !tree->depth || !tree->pos_id || !tree->score ||
        !tree->anc)
      return fail(GLANCE_ERR_INVALID_ARG, "%s: null array in tree %d", who, r);
  }
  const WsLayout w = ws_layout(B, L, V, N);
  const size_t pops_at = w.total;  // shared budget: the pops after the regular layout
  const size_t need = shared ? pops_at + sizeof(PopRec) * kMaxN * B : w.total;
  if (workspace_bytes < need)
    return fail(GLANCE_ERR_CAPACITY, "%s: workspace %zu bytes < %zu needed", who,
                workspace_bytes, need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);

  BuildParams p;
  p.logits = draft_logits;
  p.is_bf16 = dtype == GLANCE_BF16;
  p.B = B;
  p.L = L;
  p.V = V;
  p.N = N;
  p.K = N < V ? N : V;
  p.C = (V + kChunk - 1) / kChunk;
  p.root_token = root_token;
  p.t_len = t_len;
  for (int r = 0; r < kMaxB; ++r) p.tree[r] = trees[r < B ? r : 0];
  char* ws = static_cast<char*>(workspace);
  p.tickets = reinterpret_cast<uint32_t*>(ws + w.tickets);
  p.chunk_m = reinterpret_cast<float*>(ws + w.chunk_m);
  p.chunk_s = reinterpret_cast<float*>(ws + w.chunk_s);
  p.cand = reinterpret_cast<unsigned long long*>(ws + w.cand);
  p.top_tok = reinterpret_cast<int32_t*>(ws + w.top_tok);
  p.top_logq = reinterpret_cast<float*>(ws + w.top_logq);
  p.search_only = shared ? 1 : 0;
  p.pops_out = shared ? static_cast<void*>(ws + pops_at) : nullptr;

  // dynamic smem: the chunk's logits during selection, the tree search after
  // dynamic smem: the chunk's logits during selection, the row's candidate
  // keys during the row merge, the tree search after
  size_t dyn = 16 * ((sizeof(float) * 2 * L * p.K + 15) / 16) + sizeof(TreeSmem) + sizeof(LevelSmem);
  if (dyn < sizeof(float) * kChunk) dyn = sizeof(float) * kChunk;
  const size_t cand_bytes = sizeof(unsigned long long) * static_cast<size_t>(p.C) * p.K;
  if (dyn < cand_bytes) dyn = cand_bytes;
  const bool vec = V % 4 == 0 && glance::aligned16(draft_logits);
  void (*kern)(const BuildParams);
  if (p.is_bf16)
    kern = vec ? build_tree_kernel<true, true> : build_tree_kernel<true, false>;
  else
    kern = vec ? build_tree_kernel<false, true> : build_tree_kernel<false, false>;
  cudaError_t e = glance::ensure_smem(reinterpret_cast<const void*>(kern), static_cast<int>(dyn));
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  kern<<<dim3(L * p.C, B), kThreads, dyn, static_cast<cudaStream_t>(stream)>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  if (shared) {
    const size_t dyn2 = sizeof(TreeSmem) + sizeof(int) * L * p.K + sizeof(float) * B * N;
    e = glance::ensure_smem(reinterpret_cast<const void*>(shared_pack_kernel), static_cast<int>(dyn2));
    if (e != cudaSuccess) return glance::cuda_fail(e, who);
    shared_pack_kernel<<<B, kThreads, dyn2, static_cast<cudaStream_t>(stream)>>>(p, *shared);
    e = cudaGetLastError();
    if (e != cudaSuccess) return glance::cuda_fail(e, who);
  }
  return GLANCE_OK;
}

}  // namespace

extern "C" size_t glance_build_tree_workspace_bytes(int L, int V, int N) {
  if (!sizes_ok(L, V, N)) return 0;
  return ws_layout(1, L, V, N).total;
}

extern "C" glance_status glance_build_tree(const void* draft_logits, glance_dtype dtype, int L,
                                           int V, int N, const int32_t* root_token,
                                           const int32_t* t_len, const glance_tree* tree,
                                           void* workspace, size_t workspace_bytes,
                                           void* stream) {
  return launch_build("glance_build_tree", draft_logits, dtype, 1, L, V, N, root_token, t_len,
                      tree, workspace, workspace_bytes, stream);
}

extern "C" size_t glance_build_tree_batched_workspace_bytes(int B, int L, int V, int N) {
  if (B < 1 || B > kMaxB || !sizes_ok(L, V, N)) return 0;
  return ws_layout(B, L, V, N).total;
}

extern "C" glance_status glance_build_tree_batched(const void* draft_logits, glance_dtype dtype,
                                                   int B, int L, int V, int N,
                                                   const int32_t* root_token,
                                                   const int32_t* t_len, const glance_tree* trees,
                                                   void* workspace, size_t workspace_bytes,
                                                   void* stream) {
  return launch_build("glance_build_tree_batched", draft_logits, dtype, B, L, V, N, root_token,
                      t_len, trees, workspace, workspace_bytes, stream);
}

extern "C" size_t glance_build_tree_shared_workspace_bytes(int B, int L, int V, int N_max) {
  if (B < 1 || B > kMaxB || !sizes_ok(L, V, N_max)) return 0;
  return ws_layout(B, L, V, N_max).total + sizeof(PopRec) * kMaxN * B;
}

extern "C" glance_status glance_build_tree_shared(const void* draft_logits, glance_dtype dtype,
                                                  int B, int L, int V, int N_max, int N_total,
                                                  const int32_t* root_token, const int32_t* t_len,
                                                  const float* root_entropy, float law_b0,
                                                  float law_b1, const glance_tree* trees,
                                                  int32_t* n_active, void* workspace,
                                                  size_t workspace_bytes, void* stream) {
  const char* who = "glance_build_tree_shared";
  if (!n_active) return glance::fail(GLANCE_ERR_INVALID_ARG, "%s: null n_active", who);
  if (N_total < 0) return glance::fail(GLANCE_ERR_INVALID_ARG, "%s: N_total must be >= 0", who);
  if (root_entropy && !(isfinite(law_b0) && isfinite(law_b1)))
    return glance::fail(GLANCE_ERR_INVALID_ARG, "%s: law coefficients must be finite", who);
  SharedArgs sa{N_total, root_entropy, law_b0, law_b1, n_active};
  return launch_build(who, draft_logits, dtype, B, L, V, N_max, root_token, t_len, trees,
                      workspace, workspace_bytes, stream, &sa);
}
