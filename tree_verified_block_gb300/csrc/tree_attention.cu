// Ancestor-masked tree attention (one layer).
//
// Paper: "Vision Is Not Overhead ..." (arXiv 2609.00355), Definition 1 and
// the proof of Theorem 1 (Appendix B.1): the tree rows are packed into one
// target pass whose mask lets the row of a depth-d node see the cached prefix,
// the root and its own ancestors only; masking changes the layout, not the
// row-level conditioning.
//
// Visible keys of packed row i: prefix slots 0..T-1, and tree slot T + k for
// every row k with bit (i, k) of the ancestor mask. Slots past T + N are never
// visible. Scores (q . k) * scale, softmax over the visible keys, weighted sum
// of values. T is read from device memory.
//
// bf16 / head_dim 128 path (tcgen05):
//   CTA = (kv head g, tile of 128 query rows, key split), 384 threads. The 128
//   query rows of a tile are (q head, packed row) pairs of the heads that share
//   kv head g (grouped-query attention), each head's rows padded to a power of
//   two. Warp 0 issues TMA loads (Q once, then K and V tiles of 128 slots into
//   a three-stage ring); warp 1 issues the MMAs: S = Q K^T into one of two
//   tensor-memory S buffers, so the next tile's S is computed while this
//   tile's softmax runs, then O += P V with P read from tensor memory. Q is
//   an operand from tensor memory too: the softmax threads copy the landed
//   Q tile there once, so the S products read only K from shared memory.
//   Warps 4..11 run the softmax, two threads per query row (one TMEM lane,
//   64 keys each, lanes t and t + 16 of one warp; they exchange their row
//   maxima and sums with a shuffle):
//   they read S with tcgen05.ld, apply the key mask in registers (the row's
//   ancestor words sit in registers and become one 32-bit visibility word per
//   32 slots), run the online softmax in base 2, write P as bf16 pairs and
//   rescale O in tensor memory when the running max grows.
//   The key range [0, T + N + 1) is split over up to 16 CTAs per (g, q tile)
//   so that the grid fills the SMs with one CTA each; the launch is
//   cooperative, so all CTAs are resident at once. Each CTA writes its
//   unnormalised partial O and (m, l) per row to the workspace (L2-resident),
//   announces itself on the group's counter (release), waits for the other
//   splits (acquire, bounded by a timeout that sets the device status), and
//   merges the rows it owns. One launch per layer.
// fp32 path (any head_dim multiple of 32 up to 128): plain CUDA cores, one
//   CTA per (row, q head), keys in chunks of 128 with an online softmax.
#include "glance_internal.cuh"

GLANCE_DEFINE_STATUS_WORD(status_attention)

using namespace glance_dev;

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ fp32 path

struct F32Params {
  const float* q;
  const float* k;
  const float* v;
  float* out;
  const uint64_t* anc;
  const int32_t* t_len;
  int rows, Hq, Hkv, D, W, t_cap;
  long long head_stride, row_stride;  // elements
  float scale;
};

constexpr int kF32Threads = 128;

__global__ void __launch_bounds__(kF32Threads) tree_attention_f32_kernel(const F32Params p) {
  const int i = blockIdx.x / p.Hq;
  const int h = blockIdx.x % p.Hq;
  const int g = h / (p.Hq / p.Hkv);
  __shared__ float s_q[128];
  __shared__ float s_p[kF32Threads];
  __shared__ int s_tree[256];
  __shared__ int s_ntree;
  __shared__ float s_red[kF32Threads / 32];
  const int T = *p.t_len;
  if (T < 0 || T + p.rows > p.t_cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(GLANCE_DEV_TREE_CAPACITY);
    return;
  }
  for (int d = threadIdx.x; d < p.D; d += kF32Threads)
    s_q[d] = p.q[(static_cast<size_t>(i) * p.Hq + h) * p.D + d];
  if (threadIdx.x == 0) {
    int n = 0;
    for (int w = 0; w < p.W; ++w) {
      uint64_t word = p.anc[i * p.W + w];
      while (word) {
        const int b = __ffsll(static_cast<long long>(word)) - 1;
        word &= word - 1;
        const int k = 64 * w + b;
        if (k < p.rows) s_tree[n++] = k;
      }
    }
    s_ntree = n;
  }
  __syncthreads();
  const int n_keys = T + s_ntree;
  const float* kh = p.k + g * p.head_stride;
  const float* vh = p.v + g * p.head_stride;
  float m = -INFINITY, l = 0.f;
  float acc = 0.f;  // thread t < D owns output dim t (D <= 128 = threads)
  for (int c0 = 0; c0 < n_keys; c0 += kF32Threads) {
    const int j = c0 + threadIdx.x;
    float s = -INFINITY;
    if (j < n_keys) {
      const int slot = j < T ? j : T + s_tree[j - T];
      const float* kr = kh + (GLANCE_IN_BOUNDS(slot, p.t_cap) ? slot : 0) * p.row_stride;
      float dot = 0.f;
      for (int d = 0; d < p.D; ++d) dot = fmaf(s_q[d], kr[d], dot);
      s = dot * p.scale;
    }
    float cm = s;
#pragma unroll
    for (int o = 16; o; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = cm;
    __syncthreads();
    cm = s_red[0];
    for (int w = 1; w < kF32Threads / 32; ++w) cm = fmaxf(cm, s_red[w]);
    const float m_new = fmaxf(m, cm);
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    const float pj = (j < n_keys) ? expf(s - m_new) : 0.f;
    s_p[threadIdx.x] = pj;
    __syncthreads();
    float psum = 0.f;
    const int cn = min(kF32Threads, n_keys - c0);
    for (int jj = 0; jj < cn; ++jj) psum += s_p[jj];
    l = l * alpha + psum;
    if (threadIdx.x < p.D) {
      float a = acc * alpha;
      for (int jj = 0; jj < cn; ++jj) {
        const int jk = c0 + jj;
        const int slot = jk < T ? jk : T + s_tree[jk - T];
        if (GLANCE_IN_BOUNDS(slot, p.t_cap)) a = fmaf(s_p[jj], vh[slot * p.row_stride + threadIdx.x], a);
      }
      acc = a;
    }
    m = m_new;
    __syncthreads();
  }
  const size_t oidx = (static_cast<size_t>(i) * p.Hq + h) * p.D + threadIdx.x;
  if (threadIdx.x < p.D && GLANCE_IN_BOUNDS(oidx, static_cast<size_t>(p.rows) * p.Hq * p.D)) p.out[oidx] = acc / l;
}

// ------------------------------------------------------------------ bf16 path

constexpr int kD = 128;          // head_dim
constexpr int kBM = 128;         // query rows per tile (MMA M)
constexpr int kBN = 128;         // key slots per tile (MMA N of S, K of PV)
constexpr int kStages = 3;       // K/V ring depth
constexpr int kPreTiles = 1;     // prefix key tiles fetched before the dependency wait
constexpr int kThreads = 384;    // 12 warps: TMA, MMA, TMEM, idle, 2 x 4 softmax
constexpr int kTmemCols = 512;   // S0 (128) | S1 (128) | O (128) | P (64) | Q (64)
constexpr int kMaxSplit = 16;    // key splits of one (kv head, q tile)
constexpr int kMaxB = 16;        // requests of one batched call
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // pipeline wait limit: 2 s
constexpr uint32_t kHalfBytes = kBN * 128;          // 64 head dims x 128 slots, bf16: 16 KB
constexpr uint32_t kQBytes = 2 * kBM * 128;         // 32 KB
constexpr uint32_t kKVStageBytes = 4 * kHalfBytes;  // K and V, two halves each: 64 KB
constexpr uint32_t kRingBytes = kStages * kKVStageBytes;
constexpr size_t kSmemBytes = 1024 /*align*/ + kQBytes + kRingBytes + 1280;

// B requests, CTAs request-major: request r owns CTAs [cta0[r], cta0[r+1]),
// (kv head g, q tile qt, split) with the split fastest. A group is one
// (request, g, qt); its n_split[r] CTAs cover the request's key range.
// NB: capacity of the per-request arrays (1 for single-request calls, so
// that their parameter block stays small).
template <int NB>
struct Bf16Params {
  const uint64_t* anc[NB];
  const int32_t* t_len[NB];
  int t_cap[NB];
  int cta0[NB + 1];
  int n_split[NB];
  int slot0[NB];             // first partial slot of the request's groups
  __nv_bfloat16* out;        // [B][rows][Hq][128]
  uint4* part_o;             // [slots][16 dim octets][128 rows] partial O / l, bf16
  float2* part_ml;           // [slots][128] (running max, sum) per row
  uint32_t* arrive;          // [groups] split arrivals, then [groups] departures
  int B, rows, Hq, Hkv, G, Rp, n_qt, W;
  int box_rows;              // rows per Q box = min(Rp, 128)
  int ticket_merge;          // 1: the last split CTA of a group merges it (any grid);
                             // 0: all splits wait for each other (cooperative launch)
  float scale_log2;          // scale * log2(e)
  unsigned long long wait_ns;  // limit of every pipeline wait
  int withhold_v;            // 1: the producer never copies the V of a CTA's last key tile
                             //    (the timeout check's wait that runs out)
  int n_slots;               // partial slots in the workspace (bounds-checked build)
};

// K and V tensor maps of every request's cache of this layer
template <int NB>
struct KVMaps {
  CUtensorMap k[NB];
  CUtensorMap v[NB];
};

struct __align__(8) Bars {
  uint64_t q_full;
  uint64_t q_tmem;           // Q copied from shared to tensor memory (the softmax threads)
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_ready;
  uint64_t o_done;
  uint64_t merge_full;       // ticket-mode merge: partials staged in shared memory
  uint64_t mma_drain;        // every MMA of the CTA has finished
  uint32_t tmem_base;
  int abort_flag;
  int ticket_last;           // ticket mode: this CTA completed the group's count and merges it
};
static_assert(sizeof(Bars) <= 1280, "barrier block");

__device__ __forceinline__ void fail_pipeline(Bars* bars) {
  report(GLANCE_DEV_PIPELINE_TIMEOUT);
  atomicExch(&bars->abort_flag, 1);
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* bars,
                                              unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*reinterpret_cast<volatile int*>(&bars->abort_flag)) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

// Key run of one split: [k0, k1) of [0, n_keys), equal runs of `per` slots
// (a multiple of `align`: 32 when the splits of a group wait for each other,
// so that they finish together; a whole tile in ticket mode, where a split
// that finishes early frees its SM for the next wave); its key tiles are the
// 128-slot pieces of the run, the last one `cols` wide (rounded up to 32; the
// QK^T and PV products of that tile stop there).
struct SplitRun {
  int k0, k1, n_tiles;
  __device__ __forceinline__ int tile_key0(int j) const { return k0 + j * kBN; }
  __device__ __forceinline__ int tile_cols(int j) const {
    const int c = (k1 - tile_key0(j) + 31) / 32 * 32;
    return c > kBN ? kBN : c;
  }
};
__device__ __forceinline__ SplitRun split_run(int n_keys, int n_split, int split, int align) {
  const int per = ((n_keys + n_split - 1) / n_split + align - 1) / align * align;
  SplitRun r;
  r.k0 = split * per;
  r.k1 = r.k0 + per < n_keys ? r.k0 + per : n_keys;
  r.n_tiles = r.k1 > r.k0 ? (r.k1 - r.k0 + kBN - 1) / kBN : 0;
  if (r.n_tiles == 0) r.k1 = r.k0;
  return r;
}

// PV steps of 16 slots for key tile j: up to the tile's columns, and for the
// last tile of the key range up to the first step boundary past n_keys.
__device__ __forceinline__ int pv_steps(const SplitRun& run, int j, int n_keys) {
  const int key0 = run.tile_key0(j);
  const int steps = run.tile_cols(j) / 16;
  return key0 + steps * 16 > n_keys ? (n_keys - key0 + 15) / 16 : steps;
}

// word w (0..3) of a row's ancestor mask, 0 outside, without dynamic indexing
__device__ __forceinline__ uint64_t anc_word(const uint64_t (&a)[4], int w) {
  return w == 0 ? a[0] : w == 1 ? a[1] : w == 2 ? a[2] : w == 3 ? a[3] : 0ull;
}

// Visibility of 32 consecutive key slots starting at tree index kb (= slot - T;
// negative for prefix slots): bit i is set iff slot kb + i is a prefix slot, or
// a tree row (kb + i < rows) on the row's ancestor list.
__device__ __forceinline__ uint32_t visible32(const uint64_t (&a)[4], int kb, int rows) {
  if (kb <= -32) return 0xFFFFFFFFu;
  uint32_t tree_bits;
  if (kb < 0) {
    tree_bits = static_cast<uint32_t>(a[0] << (-kb));
  } else {
    const int w = kb >> 6, o = kb & 63;
    const uint64_t lo = anc_word(a, w), hi = anc_word(a, w + 1);
    tree_bits = static_cast<uint32_t>(o ? (lo >> o) | (hi << (64 - o)) : lo);
  }
  const int lim = rows - kb;  // bits i < lim are tree rows
  const uint32_t rows_mask = lim >= 32 ? 0xFFFFFFFFu : lim <= 0 ? 0u : ((1u << lim) - 1u);
  const uint32_t prefix_mask = kb < 0 ? ((1u << (-kb)) - 1u) : 0u;
  return prefix_mask | (tree_bits & rows_mask);
}

// Ticket mode: the last split of a group merges all 128 rows from shared
// memory (the K/V ring and Q area are idle by now). The splits' (m, l) go
// first, then their partials (O_s / l_s, bf16, 32 KB per split, contiguous in
// the workspace) in chunks of kMergeChunk splits, one bulk copy each. Called
// by the 256 softmax threads; thread (lrow, half) owns 64 output dims of row
// lrow.
constexpr int kMergeMlBytes = kMaxSplit * kBM * 8;  // [S][128] float2
constexpr int kMergeWBytes = kMaxSplit * kBM * 4;   // [S][128] weights
constexpr int kMergeChunk =
    static_cast<int>((kQBytes + kRingBytes - kMergeMlBytes - kMergeWBytes) / (kBM * kD * 2));

template <typename P>
__device__ __noinline__ void ticket_merge(const P& p, Bars* bars, unsigned char* area, int slot, int S, int qt,
                             int g, int q_row0, int half, int lrow) {
  if (!GLANCE_IN_BOUNDS(slot + S - 1, p.n_slots)) return;  // uniform across the 256 threads
  const float2* s_ml = reinterpret_cast<const float2*>(area);
  float* s_w = reinterpret_cast<float*>(area + kMergeMlBytes);
  unsigned char* s_o = area + kMergeMlBytes + kMergeWBytes;
  const int n_chunks = (S + kMergeChunk - 1) / kMergeChunk;
  if (threadIdx.x == 128) {
    // the other splits' partials were acquired through the group counter
    // (generic proxy); the bulk copies read them through the async proxy
    fence_proxy_async_global();
    const int c0 = S < kMergeChunk ? S : kMergeChunk;
    mbar_arrive_expect_tx(&bars->merge_full,
                          static_cast<uint32_t>(S * kBM * 8 + c0 * kBM * kD * 2));
    bulk_copy_g2s(area, p.part_ml + static_cast<size_t>(slot) * kBM,
                  static_cast<uint32_t>(S * kBM * 8), &bars->merge_full);
    bulk_copy_g2s(s_o, p.part_o + static_cast<size_t>(slot) * 16 * kBM,
                  static_cast<uint32_t>(c0 * kBM * kD * 2), &bars->merge_full);
  }
  const bool got = mbar_wait(&bars->merge_full, 0, p.wait_ns);
  if (half == 0) {
    float M = -INFINITY;
    for (int sx = 0; sx < S; ++sx) M = fmaxf(M, s_ml[sx * kBM + lrow].x);
    float Lt = 0.f;
    for (int sx = 0; sx < S; ++sx) {
      const float2 ml = s_ml[sx * kBM + lrow];
      const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M) * ml.y;
      s_w[sx * kBM + lrow] = w;
      Lt += w;
    }
    const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
    for (int sx = 0; sx < S; ++sx) s_w[sx * kBM + lrow] *= inv;
  }
  // one answer for all 256 threads, so that they leave the loop together
  bool bad = named_bar_or(1, 256, !got);
  float acc[64];
#pragma unroll
  for (int e = 0; e < 64; ++e) acc[e] = 0.f;
  for (int k = 0; k < n_chunks && !bad; ++k) {
    const int base = k * kMergeChunk;
    const int cnt = S - base < kMergeChunk ? S - base : kMergeChunk;
    if (k > 0) {
      named_bar(1, 256);  // every thread is done with the previous chunk
      if (threadIdx.x == 128) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars->merge_full, static_cast<uint32_t>(cnt * kBM * kD * 2));
        bulk_copy_g2s(s_o, p.part_o + static_cast<size_t>(slot + base) * 16 * kBM,
                      static_cast<uint32_t>(cnt * kBM * kD * 2), &bars->merge_full);
      }
      bad = named_bar_or(1, 256, !mbar_wait(&bars->merge_full, k & 1, p.wait_ns));
      if (bad) break;
    }
    for (int sx = 0; sx < cnt; ++sx) {
      const float w = s_w[(base + sx) * kBM + lrow];
      if (w == 0.f) continue;
      const uint4* src = reinterpret_cast<const uint4*>(s_o) + (sx * 16 + 8 * half) * kBM + lrow;
#pragma unroll
      for (int o = 0; o < 8; ++o) {
        const uint4 v = src[o * kBM];
        const uint32_t av[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[8 * o + 2 * e] += w * __uint_as_float(av[e] << 16);
          acc[8 * o + 2 * e + 1] += w * __uint_as_float(av[e] & 0xFFFF0000u);
        }
      }
    }
  }
  if (bad) {
    report(GLANCE_DEV_PIPELINE_TIMEOUT);
    return;
  }
  const int oq = qt * kBM + lrow;
  const int ohl = oq / p.Rp, oprow = oq % p.Rp;
  const size_t oidx = (static_cast<size_t>(q_row0 + oprow) * p.Hq + g * p.G + ohl) * kD + 64 * half;
  if (ohl < p.G && oprow < p.rows &&
      GLANCE_IN_BOUNDS(oidx + 63, static_cast<size_t>(p.B) * p.rows * p.Hq * kD)) {
    uint4* dst = reinterpret_cast<uint4*>(p.out + oidx);
#pragma unroll
    for (int o = 0; o < 8; ++o)
      dst[o] = make_uint4(pack_bf16x2(acc[8 * o], acc[8 * o + 1]), pack_bf16x2(acc[8 * o + 2], acc[8 * o + 3]),
                          pack_bf16x2(acc[8 * o + 4], acc[8 * o + 5]), pack_bf16x2(acc[8 * o + 6], acc[8 * o + 7]));
  }
}

// Softmax arithmetic on pairs: the three-input max and the packed f32x2
// FMA / add of sm_100+ take one instruction per two elements (the softmax
// warps are bound by instruction issue); each lane of a packed operation
// rounds as the scalar one does.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ unsigned long long pair_f2(float lo, float hi) {
  unsigned long long v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
  return v;
}
__device__ __forceinline__ void split_f2(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long fma_f2(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long add_f2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// One CTA = (kv head g, q tile, key split). The key splits of one (g, q tile)
// merge their partial results through the workspace once all have arrived.
template <int NB>
__global__ void __launch_bounds__(kThreads, 1)
    tree_attention_bf16_kernel(const __grid_constant__ CUtensorMap map_q,
                               const __grid_constant__ KVMaps<NB> maps,
                               const __grid_constant__ Bf16Params<NB> p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* sQ = smem;
  unsigned char* sKV = smem + kQBytes;
  Bars* bars = reinterpret_cast<Bars*>(sKV + kRingBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int req = 0;
  while (req + 1 < p.B && static_cast<int>(blockIdx.x) >= p.cta0[req + 1]) ++req;
  const int n_split = p.n_split[req];
  const int local = blockIdx.x - p.cta0[req];
  const int split = local % n_split;
  const int grp_local = local / n_split;  // g * n_qt + qt
  const int qt = grp_local % p.n_qt;
  const int g = grp_local / p.n_qt;
  const int grp = req * p.Hkv * p.n_qt + grp_local;
  const CUtensorMap* map_k = &maps.k[req];
  const CUtensorMap* map_v = &maps.v[req];
  const int q_row0 = req * p.rows;  // this request's first row in q and out

  // The next kernel in the stream may start its own prologue on free SMs now;
  // this kernel sets up barriers and tensor memory, then waits until the
  // previous kernel's writes are visible before it reads any input.
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_tmem, 256);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    mbar_init(&bars->p_ready, 256);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->merge_full, 1);
    mbar_init(&bars->mma_drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(map_k);
    tma_prefetch_desc(map_v);
  }
  if (warp == 2) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // The cache prefix (slots < T) and T itself are written only by calls that
  // let no kernel start early (accept_commit), so the first key tile that
  // lies wholly inside the prefix can be fetched before the wait; tiles that
  // hold tree rows (written by the previous kernel) wait for it.
  int pre = 0, T_pre = -1;
  if (threadIdx.x == 0) {
    T_pre = *p.t_len[req];
    if (T_pre >= 0 && T_pre + p.rows <= p.t_cap[req]) {
      const SplitRun run_pre = split_run(T_pre + p.rows, n_split, split, p.ticket_merge ? kBN : 32);
      const uint64_t pol_kv = policy_evict_first();
      for (int j = 0; j < kPreTiles && j < run_pre.n_tiles; ++j) {
        const int key0 = run_pre.tile_key0(j);
        if (key0 + run_pre.tile_cols(j) > T_pre) break;
        unsigned char* stage = sKV + j * kKVStageBytes;
        mbar_arrive_expect_tx(&bars->k_full[j], 2 * kHalfBytes);
        tma_load_3d(stage + 0 * kHalfBytes, map_k, &bars->k_full[j], 0, key0, g, pol_kv);
        tma_load_3d(stage + 1 * kHalfBytes, map_k, &bars->k_full[j], 64, key0, g, pol_kv);
        mbar_arrive_expect_tx(&bars->v_full[j], 2 * kHalfBytes);
        tma_load_3d(stage + 2 * kHalfBytes, map_v, &bars->v_full[j], 0, key0, g, pol_kv);
        tma_load_3d(stage + 3 * kHalfBytes, map_v, &bars->v_full[j], 64, key0, g, pol_kv);
        ++pre;
      }
    }
  }
  pdl_wait_prior();

  // Q does not depend on T: its copy goes out before T is read, so the two
  // round trips overlap. The thread that issues it initialised the barriers.
  if (threadIdx.x == 0) {
    const uint64_t pol_q = policy_evict_last();
    const int pieces = kBM / p.box_rows;
    int n_boxes = 0;
    for (int pc = 0; pc < pieces; ++pc) n_boxes += ((qt * kBM + pc * p.box_rows) / p.Rp < p.G) ? 2 : 0;
    mbar_arrive_expect_tx(&bars->q_full, n_boxes * p.box_rows * 128);
    for (int pc = 0; pc < pieces; ++pc) {
      const int r0 = qt * kBM + pc * p.box_rows;
      const int h = r0 / p.Rp;
      if (h >= p.G) continue;
      for (int hf = 0; hf < 2; ++hf)
        tma_load_3d(sQ + hf * (kBM * 128) + pc * p.box_rows * 128, &map_q, &bars->q_full,
                    hf * 64, g * p.G + h, q_row0 + r0 % p.Rp, pol_q);
    }
  }

  const int T = *p.t_len[req];
  // T is not written while a call can still be starting; a caller that breaks
  // that has the call give up (its prefetched tiles would be the wrong ones)
  const bool raced = __syncthreads_or(threadIdx.x == 0 && pre > 0 && T != T_pre) != 0;
  if (raced && threadIdx.x == 0) report(GLANCE_DEV_BAD_TREE);
  const bool room = !raced && T >= 0 && T + p.rows <= p.t_cap[req];
  // key tiles of this split over slots [0, T + rows)
  const int n_keys = room ? T + p.rows : 0;
  const SplitRun run = split_run(n_keys, n_split, split, p.ticket_merge ? kBN : 32);
  const int my_tiles = run.n_tiles;

  if (threadIdx.x == 0 && !room && !raced && local == 0) report(GLANCE_DEV_TREE_CAPACITY);
  // query pieces of this tile that hold no real (head, row): zero them so the
  // MMA reads finite values
  {
    const int pieces = kBM / p.box_rows;
    for (int pc = 0; pc < pieces; ++pc) {
      const int r0 = qt * kBM + pc * p.box_rows;  // first q-row of the piece
      if (r0 / p.Rp >= p.G) {
        for (int hf = 0; hf < 2; ++hf) {
          uint4* dst = reinterpret_cast<uint4*>(sQ + hf * (kBM * 128) + pc * p.box_rows * 128);
          for (int i = threadIdx.x; i < p.box_rows * 8; i += kThreads) dst[i] = make_uint4(0, 0, 0, 0);
        }
      }
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tS0 = tmem;         // S, double-buffered (fp32, 128 cols each)
  const uint32_t tO = tmem + 256;    // O (fp32, 128 cols)
  const uint32_t tP = tmem + 384;    // P (bf16 pairs, 64 cols)
  const uint32_t tQ = tmem + 448;    // Q (bf16 pairs, 64 cols): the A operand of S = Q K^T

  // softmax-thread state, live until the merge
  // Softmax warp (quarter, sub) holds the 16 rows 32 quarter + 16 sub + (lane & 15)
  // of the tile; lanes 0-15 hold keys / output dims 0-63 of those rows and
  // lanes 16-31 the other 64, so both halves of a row sit in one warp and meet
  // through a shuffle (TMEM access shape 16x32bx2).
  const bool is_sm = warp >= 4;
  const int half = is_sm ? lane >> 4 : 0;  // which 64 keys / 64 output dims
  const int quarter = warp & 3;            // TMEM lane quarter
  const int sub = is_sm ? (warp - 4) >> 2 : 0;
  const int lrow = quarter * 32 + sub * 16 + (lane & 15);
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32 + sub * 16) << 16;
  const int qrow = qt * kBM + lrow;  // index within the kv head's query rows
  const int hl = qrow / p.Rp;
  const int prow = qrow % p.Rp;
  const bool valid = hl < p.G && prow < p.rows;
  const int head = g * p.G + hl;
  float m = -INFINITY, lh = 0.f;
  bool ok = true;
  int n_issued = 0;  // K/V tiles the producer issued (after an abort: which may still land)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && my_tiles == 0) {
      // Q was issued before T was known (and prefix tiles before the wait):
      // let them land before the CTA exits
      (void)mbar_wait(&bars->q_full, 0, 50000000ull);
      for (int j = 0; j < pre; ++j) {
        (void)mbar_wait(&bars->k_full[j], 0, 50000000ull);
        (void)mbar_wait(&bars->v_full[j], 0, 50000000ull);
      }
    }
    if (lane == 0 && my_tiles > 0) {
      const uint64_t pol_kv = policy_evict_first();
      int issued = pre;
      // the timeout check's copy that is never made (the last tile's V,
      // unless it went out before the dependency wait)
      auto withheld = [&](int j) { return p.withhold_v && j == my_tiles - 1 && j >= pre; };
      for (int j = pre; j < my_tiles; ++j) {
        const int st = j % kStages;
        // Every CTA of the grid starts at once: the first tile of all of them
        // goes out alone, so that Q and K/V of tile 0 land (and the first MMA
        // starts) before the rest of the ring competes for DRAM.
        if (j == 1 && !wait_or_abort(&bars->k_full[0], 0, bars, p.wait_ns)) {
          fail_pipeline(bars);
          break;
        }
        if (j >= kStages && !wait_or_abort(&bars->kv_empty[st], ((j / kStages) - 1) & 1, bars, p.wait_ns)) {
          fail_pipeline(bars);
          break;
        }
        unsigned char* stage = sKV + st * kKVStageBytes;
        const int key0 = run.tile_key0(j);
        // K and V of a tile complete separately: QK^T needs only K, and V
        // lands while the tile's softmax runs
        mbar_arrive_expect_tx(&bars->k_full[st], 2 * kHalfBytes);
        tma_load_3d(stage + 0 * kHalfBytes, map_k, &bars->k_full[st], 0, key0, g, pol_kv);
        tma_load_3d(stage + 1 * kHalfBytes, map_k, &bars->k_full[st], 64, key0, g, pol_kv);
        if (!withheld(j)) {
          mbar_arrive_expect_tx(&bars->v_full[st], 2 * kHalfBytes);
          tma_load_3d(stage + 2 * kHalfBytes, map_v, &bars->v_full[st], 0, key0, g, pol_kv);
          tma_load_3d(stage + 3 * kHalfBytes, map_v, &bars->v_full[st], 64, key0, g, pol_kv);
        }
        ++issued;
      }
      n_issued = issued;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && my_tiles > 0) {
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, kD, false, true);
      auto issue_qk = [&](int j) -> bool {
        const int st = j % kStages;
        if (!wait_or_abort(&bars->k_full[st], (j / kStages) & 1, bars, p.wait_ns)) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(sKV + st * kKVStageBytes);
        const uint32_t tS = tS0 + (j & 1) * 128;
        const uint32_t idesc_s = idesc_bf16_f32(kBM, run.tile_cols(j), false, false);
        // A = Q from tensor memory (dims 16 kk .. 16 kk + 15 in columns 8 kk ..),
        // B = the K tile (K-major, 128-byte swizzle): only K is read from
        // shared memory, 4 KB per MMA instead of 8
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t offk = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          mma_bf16_ts(tS, tQ + kk * 8, sdesc_sw128(k_addr + offk, 16, 1024), idesc_s, kk > 0);
        }
        mma_commit(&bars->s_full[j & 1]);
        return true;
      };
      bool good = wait_or_abort(&bars->q_tmem, 0, bars, p.wait_ns) && issue_qk(0);
      for (int j = 0; good && j < my_tiles; ++j) {
        // S of the next tile goes into the other buffer while tile j's softmax runs;
        // that buffer was last read by the softmax of tile j-1, which p_ready(j-1) covered
        if (j + 1 < my_tiles && !issue_qk(j + 1)) {
          good = false;
          break;
        }
        if (!wait_or_abort(&bars->p_ready, j & 1, bars, p.wait_ns) ||
            !wait_or_abort(&bars->v_full[j % kStages], (j / kStages) & 1, bars, p.wait_ns)) {
          good = false;
          break;
        }
        tc_fence_after();
        const uint32_t v_addr = smem_u32(sKV + (j % kStages) * kKVStageBytes) + 2 * kHalfBytes;
        // O += P V over the tile's key slots, 16 per step (8 bf16-pair columns
        // of P each); the last tile of the key range stops at the first step
        // boundary past T + rows (the softmax threads zeroed the V rows of
        // that step beyond T + rows before releasing P).
        const int steps = pv_steps(run, j, n_keys);
        for (int kk = 0; kk < steps; ++kk)
          mma_bf16_ts(tO, tP + kk * 8, sdesc_sw128(v_addr + kk * 2048, kHalfBytes, 1024), idesc_o,
                      (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->o_done);
        // only stages the producer will refill need a release
        if (j + kStages < my_tiles) mma_commit(&bars->kv_empty[j % kStages]);
      }
      if (!good) fail_pipeline(bars);
    }
  } else if (is_sm) {
    // ------------------------------------------------------------ softmax
    uint64_t anc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int w = 0; w < 4; ++w)
      if (valid && w < p.W) anc[w] = p.anc[req][prow * p.W + w];
    // Q into tensor memory, in the layout of P: row = lane, column c = dims
    // (2c, 2c + 1). The Q tile in shared memory is two 128-byte-swizzled
    // halves of 64 dims (16-byte chunk c of row r at r * 128 + ((c ^ (r & 7)) * 16));
    // this thread copies the 64 dims of its half of row lrow.
    if (my_tiles > 0) {
      const bool got_q = __all_sync(0xffffffffu, wait_or_abort(&bars->q_full, 0, bars, p.wait_ns));
      if (!got_q) fail_pipeline(bars);
      uint32_t qv[32];
      const unsigned char* qrow_s = sQ + half * (kBM * 128) + lrow * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = got_q ? *reinterpret_cast<const uint4*>(qrow_s + ((c ^ (lrow & 7)) << 4))
                              : make_uint4(0u, 0u, 0u, 0u);
        qv[4 * c] = v.x;
        qv[4 * c + 1] = v.y;
        qv[4 * c + 2] = v.z;
        qv[4 * c + 3] = v.w;
      }
      tmem_st16x2<32>(tQ + lane_off, *reinterpret_cast<const uint32_t(*)[16]>(qv));
      tmem_st16x2<32>(tQ + lane_off + 16, *reinterpret_cast<const uint32_t(*)[16]>(qv + 16));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->q_tmem);
    }
    // A failed wait raises the CTA's abort flag; each warp leaves the loop as
    // a whole (warp vote) at the first tile where it sees the flag, and the
    // other warps' later waits give up on the same flag.
    for (int j = 0; j < my_tiles; ++j) {
      const int key0 = run.tile_key0(j);
      // warp-uniform: tcgen05.ld / st below are warp-collective
      const bool got_s = __all_sync(0xffffffffu, wait_or_abort(&bars->s_full[j & 1], (j >> 1) & 1, bars, p.wait_ns));
      if (!got_s) fail_pipeline(bars);
      tc_fence_after();
      const uint32_t tS = tS0 + (j & 1) * 128;
      // this thread's 64 keys of the S row
      uint32_t sr[64];
      if (got_s) {
        tmem_ld32x2<64>(tS + lane_off, *reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_ld32x2<64>(tS + lane_off + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) sr[e] = 0xFF800000u;
      }
      if (key0 + kBN > T || key0 + kBN > run.k1) {
        // slots >= T: visible only on the row's ancestor list (and < T + rows);
        // slots past this split's run (columns of the tile the products did
        // not compute, or the next split's keys) are not this CTA's
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int s0 = key0 + 64 * half + 32 * c;
          uint32_t vm = visible32(anc, s0 - T, p.rows);
          const int lim_end = run.k1 - s0;
          if (lim_end < 32) vm &= lim_end <= 0 ? 0u : ((1u << lim_end) - 1u);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            sr[32 * c + e] = ((vm >> e) & 1u) ? sr[32 * c + e] : 0xFF800000u;  // -inf
        }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int e = 0; e < 64; e += 8) {
        mx0 = max3f(mx0, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
        mx1 = max3f(mx1, __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]));
        mx2 = max3f(mx2, __uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5]));
        mx3 = max3f(mx3, __uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7]));
      }
      // scale_log2 > 0, so the max commutes with the scaling
      const float pm = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * p.scale_log2;
      const bool seen = *reinterpret_cast<volatile int*>(&bars->abort_flag) != 0;
      if (__any_sync(0xffffffffu, seen || !got_s)) {
        ok = false;
        break;  // the vote gives the whole warp the same answer
      }
      // lane ^ 16 holds the other 64 keys of the row
      const float mt = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
      // The running max only moves when some row of the warp grew by more than
      // 8 (base 2) or had no max yet: a stale max keeps P <= 2^8, cancels
      // between O and l, and lets most tiles skip the O rescale. Both halves
      // of each of the warp's 16 rows take part in the vote, so they keep the
      // same max.
      const bool grow = __any_sync(0xffffffffu, mt > m + 8.f);
      const float m_new = grow ? fmaxf(m, mt) : m;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_use);
      const float neg_m = -m_use;
      uint32_t pk[32];
      const unsigned long long sc2 = pair_f2(p.scale_log2, p.scale_log2), nm2 = pair_f2(neg_m, neg_m);
      unsigned long long ls2 = pair_f2(0.f, 0.f);  // even and odd keys' sums, as two scalar chains
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        float t0, t1;
        split_f2(fma_f2(pair_f2(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), sc2, nm2), t0, t1);
        const float p0 = ex2_approx(t0);
        const float p1 = ex2_approx(t1);
        ls2 = add_f2(ls2, pair_f2(p0, p1));
        pk[e] = pack_bf16x2(p0, p1);
      }
      float ls0, ls1;
      split_f2(ls2, ls0, ls1);
      // PV(j-1) must be done with P and O before they are rewritten
      const bool got_o =
          __all_sync(0xffffffffu, j == 0 || wait_or_abort(&bars->o_done, (j - 1) & 1, bars, p.wait_ns));
      if (!got_o) fail_pipeline(bars);
      tc_fence_after();
      if (got_o) {
        tmem_st16x2<32>(tP + lane_off, *reinterpret_cast<const uint32_t(*)[16]>(pk));
        tmem_st16x2<32>(tP + lane_off + 16, *reinterpret_cast<const uint32_t(*)[16]>(pk + 16));
        // rescale this half's 64 output dims when the running max grew
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t r[32];
            const uint32_t ta = tO + lane_off + 32 * c;
            tmem_ld32x2<64>(ta, r);
            tmem_ld_wait();
            uint32_t a[16], b[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              a[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              b[e] = __float_as_uint(__uint_as_float(r[16 + e]) * alpha);
            }
            tmem_st16x2<64>(ta, a);
            tmem_st16x2<64>(ta + 16, b);
          }
        }
        tmem_st_wait();
      }
      lh = lh * alpha + (ls0 + ls1);
      m = m_new;
      // The V rows of the key range's last PV step beyond T + rows are never
      // weighted (P = 0) but may hold anything, even NaN (0 * NaN = NaN): the
      // 256 softmax threads zero them (at most 15 rows of 256 bytes, one
      // 16-byte store each) once the tile's V has landed, before P is released.
      {
        const int key0z = run.tile_key0(j);
        const int zrows = pv_steps(run, j, n_keys) * 16 - (n_keys - key0z);
        if (zrows > 0) {
          const int t = threadIdx.x - 128;
          if (wait_or_abort(&bars->v_full[j % kStages], (j / kStages) & 1, bars, p.wait_ns)) {
            if (t < zrows * 16) {
              unsigned char* vs = sKV + (j % kStages) * kKVStageBytes + 2 * kHalfBytes;
              const int r = n_keys - key0z + (t >> 4), c = t & 15;  // row, 16-byte chunk (8 per half)
              reinterpret_cast<uint4*>(vs + (c >> 3) * kHalfBytes + r * 128)[c & 7] = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
          } else {
            fail_pipeline(bars);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->p_ready);
    }
    const bool last_ok = !ok || my_tiles == 0 || wait_or_abort(&bars->o_done, (my_tiles - 1) & 1, bars, p.wait_ns);
    if (!last_ok) fail_pipeline(bars);
    // one answer for all 256 softmax threads: the epilogue's TMEM loads are
    // warp-collective
    ok = !named_bar_or(1, 256, !ok || !last_ok);
    tc_fence_after();
  }

  // ---------------------------------------------------------------- output
  // total l of the row = sum of the two halves' partial sums (same max)
  float l = 0.f;
  if (is_sm) l = lh + __shfl_xor_sync(0xffffffffu, lh, 16);
  if (n_split == 1) {
    if (is_sm && ok && my_tiles > 0) {
      const float inv = 1.f / l;
      const size_t oidx = (static_cast<size_t>(q_row0 + prow) * p.Hq + head) * kD + 64 * half;
      const bool out_ok = valid && GLANCE_IN_BOUNDS(oidx + 63, static_cast<size_t>(p.B) * p.rows * p.Hq * kD);
      __nv_bfloat16* dst = p.out + oidx;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tmem_ld32x2<64>(tO + lane_off + 32 * c, r);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv, __uint_as_float(r[2 * e + 1]) * inv);
        if (out_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            d4[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
    }
  } else {
    // Each split CTA writes its partial O_s / l_s (bf16) and (m_s, l_s) per
    // row to the workspace (L2-resident) and publishes it on the group
    // counter with a release add. The group is then merged as
    //   O = sum_s w_s l_s (O_s / l_s) / sum_s w_s l_s,  w_s = 2^(m_s - M):
    // * cooperative mode: every split waits (acquire loads, bounded) until
    //   all have arrived and merges 1/S of the rows; the last to leave resets
    //   both counters;
    // * ticket mode: the split whose add completes the count acquires the
    //   others' partials, merges all rows and resets the counter; nobody waits.
    const int S = n_split;
    const int slot = p.slot0[req] + grp_local * S;  // first partial slot of the group
    int own0, own_rows;
    if (is_sm) {
      // column-major (dim octet, row): a warp's store covers 32 consecutive rows
      uint4* po = p.part_o + (static_cast<size_t>(slot) + split) * 16 * kBM + lrow;
      const bool slot_ok = GLANCE_IN_BOUNDS(slot + split, p.n_slots);
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        if (my_tiles > 0 && ok) {
          tmem_ld32x2<64>(tO + lane_off + 32 * c, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = 0u;
        }
#pragma unroll
        for (int v8 = 0; v8 < 4; ++v8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(r[8 * v8 + 2 * e]) * inv_l,
                               __uint_as_float(r[8 * v8 + 2 * e + 1]) * inv_l);
          if (slot_ok) po[(8 * half + 4 * c + v8) * kBM] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      if (half == 0 && slot_ok)
        p.part_ml[(static_cast<size_t>(slot) + split) * kBM + lrow] =
            make_float2(my_tiles > 0 && ok ? m : -INFINITY, l);
      named_bar(1, 256);  // this CTA's partial is written (CTA scope)
      if (threadIdx.x == 128 && GLANCE_IN_BOUNDS(grp, p.B * p.Hkv * p.n_qt)) {
        uint32_t* arrived = p.arrive + grp;
        if (p.ticket_merge) {
          const uint32_t before = atom_add_acq_rel_gpu(arrived, 1u);
          const bool last = before == static_cast<uint32_t>(S - 1);
          if (last) *arrived = 0u;  // every split has added: ready for the next call
          bars->ticket_last = last ? 1 : 0;
        } else {
          atom_add_release_gpu(arrived, 1u);  // cumulative release of the CTA's writes
          const uint64_t t0 = globaltimer_ns();
          bool done = false;
          for (uint32_t i = 0;; ++i) {
            if (ld_acquire_gpu(arrived) >= static_cast<uint32_t>(S)) {
              done = true;
              break;
            }
            if ((i & 63u) == 0 && globaltimer_ns() - t0 > p.wait_ns) break;
          }
          if (!done) report(GLANCE_DEV_PIPELINE_TIMEOUT);
          // the last split to leave resets both counters for the next call
          uint32_t* departed = p.arrive + p.B * p.Hkv * p.n_qt + grp;
          if (atomicAdd(departed, 1u) == static_cast<uint32_t>(S - 1)) {
            *arrived = 0u;
            *departed = 0u;
          }
        }
      }
      named_bar(1, 256);  // all splits' partials are visible (acquired above)
      if (p.ticket_merge) {
        own0 = 0;
        own_rows = 0;
        if (bars->ticket_last != 0) ticket_merge(p, bars, sQ, slot, S, qt, g, q_row0, half, lrow);
      } else {
        const int rpo = (kBM + S - 1) / S;  // rows per owner
        own0 = split * rpo;
        own_rows = own0 >= kBM ? 0 : (kBM - own0 < rpo ? kBM - own0 : rpo);
        if (!GLANCE_IN_BOUNDS(slot + S - 1, p.n_slots)) own_rows = 0;
      }
      // this CTA merges tile rows [own0, own0 + own_rows): (row, 8 dims) per
      // item, rows fastest so that neighbouring threads read neighbouring rows
      const int t = threadIdx.x - 128;
      const size_t grp_base = static_cast<size_t>(slot) * kBM;
      for (int item = t; item < own_rows * 16; item += 256) {
        const int c8 = item / own_rows, rr = item - c8 * own_rows;
        const int orow = own0 + rr;
        // every split's (m, l) and partial of this item, loaded together
        float2 mlr[kMaxSplit];
        uint4 pv[kMaxSplit];
#pragma unroll
        for (int sx = 0; sx < kMaxSplit; ++sx) {
          mlr[sx] = sx < S ? __ldcg(p.part_ml + grp_base + static_cast<size_t>(sx) * kBM + orow)
                           : make_float2(-INFINITY, 0.f);
          pv[sx] = sx < S ? __ldcg(p.part_o + ((static_cast<size_t>(slot) + sx) * 16 + c8) * kBM + orow)
                          : make_uint4(0u, 0u, 0u, 0u);
        }
        float M = -INFINITY;
#pragma unroll
        for (int sx = 0; sx < kMaxSplit; ++sx) M = fmaxf(M, mlr[sx].x);
        float Lt = 0.f, wts[kMaxSplit];
#pragma unroll
        for (int sx = 0; sx < kMaxSplit; ++sx) {
          wts[sx] = mlr[sx].x == -INFINITY ? 0.f : exp2f(mlr[sx].x - M) * mlr[sx].y;
          Lt += wts[sx];
        }
        const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int sx = 0; sx < kMaxSplit; ++sx) {
          if (sx < S && wts[sx] != 0.f) {
            const float w = wts[sx] * inv;
            const uint32_t av[4] = {pv[sx].x, pv[sx].y, pv[sx].z, pv[sx].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc[2 * e] += w * __uint_as_float(av[e] << 16);
              acc[2 * e + 1] += w * __uint_as_float(av[e] & 0xFFFF0000u);
            }
          }
        }
        const int oq = qt * kBM + orow;
        const int ohl = oq / p.Rp, oprow = oq % p.Rp;
        if (ohl < p.G && oprow < p.rows &&
            GLANCE_IN_BOUNDS((static_cast<size_t>(q_row0 + oprow) * p.Hq + g * p.G + ohl) * kD + 8 * c8 + 7,
                             static_cast<size_t>(p.B) * p.rows * p.Hq * kD)) {
          uint4 v;
          v.x = pack_bf16x2(acc[0], acc[1]);
          v.y = pack_bf16x2(acc[2], acc[3]);
          v.z = pack_bf16x2(acc[4], acc[5]);
          v.w = pack_bf16x2(acc[6], acc[7]);
          *reinterpret_cast<uint4*>(
              p.out + (static_cast<size_t>(q_row0 + oprow) * p.Hq + g * p.G + ohl) * kD + 8 * c8) = v;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // On the normal path every copy has landed and every MMA has finished (the
  // MMA thread waited for each tile's copies, the softmax threads for the
  // last product). After an abort some may still be in flight: the producer
  // waits for Q and its last kStages tiles (the only ones whose stage
  // barriers have not moved on) and the MMA thread for its products before
  // shared and tensor memory are released. Checked only here, after every
  // role is done, so that no role spins on them while the others work.
  if (*reinterpret_cast<volatile int*>(&bars->abort_flag)) {
    if (threadIdx.x == 0 && my_tiles > 0) {
      const int withhold_from = p.withhold_v ? my_tiles - 1 : my_tiles;
      (void)mbar_wait(&bars->q_full, 0, 50000000ull);
      for (int j = n_issued > kStages ? n_issued - kStages : 0; j < n_issued; ++j) {
        (void)mbar_wait(&bars->k_full[j % kStages], (j / kStages) & 1, 50000000ull);
        if (j < withhold_from || j < pre) (void)mbar_wait(&bars->v_full[j % kStages], (j / kStages) & 1, 50000000ull);
      }
    }
    if (warp == 1 && lane == 0 && my_tiles > 0) {
      mma_commit(&bars->mma_drain);
      (void)mbar_wait(&bars->mma_drain, 0, 50000000ull);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int next_pow2_at_least(int x, int lo) {
  int r = lo;
  while (r < x) r <<= 1;
  return r;
}

// Launch plan of one bf16 call over B requests.
struct Plan {
  int G, Rp, n_qt, box_rows;
  int n_split[kMaxB];
  int cta0[kMaxB + 1];
  int slot0[kMaxB];
  int ticket;            // merge mode (see Bf16Params::ticket_merge)
  size_t counters_bytes; // arrival / departure counters
  size_t slots;          // partial slots of 128 rows
  size_t ws_bytes;
};

// B == 1: one wave, one CTA per SM: S = SMs / groups key splits per group,
// cooperative merge. B > 1: ticket merge and any number of waves; request
// r's groups get S_r = ceil(tiles_r / tau) splits, tiles_r its key tiles at
// full capacity (t_cap), tau chosen so that the grid is about two waves.
Plan make_plan(int B, int rows, int Hq, const glance_kv* kv) {
  Plan pl;
  const int Hkv = kv[0].n_kv_heads;
  pl.G = Hq / Hkv;
  pl.Rp = next_pow2_at_least(rows, 32);
  pl.box_rows = pl.Rp < kBM ? pl.Rp : kBM;
  pl.n_qt = (pl.G * pl.Rp + kBM - 1) / kBM;
  const int gpr = Hkv * pl.n_qt;  // groups per request
  const int sms = glance::num_sms();
  if (B == 1) {
    const int sp = sms / gpr;
    pl.n_split[0] = sp < 1 ? 1 : (sp > kMaxSplit ? kMaxSplit : sp);
    pl.ticket = 0;
  } else {
    // Key tiles per split: the tau that minimises waves x (longest split +
    // 3), the 3 standing for a CTA's start-up (~3 tiles of work, measured:
    // on a ragged 8-request batch tau = 9 / 12 / 14 gave 70.3 / 55.2 / 51.8
    // us per layer at 416 / 352 / 288 CTAs).
    long long tau = 4, best = -1;
    for (long long tc = 4; tc <= 64; ++tc) {
      long long ctas = 0, longest = 0;
      for (int r = 0; r < B; ++r) {
        const long long tiles = (kv[r].t_cap + kBN - 1) / kBN;
        long long sp = (tiles + tc - 1) / tc;
        sp = sp < 1 ? 1 : (sp > kMaxSplit ? kMaxSplit : sp);
        ctas += static_cast<long long>(gpr) * sp;
        const long long per = (tiles + sp - 1) / sp;
        longest = per > longest ? per : longest;
      }
      const long long cost = (ctas + sms - 1) / sms * (longest + 3);
      if (best < 0 || cost < best) {
        best = cost;
        tau = tc;
      }
    }
    for (int r = 0; r < B; ++r) {
      const long long tiles = (kv[r].t_cap + kBN - 1) / kBN;
      long long sp = (tiles + tau - 1) / tau;
      pl.n_split[r] = static_cast<int>(sp < 1 ? 1 : (sp > kMaxSplit ? kMaxSplit : sp));
    }
    pl.ticket = 1;
  }
  pl.cta0[0] = 0;
  size_t slots = 0;
  for (int r = 0; r < B; ++r) {
    pl.cta0[r + 1] = pl.cta0[r] + gpr * pl.n_split[r];
    pl.slot0[r] = static_cast<int>(slots);
    if (pl.n_split[r] > 1) slots += static_cast<size_t>(gpr) * pl.n_split[r];
  }
  for (int r = B; r < kMaxB; ++r) {
    pl.n_split[r] = 1;
    pl.cta0[r + 1] = pl.cta0[B];
    pl.slot0[r] = static_cast<int>(slots);
  }
  pl.slots = slots;
  pl.counters_bytes = (2ull * B * gpr * sizeof(uint32_t) + 255) / 256 * 256;
  pl.ws_bytes = pl.counters_bytes + slots * kBM * (kD * sizeof(__nv_bfloat16) + sizeof(float2));
  return pl;
}

glance_status check_common(const void* q, int n_q_heads, const glance_kv* kv,
                           const glance_tree* tree, const void* out) {
  using glance::fail;
  if (!q || !kv || !tree || !out)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_tree_attention: null pointer argument");
  if (!kv->k || !kv->v || !kv->t_len || !tree->anc)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_tree_attention: null kv/tree array");
  const int rows = tree->n + 1;
  if (tree->n < 0 || rows > 256 || tree->mask_words != (rows + 63) / 64)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_tree_attention: need 1 <= N+1 <= 256 and "
                "mask_words = ceil((N+1)/64)");
  if (kv->n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % kv->n_kv_heads != 0)
    return fail(GLANCE_ERR_INVALID_ARG,
                "glance_tree_attention: n_q_heads must be a positive multiple of n_kv_heads");
  if (kv->t_cap < rows || kv->row_stride < kv->head_dim ||
      kv->head_stride < static_cast<int64_t>(kv->t_cap) * kv->row_stride)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_tree_attention: bad kv geometry");
  return GLANCE_OK;
}

// Checks shared by the bf16 single and batched calls.
glance_status check_bf16(const char* who, const void* q, int n_q_heads, const glance_kv* kv,
                         const glance_tree* trees, int B, const void* out) {
  using glance::fail;
  if (!q || !kv || !trees || !out)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: null pointer argument", who);
  if (B < 1 || B > kMaxB) return fail(GLANCE_ERR_INVALID_ARG, "%s: need 1 <= B <= %d", who, kMaxB);
  const int rows = trees[0].n + 1;
  for (int r = 0; r < B; ++r) {
    const glance_kv& x = kv[r];
    const glance_tree& t = trees[r];
    if (!x.k || !x.v || !x.t_len || !t.anc)
      return fail(GLANCE_ERR_INVALID_ARG, "%s: null kv/tree array (request %d)", who, r);
    if (t.n + 1 != rows || rows < 1 || rows > 256 || t.mask_words != (rows + 63) / 64)
      return fail(GLANCE_ERR_INVALID_ARG,
                  "%s: every tree needs the same N, 1 <= N+1 <= 256 and mask_words = "
                  "ceil((N+1)/64) (request %d)", who, r);
    if (x.dtype != GLANCE_BF16)
      return fail(r == 0 && B == 1 ? GLANCE_ERR_INVALID_ARG : GLANCE_ERR_UNSUPPORTED,
                  "%s: dtype must be BF16 here (request %d)", who, r);
    if (x.head_dim != kD) return fail(GLANCE_ERR_UNSUPPORTED, "%s: bf16 needs head_dim 128", who);
    if (x.n_kv_heads != kv[0].n_kv_heads || x.n_kv_heads < 1 || n_q_heads < 1 ||
        n_q_heads % x.n_kv_heads != 0)
      return fail(GLANCE_ERR_INVALID_ARG,
                  "%s: n_q_heads must be a positive multiple of n_kv_heads, the same for every "
                  "request (request %d)", who, r);
    if (x.t_cap < rows || x.row_stride < x.head_dim ||
        x.head_stride < static_cast<int64_t>(x.t_cap) * x.row_stride)
      return fail(GLANCE_ERR_INVALID_ARG, "%s: bad kv geometry (request %d)", who, r);
    if (!glance::aligned16(x.k) || !glance::aligned16(x.v) || (x.row_stride * 2) % 16 ||
        (x.head_stride * 2) % 16)
      return fail(GLANCE_ERR_INVALID_ARG,
                  "%s: k/v must be 16-byte aligned with 16-byte strides (request %d)", who, r);
    if (x.t_cap > (1 << 30)) return fail(GLANCE_ERR_UNSUPPORTED, "%s: t_cap too large", who);
  }
  const int G = n_q_heads / kv[0].n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(GLANCE_ERR_UNSUPPORTED, "%s: bf16 needs n_q_heads / n_kv_heads in {1, 2, 4, 8}",
                who);
  if (!glance::aligned16(q) || !glance::aligned16(out))
    return fail(GLANCE_ERR_INVALID_ARG, "%s: q and out must be 16-byte aligned", who);
  return GLANCE_OK;
}

template <int NB>
glance_status launch_bf16(const char* who, const void* q, int n_q_heads, const glance_kv* kv,
                          const glance_tree* trees, int B, float scale, void* out,
                          void* workspace, size_t workspace_bytes, cudaStream_t s,
                          unsigned long long wait_ns, int withhold_v) {
  using glance::fail;
  glance_status st = check_bf16(who, q, n_q_heads, kv, trees, B, out);
  if (st != GLANCE_OK) return st;
  const int rows = trees[0].n + 1;
  if (B > NB) return fail(GLANCE_ERR_INVALID_ARG, "%s: B too large", who);
  cudaError_t e = glance::ensure_smem(reinterpret_cast<const void*>(tree_attention_bf16_kernel<NB>),
                                      static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  const Plan pl = make_plan(B, rows, n_q_heads, kv);
  if (!workspace || workspace_bytes < pl.ws_bytes)
    return fail(GLANCE_ERR_CAPACITY, "%s: workspace %zu bytes < %zu needed", who, workspace_bytes,
                pl.ws_bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  CUtensorMap mq;
  KVMaps<NB> maps;
  {
    // all requests' rows stacked: [B * rows][Hq][128]
    const uint64_t dims[3] = {kD, static_cast<uint64_t>(n_q_heads),
                              static_cast<uint64_t>(B) * rows};
    const uint64_t strides[2] = {kD * 2ull, static_cast<uint64_t>(n_q_heads) * kD * 2ull};
    const uint32_t box[3] = {64, 1, static_cast<uint32_t>(pl.box_rows)};
    st = glance::make_map_bf16(&mq, q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, who);
    if (st != GLANCE_OK) return st;
  }
  for (int r = 0; r < NB; ++r) {
    const glance_kv& x = kv[r < B ? r : 0];
    const uint64_t dims[3] = {kD, static_cast<uint64_t>(x.t_cap),
                              static_cast<uint64_t>(x.n_kv_heads)};
    const uint64_t strides[2] = {static_cast<uint64_t>(x.row_stride) * 2ull,
                                 static_cast<uint64_t>(x.head_stride) * 2ull};
    const uint32_t box[3] = {64, kBN, 1};
    if (r >= B) {
      maps.k[r] = maps.k[0];
      maps.v[r] = maps.v[0];
      continue;
    }
    st = glance::make_map_bf16(&maps.k[r], x.k, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                               who);
    if (st != GLANCE_OK) return st;
    st = glance::make_map_bf16(&maps.v[r], x.v, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                               who);
    if (st != GLANCE_OK) return st;
  }
  Bf16Params<NB> p;
  for (int r = 0; r < NB; ++r) {
    const int rr = r < B ? r : 0;
    p.anc[r] = trees[rr].anc;
    p.t_len[r] = kv[rr].t_len;
    p.t_cap[r] = kv[rr].t_cap;
    p.n_split[r] = pl.n_split[r];
    p.slot0[r] = pl.slot0[r];
  }
  for (int r = 0; r <= NB; ++r) p.cta0[r] = pl.cta0[r];
  p.out = static_cast<__nv_bfloat16*>(out);
  {
    // [counters][partial O][partial (m, l)]
    char* ws = static_cast<char*>(workspace);
    p.arrive = reinterpret_cast<uint32_t*>(ws);
    p.part_o = reinterpret_cast<uint4*>(ws + pl.counters_bytes);
    p.part_ml = reinterpret_cast<float2*>(ws + pl.counters_bytes +
                                          pl.slots * kBM * kD * sizeof(__nv_bfloat16));
  }
  p.n_slots = static_cast<int>(pl.slots);
  p.B = B;
  p.rows = rows;
  p.Hq = n_q_heads;
  p.Hkv = kv[0].n_kv_heads;
  p.G = pl.G;
  p.Rp = pl.Rp;
  p.n_qt = pl.n_qt;
  p.W = trees[0].mask_words;
  p.box_rows = pl.box_rows;
  p.ticket_merge = pl.ticket;
  p.scale_log2 = scale * kLog2e;
  p.wait_ns = wait_ns;
  p.withhold_v = withhold_v;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.cta0[B]);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n_attr = 0;
  // may start while the previous kernel in the stream finishes (the kernel
  // waits for it with griddepcontrol.wait before reading its inputs)
  attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
  ++n_attr;
  if (!pl.ticket) {
    // the key splits of a group wait for each other: every CTA must be resident
    attr[n_attr].id = cudaLaunchAttributeCooperative;
    attr[n_attr].val.cooperative = 1;
    ++n_attr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  e = cudaLaunchKernelEx(&cfg, tree_attention_bf16_kernel<NB>, mq, maps, p);
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  return GLANCE_OK;
}

}  // namespace

extern "C" size_t glance_tree_attention_workspace_bytes(int n_rows, int n_q_heads,
                                                        const glance_kv* kv) {
  if (!kv || n_rows < 1 || n_rows > 256 || kv->n_kv_heads < 1 || n_q_heads < 1 ||
      n_q_heads % kv->n_kv_heads)
    return 0;
  if (kv->dtype != GLANCE_BF16) return 256;
  return make_plan(1, n_rows, n_q_heads, kv).ws_bytes;
}

extern "C" glance_status glance_tree_attention(const void* q, int n_q_heads, const glance_kv* kv,
                                               const glance_tree* tree, float scale, void* out,
                                               void* workspace, size_t workspace_bytes,
                                               void* stream) {
  using glance::fail;
  glance_status st = check_common(q, n_q_heads, kv, tree, out);
  if (st != GLANCE_OK) return st;
  const int rows = tree->n + 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kv->dtype == GLANCE_F32) {
    if (kv->head_dim < 32 || kv->head_dim > 128 || kv->head_dim % 32)
      return fail(GLANCE_ERR_UNSUPPORTED,
                  "glance_tree_attention: fp32 head_dim must be 32, 64, 96 or 128");
    F32Params p;
    p.q = static_cast<const float*>(q);
    p.k = static_cast<const float*>(kv->k);
    p.v = static_cast<const float*>(kv->v);
    p.out = static_cast<float*>(out);
    p.anc = tree->anc;
    p.t_len = kv->t_len;
    p.rows = rows;
    p.Hq = n_q_heads;
    p.Hkv = kv->n_kv_heads;
    p.D = kv->head_dim;
    p.W = tree->mask_words;
    p.t_cap = kv->t_cap;
    p.head_stride = kv->head_stride;
    p.row_stride = kv->row_stride;
    p.scale = scale;
    tree_attention_f32_kernel<<<rows * n_q_heads, kF32Threads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return glance::cuda_fail(e, "glance_tree_attention: launch");
    return GLANCE_OK;
  }
  if (kv->dtype != GLANCE_BF16)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_tree_attention: dtype must be F32 or BF16");
  return launch_bf16<1>("glance_tree_attention", q, n_q_heads, kv, tree, 1, scale, out,
                        workspace, workspace_bytes, s, kDefaultWaitNs, 0);
}

extern "C" size_t glance_tree_attention_batched_workspace_bytes(int B, int n_rows, int n_q_heads,
                                                                const glance_kv* kv) {
  if (!kv || B < 1 || B > kMaxB || n_rows < 1 || n_rows > 256 || n_q_heads < 1) return 0;
  for (int r = 0; r < B; ++r)
    if (kv[r].n_kv_heads != kv[0].n_kv_heads || kv[r].n_kv_heads < 1 ||
        n_q_heads % kv[r].n_kv_heads || kv[r].dtype != GLANCE_BF16 || kv[r].t_cap < 1)
      return 0;
  return make_plan(B, n_rows, n_q_heads, kv).ws_bytes;
}

extern "C" glance_status glance_tree_attention_batched(const void* q, int n_q_heads,
                                                       const glance_kv* kv,
                                                       const glance_tree* trees, int B,
                                                       float scale, void* out, void* workspace,
                                                       size_t workspace_bytes, void* stream) {
  return launch_bf16<kMaxB>("glance_tree_attention_batched", q, n_q_heads, kv, trees, B, scale,
                            out, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                            kDefaultWaitNs, 0);
}

extern "C" glance_status glance_tree_attention_timeout_check(
    const void* q, int n_q_heads, const glance_kv* kv, const glance_tree* tree, float scale,
    void* out, void* workspace, size_t workspace_bytes, unsigned long long wait_ns, void* stream) {
  using glance::fail;
  glance_status st = check_common(q, n_q_heads, kv, tree, out);
  if (st != GLANCE_OK) return st;
  if (kv->dtype != GLANCE_BF16)
    return fail(GLANCE_ERR_UNSUPPORTED, "glance_tree_attention_timeout_check: BF16 only");
  if (wait_ns < 1000ull || wait_ns > kDefaultWaitNs)
    return fail(GLANCE_ERR_INVALID_ARG,
                "glance_tree_attention_timeout_check: wait_ns must be in [1 us, 2 s]");
  return launch_bf16<1>("glance_tree_attention_timeout_check", q, n_q_heads, kv, tree, 1, scale,
                        out, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                        wait_ns, 1);
}
