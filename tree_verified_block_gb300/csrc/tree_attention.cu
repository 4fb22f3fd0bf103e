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
//   CTA = (kv head g, q tile of 128 query rows, key split). The 128 query rows
//   of a tile are (q head, packed row) pairs of the heads that share kv head g
//   (grouped-query attention), each head's rows padded to a power of two.
//   Warp 0 issues TMA loads (Q once, then K and V tiles of 128 slots into a
//   two-stage ring), warp 1 issues the MMAs (S = Q K^T into tensor memory,
//   then O += P V with P read from tensor memory), warps 4..7 own one query
//   row per thread: they read S from tensor memory, apply the key mask in
//   registers (the ancestor words of their row are held in registers), run
//   the online softmax in base 2, write P as bf16 into its own tensor-memory
//   columns (so the next tile's S = Q K^T never overwrites a P that the
//   previous PV has not read yet), and rescale O when the running max grows. Key splits write (O, m, l) partials and a
//   second kernel merges them; with one split the CTA normalises and writes
//   bf16 output itself.
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
      const float* kr = kh + slot * p.row_stride;
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
        a = fmaf(s_p[jj], vh[slot * p.row_stride + threadIdx.x], a);
      }
      acc = a;
    }
    m = m_new;
    __syncthreads();
  }
  if (threadIdx.x < p.D) p.out[(static_cast<size_t>(i) * p.Hq + h) * p.D + threadIdx.x] = acc / l;
}

// ------------------------------------------------------------------ bf16 path

constexpr int kD = 128;          // head_dim
constexpr int kBM = 128;         // query rows per tile (MMA M)
constexpr int kBN = 128;         // key slots per tile (MMA N of S, K of PV)
constexpr int kStages = 2;       // K/V ring depth
constexpr int kThreads = 256;    // 8 warps
constexpr int kTmemCols = 512;   // S (128) + O (128) + P (64, bf16 pairs), power of two
constexpr uint32_t kHalfBytes = kBN * 128;          // 64 head dims x 128 slots, bf16
constexpr uint32_t kQBytes = 2 * kBM * 128;         // 32 KB
constexpr uint32_t kKVStageBytes = 4 * kHalfBytes;  // K and V, two halves each: 64 KB
constexpr size_t kSmemBytes = 1024 /*align*/ + kQBytes + kStages * kKVStageBytes + 256;

struct Bf16Params {
  const uint64_t* anc;
  const int32_t* t_len;
  __nv_bfloat16* out;        // [rows][Hq][128]
  float* part_o;             // [S][Hkv][n_qt][128][128]
  float* part_ml;            // [S][Hkv][n_qt][128][2]
  int rows, Hq, Hkv, G, Rp, n_qt, n_split, W, t_cap;
  int box_rows;              // rows per Q box = min(Rp, 128)
  float scale_log2;          // scale * log2(e)
};

struct __align__(8) Bars {
  uint64_t q_full;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full;
  uint64_t p_ready;
  uint64_t o_done;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void fail_pipeline(Bars* bars) {
  report(GLANCE_DEV_PIPELINE_TIMEOUT);
  atomicExch(&bars->abort_flag, 1);
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* bars) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*reinterpret_cast<volatile int*>(&bars->abort_flag)) return false;
      if (globaltimer_ns() - t0 > 2000000000ull) return false;
    }
  }
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

__global__ void __launch_bounds__(kThreads, 1)
    tree_attention_bf16_kernel(const __grid_constant__ CUtensorMap map_q,
                               const __grid_constant__ CUtensorMap map_k,
                               const __grid_constant__ CUtensorMap map_v, const Bf16Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* sQ = smem;
  unsigned char* sKV = smem + kQBytes;
  Bars* bars = reinterpret_cast<Bars*>(sKV + kStages * kKVStageBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x % p.n_split;
  const int qt = (blockIdx.x / p.n_split) % p.n_qt;
  const int g = blockIdx.x / (p.n_split * p.n_qt);

  const int T = *p.t_len;
  const bool room = T >= 0 && T + p.rows <= p.t_cap;
  // key tiles of this split over slots [0, T + rows)
  const int n_keys = room ? T + p.rows : 0;
  const int n_tiles = (n_keys + kBN - 1) / kBN;
  const int tile0 = static_cast<int>((static_cast<long long>(n_tiles) * split) / p.n_split);
  const int tile1 = static_cast<int>((static_cast<long long>(n_tiles) * (split + 1)) / p.n_split);
  const int my_tiles = tile1 - tile0;

  if (threadIdx.x == 0) {
    if (!room && blockIdx.x == 0) report(GLANCE_DEV_TREE_CAPACITY);
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_ready, 128);
    mbar_init(&bars->o_done, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // query pieces of this tile that hold no real (head, row): zero them so the
  // MMA reads finite values
  {
    const int pieces = kBM / p.box_rows;
    for (int pc = 0; pc < pieces; ++pc) {
      const int r0 = qt * kBM + pc * p.box_rows;  // first q-row of the piece
      const int hl = r0 / p.Rp;
      if (hl >= p.G) {
        for (int half = 0; half < 2; ++half) {
          uint4* dst = reinterpret_cast<uint4*>(sQ + half * (kBM * 128) + pc * p.box_rows * 128);
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
  const uint32_t tS = tmem;         // S (fp32, 128 cols)
  const uint32_t tO = tmem + 128;   // O (fp32, 128 cols)
  const uint32_t tP = tmem + 256;   // P (bf16 pairs, 64 cols)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && my_tiles > 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      const uint64_t pol_kv = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      // Q: pieces of box_rows rows; piece pc covers q-rows qt*128 + pc*box_rows ...
      const int pieces = kBM / p.box_rows;
      int n_boxes = 0;
      for (int pc = 0; pc < pieces; ++pc) n_boxes += ((qt * kBM + pc * p.box_rows) / p.Rp < p.G) ? 2 : 0;
      mbar_arrive_expect_tx(&bars->q_full, n_boxes * p.box_rows * 128);
      for (int pc = 0; pc < pieces; ++pc) {
        const int r0 = qt * kBM + pc * p.box_rows;
        const int hl = r0 / p.Rp;
        if (hl >= p.G) continue;
        const int head = g * p.G + hl;
        const int row0 = r0 % p.Rp;
        for (int half = 0; half < 2; ++half)
          tma_load_3d(sQ + half * (kBM * 128) + pc * p.box_rows * 128, &map_q, &bars->q_full,
                      half * 64, head, row0, pol_q);
      }
      int issued = 0;
      for (int j = 0; j < my_tiles; ++j) {
        const int st = j % kStages;
        if (j >= kStages) {
          if (!wait_or_abort(&bars->kv_empty[st], ((j / kStages) - 1) & 1, bars)) {
            fail_pipeline(bars);
            break;
          }
        }
        unsigned char* stage = sKV + st * kKVStageBytes;
        ++issued;
        const int key0 = (tile0 + j) * kBN;
        mbar_arrive_expect_tx(&bars->kv_full[st], kKVStageBytes);
        tma_load_3d(stage + 0 * kHalfBytes, &map_k, &bars->kv_full[st], 0, key0, g, pol_kv);
        tma_load_3d(stage + 1 * kHalfBytes, &map_k, &bars->kv_full[st], 64, key0, g, pol_kv);
        tma_load_3d(stage + 2 * kHalfBytes, &map_v, &bars->kv_full[st], 0, key0, g, pol_kv);
        tma_load_3d(stage + 3 * kHalfBytes, &map_v, &bars->kv_full[st], 64, key0, g, pol_kv);
      }
      if (*reinterpret_cast<volatile int*>(&bars->abort_flag)) {
        // let copies already in flight land before the CTA's smem is released
        (void)mbar_wait(&bars->q_full, 0, 50000000ull);
        for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
          (void)mbar_wait(&bars->kv_full[j % kStages], (j / kStages) & 1, 50000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && my_tiles > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, kD, false, true);
      const uint32_t q_addr = smem_u32(sQ);
      bool ok = wait_or_abort(&bars->q_full, 0, bars);
      for (int j = 0; ok && j < my_tiles; ++j) {
        const int st = j % kStages;
        if (!wait_or_abort(&bars->kv_full[st], (j / kStages) & 1, bars)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_addr = smem_u32(sKV + st * kKVStageBytes);
        const uint32_t v_addr = k_addr + 2 * kHalfBytes;
        // S = Q K^T over head_dim 128 = 8 steps of 16
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
          const uint32_t offk = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          mma_bf16_ss(tS, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + offk, 16, 1024),
                      idesc_s, kk > 0);
        }
        mma_commit(&bars->s_full);
        // wait for P (and the O rescale) from the softmax warps
        if (!wait_or_abort(&bars->p_ready, j & 1, bars)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // O += P V over 128 key slots = 8 steps of 16 (8 bf16-pair columns of P each)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(tO, tP + kk * 8, sdesc_sw128(v_addr + kk * 2048, kHalfBytes, 1024), idesc_o,
                      (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->o_done);
        // only stages the producer will refill need a release
        if (j + kStages < my_tiles) mma_commit(&bars->kv_empty[st]);
      }
      if (!ok) fail_pipeline(bars);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------ softmax + epilogue
    const int quarter = warp - 4;  // TMEM lane quarter
    const int lrow = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int qrow = qt * kBM + lrow;  // index within the kv head's query rows
    const int hl = qrow / p.Rp;
    const int prow = qrow % p.Rp;
    const bool valid = hl < p.G && prow < p.rows;
    const int head = g * p.G + hl;
    uint64_t anc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int w = 0; w < 4; ++w)
      if (valid && w < p.W) anc[w] = p.anc[prow * p.W + w];
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < my_tiles; ++j) {
      const int key0 = (tile0 + j) * kBN;
      if (!wait_or_abort(&bars->s_full, j & 1, bars)) {
        ok = false;
        break;
      }
      // s_full(j) was committed after PV(j-1) was issued, so O and the P
      // columns of tile j-1 are released by now; this wait returns at once
      if (j > 0 && !wait_or_abort(&bars->o_done, (j - 1) & 1, bars)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool full = key0 + kBN <= T;  // all slots of the tile are prefix
      // this thread's S row: 128 fp32 in registers (four loads, one wait)
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld32(tS + lane_off + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32 * c));
      tmem_ld_wait();
      if (!full) {
        // slots >= T: visible only on the row's ancestor list (and < T + rows)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t vm = visible32(anc, key0 + 32 * c - T, p.rows);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            sr[32 * c + e] = ((vm >> e) & 1u) ? sr[32 * c + e] : 0xFF800000u;  // -inf
        }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int e = 0; e < kBN; e += 4) {
        mx0 = fmaxf(mx0, __uint_as_float(sr[e]));
        mx1 = fmaxf(mx1, __uint_as_float(sr[e + 1]));
        mx2 = fmaxf(mx2, __uint_as_float(sr[e + 2]));
        mx3 = fmaxf(mx3, __uint_as_float(sr[e + 3]));
      }
      // scale_log2 > 0, so the max commutes with the scaling
      const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * p.scale_log2;
      const float m_new = fmaxf(m, mt);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_use);
      // P = 2^(s * scale_log2 - m) as bf16 pairs, 16 columns per store
      const float neg_m = -m_use;
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = exp2f(fmaf(__uint_as_float(sr[32 * c + 2 * e]), p.scale_log2, neg_m));
          const float p1 = exp2f(fmaf(__uint_as_float(sr[32 * c + 2 * e + 1]), p.scale_log2, neg_m));
          ls0 += p0;
          ls1 += p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tP + lane_off + c * 16, pk);
      }
      const float ls = ls0 + ls1;
      // rescale O when the running max grew (O of tile j-1 is final)
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tO + lane_off + c * 32, r);
          tmem_ld_wait();
          uint32_t a[16], b[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            a[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            b[e] = __float_as_uint(__uint_as_float(r[16 + e]) * alpha);
          }
          tmem_st16(tO + lane_off + c * 32, a);
          tmem_st16(tO + lane_off + c * 32 + 16, b);
        }
      }
      tmem_st_wait();
      l = l * alpha + ls;
      m = m_new;
      tc_fence_before();
      mbar_arrive(&bars->p_ready);
    }
    if (ok && my_tiles > 0) {
      if (!wait_or_abort(&bars->o_done, (my_tiles - 1) & 1, bars)) ok = false;
    }
    if (!ok) fail_pipeline(bars);
    tc_fence_after();
    // epilogue
    if (ok && my_tiles > 0) {
      if (p.n_split == 1) {
        const float inv = 1.f / l;
        __nv_bfloat16* dst = p.out + (static_cast<size_t>(prow) * p.Hq + head) * kD;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tO + lane_off + c * 32, r);
          tmem_ld_wait();
          if (valid) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv, __uint_as_float(r[2 * e + 1]) * inv);
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              d4[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
      } else {
        const size_t tile_idx = (static_cast<size_t>(split) * p.Hkv + g) * p.n_qt + qt;
        float* po = p.part_o + (tile_idx * kBM + lrow) * kD;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tO + lane_off + c * 32, r);
          tmem_ld_wait();
          float4* d4 = reinterpret_cast<float4*>(po + c * 32);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            d4[v4] = make_float4(__uint_as_float(r[4 * v4]), __uint_as_float(r[4 * v4 + 1]),
                                 __uint_as_float(r[4 * v4 + 2]), __uint_as_float(r[4 * v4 + 3]));
        }
        p.part_ml[(tile_idx * kBM + lrow) * 2 + 0] = m;
        p.part_ml[(tile_idx * kBM + lrow) * 2 + 1] = l;
      }
    } else if (p.n_split > 1) {
      // empty split (or failure): a partial that contributes nothing
      const size_t tile_idx = (static_cast<size_t>(split) * p.Hkv + g) * p.n_qt + qt;
      p.part_ml[(tile_idx * kBM + lrow) * 2 + 0] = -INFINITY;
      p.part_ml[(tile_idx * kBM + lrow) * 2 + 1] = 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge split partials: one warp per query row, 4 head dims per lane; lane s
// holds split s's (m, l), so the loads of all splits are issued together.
__global__ void __launch_bounds__(128) combine_kernel(const Bf16Params p) {
  const int rows_per_cta = 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int flat = blockIdx.x * rows_per_cta + warp;  // over Hkv * n_qt * 128
  const int lrow = flat % kBM;
  const int qt = (flat / kBM) % p.n_qt;
  const int g = flat / (kBM * p.n_qt);
  if (g >= p.Hkv) return;
  const int qrow = qt * kBM + lrow;
  const int hl = qrow / p.Rp, prow = qrow % p.Rp;
  if (hl >= p.G || prow >= p.rows) return;
  const int head = g * p.G + hl;
  const size_t split_stride = static_cast<size_t>(p.Hkv) * p.n_qt * kBM;
  const size_t base = (static_cast<size_t>(g) * p.n_qt + qt) * kBM + lrow;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  float M = -INFINITY;  // max over all splits
  for (int s0 = 0; s0 < p.n_split; s0 += 32) {
    const int s = s0 + lane;
    const float ms = s < p.n_split ? __ldcg(p.part_ml + (s * split_stride + base) * 2) : -INFINITY;
    float mm = ms;
#pragma unroll
    for (int o = 16; o; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
    M = fmaxf(M, mm);
  }
  for (int s0 = 0; s0 < p.n_split; s0 += 32) {
    const int s = s0 + lane;
    float w = 0.f;
    if (s < p.n_split) {
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + s * split_stride + base);
      w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
      L += w * ml.y;
    }
    const int cnt = min(32, p.n_split - s0);
    float4 o[4];
    for (int i = 0; i < cnt; i += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i + u < cnt)
          o[u] = __ldcg(reinterpret_cast<const float4*>(p.part_o + ((s0 + i + u) * split_stride + base) * kD) + lane);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i + u < cnt) {
          const float wu = __shfl_sync(0xffffffffu, w, i + u);
          acc.x += wu * o[u].x;
          acc.y += wu * o[u].y;
          acc.z += wu * o[u].z;
          acc.w += wu * o[u].w;
        }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = 1.f / L;
  uint2 pk;
  pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *(reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(prow) * p.Hq + head) * kD) + lane) = pk;
}

int next_pow2_at_least(int x, int lo) {
  int r = lo;
  while (r < x) r <<= 1;
  return r;
}

struct Geometry {
  int G, Rp, n_qt, box_rows, n_split;
};

Geometry geometry(int rows, int Hq, int Hkv) {
  Geometry gm;
  gm.G = Hq / Hkv;
  gm.Rp = next_pow2_at_least(rows, 32);
  gm.box_rows = gm.Rp < kBM ? gm.Rp : kBM;
  gm.n_qt = (gm.G * gm.Rp + kBM - 1) / kBM;
  int s = glance::num_sms() / (Hkv * gm.n_qt);
  gm.n_split = s < 1 ? 1 : (s > 64 ? 64 : s);
  return gm;
}

size_t bf16_ws_bytes(int rows, int Hq, int Hkv) {
  const Geometry gm = geometry(rows, Hq, Hkv);
  if (gm.n_split == 1) return 256;
  const size_t tiles = static_cast<size_t>(gm.n_split) * Hkv * gm.n_qt;
  return (tiles * kBM * kD * sizeof(float) + 255) / 256 * 256 + tiles * kBM * 2 * sizeof(float) + 256;
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

}  // namespace

extern "C" size_t glance_tree_attention_workspace_bytes(int n_rows, int n_q_heads,
                                                        const glance_kv* kv) {
  if (!kv || n_rows < 1 || n_rows > 256 || kv->n_kv_heads < 1 || n_q_heads < 1 ||
      n_q_heads % kv->n_kv_heads)
    return 0;
  if (kv->dtype == GLANCE_F32) return 256;
  return bf16_ws_bytes(n_rows, n_q_heads, kv->n_kv_heads);
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
  if (kv->head_dim != kD)
    return fail(GLANCE_ERR_UNSUPPORTED, "glance_tree_attention: bf16 needs head_dim 128");
  const int G = n_q_heads / kv->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(GLANCE_ERR_UNSUPPORTED,
                "glance_tree_attention: bf16 needs n_q_heads / n_kv_heads in {1, 2, 4, 8}");
  if (!glance::aligned16(q) || !glance::aligned16(kv->k) || !glance::aligned16(kv->v) ||
      !glance::aligned16(out) || (kv->row_stride * 2) % 16 || (kv->head_stride * 2) % 16)
    return fail(GLANCE_ERR_INVALID_ARG,
                "glance_tree_attention: q/k/v/out must be 16-byte aligned with 16-byte strides");
  if (kv->t_cap > (1 << 30))
    return fail(GLANCE_ERR_UNSUPPORTED, "glance_tree_attention: t_cap too large");
  const Geometry gm = geometry(rows, n_q_heads, kv->n_kv_heads);
  const size_t need = bf16_ws_bytes(rows, n_q_heads, kv->n_kv_heads);
  if (!workspace || workspace_bytes < need)
    return fail(GLANCE_ERR_CAPACITY, "glance_tree_attention: workspace %zu bytes < %zu needed",
                workspace_bytes, need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_tree_attention: workspace must be 256-byte aligned");

  CUtensorMap mq, mk, mv;
  {
    const uint64_t dims[3] = {kD, static_cast<uint64_t>(n_q_heads), static_cast<uint64_t>(rows)};
    const uint64_t strides[2] = {kD * 2ull, static_cast<uint64_t>(n_q_heads) * kD * 2ull};
    const uint32_t box[3] = {64, 1, static_cast<uint32_t>(gm.box_rows)};
    st = glance::make_map_bf16(&mq, q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                               "glance_tree_attention: q map");
    if (st != GLANCE_OK) return st;
  }
  {
    const uint64_t dims[3] = {kD, static_cast<uint64_t>(kv->t_cap),
                              static_cast<uint64_t>(kv->n_kv_heads)};
    const uint64_t strides[2] = {static_cast<uint64_t>(kv->row_stride) * 2ull,
                                 static_cast<uint64_t>(kv->head_stride) * 2ull};
    const uint32_t box[3] = {64, kBN, 1};
    st = glance::make_map_bf16(&mk, kv->k, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                               "glance_tree_attention: k map");
    if (st != GLANCE_OK) return st;
    st = glance::make_map_bf16(&mv, kv->v, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                               "glance_tree_attention: v map");
    if (st != GLANCE_OK) return st;
  }
  Bf16Params p;
  p.anc = tree->anc;
  p.t_len = kv->t_len;
  p.out = static_cast<__nv_bfloat16*>(out);
  const size_t tiles = static_cast<size_t>(gm.n_split) * kv->n_kv_heads * gm.n_qt;
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                       (tiles * kBM * kD * sizeof(float) + 255) / 256 * 256);
  p.rows = rows;
  p.Hq = n_q_heads;
  p.Hkv = kv->n_kv_heads;
  p.G = gm.G;
  p.Rp = gm.Rp;
  p.n_qt = gm.n_qt;
  p.n_split = gm.n_split;
  p.W = tree->mask_words;
  p.t_cap = kv->t_cap;
  p.box_rows = gm.box_rows;
  p.scale_log2 = scale * kLog2e;
  cudaError_t e = glance::ensure_smem(reinterpret_cast<const void*>(tree_attention_bf16_kernel), static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return glance::cuda_fail(e, "glance_tree_attention: smem attribute");
  const int grid = kv->n_kv_heads * gm.n_qt * gm.n_split;
  tree_attention_bf16_kernel<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return glance::cuda_fail(e, "glance_tree_attention: launch");
  if (gm.n_split > 1) {
    const int total_rows = kv->n_kv_heads * gm.n_qt * kBM;
    combine_kernel<<<(total_rows + 3) / 4, 128, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return glance::cuda_fail(e, "glance_tree_attention: combine launch");
  }
  return GLANCE_OK;
}
