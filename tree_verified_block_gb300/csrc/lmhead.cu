// LM head with fused greedy argmax and top-2 gap.
//
// Paper: "Vision Is Not Overhead ..." (arXiv 2609.00355), Section 3.1
// (greedy decoding emits argmax_w p(w | prefix)) and Theorem 1's full
// statement in Appendix B.1 (top logit gap gamma = l_(1) - l_(2), the margin
// the tie-aware gate of Section 4.2 reads).
//
// logits[i][v] = sum_k h[i][k] W[k][v]; per row: argmax (lowest id among
// equal maxima), gap = max - (largest logit of any other id), max. The logits
// never leave the chip.
//
// bf16 path (tcgen05), M <= 128: persistent CTAs, one per SM, each walking
// vocabulary tiles of 256 columns. Warp 0 streams h (K-major, 128-byte swizzle) and W
// ([d][V] row-major, so V is the MN-major side of the B operand) through a
// 4-stage TMA ring; warp 1 issues M=128 x N=256 x K=16 MMAs into one of two
// tensor-memory accumulators; warps 4..7 each own one row (one TMEM lane),
// read the tile's 256 fp32 logits and fold them into a running
// (max, argmax, second max) held in registers across tiles, while the MMA
// warp fills the other accumulator. CTAs write per-row partials; the last CTA
// (atomic ticket) merges them, lanes over rows. M > 128 (rows of several
// requests stacked, up to 512): clusters of two CTAs split the rows and share
// each W tile through TMA multicast, one launch, W read from HBM once.
// fp32 path: CUDA cores, 128 vocabulary columns x 8 rows per CTA.
//
// Sampling mode (Section 5.4: under sampling the committed token is a draw
// from the target's own verified row): the same kernels fold l / T + g
// instead of l, g = -ln(-ln u) Gumbel noise from the counter-based generator
// Philox4x32-10 (Salmon et al., SC 2011). Column v of the row predicting
// absolute position pos of stream seq uses counter (v / 4, pos, seq, 0), key
// (seed low, seed high) and output word v % 4; u = (top 23 bits + 1/2) / 2^23.
// The argmax is then a draw from softmax(l / T), and since the noise depends
// on the predicted position only, tree rounds reproduce sampled
// autoregression of the same seed.
#include <mutex>

#include "glance_internal.cuh"

GLANCE_DEFINE_STATUS_WORD(status_lmhead)

using namespace glance_dev;

namespace {

struct Partial {
  float m1;
  int i1;
  float m2;
};

__device__ __forceinline__ void merge(Partial& a, const Partial& b) {
  if (b.m1 > a.m1 || (b.m1 == a.m1 && b.i1 < a.i1)) {
    a.m2 = fmaxf(b.m2, a.m1);
    a.m1 = b.m1;
    a.i1 = b.i1;
  } else {
    a.m2 = fmaxf(a.m2, b.m1);
  }
}

// With the entropy: s = sum_v exp(l_v - m1) and u = sum_v exp(l_v - m1) (l_v - m1)
// over the columns seen, relative to the running maximum m1; the row's entropy
// is then H = log s - u / s.
struct PartialH {
  float m1;
  int i1;
  float m2;
  float s;
  float u;
};

template <typename P>
__device__ __forceinline__ P neutral_partial();
template <>
__device__ __forceinline__ Partial neutral_partial<Partial>() {
  return Partial{-INFINITY, 0x7FFFFFFF, -INFINITY};
}
template <>
__device__ __forceinline__ PartialH neutral_partial<PartialH>() {
  return PartialH{-INFINITY, 0x7FFFFFFF, -INFINITY, 0.f, 0.f};
}

constexpr float kLog2e = 1.4426950408889634f;

// What the bf16 kernels fold per row.
constexpr int kGreedy = 0;   // argmax, gap, max of the logits
constexpr int kEntropy = 1;  // ... and the softmax entropy
constexpr int kSample = 2;   // argmax and gap of l / T + Gumbel noise

// Philox4x32-10: ten rounds of two 32x32 -> 64-bit products; the key advances
// by the Weyl increments (2^32 / golden ratio, 2^32 (sqrt 3 - 1)) per round.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += kW0;
      k1 += kW1;
    }
    // each 32 x 32 -> 64-bit product as one wide multiply
    const unsigned long long p0 = static_cast<unsigned long long>(c.x) * kM0;
    const unsigned long long p1 = static_cast<unsigned long long>(c.z) * kM1;
    const uint32_t lo0 = static_cast<uint32_t>(p0), hi0 = static_cast<uint32_t>(p0 >> 32);
    const uint32_t lo1 = static_cast<uint32_t>(p1), hi1 = static_cast<uint32_t>(p1 >> 32);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Gumbel noise from one 32-bit word: u = (k + 1/2) / 2^23 in (0, 1), k = the
// top 23 bits. The inner log needs relative accuracy near u = 1, where -ln u
// is tiny and decides the largest noise values; the outer one only absolute
// accuracy. With t = 1 - u = (2^23 - 1/2 - k) / 2^23 (exact in fp32): for
// t < 1/32 the Taylor series -ln(1 - t) = t + t^2/2 + t^3/3 + t^4/4 + t^5/5
// (relative error below t^5 / 6 < 6e-9); elsewhere -ln u > 1/32 and the
// hardware logarithm's absolute error (~1e-7) is below 4e-6 relative.
__device__ __forceinline__ float gumbel_of(uint32_t w) {
  const float k = static_cast<float>(w >> 9);
  const float u = (k + 0.5f) * (1.0f / 8388608.0f);
  const float t = (8388607.5f - k) * (1.0f / 8388608.0f);
  const float series = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 0.2f, 0.25f), 1.0f / 3.0f), 0.5f), 1.0f);
  const float nl = t < 0.03125f ? series : -__logf(u);
  return -__logf(nl);
}

// Replaces the 32 logits of columns col0.. (col0 % 4 == 0) of one row by
// l / T + g (sampling mode).
__device__ __forceinline__ void perturb_chunk(uint32_t (&r)[32], int col0, float inv_temp,
                                              uint32_t pos, uint32_t seq, uint32_t k0,
                                              uint32_t k1) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(col0 / 4 + q), pos, seq, 0u), k0, k1);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      r[4 * q + j] = __float_as_uint(fmaf(__uint_as_float(r[4 * q + j]), inv_temp, gumbel_of(ws[j])));
  }
}

// Re-expresses (s, u) relative to a new maximum M >= m.
__device__ __forceinline__ void rebase(float m, float M, float& s, float& u) {
  if (m == -INFINITY) {
    s = 0.f;
    u = 0.f;
    return;
  }
  const float f = expf(m - M);
  u = f * (u + s * (m - M));
  s *= f;
}

__device__ __forceinline__ void merge(PartialH& a, const PartialH& b) {
  const float M = fmaxf(a.m1, b.m1);
  float sa = a.s, ua = a.u, sb = b.s, ub = b.u;
  rebase(a.m1, M, sa, ua);
  rebase(b.m1, M, sb, ub);
  Partial pa{a.m1, a.i1, a.m2};
  merge(pa, Partial{b.m1, b.i1, b.m2});
  a = PartialH{pa.m1, pa.i1, pa.m2, sa + sb, ua + ub};
}

// Folds one chunk of 32 logits (columns col0.., valid below V) into the
// entropy sums; m is the running maximum after this chunk, hm the maximum the
// sums are relative to.
__device__ __forceinline__ void entropy_chunk(const uint32_t (&r)[32], int col0, int V, float m,
                                              float& hm, float& hs, float& hu) {
  if (m > hm) {
    if (hm != -INFINITY) {
      const float f = ex2_approx((hm - m) * kLog2e);
      hu = f * (hu + hs * (hm - m));
      hs *= f;
    }
    hm = m;
  }
  const int n = V - col0;
  // independent terms, summed as a tree (the epilogue runs one warp per
  // scheduler, so long dependent chains would be latency-bound)
  float ps[32], pu[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const bool ok = e < n;
    const float dx = ok ? __uint_as_float(r[e]) - hm : 0.f;
    const float pe = ok ? ex2_approx(dx * kLog2e) : 0.f;
    ps[e] = pe;
    pu[e] = pe * dx;
  }
#pragma unroll
  for (int w = 16; w; w >>= 1)
#pragma unroll
    for (int e = 0; e < w; ++e) {
      ps[e] += ps[e + w];
      pu[e] += pu[e + w];
    }
  hs += ps[0];
  hu += pu[0];
}

// Folds 32 logits of columns col0.. (valid below V) into the running
// (max, argmax, second max). The chunk is reduced as a tree first: its max,
// the lowest column holding it, and the largest other value; then merged
// (columns arrive in increasing order, so an equal maximum keeps the earlier
// id).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of 32 values as a tree of three-input maxima (17 instructions).
__device__ __forceinline__ float max32(const float (&x)[32]) {
  float t[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) t[i] = max3f(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
  t[10] = fmaxf(x[30], x[31]);
  const float u0 = max3f(t[0], t[1], t[2]), u1 = max3f(t[3], t[4], t[5]), u2 = max3f(t[6], t[7], t[8]);
  return fmaxf(max3f(u0, u1, u2), fmaxf(t[9], t[10]));
}

__device__ __forceinline__ void fold_chunk(const uint32_t (&r)[32], int col0, int V, float& m1,
                                           int& i1, float& m2) {
  const int n = V - col0;
  float x[32];
  if (n >= 32) {  // every chunk but a row's last
#pragma unroll
    for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]);
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) x[e] = e < n ? __uint_as_float(r[e]) : -INFINITY;
  }
  const float cm = max32(x);
  if (!(cm > m2)) return;  // nothing in the chunk changes the top two
  uint32_t hit = 0;
#pragma unroll
  for (int e = 0; e < 32; ++e) hit |= (x[e] == cm ? 1u : 0u) << e;
  const int ci = __ffs(static_cast<int>(hit)) - 1;
  float y[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) y[e] = e == ci ? -INFINITY : x[e];
  const float c2 = max32(y);
  if (cm > m1) {
    m2 = fmaxf(m1, c2);
    m1 = cm;
    i1 = col0 + ci;
  } else {
    m2 = fmaxf(m2, cm);
  }
}

__device__ __forceinline__ Partial load_partial(const Partial* q) {
  return Partial{__ldcg(&q->m1), __ldcg(&q->i1), __ldcg(&q->m2)};
}
__device__ __forceinline__ PartialH load_partial(const PartialH* q) {
  return PartialH{__ldcg(&q->m1), __ldcg(&q->i1), __ldcg(&q->m2), __ldcg(&q->s), __ldcg(&q->u)};
}

// Last CTA: merges every CTA's partial of each row (part[c * part_stride + r]).
// One CTA's partials are contiguous over rows, so lane i of a warp takes row
// 32 b + i of a row block b and each step's 32 loads are one contiguous run.
// The warps split the row blocks and, when there are fewer row blocks than
// warps, the CTAs too (groups); each thread issues 8 loads before it folds
// them, so the whole merge costs a few L2 round trips. The groups meet in
// `scratch` (shared memory, blockDim / 32 x 32 partials). Every fold is a
// top-2 with lowest-id ties, so the argmax, gap and maximum do not depend on
// the order; the entropy sums are rebased to the running maximum at each fold.
template <typename P, typename Out>
__device__ void merge_rows(const P* part, int n_parts, int part_stride, int M, P* scratch, Out out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int n_rb = (M + 31) / 32;
  for (int rb0 = 0; rb0 < n_rb; rb0 += nwarps) {
    const int nb = n_rb - rb0 < nwarps ? n_rb - rb0 : nwarps;  // row blocks of this pass
    const int groups = nwarps / nb;
    const int rbl = warp % nb, grp = warp / nb;
    const int r = (rb0 + rbl) * 32 + lane;
    P a = neutral_partial<P>();
    if (grp < groups && r < M) {
      for (int c0 = grp; c0 < n_parts; c0 += 8 * groups) {
        P b[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = c0 + u * groups;
          b[u] = c < n_parts ? load_partial(part + static_cast<size_t>(c) * part_stride + r) : neutral_partial<P>();
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) merge(a, b[u]);
      }
    }
    scratch[warp * 32 + lane] = a;
    __syncthreads();
    if (grp == 0 && r < M) {
      for (int gi = 1; gi < groups; ++gi) merge(a, scratch[(gi * nb + rbl) * 32 + lane]);
      out(r, a);
    }
    __syncthreads();
  }
}

__device__ void merge_partials_h(const PartialH* part, int n_parts, int part_stride, int M, PartialH* scratch,
                                 int32_t* argmax, float* gap, float* maxlogit, float* entropy) {
  merge_rows(part, n_parts, part_stride, M, scratch, [&](int r, const PartialH& a) {
    argmax[r] = a.i1;
    gap[r] = a.m1 - a.m2;
    if (maxlogit) maxlogit[r] = a.m1;
    entropy[r] = logf(a.s) - a.u / a.s;
  });
}

__device__ void merge_partials(const Partial* part, int n_parts, int part_stride, int M, Partial* scratch,
                               int32_t* argmax, float* gap, float* maxlogit) {
  merge_rows(part, n_parts, part_stride, M, scratch, [&](int r, const Partial& a) {
    argmax[r] = a.i1;
    gap[r] = a.m1 - a.m2;
    if (maxlogit) maxlogit[r] = a.m1;
  });
}

// ------------------------------------------------------------------ fp32 path

constexpr int kF32Cols = 128;
constexpr int kF32Rows = 8;
constexpr int kF32KChunk = 256;

struct F32Params {
  const float* h;
  const float* W;
  int M, d, V;
  int32_t* argmax;
  float* gap;
  float* maxlogit;
  Partial* part;  // [n_colblk][M]
  uint32_t* ticket;
  // sampling mode when position != null: fold l / T + Gumbel noise
  const int32_t* position;
  const int32_t* seq;
  float inv_temp;
  uint32_t seed_lo, seed_hi;
};

__global__ void __launch_bounds__(kF32Cols) lmhead_f32_kernel(const F32Params p) {
  __shared__ float s_h[kF32Rows][kF32KChunk];
  __shared__ Partial s_red[kF32Cols / 32][kF32Rows];
  __shared__ uint32_t s_ticket;
  const int colblk = blockIdx.x, rowgrp = blockIdx.y;
  const int v = colblk * kF32Cols + threadIdx.x;
  const int r0 = rowgrp * kF32Rows;
  float acc[kF32Rows];
#pragma unroll
  for (int r = 0; r < kF32Rows; ++r) acc[r] = 0.f;
  for (int k0 = 0; k0 < p.d; k0 += kF32KChunk) {
    const int kn = min(kF32KChunk, p.d - k0);
    __syncthreads();
    for (int i = threadIdx.x; i < kF32Rows * kF32KChunk; i += kF32Cols) {
      const int r = i / kF32KChunk, k = i % kF32KChunk;
      s_h[r][k] = (r0 + r < p.M && k < kn) ? p.h[static_cast<size_t>(r0 + r) * p.d + k0 + k] : 0.f;
    }
    __syncthreads();
    if (v < p.V) {
      for (int k = 0; k < kn; ++k) {
        const float w = p.W[static_cast<size_t>(k0 + k) * p.V + v];
#pragma unroll
        for (int r = 0; r < kF32Rows; ++r) acc[r] = fmaf(s_h[r][k], w, acc[r]);
      }
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (p.position && v < p.V) {
#pragma unroll
    for (int r = 0; r < kF32Rows; ++r) {
      if (r0 + r < p.M) {
        const uint32_t pos = static_cast<uint32_t>(p.position[r0 + r]);
        const uint32_t sq = p.seq ? static_cast<uint32_t>(p.seq[r0 + r]) : 0u;
        const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(v / 4), pos, sq, 0u),
                                      p.seed_lo, p.seed_hi);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        acc[r] = fmaf(acc[r], p.inv_temp, gumbel_of(ws[v & 3]));
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kF32Rows; ++r) {
    Partial a{v < p.V ? acc[r] : -INFINITY, v < p.V ? v : 0x7FFFFFFF, -INFINITY};
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      Partial b{__shfl_xor_sync(0xffffffffu, a.m1, o), __shfl_xor_sync(0xffffffffu, a.i1, o),
                __shfl_xor_sync(0xffffffffu, a.m2, o)};
      merge(a, b);
    }
    if (lane == 0) s_red[warp][r] = a;
  }
  __syncthreads();
  if (threadIdx.x < kF32Rows && r0 + threadIdx.x < p.M) {
    Partial a = s_red[0][threadIdx.x];
    for (int w = 1; w < kF32Cols / 32; ++w) merge(a, s_red[w][threadIdx.x]);
    const size_t at = static_cast<size_t>(colblk) * p.M + r0 + threadIdx.x;
    if (GLANCE_IN_BOUNDS(at, static_cast<size_t>(gridDim.x) * p.M)) p.part[at] = a;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_ticket = atomicAdd(p.ticket, 1u);
  __syncthreads();
  if (s_ticket != gridDim.x * gridDim.y - 1) return;
  __threadfence();
  if (threadIdx.x == 0) *p.ticket = 0;
  __shared__ Partial s_merge[kF32Cols];  // one per thread
  merge_partials(p.part, gridDim.x, p.M, p.M, s_merge, p.argmax, p.gap, p.maxlogit);
}

// ------------------------------------------------------------------ bf16 path

constexpr int kBM = 128;   // rows per MMA (M), padded with zero rows
constexpr int kBK = 64;    // one 128-byte swizzle atom of K
constexpr int kThreads = 256;
constexpr uint32_t kABytes = kBM * kBK * 2;    // one row block's K slice: 16 KB
constexpr uint32_t kWBoxBytes = kBK * 64 * 2;  // one 64 x 64 box of W: 8 KB

// Tile shape of the single-CTA kernel by the number NB of 128-row blocks of
// h it multiplies with each W stage (the library launches it with NB = 1, M
// <= 128: BN 256, 4 stages of 48 KB, two accumulator sets of 256 columns so
// the epilogue drains one while the MMA warp fills the other; larger M runs
// on CTA pairs, below).
template <int NB>
struct Shape {
  static constexpr int BN = NB == 1 ? 256 : 128;
  static constexpr int STAGES = NB <= 2 ? 4 : (NB == 3 ? 3 : 2);
  static constexpr int NBUF = NB <= 2 ? 2 : 1;
  static constexpr uint32_t kBBytes = kBK * BN * 2;
  static constexpr uint32_t kStageBytes = NB * kABytes + kBBytes;
  static constexpr size_t kSmem = 1024 + STAGES * kStageBytes + 256;
  static_assert(NB * BN * NBUF <= 512, "tensor memory");
  static_assert(kSmem <= 232448, "shared memory");
};

struct Bf16Params {
  int M, d, V, n_tiles, a_rows;  // a_rows: rows a TMA box of h writes (NB = 1)
  int32_t* argmax;
  float* gap;
  float* maxlogit;
  void* part;       // [grid][rows] Partial, or PartialH with the entropy
  uint32_t* ticket;
  float* entropy;   // [M], written by the kMode == kEntropy kernels
  // sampling mode
  float inv_temp;
  uint32_t seed_lo, seed_hi;
  const int32_t* position;  // [M] absolute position of the token each row predicts
  const int32_t* seq;       // [M] stream of each row, or null (0)
  // W packed as stage images (glance_lmhead_pack_w; NB = 1 only), or null:
  // W through its tensor map
  const unsigned char* w_packed;
};

// One contiguous copy of a packed W stage, evict-first in L2 like the
// tensor-map copies of W.
__device__ __forceinline__ void bulk_copy_g2s_evict_first(void* dst, const void* src, uint32_t bytes,
                                                          uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

template <int STAGES>
struct __align__(8) Bars {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int abort_flag;
};

template <typename BarsT>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, BarsT* bars) {
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

template <typename BarsT>
__device__ __forceinline__ void fail_pipeline(BarsT* bars) {
  report(GLANCE_DEV_PIPELINE_TIMEOUT);
  atomicExch(&bars->abort_flag, 1);
}

template <int NB, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_bf16_kernel(const __grid_constant__ CUtensorMap map_h,
                       const __grid_constant__ CUtensorMap map_w, const Bf16Params p) {
  using Sh = Shape<NB>;
  constexpr int BN = Sh::BN, STAGES = Sh::STAGES, NBUF = Sh::NBUF;
  constexpr bool kH = kMode == kEntropy, kS = kMode == kSample;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // stage s: NB A slices (16 KB each), then the W slice
  Bars<STAGES>* bars = reinterpret_cast<Bars<STAGES>*>(smem + STAGES * Sh::kStageBytes);
  __shared__ uint32_t s_ticket;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_kb = p.d / kBK;
  const int my_tiles = (p.n_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                       static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->acc_full[b], 1);
      mbar_init(&bars->acc_empty[b], 128);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  // NB = 1: rows a_rows..127 of every A stage stay zero (TMA only writes a_rows rows)
  if (NB == 1 && p.a_rows < kBM) {
    for (int s = 0; s < STAGES; ++s) {
      uint4* dst = reinterpret_cast<uint4*>(smem + s * Sh::kStageBytes + p.a_rows * 128);
      for (int i = threadIdx.x; i < (kBM - p.a_rows) * 8; i += kThreads) dst[i] = make_uint4(0, 0, 0, 0);
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // W does not depend on the previous kernel in the stream: the first stages'
  // W slices go out before the programmatic-dependent-launch wait, h after it
  const uint32_t a_bytes = NB == 1 ? static_cast<uint32_t>(p.a_rows) * kBK * 2 : NB * kABytes;
  const int n_pre = my_tiles * n_kb < STAGES ? my_tiles * n_kb : STAGES;
  // W slice (tile, kb) of one stage: four tensor-map boxes of 64 x 64, or one
  // contiguous copy of the same shared-memory image when W is packed
  auto load_w = [&](unsigned char* stage, uint64_t* bar, int tile, int kb, uint64_t pol) {
    if (NB == 1 && p.w_packed != nullptr) {
      bulk_copy_g2s_evict_first(stage + NB * kABytes,
                                p.w_packed + (static_cast<size_t>(tile) * n_kb + kb) * Sh::kBBytes,
                                Sh::kBBytes, bar, pol);
    } else {
#pragma unroll
      for (int q = 0; q < BN / 64; ++q)
        tma_load_2d(stage + NB * kABytes + q * kWBoxBytes, &map_w, bar, tile * BN + 64 * q, kb * kBK, pol);
    }
  };
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_h);
    if (p.w_packed == nullptr) tma_prefetch_desc(&map_w);
    const uint64_t pol_w = policy_evict_first();
    for (int it = 0; it < n_pre; ++it) {
      const int tile = blockIdx.x + (it / n_kb) * gridDim.x, kb = it % n_kb;
      unsigned char* stage = smem + it * Sh::kStageBytes;
      mbar_arrive_expect_tx(&bars->full[it], a_bytes + Sh::kBBytes);
      load_w(stage, &bars->full[it], tile, kb, pol_w);
    }
  }
  pdl_wait_prior();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      // NB > 1: boxes of 128 rows; rows past M are filled with zeros by TMA
      int it = 0;
      bool ok = true;
      for (int i = 0; ok && i < my_tiles; ++i) {
        const int tile = blockIdx.x + i * gridDim.x;
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % STAGES;
          unsigned char* stage = smem + st * Sh::kStageBytes;
          if (it >= n_pre) {
            if (it >= STAGES && !wait_or_abort(&bars->empty[st], ((it / STAGES) - 1) & 1, bars)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars->full[st], a_bytes + Sh::kBBytes);
            load_w(stage, &bars->full[st], tile, kb, pol_w);
          }
#pragma unroll
          for (int b = 0; b < NB; ++b)
            tma_load_2d(stage + b * kABytes, &map_h, &bars->full[st], kb * kBK, b * kBM, pol_h);
        }
      }
      if (!ok) {
        fail_pipeline(bars);
        for (int j = it > STAGES ? it - STAGES : 0; j < it; ++j)
          (void)mbar_wait(&bars->full[j % STAGES], (j / STAGES) & 1, 50000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN, false, true);
      const uint32_t s0 = smem_u32(smem);
      int it = 0;
      bool ok = true;
      const int total_it = my_tiles * n_kb;
      for (int i = 0; ok && i < my_tiles; ++i) {
        const int buf = NBUF == 2 ? (i & 1) : 0;
        const int use = NBUF == 2 ? (i >> 1) : i;  // earlier uses of this accumulator set
        if (use >= 1 && !wait_or_abort(&bars->acc_empty[buf], (use - 1) & 1, bars)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * (NB * BN);
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % STAGES;
          if (!wait_or_abort(&bars->full[st], (it / STAGES) & 1, bars)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st_addr = s0 + st * Sh::kStageBytes;
          const uint32_t b_addr = st_addr + NB * kABytes;
#pragma unroll
          for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              mma_bf16_ss(d_tmem + b * BN, sdesc_sw128(st_addr + b * kABytes + k * 32, 16, 1024),
                          sdesc_sw128(b_addr + k * 2048, kWBoxBytes, 1024), idesc,
                          (kb > 0 || k > 0) ? 1u : 0u);
          // only stages the producer will refill need a release
          if (it + STAGES < total_it) mma_commit(&bars->empty[st]);
        }
        if (!ok) break;
        mma_commit(&bars->acc_full[buf]);
      }
      if (!ok) fail_pipeline(bars);
    }
  } else if (warp >= 4) {
    const int quarter = warp - 4;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float m1[NB], m2[NB], hm[NB], hs[NB], hu[NB];
    int i1[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      m1[b] = -INFINITY;
      m2[b] = -INFINITY;
      i1[b] = 0x7FFFFFFF;
      hm[b] = -INFINITY;
      hs[b] = 0.f;
      hu[b] = 0.f;
    }
    // sampling: each of this thread's rows' predicted position and stream
    uint32_t spos[NB], sseq[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const int gr = b * kBM + row;
      spos[b] = (kS && gr < p.M) ? static_cast<uint32_t>(p.position[gr]) : 0u;
      sseq[b] = (kS && gr < p.M && p.seq) ? static_cast<uint32_t>(p.seq[gr]) : 0u;
    }
    bool ok = true;
    for (int i = 0; i < my_tiles; ++i) {
      const int buf = NBUF == 2 ? (i & 1) : 0;
      const int use = NBUF == 2 ? (i >> 1) : i;
      if (!wait_or_abort(&bars->acc_full[buf], use & 1, bars)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int v0 = (blockIdx.x + i * gridDim.x) * BN;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const uint32_t t_acc = tmem + buf * (NB * BN) + b * BN + lane_off;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(t_acc + c * 32, r);
          tmem_ld_wait();
          const int col0 = v0 + c * 32;
          if (kS) perturb_chunk(r, col0, p.inv_temp, spos[b], sseq[b], p.seed_lo, p.seed_hi);
          fold_chunk(r, col0, p.V, m1[b], i1[b], m2[b]);
          if (kH) entropy_chunk(r, col0, p.V, m1[b], hm[b], hs[b], hu[b]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->acc_empty[buf]);
    }
    if (!ok) fail_pipeline(bars);
#pragma unroll
    for (int b = 0; b < NB; ++b)
      if (b * kBM + row < p.M) {
        const size_t at = static_cast<size_t>(blockIdx.x) * (NB * kBM) + b * kBM + row;
        if (!GLANCE_IN_BOUNDS(at, static_cast<size_t>(gridDim.x) * (NB * kBM))) continue;
        if (kH)
          static_cast<PartialH*>(p.part)[at] = PartialH{m1[b], i1[b], m2[b], hs[b], hu[b]};
        else
          static_cast<Partial*>(p.part)[at] = Partial{m1[b], i1[b], m2[b]};
      }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // this CTA's part is done: the next kernel in the stream (the acceptance
  // walk) may launch and wait for the merge at its dependency wait
  pdl_launch_dependents();
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_ticket = atomicAdd(p.ticket, 1u);
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;
  __threadfence();
  if (threadIdx.x == 0) *p.ticket = 0;
  // the stage ring is idle now: it holds the merge's scratch
  if (kH)
    merge_partials_h(static_cast<const PartialH*>(p.part), gridDim.x, NB * kBM, p.M,
                     reinterpret_cast<PartialH*>(smem), p.argmax, p.gap, p.maxlogit, p.entropy);
  else
    merge_partials(static_cast<const Partial*>(p.part), gridDim.x, NB * kBM, p.M,
                   reinterpret_cast<Partial*>(smem), p.argmax, p.gap, p.maxlogit);
}

// ---------------------------------------------- bf16, M > 128: CTA pairs
//
// Rows 0..M-1 are split over the two CTAs of a cluster (rank 0: the first
// NB * 128 rows, rank 1: the next NB * 128); both walk the same vocabulary
// tiles of 256 columns in lockstep. Each loads its own rows of h and one half
// of the W tile, which it multicasts to both CTAs, so every W byte leaves L2
// once per pair and each SM requests NB * 16 + 16 KB per K slice instead of
// NB * 32 + 32 KB. A stage is refilled only when both CTAs' MMAs are done with
// it: the MMA warps' commits arrive on the stage's empty barrier in both CTAs.
//   NB = 1 (M <= 256): 4 stages of 48 KB, 2 accumulator sets of 256 columns
//   NB = 2 (M <= 512): 3 stages of 64 KB, 1 accumulator set of 2 x 256
template <int NB>
struct PairShape {
  static constexpr int BN = 256;
  static constexpr int STAGES = NB == 1 ? 4 : 3;
  static constexpr int NBUF = NB == 1 ? 2 : 1;
  static constexpr uint32_t kBBytes = kBK * BN * 2;
  static constexpr uint32_t kStageBytes = NB * kABytes + kBBytes;
  static constexpr size_t kSmem = 1024 + STAGES * kStageBytes + 256;
  // epilogue warpgroups: with one accumulator set (NB = 2) the MMAs of the
  // next tile wait for the whole fold, so each row block gets its own
  // warpgroup (two epilogue warps per scheduler, half the fold each). Four
  // (a column half each) measured slower: 512 threads cap registers at 128.
  static constexpr int EPI = NB == 2 ? 2 : 1;
  static constexpr int CH = EPI / NB > 0 ? EPI / NB : 1;  // column groups per row block
  static constexpr int kThreads = 128 + 128 * EPI;
  static_assert(NB * BN * NBUF <= 512, "tensor memory");
  static_assert(kSmem <= 232448, "shared memory");
};

template <int NB, int kMode>
__global__ void __launch_bounds__(PairShape<NB>::kThreads, 1)
    lmhead_bf16_pair_kernel(const __grid_constant__ CUtensorMap map_h,
                            const __grid_constant__ CUtensorMap map_w, const Bf16Params p) {
  using Sh = PairShape<NB>;
  constexpr int BN = Sh::BN, STAGES = Sh::STAGES, NBUF = Sh::NBUF;
  constexpr uint16_t kBoth = 0x3;
  constexpr bool kH = kMode == kEntropy, kS = kMode == kSample;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars<STAGES>* bars = reinterpret_cast<Bars<STAGES>*>(smem + STAGES * Sh::kStageBytes);
  __shared__ uint32_t s_ticket;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const int row0 = rank * NB * kBM;  // this CTA's first row of h
  const int n_kb = p.d / kBK;
  const int my_tiles = (p.n_tiles - pair + n_pairs - 1) / n_pairs;  // same for both CTAs

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 2);  // both CTAs' MMA warps release a stage
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->acc_full[b], 1);
      mbar_init(&bars->acc_empty[b], 128 * Sh::EPI);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  // both CTAs' barriers exist before either multicasts into the other
  __syncwarp();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&map_h);
      tma_prefetch_desc(&map_w);
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      int it = 0;
      bool ok = true;
      for (int i = 0; ok && i < my_tiles; ++i) {
        const int v0 = (pair + i * n_pairs) * BN;
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % STAGES;
          if (it >= STAGES && !wait_or_abort(&bars->empty[st], ((it / STAGES) - 1) & 1, bars)) {
            ok = false;
            break;
          }
          unsigned char* stage = smem + st * Sh::kStageBytes;
          // own rows of h (rows past M read as zeros) + the whole W slice, half of
          // which the peer multicasts here
          mbar_arrive_expect_tx(&bars->full[st], NB * kABytes + Sh::kBBytes);
#pragma unroll
          for (int b = 0; b < NB; ++b)
            tma_load_2d(stage + b * kABytes, &map_h, &bars->full[st], kb * kBK, row0 + b * kBM, pol_h);
#pragma unroll
          for (int q = 2 * rank; q < 2 * rank + 2; ++q)
            tma_load_2d_mcast(stage + NB * kABytes + q * kWBoxBytes, &map_w, &bars->full[st],
                              v0 + 64 * q, kb * kBK, kBoth, pol_w);
        }
      }
      if (!ok) {
        fail_pipeline(bars);
        for (int j = it > STAGES ? it - STAGES : 0; j < it; ++j)
          (void)mbar_wait(&bars->full[j % STAGES], (j / STAGES) & 1, 50000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN, false, true);
      const uint32_t s0 = smem_u32(smem);
      int it = 0;
      bool ok = true;
      const int total_it = my_tiles * n_kb;
      for (int i = 0; ok && i < my_tiles; ++i) {
        const int buf = NBUF == 2 ? (i & 1) : 0;
        const int use = NBUF == 2 ? (i >> 1) : i;
        if (use >= 1 && !wait_or_abort(&bars->acc_empty[buf], (use - 1) & 1, bars)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * (NB * BN);
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % STAGES;
          if (!wait_or_abort(&bars->full[st], (it / STAGES) & 1, bars)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st_addr = s0 + st * Sh::kStageBytes;
          const uint32_t b_addr = st_addr + NB * kABytes;
#pragma unroll
          for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              mma_bf16_ss(d_tmem + b * BN, sdesc_sw128(st_addr + b * kABytes + k * 32, 16, 1024),
                          sdesc_sw128(b_addr + k * 2048, kWBoxBytes, 1024), idesc,
                          (kb > 0 || k > 0) ? 1u : 0u);
          // stages that will be refilled: release them in both CTAs
          if (it + STAGES < total_it) mma_commit_mcast(&bars->empty[st], kBoth);
        }
        if (!ok) break;
        mma_commit(&bars->acc_full[buf]);
      }
      if (!ok) fail_pipeline(bars);
    }
  } else if (warp >= 4) {
    // warpgroup eg folds column group eg / NB (of CH) of row blocks
    // eg % NB, eg % NB + EPI, ... of the tile
    constexpr int EPI = Sh::EPI, CH = Sh::CH, NBW = (NB * CH + EPI - 1) / EPI;  // row blocks per warp
    constexpr int kCh = BN / 32 / CH;  // 32-column chunks per column group
    const int quarter = warp & 3, egw = (warp - 4) >> 2;
    const int eg = egw % (EPI / CH), cg = egw / (EPI / CH);  // row-block lane, column group
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float m1[NBW], m2[NBW], hm[NBW], hs[NBW], hu[NBW];
    int i1[NBW];
#pragma unroll
    for (int bb = 0; bb < NBW; ++bb) {
      m1[bb] = -INFINITY;
      m2[bb] = -INFINITY;
      i1[bb] = 0x7FFFFFFF;
      hm[bb] = -INFINITY;
      hs[bb] = 0.f;
      hu[bb] = 0.f;
    }
    // sampling: each of this thread's rows' predicted position and stream
    uint32_t spos[NBW], sseq[NBW];
#pragma unroll
    for (int bb = 0; bb < NBW; ++bb) {
      const int gr = row0 + (eg + bb * EPI) * kBM + row;
      spos[bb] = (kS && gr < p.M) ? static_cast<uint32_t>(p.position[gr]) : 0u;
      sseq[bb] = (kS && gr < p.M && p.seq) ? static_cast<uint32_t>(p.seq[gr]) : 0u;
    }
    bool ok = true;
    for (int i = 0; i < my_tiles; ++i) {
      const int buf = NBUF == 2 ? (i & 1) : 0;
      const int use = NBUF == 2 ? (i >> 1) : i;
      if (!wait_or_abort(&bars->acc_full[buf], use & 1, bars)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int v0 = (pair + i * n_pairs) * BN;
#pragma unroll
      for (int bb = 0; bb < NBW; ++bb) {
        const int b = eg + bb * EPI;
        const uint32_t t_acc = tmem + buf * (NB * BN) + b * BN + lane_off;
#pragma unroll 1
        for (int c = cg * kCh; c < (cg + 1) * kCh; ++c) {
          uint32_t r[32];
          tmem_ld32(t_acc + c * 32, r);
          tmem_ld_wait();
          const int col0 = v0 + c * 32;
          if (kS) perturb_chunk(r, col0, p.inv_temp, spos[bb], sseq[bb], p.seed_lo, p.seed_hi);
          fold_chunk(r, col0, p.V, m1[bb], i1[bb], m2[bb]);
          if (kH) entropy_chunk(r, col0, p.V, m1[bb], hm[bb], hs[bb], hu[bb]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->acc_empty[buf]);
    }
    if (!ok) fail_pipeline(bars);
#pragma unroll
    for (int bb = 0; bb < NBW; ++bb) {
      const int grow = row0 + (eg + bb * EPI) * kBM + row;
      if (grow < p.M) {
        const size_t at = (static_cast<size_t>(pair) * CH + cg) * (2 * NB * kBM) + grow;
        if (!GLANCE_IN_BOUNDS(at, static_cast<size_t>(n_pairs) * CH * (2 * NB * kBM))) continue;
        if (kH)
          static_cast<PartialH*>(p.part)[at] = PartialH{m1[bb], i1[bb], m2[bb], hs[bb], hu[bb]};
        else
          static_cast<Partial*>(p.part)[at] = Partial{m1[bb], i1[bb], m2[bb]};
      }
    }
  }
  tc_fence_before();
  // neither CTA leaves while the other may still touch its shared memory
  __syncwarp();
  cluster_sync_all();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // this CTA's part is done: the next kernel in the stream (the acceptance
  // walk) may launch and wait for the merge at its dependency wait
  pdl_launch_dependents();
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_ticket = atomicAdd(p.ticket, 1u);
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;
  __threadfence();
  if (threadIdx.x == 0) *p.ticket = 0;
  // the stage ring is idle now (every copy into it, the partner's multicasts
  // included, has landed): it holds the merge's scratch
  if (kH)
    merge_partials_h(static_cast<const PartialH*>(p.part), n_pairs * Sh::CH, 2 * NB * kBM, p.M,
                     reinterpret_cast<PartialH*>(smem), p.argmax, p.gap, p.maxlogit, p.entropy);
  else
    merge_partials(static_cast<const Partial*>(p.part), n_pairs * Sh::CH, 2 * NB * kBM, p.M,
                   reinterpret_cast<Partial*>(smem), p.argmax, p.gap, p.maxlogit);
}

int row_blocks(int M) { return (M + kBM - 1) / kBM; }

size_t ws_bytes_bf16(int M) {
  const int grid = glance::num_sms();
  // large enough for the partials with the entropy sums
  return 256 + (static_cast<size_t>(grid) * row_blocks(M) * kBM * sizeof(PartialH) + 255) / 256 * 256;
}

// Sampling-mode arguments (unused by the other modes).
struct SampleArgs {
  float inv_temp = 1.f;
  uint64_t seed = 0;
  const int32_t* position = nullptr;
  const int32_t* seq = nullptr;
};

void set_sample(Bf16Params& p, const SampleArgs& sa) {
  p.inv_temp = sa.inv_temp;
  p.seed_lo = static_cast<uint32_t>(sa.seed & 0xFFFFFFFFull);
  p.seed_hi = static_cast<uint32_t>(sa.seed >> 32);
  p.position = sa.position;
  p.seq = sa.seq;
}

// W [d][V] (bf16, row-major) as the shared-memory images of the M <= 128
// kernel's W stages: block (t, kb) (256 columns t, 64 rows kb of d) is 32 KB,
// four 8 KB boxes q of columns 64 q.., row r of a box at r * 128 bytes with
// its 16-byte chunk c (columns 8 c..) at chunk position c ^ (r % 8) (the
// 128-byte swizzle the tensor-map copies produce); columns >= V are zero.
// Thread i writes stored chunk i; a warp reads four whole 128-byte row
// segments.
__global__ void __launch_bounds__(256) lmhead_pack_w_kernel(const uint16_t* W, int d, int V, int n_tiles,
                                                             uint4* out) {
  const int n_kb = d / kBK;
  const size_t n_chunks = static_cast<size_t>(n_tiles) * n_kb * 4 * 64 * 8;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_chunks;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int cs = static_cast<int>(i & 7);
    size_t j = i >> 3;
    const int r = static_cast<int>(j & 63);
    j >>= 6;
    const int q = static_cast<int>(j & 3);
    j >>= 2;
    const int kb = static_cast<int>(j % n_kb);
    const int t = static_cast<int>(j / n_kb);
    const int col = t * 256 + q * 64 + 8 * (cs ^ (r & 7));  // V % 8 == 0: all 8 or none valid
    const int row = kb * kBK + r;
    out[i] = col < V ? *reinterpret_cast<const uint4*>(W + static_cast<size_t>(row) * V + col)
                     : make_uint4(0u, 0u, 0u, 0u);
  }
}

// W_packed: W as stage images (NB = 1), or null. With it, W is only used to
// describe a valid (never read) tensor map: pass the packed buffer.
template <int NB, int kMode>
glance_status launch_bf16(const void* h, const void* W, int M, int d, int V, int32_t* argmax,
                          float* gap, float* maxlogit, float* entropy, void* part, uint32_t* ticket,
                          int max_grid, cudaStream_t s, const char* who,
                          const SampleArgs& sa = SampleArgs(), const void* w_packed = nullptr) {
  using Sh = Shape<NB>;
  const int n_tiles = (V + Sh::BN - 1) / Sh::BN;
  int grid = glance::num_sms();
  if (grid > n_tiles) grid = n_tiles;
  if (grid > max_grid) grid = max_grid;
  cudaError_t e = glance::ensure_smem(reinterpret_cast<const void*>(lmhead_bf16_kernel<NB, kMode>),
                                      static_cast<int>(Sh::kSmem));
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  CUtensorMap mw, mh;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(V), static_cast<uint64_t>(d)};
    const uint64_t strides[1] = {static_cast<uint64_t>(V) * 2ull};
    const uint32_t box[2] = {64, kBK};
    glance_status st = glance::make_map_bf16(&mw, W, 2, dims, strides, box,
                                             CU_TENSOR_MAP_SWIZZLE_128B, who);
    if (st != GLANCE_OK) return st;
  }
  const int a_rows = NB == 1 ? (M + 7) / 8 * 8 : kBM;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(d) * 2ull};
    const uint32_t box[2] = {kBK, static_cast<uint32_t>(a_rows)};
    glance_status st = glance::make_map_bf16(&mh, h, 2, dims, strides, box,
                                             CU_TENSOR_MAP_SWIZZLE_128B, who);
    if (st != GLANCE_OK) return st;
  }
  Bf16Params p{M, d, V, n_tiles, a_rows, argmax, gap, maxlogit, part, ticket, entropy};
  set_sample(p, sa);
  p.w_packed = static_cast<const unsigned char*>(w_packed);
  // a programmatic dependent of the previous kernel: W streams in while it ends
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Sh::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, lmhead_bf16_kernel<NB, kMode>, mh, mw, p);
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  e = cudaGetLastError();
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  return GLANCE_OK;
}

size_t ws_bytes_f32(int M, int V) {
  const int colblks = (V + kF32Cols - 1) / kF32Cols;
  return 256 + (static_cast<size_t>(colblks) * M * sizeof(Partial) + 255) / 256 * 256;
}

// Clusters of 2 that can be resident at once with this kernel's shared
// memory, per device (queried once, after the kernel's shared-memory
// attribute is set).
template <int NB, int kMode>
int max_pairs() {
  static int cached[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * glance::num_sms());
    cfg.blockDim = dim3(PairShape<NB>::kThreads);
    cfg.dynamicSmemBytes = PairShape<NB>::kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, lmhead_bf16_pair_kernel<NB, kMode>, &cfg) != cudaSuccess ||
        n < 1)
      n = -1;
    cached[dev] = n;
  }
  return cached[dev];
}

template <int NB, int kMode>
glance_status launch_pair(const void* h, const void* W, int M, int d, int V, int32_t* argmax,
                          float* gap, float* maxlogit, float* entropy, void* part, uint32_t* ticket,
                          cudaStream_t s, const char* who, const SampleArgs& sa = SampleArgs()) {
  using Sh = PairShape<NB>;
  cudaError_t e = glance::ensure_smem(reinterpret_cast<const void*>(lmhead_bf16_pair_kernel<NB, kMode>),
                                      static_cast<int>(Sh::kSmem));
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  const int n_tiles = (V + Sh::BN - 1) / Sh::BN;
  int pairs = max_pairs<NB, kMode>();
  if (pairs < 1) return glance::fail(GLANCE_ERR_CUDA, "%s: no resident CTA pair fits", who);
  if (pairs > n_tiles) pairs = n_tiles;
  if (2 * pairs > glance::num_sms()) pairs = glance::num_sms() / 2;
  CUtensorMap mw, mh;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(V), static_cast<uint64_t>(d)};
    const uint64_t strides[1] = {static_cast<uint64_t>(V) * 2ull};
    const uint32_t box[2] = {64, kBK};
    glance_status st = glance::make_map_bf16(&mw, W, 2, dims, strides, box,
                                             CU_TENSOR_MAP_SWIZZLE_128B, who);
    if (st != GLANCE_OK) return st;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(d) * 2ull};
    const uint32_t box[2] = {kBK, static_cast<uint32_t>(kBM)};
    glance_status st = glance::make_map_bf16(&mh, h, 2, dims, strides, box,
                                             CU_TENSOR_MAP_SWIZZLE_128B, who);
    if (st != GLANCE_OK) return st;
  }
  Bf16Params p{M, d, V, n_tiles, kBM, argmax, gap, maxlogit, part, ticket, entropy};
  set_sample(p, sa);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(Sh::kThreads);
  cfg.dynamicSmemBytes = Sh::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, lmhead_bf16_pair_kernel<NB, kMode>, mh, mw, p);
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  return GLANCE_OK;
}

// bf16 LM head, one launch (W streams once for all rows): one CTA per SM for
// M <= 128, CTA pairs above. entropy == nullptr skips the entropy sums.
template <int kMode>
glance_status lmhead_bf16(const void* h, const void* W, int M, int d, int V, int32_t* argmax,
                          float* gap, float* maxlogit, float* entropy, void* part, uint32_t* ticket,
                          cudaStream_t s, const char* who, const SampleArgs& sa = SampleArgs()) {
  if (M <= kBM)
    return launch_bf16<1, kMode>(h, W, M, d, V, argmax, gap, maxlogit, entropy, part, ticket,
                                 1 << 30, s, who, sa);
  if (M <= 2 * kBM)
    return launch_pair<1, kMode>(h, W, M, d, V, argmax, gap, maxlogit, entropy, part, ticket, s,
                                 who, sa);
  return launch_pair<2, kMode>(h, W, M, d, V, argmax, gap, maxlogit, entropy, part, ticket, s, who,
                               sa);
}

glance_status check_bf16_call(const char* who, const void* h, const void* W, int M, int d, int V,
                              void* workspace, size_t workspace_bytes) {
  using glance::fail;
  if (d % kBK != 0 || V % 8 != 0)
    return fail(GLANCE_ERR_UNSUPPORTED, "%s: bf16 needs d %% 64 == 0 and V %% 8 == 0", who);
  if (!glance::aligned16(h) || !glance::aligned16(W))
    return fail(GLANCE_ERR_INVALID_ARG, "%s: h and W must be 16-byte aligned", who);
  if (workspace_bytes < ws_bytes_bf16(M))
    return fail(GLANCE_ERR_CAPACITY, "%s: workspace %zu bytes < %zu needed", who, workspace_bytes,
                ws_bytes_bf16(M));
  (void)workspace;
  return GLANCE_OK;
}

}  // namespace

extern "C" size_t glance_lmhead_argmax_workspace_bytes(int M, int d, int V, glance_dtype dtype) {
  if (M < 1 || M > 512 || d < 1 || V < 1) return 0;
  return dtype == GLANCE_BF16 ? ws_bytes_bf16(M) : ws_bytes_f32(M, V);
}

extern "C" glance_status glance_lmhead_argmax(const void* h, const void* W, glance_dtype dtype,
                                              int M, int d, int V, int32_t* argmax, float* gap,
                                              float* maxlogit, void* workspace,
                                              size_t workspace_bytes, void* stream) {
  using glance::fail;
  if (!h || !W || !argmax || !gap || !workspace)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_lmhead_argmax: null pointer argument");
  if (M < 1 || M > 512 || d < 1 || V < 1)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_lmhead_argmax: need 1 <= M <= 512, d >= 1, V >= 1");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_lmhead_argmax: workspace must be 256-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* ticket = static_cast<uint32_t*>(workspace);
  Partial* part = reinterpret_cast<Partial*>(static_cast<char*>(workspace) + 256);
  if (dtype == GLANCE_F32) {
    if (workspace_bytes < ws_bytes_f32(M, V))
      return fail(GLANCE_ERR_CAPACITY, "glance_lmhead_argmax: workspace too small");
    F32Params p{static_cast<const float*>(h), static_cast<const float*>(W), M, d, V, argmax, gap,
                maxlogit, part, ticket, nullptr, nullptr, 1.f, 0u, 0u};
    dim3 grid((V + kF32Cols - 1) / kF32Cols, (M + kF32Rows - 1) / kF32Rows);
    lmhead_f32_kernel<<<grid, kF32Cols, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return glance::cuda_fail(e, "glance_lmhead_argmax: launch");
    return GLANCE_OK;
  }
  if (dtype != GLANCE_BF16)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_lmhead_argmax: dtype must be F32 or BF16");
  glance_status st =
      check_bf16_call("glance_lmhead_argmax", h, W, M, d, V, workspace, workspace_bytes);
  if (st != GLANCE_OK) return st;
  return lmhead_bf16<kGreedy>(h, W, M, d, V, argmax, gap, maxlogit, nullptr, part, ticket, s,
                              "glance_lmhead_argmax");
}

extern "C" size_t glance_lmhead_packed_w_bytes(int d, int V) {
  if (d < kBK || d % kBK != 0 || V < 8 || V % 8 != 0) return 0;
  return static_cast<size_t>((V + 255) / 256) * (d / kBK) * Shape<1>::kBBytes;
}

extern "C" glance_status glance_lmhead_pack_w(const void* W, int d, int V, void* W_packed,
                                              size_t packed_bytes, void* stream) {
  using glance::fail;
  const char* who = "glance_lmhead_pack_w";
  if (!W || !W_packed) return fail(GLANCE_ERR_INVALID_ARG, "%s: null pointer argument", who);
  const size_t need = glance_lmhead_packed_w_bytes(d, V);
  if (need == 0)
    return fail(GLANCE_ERR_UNSUPPORTED, "%s: needs d %% 64 == 0 (d >= 64) and V %% 8 == 0", who);
  if (packed_bytes < need)
    return fail(GLANCE_ERR_CAPACITY, "%s: W_packed holds %zu bytes < %zu needed", who, packed_bytes, need);
  if (!glance::aligned16(W) || !glance::aligned16(W_packed))
    return fail(GLANCE_ERR_INVALID_ARG, "%s: W and W_packed must be 16-byte aligned", who);
  const int n_tiles = (V + 255) / 256;
  lmhead_pack_w_kernel<<<4 * glance::num_sms(), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(W), d, V, n_tiles, static_cast<uint4*>(W_packed));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  return GLANCE_OK;
}

extern "C" glance_status glance_lmhead_argmax_packed(const void* h, const void* W_packed, int M, int d,
                                                     int V, int32_t* argmax, float* gap, float* maxlogit,
                                                     void* workspace, size_t workspace_bytes,
                                                     void* stream) {
  using glance::fail;
  const char* who = "glance_lmhead_argmax_packed";
  if (!h || !W_packed || !argmax || !gap || !workspace)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: null pointer argument", who);
  if (M < 1 || M > kBM || d < 1 || V < 1)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: need 1 <= M <= 128, d >= 1, V >= 1", who);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  if (glance_lmhead_packed_w_bytes(d, V) == 0)
    return fail(GLANCE_ERR_UNSUPPORTED, "%s: needs d %% 64 == 0 (d >= 64) and V %% 8 == 0", who);
  glance_status st = check_bf16_call(who, h, W_packed, M, d, V, workspace, workspace_bytes);
  if (st != GLANCE_OK) return st;
  uint32_t* ticket = static_cast<uint32_t*>(workspace);
  Partial* part = reinterpret_cast<Partial*>(static_cast<char*>(workspace) + 256);
  return launch_bf16<1, kGreedy>(h, W_packed, M, d, V, argmax, gap, maxlogit, nullptr, part, ticket, 1 << 30,
                                 static_cast<cudaStream_t>(stream), who, SampleArgs(), W_packed);
}

extern "C" glance_status glance_lmhead_argmax_entropy(const void* h, const void* W,
                                                      glance_dtype dtype, int M, int d, int V,
                                                      int32_t* argmax, float* gap, float* maxlogit,
                                                      float* entropy, void* workspace,
                                                      size_t workspace_bytes, void* stream) {
  using glance::fail;
  const char* who = "glance_lmhead_argmax_entropy";
  if (!h || !W || !argmax || !gap || !entropy || !workspace)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: null pointer argument", who);
  if (M < 1 || M > 512 || d < 1 || V < 1)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: need 1 <= M <= 512, d >= 1, V >= 1", who);
  if (dtype != GLANCE_BF16) return fail(GLANCE_ERR_UNSUPPORTED, "%s: BF16 only", who);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  glance_status st = check_bf16_call(who, h, W, M, d, V, workspace, workspace_bytes);
  if (st != GLANCE_OK) return st;
  char* ws = static_cast<char*>(workspace);
  return lmhead_bf16<kEntropy>(h, W, M, d, V, argmax, gap, maxlogit, entropy, ws + 256,
                               reinterpret_cast<uint32_t*>(ws), static_cast<cudaStream_t>(stream),
                               who);
}

extern "C" glance_status glance_lmhead_sample(const void* h, const void* W, glance_dtype dtype,
                                              int M, int d, int V, float inv_temperature,
                                              uint64_t seed, const int32_t* position,
                                              const int32_t* seq, int32_t* tokens, float* gap,
                                              void* workspace, size_t workspace_bytes,
                                              void* stream) {
  using glance::fail;
  const char* who = "glance_lmhead_sample";
  if (!h || !W || !position || !tokens || !gap || !workspace)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: null pointer argument", who);
  if (M < 1 || M > 512 || d < 1 || V < 1)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: need 1 <= M <= 512, d >= 1, V >= 1", who);
  if (!(inv_temperature > 0.f) || !isfinite(inv_temperature))
    return fail(GLANCE_ERR_INVALID_ARG, "%s: inv_temperature must be finite and > 0", who);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* ticket = static_cast<uint32_t*>(workspace);
  char* part = static_cast<char*>(workspace) + 256;
  if (dtype == GLANCE_F32) {
    if (workspace_bytes < ws_bytes_f32(M, V)) return fail(GLANCE_ERR_CAPACITY, "%s: workspace too small", who);
    F32Params p{static_cast<const float*>(h), static_cast<const float*>(W), M, d, V, tokens, gap,
                nullptr, reinterpret_cast<Partial*>(part), ticket, position, seq, inv_temperature,
                static_cast<uint32_t>(seed & 0xFFFFFFFFull), static_cast<uint32_t>(seed >> 32)};
    dim3 grid((V + kF32Cols - 1) / kF32Cols, (M + kF32Rows - 1) / kF32Rows);
    lmhead_f32_kernel<<<grid, kF32Cols, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return glance::cuda_fail(e, who);
    return GLANCE_OK;
  }
  if (dtype != GLANCE_BF16) return fail(GLANCE_ERR_INVALID_ARG, "%s: dtype must be F32 or BF16", who);
  glance_status st = check_bf16_call(who, h, W, M, d, V, workspace, workspace_bytes);
  if (st != GLANCE_OK) return st;
  SampleArgs sa;
  sa.inv_temp = inv_temperature;
  sa.seed = seed;
  sa.position = position;
  sa.seq = seq;
  return lmhead_bf16<kSample>(h, W, M, d, V, tokens, gap, nullptr, nullptr, part, ticket, s, who, sa);
}

// ------------------------------------------------- no-allocation entry point
//
// For callers that cannot allocate device memory or hand the library a
// workspace on this path: for example code that runs while a stream is being
// captured in a mode that forbids cudaMalloc, or an engine that has reserved
// all device memory for its own pool. The scratch that glance_lmhead_argmax
// takes from its workspace (a merge ticket and one partial per CTA and row)
// lives instead in the file-scope array below. Every GPU that loads this
// library holds the array (240 KB) until the process exits.

namespace {

constexpr int kNoAllocMaxCtas = 160;
constexpr size_t kNoAllocScratchBytes =
    256 + static_cast<size_t>(kNoAllocMaxCtas) * kBM * sizeof(Partial);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The driver's current context, fetched through the runtime (no link-time
// dependency on libcuda); null if the entry point is unavailable.
CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

// Device address of g_noalloc_scratch on the current device, looked up with
// that device current (in host code the array's name is only a stand-in, not
// a device address). The address is kept per device together with the
// context it was looked up in, and looked up again when the device's context
// has changed (after cudaDeviceReset, for example).
glance_status noalloc_scratch(void** out) {
  static void* addr[64] = {nullptr};
  static CUcontext ctx[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return glance::cuda_fail(e, "glance_lmhead_argmax_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= 64)
    return glance::fail(GLANCE_ERR_UNSUPPORTED, "glance_lmhead_argmax_noalloc: device index %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  const CUcontext cur = current_context();
  if (!addr[dev] || !cur || cur != ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess)
      return glance::cuda_fail(e, "glance_lmhead_argmax_noalloc: cudaGetSymbolAddress");
    addr[dev] = p;
    ctx[dev] = current_context();
  }
  *out = addr[dev];
  return GLANCE_OK;
}

}  // namespace

extern "C" glance_status glance_lmhead_argmax_noalloc(const void* h, const void* W,
                                                      glance_dtype dtype, int M, int d, int V,
                                                      int32_t* argmax, float* gap,
                                                      float* maxlogit, void* stream) {
  using glance::fail;
  if (!h || !W || !argmax || !gap)
    return fail(GLANCE_ERR_INVALID_ARG, "glance_lmhead_argmax_noalloc: null pointer argument");
  if (dtype != GLANCE_BF16)
    return fail(GLANCE_ERR_UNSUPPORTED, "glance_lmhead_argmax_noalloc: only BF16 is supported");
  if (M < 1 || M > 512 || d < 1 || V < 1)
    return fail(GLANCE_ERR_INVALID_ARG,
                "glance_lmhead_argmax_noalloc: need 1 <= M <= 512, d >= 1, V >= 1 (got M=%d)", M);
  if (d % kBK != 0 || V % 8 != 0)
    return fail(GLANCE_ERR_UNSUPPORTED,
                "glance_lmhead_argmax_noalloc: needs d %% 64 == 0 and V %% 8 == 0");
  if (!glance::aligned16(h) || !glance::aligned16(W))
    return fail(GLANCE_ERR_INVALID_ARG,
                "glance_lmhead_argmax_noalloc: h and W must be 16-byte aligned");
  void* scratch = nullptr;
  glance_status st = noalloc_scratch(&scratch);
  if (st != GLANCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the merge ticket must start at zero (the array keeps the last call's contents)
  cudaError_t e = cudaMemsetAsync(scratch, 0, 256, s);
  if (e != cudaSuccess) return glance::cuda_fail(e, "glance_lmhead_argmax_noalloc: ticket reset");
  uint32_t* ticket = static_cast<uint32_t*>(scratch);
  Partial* part = reinterpret_cast<Partial*>(static_cast<char*>(scratch) + 256);
  // rows in blocks of 128, one launch each (the scratch holds the partials of
  // one block for at most kNoAllocMaxCtas CTAs): each launch streams all of W,
  // so a call with M > 128 reads W ceil(M / 128) times
  for (int r0 = 0; r0 < M; r0 += kBM) {
    const int mb = M - r0 < kBM ? M - r0 : kBM;
    st = launch_bf16<1, kGreedy>(static_cast<const uint16_t*>(h) + static_cast<size_t>(r0) * d, W, mb,
                               d, V, argmax + r0, gap + r0, maxlogit ? maxlogit + r0 : nullptr,
                               nullptr, part, ticket, kNoAllocMaxCtas, s,
                               "glance_lmhead_argmax_noalloc");
    if (st != GLANCE_OK) return st;
  }
  return GLANCE_OK;
}
