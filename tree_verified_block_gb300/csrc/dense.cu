// The target's dense verify layers around tree attention, at the verify
// width (M <= 128 packed rows).
//
// Paper: "Vision Is Not Overhead ..." (arXiv 2609.00355): the verify pass
// runs the frozen target once over the packed tree rows (Definition 1,
// Section 4.2) and its forward dominates a round's cost (Table 11 and the
// round-cost regression of Appendix E). The pages do not describe the layer;
// this is a Qwen3-shaped pre-norm decoder layer:
//   x -> RMSNorm -> [q | k | v] = . W_qkv -> per-head RMSNorm of q, k (when
//   weights are given) -> rotate-half RoPE at the rows' positions -> q out,
//   K/V into the cache at slots T + row -> (tree attention) -> x + . W_o
//   -> RMSNorm -> SiLU(. W_gate) * (. W_up) -> x' + . W_down.
// An RMSNorm's weight is folded into the next projection's rows by the
// caller; its 1 / rms row scale, which a projection is linear in, is applied
// to the product. The row sums of squares it needs come from the kernel that
// wrote the rows: the residual projections emit them per output tile.
//
// GEMM shape: Y[M x N] = X[M x K] W[K x N], W row-major with N contiguous
// (the MN-major B operand), bf16 in, fp32 accumulate. At M <= 128 the weights
// dominate (HBM-bound) and N / 256 output tiles are too few to occupy the
// SMs, so K is split S ways inside a thread-block cluster of S CTAs: CTA s of
// the cluster of tile t accumulates K range s in tensor memory (warp 0 streams
// X and W stages with TMA, 4 x 48 KB; warp 1 issues M=128 x N=256 x K=16 MMAs). Once
// the whole cluster is done with its stages, warps 4..7 send each row of the
// fp32 partial to the CTA that owns the row (remote stores into its shared
// memory); after a second cluster barrier each CTA sums the S partials of its
// rows and applies the epilogue. No global workspace, no grid-wide barrier. Launches
// are programmatic dependents of the previous kernel in the stream: the first
// W stages (which do not depend on it) are in flight before the wait.
#include <cstring>
#include <mutex>

#include "glance_internal.cuh"

GLANCE_DEFINE_STATUS_WORD(status_dense)

using namespace glance_dev;

namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 256;
constexpr uint32_t kABytes = kBM * kBK * 2;    // 16 KB
constexpr uint32_t kBBytes = kBK * kBN * 2;    // 32 KB
constexpr uint32_t kWBoxBytes = kBK * 64 * 2;  // one 64 x 64 box of W: 8 KB
constexpr uint32_t kStageArea = kStages * (kABytes + kBBytes);
constexpr int kPartStride = kBN + 4;           // floats per partial row in shared memory
constexpr int kMaxSplit = 16;
// received partials: [source rank][owned row][kPartStride], at most M + S - 1 rows
constexpr uint32_t kRecvBytes = (kBM + kMaxSplit) * kPartStride * 4;
constexpr int kChunkRows = 16;                 // epilogue: 16 rows at a time (16 threads a row)
constexpr size_t kSmemBytes = 1024 + kStageArea + 2048;
constexpr int kHeadDim = 128;
static_assert(kRecvBytes <= kStageArea, "received partials overlay the stages");

enum Mode : int { kResid = 0, kQKV = 1, kSwiGLU = 2 };

struct DenseParams {
  int M, K, n_kb, a_rows, mode, split;
  float eps;
  // input row norm: r[row] = 1 / sqrt(sum_t in_sumsq[t][row] / K + eps) (null: r = 1)
  const float* in_sumsq;
  int n_sumsq;
  // kResid: out_sumsq[tile][row] = sum of squares of the tile's bf16 outputs (nullable)
  float* out_sumsq;
  // kResid: out = res + X W, both [M][n_out]
  const __nv_bfloat16* res;
  __nv_bfloat16* out;
  int n_out;
  // kQKV
  int Hq, Hkv;
  const float* q_norm;      // [128] or null
  const float* k_norm;      // [128] or null
  const int32_t* pos;       // [M] position ids
  float log2_theta;
  __nv_bfloat16* q_out;     // [M][Hq][128]
  __nv_bfloat16* k_cache;   // [Hkv][t_cap][128] (strides below)
  __nv_bfloat16* v_cache;
  long long head_stride, row_stride;  // elements
  const int32_t* t_len;
  int t_cap;
  // kSwiGLU: act[M][inter] = SiLU(gate) * up
  __nv_bfloat16* act;
  int inter;
};

struct __align__(8) Bars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int failed;         // read by the cluster's other CTAs
  float r[kBM];       // 1 / rms of the rows this CTA finishes
};

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

__device__ __forceinline__ void fail_pipeline(Bars* bars) {
  report(GLANCE_DEV_PIPELINE_TIMEOUT);
  atomicExch(&bars->abort_flag, 1);
}

__device__ __forceinline__ int dsmem_ld_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Columns of a tile that thread t handles in the epilogue: 16 threads per
// row, each with two groups of 8 columns, a (from column col_a) and b (from
// col_b). Residual: 16 contiguous columns. SwiGLU: gate column j and its up
// column 128 + j. QKV: dims j0..j0+7 of one of the tile's two heads and their
// rotate-half partners j0+64..j0+71 (8 consecutive threads share a head).
__device__ __forceinline__ void epilogue_cols(int mode, int t, int& col_a, int& col_b) {
  const int sub = t % 16;
  if (mode == kResid) {
    col_a = sub * 16;
    col_b = col_a + 8;
  } else if (mode == kSwiGLU) {
    col_a = sub * 8;
    col_b = 128 + sub * 8;
  } else {
    col_a = (sub / 8) * kHeadDim + (sub % 8) * 8;
    col_b = col_a + 64;
  }
}

// Epilogue of one row's two column groups (summed products a, b, before the
// row scale r). Every thread of the block calls it (the QKV head norm and the
// residual's row sums of squares shuffle across lanes); `valid` says whether
// the row is this thread's.
__device__ void epilogue_regs(const DenseParams& p, float (&a)[8], float (&b)[8], float r, int tile, int row,
                              bool valid, int T) {
  const int t = threadIdx.x;
  int col_a, col_b;
  epilogue_cols(p.mode, t, col_a, col_b);
  if (p.mode == kResid) {
    float ss = 0.f;
    if (valid) {
      const size_t base = static_cast<size_t>(row) * p.n_out + static_cast<size_t>(tile) * kBN;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float* v8 = h ? b : a;
        const size_t at = base + (h ? col_b : col_a);
        const uint4 v = *reinterpret_cast<const uint4*>(p.res + at);
        const uint32_t rv[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o[e] = pack_bf16x2(__uint_as_float(rv[e] << 16) + v8[2 * e],
                             __uint_as_float(rv[e] & 0xFFFF0000u) + v8[2 * e + 1]);
          const float lo = __uint_as_float(o[e] << 16), hi = __uint_as_float(o[e] & 0xFFFF0000u);
          ss += lo * lo + hi * hi;  // of the stored (rounded) values
        }
        *reinterpret_cast<uint4*>(p.out + at) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    if (p.out_sumsq) {  // the row's 16 threads are 16 consecutive lanes
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (valid && t % 16 == 0) p.out_sumsq[static_cast<size_t>(tile) * p.M + row] = ss;
    }
    return;
  }
  if (p.mode == kSwiGLU) {
    if (!valid) return;
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float a2[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float g = a[2 * e + h] * r, u = b[2 * e + h] * r;
        a2[h] = g / (1.f + expf(-g)) * u;
      }
      o[e] = pack_bf16x2(a2[0], a2[1]);
    }
    *reinterpret_cast<uint4*>(p.act + static_cast<size_t>(row) * p.inter + static_cast<size_t>(tile) * 128 +
                              col_a) = make_uint4(o[0], o[1], o[2], o[3]);
    return;
  }
  // kQKV: the tile is two heads of one segment (q, k or v)
  const int hh = col_a / kHeadDim, j0 = col_a % kHeadDim;
  const int col0 = tile * kBN + hh * kHeadDim;  // first column of this head in q|k|v
  const int qcols = p.Hq * kHeadDim, kcols = p.Hkv * kHeadDim;
  const int seg = col0 < qcols ? 0 : (col0 < qcols + kcols ? 1 : 2);
  const int head = seg == 0 ? col0 / kHeadDim
                            : (seg == 1 ? (col0 - qcols) / kHeadDim : (col0 - qcols - kcols) / kHeadDim);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    a[e] *= r;
    b[e] *= r;
  }
  const float* gnorm = seg == 0 ? p.q_norm : (seg == 1 ? p.k_norm : nullptr);
  if (gnorm) {  // per-head RMSNorm over the 128 dims (8 threads, consecutive lanes)
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ss += a[e] * a[e] + b[e] * b[e];
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
    const float inv = rsqrtf(ss / kHeadDim + p.eps);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      a[e] *= inv * gnorm[j0 + e];
      b[e] *= inv * gnorm[64 + j0 + e];
    }
  }
  if (!valid) return;
  if (seg > 0 && (T < 0 || T + p.M > p.t_cap)) {  // all M rows' K/V slots must exist, else none is written
    report(GLANCE_DEV_TREE_CAPACITY);
    return;
  }
  if (seg < 2) {  // rotate-half RoPE: (a, b) -> (a cos - b sin, b cos + a sin)
    const float pos = static_cast<float>(p.pos[row]);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j = j0 + e;
      const float inv_freq = exp2f(-(2.f * j / kHeadDim) * p.log2_theta);
      float sn, cs;
      sincosf(pos * inv_freq, &sn, &cs);
      const float x = a[e], y = b[e];
      a[e] = x * cs - y * sn;
      b[e] = y * cs + x * sn;
    }
  }
  __nv_bfloat16* dst;
  if (seg == 0) {
    dst = p.q_out + (static_cast<size_t>(row) * p.Hq + head) * kHeadDim;
  } else {
    __nv_bfloat16* base = seg == 1 ? p.k_cache : p.v_cache;
    dst = base + head * p.head_stride + static_cast<long long>(T + row) * p.row_stride;
  }
  uint32_t oa[4], ob[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    oa[e] = pack_bf16x2(a[2 * e], a[2 * e + 1]);
    ob[e] = pack_bf16x2(b[2 * e], b[2 * e + 1]);
  }
  *reinterpret_cast<uint4*>(dst + j0) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  *reinterpret_cast<uint4*>(dst + 64 + j0) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
}

// Grid: one cluster of p.split CTAs per output tile (blockIdx.x = tile * S +
// rank). Every wait is bounded; a CTA that gives up still takes part in both
// cluster barriers, so its peers never wait on it forever.
__global__ void __launch_bounds__(kThreads, 1)
    dense_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                 const __grid_constant__ CUtensorMap map_b1, const DenseParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* sA = smem;
  unsigned char* sB = smem + kStages * kABytes;
  Bars* bars = reinterpret_cast<Bars*>(smem + kStageArea);
  // after phase 1 the stage area receives the cluster's partials of this
  // CTA's rows
  float* s_recv = reinterpret_cast<float*>(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.split;
  const int rank = static_cast<int>(cluster_ctarank());
  const int tile = static_cast<int>(blockIdx.x) / S;
  const int kb0 = static_cast<int>((static_cast<long long>(p.n_kb) * rank) / S);
  const int kb1 = static_cast<int>((static_cast<long long>(p.n_kb) * (rank + 1)) / S);
  const int n_it = kb1 - kb0;  // >= 1: S <= n_kb
  const uint32_t a_bytes = static_cast<uint32_t>(p.a_rows) * kBK * 2;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    bars->failed = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(&bars->tmem_base, kBN);
    tmem_relinquish();
  }
  // rows a_rows..127 of every A stage stay zero (TMA only writes a_rows rows)
  if (p.a_rows < kBM) {
    for (int s = 0; s < kStages; ++s) {
      uint4* dst = reinterpret_cast<uint4*>(sA + s * kABytes + p.a_rows * 128);
      for (int i = threadIdx.x; i < (kBM - p.a_rows) * 8; i += kThreads) dst[i] = make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  auto load_w = [&](int st, int kb, uint64_t pol) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      unsigned char* dstb = sB + st * kBBytes + q * kWBoxBytes;
      if (p.mode == kSwiGLU)  // gate columns 128 t.., then up columns 128 t..
        tma_load_2d(dstb, q < 2 ? &map_b0 : &map_b1, &bars->full[st], tile * 128 + 64 * (q & 1), kb * kBK,
                    pol);
      else
        tma_load_2d(dstb, &map_b0, &bars->full[st], tile * kBN + 64 * q, kb * kBK, pol);
    }
  };
  // W does not depend on the previous kernel: its first stages go out now
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b0);
    tma_prefetch_desc(&map_b1);
    const uint64_t pol_w = policy_evict_first();
    for (int it = 0; it < kStages && it < n_it; ++it) {
      mbar_arrive_expect_tx(&bars->full[it], a_bytes + kBBytes);
      load_w(it, kb0 + it, pol_w);
    }
  }
  pdl_wait_prior();

  // rows are owned in blocks of rows_per: CTA o of the cluster sums and
  // finishes rows o * rows_per ..
  const int rows_per = (p.M + S - 1) / S;
  const int r_begin = rank * rows_per;
  const int r_end = min(p.M, r_begin + rows_per);

  // ------------------------------------------------------------ phase 1
  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int it = 0;
      for (; it < n_it; ++it) {
        const int st = it % kStages, kb = kb0 + it;
        if (it >= kStages) {
          if (!wait_or_abort(&bars->empty[st], ((it / kStages) - 1) & 1, bars)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->full[st], a_bytes + kBBytes);
          load_w(st, kb, pol_w);
        }
        tma_load_2d(sA + st * kABytes, &map_a, &bars->full[st], kb * kBK, 0, pol_x);
      }
      if (!ok) {  // let the copies in flight land before the stage area is reused
        fail_pipeline(bars);
        for (int j = it > kStages ? it - kStages : 0; j < it; ++j)
          (void)mbar_wait(&bars->full[j % kStages], (j / kStages) & 1, 50000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, true);
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      for (int it = 0; it < n_it; ++it) {
        const int st = it % kStages;
        if (!wait_or_abort(&bars->full[st], (it / kStages) & 1, bars)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = a0 + st * kABytes, b_addr = b0 + st * kBBytes;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_bf16_ss(tmem, sdesc_sw128(a_addr + k * 32, 16, 1024), sdesc_sw128(b_addr + k * 2048, kWBoxBytes, 1024),
                      idesc, (it > 0 || k > 0) ? 1u : 0u);
        if (it + kStages < n_it) mma_commit(&bars->empty[st]);
      }
      if (ok) {
        mma_commit(&bars->acc_full);
      } else {  // the MMAs issued so far finish before the stage area is reused
        mma_commit(&bars->drain);
        (void)mbar_wait(&bars->drain, 0, 50000000ull);
        fail_pipeline(bars);
      }
    }
  } else if (warp >= 4) {
    if (!wait_or_abort(&bars->acc_full, 0, bars)) {
      ok = false;
      fail_pipeline(bars);
    }
  } else if (p.in_sumsq) {
    // warps 2 and 3: the RMSNorm row scales 1 / rms of this CTA's rows, from
    // the sums of squares the previous kernel emitted per output tile, while
    // the stages stream (8 loads in flight, summed in tile order)
    for (int lrow = threadIdx.x - 64; lrow < r_end - r_begin; lrow += 64) {
      float ss = 0.f;
      for (int t0 = 0; t0 < p.n_sumsq; t0 += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          v[u] = t0 + u < p.n_sumsq ? p.in_sumsq[static_cast<size_t>(t0 + u) * p.M + r_begin + lrow] : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) ss += v[u];
      }
      bars->r[lrow] = rsqrtf(ss / p.K + p.eps);
    }
  }
  // every role is done with its own stage area (or gave up and drained)
  const bool bad = __syncthreads_or(!ok || *reinterpret_cast<volatile int*>(&bars->abort_flag)) != 0;
  if (threadIdx.x == 0) bars->failed = bad ? 1 : 0;
  __syncwarp();
  cluster_sync_all();  // the whole cluster is done with its stage areas
  bool peer_bad = false;
  if (threadIdx.x < S) peer_bad = dsmem_ld_s32(dsmem_addr(&bars->failed, threadIdx.x)) != 0;
  const bool any_bad = __syncthreads_or(peer_bad) != 0;

  // each CTA sends its partial of every row to the row's owner (remote stores
  // into the owner's stage area)
  if (!any_bad && warp >= 4) {
    tc_fence_after();
    const int quarter = warp - 4;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int owner = row / rows_per, lrow = row - owner * rows_per;
    const int slot = rank * rows_per + lrow;
    const uint32_t dst = dsmem_addr(s_recv + slot * kPartStride, row < p.M ? owner : 0);
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_off + c * 32, r);  // warp-collective: every lane loads
      tmem_ld_wait();
      if (row < p.M) {
#pragma unroll
        for (int v = 0; v < 8; ++v)
          dsmem_st_f4(dst + (c * 32 + 4 * v) * 4, __uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                      __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kBN);
  }
  __syncwarp();
  cluster_sync_all();  // every partial has reached its owner

  // ------------------------------------------------------------ phase 2
  if (!any_bad) {
    const int T = p.mode == kQKV ? *p.t_len : 0;
    int col_a, col_b;
    epilogue_cols(p.mode, threadIdx.x, col_a, col_b);
    for (int r0 = r_begin; r0 < r_end; r0 += kChunkRows) {
      // thread: one row, two groups of 8 columns; sum over the cluster's partials
      const int row = r0 + static_cast<int>(threadIdx.x) / 16;
      const bool valid = row < r_end;
      const int lrow = valid ? row - r_begin : 0;
      float a[8], b[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) a[e] = b[e] = 0.f;
      if (valid) {
        for (int s = 0; s < S; ++s) {
          const float* src = s_recv + (s * rows_per + lrow) * kPartStride;
          const float4 a0 = *reinterpret_cast<const float4*>(src + col_a);
          const float4 a1 = *reinterpret_cast<const float4*>(src + col_a + 4);
          const float4 b0 = *reinterpret_cast<const float4*>(src + col_b);
          const float4 b1 = *reinterpret_cast<const float4*>(src + col_b + 4);
          a[0] += a0.x, a[1] += a0.y, a[2] += a0.z, a[3] += a0.w;
          a[4] += a1.x, a[5] += a1.y, a[6] += a1.z, a[7] += a1.w;
          b[0] += b0.x, b[1] += b0.y, b[2] += b0.z, b[3] += b0.w;
          b[4] += b1.x, b[5] += b1.y, b[6] += b1.z, b[7] += b1.w;
        }
      }
      const float r = p.in_sumsq && valid ? bars->r[lrow] : 1.f;
      epilogue_regs(p, a, b, r, tile, row, valid, T);
    }
  }
}

// sumsq[row] = sum_k x[row][k]^2; one warp per row.
__global__ void row_sumsq_kernel(const __nv_bfloat16* x, int M, int d, float* sumsq) {
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const __nv_bfloat16* xr = x + static_cast<size_t>(row) * d;
  float s = 0.f;
#pragma unroll 4
  for (int c = lane * 8; c < d; c += 32 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
      s += lo * lo + hi * hi;
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) sumsq[row] = s;
}

// Clusters of `size` CTAs of dense_kernel that fit on the device at once
// (queried once per device and size, after the shared-memory attribute is set).
int max_clusters(int size) {
  static int cached[64][kMaxSplit + 1] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev][size] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(size * glance::num_sms());
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, dense_kernel, &cfg) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      n = -1;
    }
    cached[dev][size] = n;
  }
  return cached[dev][size];
}

// K splits per tile: the largest S (<= 16, <= the K blocks) whose n_tiles
// clusters all fit on the device at once; 1 when even that takes more than
// one wave.
int choose_split(int n_tiles, int n_kb) {
  int best = 1;
  for (int s = 2; s <= kMaxSplit && s <= n_kb; ++s)
    if (max_clusters(s) >= n_tiles) best = s;
  return best;
}

cudaError_t ensure_attrs() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(dense_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) done[dev] = true;
  return cudaSuccess;
}

glance_status run_dense(const char* who, const void* x, int M, int K, const void* W0, const void* W1,
                        int w_cols, int n_tiles, DenseParams p, cudaStream_t s) {
  using glance::fail;
  if (M < 1 || M > kBM) return fail(GLANCE_ERR_UNSUPPORTED, "%s: need 1 <= M <= 128", who);
  if (K < kBK || K % kBK) return fail(GLANCE_ERR_UNSUPPORTED, "%s: K must be a multiple of 64", who);
  if (!glance::aligned16(x) || !glance::aligned16(W0) || !glance::aligned16(W1))
    return fail(GLANCE_ERR_INVALID_ARG, "%s: x and W must be 16-byte aligned", who);
  cudaError_t e = ensure_attrs();
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  const int a_rows = (M + 7) / 8 * 8;
  CUtensorMap ma, mb0, mb1;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(K) * 2ull};
    const uint32_t box[2] = {kBK, static_cast<uint32_t>(a_rows)};
    glance_status st = glance::make_map_bf16(&ma, x, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, who);
    if (st != GLANCE_OK) return st;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(w_cols), static_cast<uint64_t>(K)};
    const uint64_t strides[1] = {static_cast<uint64_t>(w_cols) * 2ull};
    const uint32_t box[2] = {64, kBK};
    glance_status st = glance::make_map_bf16(&mb0, W0, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, who);
    if (st != GLANCE_OK) return st;
    st = glance::make_map_bf16(&mb1, W1, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, who);
    if (st != GLANCE_OK) return st;
  }
  p.M = M;
  p.K = K;
  p.n_kb = K / kBK;
  p.split = choose_split(n_tiles, p.n_kb);
  p.a_rows = a_rows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_tiles * p.split);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, dense_kernel, ma, mb0, mb1, p);
  if (e != cudaSuccess) return glance::cuda_fail(e, who);
  return GLANCE_OK;
}

DenseParams blank_params() {
  DenseParams p;
  memset(&p, 0, sizeof(p));
  return p;
}

}  // namespace

extern "C" glance_status glance_row_sumsq(const void* x, int M, int d, float* sumsq, void* stream) {
  using glance::fail;
  if (!x || !sumsq) return fail(GLANCE_ERR_INVALID_ARG, "glance_row_sumsq: null pointer argument");
  if (M < 1 || d < 8 || d % 8 || !glance::aligned16(x))
    return fail(GLANCE_ERR_INVALID_ARG, "glance_row_sumsq: need M >= 1, d %% 8 == 0, 16-byte aligned x");
  row_sumsq_kernel<<<(M + 3) / 4, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(x), M, d, sumsq);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return glance::cuda_fail(e, "glance_row_sumsq");
  return GLANCE_OK;
}

extern "C" glance_status glance_dense_residual(const void* x, const void* W, int M, int K, int N,
                                               const void* residual, void* out, float* out_sumsq,
                                               void* stream) {
  using glance::fail;
  const char* who = "glance_dense_residual";
  if (!x || !W || !residual || !out) return fail(GLANCE_ERR_INVALID_ARG, "%s: null pointer argument", who);
  if (N < kBN || N % kBN) return fail(GLANCE_ERR_UNSUPPORTED, "%s: N must be a multiple of 256", who);
  if (!glance::aligned16(residual) || !glance::aligned16(out))
    return fail(GLANCE_ERR_INVALID_ARG, "%s: residual and out must be 16-byte aligned", who);
  DenseParams p = blank_params();
  p.mode = kResid;
  p.res = static_cast<const __nv_bfloat16*>(residual);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.n_out = N;
  p.out_sumsq = out_sumsq;
  return run_dense(who, x, M, K, W, W, N, N / kBN, p, static_cast<cudaStream_t>(stream));
}

extern "C" glance_status glance_dense_swiglu(const void* h, const void* W_gate, const void* W_up,
                                             int M, int d, int inter, const float* in_sumsq,
                                             int n_sumsq, float eps, void* act, void* stream) {
  using glance::fail;
  const char* who = "glance_dense_swiglu";
  if (!h || !W_gate || !W_up || !act) return fail(GLANCE_ERR_INVALID_ARG, "%s: null pointer argument", who);
  if (inter < 128 || inter % 128) return fail(GLANCE_ERR_UNSUPPORTED, "%s: inter must be a multiple of 128", who);
  if (!glance::aligned16(act)) return fail(GLANCE_ERR_INVALID_ARG, "%s: act must be 16-byte aligned", who);
  DenseParams p = blank_params();
  if (in_sumsq && n_sumsq < 1) return fail(GLANCE_ERR_INVALID_ARG, "%s: n_sumsq must be >= 1", who);
  p.mode = kSwiGLU;
  p.in_sumsq = in_sumsq;
  p.n_sumsq = n_sumsq;
  p.eps = eps;
  p.act = static_cast<__nv_bfloat16*>(act);
  p.inter = inter;
  return run_dense(who, h, M, d, W_gate, W_up, inter, inter / 128, p, static_cast<cudaStream_t>(stream));
}

extern "C" glance_status glance_dense_qkv(const void* h, const void* W_qkv, int M, int d, int n_q_heads,
                                          const float* in_sumsq, int n_sumsq, const float* q_norm,
                                          const float* k_norm,
                                          float eps, const int32_t* pos_id, float rope_theta,
                                          void* q_out, const glance_kv* kv, void* stream) {
  using glance::fail;
  const char* who = "glance_dense_qkv";
  if (!h || !W_qkv || !pos_id || !q_out || !kv || !kv->k || !kv->v || !kv->t_len)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: null pointer argument", who);
  if (kv->dtype != GLANCE_BF16 || kv->head_dim != kHeadDim)
    return fail(GLANCE_ERR_UNSUPPORTED, "%s: bf16 cache with head_dim 128 only", who);
  const int Hkv = kv->n_kv_heads;
  if (n_q_heads < 2 || n_q_heads % 2 || Hkv < 2 || Hkv % 2 || n_q_heads % Hkv)
    return fail(GLANCE_ERR_UNSUPPORTED, "%s: need even head counts with n_q_heads %% n_kv_heads == 0", who);
  if (!(rope_theta > 1.f)) return fail(GLANCE_ERR_INVALID_ARG, "%s: rope_theta must be > 1", who);
  if (!glance::aligned16(q_out) || !glance::aligned16(kv->k) || !glance::aligned16(kv->v) ||
      kv->row_stride < kHeadDim || (kv->row_stride * 2) % 16 || (kv->head_stride * 2) % 16 ||
      kv->head_stride < static_cast<int64_t>(kv->t_cap) * kv->row_stride || kv->t_cap < M)
    return fail(GLANCE_ERR_INVALID_ARG, "%s: bad q_out / cache layout", who);
  if (in_sumsq && n_sumsq < 1) return fail(GLANCE_ERR_INVALID_ARG, "%s: n_sumsq must be >= 1", who);
  DenseParams p = blank_params();
  p.mode = kQKV;
  p.in_sumsq = in_sumsq;
  p.n_sumsq = n_sumsq;
  p.Hq = n_q_heads;
  p.Hkv = Hkv;
  p.q_norm = q_norm;
  p.k_norm = k_norm;
  p.eps = eps;
  p.pos = pos_id;
  p.log2_theta = log2f(rope_theta);
  p.q_out = static_cast<__nv_bfloat16*>(q_out);
  p.k_cache = static_cast<__nv_bfloat16*>(kv->k);
  p.v_cache = static_cast<__nv_bfloat16*>(kv->v);
  p.head_stride = kv->head_stride;
  p.row_stride = kv->row_stride;
  p.t_len = kv->t_len;
  p.t_cap = kv->t_cap;
  const int cols = (n_q_heads + 2 * Hkv) * kHeadDim;
  return run_dense(who, h, M, d, W_qkv, W_qkv, cols, cols / kBN, p, static_cast<cudaStream_t>(stream));
}
