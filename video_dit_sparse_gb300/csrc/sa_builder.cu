// sa_builder.cu — training-free key-list builder for sm_103a (FG-Attn review,
// referee comment 2 / §4.4: score keys with the group's mean query; LoSA
// abstract: retained attention mass).
//
//   1. sa_meanq_kernel   q_avg per (b,h,g) in fp32, stored as bf16 hi + lo.
//   2. sa_score_kernel   sigma = scale * K q_avg on tcgen05 tensor cores:
//                        A = 128 keys x d, B = 128 groups x d (hi, then lo,
//                        accumulated), fp32 in TMEM; written [rows, Nk].
//                        K and mean-query tiles arrive by 2-D TMA.
//   3. sa_select_kernel  per row: the selection cut as an exact fp32 value
//                        (3-level radix descent over order-preserving keys)
//                        plus how many keys equal to the cut are kept.
//   4. sa_scan_kernel    row_ptr = exclusive prefix sum of the counts.
//   5. sa_emit_kernel    ascending indices of kept keys into col_idx.
#include "sa_device.cuh"
#include "sa_internal.h"
#include "sa_tma.h"

namespace sa {

// ------------------------------------------------------------ helpers
__device__ __forceinline__ uint16_t bf16_rn(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float bf16_f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}


template <typename T>
__device__ __forceinline__ T warp_incl_scan(T v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Exclusive scan across the block (blockDim.x a multiple of 32, <= 1024).
// `scratch` holds 32 elements.  Every thread receives the block total.
template <typename T>
__device__ __forceinline__ T block_excl_scan(T v, T* total, T* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const T incl = warp_incl_scan(v);
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    T w = lane < nw ? scratch[lane] : T(0);
    w = warp_incl_scan(w);
    scratch[lane] = w;
  }
  __syncthreads();
  const T before = warp > 0 ? scratch[warp - 1] : T(0);
  *total = scratch[nw - 1];
  __syncthreads();
  return before + incl - v;
}

// ------------------------------------------------------------ 1. mean query
template <int D>
__global__ void __launch_bounds__(256) sa_meanq_kernel(const uint16_t* __restrict__ q,
                                                       uint16_t* __restrict__ qhi,
                                                       uint16_t* __restrict__ qlo, int64_t G,
                                                       int32_t Nq, int32_t M) {
  constexpr int kChunks = D / 8, kLanes = 256 / kChunks;
  __shared__ float part[kLanes][D];
  const int64_t u = blockIdx.x, bh = u / G, g = u % G;
  const int64_t r0 = g * M, r1 = min64(r0 + M, Nq);
  const int c = threadIdx.x % kChunks, rl = threadIdx.x / kChunks;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const uint16_t* base = q + bh * Nq * D + c * 8;
  for (int64_t r = r0 + rl; r < r1; r += kLanes) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(base + r * D));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc[2 * e] += __uint_as_float(ws[e] << 16);
      acc[2 * e + 1] += __uint_as_float(ws[e] & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) part[rl][c * 8 + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kLanes; ++i) s += part[i][threadIdx.x];
    const float mean = s / static_cast<float>(r1 - r0);
    const uint16_t hi = bf16_rn(mean);
    qhi[u * D + threadIdx.x] = hi;
    qlo[u * D + threadIdx.x] = bf16_rn(mean - bf16_f(hi));
  }
}

// ------------------------------------------------------------ 2. scores
struct ScoreArgs {
  const uint16_t* k;
  const uint16_t* qhi;
  const uint16_t* qlo;
  float* scores;
  int64_t ld, G, units;
  int32_t Nk, gchunks, ksplit, tiles_per_split, ntiles;
  float scale;
  int32_t* status;
};

template <int D>
struct ScoreCfg {
  static constexpr int kStages = 3;
  static constexpr int kThreads = 32 * 6;  // 4 epilogue warps, 1 MMA warp, 1 TMA warp
  static constexpr int kTile = 128 * D * 2;  // 128 rows of d bf16
  // Each epilogue warp stages its 32 keys x 128 rows of fp32 scores (16 KB)
  // and writes them with one TMA store.
  static constexpr int kOutSlab = 32 * 128 * 4;
  static constexpr int kSmemBytes = 1024 + 2 * kTile + kStages * kTile + 4 * kOutSlab + 1024;
  static constexpr int kTmemCols = 256;
};

struct ScoreBars {
  uint64_t kfull[3], kempty[3];
  uint64_t qfull, qempty, drain;
  uint64_t dfull[2], dempty[2];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void score_unit(const ScoreArgs& a, int64_t u, int64_t* bh, int* gc,
                                           int* t0, int* t1) {
  const int64_t per_bh = int64_t(a.gchunks) * a.ksplit;
  *bh = u / per_bh;
  const int rem = static_cast<int>(u % per_bh);
  *gc = rem / a.ksplit;
  const int ks = rem % a.ksplit;
  *t0 = ks * a.tiles_per_split;
  *t1 = min(*t0 + a.tiles_per_split, a.ntiles);
}

template <int D>
__global__ void __launch_bounds__(ScoreCfg<D>::kThreads, 1)
    sa_score_kernel(const ScoreArgs a, const __grid_constant__ CUtensorMap tm_qhi,
                    const __grid_constant__ CUtensorMap tm_qlo, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_out) {
  using C = ScoreCfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQh = smem;
  uint8_t* sQl = sQh + C::kTile;
  uint8_t* sK = sQl + C::kTile;
  uint8_t* sOut = sK + S * C::kTile;
  ScoreBars* bars = reinterpret_cast<ScoreBars*>(sOut + 4 * C::kOutSlab);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars->kfull[s], 1);
      mbar_init(&bars->kempty[s], 1);
    }
    mbar_init(&bars->qfull, 1);
    mbar_init(&bars->qempty, 1);
    mbar_init(&bars->drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->dfull[b], 1);
      mbar_init(&bars->dempty[b], 128);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < 4) {
    // ------------------------------------------------------------ epilogue
    // Lane = key: the warp's 32 keys x 128 mean-query rows go to its slab as
    // [row][key] and leave with one TMA store (clipped at Nk and at G).
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float* slab = reinterpret_cast<float*>(sOut + warp * C::kOutSlab);
    const uint32_t slab_addr = smem_u32(slab);
    uint32_t t = 0;
    for (int64_t u = blockIdx.x; u < a.units; u += gridDim.x) {
      int64_t bh;
      int gc, t0, t1;
      score_unit(a, u, &bh, &gc, &t0, &t1);
      for (int tile = t0; tile < t1; ++tile, ++t) {
        const uint32_t b = t & 1;
        if (!mbar_wait(&bars->dfull[b], (t >> 1) & 1, abort)) goto done;
        tc_fence_after();
        float x[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tmem + lane_base + b * 128 + c * 32, reinterpret_cast<uint32_t*>(x + c * 32));
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bars->dempty[b]);
        // the previous tile's store must have read the slab
        if (lane == 0) bulk_wait_read();
        __syncwarp();
#pragma unroll
        for (int gi = 0; gi < 128; ++gi) slab[gi * 32 + lane] = x[gi] * a.scale;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tm_out, slab_addr, tile * 128 + warp * 32, gc * 128, static_cast<int>(bh));
          bulk_commit();
        }
      }
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16(128, 128, false, false);
      const uint32_t qh = smem_u32(sQh), ql = smem_u32(sQl), kb = smem_u32(sK);
      uint32_t t = 0, un = 0;
      bool ok = true;
      for (int64_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        int64_t bh;
        int gc, t0, t1;
        score_unit(a, u, &bh, &gc, &t0, &t1);
        if (t1 <= t0) continue;
        if (!mbar_wait(&bars->qfull, un & 1, abort)) break;
        for (int tile = t0; tile < t1; ++tile, ++t) {
          const uint32_t s = t % S, b = t & 1;
          if (!mbar_wait(&bars->kfull[s], (t / S) & 1, abort) ||
              !mbar_wait(&bars->dempty[b], ((t >> 1) & 1) ^ 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem + b * 128;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 128 * 128 + (kk & 3) * 32;
            mma_ss(d_tmem, sw128_desc(kb + s * C::kTile + off, 16, 1024), sw128_desc(qh + off, 16, 1024),
                   kIdesc, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 128 * 128 + (kk & 3) * 32;
            mma_ss(d_tmem, sw128_desc(kb + s * C::kTile + off, 16, 1024), sw128_desc(ql + off, 16, 1024),
                   kIdesc, 1u);
          }
          mma_commit(&bars->dfull[b]);
          mma_commit(&bars->kempty[s]);
          if (tile == t1 - 1) mma_commit(&bars->qempty);
        }
        ++un;
      }
      mma_commit(&bars->drain);
      const long long c0 = clock64();
      while (!mbar_test(&bars->drain, 0) && clock64() - c0 < kWaitLimitCycles) {
      }
    }
  } else if (lane == 0) {
    // ------------------------------------------------------------ loads (TMA)
    const uint32_t qh = smem_u32(sQh), ql = smem_u32(sQl), kb = smem_u32(sK);
    uint32_t t = 0, un = 0;
    for (int64_t u = blockIdx.x; u < a.units; u += gridDim.x) {
      int64_t bh;
      int gc, t0, t1;
      score_unit(a, u, &bh, &gc, &t0, &t1);
      if (t1 <= t0) continue;
      if (un > 0 && !mbar_wait(&bars->qempty, (un - 1) & 1, abort)) goto done;
      // mean-query rows bh*G + g0 .. +127 (rows of the next head or past the
      // end only feed columns that are never written)
      const int qrow = static_cast<int>(bh * a.G + int64_t(gc) * 128);
      mbar_expect_tx(&bars->qfull, 2 * C::kTile);
#pragma unroll
      for (int cb = 0; cb < D / 64; ++cb) {
        tma_load_2d(qh + cb * 128 * 128, &tm_qhi, 64 * cb, qrow, &bars->qfull);
        tma_load_2d(ql + cb * 128 * 128, &tm_qlo, 64 * cb, qrow, &bars->qfull);
      }
      for (int tile = t0; tile < t1; ++tile, ++t) {
        const uint32_t s = t % S;
        if (!mbar_wait(&bars->kempty[s], ((t / S) & 1) ^ 1, abort)) goto done;
        mbar_expect_tx(&bars->kfull[s], C::kTile);
        const int krow = static_cast<int>(bh * a.Nk + int64_t(tile) * 128);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_2d(kb + s * C::kTile + cb * 128 * 128, &tm_k, 64 * cb, krow, &bars->kfull[s]);
      }
      ++un;
    }
  }
done:
  // score stores must be complete (and off the slabs) before the block exits
  if (warp < 4 && lane == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && bars->abort) report(a.status, SA_DEVERR_TIMEOUT);
  if (warp == 4) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------ 3. select
struct SelArgs {
  const float* scores;
  int64_t ld;
  int32_t Nk, mode;
  int64_t topk;
  float log_tau;  // ln(threshold); -inf for 0
  double mass;
  uint32_t* cut;
  int32_t* ties;
  int64_t* counts;
  int32_t* col_idx;      // TOPK only: lists are emitted by the select kernel
  int64_t col_capacity;
  int32_t mask_words;    // TOPK: words of the kept-key bitmask (0: emit by re-reading the row)
  int32_t level;         // THRESHOLD compares the score itself with ln(threshold)
};

constexpr int kSelThreads = 256;            // one row per block, 4 blocks resident per SM
constexpr size_t kSelSmemBudget = 75 * 1024;  // dynamic shared memory per block: 3 or 4 blocks per SM
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBins = 1024;                 // linear bins over the undecided score range
constexpr int kBinsPerThread = kBins / kSelThreads;
constexpr int kLevels = 3;                  // bin refinements of the crossing bin
constexpr int kRank = 512;                  // exact ranking once this few keys are undecided
constexpr int kWindow = 8192;               // keys the sampled bracket may hold (indices)
constexpr int kSampleMax = kWindow;         // samples share the bracket's storage
constexpr int kNoSample = 4096;             // rows this short are selected without a sample
constexpr int kUnroll = 4;                  // float4 loads in flight per lane
constexpr int kWinUnroll = 4;               // ... in the bracket pass (16 keys per lane)
constexpr float kMassOne = 4294967296.0f;   // fixed-point unit of probability mass (2^32)

// Probability mass exp(x - max) of one key in 2^-32 units; integer sums are
// exact and order-independent, so every pass agrees on every partial sum.
__device__ __forceinline__ unsigned long long fixed_mass(float x, float rmax) {
  return __float2ull_rn(expf(x - rmax) * kMassOne);
}

// One refinement level: keys in the undecided range are spread over kBins
// linear bins starting at lo; `pick` is the bin that holds the cut.
struct SelLevel {
  float lo, inv;
  int pick;
};

__device__ __forceinline__ int lin_bin(float x, float lo, float inv, int nb) {
  const float f = (x - lo) * inv;
  return f <= 0.f ? 0 : (f >= float(nb - 1) ? nb - 1 : static_cast<int>(f));
}

struct SelSmem {
  uint32_t hist[kBins];
  unsigned long long hmass[kBins];
  float rx[kRank];
  int32_t rj[kRank];
  union {
    struct {
      int32_t j[kWindow];
    } win;
    float sample[kSampleMax];
  } u;
  SelLevel levels[kLevels];
  float fred[3][32];
  int64_t scan_c[32], scan_m[32];
  int32_t claim, n_rank, n_win, found_cnt, cut_rank;
  int64_t found_above_cnt, found_above_mass, cut_greater;
  float cut_x;
  int32_t seg_sel[kSelWarps], seg_tie[kSelWarps];
};

// Keys of one row: either the whole score row or the bracketed window.
struct RowSrc {
  const float* s;
  int n;
  __device__ __forceinline__ float x(int i) const { return s[i]; }
  __device__ __forceinline__ int j(int i) const { return i; }
};
// Keys of the bracketed window: indices in shared memory, scores re-read
// from the row (in L2 after the window pass).
struct WinSrc {
  const float* xs;
  const int32_t* js;
  int n;
  __device__ __forceinline__ float x(int i) const { return xs[i]; }
  __device__ __forceinline__ int j(int i) const { return js[i]; }
};
struct RowIdxSrc {
  const float* s;
  const int32_t* js;
  int n;
  __device__ __forceinline__ float x(int i) const { return s[js[i]]; }
  __device__ __forceinline__ int j(int i) const { return js[i]; }
};

__device__ __forceinline__ float block_min(float v, SelSmem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) sm.fred[0][warp] = v;
  __syncthreads();
  v = sm.fred[0][0];
#pragma unroll
  for (int w = 1; w < kSelWarps; ++w) v = fminf(v, sm.fred[0][w]);
  return v;
}
__device__ __forceinline__ float block_max(float v, SelSmem& sm) { return -block_min(-v, sm); }

__device__ __forceinline__ float f4_get(const float4& v, int e) {
  return e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
}

// Calls f(j, x) for every key of a row; lanes read float4s, kUnroll of them
// in flight, and the tail that does not fill a float4 is read singly.
template <class F>
__device__ __forceinline__ void for_each_key(const float* s, int Nk, F&& f) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nv = Nk >> 2;
  const float4* s4 = reinterpret_cast<const float4*>(s);
  for (int b = warp * 32 * kUnroll; b < nv; b += kSelThreads * kUnroll) {
    float4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i4 = b + u * 32 + lane;
      v[u] = i4 < nv ? __ldg(s4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i4 = b + u * 32 + lane;
      if (i4 < nv) {
#pragma unroll
        for (int e = 0; e < 4; ++e) f(4 * i4 + e, f4_get(v[u], e));
      }
    }
  }
  for (int j = 4 * nv + threadIdx.x; j < Nk; j += kSelThreads) f(j, s[j]);
}

// The exact selection among the undecided keys of `src` (all with scores in
// [lo0, hi0]); `above_cnt` / `above_mass` account for the keys above hi0.
// Keys are ranked by (score descending, index ascending).  TOPK takes rank
// k-1 as the cut; MASS the first key at which the running fixed-point mass
// reaches `target`.  Returns the cut as (order key, kept ties, row count).
template <class Src>
__device__ void exact_select(const Src& src, float lo0, float hi0, int64_t k, int64_t target,
                             bool by_mass, float rmax, int64_t above_cnt, int64_t above_mass,
                             int64_t keep_all_count, SelSmem& sm, uint32_t* cut, int32_t* ties,
                             int64_t* count) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int nlev = 0;
  bool ranked = false, all_equal = false;
  float lo = lo0, hi = hi0;
  for (int lv = 0; lv < kLevels; ++lv) {
    if (!(hi > lo)) {  // every undecided key has the same score
      all_equal = true;
      break;
    }
    const float inv = float(kBins) / (hi - lo);
    for (int i = tid; i < kBins; i += kSelThreads) {
      sm.hist[i] = 0;
      if (by_mass) sm.hmass[i] = 0ull;
    }
    if (tid == 0) {
      sm.levels[lv].lo = lo;
      sm.levels[lv].inv = inv;
      sm.levels[lv].pick = -1;
      sm.claim = -1;
    }
    __syncthreads();
    SelLevel lvl[kLevels];
#pragma unroll
    for (int i = 0; i < kLevels; ++i) lvl[i] = sm.levels[i];
    for (int base = warp * 32; base < src.n; base += kSelThreads) {
      const int i = base + lane;
      const float x = i < src.n ? src.x(i) : -INFINITY;
      bool in = i < src.n && x >= lo0 && x <= hi0;
#pragma unroll
      for (int l = 0; l < kLevels; ++l)
        if (l < lv) in = in && lin_bin(x, lvl[l].lo, lvl[l].inv, kBins) == lvl[l].pick;
      const int b = in ? lin_bin(x, lo, inv, kBins) : -1;
      const unsigned same = __match_any_sync(0xffffffffu, b);
      if (in && lane == __ffs(same) - 1) atomicAdd(&sm.hist[b], static_cast<uint32_t>(__popc(same)));
      if (in && by_mass) atomicAdd(&sm.hmass[b], fixed_mass(x, rmax));
    }
    __syncthreads();
    const int top = kBins - 1 - kBinsPerThread * tid;
    int64_t c2 = 0, m2 = 0;
#pragma unroll
    for (int e = 0; e < kBinsPerThread; ++e) {
      c2 += sm.hist[top - e];
      if (by_mass) m2 += int64_t(sm.hmass[top - e]);
    }
    int64_t ctot, mtot = 0;
    const int64_t cex = block_excl_scan<int64_t>(c2, &ctot, sm.scan_c);
    const int64_t mex = by_mass ? block_excl_scan<int64_t>(m2, &mtot, sm.scan_m) : 0;
    int64_t cum_c = above_cnt + cex, cum_m = above_mass + mex;
    for (int e = 0; e < kBinsPerThread; ++e) {
      const int bin = top - e;
      const int64_t bc = sm.hist[bin], bm = by_mass ? int64_t(sm.hmass[bin]) : 0;
      const bool cross = by_mass ? (bm > 0 && cum_m + bm >= target && cum_m < target)
                                 : (bc > 0 && cum_c + bc >= target && cum_c < target);
      if (cross && atomicCAS(&sm.claim, -1, bin) == -1) {
        sm.found_cnt = static_cast<int32_t>(bc);
        sm.found_above_cnt = cum_c - above_cnt;
        sm.found_above_mass = cum_m - above_mass;
      }
      cum_c += bc;
      cum_m += bm;
    }
    __syncthreads();
    const int bin = sm.claim;
    if (bin < 0) break;  // mass target beyond the rounded total
    if (tid == 0) sm.levels[lv].pick = bin;
    above_cnt += sm.found_above_cnt;
    above_mass += sm.found_above_mass;
    nlev = lv + 1;
    const int bc = sm.found_cnt;
    lo = lvl[lv].lo + float(bin) / inv;  // the picked bin's interval is the next range
    hi = lvl[lv].lo + float(bin + 1) / inv;
    __syncthreads();
    if (bc <= kRank) {
      ranked = true;
      break;
    }
  }
  __syncthreads();
  if (nlev == 0 && !all_equal) {
    *cut = 0;  // keep every key
    *ties = 0;
    *count = keep_all_count;
    return;
  }
  SelLevel lvl[kLevels];
#pragma unroll
  for (int i = 0; i < kLevels; ++i) lvl[i] = sm.levels[i];
  if (tid == 0) {
    sm.n_rank = 0;
    sm.cut_rank = -1;
  }
  __syncthreads();
  for (int base = warp * 32; base < src.n; base += kSelThreads) {
    const int i = base + lane;
    const float x = i < src.n ? src.x(i) : -INFINITY;
    bool in = i < src.n && x >= lo0 && x <= hi0;
#pragma unroll
    for (int l = 0; l < kLevels; ++l)
      if (l < nlev) in = in && lin_bin(x, lvl[l].lo, lvl[l].inv, kBins) == lvl[l].pick;
    const unsigned ballot = __ballot_sync(0xffffffffu, in);
    int slot0 = 0;
    if (lane == 0 && ballot) slot0 = atomicAdd(&sm.n_rank, __popc(ballot));
    slot0 = __shfl_sync(0xffffffffu, slot0, 0);
    const int slot = slot0 + __popc(ballot & ((1u << lane) - 1u));
    if (in && slot < kRank) {
      sm.rx[slot] = x;
      sm.rj[slot] = src.j(i);
    }
  }
  __syncthreads();
  const int n_und = sm.n_rank;
  const int nc = n_und < kRank ? n_und : kRank;
  if (!ranked || n_und > kRank) {
    // The undecided keys share one score (the bin is below float
    // resolution): the cut is that score and the tie rule decides.
    const float xv = sm.rx[0];
    *cut = order_key(xv);
    int32_t t;
    if (by_mass) {
      const int64_t e = static_cast<int64_t>(fixed_mass(xv, rmax));
      const int64_t need = e > 0 ? (target - above_mass + e - 1) / e : 1;
      t = static_cast<int32_t>(need < 1 ? 1 : (need > n_und ? n_und : need));
    } else {
      t = static_cast<int32_t>(min64(k - above_cnt, n_und));
    }
    *ties = t;
    *count = above_cnt + t;
    return;
  }
  for (int c = tid; c < nc; c += kSelThreads) {
    const float xc = sm.rx[c];
    const int jc = sm.rj[c];
    int rank = 0, greater = 0;
    int64_t before_m = 0;
    for (int o = 0; o < nc; ++o) {
      const float xo = sm.rx[o];
      const bool ahead = xo > xc || (xo == xc && sm.rj[o] < jc);
      rank += ahead;
      greater += xo > xc;
      if (by_mass && ahead) before_m += int64_t(fixed_mass(xo, rmax));
    }
    bool is_cut;
    if (by_mass) {
      const int64_t incl = above_mass + before_m + int64_t(fixed_mass(xc, rmax));
      is_cut = incl >= target && above_mass + before_m < target;
    } else {
      is_cut = above_cnt + rank == k - 1;
    }
    if (is_cut) {
      sm.cut_rank = rank;
      sm.cut_x = xc;
      sm.cut_greater = greater;
    }
  }
  __syncthreads();
  if (sm.cut_rank < 0) {  // rounding left the mass target unreached
    *cut = 0;
    *ties = 0;
    *count = keep_all_count;
  } else {
    *cut = order_key(sm.cut_x);
    *count = above_cnt + sm.cut_rank + 1;
    *ties = static_cast<int32_t>(*count - (above_cnt + sm.cut_greater));
  }
}

// Writes the ascending indices of a row's kept keys (score above the cut, or
// equal to it among the first `ties` such keys) to col_idx[base, end).  Each
// warp owns one contiguous segment of the row: it counts its kept keys, the
// segments' offsets come from one block-wide exchange, and a second read of
// the segment writes the indices in order.
__device__ void emit_row(const float* s, int Nk, uint32_t ck, int64_t nt, int64_t base, int64_t end,
                         int32_t* col_idx, int32_t* seg_sel, int32_t* seg_tie) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nv = (Nk + 3) >> 2;  // float4 chunks, the last one possibly partial
  const int per = (nv + kSelWarps - 1) / kSelWarps;
  const int v0 = warp * per, v1 = min(v0 + per, nv);
  const float4* s4 = reinterpret_cast<const float4*>(s);
  auto load4 = [&](int i4, float* x) {
    if (4 * i4 + 3 < Nk) {
      const float4 v = __ldg(s4 + i4);
      x[0] = v.x;
      x[1] = v.y;
      x[2] = v.z;
      x[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = 4 * i4 + e < Nk ? s[4 * i4 + e] : -INFINITY;
    }
  };
  int n_sel = 0, n_tie = 0;
  for (int b = v0; b < v1; b += 32 * kUnroll) {
    float x[kUnroll][4];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i4 = b + u * 32 + lane;
      if (i4 < v1) load4(i4, x[u]);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i4 = b + u * 32 + lane;
      if (i4 < v1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool in = 4 * i4 + e < Nk;
          const uint32_t kx = order_key(x[u][e]);
          n_sel += in && kx > ck;
          n_tie += in && kx == ck;
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    n_sel += __shfl_xor_sync(0xffffffffu, n_sel, o);
    n_tie += __shfl_xor_sync(0xffffffffu, n_tie, o);
  }
  __syncthreads();
  if (lane == 0) {
    seg_sel[warp] = n_sel;
    seg_tie[warp] = n_tie;
  }
  __syncthreads();
  int64_t sb = 0, tb = 0;
  for (int w = 0; w < warp; ++w) {
    sb += seg_sel[w];
    tb += seg_tie[w];
  }
  for (int b0 = v0; b0 < v1; b0 += 32 * kUnroll) {
    float xs[kUnroll][4];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i4 = b0 + u * 32 + lane;
      if (i4 < v1) load4(i4, xs[u]);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
    const int b = b0 + u * 32;
    if (b >= v1) break;
    const int i4 = b + lane;
    float* x = xs[u];
    bool sel[4], tie[4];
    int cs = 0, ct = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool in = i4 < v1 && 4 * i4 + e < Nk;
      const uint32_t kx = in ? order_key(x[e]) : 0u;
      sel[e] = in && kx > ck;
      tie[e] = in && kx == ck;
      cs += sel[e];
      ct += tie[e];
    }
    // exclusive prefix of (sel, tie) counts over the warp's lanes
    int ps = cs, pt = ct;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a1 = __shfl_up_sync(0xffffffffu, ps, o), a2 = __shfl_up_sync(0xffffffffu, pt, o);
      if (lane >= o) {
        ps += a1;
        pt += a2;
      }
    }
    const int tot_s = __shfl_sync(0xffffffffu, ps, 31), tot_t = __shfl_sync(0xffffffffu, pt, 31);
    int64_t ls = sb + ps - cs, lt = tb + pt - ct;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (sel[e]) {
        const int64_t pos = base + ls + min64(lt, nt);
        if (pos < end) col_idx[pos] = 4 * i4 + e;
        ++ls;
      } else if (tie[e]) {
        const int64_t pos = base + ls + lt;
        if (lt < nt && pos < end) col_idx[pos] = 4 * i4 + e;
        ++lt;
      }
    }
    sb += tot_s;
    tb += tot_t;
    }
  }
}

__device__ __forceinline__ bool by_mass_mode(const SelArgs& a) { return a.mode != SA_SELECT_TOPK; }

// Writes the indices of the set bits of kept[0, words) in ascending order to
// col_idx[base, ...).  Warp w owns a contiguous run of words; the runs'
// offsets come from one block scan of their popcounts.  A warp takes its run
// 32 words at a time (lane = word): a warp scan of the popcounts places each
// word's keys in the warp's staging buffer (1024 entries of shared memory),
// and the pass leaves in coalesced stores.
__device__ void emit_mask(const uint32_t* kept, int words, int64_t base, int32_t* col_idx,
                          int64_t* scratch, int32_t* stage_all) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = (words + kSelWarps - 1) / kSelWarps;
  const int w0 = min(words, warp * per), w1 = min(words, w0 + per);
  int64_t n = 0;
  for (int w = w0 + lane; w < w1; w += 32) n += __popc(kept[w]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  // block scan over the warps' counts (only lane 0 of each warp contributes)
  int64_t total;
  const int64_t before = block_excl_scan<int64_t>(lane == 0 ? n : 0, &total, scratch);
  int64_t pos = base + __shfl_sync(0xffffffffu, before, 0);
  int32_t* stage = stage_all + warp * 1024;
  for (int wb = w0; wb < w1; wb += 32) {
    const int w = wb + lane;
    uint32_t bits = w < w1 ? kept[w] : 0u;
    const int c = __popc(bits);
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const int cnt = __shfl_sync(0xffffffffu, x, 31);
    int off = x - c;
    while (bits) {
      stage[off++] = w * 32 + (__ffs(bits) - 1);
      bits &= bits - 1;
    }
    __syncwarp();
    for (int i = lane; i < cnt; i += 32) col_idx[pos + i] = stage[i];
    __syncwarp();
    pos += cnt;
  }
}

__global__ void __launch_bounds__(kSelThreads, 4) sa_select_kernel(const SelArgs a) {
  extern __shared__ uint8_t sel_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(sel_raw);
  // TOPK: bit j of kept[j / 32] marks key j as kept (keys above the bracket
  // during the window pass, kept keys of the window after the selection).
  uint32_t* kept = reinterpret_cast<uint32_t*>(sel_raw + sizeof(SelSmem));
  const bool use_mask = !by_mass_mode(a) && a.col_idx && a.mask_words > 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const float* s = a.scores + row * a.ld;
  const int Nk = a.Nk;
  const bool by_mass = a.mode == SA_SELECT_MASS;
  uint32_t cut = 0;
  int32_t ties = 0;
  int64_t count = Nk;
  // Every later phase reads this row (the sample, the bracket pass, the
  // window's scores, the emission): start moving all of it into L2 now, so
  // that those phases wait on L2 rather than DRAM latency.
  for (int off = tid * 32; off < Nk; off += kSelThreads * 32) prefetch_l2(s + off);

  if (a.mode == SA_SELECT_THRESHOLD) {
    // keep p_j >= tau  <=>  sigma_j >= ln tau + max + ln Z
    float mx = -INFINITY, z = 0.f;
    for_each_key(s, Nk, [&](int, float x) {
      if (x > mx) {
        z = z * expf(mx - x) + 1.f;
        mx = x;
      } else {
        z += expf(x - mx);
      }
    });
    const float rmax = block_max(mx, sm);
    float zr = (mx == -INFINITY) ? 0.f : z * expf(mx - rmax);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zr += __shfl_xor_sync(0xffffffffu, zr, o);
    __syncthreads();
    if (lane == 0) sm.fred[1][warp] = zr;
    __syncthreads();
    float rz = 0.f;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) rz += sm.fred[1][w];
    // LEVEL (dense-step statistics): the score is already ln of a probability
    const float c = a.level ? a.log_tau : a.log_tau + rmax + logf(rz);
    const uint32_t kc = (c == -INFINITY) ? 0u : order_key(c);
    int64_t n = 0;
    for_each_key(s, Nk, [&](int, float x) { n += order_key(x) >= kc; });
    int64_t total;
    block_excl_scan<int64_t>(n, &total, sm.scan_c);
    if (total > 0) {
      cut = kc > 0 ? kc - 1 : 0u;  // keys > kc - 1  <=>  keys >= kc
      ties = 0;
      count = total;
    } else {
      cut = order_key(rmax);  // none qualifies: the top-ranked key only
      ties = 1;
      count = 1;
    }
  } else if (by_mass && a.mass >= 1.0) {
    cut = 0;  // the whole mass needs every key
    ties = 0;
    count = Nk;
  } else {
    const int64_t k = min64(max64(a.topk, 1), Nk);
    float rmax = 0.f;
    // Rank or fixed-point mass the cut must reach.  Every comparison below is
    // between integers (FP64 is slow on this part): for an integer sum x,
    // x >= mass * total  <=>  x >= ceil(mass * total).
    int64_t target = k;
    if (by_mass) {
      float mx = -INFINITY;
      for_each_key(s, Nk, [&](int, float x) { mx = fmaxf(mx, x); });
      rmax = block_max(mx, sm);
      unsigned long long zt = 0;
      for_each_key(s, Nk, [&](int, float x) { zt += fixed_mass(x, rmax); });
      int64_t ztot;
      block_excl_scan<int64_t>(static_cast<int64_t>(zt), &ztot, sm.scan_m);
      target = static_cast<int64_t>(ceil(a.mass * static_cast<double>(ztot)));
    }
    // ---- bracket the cut from an evenly strided sample of the row
    float lo = -INFINITY, hi = INFINITY;
    if (Nk > kNoSample) {
      const int S = Nk / 4 < kSampleMax ? (Nk / 4 > 1024 ? Nk / 4 : 1024) : kSampleMax;
      const int stride = Nk / S;  // >= 1: samples j = i*stride, evenly spread over the row
      float smn = INFINITY, smx = -INFINITY;
#pragma unroll 8
      for (int i = tid; i < S; i += kSelThreads) {
        const float x = __ldg(s + i * stride);
        sm.u.sample[i] = x;
        smn = fminf(smn, x);
        smx = fmaxf(smx, x);
      }
      smn = block_min(smn, sm);
      smx = block_max(smx, sm);
      if (smx > smn) {
        const float inv = float(kBins) / (smx - smn);
        for (int i = tid; i < kBins; i += kSelThreads) {
          sm.hist[i] = 0;
          if (by_mass) sm.hmass[i] = 0ull;
        }
        __syncthreads();
        for (int i = tid; i < S; i += kSelThreads) {
          const float x = sm.u.sample[i];
          const int bn = lin_bin(x, smn, inv, kBins);
          atomicAdd(&sm.hist[bn], 1u);
          if (by_mass) atomicAdd(&sm.hmass[bn], fixed_mass(x, rmax));
        }
        __syncthreads();
        const int top = kBins - 1 - kBinsPerThread * tid;
        int64_t c4 = 0, m4 = 0;
#pragma unroll
        for (int e = 0; e < kBinsPerThread; ++e) {
          c4 += sm.hist[top - e];
          if (by_mass) m4 += int64_t(sm.hmass[top - e]);
        }
        int64_t ctot, mtot = 0;
        const int64_t cex = block_excl_scan<int64_t>(c4, &ctot, sm.scan_c);
        const int64_t mex = by_mass ? block_excl_scan<int64_t>(m4, &mtot, sm.scan_m) : 0;
        // expected rank of the cut among the samples, counted from the top
        float p;
        if (by_mass) {
          if (tid == 0) sm.found_above_cnt = S;  // no crossing: bracket everything below the top
          __syncthreads();
          const int64_t share = static_cast<int64_t>(ceil(a.mass * static_cast<double>(mtot)));
          int64_t cm = mex, cc = cex;
          for (int e = 0; e < kBinsPerThread; ++e) {
            const int64_t bm = int64_t(sm.hmass[top - e]), bc = sm.hist[top - e];
            if (bm > 0 && cm + bm >= share && cm < share) sm.found_above_cnt = cc + bc;
            cm += bm;
            cc += bc;
          }
          __syncthreads();
          p = float(sm.found_above_cnt);
        } else {
          p = float(k) * float(S) / float(Nk);
        }
        const float q = fminf(fmaxf(p / float(S), 0.f), 1.f);
        const float delta = 5.f * sqrtf(float(S) * q * (1.f - q)) + 16.f;
        const float r_hi = p - delta, r_lo = p + delta;  // sample ranks bounding the cut
        if (tid == 0) {
          sm.fred[2][0] = INFINITY;
          sm.fred[2][1] = -INFINITY;
        }
        __syncthreads();
        int64_t cc = cex;
        for (int e = 0; e < kBinsPerThread; ++e) {
          const int bn = top - e;
          const int64_t bc = sm.hist[bn];
          // this bin covers sample ranks [cc, cc + bc)
          if (bc > 0 && r_hi >= float(cc) && r_hi < float(cc + bc)) sm.fred[2][0] = smn + float(bn + 1) / inv;
          if (bc > 0 && r_lo >= float(cc) && r_lo < float(cc + bc)) sm.fred[2][1] = smn + float(bn) / inv;
          cc += bc;
        }
        __syncthreads();
        hi = r_hi >= 0.f ? sm.fred[2][0] : INFINITY;
        lo = r_lo < float(S) ? sm.fred[2][1] : -INFINITY;
      } else {
        lo = hi = smn;  // flat sample: try its single value, fall back if wrong
      }
      __syncthreads();  // the sample's storage becomes the bracket's
    }
    // ---- one pass: count the keys above the bracket, collect those inside
    if (tid == 0) sm.n_win = 0;
    __syncthreads();
    int64_t c_above = 0;
    unsigned long long m_above = 0, m_win = 0;
    {
      const int nv = Nk >> 2;
      const float4* s4 = reinterpret_cast<const float4*>(s);
      constexpr int U = kWinUnroll;
      // Keys past the row read as NaN: every comparison with them is false.
      const float nan = __int_as_float(0x7fffffff);
      for (int b = warp * 32 * U; b < nv + 32 * U; b += kSelThreads * U) {
        float x[U][4];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i4 = b + u * 32 + lane;
          if (i4 < nv) {
            const float4 v = __ldg(s4 + i4);
            x[u][0] = v.x;
            x[u][1] = v.y;
            x[u][2] = v.z;
            x[u][3] = v.w;
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) x[u][e] = 4 * i4 + e < Nk ? s[4 * i4 + e] : nan;
          }
        }
        if (b >= nv && (4 * b >= Nk)) break;
        // bit u*4+e: key 4*(b + 32u + lane) + e
        uint32_t in_mask = 0, above_bits = 0;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float xv = x[u][e];
            const bool above = xv > hi;
            const bool inw = xv >= lo && !above;
            above_bits |= (above ? 1u : 0u) << (u * 4 + e);
            in_mask |= (inw ? 1u : 0u) << (u * 4 + e);
            if (by_mass && (above || inw)) {
              const unsigned long long fm = fixed_mass(xv, rmax);
              if (above) m_above += fm;
              else m_win += fm;
            }
          }
        c_above += __popc(above_bits);
        const int n_in = __popc(in_mask);
        if (use_mask) {
          // eight lanes hold the 32 keys of one mask word: OR their nibbles
#pragma unroll
          for (int u = 0; u < U; ++u) {
            uint32_t w = ((above_bits >> (u * 4)) & 0xFu) << (4 * (lane & 7));
            w |= __shfl_xor_sync(0xffffffffu, w, 1);
            w |= __shfl_xor_sync(0xffffffffu, w, 2);
            w |= __shfl_xor_sync(0xffffffffu, w, 4);
            const int word = (b + u * 32 + lane) >> 3;
            if ((lane & 7) == 0 && word < a.mask_words) kept[word] = w;
          }
        }
        // warp-aggregated append of this lane's in-bracket keys
        int pre = n_in;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, pre, o);
          if (lane >= o) pre += t;
        }
        const int tot = __shfl_sync(0xffffffffu, pre, 31);
        if (tot == 0) continue;
        int slot0 = 0;
        if (lane == 0) slot0 = atomicAdd(&sm.n_win, tot);
        int slot = __shfl_sync(0xffffffffu, slot0, 0) + pre - n_in;
        for (uint32_t m = in_mask; m; m &= m - 1, ++slot) {
          const int bit = __ffs(m) - 1;
          if (slot < kWindow) sm.u.win.j[slot] = 4 * (b + (bit >> 2) * 32 + lane) + (bit & 3);
        }
      }
    }
    int64_t above_cnt, above_mass = 0, win_mass = 0;
    block_excl_scan<int64_t>(c_above, &above_cnt, sm.scan_c);
    if (by_mass) {
      block_excl_scan<int64_t>(static_cast<int64_t>(m_above), &above_mass, sm.scan_m);
      block_excl_scan<int64_t>(static_cast<int64_t>(m_win), &win_mass, sm.scan_c);
    }
    const int n_win = sm.n_win;
    const bool bracketed =
        n_win <= kWindow && (by_mass ? (above_mass < target && target <= above_mass + win_mass)
                                     : (above_cnt < k && k <= above_cnt + n_win));
    // A window of at most kWindow/2 keys gets its scores copied next to the
    // indices (one gather from L2), so the selection passes read shared memory.
    const bool win_x = n_win <= kWindow / 2;
    float* wx = reinterpret_cast<float*>(sm.u.win.j + kWindow / 2);
    if (bracketed) {
      float wmn = INFINITY, wmx = -INFINITY;
      for (int i = tid; i < n_win; i += kSelThreads) {
        const float xv = s[sm.u.win.j[i]];
        if (win_x) wx[i] = xv;
        wmn = fminf(wmn, xv);
        wmx = fmaxf(wmx, xv);
      }
      wmn = block_min(wmn, sm);  // (its barriers also publish wx)
      wmx = block_max(wmx, sm);
      if (win_x)
        exact_select(WinSrc{wx, sm.u.win.j, n_win}, wmn, wmx, k, target, by_mass, rmax, above_cnt,
                     above_mass, Nk, sm, &cut, &ties, &count);
      else
        exact_select(RowIdxSrc{s, sm.u.win.j, n_win}, wmn, wmx, k, target, by_mass, rmax, above_cnt,
                     above_mass, Nk, sm, &cut, &ties, &count);
    } else {
      // The sample missed (or the bracket overflowed): select over the row.
      float mn = INFINITY, mx = -INFINITY;
      for_each_key(s, Nk, [&](int, float x) {
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
      });
      mn = block_min(mn, sm);
      mx = block_max(mx, sm);
      exact_select(RowSrc{s, Nk}, mn, mx, k, target, by_mass, rmax, 0, 0, Nk, sm, &cut, &ties, &count);
    }
    if (!by_mass && a.col_idx) {
      // TOPK: every row holds exactly k keys, so row r starts at r*k.
      const int64_t base = row * k;
      if (base + k <= a.col_capacity) {
        // The bitmask serves when the cut fell in the bracket and keeps all of
        // its ties (every key equal to the cut lies in the window); else the
        // row is read again.
        bool from_mask = use_mask && bracketed;
        if (from_mask) {
          int nt = 0;
          for (int i = tid; i < n_win; i += kSelThreads)
            nt += order_key(win_x ? wx[i] : s[sm.u.win.j[i]]) == cut;
          int64_t nt_all;
          block_excl_scan<int64_t>(nt, &nt_all, sm.scan_c);
          from_mask = nt_all == ties;
        }
        if (from_mask) {
          for (int i = tid; i < n_win; i += kSelThreads) {
            const int j = sm.u.win.j[i];
            if (order_key(win_x ? wx[i] : s[j]) >= cut) atomicOr(&kept[j >> 5], 1u << (j & 31));
          }
          __syncthreads();
          // the window's indices are no longer needed: its storage stages the lists
          emit_mask(kept, a.mask_words, base, a.col_idx, sm.scan_c, sm.u.win.j);
        } else {
          emit_row(s, Nk, cut, ties, base, base + k, a.col_idx, sm.seg_sel, sm.seg_tie);
        }
      }
    }
  }
  if (tid == 0) {
    a.cut[row] = cut;
    a.ties[row] = ties;
    a.counts[row] = count;
  }
}

// ------------------------------------------------------------ 4. scan
__global__ void __launch_bounds__(1024) sa_scan_kernel(const int64_t* counts, int64_t rows,
                                                       int64_t* row_ptr, int64_t* nnz,
                                                       int64_t capacity, int32_t* status) {
  __shared__ int64_t scratch[32];
  const int64_t per = (rows + blockDim.x - 1) / blockDim.x;
  const int64_t r0 = min64(rows, threadIdx.x * per), r1 = min64(rows, r0 + per);
  int64_t local = 0;
  for (int64_t r = r0; r < r1; ++r) local += counts[r];
  int64_t total;
  int64_t run = block_excl_scan<int64_t>(local, &total, scratch);
  for (int64_t r = r0; r < r1; ++r) {
    row_ptr[r] = run;
    run += counts[r];
  }
  if (threadIdx.x == 0) {
    row_ptr[rows] = total;
    *nnz = total;
    if (total > capacity) report(status, SA_DEVERR_CAPACITY);
  }
}

// ------------------------------------------------------------ 5. emit
// THRESHOLD and MASS: lists are written after row_ptr is known.
__global__ void __launch_bounds__(kSelThreads) sa_emit_kernel(const float* scores, int64_t ld,
                                                              int32_t Nk, const uint32_t* cut,
                                                              const int32_t* ties,
                                                              const int64_t* row_ptr,
                                                              int32_t* col_idx, int64_t capacity) {
  __shared__ int32_t seg_sel[kSelWarps], seg_tie[kSelWarps];
  const int64_t row = blockIdx.x;
  const int64_t base = row_ptr[row], end = row_ptr[row + 1];
  if (end > capacity) return;  // reported by the scan
  emit_row(scores + row * ld, Nk, cut[row], ties[row], base, end, col_idx, seg_sel, seg_tie);
}

// ------------------------------------------------------------ validator
__global__ void __launch_bounds__(256) sa_validate_kernel(const int64_t* row_ptr,
                                                          const int32_t* col_idx, int64_t rows,
                                                          int64_t nnz, int32_t Nk,
                                                          int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int64_t b0 = row_ptr[row], b1 = row_ptr[row + 1];
  if (lane == 0) {
    if ((row == 0 && b0 != 0) || (row == rows - 1 && b1 != nnz)) report(status, SA_DEVERR_ROW_PTR);
  }
  if (b0 < 0 || b1 < b0 || b1 > nnz) {
    if (lane == 0) report(status, SA_DEVERR_ROW_PTR);
    return;
  }
  bool bad = false;
  for (int64_t p = b0 + lane; p < b1; p += 32) {
    const int32_t x = col_idx[p];
    if (x < 0 || x >= Nk) bad = true;
    if (p > b0 && col_idx[p - 1] >= x) bad = true;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) report(status, SA_DEVERR_INDEX);
}

// ------------------------------------------------------------ host side
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

BuildLayout build_layout(int64_t rows, int32_t Nk, int32_t d) {
  BuildLayout L;
  L.ld = (int64_t(Nk) + 3) & ~int64_t(3);
  size_t off = 0;
  L.qhi = off;
  off = align256(off + size_t(rows) * d * 2);
  L.qlo = off;
  off = align256(off + size_t(rows) * d * 2);
  L.scores = off;
  off = align256(off + size_t(rows) * size_t(L.ld) * 4);
  L.cut = off;
  off = align256(off + size_t(rows) * 4);
  L.ties = off;
  off = align256(off + size_t(rows) * 4);
  L.counts = off;
  off = align256(off + size_t(rows) * 8);
  L.misc = off;
  off = align256(off + 16);
  L.total = off;
  return L;
}

template <int D>
static cudaError_t launch_scores(const BuildArgs& a, int num_sms, cudaStream_t st, int32_t* status) {
  using C = ScoreCfg<D>;
  ScoreArgs s;
  s.k = a.k;
  s.qhi = reinterpret_cast<const uint16_t*>(a.ws + a.L.qhi);
  s.qlo = reinterpret_cast<const uint16_t*>(a.ws + a.L.qlo);
  s.scores = reinterpret_cast<float*>(a.ws + a.L.scores);
  s.ld = a.L.ld;
  s.G = a.G;
  s.Nk = a.Nk;
  s.gchunks = static_cast<int32_t>((a.G + 127) / 128);
  s.ntiles = (a.Nk + 127) / 128;
  const int64_t base = int64_t(a.BH) * s.gchunks;
  int64_t ks = (2 * int64_t(num_sms) + base - 1) / base;
  ks = ks < 1 ? 1 : (ks > s.ntiles ? s.ntiles : ks);
  s.tiles_per_split = static_cast<int32_t>((s.ntiles + ks - 1) / ks);
  s.ksplit = (s.ntiles + s.tiles_per_split - 1) / s.tiles_per_split;
  s.units = base * s.ksplit;
  s.scale = a.scale;
  s.status = status;
  CUtensorMap tm_qhi, tm_qlo, tm_k, tm_out;
  if (!make_rows_map(&tm_qhi, s.qhi, uint64_t(a.rows), D, 128) ||
      !make_rows_map(&tm_qlo, s.qlo, uint64_t(a.rows), D, 128) ||
      !make_rows_map(&tm_k, a.k, uint64_t(a.BH) * a.Nk, D, 128) ||
      !make_scores_map(&tm_out, s.scores, static_cast<uint32_t>(a.Nk), uint64_t(a.G), uint64_t(a.BH),
                       uint64_t(s.ld)))
    return cudaErrorInvalidValue;
  auto kern = sa_score_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t grid = s.units < num_sms ? s.units : num_sms;
  kern<<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, st>>>(s, tm_qhi, tm_qlo, tm_k, tm_out);
  return cudaGetLastError();
}

cudaError_t launch_colstat(const BuildArgs& b, float* scores, int32_t* status, int num_sms,
                           cudaStream_t st);

cudaError_t launch_build_index(const BuildArgs& a, int num_sms, cudaStream_t st) {
  int64_t* misc = reinterpret_cast<int64_t*>(a.ws + a.L.misc);
  int32_t* status = reinterpret_cast<int32_t*>(misc + 1);
  cudaError_t e = cudaMemsetAsync(misc, 0, 16, st);
  if (e != cudaSuccess) return e;
  if (a.stat >= 0) {
    // dense-step statistics of the full attention probabilities
    e = launch_colstat(a, reinterpret_cast<float*>(a.ws + a.L.scores), status, num_sms, st);
    if (e != cudaSuccess) return e;
  } else {
    uint16_t* qhi = reinterpret_cast<uint16_t*>(a.ws + a.L.qhi);
    uint16_t* qlo = reinterpret_cast<uint16_t*>(a.ws + a.L.qlo);
    if (a.d == 128)
      sa_meanq_kernel<128><<<static_cast<unsigned>(a.rows), 256, 0, st>>>(a.q, qhi, qlo, a.G, a.Nq, a.M);
    else
      sa_meanq_kernel<64><<<static_cast<unsigned>(a.rows), 256, 0, st>>>(a.q, qhi, qlo, a.G, a.Nq, a.M);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = a.d == 128 ? launch_scores<128>(a, num_sms, st, status) : launch_scores<64>(a, num_sms, st, status);
    if (e != cudaSuccess) return e;
  }
  SelArgs s;
  s.scores = reinterpret_cast<const float*>(a.ws + a.L.scores);
  s.ld = a.L.ld;
  s.Nk = a.Nk;
  s.mode = a.mode;
  s.topk = a.topk;
  s.log_tau = a.threshold > 0.0 ? static_cast<float>(log(a.threshold)) : -INFINITY;
  s.mass = a.mass;
  s.level = a.stat >= 0 ? 1 : 0;
  s.cut = reinterpret_cast<uint32_t*>(a.ws + a.L.cut);
  s.ties = reinterpret_cast<int32_t*>(a.ws + a.L.ties);
  s.counts = reinterpret_cast<int64_t*>(a.ws + a.L.counts);
  s.col_idx = a.mode == SA_SELECT_TOPK ? a.col_idx : nullptr;
  s.col_capacity = a.col_capacity;
  // TOPK lists come from a kept-key bitmask in shared memory (rows up to
  // ~200K keys); longer rows are read a second time instead.
  const int words = (a.Nk + 31) / 32;
  s.mask_words = (a.mode == SA_SELECT_TOPK && sizeof(SelSmem) + size_t(words) * 4 <= kSelSmemBudget) ? words : 0;
  const size_t sel_smem = sizeof(SelSmem) + size_t(s.mask_words) * 4;
  e = cudaFuncSetAttribute(sa_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sel_smem));
  if (e != cudaSuccess) return e;
  sa_select_kernel<<<static_cast<unsigned>(a.rows), kSelThreads, sel_smem, st>>>(s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  sa_scan_kernel<<<1, 1024, 0, st>>>(s.counts, a.rows, a.row_ptr, misc, a.col_capacity, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.mode != SA_SELECT_TOPK)
    sa_emit_kernel<<<static_cast<unsigned>(a.rows), kSelThreads, 0, st>>>(
        s.scores, s.ld, a.Nk, s.cut, s.ties, a.row_ptr, a.col_idx, a.col_capacity);
  return cudaGetLastError();
}

cudaError_t launch_validate(const int64_t* row_ptr, const int32_t* col_idx, int64_t rows,
                            int64_t nnz, int32_t Nk, int32_t* status, cudaStream_t st) {
  const int64_t blocks = (rows + 7) / 8;
  sa_validate_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(row_ptr, col_idx, rows, nnz, Nk,
                                                                  status);
  return cudaGetLastError();
}

}  // namespace sa
