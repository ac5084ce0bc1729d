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
//                        plus how many keys equal to the cut are kept.  A
//                        strided sample of the row brackets the cut, one pass
//                        collects the keys inside the bracket (and marks those
//                        above it), and an exact ranking among them settles it;
//                        a bracket the sample misses falls back to a ranking
//                        of the whole row.  TOPK lists are written here.
//   4. sa_scan_kernel    row_ptr = exclusive prefix sum of the counts.
//   5. sa_emit_kernel    ascending indices of kept keys into col_idx.
//   6. TOPK over >= 8192 keys without the score matrix: sample scores of every
//      8th key (sa_score_kernel), a per-row bracket of the cut
//      (sa_bracket_kernel), a classifying score pass that marks keys above the
//      bracket and stores the ones inside it (sa_rowscore_kernel), and the
//      exact cut and emission (sa_topk_finalize_kernel).
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
  // score only the (head, 128-row chunk) units flagged non-zero here
  const int32_t* unit_filter = nullptr;
};

__device__ __forceinline__ bool skip_unit(const ScoreArgs& a, int64_t bh, int gc) {
  return a.unit_filter && a.unit_filter[bh * a.gchunks + gc] == 0;
}

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
      if (skip_unit(a, bh, gc)) continue;
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
        if (t1 <= t0 || skip_unit(a, bh, gc)) continue;
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
      if (t1 <= t0 || skip_unit(a, bh, gc)) continue;
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
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_3d(kb + s * C::kTile + cb * 128 * 128, &tm_k, 64 * cb, tile * 128, static_cast<int>(bh),
                      &bars->kfull[s]);
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
  const int32_t* row_list = nullptr;   // select only these rows (count in *row_count)
  const int32_t* row_count = nullptr;
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

template <class Sm>
__device__ __forceinline__ float block_min(float v, Sm& sm) {
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
template <class Sm>
__device__ __forceinline__ float block_max(float v, Sm& sm) { return -block_min(-v, sm); }
// Both at once, with one pair of barriers.
template <class Sm>
__device__ __forceinline__ void block_minmax(float* mn, float* mx, Sm& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float a = *mn, b = *mx;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fminf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  __syncthreads();
  if (lane == 0) {
    sm.fred[0][warp] = a;
    sm.fred[1][warp] = b;
  }
  __syncthreads();
  a = sm.fred[0][0];
  b = sm.fred[1][0];
#pragma unroll
  for (int w = 1; w < kSelWarps; ++w) {
    a = fminf(a, sm.fred[0][w]);
    b = fmaxf(b, sm.fred[1][w]);
  }
  *mn = a;
  *mx = b;
}

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
// col_idx[base, ...) and returns true, or, when `expect` >= 0 and the number
// of set bits differs from it, writes nothing and returns false (the same in
// every thread).  `write` false only counts.  Warp w owns a contiguous run of
// words; the runs' offsets come from one block scan of their popcounts.  A
// warp takes its run 32 words at a time (lane = word): a warp scan of the
// popcounts places each word's keys in the warp's staging buffer (1024 entries
// of shared memory), and the pass leaves in coalesced stores.  A lane expands
// its word bit by bit, in 32 fixed predicated steps when some word of the 32
// has more than 8 keys (a loop over set bits would run as long as the warp's
// fullest word), else in a loop over its set bits.
__device__ bool emit_mask(const uint32_t* kept, int words, int64_t base, int32_t* col_idx,
                          int64_t* scratch, int32_t* stage_all, int64_t expect = -1,
                          bool write = true) {
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
  if (expect >= 0 && total != expect) return false;
  if (!write) return true;
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
    const int jb = w * 32;
    if (__reduce_max_sync(0xffffffffu, static_cast<unsigned>(c)) > 8u) {
#pragma unroll
      for (int b = 0; b < 32; ++b)
        if (bits & (1u << b)) stage[off++] = jb + b;
    } else {
      while (bits) {
        stage[off++] = jb + (__ffs(bits) - 1);
        bits &= bits - 1;
      }
    }
    __syncwarp();
    for (int i = lane; i < cnt; i += 32) col_idx[pos + i] = stage[i];
    __syncwarp();
    pos += cnt;
  }
  return true;
}

// The selection of one score row by the whole block.  TOPK: bit j of
// kept[j / 32] marks key j as kept (keys above the bracket during the window
// pass, kept keys of the window after the selection).
__device__ void select_row(const SelArgs& a, const int64_t row, SelSmem& sm, uint32_t* kept) {
  const bool use_mask = !by_mass_mode(a) && a.col_idx && a.mask_words > 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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

// One row per block, or (row_list set) the listed rows only: the rows that
// the TOPK path without a score matrix could not bracket, whose scores the
// score kernel has written for this kernel.
template <bool LIST>
__global__ void __launch_bounds__(kSelThreads, 4) sa_select_kernel(const SelArgs a) {
  extern __shared__ uint8_t sel_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(sel_raw);
  uint32_t* kept = reinterpret_cast<uint32_t*>(sel_raw + sizeof(SelSmem));
  if (!LIST) {
    select_row(a, blockIdx.x, sm, kept);
    return;
  }
  const int n = *a.row_count;
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    select_row(a, a.row_list[i], sm, kept);
    __syncthreads();
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

// ------------------------------------------------------------ 6. TOPK without a score matrix
// TOPK lists need each row's k-th largest score and the keys above it, not the
// scores themselves, so the fp32 score matrix (rows x Nk, written once and read
// several times by the select kernel) is replaced by three passes:
//   sa_score_kernel<D>            scores of every stride-th key (a strided TMA
//                                 map over K) into a small sample matrix;
//   sa_bracket_kernel             per row, two score values lo <= hi around the
//                                 cut: the sample's order statistics at the
//                                 expected rank of the cut -/+ four binomial
//                                 standard deviations;
//   sa_rowscore_kernel<D>         every score, classified as it leaves TMEM:
//                                 above hi -> a bit of the row's keep-mask, in
//                                 [lo, hi] -> an (index, score) candidate;
//   sa_topk_finalize_kernel       the exact cut among the candidates (the
//                                 select kernel's histogram descent), their
//                                 bits, and ascending emission from the mask.
// The score MMA here puts the mean queries on TMEM lanes (A = 128 groups x d,
// B = 128 keys x d), so a thread owns one row and builds its mask words and
// candidate list without any exchange.  A row whose bracket misses the cut or
// overflows its candidate storage is listed; the score kernel then writes the
// fp32 scores of the listed rows' units and the select kernel selects those
// rows, so the lists are exact in every case.
// Key split ks of a unit takes the key tiles ks, ks + ksplit, ... (spread
// over the whole sequence, so that every split sees about the same share of
// a row's candidates however they cluster); each (row, split, 32-column part
// of the tile) has its own candidate region of `cap` slots.
struct RowScoreArgs {
  int64_t G, units;
  int32_t Nk, gchunks, ksplit, ntiles;
  float scale;
  const float2* lohi;   // (lo, hi) per row
  uint32_t* mask;       // [rows, ld_mask] words, bit j mod 32 of word j / 32: key j above hi
  int64_t ld_mask;
  uint2* cand;          // [rows, 4 * ksplit regions, cap]: (key, score bits)
  int32_t cap;
  int32_t* nabove;      // [rows, 4 * ksplit]: keys above hi
  int32_t* ncand;       // [rows, 4 * ksplit]: keys in [lo, hi] (may exceed cap)
  int32_t* status;
};

template <int D>
struct RowScoreCfg {
  static constexpr int kStages = 3;
  // four per TMEM lane quarter, one 32-key column part of the tile each
  static constexpr int kParts = 4;
  static constexpr int kEpiWarps = 4 * kParts;
  static constexpr int kMmaWarp = kEpiWarps, kTmaWarp = kEpiWarps + 1;
  static constexpr int kThreads = 32 * (kEpiWarps + 2);
  static constexpr int kTile = 128 * D * 2;  // 128 rows of d bf16
  // each epilogue warp stages its 32 rows x 32 raw scores, [c / 4][lane] float4s
  static constexpr int kStage = 32 * 32 * 4;
  static constexpr int kSmemBytes = 1024 + 2 * kTile + kStages * kTile + kEpiWarps * kStage + 1024;
  static constexpr int kTmemCols = 256;      // two 128-column accumulators
};

__device__ __forceinline__ void rs_unit(const RowScoreArgs& a, int64_t u, int64_t* bh, int* gc,
                                        int* ks) {
  const int64_t per_bh = int64_t(a.gchunks) * a.ksplit;
  *bh = u / per_bh;
  const int rem = static_cast<int>(u % per_bh);
  *gc = rem / a.ksplit;
  *ks = rem % a.ksplit;
}

// For s > 0: the largest x with fl(x * s) <= hi (+inf for hi = +inf), and
// the smallest x with fl(x * s) >= lo (-inf for lo = -inf); rounding is
// monotone in x, so a few ulp steps from the quotient find them.  A zero
// result is returned as +0 (floor) or -0 (ceil), so that the sign of
// floor - x and of x - ceil is that of the comparison.
__device__ __forceinline__ float score_floor(float hi, float s) {
  if (!(hi < INFINITY)) return INFINITY;
  float x = hi / s;
  for (int i = 0; i < 8 && x * s > hi; ++i) x = nextafterf(x, -INFINITY);
  for (int i = 0; i < 8 && nextafterf(x, INFINITY) * s <= hi; ++i) x = nextafterf(x, INFINITY);
  return x == 0.f ? 0.f : x;
}
__device__ __forceinline__ float score_ceil(float lo, float s) {
  if (!(lo > -INFINITY)) return -INFINITY;
  float x = lo / s;
  for (int i = 0; i < 8 && x * s < lo; ++i) x = nextafterf(x, INFINITY);
  for (int i = 0; i < 8 && nextafterf(x, -INFINITY) * s >= lo; ++i) x = nextafterf(x, -INFINITY);
  return x == 0.f ? -0.f : x;
}

template <int D>
__global__ void __launch_bounds__(RowScoreCfg<D>::kThreads, 1)
    sa_rowscore_kernel(const RowScoreArgs a, const __grid_constant__ CUtensorMap tm_qhi,
                       const __grid_constant__ CUtensorMap tm_qlo,
                       const __grid_constant__ CUtensorMap tm_k) {
  using C = RowScoreCfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQh = smem;
  uint8_t* sQl = sQh + C::kTile;
  uint8_t* sK = sQl + C::kTile;
  uint8_t* sStage = sK + S * C::kTile;
  ScoreBars* bars = reinterpret_cast<ScoreBars*>(sStage + C::kEpiWarps * C::kStage);
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
      mbar_init(&bars->dempty[b], C::kEpiWarps);  // one arrival per epilogue warp
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < C::kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    // Thread = one mean-query row (TMEM lane), 32 key columns of each tile.
    // Four warps share a lane quarter, so that a sub-partition has four
    // epilogue warps to hide the latency of each one's chain of steps.
    const int quarter = warp & 3, part = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int gi = quarter * 32 + lane;
    uint32_t t = 0;
    for (int64_t u = blockIdx.x; u < a.units; u += gridDim.x) {
      int64_t bh;
      int gc, ks;
      rs_unit(a, u, &bh, &gc, &ks);
      const int64_t g = int64_t(gc) * 128 + gi;
      const bool valid = g < a.G;
      const int64_t row = bh * a.G + g;
      const int64_t region = (row * a.ksplit + ks) * C::kParts + part;
      // scale > 0: scale*x > hi <=> x > xa and scale*x < lo <=> x < xb, with
      // xa the largest x whose rounded score is <= hi, xb the smallest whose
      // rounded score is >= lo (found from the quotients by stepping ulps)
      float xa = 0.f, xb = 0.f;
      if (valid) {
        const float2 b = a.lohi[row];
        xa = score_floor(b.y, a.scale);
        xb = score_ceil(b.x, a.scale);
      }
      uint2* cbase = a.cand + region * a.cap;
      const int cap = a.cap;
      const int64_t lane_step = int64_t(C::kParts) * a.ksplit * cap;  // one row further
      int nab = 0, nc = 0;
      for (int tile = ks; tile < a.ntiles; tile += a.ksplit, ++t) {
        const uint32_t b = t & 1;
        // (the whole warp leaves together: the steps below are warp-collective)
        const bool got = mbar_wait(&bars->dfull[b], (t >> 1) & 1, abort);
        if (!__all_sync(0xffffffffu, got)) goto done;
        tc_fence_after();
        float x[32];
        tmem_ld32(tmem + lane_base + b * 128 + part * 32, reinterpret_cast<uint32_t*>(x));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->dempty[b]);
        // (rows past G take part in the warp's collective steps with no keys)
        const int j0 = tile * 128 + part * 32;
        // key c is above when xa - x < 0 and below when x - xb < 0 (for floats
        // p != q, p - q is never zero; xa is never -0 and xb never +0): the
        // sign bits are funnel-shifted into a word, highest key first, in
        // four chains of 16 keys
        uint32_t a0 = 0u, a1 = 0u, b0 = 0u, b1 = 0u;
#pragma unroll
        for (int c = 15; c >= 0; --c) {
          a0 = shl_in(a0, __float_as_uint(xa - x[c]));
          a1 = shl_in(a1, __float_as_uint(xa - x[16 + c]));
          b0 = shl_in(b0, __float_as_uint(x[c] - xb));
          b1 = shl_in(b1, __float_as_uint(x[16 + c] - xb));
        }
        uint32_t w = (a1 << 16) | a0;
        uint32_t cw = ~(w | (b1 << 16) | b0);  // neither above nor below
        if (j0 + 32 > a.Nk || !valid) {
          const int r = valid ? a.Nk - j0 : 0;  // keys of this part that exist
          const uint32_t keep = r >= 32 ? 0xFFFFFFFFu : (r <= 0 ? 0u : (1u << r) - 1u);
          w &= keep;
          cw &= keep;
        }
        if (valid) {
          nab += __popc(w);
          a.mask[row * a.ld_mask + (j0 >> 5)] = w;
        }
        // The candidates' scores leave through the warp's staging area, the
        // whole warp at once: the warp's candidates of this part, row (lane)
        // by row and key by key, are numbered by a warp scan of the rows'
        // counts, and lane l takes numbers l, l + 32, ...: it finds the row
        // holding its number (a binary search over the scan) and the key (the
        // r-th set bit of that row's word).  A row's candidates fall on
        // consecutive lanes and land in consecutive slots.
        const int cnt = __popc(cw);
        const int incl = warp_incl_scan(cnt);
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (total > 0) {
          float4* st4 = reinterpret_cast<float4*>(sStage + warp * C::kStage);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4)
            st4[c4 * 32 + lane] = make_float4(x[4 * c4], x[4 * c4 + 1], x[4 * c4 + 2], x[4 * c4 + 3]);
          __syncwarp();
          const float* st = reinterpret_cast<const float*>(st4);
          const int excl = incl - cnt;
          for (int i0 = 0; i0 < total; i0 += 32) {  // (total is the same in every lane)
            const int i = i0 + lane;
            int o = 0;  // the owner: the number of rows whose inclusive count is <= i
#pragma unroll
            for (int step = 16; step > 0; step >>= 1)
              if (__shfl_sync(0xffffffffu, incl, o + step - 1) <= i) o += step;
            int r = i - __shfl_sync(0xffffffffu, excl, o);
            uint32_t m = __shfl_sync(0xffffffffu, cw, o);
            const int slot = __shfl_sync(0xffffffffu, nc, o) + r;
            if (i < total) {
              int c = 0;  // the r-th set bit (0-based) of m
#pragma unroll
              for (int wdt = 16; wdt > 0; wdt >>= 1) {
                const int p = __popc(m & ((1u << wdt) - 1u));
                if (r >= p) {
                  r -= p;
                  c += wdt;
                  m >>= wdt;
                }
              }
              if (slot < cap)
                cbase[int64_t(o - lane) * lane_step + slot] =
                    make_uint2(static_cast<uint32_t>(j0 + c),
                               __float_as_uint(st[((c >> 2) * 32 + o) * 4 + (c & 3)] * a.scale));
            }
          }
          nc += cnt;
          __syncwarp();
        }
      }
      if (valid) {
        a.nabove[region] = nab;
        a.ncand[region] = nc;
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16(128, 128, false, false);
      const uint32_t qh = smem_u32(sQh), ql = smem_u32(sQl), kb = smem_u32(sK);
      uint32_t t = 0, un = 0;
      bool ok = true;
      for (int64_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        int64_t bh;
        int gc, ks;
        rs_unit(a, u, &bh, &gc, &ks);
        if (ks >= a.ntiles) continue;
        if (!mbar_wait(&bars->qfull, un & 1, abort)) break;
        for (int tile = ks; tile < a.ntiles; tile += a.ksplit, ++t) {
          const uint32_t s = t % S, b = t & 1;
          if (!mbar_wait(&bars->kfull[s], (t / S) & 1, abort) ||
              !mbar_wait(&bars->dempty[b], ((t >> 1) & 1) ^ 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem + b * 128;
          // D[group][key] = q_hi . k, then += q_lo . k
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 128 * 128 + (kk & 3) * 32;
            mma_ss(d_tmem, sw128_desc(qh + off, 16, 1024), sw128_desc(kb + s * C::kTile + off, 16, 1024),
                   kIdesc, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 128 * 128 + (kk & 3) * 32;
            mma_ss(d_tmem, sw128_desc(ql + off, 16, 1024), sw128_desc(kb + s * C::kTile + off, 16, 1024),
                   kIdesc, 1u);
          }
          mma_commit(&bars->dfull[b]);
          mma_commit(&bars->kempty[s]);
          if (tile + a.ksplit >= a.ntiles) mma_commit(&bars->qempty);
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
      int gc, ks;
      rs_unit(a, u, &bh, &gc, &ks);
      if (ks >= a.ntiles) continue;
      if (un > 0 && !mbar_wait(&bars->qempty, (un - 1) & 1, abort)) goto done;
      // mean-query rows bh*G + gc*128 .. +127 (rows past the head only feed
      // rows that are never written)
      const int qrow = static_cast<int>(bh * a.G + int64_t(gc) * 128);
      mbar_expect_tx(&bars->qfull, 2 * C::kTile);
#pragma unroll
      for (int cb = 0; cb < D / 64; ++cb) {
        tma_load_2d(qh + cb * 128 * 128, &tm_qhi, 64 * cb, qrow, &bars->qfull);
        tma_load_2d(ql + cb * 128 * 128, &tm_qlo, 64 * cb, qrow, &bars->qfull);
      }
      for (int tile = ks; tile < a.ntiles; tile += a.ksplit, ++t) {
        const uint32_t s = t % S;
        if (!mbar_wait(&bars->kempty[s], ((t / S) & 1) ^ 1, abort)) goto done;
        mbar_expect_tx(&bars->kfull[s], C::kTile);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_3d(kb + s * C::kTile + cb * 128 * 128, &tm_k, 64 * cb, tile * 128, static_cast<int>(bh),
                      &bars->kfull[s]);
      }
      ++un;
    }
  }
done:
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && bars->abort) report(a.status, SA_DEVERR_TIMEOUT);
  if (warp == C::kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Per row (one warp each): lo <= hi around the cut from the row's samples.
// The samples are spread over kBrBins linear bins between the minimum and
// maximum of the first 1024 of them, widened by an eighth (samples outside go
// to the end bins, whose outer edges count as -inf and inf); hi is the upper
// edge of the bin
// holding sample rank r_hi (counted from the top, 0-based) and lo the lower
// edge of the bin holding rank r_lo, so at most r_hi samples lie above hi and
// more than r_lo at or above lo.  A non-finite estimate gives (-inf, inf):
// every key a candidate.
// Bin b lives at word b + b / 32 of the warp's histogram: a lane scans 32
// consecutive bins, and the pad word puts the 32 lanes' reads of one step in 32
// different banks.
constexpr int kBrBins = 1024;
constexpr int kBrWarps = 4;
__device__ __forceinline__ int br_slot(int b) { return b + (b >> 5); }
__global__ void __launch_bounds__(32 * kBrWarps) sa_bracket_kernel(const float* samp, int64_t ld_samp,
                                                                    int32_t S, int64_t rows, float r_hi,
                                                                    float r_lo, float2* lohi) {
  __shared__ uint32_t hist_all[kBrWarps][kBrBins + kBrBins / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = int64_t(blockIdx.x) * kBrWarps + warp;
  if (row >= rows) return;  // warps are independent: no block barrier below
  uint32_t* hist = hist_all[warp];
  const float* x = samp + row * ld_samp;
  const float nan = __int_as_float(0x7fffffff);
  float mn = INFINITY, mx = -INFINITY;
  {
    const int ne = S < 1024 ? S : 1024;
    float v[32];
#pragma unroll
    for (int m = 0; m < 32; ++m) v[m] = lane + 32 * m < ne ? x[lane + 32 * m] : nan;
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      mn = fminf(mn, v[m]);
      mx = fmaxf(mx, v[m]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  float lo = -INFINITY, hi = INFINITY;
  float span = mx - mn;
  if (isfinite(mn) && isfinite(mx) && isfinite(span)) {
    // the estimate's range widened by an eighth (half on each side), or
    // narrow bins centred on a flat estimate
    if (span > 0.f) {
      mn -= span * 0.0625f;
      span *= 1.125f;
    } else {
      span = fabsf(mn) * 0x1p-10f + 0x1p-100f;
      mn -= 0.5f * span;
    }
    const float inv = float(kBrBins) / span;
    for (int i = lane; i < kBrBins + kBrBins / 32; i += 32) hist[i] = 0;
    __syncwarp();
    const int nf4 = S >> 2;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    for (int f0 = 0; f0 < nf4; f0 += 32 * 8) {
      float4 q4[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int f = f0 + 32 * u + lane;
        q4[u] = f < nf4 ? x4[f] : make_float4(nan, nan, nan, nan);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float e[4] = {q4[u].x, q4[u].y, q4[u].z, q4[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (e[c] == e[c]) atomicAdd(&hist[br_slot(lin_bin(e[c], mn, inv, kBrBins))], 1u);
      }
    }
    for (int i = 4 * nf4 + lane; i < S; i += 32) {
      const float v = x[i];
      if (v == v) atomicAdd(&hist[br_slot(lin_bin(v, mn, inv, kBrBins))], 1u);
    }
    __syncwarp();
    constexpr int per = kBrBins / 32;
    const int top = kBrBins - 1 - per * lane;  // lane 0 holds the highest bins
    uint32_t tot = 0;
#pragma unroll 8
    for (int e = 0; e < per; ++e) tot += hist[br_slot(top - e)];
    uint32_t c = warp_incl_scan(tot) - tot;  // samples in higher bins
    float hv = INFINITY, lv = -INFINITY;
    bool got_hi = false, got_lo = false;
    for (int e = 0; e < per; ++e) {
      const int bin = top - e;
      const uint32_t n = hist[br_slot(bin)];
      if (n > 0) {
        if (r_hi >= float(c) && r_hi < float(c + n)) {
          got_hi = true;
          hv = bin == kBrBins - 1 ? INFINITY : mn + float(bin + 1) / inv;
        }
        if (r_lo >= float(c) && r_lo < float(c + n)) {
          got_lo = true;
          lv = bin == 0 ? -INFINITY : mn + float(bin) / inv;
        }
      }
      c += n;
    }
    const unsigned bh_ = __ballot_sync(0xffffffffu, got_hi), bl_ = __ballot_sync(0xffffffffu, got_lo);
    if (bh_) hi = __shfl_sync(0xffffffffu, hv, __ffs(bh_) - 1);
    if (bl_) lo = __shfl_sync(0xffffffffu, lv, __ffs(bl_) - 1);
    if (hi < lo) hi = lo;
  }
  if (lane == 0) lohi[row] = make_float2(lo, hi);
}

struct FinArgs {
  int64_t rows, G, k;
  int32_t Nk, nreg, cap, gchunks, all_keys;
  const uint32_t* mask;
  int64_t ld_mask;
  const uint2* cand;
  const int32_t* nabove;
  const int32_t* ncand;
  int32_t* col_idx;
  int64_t col_capacity;
  int64_t* counts;
  int64_t* row_ptr;     // TOPK: every row holds k keys, so row_ptr[r] = r * k
  int64_t* nnz;
  int32_t* fail_rows;   // rows left to the score + select kernels
  int32_t* fail_count;
  int32_t* fail_units;  // [BH * gchunks] non-zero: that unit's scores are needed
};
constexpr int kFinCand = kWindow / 2;  // candidates a row may hold
// The finalize's shared memory (then the row's keep-mask, 16-byte aligned):
// small enough for four blocks per SM
struct FinSmem {
  uint32_t hist[kBins];
  float rx[kRank];
  int32_t rj[kRank];
  int32_t cand[2 * kFinCand];  // keys, then scores; afterwards the mask words' offsets
  float fred[3][32];
  int64_t scan_c[32];
  int64_t found_above_cnt, cut_greater;
  int32_t claim, n_rank, cut_rank, n_win, found_cnt;
  float cut_x;
};
constexpr size_t kFinMaskOff = (sizeof(FinSmem) + 15) & ~size_t(15);

__global__ void __launch_bounds__(kSelThreads, 4) sa_topk_finalize_kernel(const FinArgs a) {
  extern __shared__ __align__(16) uint8_t fin_raw[];
  FinSmem& sm = *reinterpret_cast<FinSmem*>(fin_raw);
  uint32_t* kept = reinterpret_cast<uint32_t*>(fin_raw + kFinMaskOff);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int64_t k = a.k, base = row * k;
  if (tid == 0) {
    a.row_ptr[row] = base;
    if (row == 0) {
      a.row_ptr[a.rows] = a.rows * k;
      *a.nnz = a.rows * k;
    }
  }
  if (a.all_keys) {  // k == Nk: every key, in order
    if (base + k <= a.col_capacity)
      for (int j = tid; j < a.Nk; j += kSelThreads) a.col_idx[base + j] = j;
    if (tid == 0) a.counts[row] = k;
    return;
  }
  const int32_t* nab = a.nabove + row * a.nreg;
  const int32_t* ncd = a.ncand + row * a.nreg;
  __shared__ int32_t reg_off[65];
  if (tid < 32) {
    int64_t above = 0;
    int ntot = 0, over = 0;
    for (int r = lane; r < a.nreg; r += 32) {  // (nreg <= 64)
      above += nab[r];
      const int c = ncd[r];
      over |= c > a.cap || c < 0;  // (a negative count: a damaged workspace)
      ntot += c;
    }
    // region offsets in the packed candidate list
    const int ca = lane < a.nreg ? max(0, min(ncd[lane], a.cap)) : 0;
    const int cb = lane + 32 < a.nreg ? max(0, min(ncd[lane + 32], a.cap)) : 0;
    const int ia = warp_incl_scan(ca);
    const int ib = warp_incl_scan(cb) + __shfl_sync(0xffffffffu, ia, 31);
    reg_off[lane + 1] = ia;
    reg_off[lane + 33] = ib;
    if (lane == 0) reg_off[0] = 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      above += __shfl_xor_sync(0xffffffffu, above, o);
      ntot += __shfl_xor_sync(0xffffffffu, ntot, o);
      over |= __shfl_xor_sync(0xffffffffu, over, o);
    }
    if (tid == 0) {
      sm.found_above_cnt = above;
      sm.n_win = ntot;
      sm.found_cnt = over;
    }
  }
  // the row goes to the score + select kernels
  auto leave = [&]() {
    if (tid == 0) {
      const int32_t i = atomicAdd(a.fail_count, 1);
      a.fail_rows[i] = static_cast<int32_t>(row);
      const int64_t bh = row / a.G, g = row % a.G;
      a.fail_units[bh * a.gchunks + g / 128] = 1;
    }
  };
  __syncthreads();
  const int64_t above = sm.found_above_cnt;
  const int ntot = sm.n_win;
  if (!(sm.found_cnt == 0 && above <= k && k <= above + ntot && ntot <= kFinCand)) {
    leave();
    return;
  }
  const int words = static_cast<int>((a.Nk + 31) / 32);
  {  // the keys above the bracket
    const uint4* mrow = reinterpret_cast<const uint4*>(a.mask + row * a.ld_mask);
    for (int w = tid; w < static_cast<int>(a.ld_mask / 4); w += kSelThreads)
      reinterpret_cast<uint4*>(kept)[w] = mrow[w];
  }
  int32_t* cj = sm.cand;
  float* cx = reinterpret_cast<float*>(sm.cand + kFinCand);
  const int64_t need = k - above;  // candidates to keep
  if (need > 0) {
    // candidate i of the packed list: region r with reg_off[r] <= i < reg_off[r+1];
    // up to eight loads in flight per thread
    const uint2* src = a.cand + row * int64_t(a.nreg) * a.cap;
    float wmn = INFINITY, wmx = -INFINITY;
    for (int i0 = 0; i0 < ntot; i0 += 8 * kSelThreads) {
      uint2 e[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kSelThreads + tid;
        if (i < ntot) {
          int r = 0;  // the last region with reg_off[r] <= i
#pragma unroll
          for (int step = 32; step > 0; step >>= 1)
            if (r + step < a.nreg && reg_off[r + step] <= i) r += step;
          e[u] = src[int64_t(r) * a.cap + (i - reg_off[r])];
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kSelThreads + tid;
        if (i < ntot) {
          const float xv = __uint_as_float(e[u].y);
          cj[i] = static_cast<int32_t>(e[u].x);
          cx[i] = xv;
          wmn = fminf(wmn, xv);
          wmx = fmaxf(wmx, xv);
        }
      }
    }
    block_minmax(&wmn, &wmx, sm);  // (its barriers also publish cx, cj)
    // The need-th candidate by (score descending, key ascending): one
    // histogram over kBins linear bins of [wmn, wmx], the bin where the
    // count from the top reaches need, then an exact ranking of that bin's
    // candidates.  Equal scores share a bin; a bin too full to rank leaves
    // the row to the select kernel.
    uint32_t cut;
    int64_t ties;
    const bool flat = !(wmx > wmn);
    const float inv = flat ? 0.f : float(kBins) / (wmx - wmn);
    for (int i = tid; i < kBins; i += kSelThreads) sm.hist[i] = 0;
    if (tid == 0) {
      sm.claim = -1;
      sm.n_rank = 0;
      sm.cut_rank = -1;
    }
    __syncthreads();
    if (!flat)
      for (int i = tid; i < ntot; i += kSelThreads) atomicAdd(&sm.hist[lin_bin(cx[i], wmn, inv, kBins)], 1u);
    else if (tid == 0)
      sm.hist[0] = static_cast<uint32_t>(ntot);
    __syncthreads();
    const int top = kBins - 1 - kBinsPerThread * tid;  // thread 0 holds the highest bins
    int64_t c4 = 0;
#pragma unroll
    for (int e = 0; e < kBinsPerThread; ++e) c4 += sm.hist[top - e];
    int64_t ctot;
    int64_t cum = block_excl_scan<int64_t>(c4, &ctot, sm.scan_c);
    for (int e = 0; e < kBinsPerThread; ++e) {
      const int bin = top - e;
      const int64_t bc = sm.hist[bin];
      if (bc > 0 && cum < need && cum + bc >= need) {
        sm.claim = bin;
        sm.found_above_cnt = cum;  // candidates in higher bins
      }
      cum += bc;
    }
    __syncthreads();
    const int bin = sm.claim;
    const int64_t higher = sm.found_above_cnt;
    const int nb = bin >= 0 ? static_cast<int>(sm.hist[bin]) : 0;
    if (bin < 0 || nb > kRank) {
      leave();
      return;
    }
    // the bin's candidates
    for (int base_i = warp * 32; base_i < ntot; base_i += kSelThreads) {
      const int i = base_i + lane;
      const bool in = i < ntot && (flat || lin_bin(cx[i], wmn, inv, kBins) == bin);
      const unsigned bal = __ballot_sync(0xffffffffu, in);
      int s0 = 0;
      if (lane == 0 && bal) s0 = atomicAdd(&sm.n_rank, __popc(bal));
      const int slot = __shfl_sync(0xffffffffu, s0, 0) + __popc(bal & ((1u << lane) - 1u));
      if (in && slot < kRank) {
        sm.rx[slot] = cx[i];
        sm.rj[slot] = cj[i];
      }
    }
    __syncthreads();
    for (int c = tid; c < nb; c += kSelThreads) {
      const float xc = sm.rx[c];
      const int jc = sm.rj[c];
      int rank = 0, greater = 0;
      for (int o = 0; o < nb; ++o) {
        const float xo = sm.rx[o];
        rank += xo > xc || (xo == xc && sm.rj[o] < jc);
        greater += xo > xc;
      }
      if (higher + rank == need - 1) {
        sm.cut_rank = rank;
        sm.cut_x = xc;
        sm.cut_greater = greater;
      }
    }
    __syncthreads();
    if (sm.cut_rank < 0) {  // (never)
      leave();
      return;
    }
    cut = order_key(sm.cut_x);
    ties = need - (higher + sm.cut_greater);  // keys equal to the cut that are kept
    // keys equal to the cut: all in this bin; the lowest indices are kept
    int n_eq = 0;
    for (int c = 0; c < nb; ++c) n_eq += order_key(sm.rx[c]) == cut;
    const bool rank_ties = ties < n_eq;
    for (int i = tid; i < ntot; i += kSelThreads) {
      const uint32_t kx = order_key(cx[i]);
      const int j = cj[i];
      bool keep = kx > cut;
      if (kx == cut) {
        if (!rank_ties) {
          keep = true;
        } else {
          int before = 0;  // lower indices first among equal scores
          for (int c = 0; c < nb; ++c) before += order_key(sm.rx[c]) == cut && sm.rj[c] < j;
          keep = before < ties;
        }
      }
      // (a key outside [0, Nk), which only a damaged workspace could hold,
      // sets no bit: the count check below then leaves the row to the
      // select kernel)
      if (keep && static_cast<uint32_t>(j) < static_cast<uint32_t>(a.Nk)) atomicOr(&kept[j >> 5], 1u << (j & 31));
    }
  }
  __syncthreads();
  // ascending emission of exactly k kept keys (else the row is left to the
  // select kernel), staged per warp in the candidates' storage (free now)
  if (!emit_mask(kept, words, base, a.col_idx, sm.scan_c, sm.cand, k, base + k <= a.col_capacity)) {
    leave();
    return;
  }
  if (tid == 0) a.counts[row] = k;
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
  L.fail = off;
  off = align256(off + 256 + size_t(rows) * 8);
  L.total = off;
  return L;
}

// Scores of every stride-th key (nkeys of them per head; stride 1 and nkeys
// Nk: every key) into `out`, fp32 [rows, ld]; only the units flagged in
// unit_filter when it is given.
template <int D>
static cudaError_t launch_scores(const BuildArgs& a, int num_sms, cudaStream_t st, int32_t* status,
                                 const int32_t* unit_filter = nullptr, float* out = nullptr,
                                 int64_t ld = 0, int32_t nkeys = 0, int32_t stride = 1) {
  using C = ScoreCfg<D>;
  if (!out) {
    out = reinterpret_cast<float*>(a.ws + a.L.scores);
    ld = a.L.ld;
    nkeys = a.Nk;
    stride = 1;
  }
  ScoreArgs s;
  s.k = a.k;
  s.qhi = reinterpret_cast<const uint16_t*>(a.ws + a.L.qhi);
  s.qlo = reinterpret_cast<const uint16_t*>(a.ws + a.L.qlo);
  s.scores = out;
  s.ld = ld;
  s.G = a.G;
  s.Nk = nkeys;
  s.gchunks = static_cast<int32_t>((a.G + 127) / 128);
  s.ntiles = (nkeys + 127) / 128;
  const int64_t base = int64_t(a.BH) * s.gchunks;
  int64_t ks = (2 * int64_t(num_sms) + base - 1) / base;
  // with a unit filter (a few units flagged) the flagged units' keys are
  // split finely, so that they spread over the SMs; the rest are skipped
  if (unit_filter) ks = 64;
  ks = ks < 1 ? 1 : (ks > s.ntiles ? s.ntiles : ks);
  s.tiles_per_split = static_cast<int32_t>((s.ntiles + ks - 1) / ks);
  s.ksplit = (s.ntiles + s.tiles_per_split - 1) / s.tiles_per_split;
  s.units = base * s.ksplit;
  s.scale = a.scale;
  s.status = status;
  s.unit_filter = unit_filter;
  CUtensorMap tm_qhi, tm_qlo, tm_k, tm_out;
  if (!make_rows_map(&tm_qhi, s.qhi, uint64_t(a.rows), D, 128) ||
      !make_rows_map(&tm_qlo, s.qlo, uint64_t(a.rows), D, 128) ||
      !make_keys_map(&tm_k, a.k, D, uint64_t(nkeys), uint64_t(a.Nk), uint64_t(a.BH), uint64_t(stride)) ||
      !make_scores_map(&tm_out, s.scores, static_cast<uint32_t>(nkeys), uint64_t(a.G), uint64_t(a.BH),
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

// Buffers of the TOPK path without a score matrix, carved from the scores
// region of the workspace; ok = false when they do not fit (the score matrix
// path is used instead).
struct TopkPlan {
  bool ok = false;
  int32_t stride = 8, S = 0, gchunks = 0;
  int32_t ksplit = 0, ntiles = 0;  // classifying pass
  int32_t nreg = 0, cap = 0;       // candidate regions per row, slots per region
  int64_t ld_samp = 0, ld_mask = 0;
  float r_hi = 0.f, r_lo = 0.f;
  size_t samp = 0, lohi = 0, mask = 0, cand = 0, nabove = 0, ncand = 0;
};

static TopkPlan plan_topk(const BuildArgs& a, int num_sms) {
  TopkPlan P;
  const int64_t k = a.topk;
  // (a whole number of samples per head keeps the strided key map's head
  // stride a multiple of its row stride)
  if (a.Nk < 8192 || a.Nk % P.stride != 0 || k >= a.Nk || k < 1 || !(a.scale > 0.f)) return P;
  P.gchunks = static_cast<int32_t>((a.G + 127) / 128);
  const int64_t base = int64_t(a.BH) * P.gchunks;
  P.S = a.Nk / P.stride;
  P.ntiles = (a.Nk + 127) / 128;
  P.ld_samp = (int64_t(P.S) + 3) & ~int64_t(3);
  P.ld_mask = int64_t(P.ntiles) * 4;
  // The cut's sample rank (from the top) is binomial around p: bracket it by
  // four standard deviations and 16 ranks each way.
  const double q = double(k) / double(a.Nk), p = q * P.S;
  const double dev = 4.0 * sqrt(double(P.S) * q * (1.0 - q)) + 16.0;
  P.r_hi = static_cast<float>(p - dev);
  P.r_lo = static_cast<float>(p + dev);
  // expected keys in the bracket; the finalize takes up to kFinCand of them
  const double window = (2.0 * dev / P.S) * a.Nk;
  if (window > 0.85 * kFinCand) return P;  // the bracket would often overflow the finalize
  // the row's mask in shared memory, its word offsets in the window storage
  if (kFinMaskOff + size_t(P.ld_mask) * 4 > 160 * 1024 || P.ld_mask > 2 * kFinCand) return P;
  const size_t rows = size_t(a.rows), region = rows * size_t(a.L.ld) * 4;
  // Key splits: among the counts (at most 16, so at most 64 candidate regions
  // per row) whose regions fit the scores region, the one that minimises the
  // tiles of the busiest SM, counting two tiles of start-up per unit.  A
  // region takes what the scores region holds, up to kFinCand slots; its
  // expected share of the bracket (tiles spread over the sequence) must fit
  // twice over, plus 96.
  int64_t best = -1;
  for (int ks = 1; ks <= 16 && ks <= P.ntiles; ++ks) {
    const int nreg = 4 * ks;
    size_t off = 0;
    const size_t samp = off;
    off = align256(off + rows * size_t(P.ld_samp) * 4);
    const size_t lohi = off;
    off = align256(off + rows * 8);
    const size_t mask = off;
    off = align256(off + rows * size_t(P.ld_mask) * 4);
    const size_t nab = off;
    off = align256(off + rows * size_t(nreg) * 4);
    const size_t ncd = off;
    off = align256(off + rows * size_t(nreg) * 4);
    if (off >= region) break;  // (more regions only take more room)
    const int64_t room = static_cast<int64_t>((region - off) / (rows * size_t(nreg) * 8));
    const int64_t cap = (room < kFinCand ? room : kFinCand) & ~int64_t(1);  // (even: every region starts 16-byte aligned)
    if (cap < 2.0 * window / nreg + 96) continue;
    const int64_t units = base * ks, waves = (units + num_sms - 1) / num_sms;
    const int64_t cost = waves * ((P.ntiles + ks - 1) / ks + 2);
    if (best >= 0 && cost >= best) continue;
    best = cost;
    P.ksplit = ks;
    P.nreg = nreg;
    P.cap = static_cast<int32_t>(cap);
    P.samp = samp;
    P.lohi = lohi;
    P.mask = mask;
    P.nabove = nab;
    P.ncand = ncd;
    P.cand = off;
    P.ok = true;
  }
  return P;
}

template <int D>
static cudaError_t launch_rowscore(const BuildArgs& a, const TopkPlan& P, int num_sms, cudaStream_t st,
                                   int32_t* status) {
  using C = RowScoreCfg<D>;
  uint8_t* reg = a.ws + a.L.scores;
  RowScoreArgs r;
  r.G = a.G;
  r.Nk = a.Nk;
  r.gchunks = P.gchunks;
  r.ntiles = P.ntiles;
  r.ksplit = P.ksplit;
  r.units = int64_t(a.BH) * P.gchunks * r.ksplit;
  r.scale = a.scale;
  r.lohi = reinterpret_cast<const float2*>(reg + P.lohi);
  r.mask = reinterpret_cast<uint32_t*>(reg + P.mask);
  r.ld_mask = P.ld_mask;
  r.cand = reinterpret_cast<uint2*>(reg + P.cand);
  r.cap = P.cap;
  r.nabove = reinterpret_cast<int32_t*>(reg + P.nabove);
  r.ncand = reinterpret_cast<int32_t*>(reg + P.ncand);
  r.status = status;
  CUtensorMap tm_qhi, tm_qlo, tm_k;
  if (!make_rows_map(&tm_qhi, a.ws + a.L.qhi, uint64_t(a.rows), D, 128) ||
      !make_rows_map(&tm_qlo, a.ws + a.L.qlo, uint64_t(a.rows), D, 128) ||
      !make_keys_map(&tm_k, a.k, D, uint64_t(a.Nk), uint64_t(a.Nk), uint64_t(a.BH), 1u))
    return cudaErrorInvalidValue;
  auto kern = sa_rowscore_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t grid = r.units < num_sms ? r.units : num_sms;
  kern<<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, st>>>(r, tm_qhi, tm_qlo, tm_k);
  return cudaGetLastError();
}

// TOPK lists without the score matrix (see section 6); rows it cannot
// bracket go through the score and select kernels afterwards.
static cudaError_t launch_topk_direct(const BuildArgs& a, const TopkPlan& P, bool all_keys,
                                      int num_sms, cudaStream_t st, int32_t* status) {
  cudaError_t e;
  uint8_t* reg = a.ws + a.L.scores;
  int32_t* fail_count = reinterpret_cast<int32_t*>(a.ws + a.L.fail);
  int32_t* fail_rows = reinterpret_cast<int32_t*>(a.ws + a.L.fail + 256);
  int32_t* fail_units = fail_rows + a.rows;
  if (!all_keys) {
    float* samp = reinterpret_cast<float*>(reg + P.samp);
    e = a.d == 128 ? launch_scores<128>(a, num_sms, st, status, nullptr, samp, P.ld_samp, P.S, P.stride)
                   : launch_scores<64>(a, num_sms, st, status, nullptr, samp, P.ld_samp, P.S, P.stride);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (a.rows + kBrWarps - 1) / kBrWarps;
    sa_bracket_kernel<<<static_cast<unsigned>(blocks), 32 * kBrWarps, 0, st>>>(
        reinterpret_cast<const float*>(reg + P.samp), P.ld_samp, P.S, a.rows, P.r_hi, P.r_lo,
        reinterpret_cast<float2*>(reg + P.lohi));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = a.d == 128 ? launch_rowscore<128>(a, P, num_sms, st, status)
                   : launch_rowscore<64>(a, P, num_sms, st, status);
    if (e != cudaSuccess) return e;
    // fail count and unit flags start at zero (the rows list needs no clearing)
    if ((e = cudaMemsetAsync(fail_count, 0, 4, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(fail_units, 0, size_t(a.rows) * 4, st)) != cudaSuccess) return e;
  }
  FinArgs f;
  f.rows = a.rows;
  f.G = a.G;
  f.k = all_keys ? a.Nk : a.topk;
  f.Nk = a.Nk;
  f.nreg = P.nreg;
  f.cap = P.cap;
  f.gchunks = P.gchunks;
  f.all_keys = all_keys ? 1 : 0;
  f.mask = reinterpret_cast<const uint32_t*>(reg + P.mask);
  f.ld_mask = P.ld_mask;
  f.cand = reinterpret_cast<const uint2*>(reg + P.cand);
  f.nabove = reinterpret_cast<const int32_t*>(reg + P.nabove);
  f.ncand = reinterpret_cast<const int32_t*>(reg + P.ncand);
  f.col_idx = a.col_idx;
  f.col_capacity = a.col_capacity;
  f.counts = reinterpret_cast<int64_t*>(a.ws + a.L.counts);
  f.row_ptr = a.row_ptr;
  f.nnz = reinterpret_cast<int64_t*>(a.ws + a.L.misc);
  f.fail_rows = fail_rows;
  f.fail_count = fail_count;
  f.fail_units = fail_units;
  const size_t fin_smem = all_keys ? 0 : kFinMaskOff + size_t(P.ld_mask) * 4;
  e = cudaFuncSetAttribute(sa_topk_finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(fin_smem));
  if (e != cudaSuccess) return e;
  sa_topk_finalize_kernel<<<static_cast<unsigned>(a.rows), kSelThreads, fin_smem, st>>>(f);
  return cudaGetLastError();
}

cudaError_t launch_build_index(const BuildArgs& a, int num_sms, cudaStream_t st) {
  int64_t* misc = reinterpret_cast<int64_t*>(a.ws + a.L.misc);
  int32_t* status = reinterpret_cast<int32_t*>(misc + 1);
  cudaError_t e = cudaMemsetAsync(misc, 0, 16, st);
  if (e != cudaSuccess) return e;
  // TOPK by mean query: lists without the score matrix when its buffers fit
  const bool topk = a.stat < 0 && a.mode == SA_SELECT_TOPK;
  const bool all_keys = topk && a.topk >= a.Nk;
  TopkPlan P;
  if (topk && !all_keys) P = plan_topk(a, num_sms);
  const bool direct = all_keys || P.ok;
  if (a.stat >= 0) {
    // dense-step statistics of the full attention probabilities
    e = launch_colstat(a, reinterpret_cast<float*>(a.ws + a.L.scores), status, num_sms, st);
    if (e != cudaSuccess) return e;
  } else if (!all_keys) {
    uint16_t* qhi = reinterpret_cast<uint16_t*>(a.ws + a.L.qhi);
    uint16_t* qlo = reinterpret_cast<uint16_t*>(a.ws + a.L.qlo);
    if (a.d == 128)
      sa_meanq_kernel<128><<<static_cast<unsigned>(a.rows), 256, 0, st>>>(a.q, qhi, qlo, a.G, a.Nq, a.M);
    else
      sa_meanq_kernel<64><<<static_cast<unsigned>(a.rows), 256, 0, st>>>(a.q, qhi, qlo, a.G, a.Nq, a.M);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (direct) {
      e = launch_topk_direct(a, P, false, num_sms, st, status);
      if (e != cudaSuccess) return e;
      // the rows it left: their units' scores, then the select kernel on them
      const int32_t* fail_units = reinterpret_cast<const int32_t*>(a.ws + a.L.fail + 256) + a.rows;
      e = a.d == 128 ? launch_scores<128>(a, num_sms, st, status, fail_units)
                     : launch_scores<64>(a, num_sms, st, status, fail_units);
    } else {
      e = a.d == 128 ? launch_scores<128>(a, num_sms, st, status) : launch_scores<64>(a, num_sms, st, status);
    }
    if (e != cudaSuccess) return e;
  } else {
    e = launch_topk_direct(a, P, true, num_sms, st, status);
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
  if (!all_keys) {
    auto kern = direct ? sa_select_kernel<true> : sa_select_kernel<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sel_smem));
    if (e != cudaSuccess) return e;
    int64_t grid = a.rows;
    if (direct) {  // only the rows the direct path left
      s.row_count = reinterpret_cast<const int32_t*>(a.ws + a.L.fail);
      s.row_list = s.row_count + 64;
      grid = a.rows < 4 * int64_t(num_sms) ? a.rows : 4 * int64_t(num_sms);
    }
    kern<<<static_cast<unsigned>(grid), kSelThreads, sel_smem, st>>>(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (!direct) {  // (the TOPK path's finalize writes row_ptr and nnz)
    sa_scan_kernel<<<1, 1024, 0, st>>>(s.counts, a.rows, a.row_ptr, misc, a.col_capacity, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
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
