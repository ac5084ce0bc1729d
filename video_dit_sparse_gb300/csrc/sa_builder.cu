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

// Monotone map float -> uint32 (larger score, larger key).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
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
  static constexpr int kStages = 4;
  static constexpr int kThreads = 32 * 6;  // 4 epilogue warps, 1 MMA warp, 1 TMA warp
  static constexpr int kTile = 128 * D * 2;  // 128 rows of d bf16
  static constexpr int kSmemBytes = 1024 + 2 * kTile + kStages * kTile + 1024;
  static constexpr int kTmemCols = 256;
};

struct ScoreBars {
  uint64_t kfull[4], kempty[4];
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
                    const __grid_constant__ CUtensorMap tm_qlo, const __grid_constant__ CUtensorMap tm_k) {
  using C = ScoreCfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQh = smem;
  uint8_t* sQl = sQh + C::kTile;
  uint8_t* sK = sQl + C::kTile;
  ScoreBars* bars = reinterpret_cast<ScoreBars*>(sK + S * C::kTile);
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
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t t = 0;
    for (int64_t u = blockIdx.x; u < a.units; u += gridDim.x) {
      int64_t bh;
      int gc, t0, t1;
      score_unit(a, u, &bh, &gc, &t0, &t1);
      const int64_t g0 = int64_t(gc) * 128;
      const int ng = static_cast<int>(min64(128, a.G - g0));
      float* dst0 = a.scores + (bh * a.G + g0) * a.ld;
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
        const int64_t key = int64_t(tile) * 128 + warp * 32 + lane;
        if (key < a.Nk) {
          float* dst = dst0 + key;
#pragma unroll
          for (int gi = 0; gi < 128; ++gi)
            if (gi < ng) dst[int64_t(gi) * a.ld] = x[gi] * a.scale;
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
};

constexpr int kSelThreads = 1024;
constexpr int kBins = 2048;                 // radix levels of 11, 11 and 10 bits
constexpr float kMassOne = 4294967296.0f;   // fixed-point unit of probability mass (2^32)

// Probability mass exp(x - max) of one key in 2^-32 units; integer sums are
// exact and order-independent, so every thread agrees on the crossing bin.
__device__ __forceinline__ unsigned long long fixed_mass(float x, float rmax) {
  return __float2ull_rn(expf(x - rmax) * kMassOne);
}

__global__ void __launch_bounds__(kSelThreads) sa_select_kernel(const SelArgs a) {
  __shared__ uint32_t hist[kBins];
  __shared__ unsigned long long hmass[kBins];
  __shared__ float red_m[32], red_z[32];
  __shared__ int64_t scan_c[32], scan_m[32];
  __shared__ int32_t claim;
  __shared__ int32_t found_cnt;
  __shared__ int64_t found_above_cnt, found_above_mass;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const float* s = a.scores + row * a.ld;
  const int Nk = a.Nk;

  float rmax = -INFINITY, rz = 0.f;
  if (a.mode != SA_SELECT_TOPK) {
    // row max and sum of exp(x - max), one pass with rescaling
    float m = -INFINITY, z = 0.f;
    for (int j = tid; j < Nk; j += kSelThreads) {
      const float x = s[j];
      if (x > m) {
        z = z * expf(m - x) + 1.f;
        m = x;
      } else {
        z += expf(x - m);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), z2 = __shfl_xor_sync(0xffffffffu, z, o);
      const float mm = fmaxf(m, m2);
      z = (m == -INFINITY ? 0.f : z * expf(m - mm)) + (m2 == -INFINITY ? 0.f : z2 * expf(m2 - mm));
      m = mm;
    }
    if (lane == 0) {
      red_m[warp] = m;
      red_z[warp] = z;
    }
    __syncthreads();
    if (warp == 0) {
      m = red_m[lane];
      z = red_z[lane];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), z2 = __shfl_xor_sync(0xffffffffu, z, o);
        const float mm = fmaxf(m, m2);
        z = (m == -INFINITY ? 0.f : z * expf(m - mm)) + (m2 == -INFINITY ? 0.f : z2 * expf(m2 - mm));
        m = mm;
      }
      if (lane == 0) {
        red_m[0] = m;
        red_z[0] = z;
      }
    }
    __syncthreads();
    rmax = red_m[0];
    rz = red_z[0];
  }

  uint32_t cut = 0;
  int32_t ties = 0;
  int64_t count = Nk;
  if (a.mode == SA_SELECT_THRESHOLD) {
    // keep p_j >= tau  <=>  sigma_j >= ln tau + max + ln Z
    const float c = a.log_tau + rmax + logf(rz);
    const uint32_t kc = (c == -INFINITY) ? 0u : order_key(c);
    int64_t n = 0;
    for (int j = tid; j < Nk; j += kSelThreads) n += order_key(s[j]) >= kc;
    int64_t total;
    block_excl_scan<int64_t>(n, &total, scan_c);
    if (total > 0) {
      cut = kc > 0 ? kc - 1 : 0u;  // keys > kc - 1  <=>  keys >= kc
      ties = 0;
      count = total;
    } else {
      cut = order_key(rmax);  // none qualifies: the top-ranked key only
      ties = 1;
      count = 1;
    }
  } else if (a.mode == SA_SELECT_MASS && a.mass >= 1.0) {
    cut = 0;  // the whole mass needs every key
    ties = 0;
    count = Nk;
  } else {
    const bool by_mass = a.mode == SA_SELECT_MASS;
    const int64_t k = min64(max64(a.topk, 1), Nk);
    double target = static_cast<double>(k);
    uint32_t prefix = 0, pmask = 0;
    int64_t above_cnt = 0, above_mass = 0;
    int32_t last_cnt = 0;
    bool keep_all = false;
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
    for (int lv = 0; lv < 3; ++lv) {
      const int shift = shifts[lv], nb = 1 << widths[lv];
      for (int i = tid; i < kBins; i += kSelThreads) {
        hist[i] = 0;
        hmass[i] = 0ull;
      }
      if (tid == 0) claim = -1;
      __syncthreads();
      for (int j = tid; j < Nk; j += kSelThreads) {
        const float x = s[j];
        const uint32_t kx = order_key(x);
        if ((kx & pmask) == prefix) {
          const uint32_t bin = (kx >> shift) & (nb - 1);
          atomicAdd(&hist[bin], 1u);
          if (by_mass) atomicAdd(&hmass[bin], fixed_mass(x, rmax));
        }
      }
      __syncthreads();
      // Thread t owns bins nb-1-2t and nb-2-2t (descending score order).
      const int top = nb - 1 - 2 * tid;
      int64_t c2 = 0, m2 = 0;
      if (top >= 0) {
        c2 = int64_t(hist[top]) + hist[top - 1];
        m2 = int64_t(hmass[top]) + int64_t(hmass[top - 1]);
      }
      int64_t ctot, mtot;
      const int64_t cex = block_excl_scan<int64_t>(c2, &ctot, scan_c);
      const int64_t mex = block_excl_scan<int64_t>(m2, &mtot, scan_m);
      if (by_mass && lv == 0) target = a.mass * static_cast<double>(mtot);
      if (top >= 0) {
        int64_t cum_c = above_cnt + cex, cum_m = above_mass + mex;
        for (int e = 0; e < 2; ++e) {
          const int bin = top - e;
          const int64_t bc = hist[bin], bm = int64_t(hmass[bin]);
          const bool cross = by_mass
                                 ? (bm > 0 && double(cum_m + bm) >= target && double(cum_m) < target)
                                 : (bc > 0 && double(cum_c + bc) >= target && double(cum_c) < target);
          if (cross && atomicCAS(&claim, -1, bin) == -1) {
            found_cnt = static_cast<int32_t>(bc);
            found_above_cnt = cum_c - above_cnt;
            found_above_mass = cum_m - above_mass;
          }
          cum_c += bc;
          cum_m += bm;
        }
      }
      __syncthreads();
      const int bin = claim;
      if (bin < 0) {
        keep_all = true;  // target not reachable through rounding: keep every key
        break;
      }
      prefix |= static_cast<uint32_t>(bin) << shift;
      pmask |= static_cast<uint32_t>(nb - 1) << shift;
      above_cnt += found_above_cnt;
      above_mass += found_above_mass;
      last_cnt = found_cnt;
      __syncthreads();
    }
    if (keep_all) {
      cut = 0;
      ties = 0;
      count = Nk;
    } else if (by_mass) {
      // every key equal to the cut carries the same fixed-point mass
      const double e = static_cast<double>(fixed_mass(key_value(prefix), rmax));
      const double need = e > 0.0 ? ceil((target - double(above_mass)) / e) : 1.0;
      const int32_t n = need < 1.0 ? 1 : (need > double(last_cnt) ? last_cnt : static_cast<int32_t>(need));
      cut = prefix;
      ties = n;
      count = above_cnt + n;
    } else {
      cut = prefix;
      ties = static_cast<int32_t>(k - above_cnt);
      count = k;
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
__global__ void __launch_bounds__(kSelThreads) sa_emit_kernel(const float* scores, int64_t ld,
                                                              int32_t Nk, const uint32_t* cut,
                                                              const int32_t* ties,
                                                              const int64_t* row_ptr,
                                                              int32_t* col_idx, int64_t capacity) {
  __shared__ int32_t scratch[32];
  const int64_t row = blockIdx.x;
  const int64_t base = row_ptr[row], end = row_ptr[row + 1];
  if (end > capacity) return;  // reported by the scan
  const float* s = scores + row * ld;
  const uint32_t ck = cut[row];
  const int64_t nt = ties[row];
  int64_t run_sel = 0, run_tie = 0;
  for (int64_t c0 = 0; c0 < Nk; c0 += 4 * kSelThreads) {
    const int64_t j0 = c0 + 4 * threadIdx.x;
    float x[4];
    if (j0 + 3 < Nk) {
      const float4 v = *reinterpret_cast<const float4*>(s + j0);
      x[0] = v.x;
      x[1] = v.y;
      x[2] = v.z;
      x[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = j0 + e < Nk ? s[j0 + e] : -INFINITY;
    }
    bool sel[4], tie[4];
    int32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool in = j0 + e < Nk;
      const uint32_t kx = order_key(x[e]);
      sel[e] = in && kx > ck;
      tie[e] = in && kx == ck;
      packed += (sel[e] ? 1 : 0) + (tie[e] ? 0x10000 : 0);
    }
    int32_t total;
    const int32_t ex = block_excl_scan<int32_t>(packed, &total, scratch);
    int64_t sb = run_sel + (ex & 0xFFFF), tb = run_tie + (ex >> 16);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (sel[e]) {
        const int64_t pos = base + sb + min64(tb, nt);
        if (pos < end) col_idx[pos] = static_cast<int32_t>(j0 + e);
        ++sb;
      } else if (tie[e]) {
        const int64_t pos = base + sb + tb;
        if (tb < nt && pos < end) col_idx[pos] = static_cast<int32_t>(j0 + e);
        ++tb;
      }
    }
    run_sel += total & 0xFFFF;
    run_tie += total >> 16;
  }
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
  CUtensorMap tm_qhi, tm_qlo, tm_k;
  if (!make_rows_map(&tm_qhi, s.qhi, uint64_t(a.rows), D, 128) ||
      !make_rows_map(&tm_qlo, s.qlo, uint64_t(a.rows), D, 128) ||
      !make_rows_map(&tm_k, a.k, uint64_t(a.BH) * a.Nk, D, 128))
    return cudaErrorInvalidValue;
  auto kern = sa_score_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t grid = s.units < num_sms ? s.units : num_sms;
  kern<<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, st>>>(s, tm_qhi, tm_qlo, tm_k);
  return cudaGetLastError();
}

cudaError_t launch_build_index(const BuildArgs& a, int num_sms, cudaStream_t st) {
  int64_t* misc = reinterpret_cast<int64_t*>(a.ws + a.L.misc);
  int32_t* status = reinterpret_cast<int32_t*>(misc + 1);
  cudaError_t e = cudaMemsetAsync(misc, 0, 16, st);
  if (e != cudaSuccess) return e;
  uint16_t* qhi = reinterpret_cast<uint16_t*>(a.ws + a.L.qhi);
  uint16_t* qlo = reinterpret_cast<uint16_t*>(a.ws + a.L.qlo);
  if (a.d == 128)
    sa_meanq_kernel<128><<<static_cast<unsigned>(a.rows), 256, 0, st>>>(a.q, qhi, qlo, a.G, a.Nq, a.M);
  else
    sa_meanq_kernel<64><<<static_cast<unsigned>(a.rows), 256, 0, st>>>(a.q, qhi, qlo, a.G, a.Nq, a.M);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = a.d == 128 ? launch_scores<128>(a, num_sms, st, status) : launch_scores<64>(a, num_sms, st, status);
  if (e != cudaSuccess) return e;
  SelArgs s;
  s.scores = reinterpret_cast<const float*>(a.ws + a.L.scores);
  s.ld = a.L.ld;
  s.Nk = a.Nk;
  s.mode = a.mode;
  s.topk = a.topk;
  s.log_tau = a.threshold > 0.0 ? static_cast<float>(log(a.threshold)) : -INFINITY;
  s.mass = a.mass;
  s.cut = reinterpret_cast<uint32_t*>(a.ws + a.L.cut);
  s.ties = reinterpret_cast<int32_t*>(a.ws + a.L.ties);
  s.counts = reinterpret_cast<int64_t*>(a.ws + a.L.counts);
  sa_select_kernel<<<static_cast<unsigned>(a.rows), kSelThreads, 0, st>>>(s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  sa_scan_kernel<<<1, 1024, 0, st>>>(s.counts, a.rows, a.row_ptr, misc, a.col_capacity, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
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
