// sa_colstat.cu — dense-step key lists for sm_103a.
//
// FG-Attn review, cached mask (its free parameters and Fig. 10): after a
// dense denoising step a slice (query group g, key j) is kept when at least
// one of its full-attention scores reaches tau_cached = 0.5/N, and the mask
// is reused by the following sparse steps.  Chipmunk review, major comment 2
// / Alg. 4: columns are ranked by the sum of their attention probabilities
// over the group, with the softmax constants of an earlier step.  Both need,
// for every unit and key, one statistic of
//     p_ij = exp(scale q_i.k_j - lse_i),   i in the group's rows,
// where lse_i is the dense step's row log-sum-exp (the dense forward's lse
// output).  sa_colstat_kernel writes ln max_i p_ij or ln sum_i p_ij for every
// key into the builder's score matrix; the select, scan and emit kernels of
// the mean-query builder then apply TOPK, MASS or a LEVEL threshold to it.
//
// Per unit the queries of GPU groups (NQ = 256 columns: two groups of at
// most 128 rows, or one of up to 256) stay in shared memory and K tiles of
// 128 keys stream in by TMA.  One tcgen05 MMA chain per tile gives
// S^T = K_tile Q^T in TMEM with keys on the 128 lanes and queries on the
// columns, so each epilogue thread owns one key and reduces over each
// group's queries in registers (no cross-lane reduction).  Two groups per
// unit read every K tile once for both: 256 flops per K byte from L2.
#include <cfloat>

#include "sa_device.cuh"
#include "sa_internal.h"
#include "sa_tma.h"

namespace sa {

struct ColArgs {
  const float* lse;  // [B*H*Nq] natural-log row normaliser
  float* out;        // score matrix [rows, ld]
  int64_t ld, G, rows;
  int32_t Nq, Nk, M;
  float sl;          // scale * log2(e)
  int32_t stat;      // 0 max, 1 sum
  int32_t gpu;       // groups per unit: 2 when M <= 128, else 1
  int64_t units;     // B*H*ceil(G/gpu)
  int64_t uph;       // units per head
  int32_t* status;
};

template <int D, int NQ>
struct ColCfg {
  static constexpr int kStages = 4;
  // two sets of 4 epilogue warps (set s takes the tiles in TMEM buffer s),
  // 1 MMA warp, 1 TMA warp
  static constexpr int kEpiWarps = 8;
  static constexpr int kMmaWarp = kEpiWarps, kTmaWarp = kEpiWarps + 1;
  static constexpr int kThreads = 32 * (kEpiWarps + 2);
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kQBytes = NQ * D * 2;
  // each epilogue warp keeps its own copy of the unit's lse column (no
  // cross-warp barrier that an aborting warp could leave waiting)
  static constexpr int kSmemBytes = 1024 + kQBytes + kStages * kTile + kEpiWarps * NQ * 4 + 1024;
  static constexpr int kTmemCols = 2 * NQ;
  static_assert(NQ == 256, "query columns");
};

struct ColBars {
  uint64_t kfull[4], kempty[4];
  uint64_t qfull, qempty, drain;
  uint64_t dfull[2], dempty[2];
  uint32_t tmem_base;
  int abort;
};

template <int D, int NQ>
__global__ void __launch_bounds__(ColCfg<D, NQ>::kThreads, 1)
    sa_colstat_kernel(const ColArgs a, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k) {
  using C = ColCfg<D, NQ>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::kQBytes;
  float* sL = reinterpret_cast<float*>(sK + S * C::kTile);  // per warp: lse in exp2 units per query column
  ColBars* bars = reinterpret_cast<ColBars*>(sL + C::kEpiWarps * NQ);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = (a.Nk + 127) / 128;
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
    // Thread = key (TMEM lane); the group's queries are the columns.  Warp
    // set `es` handles the tiles that land in TMEM buffer es.
    const int es = warp / 4, tid = threadIdx.x % 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    float* wL = sL + warp * NQ;
    uint32_t t = 0;
    constexpr int kCols = NQ;  // query columns of one unit
    for (int64_t u = blockIdx.x; u < a.units; u += gridDim.x) {
      const int64_t bh = u / a.uph, g0 = (u % a.uph) * a.gpu;
      const int slot_cols = NQ / a.gpu;  // 128 or 256 columns per group
      // group slot s covers columns [s*slot_cols, ...) and rows g0+s of the head
      int nrows[2], nch[2];
#pragma unroll
      for (int sl = 0; sl < 2; ++sl) {
        const int64_t g = g0 + sl;
        nrows[sl] = (sl < a.gpu && g < a.G) ? static_cast<int>(min64(a.M, a.Nq - g * a.M)) : 0;
        nch[sl] = (nrows[sl] + 31) / 32;
      }
      // Columns past a group's rows, and rows without a finite lse, get
      // +inf: their exponent is -inf and they add nothing.
      __syncwarp();  // every lane is done with the previous unit's columns
      for (int c = lane; c < kCols; c += 32) {
        const int sl = c / slot_cols, r = c % slot_cols;
        float v = INFINITY;
        if (r < (sl == 0 ? nrows[0] : nrows[1])) {
          const float l = __ldg(a.lse + bh * a.Nq + (g0 + sl) * a.M + r);
          if (isfinite(l)) v = l * 1.4426950408889634f;
        }
        wL[c] = v;
      }
      __syncwarp();
      const float sl_ = a.sl;
      for (int tile = 0; tile < ntiles; ++tile, ++t) {
        const uint32_t b = t & 1;
        if (b != static_cast<uint32_t>(es)) continue;
        if (!mbar_wait(&bars->dfull[b], (t >> 1) & 1, abort)) goto done;
        tc_fence_after();
        const uint32_t sbase = tmem + lane_base + b * NQ;
        float res[2];
#pragma unroll
        for (int sl = 0; sl < 2; ++sl) {
          const int c0 = sl * slot_cols / 32, c1 = c0 + nch[sl];
          if (a.stat == 0) {
            // ln max_i p_ij = ln2 * max_i (sl x_ij - lse2_i)
            float m = -INFINITY;
            for (int c = c0; c < c1; ++c) {
              uint32_t r[32];
              tmem_ld32(sbase + c * 32, r);
              tmem_ld_wait();
              const float4* l4 = reinterpret_cast<const float4*>(wL + c * 32);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float4 L = l4[e];
                const float y0 = fmaf(__uint_as_float(r[4 * e]), sl_, -L.x);
                const float y1 = fmaf(__uint_as_float(r[4 * e + 1]), sl_, -L.y);
                const float y2 = fmaf(__uint_as_float(r[4 * e + 2]), sl_, -L.z);
                const float y3 = fmaf(__uint_as_float(r[4 * e + 3]), sl_, -L.w);
                m = fmax3(m, fmaxf(y0, y1), fmaxf(y2, y3));
              }
            }
            res[sl] = m * 0.69314718055994531f;
          } else {
            // ln sum_i p_ij, accumulated relative to a running maximum so that
            // it never underflows: per 32-query chunk a max and a sum of exp2.
            float mt = -INFINITY, st = 0.f;
            for (int c = c0; c < c1; ++c) {
              uint32_t r[32];
              tmem_ld32(sbase + c * 32, r);
              tmem_ld_wait();
              const float4* l4 = reinterpret_cast<const float4*>(wL + c * 32);
              float y[32];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float4 L = l4[e];
                y[4 * e] = fmaf(__uint_as_float(r[4 * e]), sl_, -L.x);
                y[4 * e + 1] = fmaf(__uint_as_float(r[4 * e + 1]), sl_, -L.y);
                y[4 * e + 2] = fmaf(__uint_as_float(r[4 * e + 2]), sl_, -L.z);
                y[4 * e + 3] = fmaf(__uint_as_float(r[4 * e + 3]), sl_, -L.w);
              }
              float mc = y[0];
#pragma unroll
              for (int e = 1; e < 31; e += 2) mc = fmax3(mc, y[e], y[e + 1]);
              mc = fmaxf(mc, y[31]);
              // (branch-free: a chunk in which no row counts has mc = -inf and
              // adds exp2(-inf) = 0 terms; the warp stays converged for the
              // next TMEM load)
              const float mr = mc == -INFINITY ? 0.f : mc;
              float s0 = 0.f, s1 = 0.f;
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                s0 += fast_exp2(y[e] - mr);
                s1 += fast_exp2(y[e + 1] - mr);
              }
              const float mn = fmaxf(mt, mc);
              const float ms = mn == -INFINITY ? 0.f : mn;
              st = st * fast_exp2(mt - ms) + (s0 + s1) * fast_exp2(mr - ms);
              mt = mn;
            }
            res[sl] = mt == -INFINITY ? -INFINITY : (mt + __log2f(st)) * 0.69314718055994531f;
          }
        }
        tc_fence_before();
        mbar_arrive(&bars->dempty[b]);
        const int key = tile * 128 + tid;
        // a key no row counts for (every lse non-finite) ranks lowest, finite
        if (key < a.Nk) {
#pragma unroll
          for (int sl = 0; sl < 2; ++sl)
            if (nrows[sl] > 0) {
              const int64_t row = bh * a.G + g0 + sl;
              a.out[row * a.ld + key] = res[sl] >= -FLT_MAX ? res[sl] : -FLT_MAX;
            }
        }
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16(128, NQ, false, false);
      const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK);
      uint32_t t = 0, un = 0;
      bool ok = true;
      for (int64_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        if (!mbar_wait(&bars->qfull, un & 1, abort)) break;
        for (int tile = 0; tile < ntiles; ++tile, ++t) {
          const uint32_t s = t % S, b = t & 1;
          if (!mbar_wait(&bars->kfull[s], (t / S) & 1, abort) ||
              !mbar_wait(&bars->dempty[b], ((t >> 1) & 1) ^ 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem + b * NQ;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = k_addr + s * C::kTile + (kk >> 2) * 128 * 128 + (kk & 3) * 32;
            const uint32_t qa = q_addr + (kk >> 2) * NQ * 128 + (kk & 3) * 32;
            mma_ss(d_tmem, sw128_desc(ka, 16, 1024), sw128_desc(qa, 16, 1024), kIdesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->dfull[b]);
          mma_commit(&bars->kempty[s]);
          if (tile == ntiles - 1) mma_commit(&bars->qempty);
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
    const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK);
    uint32_t t = 0, un = 0;
    for (int64_t u = blockIdx.x; u < a.units; u += gridDim.x) {
      const int64_t bh = u / a.uph, g0 = (u % a.uph) * a.gpu;
      if (un > 0 && !mbar_wait(&bars->qempty, (un - 1) & 1, abort)) goto done;
      // 128-row blocks of queries: with two groups per unit, block s holds
      // rows (g0+s)*M ..; with one, blocks 0 and 1 hold rows g0*M .. +255.
      // Rows past a group or the head only feed columns whose lse is +inf;
      // rows past the tensor read as zeros.
      mbar_expect_tx(&bars->qfull, C::kQBytes);
#pragma unroll
      for (int rb = 0; rb < NQ / 128; ++rb) {
        const int64_t r0 = a.gpu == 2 ? (g0 + rb) * a.M : g0 * a.M + rb * 128;
        const int qrow = static_cast<int>(bh * a.Nq + r0);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_2d(q_addr + cb * NQ * 128 + rb * 128 * 128, &tm_q, 64 * cb, qrow, &bars->qfull);
      }
      for (int tile = 0; tile < ntiles; ++tile, ++t) {
        const uint32_t s = t % S;
        if (!mbar_wait(&bars->kempty[s], ((t / S) & 1) ^ 1, abort)) goto done;
        mbar_expect_tx(&bars->kfull[s], C::kTile);
        const int krow = static_cast<int>(bh * a.Nk + int64_t(tile) * 128);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_2d(k_addr + s * C::kTile + cb * 128 * 128, &tm_k, 64 * cb, krow, &bars->kfull[s]);
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

template <int D, int NQ>
static cudaError_t launch_cs(const ColArgs& a, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                             int num_sms, cudaStream_t st) {
  using C = ColCfg<D, NQ>;
  auto kern = sa_colstat_kernel<D, NQ>;
  // At least half the SM's shared memory: one CTA per SM, which owns the
  // SM's TMEM (two CTAs of 512 columns would serialise on the allocation).
  const int smem = C::kSmemBytes > 120 * 1024 ? C::kSmemBytes : 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = a.units < num_sms ? a.units : num_sms;
  kern<<<static_cast<unsigned>(grid), C::kThreads, smem, st>>>(a, tm_q, tm_k);
  return cudaGetLastError();
}

cudaError_t launch_colstat(const BuildArgs& b, float* scores, int32_t* status, int num_sms,
                           cudaStream_t st) {
  ColArgs a;
  a.lse = b.lse;
  a.out = scores;
  a.ld = b.L.ld;
  a.G = b.G;
  a.rows = b.rows;
  a.Nq = b.Nq;
  a.Nk = b.Nk;
  a.M = b.M;
  a.sl = static_cast<float>(static_cast<double>(b.scale) * 1.4426950408889634);
  a.stat = b.stat;
  a.gpu = b.M <= 128 ? 2 : 1;
  a.uph = (b.G + a.gpu - 1) / a.gpu;
  a.units = int64_t(b.BH) * a.uph;
  a.status = status;
  CUtensorMap tm_q, tm_k;
  if (!make_rows_map(&tm_q, b.q, uint64_t(b.BH) * b.Nq, b.d, 128) ||
      !make_rows_map(&tm_k, b.k, uint64_t(b.BH) * b.Nk, b.d, 128))
    return cudaErrorInvalidValue;
  return b.d == 128 ? launch_cs<128, 256>(a, tm_q, tm_k, num_sms, st)
                    : launch_cs<64, 256>(a, tm_q, tm_k, num_sms, st);
}

}  // namespace sa
