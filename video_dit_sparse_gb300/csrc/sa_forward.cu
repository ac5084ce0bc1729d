// sa_forward.cu — fused column-sparse attention forward for sm_103a.
//
// One persistent CTA per SM walks (batch, head, group) units in head-major
// order.  Per unit it keeps the group's queries in shared memory and streams
// the unit's kept keys in tiles of BN:
//   gather warps  copy the listed K and V rows (16-byte cp.async per chunk;
//                 each stage's mbarrier completes when the copies land) into
//                 128B-swizzled tiles — the FG-Attn review's gather-load
//                 (What carries the argument): the next tile's indices are
//                 loaded into registers while this tile's copies are issued,
//                 and rows land in tensor-core-ready shared-memory tiles.
//                 The query tile arrives by one 2-D TMA load per 64 columns;
//   the MMA warp  issues S = Q K^T (tcgen05, fp32 in TMEM, double-buffered)
//                 and O += P V with P read from TMEM;
//   softmax warps keep the running max / sum per query row in registers
//                 (DiT page, "Online Softmax"), write P as bf16 over S in
//                 TMEM and rescale O only when the running max must grow by
//                 2^32 (exact after the final division by the sum): for
//                 128-row groups a unit finds a row max in its first tile
//                 and then only in the rare tiles whose P overflow that bound;
//                 the epilogue writes O / l in bf16 and lse = m + ln l.
// The softmax is restricted to the kept keys (Chipmunk review, major
// comment 1, Alg. 3).  Groups longer than 128 rows (C = 192) use two
// 128-row blocks that share every K/V tile: 128-key tiles, each softmax
// thread working its row in two 64-key halves, Q read from shared memory.
// Without index lists every unit
// keeps all keys in order (dense attention, the dense step of a cached
// mask).
//
// The DELTA variant is the Chipmunk review's sparse delta (Eq. 1 with the
// normalisation constants of an earlier step, Appendix B.2): no running max
// and no renormalisation; P = exp(l - lse_ref) with the caller's per-row
// lse_ref, and the epilogue writes base + sign * P V.  Without the final
// division nothing cancels the rounding of P, so P goes to the PV MMA as two
// bf16 terms (hi and the rounded remainder, in the two halves of the S
// buffer) and O accumulates both products.
#include <atomic>

#include "sa_device.cuh"
#include "sa_internal.h"
#include "sa_tma.h"

namespace sa {

template <int D, int RB, int BN, int STAGES>
struct FwdCfg {
  // 4*RB softmax warps (one per 32 rows of each 128-row block), one
  // MMA-issuing warp, then the gather warps.
  static constexpr int kSoftmaxWarps = 4 * RB;
  static constexpr int kMmaWarp = kSoftmaxWarps;
  static constexpr int kProdWarp0 = kSoftmaxWarps + 1;
  // 128-row groups: seven gather warps (12 warps in all), with the softmax
  // warpgroup's registers raised (its threads hold a 128-float S row) and the
  // rest lowered after launch; longer groups: three, no split (their eight
  // softmax warps hold half rows).
  static constexpr int kProdWarps = RB == 1 ? 7 : 3;
  static constexpr int kProdThreads = 32 * kProdWarps;
  static constexpr int kThreads = 32 * (kSoftmaxWarps + 1 + kProdWarps);
  // setmaxnreg acts per warpgroup: the four softmax warps (one warpgroup) go
  // up, the other two warpgroups down.  A split inside a warpgroup never
  // completes.
  static constexpr bool kRegSplit = RB == 1;
  static constexpr int kRegSoftmax = 240, kRegOther = 80;
  static_assert(!kRegSplit || (kSoftmaxWarps % 4 == 0 && kThreads % 128 == 0),
                "register split by whole warpgroups");
  static_assert(!kRegSplit || (kRegSoftmax * 4 + kRegOther * (kThreads / 32 - 4)) * 32 <=
                                  (65536 / kThreads / 8 * 8) * kThreads,
                "register split exceeds the launch's registers");
  // Gather mapping: 8 lanes per row, lane copies 16-byte chunks sub, sub+8
  // (one 128-byte line of 4 rows per copy instruction).
  static constexpr int kLanesPerRow = 8;
  static constexpr int kChunksPerLane = (D / 8) / kLanesPerRow;
  static constexpr int kRowStep = kProdThreads / kLanesPerRow;
  static constexpr int kKVRowsPerThread = (BN + kRowStep - 1) / kRowStep;
  // Lazy rescale: O and the row sums are rescaled only when the running max
  // must grow (a tile's P against it would sum past 2^kRescaleLog2, or, for
  // 192-row groups, the tile's max exceeds it by kRescaleLog2).  P stays
  // <= 2^32 and O, l within fp32.
  static constexpr float kRescaleLog2 = 32.f;
  static constexpr float kRescaleLimit = 4294967296.f;  // 2^kRescaleLog2
  // Tiles that cannot need a row max skip it (see the softmax warps): the
  // 128-row path here, the half-tile path (kHalves) by the same sum check
  // (the delta has a fixed normaliser: no max at all).
  static constexpr bool kLazyMax = RB == 1;
  // groups of more than 128 rows with 128-key tiles: each softmax thread
  // takes its row's tile in two 64-key halves (a 128-float row would not fit
  // the 168 registers of a 12-warp block without a register split)
  static constexpr bool kHalves = RB == 2 && BN == 128;
  static constexpr int kQBlock = 128 * D * 2;    // one 128-row block of Q
  static constexpr int kQBytes = RB * kQBlock;
  static constexpr int kTile = BN * D * 2;       // one K or V tile
  static constexpr int kSCols = RB * BN;         // TMEM columns per S buffer
  // 128-row groups double-buffer S; with two row blocks each block has one S
  // buffer (the MMA warp issues PV(j-1) of a block before QK(j) of the same
  // block, so the tensor core, which runs one thread's MMAs in order, reads P
  // before S is overwritten).  Where Q fits in TMEM beside S and O (below),
  // the QK MMAs read only K from shared memory; otherwise (two row blocks of
  // 128-key tiles) they read Q from its shared-memory tile.
  static constexpr int kSBufs = RB == 2 ? 1 : 2;
  static constexpr int kOCol = kSBufs * kSCols;
  static __device__ __forceinline__ uint32_t sbuf(uint32_t tt) { return kSBufs == 2 ? (tt & 1u) : 0u; }
  static __device__ __forceinline__ uint32_t sphase(uint32_t tt) {
    return kSBufs == 2 ? ((tt >> 1) & 1u) : (tt & 1u);
  }
  // Q moves from shared memory into TMEM (D/2 columns per 128-row block) once
  // per unit, so the QK^T MMAs read only K from shared memory, when TMEM has
  // room for it.
  static constexpr int kQCol = kOCol + RB * D;
  static constexpr bool kQTmem = kQCol + RB * D / 2 <= 512;
  static constexpr int kUsedCols = kQCol + (kQTmem ? RB * D / 2 : 0);
  static constexpr int kTmemCols = kUsedCols <= 128 ? 128 : (kUsedCols <= 256 ? 256 : 512);
  static constexpr int kBarBytes = 1024;
  static constexpr int kSmemBytes = 1024 + kQBytes + 2 * STAGES * kTile + kBarBytes;
  static_assert(kUsedCols <= 512, "TMEM budget");
  static_assert(BN % 64 == 0 && D % 64 == 0, "tile shapes");
  static_assert(kProdThreads % kLanesPerRow == 0 && kChunksPerLane >= 1, "gather mapping");
};

// The CTA's unit sequence reaches every role through a ring of kRing slots
// in shared memory: the first gather thread, which starts each unit before
// any other role, fills the slot of the unit after next once every role has
// read the slot's previous unit; -1 ends the sequence.  Two slots keep at
// most one unit drawn ahead of the slowest role, so that units drawn from the
// shared counter do not pile up in one CTA.
constexpr int kRing = 2;

// The f-th unit of this CTA: from the launch's counter (dynamic: a CTA that
// finishes early takes more units, so ragged lists balance), else units
// b, b + gridDim.x, ...; -1 past the last unit.
__device__ __forceinline__ int64_t draw_unit(const FwdArgs& a, uint32_t f) {
  const int64_t u = a.sched ? static_cast<int64_t>(atomicAdd(a.sched, 1u))
                            : static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(f) * gridDim.x;
  return u < a.units ? u : -1;
}

template <int RB, int STAGES>
struct FwdBars {
  uint64_t kfull[STAGES], vfull[STAGES], kempty[STAGES], vempty[STAGES];
  uint64_t qfull, qempty, drain;
  uint64_t ring_full[kRing], ring_empty[kRing];
  int64_t ring_u[kRing];
  uint64_t sfull[2][RB], pfull[2][RB], pvdone[2][RB], ofree[RB];
  uint32_t tmem_base;
  int abort;
};

// Unit number i of this CTA from the ring (-1: no more units).  Every
// thread of a reading warp calls it; `release` (one lane per reading warp,
// after the warp has read the slot) frees the slot for the unit after next.
template <class Bars>
__device__ __forceinline__ bool ring_read(Bars* bars, uint32_t i, int64_t* u, bool release,
                                          volatile int* abort) {
  const uint32_t s = i % kRing;
  if (!mbar_wait(&bars->ring_full[s], (i / kRing) & 1, abort)) return false;
  *u = bars->ring_u[s];
  __syncwarp(__activemask());
  if (release) mbar_arrive(&bars->ring_empty[s]);
  return true;
}

// Unit u's list bounds.  A malformed row_ptr pair makes the unit empty.
template <bool DENSE>
__device__ __forceinline__ int64_t unit_list(const FwdArgs& a, int64_t u, int64_t* begin,
                                             bool* bad) {
  if (DENSE) {
    *bad = false;
    *begin = 0;
    return a.Nk;
  }
  const int64_t b0 = __ldg(a.row_ptr + u), b1 = __ldg(a.row_ptr + u + 1);
  if (b0 < 0 || b1 < b0 || b1 > a.nnz) {
    *bad = true;
    *begin = 0;
    return 0;
  }
  *bad = false;
  *begin = b0;
  return b1 - b0;
}

// Writes row values o[c] = base[c] + sign * acc[c] * inv for 32 columns
// starting at column c0 (bf16 RNE or fp32 output).
__device__ __forceinline__ void store_row32(const FwdArgs& a, int64_t orow_off, int c0,
                                            const uint32_t* acc, float mul, bool delta) {
  float v[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(acc[e]) * mul;
  if (delta && a.base) {
    const float4* b4 = reinterpret_cast<const float4*>(a.base + orow_off + c0);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float4 b = __ldg(b4 + e);
      v[4 * e] += b.x;
      v[4 * e + 1] += b.y;
      v[4 * e + 2] += b.z;
      v[4 * e + 3] += b.w;
    }
  }
  if (a.out_fp32) {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(a.o) + orow_off + c0);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      dst[e] = make_uint4(__float_as_uint(v[4 * e]), __float_as_uint(v[4 * e + 1]),
                          __float_as_uint(v[4 * e + 2]), __float_as_uint(v[4 * e + 3]));
  } else {
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) w[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + orow_off + c0);
#pragma unroll
    for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
  }
}

// DENSE (no lists) is a template parameter: a run-time choice inside the
// gather warps' index loads costs a fifth of the sparse kernel's speed.
template <int D, int RB, int BN, int STAGES, bool DELTA, bool DENSE>
__global__ void __launch_bounds__(FwdCfg<D, RB, BN, STAGES>::kThreads, 1)
    sa_forward_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap tmq) {
  using C = FwdCfg<D, RB, BN, STAGES>;
  using Bars = FwdBars<RB, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::kQBytes;
  uint8_t* sV = sK + STAGES * C::kTile;
  Bars* bars = reinterpret_cast<Bars*>(sV + STAGES * C::kTile);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->kfull[s], C::kProdThreads);
      mbar_init(&bars->vfull[s], C::kProdThreads);
      mbar_init(&bars->kempty[s], 1);
      mbar_init(&bars->vempty[s], 1);
    }
    mbar_init(&bars->qfull, 1);
    mbar_init(&bars->qempty, 1);
    mbar_init(&bars->drain, 1);
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&bars->ring_full[r], 1);
      // one arrival from each reader: the MMA thread, every softmax and gather warp
      mbar_init(&bars->ring_empty[r], 1 + C::kSoftmaxWarps + C::kProdWarps);
    }
    for (int b = 0; b < 2; ++b)
      for (int r = 0; r < RB; ++r) {
        mbar_init(&bars->sfull[b][r], 1);
        mbar_init(&bars->pfull[b][r], 128);
        mbar_init(&bars->pvdone[b][r], 1);
      }
    for (int r = 0; r < RB; ++r) mbar_init(&bars->ofree[r], 128);
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
  const int64_t G = a.G;
  if (C::kRegSplit) {
    if (warp < 4)
      reg_alloc<C::kRegSoftmax>();
    else
      reg_dealloc<C::kRegOther>();
  }

  if (warp < C::kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax
    const int rb = warp >> 2, quarter = warp & 3;
    const int row_in_unit = rb * 128 + quarter * 32 + lane;
    // A warp whose 32 rows lie past every group (the padding rows of a
    // 192-row group in its second 128-row block) skips the softmax work.
    const bool idle = rb * 128 + quarter * 32 >= a.M;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t t = 0, un = 0;
    for (uint32_t i = 0;; ++i) {
      int64_t u;
      if (!ring_read(bars, i, &u, lane == 0, abort)) goto done;
      if (u < 0) break;
      int64_t begin;
      bool bad;
      const int64_t len = unit_list<DENSE>(a, u, &begin, &bad);
      if (bad && threadIdx.x == 0) report(a.status, SA_DEVERR_ROW_PTR);
      const int64_t bh = u / G, g = u % G;
      const int64_t grow = g * a.M + row_in_unit;
      const bool valid = row_in_unit < a.M && grow < a.Nq;
      const int64_t orow_off = (bh * a.Nq + grow) * D;
      const uint32_t n = static_cast<uint32_t>((len + BN - 1) / BN);
      if (n == 0) {
        if (DELTA) {
          if (valid) {
            const uint32_t zero[32] = {};
#pragma unroll
            for (int c = 0; c < D / 32; ++c) store_row32(a, orow_off, c * 32, zero, 0.f, true);
          }
          continue;
        }
        if (valid) {
          const uint4 z = make_uint4(0, 0, 0, 0);
          uint4* dst = a.out_fp32 ? reinterpret_cast<uint4*>(static_cast<float*>(a.o) + orow_off)
                                  : reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + orow_off);
          const int n16 = a.out_fp32 ? D / 4 : D / 8;
          for (int c = 0; c < n16; ++c) dst[c] = z;
          if (a.lse) a.lse[bh * a.Nq + grow] = -INFINITY;
        }
        continue;
      }
      const float sl = a.scale_log2;  // |scale| * log2(e) > 0
      float m = -INFINITY, l = 0.f, lr = 0.f;
      if (DELTA) {
        // the fixed normaliser in exp2 units; a row without a finite one adds nothing
        const float lr0 = valid ? __ldg(a.lse_ref + bh * a.Nq + grow) : INFINITY;
        m = isfinite(lr0) ? lr0 * 1.4426950408889634f : INFINITY;
      }
      // One S tile: row max, exponentials, sums, P back into TMEM.
      auto tile = [&](uint32_t j) -> bool {
        const uint32_t tt = t + j, b = C::sbuf(tt);
        const int nvalid = static_cast<int>(min64(BN, len - int64_t(j) * BN));
        if (!mbar_wait(&bars->sfull[b][rb], C::sphase(tt), abort)) return false;
        if (idle) {  // rows past the group: their P and O are never used
          mbar_arrive(&bars->pfull[b][rb]);
          return true;
        }
        tc_fence_after();
        const uint32_t sbase = tmem + lane_base + b * C::kSCols + rb * BN;
        // O, l and lr times 2^(m - mn) with m raised to mn where `raise`
        // (warp-collective: every lane takes part, alpha = 1 where not raised).
        auto rescale = [&](bool raise, float mn) -> bool {
          // O must hold PV of the previous tile before it is rescaled.
          const uint32_t tp = tt - 1;
          if (!mbar_wait(&bars->pvdone[C::sbuf(tp)][rb], C::sphase(tp), abort)) return false;
          tc_fence_after();
          float alpha = 1.f;
          if (raise) {
            alpha = fast_exp2(m - mn);
            m = mn;
          }
          l *= alpha;
          lr *= alpha;
          const uint32_t obase = tmem + lane_base + C::kOCol + rb * D;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(obase + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(obase + c * 32, r);
          }
          tmem_st_wait();
          return true;
        };
        if constexpr (C::kHalves && DELTA) {
          // The delta's tile in two 64-key halves, each finished before the
          // next is loaded (a fixed normaliser needs no check): its P as bf16
          // hi and remainder goes to the half's own S columns (hi to the first
          // 32, remainder to the last 32), which the PV MMAs read that way.
          constexpr int H = BN / 2;
          const uint64_t sl2 = f2(sl, sl), nm2 = f2(-m, -m);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float x[H];
#pragma unroll
            for (int c = 0; c < H / 32; ++c)
              tmem_ld32(sbase + h * H + c * 32, reinterpret_cast<uint32_t*>(x + c * 32));
            tmem_ld_wait();
            if (nvalid < (h + 1) * H) {  // tail tile: columns past the list do not exist
#pragma unroll
              for (int c = 0; c < H; ++c)
                if (h * H + c >= nvalid) x[c] = -INFINITY;
            }
            uint32_t phi[H / 2], plo[H / 2];
#pragma unroll
            for (int c = 0; c < H / 2; ++c) {
              const uint64_t y = fma2(f2(x[2 * c], x[2 * c + 1]), sl2, nm2);
              const float p0 = fast_exp2(f2lo(y)), p1 = fast_exp2(f2hi(y));
              phi[c] = pack_bf16(p0, p1);
              plo[c] = pack_bf16(p0 - __uint_as_float(phi[c] << 16), p1 - __uint_as_float(phi[c] & 0xFFFF0000u));
            }
            tmem_st32(sbase + h * H, phi);
            tmem_st32(sbase + h * H + H / 2, plo);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars->pfull[b][rb]);
          return true;
        } else if constexpr (C::kHalves) {
          static_assert(BN == 128, "half tiles: 128-key tiles");
          // The tile in two 64-key halves (keys 0-63 in S columns 0-63, keys
          // 64-127 in 64-127): a thread holds one half's scores and both
          // halves' P, which is stored only once the tile's sum check has
          // passed (the slow path reloads the first half's scores from S).
          constexpr int H = BN / 2;
          float x[H];
          uint32_t pa[H / 2], pb[H / 2];
          uint64_t ps[4];
          float pr[4];
          auto load_half = [&](int h) {
#pragma unroll
            for (int c = 0; c < H / 32; ++c)
              tmem_ld32(sbase + h * H + c * 32, reinterpret_cast<uint32_t*>(x + c * 32));
            tmem_ld_wait();
            if (nvalid < (h + 1) * H) {  // tail tile: columns past the list do not exist
#pragma unroll
              for (int c = 0; c < H; ++c)
                if (h * H + c >= nvalid) x[c] = -INFINITY;
            }
          };
          auto half_max = [&]() -> float {  // scaled max of the half in x
            float t8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) t8[i] = fmaxf(x[i], x[8 + i]);
#pragma unroll
            for (int c = 16; c < H; c += 16)
#pragma unroll
              for (int i = 0; i < 8; ++i) t8[i] = fmax3(t8[i], x[c + i], x[c + 8 + i]);
            return sl * fmax3(fmax3(t8[0], t8[1], t8[2]), fmax3(t8[3], t8[4], t8[5]), fmaxf(t8[6], t8[7]));
          };
          auto half_exps = [&](float mm, uint32_t* pp) {  // P of the half in x, into the sums
            const uint64_t sl2 = f2(sl, sl), nm2 = f2(-mm, -mm);
#pragma unroll
            for (int c = 0; c < H / 2; ++c) {
              const uint64_t y = fma2(f2(x[2 * c], x[2 * c + 1]), sl2, nm2);
              const float p0 = fast_exp2(f2lo(y)), p1 = fast_exp2(f2hi(y));
              pp[c] = pack_bf16(p0, p1);
              ps[c & 3] = add2(ps[c & 3], f2(p0, p1));
              pr[c & 3] = add_bf16x2(pp[c], pr[c & 3]);
            }
          };
          auto zero_sums = [&]() {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              ps[i] = 0;
              pr[i] = 0.f;
            }
          };
          float ts, tr;
          auto tile_sums = [&]() {
            const uint64_t s2 = add2(add2(ps[0], ps[1]), add2(ps[2], ps[3]));
            ts = f2lo(s2) + f2hi(s2);
            tr = (pr[0] + pr[1]) + (pr[2] + pr[3]);
          };
          zero_sums();
          if (j == 0) {  // the unit's first tile sets the running max
            load_half(0);
            float mx = half_max();
            load_half(1);
            mx = fmaxf(mx, half_max());
            m = mx;
            half_exps(m, pb);
            load_half(0);
            half_exps(m, pa);
          } else {
            load_half(0);
            half_exps(m, pa);
            load_half(1);
            half_exps(m, pb);
          }
          tile_sums();
          if (j > 0 && __any_sync(0xffffffffu, !(ts <= C::kRescaleLimit))) {
            float mx = half_max();  // the second half, still in x
            load_half(0);
            mx = fmaxf(mx, half_max());
            if (!rescale(!(ts <= C::kRescaleLimit), fmaxf(m, mx))) return false;
            zero_sums();
            load_half(0);  // (again: no scores are held across the rescale)
            half_exps(m, pa);
            load_half(1);
            half_exps(m, pb);
            tile_sums();
          }
          l += ts;
          lr += tr;
          // P of keys 0-63 to columns 0-31, of keys 64-127 to columns 32-63
          tmem_st32(sbase, pa);
          tmem_st32(sbase + 32, pb);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars->pfull[b][rb]);
          return true;
        } else {
        float x[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(sbase + c * 32, reinterpret_cast<uint32_t*>(x + c * 32));
        tmem_ld_wait();
        if (nvalid < BN) {  // tail tile: columns past the list do not exist
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= nvalid) x[c] = -INFINITY;
        }
        // Row max of the raw scores (scale > 0 commutes with max), scaled:
        // 3-input maxima in 8 chains.
        auto row_max = [&]() -> float {
          float t8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) t8[i] = fmaxf(x[i], x[8 + i]);
#pragma unroll
          for (int c = 16; c < BN; c += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i) t8[i] = fmax3(t8[i], x[c + i], x[c + 8 + i]);
          return sl * fmax3(fmax3(t8[0], t8[1], t8[2]), fmax3(t8[3], t8[4], t8[5]), fmaxf(t8[6], t8[7]));
        };
        // P = exp2(s*x - mm): a packed two-lane FFMA per pair, then EX2.  The
        // fp32 sum of P gives the log-sum-exp; O is normalised by the sum of
        // the bf16-rounded P that the PV MMA consumes, so that O stays a
        // convex combination of V rows whatever the rounding.
        uint32_t p[BN / 2];
        uint32_t plo[DELTA ? BN / 2 : 1];
        auto exps = [&](float mm, float* sum, float* sum_r) {
          const uint64_t sl2 = f2(sl, sl), nm2 = f2(-mm, -mm);
          // eight partial sums of each kind: short dependency chains
          uint64_t ps[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          float pr[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c = 0; c < BN / 2; ++c) {
            const uint64_t y = fma2(f2(x[2 * c], x[2 * c + 1]), sl2, nm2);
            const float p0 = fast_exp2(f2lo(y)), p1 = fast_exp2(f2hi(y));
            p[c] = pack_bf16(p0, p1);
            if (!DELTA) {
              ps[c & 7] = add2(ps[c & 7], f2(p0, p1));
              pr[c & 7] = add_bf16x2(p[c], pr[c & 7]);
            } else {
              plo[c] = pack_bf16(p0 - __uint_as_float(p[c] << 16), p1 - __uint_as_float(p[c] & 0xFFFF0000u));
            }
          }
          const uint64_t s2 = add2(add2(add2(ps[0], ps[1]), add2(ps[2], ps[3])),
                                   add2(add2(ps[4], ps[5]), add2(ps[6], ps[7])));
          *sum = f2lo(s2) + f2hi(s2);
          *sum_r = ((pr[0] + pr[1]) + (pr[2] + pr[3])) + ((pr[4] + pr[5]) + (pr[6] + pr[7]));
        };
        // The running max m moves only when a tile needs it (lazy rescale);
        // the first tile of a unit sets it to that tile's max.  128-row
        // groups: a later tile's P are computed against the current m, and
        // only when their sum exceeds 2^kRescaleLog2 (so some P might: P >= 0)
        // does the warp take the tile's exact max, raise m to it, rescale and
        // compute P again, so most tiles need no row max at all.  192-row
        // groups (64-key tiles): every tile's max, m raised when it grows by
        // more than kRescaleLog2.  Every P the PV MMA consumes is
        // <= 2^kRescaleLog2.
        float ts = 0.f, tr = 0.f;
        if (!DELTA && (j == 0 || !C::kLazyMax)) {
          const float mx = row_max();
          if (j == 0) {
            m = mx;
          } else if (__any_sync(0xffffffffu, mx > m + C::kRescaleLog2)) {
            if (!rescale(mx > m + C::kRescaleLog2, mx)) return false;
          }
        }
        exps(m, &ts, &tr);
        if (C::kLazyMax && !DELTA && j > 0 && __any_sync(0xffffffffu, !(ts <= C::kRescaleLimit))) {
          const float mx = row_max();
          if (!rescale(!(ts <= C::kRescaleLimit), fmaxf(m, mx))) return false;
          exps(m, &ts, &tr);
        }
        if (!DELTA) {
          l += ts;
          lr += tr;
        }
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) tmem_st32(sbase + c * 32, p + c * 32);
        if (DELTA) {
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) tmem_st32(sbase + BN / 2 + c * 32, plo + c * 32);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->pfull[b][rb]);
        return true;
        }
      };
      for (uint32_t j = 0; j < n; ++j)
        if (!tile(j)) goto done;
      {
        const uint32_t tl = t + n - 1;
        if (!mbar_wait(&bars->pvdone[C::sbuf(tl)][rb], C::sphase(tl), abort)) goto done;
        tc_fence_after();
        const float inv = DELTA ? a.sign : 1.f / lr;
        const uint32_t obase = tmem + lane_base + C::kOCol + rb * D;
        if (!idle) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(obase + c * 32, r);
            tmem_ld_wait();
            if (valid) store_row32(a, orow_off, c * 32, r, inv, DELTA);
          }
        }
        if (!DELTA && valid && a.lse) a.lse[bh * a.Nq + grow] = m * 0.69314718055994531f + __logf(l);
        tc_fence_before();
        mbar_arrive(&bars->ofree[rb]);
      }
      t += n;
      ++un;
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      // a negative scale negates the scores: B (= K) negated inside the MMA
      const uint32_t kIdescS = a.neg_scale ? idesc_negate_b(idesc_bf16(128, BN, false, false))
                                           : idesc_bf16(128, BN, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(128, D, false, true);
      const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
      // Descriptor halves: the high words are constant, the low word holds the
      // start address in 16-byte units (tiles lie below 256 KB of shared memory,
      // so adding to it never carries into the leading-offset field).
      const uint64_t dq = sw128_desc(q_addr, 16, 1024), dk = sw128_desc(k_addr, 16, 1024);
      const uint64_t dv = sw128_desc(v_addr, BN * 128, 1024);
      const uint32_t q_lo = static_cast<uint32_t>(dq), q_hi = static_cast<uint32_t>(dq >> 32);
      const uint32_t k_lo = static_cast<uint32_t>(dk), k_hi = static_cast<uint32_t>(dk >> 32);
      const uint32_t v_lo = static_cast<uint32_t>(dv), v_hi = static_cast<uint32_t>(dv >> 32);
      uint32_t t = 0, un = 0;
      bool ok = true;
      // V tile of tile tt has landed in shared memory.
      auto v_ready = [&](uint32_t tt) -> bool {
        if (!mbar_wait(&bars->vfull[tt % STAGES], (tt / STAGES) & 1, abort)) return false;
        fence_proxy_async_smem();  // V rows were written through the generic proxy
        return true;
      };
      // O += P V of row block rb for tile tt (first: overwrite O).
      auto pv_block = [&](uint32_t tt, int rb, bool first) -> bool {
        const uint32_t s = tt % STAGES, b = C::sbuf(tt);
        if (!mbar_wait(&bars->pfull[b][rb], C::sphase(tt), abort)) return false;
        if (first && un > 0 && !mbar_wait(&bars->ofree[rb], (un - 1) & 1, abort)) return false;
        tc_fence_after();
        const uint32_t a_tmem = tmem + b * C::kSCols + rb * BN;
        const uint32_t d_tmem = tmem + C::kOCol + rb * D;
        const uint32_t vs_lo = v_lo + ((s * C::kTile) >> 4);
        // P of keys 16kk..16kk+15: columns 8kk.. of the S buffer; the delta's
        // remainder in the second half of the buffer, or, for half tiles, each
        // 64-key half's P hi then remainder in that half's columns
        auto p_col = [&](int kk, bool rem) -> uint32_t {
          if (C::kHalves && DELTA) return (kk >> 2) * (BN / 2) + (rem ? BN / 4 : 0) + (kk & 3) * 8;
          return (rem ? BN / 2 : 0) + kk * 8;
        };
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts_w(d_tmem, a_tmem + p_col(kk, false), vs_lo + ((kk * 2048) >> 4), v_hi, kIdescPV,
                   (!first || kk > 0) ? 1u : 0u);
        if (DELTA) {  // the remainder of P
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts_w(d_tmem, a_tmem + p_col(kk, true), vs_lo + ((kk * 2048) >> 4), v_hi, kIdescPV, 1u);
        }
        mma_commit(&bars->pvdone[b][rb]);
        return true;
      };
      // O += P V for tile tt, every row block, then the V stage is free.
      auto pv = [&](uint32_t tt, bool first) -> bool {
        if (!v_ready(tt)) return false;
#pragma unroll
        for (int rb = 0; rb < RB; ++rb)
          if (!pv_block(tt, rb, first)) return false;
        mma_commit(&bars->vempty[tt % STAGES]);
        return true;
      };
      for (uint32_t i = 0; ok; ++i) {
        int64_t u;
        if (!ring_read(bars, i, &u, true, abort)) break;
        if (u < 0) break;
        int64_t begin;
        bool bad;
        const int64_t len = unit_list<DENSE>(a, u, &begin, &bad);
        const uint32_t n = static_cast<uint32_t>((len + BN - 1) / BN);
        if (n == 0) continue;
        if (!mbar_wait(&bars->qfull, un & 1, abort)) break;
        if (C::kQTmem) {
          // Q into TMEM, then the shared-memory copy is free for the next unit.
          tc_fence_after();
#pragma unroll
          for (int rb = 0; rb < RB; ++rb)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tmem_cp_128x256b(tmem + C::kQCol + rb * (D / 2) + kk * 8,
                               q_lo + ((rb * C::kQBlock + (kk >> 2) * 128 * 128 + (kk & 3) * 32) >> 4), q_hi);
          mma_commit(&bars->qempty);
        }
        for (uint32_t j = 0; j < n && ok; ++j) {
          const uint32_t tt = t + j, s = tt % STAGES, b = C::sbuf(tt);
          if (!mbar_wait(&bars->kfull[s], (tt / STAGES) & 1, abort)) { ok = false; break; }
          fence_proxy_async_smem();  // K rows were written through the generic proxy
          tc_fence_after();
          // one S buffer per block: PV(j-1) of a block goes before its QK(j)
          const bool interleave = C::kSBufs == 1 && j >= 1;
          if (interleave && !v_ready(tt - 1)) { ok = false; break; }
          const uint32_t ks_lo = k_lo + ((s * C::kTile) >> 4);
#pragma unroll
          for (int rb = 0; rb < RB; ++rb) {
            if (interleave && !pv_block(tt - 1, rb, j == 1)) { ok = false; break; }
            const uint32_t d_tmem = tmem + b * C::kSCols + rb * BN;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t kb_lo = ks_lo + (((kk >> 2) * BN * 128 + (kk & 3) * 32) >> 4);
              if (C::kQTmem)
                mma_ts_w(d_tmem, tmem + C::kQCol + rb * (D / 2) + kk * 8, kb_lo, k_hi, kIdescS,
                         kk > 0 ? 1u : 0u);
              else
                mma_ss_w(d_tmem, q_lo + ((rb * C::kQBlock + (kk >> 2) * 128 * 128 + (kk & 3) * 32) >> 4),
                         q_hi, kb_lo, k_hi, kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bars->sfull[b][rb]);
          }
          if (!ok) break;
          if (interleave) mma_commit(&bars->vempty[(tt - 1) % STAGES]);
          mma_commit(&bars->kempty[s]);
          if (!C::kQTmem && j == n - 1) mma_commit(&bars->qempty);
          if (C::kSBufs == 2 && j >= 1 && !pv(tt - 1, j == 1)) ok = false;
        }
        if (ok && !pv(t + n - 1, n == 1)) ok = false;
        t += n;
        ++un;
      }
      // Every MMA issued above must finish before TMEM is released.
      mma_commit(&bars->drain);
      const long long t0 = clock64();
      while (!mbar_test(&bars->drain, 0) && clock64() - t0 < kWaitLimitCycles) {
      }
    }
  } else {
    // ------------------------------------------------------------ gather
    // Thread pt copies 16-byte chunks (pt mod 8) + 8c of tile rows pt/8, +28, ...
    // Copies never block the gather warps: each stage's "full" barrier is
    // completed by the copies themselves (cp.async.mbarrier.arrive.noinc).
    // The next tile's indices are loaded while this tile's copies are issued
    // and are not inspected before their own tile, so their latency hides
    // behind a whole tile of work.
    const int pt = threadIdx.x - C::kProdWarp0 * 32;
    const int sub = pt % C::kLanesPerRow;
    const int row0 = pt / C::kLanesPerRow;
    // Shared-memory offset of chunk `sub` of this thread's i-th row (the
    // chunks sub + 8c lie c column blocks further on).  The row step is 4
    // modulo 8, so the swizzle takes two values: two registers, not one per row.
    static_assert(C::kRowStep % 8 == 4, "row step");
    const uint32_t off_even = sw128_offset(row0, sub, BN), off_odd = sw128_offset(row0 + 4, sub, BN) - 512;
    auto dst_off = [&](int i) -> uint32_t {
      return static_cast<uint32_t>(i * C::kRowStep * 128) + ((i & 1) ? off_odd : off_even);
    };
    const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
    uint32_t t = 0, un = 0;
    bool bad_index = false;
    // Three index buffers in rotation: tile j's K copies read buffer j mod 3,
    // its V copies (one step later) the same buffer, and tile j+1's indices
    // load into buffer (j+1) mod 3 a whole step before they are first used.
    int ia[C::kKVRowsPerThread], ib[C::kKVRowsPerThread], ic[C::kKVRowsPerThread];
#pragma unroll
    for (int i = 0; i < C::kKVRowsPerThread; ++i) ia[i] = ib[i] = ic[i] = 0;
    // the unit drawn for the ring slot after next (pt 0 only): the counter's
    // answer is first needed a whole unit after the draw is issued
    int64_t drawn = -1;
    if (pt == 0) {
      bars->ring_u[0] = draw_unit(a, 0);
      mbar_arrive(&bars->ring_full[0]);
      if (bars->ring_u[0] >= 0) drawn = draw_unit(a, 1);
    }
    for (uint32_t i = 0;; ++i) {
      int64_t u;
      if (!ring_read(bars, i, &u, lane == 0, abort)) goto done;
      if (u < 0) break;
      if (pt == 0) {
        // slot i + 1 takes the unit drawn during unit i - 1, once every role
        // has read its previous unit (i - 1)
        const uint32_t f = i + 1, s = f % kRing;
        if (f >= kRing && !mbar_wait(&bars->ring_empty[s], ((f / kRing) - 1) & 1, abort)) goto done;
        bars->ring_u[s] = drawn;
        mbar_arrive(&bars->ring_full[s]);
        if (drawn >= 0) drawn = draw_unit(a, f + 1);
      }
      int64_t begin;
      bool bad;
      const int64_t len = unit_list<DENSE>(a, u, &begin, &bad);
      const uint32_t n = static_cast<uint32_t>((len + BN - 1) / BN);
      if (n == 0) continue;
      const int64_t bh = u / G, g = u % G;
      const uint16_t* kh = a.k + bh * a.Nk * D + sub * 8;
      const uint16_t* vh = a.v + bh * a.Nk * D + sub * 8;
      auto load_indices = [&](uint32_t jj, int* dst) {
#pragma unroll
        for (int i = 0; i < C::kKVRowsPerThread; ++i) {
          const int r = row0 + i * C::kRowStep;
          const int64_t pos = int64_t(jj) * BN + r;
          if (r < BN && pos < len) dst[i] = DENSE ? static_cast<int>(pos) : __ldg(a.col_idx + begin + pos);
        }
      };
      // Issue one tile's copies: rows past the list, and flagged indices
      // outside [0, Nk), are zero-filled.
      auto issue = [&](uint32_t jj, const int* idx, uint32_t dst_base, const uint16_t* src_head,
                       const uint16_t* any) {
        const int64_t rem = len - int64_t(jj) * BN;  // list rows from this tile on
        const int lim = rem < BN ? static_cast<int>(rem) : BN;
#pragma unroll
        for (int i = 0; i < C::kKVRowsPerThread; ++i) {
          const int r = row0 + i * C::kRowStep;
          if (r >= BN) break;
          const bool in_list = r < lim;
          const bool ok = in_list && static_cast<uint32_t>(idx[i]) < static_cast<uint32_t>(a.Nk);
          bad_index |= in_list && !ok;
          const uint16_t* src = ok ? src_head + int64_t(idx[i]) * D : any;
          const uint32_t dst = dst_base + dst_off(i);
#pragma unroll
          for (int c = 0; c < C::kChunksPerLane; ++c)
            cp_async16(dst + c * BN * 128, src + 64 * c, ok ? 16u : 0u);
        }
      };
      load_indices(0, ia);
      if (pt == 0) {
        // query rows g*M .. g*M + 128*RB - 1 of this head (rows past the
        // group feed only rows that are never written; past the tensor: zeros)
        if (un > 0 && !mbar_wait(&bars->qempty, (un - 1) & 1, abort)) goto done;
        mbar_expect_tx(&bars->qfull, C::kQBytes);
#pragma unroll
        for (int rb = 0; rb < RB; ++rb)
#pragma unroll
          for (int cb = 0; cb < D / 64; ++cb)
            tma_load_2d(q_addr + rb * C::kQBlock + cb * 128 * 128, &tmq, 64 * cb,
                        static_cast<int>(bh * a.Nq + g * a.M + rb * 128), &bars->qfull);
      }
      auto step = [&](uint32_t j, const int* kb, const int* vb, int* nb) -> bool {
        const uint32_t tt = t + j;
        if (j < n) {
          if (j + 1 < n) load_indices(j + 1, nb);
          const uint32_t s = tt % STAGES;
          if (!mbar_wait(&bars->kempty[s], ((tt / STAGES) & 1) ^ 1, abort)) return false;
          issue(j, kb, k_addr + s * C::kTile, kh, a.k);
          cp_async_arrive_noinc(&bars->kfull[s]);
        }
        if (j >= 1) {
          const uint32_t tp = tt - 1, s = tp % STAGES;
          if (!mbar_wait(&bars->vempty[s], ((tp / STAGES) & 1) ^ 1, abort)) return false;
          issue(j - 1, vb, v_addr + s * C::kTile, vh, a.v);
          cp_async_arrive_noinc(&bars->vfull[s]);
        }
        return true;
      };
      bool ok = true;
      for (uint32_t j = 0; j <= n && ok; j += 3) {
        ok = step(j, ia, ic, ib);
        if (ok && j + 1 <= n) ok = step(j + 1, ib, ia, ic);
        if (ok && j + 2 <= n) ok = step(j + 2, ic, ib, ia);
      }
      if (!ok) goto done;
      t += n;
      ++un;
    }
    cp_async_wait<0>();
    if (bad_index) report(a.status, SA_DEVERR_INDEX);
  }
done:
  if (warp >= C::kProdWarp0) cp_async_wait<0>();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && bars->abort) report(a.status, SA_DEVERR_TIMEOUT);
  if (warp == C::kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int RB, int BN, int STAGES, bool DELTA>
static cudaError_t launch(const FwdArgs& a, const CUtensorMap& tmq, int num_sms,
                          cudaStream_t stream) {
  using C = FwdCfg<D, RB, BN, STAGES>;
  auto kern = a.dense ? sa_forward_kernel<D, RB, BN, STAGES, DELTA, true>
                      : sa_forward_kernel<D, RB, BN, STAGES, DELTA, false>;
  // At least half the SM's shared memory, so that one CTA owns each SM's TMEM.
  const int smem = C::kSmemBytes > 120 * 1024 ? C::kSmemBytes : 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (C::kRegSplit) {
    // setmaxnreg.inc waits until the block's launch registers cover the new
    // split; the compiler may launch with fewer than the maximum, so check
    // the compiled count before any launch (never a block that could wait
    // forever)
    static std::atomic<int> regs_ok{0};  // 0 unknown, 1 enough, 2 too few (per instantiation)
    if (regs_ok.load() == 0) {
      cudaFuncAttributes attr;
      if ((e = cudaFuncGetAttributes(&attr, kern)) != cudaSuccess) return e;
      const long need = long(C::kRegSoftmax) * 4 * 32 + long(C::kRegOther) * (C::kThreads - 4 * 32);
      regs_ok.store(long(attr.numRegs) * C::kThreads >= need ? 1 : 2);
    }
    if (regs_ok.load() != 1) return cudaErrorLaunchOutOfResources;
  }
  const int64_t grid = a.units < num_sms ? a.units : num_sms;
  kern<<<static_cast<unsigned>(grid), C::kThreads, smem, stream>>>(a, tmq);
  return cudaGetLastError();
}

// Unit counters of the dynamic schedule.  Each launch takes the next slot and
// clears it on its own stream just before the kernel, so launches in flight
// at the same time count in different slots (as long as fewer than
// kSchedSlots are in flight at once).
constexpr int kSchedSlots = 256;
__device__ uint32_t g_sched[kSchedSlots];
std::atomic<uint32_t> g_sched_next{0};

template <bool DELTA>
static cudaError_t launch_any(FwdArgs a, int d, int num_sms, cudaStream_t stream) {
  if (a.units <= 0) return cudaSuccess;
  if (a.units > num_sms) {  // more units than CTAs: draw them dynamically
    void* base = nullptr;
    if (symbol_address(g_sched, 1, &base) != SA_OK) return cudaErrorInvalidSymbol;
    a.sched = static_cast<uint32_t*>(base) + g_sched_next.fetch_add(1) % kSchedSlots;
    cudaError_t e = cudaMemsetAsync(a.sched, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return e;
  }
  const int64_t bh = a.units / a.G;
  CUtensorMap tmq;
  if (!make_rows_map(&tmq, a.q, uint64_t(bh) * a.Nq, d, 128)) return cudaErrorInvalidValue;
  // groups of more than 128 rows: 128-key tiles in halves (Q then stays in
  // shared memory: two S blocks and two O blocks fill TMEM)
  if (d == 128) {
    return a.M <= 128 ? launch<128, 1, 128, 3, DELTA>(a, tmq, num_sms, stream)
                      : launch<128, 2, 128, 2, DELTA>(a, tmq, num_sms, stream);
  }
  return a.M <= 128 ? launch<64, 1, 128, 4, DELTA>(a, tmq, num_sms, stream)
                    : launch<64, 2, 128, 4, DELTA>(a, tmq, num_sms, stream);
}

cudaError_t launch_forward(const FwdArgs& a, int d, int num_sms, cudaStream_t stream) {
  return launch_any<false>(a, d, num_sms, stream);
}

cudaError_t launch_forward_delta(const FwdArgs& a, int d, int num_sms, cudaStream_t stream) {
  return launch_any<true>(a, d, num_sms, stream);
}

}  // namespace sa
