// sa_format.cu — other index formats into the CSR lists the forward reads.
//
//  * Bit-packed keep-masks (Chipmunk review, "Bitpacked Sparsity Masks": one
//    bit per mask entry instead of a byte): per index row ceil(Nk/32) uint32
//    words, key j is bit j % 32 of word j / 32; bits past Nk are ignored.
//  * Block-sparse masks (FG-Attn review, "The pith" and Fig. 6: masks of
//    block-sparse methods feed the slice kernel directly): one byte per
//    (query group, block of block_k keys), non-zero = every key of the block
//    kept (the last block may be short).
//
// Three launches each: per-row counts written to row_ptr[1..rows], an
// in-place prefix sum (row_ptr[0] = 0), and the emission of ascending indices
// (one warp per row).  Rows whose lists would pass col_capacity are not
// written.
#include "sa_device.cuh"
#include "sa_internal.h"

namespace sa {

__device__ __forceinline__ uint32_t tail_mask(int32_t Nk, int32_t w) {
  const int32_t rem = Nk - w * 32;  // keys in word w
  return rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int warp_excl_scan(int v, int* total) {
  const int lane = threadIdx.x & 31;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  *total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

// row_ptr[r+1] = number of kept keys of row r
__global__ void __launch_bounds__(256) sa_fmt_count_kernel(const FmtArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < a.rows; r += nwarps) {
    int n = 0;
    if (a.words) {
      const uint32_t* row = a.words + r * a.W;
      for (int w = lane; w < a.W; w += 32) n += __popc(__ldg(row + w) & tail_mask(a.Nk, w));
    } else {
      const uint8_t* row = a.blocks + r * a.W;
      for (int b = lane; b < a.W; b += 32)
        if (__ldg(row + b)) n += min(a.block_k, a.Nk - b * a.block_k);
    }
    n = warp_sum(n);
    if (lane == 0) a.row_ptr[r + 1] = n;
  }
}

// In place: row_ptr[0] = 0, row_ptr[r+1] = sum of the counts of rows 0..r.
// One block; each thread owns a contiguous run of rows and reads each count
// before it overwrites it.
__global__ void __launch_bounds__(1024) sa_fmt_scan_kernel(int64_t* row_ptr, int64_t rows) {
  __shared__ int64_t part[1024];
  const int64_t per = (rows + blockDim.x - 1) / blockDim.x;
  const int64_t r0 = min64(rows, threadIdx.x * per), r1 = min64(rows, r0 + per);
  int64_t local = 0;
  for (int64_t r = r0; r < r1; ++r) local += row_ptr[r + 1];
  part[threadIdx.x] = local;
  __syncthreads();
  // exclusive prefix of the per-thread sums (a Hillis-Steele pass over 1024)
  for (int o = 1; o < 1024; o <<= 1) {
    const int64_t add = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
    __syncthreads();
    part[threadIdx.x] += add;
    __syncthreads();
  }
  int64_t run = part[threadIdx.x] - local;
  for (int64_t r = r0; r < r1; ++r) {
    run += row_ptr[r + 1];
    row_ptr[r + 1] = run;
  }
  if (threadIdx.x == 0) row_ptr[0] = 0;
}

// One warp per row.  Bit mask: 32 consecutive words per pass, offsets from a
// warp scan of their popcounts; the pass's keys are staged in shared memory
// and leave in coalesced stores.  Block mask: the kept blocks of each pass of
// 32 are taken in order and the whole warp writes each block's key range.
__global__ void __launch_bounds__(256) sa_fmt_emit_kernel(const FmtArgs a) {
  __shared__ int32_t stage_all[8 * 1024];
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < a.rows; r += nwarps) {
    const int64_t end = a.row_ptr[r + 1];
    if (end > a.capacity) continue;  // does not fit: reported by the caller's nnz check
    int64_t pos = a.row_ptr[r];
    if (a.words) {
      int32_t* stage = stage_all + (threadIdx.x >> 5) * 1024;  // 32 words x 32 bits
      const uint32_t* row = a.words + r * a.W;
      for (int w0 = 0; w0 < a.W; w0 += 32) {
        const int w = w0 + lane;
        const uint32_t mine = w < a.W ? (__ldg(row + w) & tail_mask(a.Nk, w)) : 0u;
        int total;
        const int start = warp_excl_scan(__popc(mine), &total);  // word offsets in this pass
        // each lane puts its word's keys at their offsets in the warp's
        // staging buffer, then the warp copies the pass out in order
        uint32_t bits = mine;
        int o = start;
        while (bits) {
          stage[o++] = w * 32 + (__ffs(bits) - 1);
          bits &= bits - 1;
        }
        __syncwarp();
        for (int i = lane; i < total; i += 32) a.col_idx[pos + i] = stage[i];
        __syncwarp();
        pos += total;
      }
    } else {
      const uint8_t* row = a.blocks + r * a.W;
      for (int b0 = 0; b0 < a.W; b0 += 32) {
        const int b = b0 + lane;
        unsigned kept = __ballot_sync(0xffffffffu, b < a.W && __ldg(row + min(b, a.W - 1)) != 0);
        while (kept) {
          const int kb = b0 + __ffs(kept) - 1;
          kept &= kept - 1;
          const int k0 = kb * a.block_k, len = min(a.block_k, a.Nk - k0);
          for (int i = lane; i < len; i += 32) a.col_idx[pos + i] = k0 + i;
          pos += len;
        }
      }
    }
  }
}

cudaError_t launch_index_from_mask(const FmtArgs& a, int num_sms, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  int64_t blocks = (a.rows + 7) / 8;  // 8 warps per block, a warp per row
  const int64_t cap = int64_t(num_sms) * 16;
  blocks = blocks < cap ? blocks : cap;
  sa_fmt_count_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sa_fmt_scan_kernel<<<1, 1024, 0, st>>>(a.row_ptr, a.rows);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  sa_fmt_emit_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
