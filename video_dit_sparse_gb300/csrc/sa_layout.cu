// sa_layout.cu — token-layout kernels on either side of the attention path.
//
//  * Voxel reordering (Chipmunk review, "What carries the argument" / Alg. 1):
//    the tokens of a (T, Hh, W) latent grid are reordered so that every
//    contiguous run of vt*vh*vw tokens is one spatio-temporal voxel; voxels
//    follow raster order over the voxel grid, tokens raster order inside a
//    voxel, and voxels at the far edges are clipped to what remains.  The
//    inverse restores raster order after attention.
//  * Rolling KV window (DiT page, "The Architecture"): the cache keeps S chunk
//    slots in chronological order; slot 0 is the first chunk (the attention
//    sink, never replaced).  A new chunk fills the next free slot; once the
//    window is full the non-sink chunks move one slot towards the sink (the
//    oldest leaves) and the new chunk takes the last slot.
//
// Both move whole rows of d bf16 values and are bound by HBM bandwidth: each
// thread moves 16-byte pieces, a warp covers whole 128-byte lines.
#include "sa_device.cuh"
#include "sa_internal.h"

namespace sa {

// Position of raster token r = (t*Hh + h)*W + w in the voxel-ordered
// sequence.  Earlier voxel slabs along t are full (only the last is clipped),
// as are earlier voxel rows along h inside a slab and earlier voxels along w.
__device__ __forceinline__ uint32_t voxel_pos(uint32_t r, const VoxArgs& a) {
  const uint32_t HW = a.Hh * a.W;
  const uint32_t t = r / HW, rem = r - t * HW, h = rem / a.W, w = rem - h * a.W;
  const uint32_t ta = t / a.vt, ha = h / a.vh, wa = w / a.vw;
  const uint32_t t0 = ta * a.vt, h0 = ha * a.vh, w0 = wa * a.vw;
  const uint32_t st = min(a.vt, a.T - t0), sh = min(a.vh, a.Hh - h0), sw = min(a.vw, a.W - w0);
  const uint32_t base = t0 * HW + ha * st * a.vh * a.W + wa * st * sh * a.vw;
  return base + ((t - t0) * sh + (h - h0)) * sw + (w - w0);
}

// One warp handles 32 consecutive rows of one head at a time: each lane works
// out one row's voxel position, then the warp moves the rows together, every
// row's 16-byte pieces spread over `pieces` consecutive lanes.
__global__ void __launch_bounds__(256) sa_voxel_permute_kernel(const VoxArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t batches_per_head = (int64_t(a.N) + 31) / 32;
  const int64_t batches = a.BH * batches_per_head;
  const int pieces = a.pieces;             // 16-byte pieces per row (d / 8)
  const int rows_per_pass = 32 / pieces;   // rows moved by one warp instruction
  const int sub = lane % pieces, slot = lane / pieces;
  for (int64_t bt = warp; bt < batches; bt += nwarps) {
    const int64_t bh = bt / batches_per_head;
    const uint32_t r0 = static_cast<uint32_t>((bt % batches_per_head) * 32);
    const uint32_t my_r = r0 + lane;
    const uint32_t my_pos = my_r < a.N ? voxel_pos(my_r, a) : 0u;
    const uint4* xh = a.x + bh * int64_t(a.N) * pieces;
    uint4* yh = a.y + bh * int64_t(a.N) * pieces;
    for (int i = 0; i < 32; i += rows_per_pass) {
      const int src_lane = i + slot;
      const uint32_t r = r0 + src_lane;
      const uint32_t pos = __shfl_sync(0xffffffffu, my_pos, src_lane);
      if (r < a.N && slot < rows_per_pass) {
        // forward: y[pos(r)] = x[r]; inverse: y[r] = x[pos(r)]
        const uint32_t from = a.inverse ? pos : r, to = a.inverse ? r : pos;
        yh[int64_t(to) * pieces + sub] = __ldg(xh + int64_t(from) * pieces + sub);
      }
    }
  }
}

// K (blockIdx.y = 0) or V (1): moves the pieces of one chunk position e of
// every slot, so a thread reads slot s+1 before it writes slot s+1 and no
// other thread touches position e.
__global__ void __launch_bounds__(256) sa_kv_window_kernel(const KvArgs a) {
  uint4* c = blockIdx.y == 0 ? a.ck : a.cv;
  const uint4* n = blockIdx.y == 0 ? a.nk : a.nv;
  const int64_t total = a.BH * a.L16;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t bh = i / a.L16, e = i - bh * a.L16;
    uint4* ch = c + bh * a.S * a.L16 + e;
    const uint4 v = __ldg(n + i);
    if (a.slot >= 0) {
      ch[int64_t(a.slot) * a.L16] = v;
    } else {
      for (int s = 1; s + 1 < a.S; ++s) ch[int64_t(s) * a.L16] = ch[int64_t(s + 1) * a.L16];
      ch[int64_t(a.S - 1) * a.L16] = v;
    }
  }
}

cudaError_t launch_voxel_permute(const VoxArgs& a, int num_sms, cudaStream_t st) {
  const int64_t batches = a.BH * ((int64_t(a.N) + 31) / 32);
  int64_t blocks = (batches + 7) / 8;
  const int64_t cap = int64_t(num_sms) * 8;
  blocks = blocks < cap ? blocks : cap;
  if (blocks < 1) return cudaSuccess;
  sa_voxel_permute_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_kv_window(const KvArgs& a, int num_sms, cudaStream_t st) {
  const int64_t total = a.BH * a.L16;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = int64_t(num_sms) * 8;
  blocks = blocks < cap ? blocks : cap;
  if (blocks < 1) return cudaSuccess;
  sa_kv_window_kernel<<<dim3(static_cast<unsigned>(blocks), 2), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
