// sa_internal.h — launch interfaces between the C ABI (sa_api.cu) and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sparse_attn.h"

namespace sa {

struct FwdArgs {
  const uint16_t* q;  // bf16 bits [B,H,Nq,d]
  const uint16_t* k;  // bf16 bits [B,H,Nk,d]
  const uint16_t* v;
  const int64_t* row_ptr;
  const int32_t* col_idx;
  int64_t nnz;
  void* o;            // [B,H,Nq,d]: bf16 bits, or fp32 when out_fp32
  float* lse;         // [B,H,Nq] or null
  int32_t* status;    // device status word or null
  int64_t units;      // B*H*G
  int64_t G;
  int32_t Nq, Nk, M;
  int32_t out_fp32;
  int32_t neg_scale;  // scale < 0: the QK MMA negates K, and scale_log2 = |scale| log2(e)
  float scale_log2;   // |scale| * log2(e)
  int32_t dense = 0;  // no lists: every unit keeps keys 0 .. Nk-1
  // unit counter of the launch (zero when it starts), or null: static schedule
  uint32_t* sched = nullptr;
  // sparse delta (launch_forward_delta): o = base + sign * sum_j exp(l_ij - lse_i) v_j
  const float* lse_ref = nullptr;  // [B,H,Nq] natural-log normaliser per query row
  const float* base = nullptr;     // [B,H,Nq,d] fp32 or null (zero)
  float sign = 1.f;
};

cudaError_t launch_forward(const FwdArgs& a, int d, int num_sms, cudaStream_t stream);
cudaError_t launch_forward_delta(const FwdArgs& a, int d, int num_sms, cudaStream_t stream);

// Index builder.  The workspace holds, in order (each 256-byte aligned):
//   qhi, qlo   bf16 [rows, d]   mean query split as hi + lo
//   scores     fp32 [rows, ld]  ld = Nk rounded up to a multiple of 4
//   cut        uint32 [rows]    order-preserving key of the selection cut
//   ties       int32 [rows]     keys equal to the cut that are kept
//   counts     int64 [rows]     kept keys per row
//   misc       int64 nnz, int32 status
//   fail       int32 count (own 256 bytes), int32 [rows] rows, int32 [rows] units:
//              rows the TOPK path without a score matrix leaves to the select
//              kernel, and the (head, 128-row chunk) units whose scores they need
// The TOPK path without a score matrix keeps its sample scores, brackets,
// keep-masks and candidates inside the scores region.
struct BuildLayout {
  size_t qhi, qlo, scores, cut, ties, counts, misc, fail, total;
  int64_t ld;
};
BuildLayout build_layout(int64_t rows, int32_t Nk, int32_t d);

struct BuildArgs {
  const uint16_t* q;
  const uint16_t* k;
  // dense-step lists: stat >= 0 ranks keys by ln max_i / ln sum_i of
  // exp(scale q_i.k_j - lse_i) over the group's rows instead of the mean-query
  // score, and THRESHOLD compares that statistic itself with the threshold
  const float* lse = nullptr;
  int32_t stat = -1;  // -1 mean query, 0 column max, 1 column sum
  int64_t* row_ptr;
  int32_t* col_idx;
  int64_t col_capacity;
  uint8_t* ws;
  BuildLayout L;
  int64_t rows, G;
  int32_t BH, Nq, Nk, d, M;
  float scale;
  int32_t mode;
  int64_t topk;
  double threshold, mass;
};

cudaError_t launch_build_index(const BuildArgs& a, int num_sms, cudaStream_t stream);

// Voxel reordering of [BH, N, d] bf16 rows (N = T*Hh*W < 2^31).
struct VoxArgs {
  const uint4* x;
  uint4* y;
  int64_t BH;
  uint32_t N, T, Hh, W, vt, vh, vw;
  int32_t pieces;   // 16-byte pieces per row: d / 8 (a divisor of 32)
  int32_t inverse;  // 0: raster -> voxel order, 1: back
};
cudaError_t launch_voxel_permute(const VoxArgs& a, int num_sms, cudaStream_t stream);

// Rolling KV window append of one chunk to caches of S slots.
struct KvArgs {
  uint4* ck;
  uint4* cv;
  const uint4* nk;
  const uint4* nv;
  int64_t BH, L16;  // heads; 16-byte pieces per chunk per head
  int32_t S;        // slots (>= 2)
  int32_t slot;     // slot to fill, or -1: roll (sink stays) and fill the last
};
cudaError_t launch_kv_window(const KvArgs& a, int num_sms, cudaStream_t stream);

// Bit-packed (words) or block (blocks) keep-masks to CSR lists.
struct FmtArgs {
  const uint32_t* words;   // [rows, W] or null
  const uint8_t* blocks;   // [rows, W] or null
  int64_t* row_ptr;
  int32_t* col_idx;
  int64_t rows, capacity;
  int32_t W, Nk, block_k;
};
cudaError_t launch_index_from_mask(const FmtArgs& a, int num_sms, cudaStream_t stream);

// sparse_attn_layer_from_host splits a layer into at most this many chunks.
constexpr int kMaxPipelineChunks = 64;

// ------------------------------------------------------------ host checks
// Shared by every entry point (sa_api.cu defines them).
struct Dims {
  int64_t G, rows;
};
// Shapes, scale, head dim, group size, output dtype and the 32-bit limits
// (rows of the per-row kernels, TMA row coordinates).
sa_status check_problem(const sa_problem* p, Dims* dims);
// The selection rule of a builder call; `stat` < 0 for mean-query scores,
// else the column statistic (its THRESHOLD range differs).
sa_status check_select(const sa_problem* p, const sa_select* sel, int32_t stat);
// Checks that the current device is an sm_103 GPU and gives its SM count;
// also resolves the driver's address-range query used by in_device_allocation.
sa_status device_info(int* num_sms);
// [p, p + bytes) lies inside one device allocation of the current context.
bool in_device_allocation(const void* p, uint64_t bytes);
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Every argument rule of a builder call except those on the scratch pointer
// itself: `scratch_bytes` below the problem's workspace size returns
// `scratch_short`.  Fills `a` (a->ws left null) and the SM count.
sa_status prepare_build(const sa_problem* p, const sa_select* sel, int32_t stat, const void* q,
                        const void* k, const float* lse, int64_t* row_ptr, int32_t* col_idx,
                        int64_t col_capacity, int64_t* nnz_out_host, size_t scratch_bytes,
                        sa_status scratch_short, BuildArgs* a, int* num_sms);
// Launches the builder on a.ws; with nnz_out_host, synchronises the stream
// and reports nnz and the device status.
sa_status run_build(const BuildArgs& a, int num_sms, int64_t* nnz_out_host, cudaStream_t s);

// Device address of a __device__ variable (`symbol`, its host-side name) in
// the current context, looked up once per (device, context) and cached under
// `id` (0: the builder's fixed scratch, 1: the forward's unit counters).
sa_status symbol_address(const void* symbol, int id, void** addr);

// A named NVTX range around a host call (shows the entry point's launches
// in a profiler's timeline; costs nothing measurable without one).
struct NvtxRange {
  explicit NvtxRange(const char* name);
  ~NvtxRange();
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

cudaError_t launch_validate(const int64_t* row_ptr, const int32_t* col_idx, int64_t rows,
                            int64_t nnz, int32_t Nk, int32_t* status, cudaStream_t stream);

}  // namespace sa
