// sa_noalloc.cu — sparse_attn_build_index_noalloc: the index builder for
// callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory at the point they build
// index lists: code running inside a framework's stream-ordered allocator
// hook or a pre-allocated inference runtime that forbids allocations after
// start-up, plugins of host applications that only hand over tensor
// pointers, and C callers without a CUDA allocator of their own.  For them
// the builder's scratch (mean queries, the fp32 score matrix, per-row
// selection results, counters) lives in one fixed array of
// SA_NOALLOC_WORKSPACE_BYTES that the library owns.
//
// The array is a file-scope __device__ variable: every GPU on which this
// library's code is loaded holds it until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on
// each device looks the address up with cudaGetSymbolAddress while that
// device is current and caches it.  All calls share the array: calls that
// overlap on the GPU (concurrent streams, or several host threads) race on
// it and must be serialised by the caller.  Nothing here allocates.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "sa_internal.h"
#include "sparse_attn.h"

namespace {

constexpr size_t kScratchBytes = SA_NOALLOC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::atomic<void*> g_scratch_addr[kMaxDevices];
std::atomic<int> g_num_sms[kMaxDevices];

using AddrRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);
std::atomic<AddrRangeFn> g_range_fn{nullptr};

// Device address of g_scratch and the SM count of the current device,
// looked up once per device (the first call on a device does this set-up).
sa_status scratch_for_current_device(void** addr, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SA_ERR_UNSUPPORTED;
  void* p = g_scratch_addr[dev].load();
  if (!p) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SA_ERR_CUDA;
    if (major != 10 || minor != 3) return SA_ERR_UNSUPPORTED;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return SA_ERR_CUDA;
    g_num_sms[dev].store(n);
    g_scratch_addr[dev].store(p);
  }
  if (!g_range_fn.load()) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return SA_ERR_CUDA;
    g_range_fn.store(reinterpret_cast<AddrRangeFn>(fn));
  }
  *addr = p;
  *sms = g_num_sms[dev].load();
  return SA_OK;
}

bool inside_allocation(const void* p, uint64_t bytes) {
  if (!p) return false;
  CUdeviceptr base = 0;
  size_t size = 0;
  const CUdeviceptr dp = reinterpret_cast<CUdeviceptr>(p);
  if (g_range_fn.load()(&base, &size, dp) != CUDA_SUCCESS) return false;
  return dp >= base && bytes <= size && dp - base <= size - bytes;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" sa_status sparse_attn_build_index_noalloc(const sa_problem* p, const sa_select* sel,
                                                     const void* q, const void* k,
                                                     int64_t* row_ptr, int32_t* col_idx,
                                                     int64_t col_capacity, int64_t* nnz_out_host,
                                                     sa_stream_t stream) {
  // Same argument rules as sparse_attn_build_index, without a workspace.
  if (!p || p->B < 1 || p->H < 1 || p->Nq < 1 || p->Nk < 1 || p->d < 1 || p->group_size < 1 ||
      !std::isfinite(p->scale) || p->scale == 0.f)
    return SA_ERR_INVALID_ARG;
  if (p->d != 64 && p->d != 128) return SA_ERR_UNSUPPORTED;
  if (p->group_size > 256) return SA_ERR_UNSUPPORTED;
  if (p->out_dtype != SA_OUT_BF16 && p->out_dtype != SA_OUT_FP32) return SA_ERR_INVALID_ARG;
  const int64_t G = (int64_t(p->Nq) + p->group_size - 1) / p->group_size;
  const int64_t rows = int64_t(p->B) * p->H * G;
  if (!sel || sel->mode < SA_SELECT_TOPK || sel->mode > SA_SELECT_MASS) return SA_ERR_INVALID_ARG;
  if (sel->mode == SA_SELECT_TOPK && sel->topk < 1) return SA_ERR_INVALID_ARG;
  if (sel->mode == SA_SELECT_THRESHOLD && !(sel->threshold >= 0.0 && sel->threshold <= 1.0))
    return SA_ERR_INVALID_ARG;
  if (sel->mode == SA_SELECT_MASS && !(sel->mass > 0.0 && sel->mass <= 1.0)) return SA_ERR_INVALID_ARG;
  if (!q || !k || !row_ptr || col_capacity < 0 || (col_capacity > 0 && !col_idx))
    return SA_ERR_INVALID_ARG;
  if (!aligned_to(q, 16) || !aligned_to(k, 16) || !aligned_to(row_ptr, 8) ||
      (col_idx && !aligned_to(col_idx, 4)))
    return SA_ERR_INVALID_ARG;
  // The problem's scratch must fit the fixed array: rejected, nothing launched.
  const sa::BuildLayout L = sa::build_layout(rows, p->Nk, p->d);
  if (L.total > kScratchBytes) return SA_ERR_UNSUPPORTED;
  if (sel->mode == SA_SELECT_TOPK) {
    const int64_t kk = sel->topk < p->Nk ? sel->topk : p->Nk;
    if (rows * kk > col_capacity) {
      if (nnz_out_host) *nnz_out_host = rows * kk;
      return SA_ERR_CAPACITY;
    }
  } else if (col_capacity < rows * p->Nk && !nnz_out_host) {
    return SA_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  int sms = 0;
  sa_status st = scratch_for_current_device(&scratch, &sms);
  if (st != SA_OK) return st;
  const uint64_t qbytes = uint64_t(p->B) * p->H * p->Nq * p->d * 2;
  const uint64_t kbytes = uint64_t(p->B) * p->H * p->Nk * p->d * 2;
  if (!inside_allocation(q, qbytes) || !inside_allocation(k, kbytes) ||
      !inside_allocation(row_ptr, uint64_t(rows + 1) * 8) ||
      (col_capacity > 0 && !inside_allocation(col_idx, uint64_t(col_capacity) * 4)))
    return SA_ERR_INVALID_ARG;

  sa::BuildArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.row_ptr = row_ptr;
  a.col_idx = col_idx;
  a.col_capacity = col_capacity;
  a.ws = static_cast<uint8_t*>(scratch);
  a.L = L;
  a.rows = rows;
  a.G = G;
  a.BH = p->B * p->H;
  a.Nq = p->Nq;
  a.Nk = p->Nk;
  a.d = p->d;
  a.M = p->group_size;
  a.scale = p->scale;
  a.mode = sel->mode;
  a.topk = sel->topk;
  a.threshold = sel->threshold;
  a.mass = sel->mass;
  // launch_build_index clears the counters it accumulates into (nnz, status);
  // every other scratch byte it reads is written earlier in the same call.
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (sa::launch_build_index(a, sms, s) != cudaSuccess) return SA_ERR_CUDA;
  if (nnz_out_host) {
    int64_t misc[2] = {0, 0};
    if (cudaMemcpyAsync(misc, a.ws + L.misc, sizeof misc, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return SA_ERR_CUDA;
    *nnz_out_host = misc[0];
    const int32_t dev_status = static_cast<int32_t>(misc[1] & 0xFFFFFFFF);
    if (dev_status & SA_DEVERR_TIMEOUT) return SA_ERR_TIMEOUT;
    if (dev_status & SA_DEVERR_CAPACITY) return SA_ERR_CAPACITY;
  }
  return SA_OK;
}
