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
// library's code is loaded holds it until the process exits, and each CUDA
// context on a device has its own instance.  Host code cannot use the
// array's name as a device address, so the first call in each context looks
// the address up with cudaGetSymbolAddress while that context is current and
// caches it together with the context it belongs to; a call from another
// context on the same device looks it up again.  All calls share the array:
// calls that overlap on the GPU (concurrent streams, or several host
// threads) race on it and must be serialised by the caller.  Nothing here
// allocates.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sa_internal.h"
#include "sparse_attn.h"

namespace {

constexpr size_t kScratchBytes = SA_NOALLOC_WORKSPACE_BYTES;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

}  // namespace

extern "C" sa_status sparse_attn_build_index_noalloc(const sa_problem* p, const sa_select* sel,
                                                     const void* q, const void* k,
                                                     int64_t* row_ptr, int32_t* col_idx,
                                                     int64_t col_capacity, int64_t* nnz_out_host,
                                                     sa_stream_t stream) {
  // The argument rules of sparse_attn_build_index; a problem whose scratch
  // does not fit the fixed array is refused before anything is enqueued.
  sa::BuildArgs a;
  int sms = 0;
  sa_status st = sa::prepare_build(p, sel, -1, q, k, nullptr, row_ptr, col_idx, col_capacity,
                                   nnz_out_host, kScratchBytes, SA_ERR_UNSUPPORTED, &a, &sms);
  if (st != SA_OK) return st;
  void* scratch = nullptr;
  if ((st = sa::symbol_address(g_scratch, 0, &scratch)) != SA_OK) return st;
  a.ws = static_cast<uint8_t*>(scratch);
  // launch_build_index clears the counters it accumulates into (nnz, status);
  // every other scratch byte it reads is written earlier in the same call.
  return sa::run_build(a, sms, nnz_out_host, reinterpret_cast<cudaStream_t>(stream));
}
