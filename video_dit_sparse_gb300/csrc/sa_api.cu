// sa_api.cu — the C ABI (include/sparse_attn.h): argument checks, buffer
// extent checks, workspace sizing, launch and status mapping.
#include <cuda.h>
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "sa_internal.h"
#include "sparse_attn.h"

namespace {

constexpr int32_t kVersion = 1 * 10000 + 1 * 100 + 0;
constexpr int kMaxDevices = 64;

std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_ok[kMaxDevices];  // 0 unknown, 1 sm_103, 2 other

using AddrRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);
std::atomic<AddrRangeFn> g_addr_range{nullptr};

}  // namespace

namespace sa {

sa_status check_problem(const sa_problem* p, Dims* dims) {
  if (!p) return SA_ERR_INVALID_ARG;
  if (p->B < 1 || p->H < 1 || p->Nq < 1 || p->Nk < 1 || p->d < 1 || p->group_size < 1)
    return SA_ERR_INVALID_ARG;
  if (!std::isfinite(p->scale) || p->scale == 0.f) return SA_ERR_INVALID_ARG;
  if (p->d != 64 && p->d != 128) return SA_ERR_UNSUPPORTED;
  if (p->group_size > 256) return SA_ERR_UNSUPPORTED;
  if (p->out_dtype != SA_OUT_BF16 && p->out_dtype != SA_OUT_FP32) return SA_ERR_INVALID_ARG;
  dims->G = (int64_t(p->Nq) + p->group_size - 1) / p->group_size;
  dims->rows = int64_t(p->B) * p->H * dims->G;
  if (dims->rows >= (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;  // grid.x of the per-row kernels
  // TMA row coordinates are 32-bit: all query rows and all key rows of the batch
  const int64_t bh = int64_t(p->B) * p->H;
  if (bh * p->Nq >= (int64_t(1) << 31) || bh * p->Nk >= (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;
  return SA_OK;
}

sa_status check_select(const sa_problem* p, const sa_select* sel, int32_t stat) {
  if (!sel || sel->mode < SA_SELECT_TOPK || sel->mode > SA_SELECT_MASS) return SA_ERR_INVALID_ARG;
  if (sel->mode == SA_SELECT_TOPK && sel->topk < 1) return SA_ERR_INVALID_ARG;
  if (sel->mode == SA_SELECT_THRESHOLD) {
    // a probability for the mean-query rule and the column maximum; a column
    // sum can reach the group's row count
    const double tmax = stat == 1 ? double(p->group_size) : 1.0;
    if (!(sel->threshold >= 0.0 && sel->threshold <= tmax)) return SA_ERR_INVALID_ARG;
  }
  if (sel->mode == SA_SELECT_MASS && !(sel->mass > 0.0 && sel->mass <= 1.0)) return SA_ERR_INVALID_ARG;
  return SA_OK;
}

sa_status device_info(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SA_ERR_UNSUPPORTED;
  int ok = g_ok[dev].load();
  if (ok == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaFree(nullptr) != cudaSuccess ||  // makes a context current (the primary one if none is)
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SA_ERR_CUDA;
    g_sms[dev].store(sms);
    ok = (major == 10 && minor == 3) ? 1 : 2;
    g_ok[dev].store(ok);
  }
  if (ok != 1) return SA_ERR_UNSUPPORTED;
  *num_sms = g_sms[dev].load();
  if (!g_addr_range.load()) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return SA_ERR_CUDA;
    g_addr_range.store(reinterpret_cast<AddrRangeFn>(fn));
  }
  return SA_OK;
}

// Catches host pointers, freed memory and buffers too small for the stated
// shape before any kernel could touch them.  device_info() resolves the
// query first.
bool in_device_allocation(const void* p, uint64_t bytes) {
  if (!p) return false;
  const AddrRangeFn fn = g_addr_range.load();
  if (!fn) return false;
  CUdeviceptr base = 0;
  size_t size = 0;
  const CUdeviceptr dp = reinterpret_cast<CUdeviceptr>(p);
  if (fn(&base, &size, dp) != CUDA_SUCCESS) return false;
  return dp >= base && bytes <= size && dp - base <= size - bytes;
}

// Per device and symbol: the context whose instance of the symbol `addr`
// points into.  Every CUDA context holds its own copy of a __device__
// variable, so a call from another context looks the address up again.
namespace {
constexpr int kMaxSymbols = 4;
struct SymbolSlot {
  CUcontext ctx = nullptr;
  void* addr = nullptr;
};
std::mutex g_sym_mu;
SymbolSlot g_sym[kMaxDevices][kMaxSymbols];
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn g_ctx_current = nullptr;  // guarded by g_sym_mu
}  // namespace

sa_status symbol_address(const void* symbol, int id, void** addr) {
  int dev = 0;
  if (id < 0 || id >= kMaxSymbols) return SA_ERR_INVALID_ARG;
  if (cudaGetDevice(&dev) != cudaSuccess) return SA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_sym_mu);
  if (!g_ctx_current) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return SA_ERR_CUDA;
    g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return SA_ERR_CUDA;
  SymbolSlot& s = g_sym[dev][id];
  if (s.ctx != ctx || !s.addr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || !p) return SA_ERR_CUDA;
    s.ctx = ctx;
    s.addr = p;
  }
  *addr = s.addr;
  return SA_OK;
}

NvtxRange::NvtxRange(const char* name) { nvtxRangePushA(name); }
NvtxRange::~NvtxRange() { nvtxRangePop(); }

sa_status prepare_build(const sa_problem* p, const sa_select* sel, int32_t stat, const void* q,
                        const void* k, const float* lse, int64_t* row_ptr, int32_t* col_idx,
                        int64_t col_capacity, int64_t* nnz_out_host, size_t scratch_bytes,
                        sa_status scratch_short, BuildArgs* a, int* num_sms) {
  Dims dims;
  sa_status st = check_problem(p, &dims);
  if (st != SA_OK) return st;
  if ((st = check_select(p, sel, stat)) != SA_OK) return st;
  if (!q || !k || !row_ptr || col_capacity < 0) return SA_ERR_INVALID_ARG;
  if (stat >= 0 && (!lse || !aligned(lse, 4))) return SA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(row_ptr, 8) || (col_idx && !aligned(col_idx, 4)))
    return SA_ERR_INVALID_ARG;
  const BuildLayout L = build_layout(dims.rows, p->Nk, p->d);
  if (scratch_bytes < L.total) return scratch_short;
  const int64_t max_nnz = dims.rows * p->Nk;
  if (sel->mode == SA_SELECT_TOPK) {
    const int64_t kk = sel->topk < p->Nk ? sel->topk : p->Nk;
    if (dims.rows * kk > col_capacity) {
      if (nnz_out_host) *nnz_out_host = dims.rows * kk;
      return SA_ERR_CAPACITY;
    }
  } else if (col_capacity < max_nnz && !nnz_out_host) {
    return SA_ERR_INVALID_ARG;  // data-dependent nnz needs the synchronous report
  }
  if (col_capacity > 0 && !col_idx) return SA_ERR_INVALID_ARG;
  if ((st = device_info(num_sms)) != SA_OK) return st;
  const uint64_t qbytes = uint64_t(p->B) * p->H * p->Nq * p->d * 2;
  const uint64_t kbytes = uint64_t(p->B) * p->H * p->Nk * p->d * 2;
  if (!in_device_allocation(q, qbytes) || !in_device_allocation(k, kbytes) ||
      !in_device_allocation(row_ptr, uint64_t(dims.rows + 1) * 8) ||
      (stat >= 0 && !in_device_allocation(lse, uint64_t(p->B) * p->H * p->Nq * 4)) ||
      (col_capacity > 0 && !in_device_allocation(col_idx, uint64_t(col_capacity) * 4)))
    return SA_ERR_INVALID_ARG;
  a->q = static_cast<const uint16_t*>(q);
  a->k = static_cast<const uint16_t*>(k);
  a->lse = lse;
  a->stat = stat;
  a->row_ptr = row_ptr;
  a->col_idx = col_idx;
  a->col_capacity = col_capacity;
  a->ws = nullptr;
  a->L = L;
  a->rows = dims.rows;
  a->G = dims.G;
  a->BH = p->B * p->H;
  a->Nq = p->Nq;
  a->Nk = p->Nk;
  a->d = p->d;
  a->M = p->group_size;
  a->scale = p->scale;
  a->mode = sel->mode;
  a->topk = sel->topk;
  a->threshold = sel->threshold;
  a->mass = sel->mass;
  return SA_OK;
}

sa_status run_build(const BuildArgs& a, int num_sms, int64_t* nnz_out_host, cudaStream_t s) {
  NvtxRange range("sparse_attn_build_index");
  if (launch_build_index(a, num_sms, s) != cudaSuccess) return SA_ERR_CUDA;
  if (nnz_out_host) {
    int64_t misc[2] = {0, 0};
    if (cudaMemcpyAsync(misc, a.ws + a.L.misc, sizeof misc, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return SA_ERR_CUDA;
    *nnz_out_host = misc[0];
    const int32_t dev_status = static_cast<int32_t>(misc[1] & 0xFFFFFFFF);
    if (dev_status & SA_DEVERR_TIMEOUT) return SA_ERR_TIMEOUT;
    if (dev_status & SA_DEVERR_CAPACITY) return SA_ERR_CAPACITY;
  }
  return SA_OK;
}

}  // namespace sa

namespace {

using sa::aligned;
using sa::check_problem;
using sa::device_info;
using sa::Dims;
using sa::in_device_allocation;

sa_status map_cuda(cudaError_t e) { return e == cudaSuccess ? SA_OK : SA_ERR_CUDA; }

}  // namespace

extern "C" {

const char* sparse_attn_status_string(sa_status s) {
  switch (s) {
    case SA_OK: return "ok";
    case SA_ERR_INVALID_ARG: return "invalid argument";
    case SA_ERR_UNSUPPORTED: return "unsupported problem or device";
    case SA_ERR_CAPACITY: return "col_idx capacity too small";
    case SA_ERR_BAD_INDEX: return "malformed index lists";
    case SA_ERR_TIMEOUT: return "device wait timed out";
    case SA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

int32_t sparse_attn_version(void) { return kVersion; }

size_t sparse_attn_build_index_workspace_size(const sa_problem* p) {
  Dims dims;
  if (check_problem(p, &dims) != SA_OK) return 0;
  return sa::build_layout(dims.rows, p->Nk, p->d).total;
}

}  // extern "C"

namespace {

// Shared by the mean-query and the dense-step builders: stat < 0 selects
// the mean-query scores, otherwise the column statistic of p_ij =
// exp(scale q_i.k_j - lse_i) (0 max, 1 sum) with `lse` [B,H,Nq].
sa_status build_common(const sa_problem* p, const sa_select* sel, int32_t stat, const void* q,
                       const void* k, const float* lse, int64_t* row_ptr, int32_t* col_idx,
                       int64_t col_capacity, int64_t* nnz_out_host, void* workspace,
                       size_t workspace_bytes, sa_stream_t stream) {
  if (!workspace || !aligned(workspace, 256)) return SA_ERR_INVALID_ARG;
  sa::BuildArgs a;
  int sms = 0;
  sa_status st = sa::prepare_build(p, sel, stat, q, k, lse, row_ptr, col_idx, col_capacity, nnz_out_host,
                                   workspace_bytes, SA_ERR_INVALID_ARG, &a, &sms);
  if (st != SA_OK) return st;
  if (!in_device_allocation(workspace, a.L.total)) return SA_ERR_INVALID_ARG;
  a.ws = static_cast<uint8_t*>(workspace);
  return sa::run_build(a, sms, nnz_out_host, reinterpret_cast<cudaStream_t>(stream));
}

// Bit-packed (words) or block (blocks, block_k) masks to CSR.
sa_status index_from_mask(const sa_problem* p, const uint32_t* words, const uint8_t* blocks,
                          int32_t block_k, int64_t* row_ptr, int32_t* col_idx, int64_t col_capacity,
                          int64_t* nnz_out_host, sa_stream_t stream) {
  Dims dims;
  sa_status st = check_problem(p, &dims);
  if (st != SA_OK) return st;
  if (!row_ptr || col_capacity < 0 || (col_capacity > 0 && !col_idx)) return SA_ERR_INVALID_ARG;
  if (!aligned(row_ptr, 8) || (col_idx && !aligned(col_idx, 4)) || (words && !aligned(words, 4)))
    return SA_ERR_INVALID_ARG;
  if (blocks && block_k < 1) return SA_ERR_INVALID_ARG;
  if (col_capacity < dims.rows * p->Nk && !nnz_out_host) return SA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_info(&sms)) != SA_OK) return st;
  const int64_t W = words ? (int64_t(p->Nk) + 31) / 32 : (int64_t(p->Nk) + block_k - 1) / block_k;
  const uint64_t mask_bytes = uint64_t(dims.rows) * uint64_t(W) * (words ? 4 : 1);
  if (!in_device_allocation(words ? static_cast<const void*>(words) : static_cast<const void*>(blocks), mask_bytes) ||
      !in_device_allocation(row_ptr, uint64_t(dims.rows + 1) * 8) ||
      (col_capacity > 0 && !in_device_allocation(col_idx, uint64_t(col_capacity) * 4)))
    return SA_ERR_INVALID_ARG;
  sa::FmtArgs a;
  a.words = words;
  a.blocks = blocks;
  a.row_ptr = row_ptr;
  a.col_idx = col_idx;
  a.rows = dims.rows;
  a.capacity = col_capacity;
  a.W = static_cast<int32_t>(W);
  a.Nk = p->Nk;
  a.block_k = words ? 32 : block_k;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  sa::NvtxRange range(words ? "sparse_attn_index_from_bitmask" : "sparse_attn_index_from_block_mask");
  if ((st = map_cuda(sa::launch_index_from_mask(a, sms, s))) != SA_OK) return st;
  if (nnz_out_host) {
    int64_t nnz = 0;
    if (cudaMemcpyAsync(&nnz, row_ptr + dims.rows, 8, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return SA_ERR_CUDA;
    *nnz_out_host = nnz;
    if (nnz > col_capacity) return SA_ERR_CAPACITY;
  }
  return SA_OK;
}

// Argument checks and FwdArgs shared by the forward and the sparse delta.
// row_ptr == col_idx == NULL: every unit keeps all keys (nnz ignored).
sa_status forward_args(const sa_problem* p, const void* q, const void* k, const void* v,
                       const int64_t* row_ptr, const int32_t* col_idx, int64_t nnz, void* o,
                       float* lse, int32_t* dev_status, sa::FwdArgs* a, int* sms) {
  Dims dims;
  sa_status st = check_problem(p, &dims);
  if (st != SA_OK) return st;
  const bool dense = !row_ptr && !col_idx;
  if (!q || !k || !v || !o || (!dense && (!row_ptr || nnz < 0 || (nnz > 0 && !col_idx))))
    return SA_ERR_INVALID_ARG;
  if (dense) nnz = 0;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      (row_ptr && !aligned(row_ptr, 8)) || (col_idx && !aligned(col_idx, 4)) || (lse && !aligned(lse, 4)) ||
      (dev_status && !aligned(dev_status, 4)))
    return SA_ERR_INVALID_ARG;
  if ((st = device_info(sms)) != SA_OK) return st;
  const uint64_t qbytes = uint64_t(p->B) * p->H * p->Nq * p->d * 2;
  const uint64_t kbytes = uint64_t(p->B) * p->H * p->Nk * p->d * 2;
  const uint64_t obytes = p->out_dtype == SA_OUT_FP32 ? 2 * qbytes : qbytes;
  if (!in_device_allocation(q, qbytes) || !in_device_allocation(k, kbytes) ||
      !in_device_allocation(v, kbytes) || !in_device_allocation(o, obytes) ||
      (!dense && !in_device_allocation(row_ptr, uint64_t(dims.rows + 1) * 8)) ||
      (nnz > 0 && !in_device_allocation(col_idx, uint64_t(nnz) * 4)) ||
      (lse && !in_device_allocation(lse, uint64_t(p->B) * p->H * p->Nq * 4)) ||
      (dev_status && !in_device_allocation(dev_status, 4)))
    return SA_ERR_INVALID_ARG;
  a->q = static_cast<const uint16_t*>(q);
  a->k = static_cast<const uint16_t*>(k);
  a->v = static_cast<const uint16_t*>(v);
  a->row_ptr = row_ptr;
  a->col_idx = col_idx;
  a->nnz = nnz;
  a->dense = dense ? 1 : 0;
  a->o = o;
  a->out_fp32 = p->out_dtype == SA_OUT_FP32 ? 1 : 0;
  a->lse = lse;
  a->status = dev_status;
  a->units = dims.rows;
  a->G = dims.G;
  a->Nq = p->Nq;
  a->Nk = p->Nk;
  a->M = p->group_size;
  a->neg_scale = p->scale < 0.f ? 1 : 0;
  a->scale_log2 = static_cast<float>(std::fabs(static_cast<double>(p->scale)) * 1.4426950408889634);
  return SA_OK;
}

}  // namespace

extern "C" {

sa_status sparse_attn_build_index(const sa_problem* p, const sa_select* sel, const void* q,
                                  const void* k, int64_t* row_ptr, int32_t* col_idx,
                                  int64_t col_capacity, int64_t* nnz_out_host, void* workspace,
                                  size_t workspace_bytes, sa_stream_t stream) {
  return build_common(p, sel, -1, q, k, nullptr, row_ptr, col_idx, col_capacity, nnz_out_host,
                      workspace, workspace_bytes, stream);
}

sa_status sparse_attn_build_index_dense(const sa_problem* p, const sa_select* sel, int32_t stat,
                                        const void* q, const void* k, const float* lse,
                                        int64_t* row_ptr, int32_t* col_idx, int64_t col_capacity,
                                        int64_t* nnz_out_host, void* workspace,
                                        size_t workspace_bytes, sa_stream_t stream) {
  if (stat != SA_COLSTAT_MAX && stat != SA_COLSTAT_SUM) return SA_ERR_INVALID_ARG;
  return build_common(p, sel, stat, q, k, lse, row_ptr, col_idx, col_capacity, nnz_out_host,
                      workspace, workspace_bytes, stream);
}

sa_status sparse_attn_forward(const sa_problem* p, const void* q, const void* k, const void* v,
                              const int64_t* row_ptr, const int32_t* col_idx, int64_t nnz,
                              void* o, float* lse, int32_t* dev_status, sa_stream_t stream) {
  sa::FwdArgs a;
  int sms = 0;
  sa_status st = forward_args(p, q, k, v, row_ptr, col_idx, nnz, o, lse, dev_status, &a, &sms);
  if (st != SA_OK) return st;
  sa::NvtxRange range(a.dense ? "sparse_attn_forward (dense)" : "sparse_attn_forward");
  return map_cuda(sa::launch_forward(a, p->d, sms, reinterpret_cast<cudaStream_t>(stream)));
}

sa_status sparse_attn_forward_delta(const sa_problem* p, const void* q, const void* k,
                                    const void* v, const int64_t* row_ptr,
                                    const int32_t* col_idx, int64_t nnz, const float* lse_ref,
                                    const float* base, float sign, void* o, int32_t* dev_status,
                                    sa_stream_t stream) {
  sa::FwdArgs a;
  int sms = 0;
  sa_status st = forward_args(p, q, k, v, row_ptr, col_idx, nnz, o, nullptr, dev_status, &a, &sms);
  if (st != SA_OK) return st;
  if (!lse_ref || !aligned(lse_ref, 4) || !std::isfinite(sign) || (base && !aligned(base, 16)))
    return SA_ERR_INVALID_ARG;
  const uint64_t rows = uint64_t(p->B) * p->H * p->Nq;
  const uint64_t base_bytes = rows * p->d * 4;
  const uint64_t obytes = rows * p->d * (p->out_dtype == SA_OUT_FP32 ? 4 : 2);
  if (!in_device_allocation(lse_ref, rows * 4) || (base && !in_device_allocation(base, base_bytes)))
    return SA_ERR_INVALID_ARG;
  if (base && base != o) {
    // distinct buffers must not overlap (in-place needs o == base, fp32 output)
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(base), o0 = reinterpret_cast<uintptr_t>(o);
    if (b0 < o0 + obytes && o0 < b0 + base_bytes) return SA_ERR_INVALID_ARG;
  }
  if (base && base == o && p->out_dtype != SA_OUT_FP32) return SA_ERR_INVALID_ARG;
  a.lse_ref = lse_ref;
  a.base = base;
  a.sign = sign;
  sa::NvtxRange range("sparse_attn_forward_delta");
  return map_cuda(sa::launch_forward_delta(a, p->d, sms, reinterpret_cast<cudaStream_t>(stream)));
}

sa_status sparse_attn_index_from_bitmask(const sa_problem* p, const uint32_t* mask_words,
                                         int64_t* row_ptr, int32_t* col_idx, int64_t col_capacity,
                                         int64_t* nnz_out_host, sa_stream_t stream) {
  if (!mask_words) return SA_ERR_INVALID_ARG;
  return index_from_mask(p, mask_words, nullptr, 0, row_ptr, col_idx, col_capacity, nnz_out_host, stream);
}

sa_status sparse_attn_index_from_block_mask(const sa_problem* p, int32_t block_k,
                                            const uint8_t* block_mask, int64_t* row_ptr,
                                            int32_t* col_idx, int64_t col_capacity,
                                            int64_t* nnz_out_host, sa_stream_t stream) {
  if (!block_mask) return SA_ERR_INVALID_ARG;
  return index_from_mask(p, nullptr, block_mask, block_k, row_ptr, col_idx, col_capacity, nnz_out_host,
                         stream);
}

sa_status sparse_attn_voxel_permute(const sa_voxel_grid* g, int32_t BH, int32_t d, const void* x,
                                    void* y, int32_t inverse, sa_stream_t stream) {
  if (!g || BH < 1 || !x || !y || (inverse != 0 && inverse != 1)) return SA_ERR_INVALID_ARG;
  if (g->T < 1 || g->Hh < 1 || g->W < 1 || g->vt < 1 || g->vh < 1 || g->vw < 1) return SA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return SA_ERR_UNSUPPORTED;
  const int64_t N = int64_t(g->T) * g->Hh * g->W;
  if (N >= (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(y, 16)) return SA_ERR_INVALID_ARG;
  int sms = 0;
  sa_status st = device_info(&sms);
  if (st != SA_OK) return st;
  const uint64_t bytes = uint64_t(BH) * uint64_t(N) * uint64_t(d) * 2;
  if (!in_device_allocation(x, bytes) || !in_device_allocation(y, bytes)) return SA_ERR_INVALID_ARG;
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), y0 = reinterpret_cast<uintptr_t>(y);
  if (x0 < y0 + bytes && y0 < x0 + bytes) return SA_ERR_INVALID_ARG;  // out of place only
  sa::VoxArgs a;
  a.x = static_cast<const uint4*>(x);
  a.y = static_cast<uint4*>(y);
  a.BH = BH;
  a.N = static_cast<uint32_t>(N);
  a.T = g->T;
  a.Hh = g->Hh;
  a.W = g->W;
  a.vt = g->vt;
  a.vh = g->vh;
  a.vw = g->vw;
  a.pieces = d / 8;
  a.inverse = inverse;
  sa::NvtxRange range("sparse_attn_voxel_permute");
  return map_cuda(sa::launch_voxel_permute(a, sms, reinterpret_cast<cudaStream_t>(stream)));
}

sa_status sparse_attn_kv_window_append(int32_t BH, int32_t d, int32_t chunk_tokens, int32_t slots,
                                       int64_t chunks_before, void* cache_k, void* cache_v,
                                       const void* new_k, const void* new_v,
                                       int64_t* valid_tokens, sa_stream_t stream) {
  if (BH < 1 || chunk_tokens < 1 || slots < 2 || slots > 64 || chunks_before < 0) return SA_ERR_INVALID_ARG;
  if (!cache_k || !cache_v || !new_k || !new_v) return SA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return SA_ERR_UNSUPPORTED;
  if (!aligned(cache_k, 16) || !aligned(cache_v, 16) || !aligned(new_k, 16) || !aligned(new_v, 16))
    return SA_ERR_INVALID_ARG;
  int sms = 0;
  sa_status st = device_info(&sms);
  if (st != SA_OK) return st;
  const uint64_t chunk = uint64_t(BH) * uint64_t(chunk_tokens) * uint64_t(d) * 2;
  const uint64_t cache = chunk * uint64_t(slots);
  if (!in_device_allocation(cache_k, cache) || !in_device_allocation(cache_v, cache) ||
      !in_device_allocation(new_k, chunk) || !in_device_allocation(new_v, chunk))
    return SA_ERR_INVALID_ARG;
  sa::KvArgs a;
  a.ck = static_cast<uint4*>(cache_k);
  a.cv = static_cast<uint4*>(cache_v);
  a.nk = static_cast<const uint4*>(new_k);
  a.nv = static_cast<const uint4*>(new_v);
  a.BH = BH;
  a.L16 = int64_t(chunk_tokens) * d / 8;
  a.S = slots;
  a.slot = chunks_before < slots ? static_cast<int32_t>(chunks_before) : -1;
  sa::NvtxRange range("sparse_attn_kv_window_append");
  if ((st = map_cuda(sa::launch_kv_window(a, sms, reinterpret_cast<cudaStream_t>(stream)))) != SA_OK)
    return st;
  if (valid_tokens) *valid_tokens = int64_t(chunks_before + 1 < slots ? chunks_before + 1 : slots) * chunk_tokens;
  return SA_OK;
}

sa_status sparse_attn_validate_index(const sa_problem* p, const int64_t* row_ptr,
                                     const int32_t* col_idx, int64_t nnz, int32_t* dev_status,
                                     sa_stream_t stream) {
  Dims dims;
  sa_status st = check_problem(p, &dims);
  if (st != SA_OK) return st;
  if (!row_ptr || !dev_status || nnz < 0 || (nnz > 0 && !col_idx)) return SA_ERR_INVALID_ARG;
  if (!aligned(row_ptr, 8) || !aligned(dev_status, 4) || (col_idx && !aligned(col_idx, 4)))
    return SA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_info(&sms)) != SA_OK) return st;
  if (!in_device_allocation(row_ptr, uint64_t(dims.rows + 1) * 8) ||
      (nnz > 0 && !in_device_allocation(col_idx, uint64_t(nnz) * 4)) ||
      !in_device_allocation(dev_status, 4))
    return SA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t flags = 0;
  if (cudaMemsetAsync(dev_status, 0, 4, s) != cudaSuccess) return SA_ERR_CUDA;
  if ((st = map_cuda(sa::launch_validate(row_ptr, col_idx, dims.rows, nnz, p->Nk, dev_status, s))) != SA_OK)
    return st;
  if (cudaMemcpyAsync(&flags, dev_status, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return SA_ERR_CUDA;
  return flags ? SA_ERR_BAD_INDEX : SA_OK;
}

}  // extern "C"
