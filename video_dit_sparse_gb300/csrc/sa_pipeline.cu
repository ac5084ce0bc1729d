// sa_pipeline.cu — one attention layer from host buffers, copies overlapped
// with the computation.
//
// The layer's (batch, head) pairs are independent: each has its own queries,
// keys, values and key lists.  sparse_attn_layer_from_host splits them into
// chunks of consecutive heads and runs three streams: the copy-in stream
// moves chunk c's Q, K, V from pinned host memory to the device, the compute
// stream builds chunk c's lists and runs its forward once they have landed,
// and the copy-out stream returns chunk c's O (and LSE) as soon as its
// forward is done.  While chunk c computes, chunk c+1 is arriving and chunk
// c-1 is leaving.  Every copy is one cudaMemcpyAsync of a contiguous range.
#include <cuda_runtime.h>

#include <cstdint>

#include "sa_internal.h"
#include "sparse_attn.h"

namespace {

struct Events {
  cudaEvent_t e[3 * sa::kMaxPipelineChunks + 2];
  int n = 0;
  ~Events() {
    for (int i = 0; i < n; ++i) cudaEventDestroy(e[i]);
  }
  cudaEvent_t make() {
    if (n >= 3 * sa::kMaxPipelineChunks + 2) return nullptr;
    if (cudaEventCreateWithFlags(&e[n], cudaEventDisableTiming) != cudaSuccess) return nullptr;
    return e[n++];
  }
};

}  // namespace

extern "C" sa_status sparse_attn_layer_from_host(
    const sa_problem* p, const sa_select* sel, const void* q_host, const void* k_host,
    const void* v_host, void* o_host, float* lse_host, void* q_dev, void* k_dev, void* v_dev,
    void* o_dev, float* lse_dev, int64_t* row_ptr, int32_t* col_idx, int64_t col_capacity,
    void* workspace, size_t workspace_bytes, int32_t heads_per_chunk, sa_stream_t compute,
    sa_stream_t copy_in, sa_stream_t copy_out) {
  if (!p || !sel || !q_host || !k_host || !v_host || !o_host || !q_dev || !k_dev || !v_dev || !o_dev)
    return SA_ERR_INVALID_ARG;
  if ((lse_host != nullptr) != (lse_dev != nullptr)) return SA_ERR_INVALID_ARG;
  // Every check on the whole layer comes before the first copy is enqueued:
  // a short or misaligned staging buffer is an INVALID_ARG with nothing on
  // any stream.
  sa::Dims dims;
  sa_status st0 = sa::check_problem(p, &dims);
  if (st0 != SA_OK) return st0;
  if ((st0 = sa::check_select(p, sel, -1)) != SA_OK) return st0;
  if (!sa::aligned(q_dev, 16) || !sa::aligned(k_dev, 16) || !sa::aligned(v_dev, 16) ||
      !sa::aligned(o_dev, 16) || (lse_dev && !sa::aligned(lse_dev, 4)) || !row_ptr ||
      !sa::aligned(row_ptr, 8) || !col_idx || !sa::aligned(col_idx, 4) || !workspace ||
      !sa::aligned(workspace, 256) || col_capacity < 1)
    return SA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st0 = sa::device_info(&sms)) != SA_OK) return st0;
  {
    const uint64_t qb = uint64_t(p->B) * p->H * p->Nq * p->d * 2;
    const uint64_t kb = uint64_t(p->B) * p->H * p->Nk * p->d * 2;
    const uint64_t ob = p->out_dtype == SA_OUT_FP32 ? 2 * qb : qb;
    if (!sa::in_device_allocation(q_dev, qb) || !sa::in_device_allocation(k_dev, kb) ||
        !sa::in_device_allocation(v_dev, kb) || !sa::in_device_allocation(o_dev, ob) ||
        (lse_dev && !sa::in_device_allocation(lse_dev, uint64_t(p->B) * p->H * p->Nq * 4)) ||
        !sa::in_device_allocation(col_idx, uint64_t(col_capacity) * 4) ||
        !sa::in_device_allocation(workspace, workspace_bytes))
      return SA_ERR_INVALID_ARG;
  }
  const int64_t BH = int64_t(p->B) * p->H;
  // Chunk schedule: only the first chunk's copy in and the last chunk's
  // computation and copy out are not hidden, so with more than two heads the
  // first and the last chunk hold one head each.  The heads between them
  // form chunks of 1, 2, 4, ... heads up to hc (default: the middle split in
  // three), then hc: a chunk's copy in then takes about as long as the
  // computation of the chunk before it (a head's copy is shorter than its
  // computation), so the compute stream does not wait for a large first
  // copy.
  const int64_t mid = BH > 2 ? BH - 2 : 0;
  int64_t hc = heads_per_chunk > 0 ? heads_per_chunk : (mid > 0 ? (mid + 2) / 3 : BH);
  if (hc > BH) hc = BH;
  int64_t starts[sa::kMaxPipelineChunks + 1];
  int64_t nchunks = 0;
  {
    int64_t h = 0, size = mid > 0 ? 1 : hc;
    if (mid > 0) starts[nchunks++] = h++;
    while (h < BH - (mid > 0 ? 1 : 0)) {
      if (nchunks >= sa::kMaxPipelineChunks) return SA_ERR_UNSUPPORTED;
      starts[nchunks++] = h;
      h += size < hc ? size : hc;
      size *= 2;
      if (mid > 0 && h > BH - 1) h = BH - 1;
    }
    if (mid > 0) {
      if (nchunks >= sa::kMaxPipelineChunks) return SA_ERR_UNSUPPORTED;
      starts[nchunks++] = BH - 1;
    }
    starts[nchunks] = BH;
  }
  // each chunk is a problem of hc heads (B = 1) on the same lists, workspace
  // and capacity: the compute stream runs the chunks one after another
  sa_problem cp = *p;
  cp.B = 1;
  cp.H = static_cast<int32_t>(hc);
  const size_t ws_need = sparse_attn_build_index_workspace_size(&cp);
  if (ws_need == 0 || workspace_bytes < ws_need) return SA_ERR_INVALID_ARG;
  const int64_t G = dims.G;
  const int64_t kmax = sel->mode == SA_SELECT_TOPK ? (sel->topk < p->Nk ? sel->topk : p->Nk) : p->Nk;
  if (col_capacity < hc * G * kmax) return SA_ERR_CAPACITY;  // one chunk's lists, without a sync
  if (!sa::in_device_allocation(row_ptr, uint64_t(hc * G + 1) * 8)) return SA_ERR_INVALID_ARG;
  sa::NvtxRange range("sparse_attn_layer_from_host");
  cudaStream_t sc = reinterpret_cast<cudaStream_t>(compute);
  cudaStream_t si = copy_in ? reinterpret_cast<cudaStream_t>(copy_in) : sc;
  cudaStream_t so = copy_out ? reinterpret_cast<cudaStream_t>(copy_out) : sc;
  const size_t qh = size_t(p->Nq) * p->d * 2, kh = size_t(p->Nk) * p->d * 2;
  const size_t oh = size_t(p->Nq) * p->d * (p->out_dtype == SA_OUT_FP32 ? 4 : 2);
  const size_t lh = size_t(p->Nq) * 4;
  Events ev;
  // the copies of this call start after everything an earlier call left on
  // the compute stream (its staging buffers may still be in use there)
  if (si != sc) {
    cudaEvent_t start = ev.make();
    if (!start || cudaEventRecord(start, sc) != cudaSuccess || cudaStreamWaitEvent(si, start, 0) != cudaSuccess)
      return SA_ERR_CUDA;
  }
  for (int64_t c = 0; c < nchunks; ++c) {
    const int64_t h0 = starts[c], nh = starts[c + 1] - h0;
    cp.H = static_cast<int32_t>(nh);
    auto at = [](const void* base, size_t per_head, int64_t h) {
      return static_cast<const uint8_t*>(base) + per_head * size_t(h);
    };
    auto atm = [](void* base, size_t per_head, int64_t h) {
      return static_cast<uint8_t*>(base) + per_head * size_t(h);
    };
    // copy in
    if (cudaMemcpyAsync(atm(q_dev, qh, h0), at(q_host, qh, h0), qh * nh, cudaMemcpyHostToDevice, si) != cudaSuccess ||
        cudaMemcpyAsync(atm(k_dev, kh, h0), at(k_host, kh, h0), kh * nh, cudaMemcpyHostToDevice, si) != cudaSuccess ||
        cudaMemcpyAsync(atm(v_dev, kh, h0), at(v_host, kh, h0), kh * nh, cudaMemcpyHostToDevice, si) != cudaSuccess)
      return SA_ERR_CUDA;
    if (si != sc) {
      cudaEvent_t in = ev.make();
      if (!in || cudaEventRecord(in, si) != cudaSuccess || cudaStreamWaitEvent(sc, in, 0) != cudaSuccess)
        return SA_ERR_CUDA;
    }
    // compute: lists, then the forward (no synchronisation: capacity covers the chunk)
    sa_status st = sparse_attn_build_index(&cp, sel, at(q_dev, qh, h0), at(k_dev, kh, h0), row_ptr, col_idx,
                                           col_capacity, nullptr, workspace, workspace_bytes, compute);
    if (st != SA_OK) return st;
    st = sparse_attn_forward(&cp, at(q_dev, qh, h0), at(k_dev, kh, h0), at(v_dev, kh, h0), row_ptr, col_idx,
                             col_capacity, atm(o_dev, oh, h0),
                             lse_dev ? reinterpret_cast<float*>(atm(lse_dev, lh, h0)) : nullptr, nullptr, compute);
    if (st != SA_OK) return st;
    if (so != sc) {
      cudaEvent_t done = ev.make();
      if (!done || cudaEventRecord(done, sc) != cudaSuccess || cudaStreamWaitEvent(so, done, 0) != cudaSuccess)
        return SA_ERR_CUDA;
    }
    // copy out
    if (cudaMemcpyAsync(atm(o_host, oh, h0), at(o_dev, oh, h0), oh * nh, cudaMemcpyDeviceToHost, so) != cudaSuccess)
      return SA_ERR_CUDA;
    if (lse_dev &&
        cudaMemcpyAsync(atm(lse_host, lh, h0), at(lse_dev, lh, h0), lh * nh, cudaMemcpyDeviceToHost, so) != cudaSuccess)
      return SA_ERR_CUDA;
  }
  // the compute stream waits for the last copy out: synchronising it is enough
  if (so != sc) {
    cudaEvent_t last = ev.make();
    if (!last || cudaEventRecord(last, so) != cudaSuccess || cudaStreamWaitEvent(sc, last, 0) != cudaSuccess)
      return SA_ERR_CUDA;
  }
  return SA_OK;
}
