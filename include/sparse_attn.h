/*
 * sparse_attn.h — C ABI of the column-sparse (Mx1-slice) attention library
 * (libsparse_attn.so, hand-written CUDA kernels for sm_103a / GB300).
 *
 * The operation, as the video-DiT pages state it:
 *  - FG-Attn review (arXiv 2509.16518), "The pith" and "What carries the
 *    argument": attention scores are skipped per Mx1 slice — M contiguous
 *    queries against one key — so each group of M queries keeps its own list
 *    of key indices, and only those K/V rows are gathered into dense tiles.
 *  - Chipmunk review (arXiv 2506.03275), "What carries the argument": the
 *    same idea with [C,1] column chunks, C = 192 voxel-ordered tokens; major
 *    comment 1 / Alg. 3: the softmax is renormalised over the selected keys
 *    only (restricted softmax).
 *  - FG-Attn review, referee comment 2 (§4.4): the list is built without
 *    training by scoring every key with the group's average query,
 *    k . q_avg / sqrt(D); LoSA abstract (mlsift.com list): or by keeping the
 *    smallest key set that retains 99 % of the attention mass.
 *  - DiT page (woonyee.org), "Self Attention" and "Online Softmax":
 *    O = softmax(Q K^T / sqrt(d)) V per head, computed tile by tile with a
 *    running max, running sum and running output.
 *  - FG-Attn review, cached mask (free parameters; Fig. 10): at a dense step
 *    a slice is kept when one of its full-attention scores reaches
 *    tau_cached = 0.5/N, and the mask is reused by later steps.  Chipmunk
 *    review, major comment 2 / Alg. 4: top-k columns by the column sums of
 *    the attention probabilities; Eq. 1 with Appendix B.2: the sparse delta
 *    reuses the normalisation constants of an earlier step.
 *
 * Conventions shared by every entry point
 *  - Tensors are row-major [B, H, N, d] with d contiguous (BHND), bf16.
 *  - Query group g of a head covers query rows [g*M, min((g+1)*M, Nq));
 *    G = ceil(Nq / M) groups per head; "rows" of an index are the
 *    B*H*G (batch, head, group) units in that order.
 *  - Index lists are CSR: row_ptr int64 [B*H*G + 1], col_idx int32 [nnz];
 *    the keys of unit u are col_idx[row_ptr[u] .. row_ptr[u+1]).
 *  - Every pointer argument marked "device" must be a CUDA device (or
 *    managed) address on the current device; the caller owns all memory.
 *    q, k, v, o and the workspace must be 16-byte aligned; row_ptr 8-byte;
 *    col_idx and lse 4-byte.
 *  - All work is enqueued on `stream` (NULL = legacy default stream) and is
 *    asynchronous unless a function says it synchronises.  Argument errors
 *    are returned before anything is enqueued.
 *  - No function allocates device memory, and none falls back to the CPU.
 *  - Supported: d in {64, 128}; 1 <= M <= 256; 1 <= Nq, Nk < 2^31.
 */
#ifndef SPARSE_ATTN_H
#define SPARSE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st* sa_stream_t;

typedef enum {
  SA_OK = 0,
  SA_ERR_INVALID_ARG = 1,  /* bad pointer, alignment, shape or mode */
  SA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. d = 96) or no sm_103a device */
  SA_ERR_CAPACITY = 3,     /* col_capacity smaller than the lists need */
  SA_ERR_BAD_INDEX = 4,    /* index lists malformed (see sparse_attn_validate_index) */
  SA_ERR_TIMEOUT = 5,      /* a device-side wait gave up; outputs are incomplete */
  SA_ERR_CUDA = 6          /* a CUDA runtime call or launch failed */
} sa_status;

/* Bits a kernel ORs into the optional device status word (int32). */
#define SA_DEVERR_ROW_PTR 1   /* row_ptr not monotone / out of [0, nnz] */
#define SA_DEVERR_INDEX 2     /* a key index outside [0, Nk) or lists not ascending */
#define SA_DEVERR_TIMEOUT 4   /* a bounded wait ran out */
#define SA_DEVERR_CAPACITY 8  /* the builder's lists did not fit col_capacity */

typedef enum {
  SA_SELECT_TOPK = 0,       /* keep the topk highest-scoring keys */
  SA_SELECT_THRESHOLD = 1,  /* keep keys whose mean-query probability >= threshold */
  SA_SELECT_MASS = 2        /* keep the fewest top keys whose probability sum >= mass */
} sa_select_mode;

/* Column statistic of the dense-step builder (sparse_attn_build_index_dense). */
#define SA_COLSTAT_MAX 0  /* max over the group's queries of p_ij (FG-Attn cached mask) */
#define SA_COLSTAT_SUM 1  /* sum over the group's queries of p_ij (Chipmunk column sums) */

/* Element type of the attention output o. */
#define SA_OUT_BF16 0
#define SA_OUT_FP32 1

typedef struct {
  int32_t B, H;       /* batch, heads */
  int32_t Nq, Nk;     /* query tokens, key/value tokens per head */
  int32_t d;          /* head dimension: 64 or 128 */
  int32_t group_size; /* M: contiguous queries sharing one key list (128, or C = 192) */
  float scale;        /* softmax scale, normally 1/sqrt(d); finite, non-zero */
  int32_t out_dtype;  /* SA_OUT_BF16 (0, default) or SA_OUT_FP32; forward only */
} sa_problem;

typedef struct {
  int32_t mode;       /* sa_select_mode */
  int64_t topk;       /* TOPK: number of keys, clamped to [1, Nk] */
  double threshold;   /* THRESHOLD: tau in [0, 1] */
  double mass;        /* MASS: rho in (0, 1] */
} sa_select;

/*
 * Bytes of device workspace sparse_attn_build_index needs for this problem
 * (mean queries, room for the fp32 score matrix of every group against every
 * key, per-row selection results, counters and a list of rows).  TOPK over
 * at least 8192 keys uses the score matrix's room for smaller buffers (a
 * sampled score matrix, per-row brackets, keep-masks and candidates) and
 * writes full score rows only for rows those cannot settle.  0 if the
 * problem is invalid.
 */
size_t sparse_attn_build_index_workspace_size(const sa_problem* problem);

/*
 * Builds the per-group key lists (FG-Attn review, §4.4 pooling mask; LoSA's
 * retained-mass rule).  For each unit (b, h, g):
 *   q_avg = mean of the group's query rows;
 *   sigma_j = scale * (q_avg . k_j) for every key j < Nk;
 *   keys ranked by (sigma descending, index ascending), then
 *     TOPK:      the first min(topk, Nk) keys;
 *     THRESHOLD: keys with p_j = exp(sigma_j - logsumexp(sigma)) >= threshold,
 *                or the top-ranked key if none qualifies;
 *     MASS:      the shortest ranked prefix whose sum of p_j reaches mass.
 * Lists are written ascending into col_idx with row_ptr as their CSR offsets
 * (row_ptr[0] = 0, row_ptr[rows] = nnz).  Scores are computed in fp32 from
 * an fp32 mean query (split into two bf16 terms for the tensor cores), so a
 * key whose score lies within rounding of the cut may fall either side.
 * TOPK over at least 8192 keys (a multiple of 8, scale > 0) finds each row's
 * cut without storing the scores: a sample of every 8th key brackets the
 * cut, a second scoring pass marks the keys above the bracket and keeps
 * those inside it, and the exact cut is taken among them; rows whose bracket
 * misses are selected from their full scores afterwards, so the lists are
 * the same as by full sorting in every case.
 *
 *  q, k          device bf16 [B,H,Nq,d], [B,H,Nk,d]
 *  row_ptr       device int64 [B*H*G + 1], written
 *  col_idx       device int32 [col_capacity], written
 *  col_capacity  entries available in col_idx
 *  nnz_out_host  host int64, nullable.  If set, the call synchronises the
 *                stream, stores nnz and reports SA_ERR_CAPACITY /
 *                SA_ERR_TIMEOUT.  In THRESHOLD and MASS modes nnz is data
 *                dependent: unless col_capacity >= B*H*G*Nk, nnz_out_host
 *                must be given (else SA_ERR_INVALID_ARG).  In TOPK mode nnz
 *                is B*H*G*min(topk,Nk) and is checked up front.
 *  workspace     device, >= sparse_attn_build_index_workspace_size bytes;
 *                contents on entry do not matter; must not be shared with a
 *                concurrent call.
 * Lists that would overflow col_capacity are not written (row_ptr still is).
 */
sa_status sparse_attn_build_index(const sa_problem* problem, const sa_select* select,
                                  const void* q, const void* k, int64_t* row_ptr,
                                  int32_t* col_idx, int64_t col_capacity,
                                  int64_t* nnz_out_host, void* workspace,
                                  size_t workspace_bytes, sa_stream_t stream);

/*
 * The index builder for callers that cannot allocate device memory.  The
 * paper has no counterpart: this entry point exists for callers such as
 * runtimes that forbid allocation after start-up, allocator hooks, or plugins
 * that are handed tensor pointers but no allocator.
 *
 * Same operation, arguments, results and errors as sparse_attn_build_index,
 * without the workspace: the builder's scratch lives in one library-owned
 * device array of SA_NOALLOC_WORKSPACE_BYTES (32 MiB), which every GPU that
 * loads this code holds until the process exits.  A problem whose
 * sparse_attn_build_index_workspace_size exceeds that returns
 * SA_ERR_UNSUPPORTED before anything is enqueued.  Each CUDA context on a
 * device holds its own instance of the array: the first call in a context
 * (for most callers, the device's primary context) looks up its device
 * address (cudaGetSymbolAddress) with that context current, and a call from
 * another context looks it up again; make the first call in each context
 * before any stream capture.
 * Every call shares the array and leaves its contents behind: calls that
 * overlap on the GPU (other streams, other host threads) race on it and must
 * be serialised by the caller.  Calls no allocating function.
 */
#define SA_NOALLOC_WORKSPACE_BYTES (32u << 20)

sa_status sparse_attn_build_index_noalloc(const sa_problem* problem, const sa_select* select,
                                          const void* q, const void* k, int64_t* row_ptr,
                                          int32_t* col_idx, int64_t col_capacity,
                                          int64_t* nnz_out_host, sa_stream_t stream);

/*
 * Key lists from the attention probabilities of a dense step (FG-Attn
 * review, cached mask; Chipmunk review, Alg. 4 column sums).  For each unit
 * (b, h, g) and key j < Nk:
 *   p_ij   = exp(scale * q_i . k_j - lse_i)   for the group's query rows i,
 *   stat_j = max_i p_ij (SA_COLSTAT_MAX) or sum_i p_ij (SA_COLSTAT_SUM),
 * where lse_i is the natural-log log-sum-exp of row i over all Nk keys, as
 * sparse_attn_forward writes it in its dense mode (row_ptr = col_idx = NULL).
 * Rows whose lse is not finite count for nothing.  Keys are ranked by
 * (stat descending, index ascending), then
 *   TOPK:      the first min(topk, Nk) keys;
 *   THRESHOLD: keys with stat_j >= threshold (the statistic itself; the
 *              cached mask uses threshold = 0.5 / Nk with SA_COLSTAT_MAX),
 *              or the top-ranked key if none qualifies; threshold in
 *              [0, 1] for MAX, [0, group_size] for SUM;
 *   MASS:      the shortest ranked prefix whose stat sum reaches mass times
 *              the sum over all keys (LoSA's retained mass, exact at the
 *              dense step with SA_COLSTAT_SUM).
 * Lists, workspace (sparse_attn_build_index_workspace_size bytes), capacity
 * rules, nnz_out_host, synchronisation and errors are those of
 * sparse_attn_build_index.  Statistics are computed in fp32 from
 * tensor-core scores (bf16 inputs, fp32 accumulation), so a key whose
 * statistic lies within rounding of the cut may fall either side.
 *
 *  stat          SA_COLSTAT_MAX or SA_COLSTAT_SUM (else SA_ERR_INVALID_ARG)
 *  lse           device fp32 [B,H,Nq], 4-byte aligned
 */
sa_status sparse_attn_build_index_dense(const sa_problem* problem, const sa_select* select,
                                        int32_t stat, const void* q, const void* k,
                                        const float* lse, int64_t* row_ptr, int32_t* col_idx,
                                        int64_t col_capacity, int64_t* nnz_out_host,
                                        void* workspace, size_t workspace_bytes,
                                        sa_stream_t stream);

/*
 * Column-sparse attention forward (FG-Attn review, "What carries the
 * argument": gather-load of the listed K/V rows into tensor-core tiles;
 * Chipmunk review, Alg. 3: softmax renormalised over the kept keys).
 * For each query row i of unit u with kept keys K_u = col_idx[row_ptr[u]..):
 *   l_ij = scale * q_i . k_j  (j in K_u),   m_i = max_j l_ij,
 *   o_i = sum_j exp(l_ij - m_i) v_j / sum_j exp(l_ij - m_i),
 *   lse_i = m_i + ln sum_j exp(l_ij - m_i)     (natural log).
 * An empty list gives o_i = 0 and lse_i = -inf.  Duplicate indices count
 * twice; order within a list does not matter.
 *
 *  q             device bf16 [B,H,Nq,d]
 *  k, v          device bf16 [B,H,Nk,d]
 *  row_ptr       device int64 [B*H*G + 1]
 *  col_idx       device int32 [nnz]
 *  nnz           length of col_idx; every row_ptr entry must lie in [0, nnz]
 *                row_ptr = col_idx = NULL: dense mode, every unit keeps keys
 *                0 .. Nk-1 and nnz is ignored (the dense step whose lse
 *                feeds sparse_attn_build_index_dense); only one of the two
 *                NULL is SA_ERR_INVALID_ARG
 *  o             device [B,H,Nq,d], written: bf16 (the fp32 result rounded to
 *                nearest even) or fp32, per problem->out_dtype
 *  lse           device fp32 [B,H,Nq], written; nullable
 *  dev_status    device int32, nullable.  Malformed input never makes the
 *                kernel read out of bounds: a unit whose row_ptr pair is out
 *                of order or outside [0, nnz] is treated as empty, and an index
 *                outside [0, Nk) as a zero K/V row; the matching
 *                SA_DEVERR_* bit is ORed into *dev_status (never cleared).
 */
sa_status sparse_attn_forward(const sa_problem* problem, const void* q, const void* k,
                              const void* v, const int64_t* row_ptr, const int32_t* col_idx,
                              int64_t nnz, void* o, float* lse, int32_t* dev_status,
                              sa_stream_t stream);

/*
 * Sparse-delta attention (Chipmunk review, "What carries the argument" and
 * Eq. 1 as its referee reads it; Appendix B.2: the softmax normalisation of
 * an earlier step is reused).  For each query row i of unit u with kept
 * keys K_u:
 *   o_i = base_i + sign * sum_{j in K_u} exp(scale * q_i . k_j - lse_ref_i) v_j
 * — a masked full softmax with the caller's normaliser, not renormalised
 * over K_u.  With lse_ref from a dense step (sparse_attn_forward's dense
 * mode), sign = -1 and base = that step's output (fp32), the call writes the
 * cache of the keys outside the lists; a later step adds its own kept keys'
 * terms back with sign = +1 and base = the cache.  With every key kept, the
 * true lse, base = NULL and sign = 1 it is dense attention.  A row whose
 * lse_ref is not finite gets base_i (or 0).
 *
 *  q, k, v, row_ptr, col_idx, nnz, dev_status   as for sparse_attn_forward
 *                (row_ptr = col_idx = NULL keeps every key)
 *  lse_ref       device fp32 [B,H,Nq], natural log, 4-byte aligned
 *  base          device fp32 [B,H,Nq,d], 16-byte aligned; NULL = zeros
 *  sign          finite multiplier of the sum (normally +1 or -1)
 *  o             device [B,H,Nq,d] in problem->out_dtype; may be base itself
 *                when the output is fp32 (in place), must not overlap it
 *                otherwise
 */
sa_status sparse_attn_forward_delta(const sa_problem* problem, const void* q, const void* k,
                                    const void* v, const int64_t* row_ptr,
                                    const int32_t* col_idx, int64_t nnz, const float* lse_ref,
                                    const float* base, float sign, void* o, int32_t* dev_status,
                                    sa_stream_t stream);

/*
 * One attention layer from host memory: copies overlapped with computation.
 * (The pages describe no host interface; this is the runtime around the two
 * calls above.)  The B*H (batch, head) pairs are split into chunks of
 * consecutive heads: with more than two heads the first and the last chunk
 * hold one head each (their copies are the ones computation cannot hide)
 * and the heads between form chunks of 1, 2, 4, ... heads up to
 * heads_per_chunk (0: the middle split in three), then heads_per_chunk, so
 * that each chunk's copy in is hidden behind the previous chunk's
 * computation from the start; at most 64 chunks.  For each chunk, on copy_in: Q, K, V from
 * host to the device staging buffers; on compute, once they have landed:
 * sparse_attn_build_index (this select, no synchronisation) and
 * sparse_attn_forward; on copy_out, once that is done: O (and LSE) back to
 * the host.  Chunk c+1 arrives and chunk c-1 leaves while chunk c computes.
 * Every copy is one cudaMemcpyAsync of a contiguous range.  The call
 * returns after enqueueing; the compute stream waits for the last copy, so
 * synchronising `compute` completes the layer.  Copies of a call start only
 * after the work an earlier call left on `compute`.
 *   q_host, k_host, v_host   host bf16 [B,H,N,d]; pinned for the copies to overlap
 *   o_host, lse_host         host outputs (o per problem->out_dtype; lse fp32
 *                            [B,H,Nq], nullable together with lse_dev)
 *   q_dev ... lse_dev        device staging of the same full shapes
 *   row_ptr, col_idx, workspace
 *                            device scratch for ONE chunk: row_ptr
 *                            [heads_per_chunk*G + 1], col_idx of col_capacity
 *                            >= heads_per_chunk*G*k (TOPK) or
 *                            heads_per_chunk*G*Nk (else; SA_ERR_CAPACITY
 *                            otherwise), workspace of the build's size for a
 *                            problem of heads_per_chunk heads (0 stands for
 *                            ceil((B*H - 2) / 3) when B*H > 2, else B*H)
 *   compute, copy_in, copy_out   streams; a NULL copy stream means `compute`
 * The lists are scratch (each chunk overwrites them).  Argument errors of
 * the inner calls are returned as they are; nothing is allocated except the
 * events that order the streams.
 */
sa_status sparse_attn_layer_from_host(const sa_problem* problem, const sa_select* select,
                                      const void* q_host, const void* k_host, const void* v_host,
                                      void* o_host, float* lse_host, void* q_dev, void* k_dev,
                                      void* v_dev, void* o_dev, float* lse_dev, int64_t* row_ptr,
                                      int32_t* col_idx, int64_t col_capacity, void* workspace,
                                      size_t workspace_bytes, int32_t heads_per_chunk,
                                      sa_stream_t compute, sa_stream_t copy_in, sa_stream_t copy_out);

/*
 * Index lists from other mask formats (the forward reads CSR).
 *
 * Bit-packed keep-mask (Chipmunk review, "Bitpacked Sparsity Masks": one bit
 * per entry, 8x smaller than a byte mask): for each index row (unit b, h, g)
 * ceil(Nk/32) uint32 words; key j is kept when bit (j % 32) of word j / 32
 * is set (LSB first; the same bits as numpy.packbits(..., bitorder="little")
 * of a row padded to a multiple of 32).  Bits past Nk are ignored.
 *   mask_words  device uint32 [B*H*G, ceil(Nk/32)], 4-byte aligned
 *
 * Block-sparse mask (FG-Attn review, "The pith" and Fig. 6: masks of
 * block-sparse attention methods feed the slice kernel directly): one byte
 * per (index row, key block of block_k keys); non-zero keeps every key of the
 * block (the last block holds Nk - (nb-1)*block_k keys).  Query blocks are
 * the query groups of problem->group_size rows.
 *   block_mask  device uint8 [B*H*G, ceil(Nk/block_k)]; block_k >= 1
 *
 * Both write ascending lists into col_idx with row_ptr as their offsets
 * (rows may be empty).  row_ptr, col_idx, col_capacity, nnz_out_host:
 * as for sparse_attn_build_index (nnz is data dependent: unless col_capacity
 * >= B*H*G*Nk, nnz_out_host must be given; with it the call synchronises and
 * returns SA_ERR_CAPACITY if the lists do not fit — rows that do not fit are
 * not written).  Only problem's B, H, Nq, Nk, d and group_size are used.
 */
sa_status sparse_attn_index_from_bitmask(const sa_problem* problem, const uint32_t* mask_words,
                                         int64_t* row_ptr, int32_t* col_idx, int64_t col_capacity,
                                         int64_t* nnz_out_host, sa_stream_t stream);

sa_status sparse_attn_index_from_block_mask(const sa_problem* problem, int32_t block_k,
                                            const uint8_t* block_mask, int64_t* row_ptr,
                                            int32_t* col_idx, int64_t col_capacity,
                                            int64_t* nnz_out_host, sa_stream_t stream);

/*
 * Token layout on either side of the attention path.
 *
 * Voxel reordering (Chipmunk review, "What carries the argument" / Alg. 1):
 * tokens of a (T, Hh, W) latent grid, raster order t*Hh*W + h*W + w, are
 * reordered so that each contiguous run of vt*vh*vw tokens is one voxel:
 * voxels in raster order over the voxel grid, tokens in raster order inside
 * a voxel; voxels at the far edges of a grid they do not tile are clipped.
 * With voxels of M (or C) tokens, query group g of the reordered sequence is
 * voxel g.
 *   grid      T, Hh, W >= 1 and the voxel vt, vh, vw >= 1; N = T*Hh*W < 2^31
 *   x, y      device bf16 [BH, N, d], 16-byte aligned, not overlapping
 *   inverse   0: y[n] = x[order[n]] (raster -> voxel), 1: y[order[n]] = x[n]
 * d in {64, 128}.  Asynchronous; errors as for the other entry points.
 */
typedef struct {
  int32_t T, Hh, W;    /* latent grid (frames, height, width in tokens) */
  int32_t vt, vh, vw;  /* voxel shape */
} sa_voxel_grid;

sa_status sparse_attn_voxel_permute(const sa_voxel_grid* grid, int32_t BH, int32_t d, const void* x,
                                    void* y, int32_t inverse, sa_stream_t stream);

/*
 * Rolling KV window (DiT page, "The Architecture": a window of 4 chunks,
 * the first chunk a permanent attention sink, then the 2 most recent chunks
 * and the current one; "roll the cache if the 4-chunk window is full (sink
 * stays)").  The caches hold `slots` chunks of chunk_tokens rows in
 * chronological order.  Appending the chunk numbered chunks_before (0 for
 * the first): while chunks_before < slots it fills slot chunks_before;
 * otherwise slots 1 .. slots-2 take the contents of slots 2 .. slots-1 (the
 * oldest non-sink chunk leaves), the new chunk fills the last slot and slot
 * 0 never changes.  K and V move alike, in place.
 *   cache_k, cache_v  device bf16 [BH, slots * chunk_tokens, d], 16-byte aligned
 *   new_k, new_v      device bf16 [BH, chunk_tokens, d], 16-byte aligned
 *   valid_tokens      host, nullable: keys valid after the append,
 *                     min(chunks_before + 1, slots) * chunk_tokens
 * 2 <= slots <= 64; d in {64, 128}.  Asynchronous.
 */
sa_status sparse_attn_kv_window_append(int32_t BH, int32_t d, int32_t chunk_tokens, int32_t slots,
                                       int64_t chunks_before, void* cache_k, void* cache_v,
                                       const void* new_k, const void* new_v,
                                       int64_t* valid_tokens, sa_stream_t stream);

/*
 * Checks index lists without trapping: row_ptr[0] == 0, row_ptr[rows] == nnz,
 * row_ptr non-decreasing, every index in [0, Nk) and strictly ascending
 * within its row.  dev_status is a caller-provided device int32 used as the
 * flag word (cleared first).  Synchronises the stream.  Returns SA_OK or
 * SA_ERR_BAD_INDEX.
 */
sa_status sparse_attn_validate_index(const sa_problem* problem, const int64_t* row_ptr,
                                     const int32_t* col_idx, int64_t nnz,
                                     int32_t* dev_status, sa_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char* sparse_attn_status_string(sa_status status);

/* Library version: major*10000 + minor*100 + patch. */
int32_t sparse_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_ATTN_H */
