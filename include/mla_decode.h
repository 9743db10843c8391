/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) paged MLA decode library
 * (libmla.so).
 *
 * What it computes.  Multi-head Latent Attention decode after weight
 * absorption: h_q query heads of dimension 576 attend to ONE shared paged KV
 * head whose 576-dim rows (512 latent + 64 RoPE) serve as K, and whose first
 * 512 dims serve as V ("[DeepSeek-3] FlashMLA：把 MLA 的 KV Cache 优势变成 GPU
 * 吞吐", sec. 2 "Weight Absorption" and sec. 3 "一个 576 维缓存为什么同时充当 K
 * 和 V").  For request i, query token s, head h:
 *     visible  = { t < L_i : !causal || t <= L_i - s_q + s }
 *     kv_t     = k_cache[block_table[i][t / 64]][t % 64][0][:]
 *     x_t      = softmax_scale * dot(q[i][s][h][:], kv_t[0:576])
 *     lse[i][h][s] = ln sum_t exp(x_t)                    (natural log)
 *     out[i][s][h][:] = sum_t exp(x_t - lse) * kv_t[0:512]
 * An empty visible set gives out = 0 and lse = -inf.  The causal rule is the
 * bottom-right aligned triangle ("3.4 Attention kernel", 代码).
 *
 * The two calls follow the API of "FlashMLA 新内核深度解析" (section "如何在
 * 仓库中验证与复现"): get_mla_metadata(cache_seqlens, s_q*h_q//h_kv, h_kv, ...)
 * -> (tile_scheduler_metadata, num_splits), then flash_mla_with_kvcache(q,
 * kvcache, block_table, cache_seqlens, dv, metadata, num_splits, causal) ->
 * (out, lse).  Here they are mla_get_metadata and mla_decode_fwd.
 *
 * Conventions for every function:
 *   - returns MLA_OK (0) or a negative MLA_ERR_* code; mla_strerror() names it;
 *   - every pointer argument named *_dev is DEVICE memory, owned by the
 *     caller; the library never allocates, frees or retains memory;
 *   - work is enqueued asynchronously on `stream` (a cudaStream_t, 0 = the
 *     legacy default stream) on the CURRENT device; no call synchronises the
 *     stream except mla_last_device_error;
 *   - argument errors are detected on the host before anything is enqueued
 *     and leave every buffer untouched;
 *   - errors that only the device can see (a sequence longer than its
 *     block-table row, metadata built for another shape, a pipeline wait that
 *     exceeded its time budget) are recorded in a per-device error word and
 *     reported by mla_last_device_error().
 * Supported: bf16 q / k_cache / out, fp32 lse, d_qk = 576, d_v = 512 (other
 * sizes through mla_decode_fwd_dims), page
 * size 64, batch * h_kv <= 16384, GPUs of compute capability 10.3 (GB300);
 * other shapes return MLA_ERR_UNSUPPORTED.
 *
 * Several cache heads (h_kv > 1; "[DeepSeek-3] FlashMLA", sec. 4: k_cache is
 * [blocks, 64, h_kv, 576] and the dense tests cover MQA and GQA): query heads
 * j*g .. j*g+g-1 (g = h_q / h_kv) attend to cache head j, each group as in the
 * definition above.  h_q must be a multiple of h_kv, and g must divide 64 or
 * be a multiple of 64 (else MLA_ERR_UNSUPPORTED); the heads of a token are
 * adjacent in the cache (head stride 576).  Not with sparse decode or the FP8
 * layout (MLA_ERR_UNSUPPORTED).
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *mla_stream_t; /* same type as cudaStream_t */

/* Every entry point below is exported from libmla.so (built with hidden
 * default visibility, so nothing else is). */
#ifndef MLA_API
#define MLA_API __attribute__((visibility("default")))
#endif

enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARGUMENT = -1,   /* null pointer, bad size or stride       */
    MLA_ERR_UNSUPPORTED = -2,        /* shape/layout not built, or wrong GPU    */
    MLA_ERR_WORKSPACE_TOO_SMALL = -3,
    MLA_ERR_CUDA = -4,               /* a CUDA runtime call failed              */
    MLA_ERR_DEVICE_TIMEOUT = -5,     /* device: a pipeline wait ran out         */
    MLA_ERR_METADATA_MISMATCH = -6,  /* device: metadata built for other shapes */
    MLA_ERR_NO_DEVICE = -7,          /* no CUDA device visible                  */
    MLA_ERR_SEQ_TOO_LONG = -8,       /* device: L_i > 64 * max_blocks_per_seq   */
    MLA_ERR_BAD_ALIGNMENT = -9,      /* a pointer/stride breaks 16-byte rules   */
    MLA_ERR_BAD_INDEX = -10          /* device: a sparse index past the cache   */
};

#define MLA_HEAD_DIM_QK 576
#define MLA_HEAD_DIM_V 512
#define MLA_PAGE_SIZE 64

/* Human-readable name of a status code (static string, never NULL). */
MLA_API const char *mla_strerror(int code);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
MLA_API int mla_version(void);

/*
 * mla_metadata_size -- bytes of the two metadata buffers for a problem shape.
 * Source: "FlashMLA 新内核深度解析", section "Tile Scheduler" (DecodingSchedMeta
 * per SM part, num_splits per request).
 *   meta_bytes: int32 header[8] + max(num_sm_parts, 256) records of 8 int32
 *     each, where num_sm_parts = max(1, SMs / ceil(s_q*h_q / h_kv / 64)) on the
 *     current device (records past num_sm_parts are not written; the room lets
 *     a decode CTA read its record before it has checked the header);
 *   num_splits_bytes: int32[batch + 1].
 * With h_kv > 1 the plan's requests are the (request, cache head) pairs:
 * num_splits is int32[batch * h_kv + 1] and a tile has s_q*h_q/h_kv rows.
 * Either output pointer may be NULL.  Errors: INVALID_ARGUMENT for
 * batch < 1, h_q < 1, s_q < 1, h_kv < 1 or h_q not a multiple of h_kv;
 * UNSUPPORTED for the head groupings above; NO_DEVICE / CUDA when the device
 * cannot be queried.
 */
MLA_API int mla_metadata_size(int batch, int h_q, int s_q, int h_kv, size_t *meta_bytes,
                      size_t *num_splits_bytes);

/*
 * mla_get_metadata -- build the tile-scheduler plan on the device.
 * Source: "FlashMLA 新内核深度解析", section "Tile Scheduler" (one warp counts
 * every request's 64-token blocks, caps each SM part at
 * payload = ceil(total / num_sm_parts) + fixed overhead, and walks the requests
 * greedily, splitting a request over parts when it does not fit).
 *   cache_seqlens_dev : int32[batch], device.  Negative values count as 0.
 *   meta_dev          : device buffer of mla_metadata_size() meta_bytes,
 *                       16-byte aligned; receives header + part records.
 *   num_splits_dev    : device int32[batch + 1]; receives the prefix sum of the
 *                       number of pieces each request is cut into.
 * The plan is valid for mla_decode_fwd calls with the same batch, s_q, h_q,
 * h_kv, cache_seqlens and device; it may be reused across layers of one step
 * ("[DeepSeek-3] FlashMLA", sec. 5).  Enqueues one kernel on `stream`.
 */
MLA_API int mla_get_metadata(const int32_t *cache_seqlens_dev, int batch, int h_q, int s_q, int h_kv,
                     void *meta_dev, int32_t *num_splits_dev, mla_stream_t stream);

/*
 * mla_workspace_size -- bytes of split-KV scratch mla_decode_fwd needs:
 * fp32 partial outputs [pieces][s_q*h_q][512] and partial log-sum-exps
 * [pieces][s_q*h_q], with pieces <= batch + num_sm_parts (every part boundary
 * adds at most one piece).  Source: "[DeepSeek-3] FlashMLA", sec. 6
 * (out_accum / lse_accum), "CUTLASS 从零重写 FlashAttention：Split KV 并行优化
 * 实战" sec. 3.1 (caller-preallocated, aligned workspace).
 */
MLA_API int mla_workspace_size(int batch, int h_q, int s_q, int h_kv, size_t *bytes);

/*
 * mla_decode_fwd -- paged MLA decode: out, lse from q and the paged cache.
 * Sources: "[DeepSeek-3] FlashMLA", sec. 3-7 (definition, paging, split-KV,
 * online softmax); "FlashMLA 新内核深度解析", sections "细粒度 TMA copy-GEMM 流水
 * 线", "缓存提示", "Programmatic Dependent Launch", "Tile Scheduler".
 *
 *   q_dev        bf16 [batch][s_q][h_q][576]; the 576 dims and the (s_q, h_q)
 *                rows are packed (row stride 576, s stride h_q*576 elements);
 *                q_batch_stride (elements) is free but a multiple of 8.
 *                16-byte aligned.
 *   k_cache_dev  bf16 [num_pages][64][h_kv][576]; k_page_stride and
 *                k_token_stride in elements, multiples of 8, the 576 dims
 *                of a head contiguous and the h_kv heads of a token adjacent
 *                (k_token_stride >= h_kv * 576).  16-byte aligned.  Slots of the last page of a
 *                sequence beyond its length never influence the result.
 *   block_table_dev int32 [batch][max_blocks_per_seq], row stride
 *                bt_batch_stride (elements).  Entries for blocks
 *                < ceil(L_i / 64) must name pages in [0, num_pages); an entry
 *                outside reads zeros (never out-of-bounds memory).
 *   cache_seqlens_dev int32 [batch].
 *   softmax_scale  multiplies q.k (the examples use 576^-0.5).
 *   causal         0 or 1 (bottom-right aligned mask over the s_q tokens).
 *   meta_dev, num_splits_dev  from mla_get_metadata for the same shapes.
 *   workspace_dev  >= mla_workspace_size() bytes, 256-byte aligned.
 *   out_dev      bf16 [batch][s_q][h_q][512]; element strides out_batch_stride,
 *                out_s_stride, out_h_stride; dims contiguous; 16-byte aligned
 *                rows.
 *   lse_dev      fp32 [batch][h_q][s_q], contiguous.
 * Enqueues the decode kernel and (programmatically dependent) the combine
 * kernel on `stream`.  Graph-capturable: no allocation, no synchronisation.
 * Programmatic dependent launch ("FlashMLA 新内核深度解析", section
 * "Programmatic Dependent Launch"): each kernel lets the next kernel on the
 * stream launch right after its own prologue, and waits for the previous one
 * (griddepcontrol.wait) before it reads its inputs or writes anything.  A
 * caller's kernel launched after this call with the programmatic-serialization
 * attribute must likewise wait (cudaGridDependencySynchronize) before it reads
 * out or lse; kernels launched without that attribute are ordered as usual.
 */
MLA_API int mla_decode_fwd(const void *q_dev, int64_t q_batch_stride, const void *k_cache_dev,
                   int64_t k_page_stride, int64_t k_token_stride, int num_pages, int page_size,
                   const int32_t *block_table_dev, int64_t bt_batch_stride,
                   int max_blocks_per_seq, const int32_t *cache_seqlens_dev, int batch, int s_q,
                   int h_q, int h_kv, float softmax_scale, int causal, const void *meta_dev,
                   const int32_t *num_splits_dev, void *workspace_dev, size_t workspace_bytes,
                   void *out_dev, int64_t out_batch_stride, int64_t out_s_stride,
                   int64_t out_h_stride, float *lse_dev, mla_stream_t stream);

/*
 * mla_decode_fwd_dims -- mla_decode_fwd for other head sizes: q rows and
 * cache rows of d_qk dims, out rows of d_v dims, V again the first d_v dims
 * of each cache row.  The pages' decode has d_qk = 576, d_v = 512 ("[DeepSeek-3]
 * FlashMLA", sec. 3; the reference tests' configuration in "FlashMLA 新内核深度
 * 解析", "如何在仓库中验证与复现"); this call takes any d_qk and d_v that are
 * multiples of 64 with 64 <= d_v <= d_qk <= 576 and d_v <= 512, for one cache
 * head (h_kv = 1), bf16, on the single-CTA kernel.  Other sizes return
 * MLA_ERR_UNSUPPORTED.  Strides and layouts as mla_decode_fwd with 576 read
 * as d_qk and 512 as d_v: q [batch][s_q][h_q][d_qk], k_cache
 * [num_pages][64][1][d_qk] (k_token_stride >= d_qk), out
 * [batch][s_q][h_q][d_v] (out_h_stride >= d_v).  The plan and the workspace
 * are those of mla_get_metadata / mla_workspace_size for the same batch,
 * h_q, s_q and h_kv.  d_qk = 576, d_v = 512 is exactly mla_decode_fwd.
 */
MLA_API int mla_decode_fwd_dims(const void *q_dev, int64_t q_batch_stride, const void *k_cache_dev,
                                int64_t k_page_stride, int64_t k_token_stride, int num_pages,
                                int page_size, const int32_t *block_table_dev,
                                int64_t bt_batch_stride, int max_blocks_per_seq,
                                const int32_t *cache_seqlens_dev, int batch, int s_q, int h_q,
                                int h_kv, int d_qk, int d_v, float softmax_scale, int causal,
                                const void *meta_dev, const int32_t *num_splits_dev,
                                void *workspace_dev, size_t workspace_bytes, void *out_dev,
                                int64_t out_batch_stride, int64_t out_s_stride,
                                int64_t out_h_stride, float *lse_dev, mla_stream_t stream);

/*
 * mla_decode_splitkv / mla_decode_combine -- the two kernels mla_decode_fwd
 * enqueues, callable one at a time (the split-KV kernel and the combine kernel
 * of "FlashMLA 新内核深度解析", section "Programmatic Dependent Launch").
 * mla_decode_fwd(args) is exactly mla_decode_splitkv(args) followed by
 * mla_decode_combine(...) on the same stream; separately they let a caller
 * place events between the two (e.g. to time each kernel).
 *
 * mla_decode_splitkv takes mla_decode_fwd's arguments and has the same
 * checks and errors.  It writes out/lse of every request the plan kept in one
 * piece, and the partial results of split requests into the workspace.
 *
 * mla_decode_combine merges the partials of split requests into out/lse.
 * Arguments have the meaning they have in mla_decode_fwd; workspace_dev must
 * hold the partials the matching mla_decode_splitkv call wrote.  It is
 * launched as a programmatic dependent of the preceding kernel on `stream`.
 */
MLA_API int mla_decode_splitkv(const void *q_dev, int64_t q_batch_stride, const void *k_cache_dev,
                               int64_t k_page_stride, int64_t k_token_stride, int num_pages,
                               int page_size, const int32_t *block_table_dev,
                               int64_t bt_batch_stride, int max_blocks_per_seq,
                               const int32_t *cache_seqlens_dev, int batch, int s_q, int h_q,
                               int h_kv, float softmax_scale, int causal, const void *meta_dev,
                               const int32_t *num_splits_dev, void *workspace_dev,
                               size_t workspace_bytes, void *out_dev, int64_t out_batch_stride,
                               int64_t out_s_stride, int64_t out_h_stride, float *lse_dev,
                               mla_stream_t stream);
MLA_API int mla_decode_combine(const void *meta_dev, const int32_t *num_splits_dev,
                               void *workspace_dev, size_t workspace_bytes, int batch, int s_q,
                               int h_q, int h_kv, void *out_dev, int64_t out_batch_stride,
                               int64_t out_s_stride, int64_t out_h_stride, float *lse_dev,
                               mla_stream_t stream);

/*
 * mla_decode_fwd_noalloc -- mla_decode_fwd for callers that cannot allocate
 * device memory.  The paper has no counterpart: this is a service of this
 * library.
 *
 * Who needs it.  Some callers may not call cudaMalloc (or any allocator) at
 * the point where they decode:
 *   - a plugin inside a host framework that owns the whole device memory pool
 *     and hands the plugin no allocator;
 *   - a serving loop that forbids device allocation on its hot path, because
 *     cudaMalloc can synchronise the device and stall every other stream;
 *   - a process that has already reserved device memory up to its limit.
 * They still own and pass every input and output; only the split-KV scratch
 * (the `workspace` of mla_decode_fwd) is supplied by the library.
 *
 * Arguments and results are those of mla_decode_fwd without workspace_dev and
 * workspace_bytes.  The scratch is one static device array of
 * MLA_NOALLOC_SCRATCH_BYTES (32 MiB) inside libmla.so: every GPU that loads
 * the library keeps those 32 MiB until the process exits.  A problem whose
 * mla_workspace_size() exceeds it is refused with MLA_ERR_WORKSPACE_TOO_SMALL
 * before anything is enqueued (e.g. batch 64 x h_q 16 needs ~7 MB and fits;
 * batch 64 x h_q 128 needs ~37 MB and does not).
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress); make that first call before any stream
 * capture.  All calls on a device share the one array and it keeps whatever
 * the last call left there; nothing in it needs to start at zero, because
 * every partial the combine reads is written earlier by the same call.  Calls
 * whose work overlaps on the GPU (e.g. on two streams at once) race on the
 * array and give wrong results: serialise them.  Allocates nothing and calls
 * no allocating routine.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
MLA_API int mla_decode_fwd_noalloc(const void *q_dev, int64_t q_batch_stride,
                                   const void *k_cache_dev, int64_t k_page_stride,
                                   int64_t k_token_stride, int num_pages, int page_size,
                                   const int32_t *block_table_dev, int64_t bt_batch_stride,
                                   int max_blocks_per_seq, const int32_t *cache_seqlens_dev,
                                   int batch, int s_q, int h_q, int h_kv, float softmax_scale,
                                   int causal, const void *meta_dev,
                                   const int32_t *num_splits_dev, void *out_dev,
                                   int64_t out_batch_stride, int64_t out_s_stride,
                                   int64_t out_h_stride, float *lse_dev, mla_stream_t stream);

/*
 * mla_decode_fp8_fwd -- mla_decode_fwd over a cache in the FP8 layout of
 * "[DeepSeek-3] FlashMLA：把 MLA 的 KV Cache 优势变成 GPU 吞吐", sec. 12: every
 * token takes 656 bytes,
 *     bytes [0, 512)    512 float8_e4m3 values: latent dims 0..511
 *     bytes [512, 528)  4 fp32 scales, scale j for latent dims 128j..128j+127
 *     bytes [528, 656)  64 bf16 values: RoPE dims 512..575
 * The kernel dequantises each row to k[c] = bf16(e4m3 * scale) (c < 512,
 * round to nearest even) next to the bf16 RoPE and computes what
 * mla_decode_fwd computes over those rows.
 *   k_cache_dev  uint8 [num_pages][64][h_kv = 1][656]: the rows of a page
 *                packed (row stride 656 bytes), pages k_page_stride_bytes
 *                apart (>= 41984, a multiple of 16); 16-byte aligned.  A
 *                block-table entry outside [0, num_pages) reads zeros.
 *   everything else as mla_decode_fwd; the metadata from mla_get_metadata.
 * Runs the kernel that keeps most of Q in tensor memory where mla_decode_fwd
 * would (s_q * h_q <= 32 by default, or as mla_set_decode_kernel chose), with
 * four more warps that dequantise each page in shared memory; otherwise the
 * single-CTA kernel, which runs any plan mla_get_metadata made.
 * Enqueues the decode kernel and the combine kernel on `stream`;
 * graph-capturable.
 */
MLA_API int mla_decode_fp8_fwd(const void *q_dev, int64_t q_batch_stride, const void *k_cache_dev,
                               int64_t k_page_stride_bytes, int num_pages, int page_size,
                               const int32_t *block_table_dev, int64_t bt_batch_stride,
                               int max_blocks_per_seq, const int32_t *cache_seqlens_dev,
                               int batch, int s_q, int h_q, int h_kv, float softmax_scale,
                               int causal, const void *meta_dev, const int32_t *num_splits_dev,
                               void *workspace_dev, size_t workspace_bytes, void *out_dev,
                               int64_t out_batch_stride, int64_t out_s_stride,
                               int64_t out_h_stride, float *lse_dev, mla_stream_t stream);

/*
 * Sparse decode -- attention over a per-query-token list of selected cache
 * positions instead of a request's whole prefix.  Source: "[DeepSeek-3]
 * FlashMLA：把 MLA 的 KV Cache 优势变成 GPU 吞吐", sec. 11 (Sparse FlashMLA: an
 * upper layer picks top-k tokens per query token and passes their physical
 * positions, index = page_id * 64 + offset, so no block table is needed; the
 * kernel gathers those rows and runs QK -> online softmax -> PV).
 * For request i, query token s, head h, with keys
 *     K(i, s) = [ indices[i][s][k] : 0 <= k < topk, 0 <= index < num_pages * 64 ]
 *     x_k     = softmax_scale * dot(q[i][s][h][:], row(index_k)[0:576]),
 *               row(n) = k_cache[n / 64][n % 64][0][:]
 *     lse[i][h][s]    = ln sum_k exp(x_k)
 *     out[i][s][h][:] = sum_k exp(x_k - lse) * row(index_k)[0:512]
 * The page leaves these open; this library reads them as:
 *   - an index < 0 is padding and adds no key;
 *   - an index >= num_pages * 64 adds no key and is reported as
 *     MLA_ERR_BAD_INDEX by mla_last_device_error (the call still completes);
 *   - a position listed twice counts twice (the list is attended as given);
 *   - no causal mask (the selector decides what each token may see);
 *   - an empty key set gives out = 0 and lse = -inf.
 *
 * mla_metadata_size_sparse / mla_workspace_size_sparse: buffer sizes, as
 *   mla_metadata_size / mla_workspace_size (num_splits is int32[batch*s_q + 1]).
 * mla_get_metadata_sparse: the split plan for lists of `topk` entries (every
 *   (i, s) pair is one unit of topk keys).  Enqueues one kernel on `stream`.
 * mla_decode_sparse_fwd: arguments as mla_decode_fwd, with
 *   indices_dev  int32 [batch][s_q][topk], contiguous, 4-byte aligned (may
 *                be NULL when topk == 0);
 *   q_dev        as mla_decode_fwd, and when batch > 1 and s_q > 1 also
 *                q_batch_stride == s_q * h_q * 576 (else MLA_ERR_UNSUPPORTED);
 *   k_cache_dev  as mla_decode_fwd, with the pages packed back to back:
 *                k_page_stride == 64 * k_token_stride (else UNSUPPORTED),
 *                num_pages * 64 < 2^31;
 *   out_dev, lse_dev as mla_decode_fwd.
 * Constraints: batch * s_q <= 16384, 0 <= topk <= 2^24, h_kv = 1.
 * Enqueues the decode kernel and the combine kernel on `stream`;
 * graph-capturable.  The decode kernel is the CTA pair when the dense
 * choice for a tile of h_q rows is the pair (by default h_q >= 128; see
 * mla_set_decode_kernel), else the single-CTA kernel (the TQ kernel does no
 * row gather); mla_get_metadata_sparse plans for the same kernel.
 */
MLA_API int mla_metadata_size_sparse(int batch, int h_q, int s_q, int h_kv, size_t *meta_bytes,
                                     size_t *num_splits_bytes);
MLA_API int mla_get_metadata_sparse(int topk, int batch, int h_q, int s_q, int h_kv,
                                    void *meta_dev, int32_t *num_splits_dev, mla_stream_t stream);
MLA_API int mla_workspace_size_sparse(int batch, int h_q, int s_q, int h_kv, size_t *bytes);
MLA_API int mla_decode_sparse_fwd(const void *q_dev, int64_t q_batch_stride,
                                  const void *k_cache_dev, int64_t k_page_stride,
                                  int64_t k_token_stride, int num_pages, int page_size,
                                  const int32_t *indices_dev, int topk, int batch, int s_q,
                                  int h_q, int h_kv, float softmax_scale, const void *meta_dev,
                                  const int32_t *num_splits_dev, void *workspace_dev,
                                  size_t workspace_bytes, void *out_dev, int64_t out_batch_stride,
                                  int64_t out_s_stride, int64_t out_h_stride, float *lse_dev,
                                  mla_stream_t stream);

/*
 * mla_last_device_error -- synchronise `stream`, then read and clear the
 * current device's error word.  *code receives MLA_OK or the first device-side
 * MLA_ERR_* recorded since the last call.  Returns MLA_ERR_CUDA if the
 * synchronisation itself failed.
 */
MLA_API int mla_last_device_error(mla_stream_t stream, int *code);

/*
 * mla_set_wait_budget_ns -- wall-clock budget of every pipeline wait inside
 * the decode kernel (default 2e9 ns).  When a wait runs out the kernel records
 * MLA_ERR_DEVICE_TIMEOUT, drains its own copies and returns.  Tests use a tiny
 * budget to exercise that path; 0 restores the default.  Process-wide.
 */
MLA_API int mla_set_wait_budget_ns(uint64_t budget_ns);

/*
 * mla_set_fixed_overhead -- the scheduler's fixed per-piece overhead in
 * 64-token blocks (fixed_overhead_num_blocks in the "Tile Scheduler" section;
 * 0 is raised to 1 and values above 4096 are lowered to 4096).  By default
 * it follows the kernel the plan is made for: 2 for the single-CTA kernel, 4
 * for the tensor-memory-Q kernel, 5 for the CTA-pair kernel (about what a
 * request boundary costs each in pages).  Affects only load balance, never
 * results.  Process-wide; negative restores the per-kernel defaults.
 */
MLA_API int mla_set_fixed_overhead(int blocks);

/*
 * mla_set_decode_kernel -- which decode kernel mla_decode_fwd and
 * mla_decode_splitkv launch.  Process-wide; all compute the same function.
 *   MLA_KERNEL_AUTO   (default) MLA_KERNEL_TQ when s_q * h_q <= 32,
 *                     MLA_KERNEL_DUO when s_q * h_q >= 128 (one cache head),
 *                     else MLA_KERNEL_SINGLE.
 *   MLA_KERNEL_SINGLE one CTA per SM part and 64-row query tile,
 *                     Q in shared memory, two KV pages in flight.
 *   MLA_KERNEL_TQ     one CTA per SM part and query tile with Q's dims
 *                     0..447 in tensor memory (the A operand of QK^T, as in
 *                     "Blackwell 多轨矩乘(multi-rail GEMM)", sec. 1), so that
 *                     three KV pages fit in shared memory for tiles of at
 *                     most 32 query rows (two otherwise).
 *   MLA_KERNEL_DUO    a 2-CTA cluster per SM pair and 128-row query tile:
 *                     the two CTAs split every page by head dims, and one
 *                     tcgen05 MMA (cta_group::2, M = 128) feeds all 128 rows
 *                     from each K/V byte; Q's two halves of the latent dims
 *                     sit in the two TMEM lane groups and the partial QK^T
 *                     scores are added after the MMA ("Blackwell 多轨矩乘
 *                     (multi-rail GEMM)", sec. 2 and 4.3).  Tiles of 128 rows
 *                     and one cache head (otherwise MLA_KERNEL_SINGLE runs).
 * The split plan depends on the kernel (its number of SM parts), so metadata
 * must be rebuilt after a switch; a decode call with metadata built for a
 * kernel with another part count records MLA_ERR_METADATA_MISMATCH on the
 * device.  Returns MLA_ERR_INVALID_ARGUMENT for an unknown kind.
 * mla_get_decode_kernel returns the current kind.
 */
#define MLA_KERNEL_SINGLE 1
#define MLA_KERNEL_TQ 2
#define MLA_KERNEL_AUTO 3
#define MLA_KERNEL_DUO 4
MLA_API int mla_set_decode_kernel(int kind);
MLA_API int mla_get_decode_kernel(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
