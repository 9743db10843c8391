// mla_internal.h -- declarations shared by the translation units of libmla.so
// (host launchers and the kernel parameter blocks).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla_decode.h"

namespace mla {

constexpr int kDqk = 576;        // K / Q head dim (512 latent + 64 RoPE)
constexpr int kDv = 512;         // V head dim: the first 512 dims of the same row
constexpr int kPage = 64;        // tokens per KV page
constexpr int kTileM = 64;       // query rows per CTA (one weight-stationary MMA row tile)
constexpr int kChunks = kDqk / 64;  // 64-dim chunks of one row: 9
constexpr int kChunkBytes = 64 * 128;  // one [64 rows][64 dims] bf16 chunk, 128B-swizzled
constexpr int kMetaHeader = 8;   // int32 header words before the part records
constexpr int kMetaFields = 8;   // int32 words per part record
// Every metadata buffer has room for at least this many part records, so a
// decode CTA with a smaller part index may read its record beside the header
// (and use it only once the header matches).
constexpr int kMetaMinParts = 256;
constexpr int kMetaMagic = 0x4D4C4131;  // "MLA1"

// Part record fields (the DecodingSchedMeta of the Tile Scheduler section).
enum MetaField {
    kBeginReq = 0,
    kEndReq = 1,
    kBeginBlock = 2,
    kEndBlock = 3,
    kBeginSplit = 4,
    kFirstSplit = 5,
    kLastSplit = 6,
    kPad = 7
};
// Header fields.
enum MetaHeader {
    kHMagic = 0,
    kHBatch = 1,
    kHRows = 2,
    kHParts = 3,
    kHMTiles = 4,
    kHFixed = 5,
    kHPage = 6,
    kHPieces = 7
};

struct DecodeParams {
    const int32_t* block_table;
    int64_t bt_stride;
    int max_blocks;
    const int32_t* seqlens;
    const int32_t* meta;
    const int32_t* num_splits;
    __nv_bfloat16* out;
    int64_t out_sb, out_ss, out_sh;
    float* lse;
    float* oaccum;    // [pieces][R][512]
    float* lseaccum;  // [pieces][R], log2 domain
    int batch, s_q, h_q, R, n_mtiles, num_parts;
    int q_box_rows;   // rows one Q tile load brings (min(64, R); 64 in the CTA-pair kernel)
    float scale_log2; // softmax_scale * log2(e)
    int causal;
    int* error_word;
    uint64_t budget_ns;
    // Sparse decode ("[DeepSeek-3] FlashMLA", sec. 11): the kernel's requests
    // are the (i, s) query tokens, each with its own key list of topk
    // physical positions indices[(i * fold + s) * topk + k] (< 0: padding),
    // gathered row by row from the cache (pages packed back to back).
    // sparse == 0: dense decode through block_table.  (indices may be null
    // when topk == 0.)
    int sparse;
    const int32_t* indices;
    int topk;
    int64_t num_tokens;  // num_pages * 64: positions past it are reported
    const uint8_t* kv_bytes;  // cache base; row n starts at kv_bytes + n * kv_token_bytes
    int64_t kv_token_bytes;
    int fold;            // sparse: s_q of the caller (request r = i * fold + s); dense: 0
    // FP8 cache ("[DeepSeek-3] FlashMLA", sec. 12; decode_kernel only): rows
    // of 656 bytes (512 e4m3, 4 fp32 scales, 64 bf16 RoPE), a page of 64 rows
    // packed at kv_bytes + page * kv_page_bytes; num_tokens = num_pages * 64.
    int fp8;
    int64_t kv_page_bytes;
    // Cache heads ("[DeepSeek-3] FlashMLA", sec. 4: k_cache [blocks, 64, h_kv,
    // 576]): dense requests are (i, cache head j) pairs r = i * kvh + j whose
    // rows are s * grp + hh for query head j * grp + hh (grp = h_q / kvh).
    // kvh = 1, grp = h_q: one cache head.
    int kvh, grp;
    // decode_kernel only: 1 = P of each page in that page's RoPE chunk (the
    // softmax may run a page ahead of PV), 0 = one P buffer.
    int stage_p;
    // decode_kernel's head-size instantiation only: K / Q rows of nc 64-dim
    // chunks (d = 64 nc <= 576), V their first nv chunks (dv = 64 nv <= 512);
    // the partials in oaccum are rows of dv floats.
    int nc, nv;
};

// Output address of (kernel request r, row) for every layout: dense
// requests are (i, cache head j) pairs with rows s * grp + hh (query head
// j * grp + hh); sparse requests fold (i, s) and their rows are heads.
struct OutMap {
    int64_t out_off;   // element offset into out
    int64_t lse_idx;   // element index into lse [b][h_q][s_q]
};
__device__ __forceinline__ OutMap out_map(int r, int row, int h_q, int s_q, int fold, int kvh,
                                          int grp, int64_t out_sb, int64_t out_ss,
                                          int64_t out_sh) {
    OutMap m;
    if (fold > 0) {
        const int i = r / fold, s = r % fold;
        m.out_off = i * out_sb + s * out_ss + row * out_sh;
        m.lse_idx = (static_cast<int64_t>(i) * h_q + row) * fold + s;
    } else {
        const int i = r / kvh, j = r % kvh;
        const int s = row / grp, h = j * grp + row % grp;
        m.out_off = i * out_sb + s * out_ss + h * out_sh;
        m.lse_idx = (static_cast<int64_t>(i) * h_q + h) * s_q + s;
    }
    return m;
}

struct CombineParams {
    const int32_t* meta;
    const int32_t* num_splits;
    const float* oaccum;
    const float* lseaccum;
    __nv_bfloat16* out;
    int64_t out_sb, out_ss, out_sh;
    float* lse;
    int batch, s_q, h_q, R;
    int num_parts;  // SM parts of the plan (bounds the pieces: batch + num_parts)
    int fold;      // as DecodeParams::fold
    int kvh, grp;  // as DecodeParams::kvh, grp
    int dv;        // partial row length (512, or a head-size call's dv)
};

// Host launchers (return a cudaError_t).
// Request r has seqlens[r / seq_div] keys (seq_div = h_kv: the cache heads
// of one sequence); seqlens == nullptr: every request has uniform_len keys.
cudaError_t launch_sched(const int32_t* seqlens, int seq_div, int uniform_len, int batch, int R,
                         int num_parts, int n_mtiles, int fixed_overhead, int32_t* meta,
                         int32_t* num_splits, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& q_map,
                          const CUtensorMap& kv_map, cudaStream_t stream);
cudaError_t launch_decode_tq(const DecodeParams& p, const CUtensorMap& q_map,
                             const CUtensorMap& kv_map, cudaStream_t stream);
cudaError_t launch_decode_duo(const DecodeParams& p, const CUtensorMap& q_map,
                              const CUtensorMap& kv_map, cudaStream_t stream);
int duo_max_active_clusters();  // on the current device; 0 when the query fails
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool pdl);
int sched_max_batch();

}  // namespace mla
