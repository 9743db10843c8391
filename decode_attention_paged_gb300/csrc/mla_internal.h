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
    int q_box_rows;   // rows one Q tile load brings (min(64, R))
    float scale_log2; // softmax_scale * log2(e)
    int causal;
    int* error_word;
    uint64_t budget_ns;
};

struct CombineParams {
    const int32_t* meta;
    const int32_t* num_splits;
    const float* oaccum;
    const float* lseaccum;
    __nv_bfloat16* out;
    int64_t out_sb, out_ss, out_sh;
    float* lse;
    int batch, s_q, h_q, R;
};

// Host launchers (return a cudaError_t).
cudaError_t launch_sched(const int32_t* seqlens, int batch, int R, int num_parts, int n_mtiles,
                         int fixed_overhead, int32_t* meta, int32_t* num_splits,
                         cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& q_map,
                          const CUtensorMap& kv_map, cudaStream_t stream);
cudaError_t launch_decode_tq(const DecodeParams& p, const CUtensorMap& q_map,
                             const CUtensorMap& kv_map, cudaStream_t stream);
cudaError_t launch_decode_pair(const DecodeParams& p, const CUtensorMap& q_map,
                               const CUtensorMap& kv_map, cudaStream_t stream);
int pair_max_active_clusters();  // on the current device; 0 when the query fails
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool pdl);
int sched_max_batch();

}  // namespace mla
