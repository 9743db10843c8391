// mla_sched.cu -- device tile scheduler: builds the split-KV plan from the
// sequence lengths.
//
// Source: "FlashMLA 新内核深度解析：Seesaw 调度、细粒度 TMA 流水线与 H800 上的 660
// TFlops MLA 解码", section "Tile Scheduler：跨 SM 的负载均衡".  One warp counts
// the 64-token blocks of every request, sets the per-part cap
//     payload = ceil(total / num_sm_parts) + fixed_overhead,
// and walks the requests in order, filling each SM part greedily and cutting a
// request into several pieces when it does not fit.  It records one
// DecodingSchedMeta record per part and num_splits, the prefix sum of pieces
// per request, for the combine.
//
// Readings of what that section leaves open:
//   - total = sum_i (blocks_i + fixed_overhead): every piece costs its blocks
//     plus the fixed overhead (a request cut in two pays it twice);
//   - a part that cannot take the rest of the current request takes
//     (remaining - overhead) blocks of it when that is at least one block,
//     otherwise it closes; the last part takes whatever is still unassigned;
//   - pieces are numbered request by request; num_splits[i] is the index of
//     request i's first piece and num_splits[batch] their total.
// The plan only balances work: any valid plan gives the same attention result.
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

__device__ __forceinline__ int64_t blocks_of(int32_t L) {
    return L > 0 ? (static_cast<int64_t>(L) + kPage - 1) / kPage : 0;
}

__global__ void __launch_bounds__(32) sched_kernel(const int32_t* __restrict__ seqlens, int batch,
                                                   int R, int num_parts, int n_mtiles, int fixed,
                                                   int32_t* meta, int32_t* num_splits) {
    // Let the decode kernel (programmatically dependent) run its prologue now;
    // it waits for this grid's completion before reading the plan.
    pdl_launch_dependents();
    const int lane = threadIdx.x;
    int64_t tot = 0;
    for (int i = lane; i < batch; i += 32) tot += blocks_of(seqlens[i]) + fixed;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    const int64_t payload = (tot + num_parts - 1) / num_parts + fixed;

    if (lane == 0) {
        int32_t* rec0 = meta + kMetaHeader;
        int now_req = 0;
        int64_t now_block = 0;
        int64_t nb_now = batch > 0 ? blocks_of(seqlens[0]) : 0;
        int piece = 0;
        for (int p = 0; p < num_parts; ++p) {
            int32_t* rec = rec0 + static_cast<int64_t>(p) * kMetaFields;
            if (now_req >= batch) {
                rec[kBeginReq] = batch;
                rec[kEndReq] = batch - 1;
                rec[kBeginBlock] = 0;
                rec[kEndBlock] = 0;
                rec[kBeginSplit] = piece;
                rec[kFirstSplit] = 0;
                rec[kLastSplit] = 0;
                rec[kPad] = 0;
                continue;
            }
            rec[kBeginReq] = now_req;
            rec[kBeginBlock] = static_cast<int32_t>(now_block);
            rec[kBeginSplit] = piece;
            int64_t remain = payload;
            int end_req = now_req;
            int64_t end_block = 0;
            while (now_req < batch) {
                const int64_t cost = nb_now - now_block + fixed;
                if (p == num_parts - 1 || cost <= remain) {
                    if (now_block == 0) num_splits[now_req] = piece;
                    ++piece;
                    remain -= cost;
                    end_req = now_req;
                    end_block = nb_now;
                    ++now_req;
                    now_block = 0;
                    nb_now = now_req < batch ? blocks_of(seqlens[now_req]) : 0;
                } else if (remain > fixed) {
                    if (now_block == 0) num_splits[now_req] = piece;
                    ++piece;
                    now_block += remain - fixed;
                    end_req = now_req;
                    end_block = now_block;
                    break;
                } else {
                    break;
                }
            }
            rec[kEndReq] = end_req;
            rec[kEndBlock] = static_cast<int32_t>(end_block);
            rec[kPad] = 0;
        }
        num_splits[batch] = piece;
        meta[kHMagic] = kMetaMagic;
        meta[kHBatch] = batch;
        meta[kHRows] = R;
        meta[kHParts] = num_parts;
        meta[kHMTiles] = n_mtiles;
        meta[kHFixed] = fixed;
        meta[kHPage] = kPage;
        meta[kHPieces] = piece;
    }
    __syncwarp();
    // Split flags need every request's final piece count.
    for (int p = lane; p < num_parts; p += 32) {
        int32_t* rec = meta + kMetaHeader + static_cast<int64_t>(p) * kMetaFields;
        const int br = rec[kBeginReq], er = rec[kEndReq];
        if (br >= batch) continue;
        rec[kFirstSplit] = (num_splits[br + 1] - num_splits[br]) > 1;
        rec[kLastSplit] = (num_splits[er + 1] - num_splits[er]) > 1;
    }
}

cudaError_t launch_sched(const int32_t* seqlens, int batch, int R, int num_parts, int n_mtiles,
                         int fixed_overhead, int32_t* meta, int32_t* num_splits,
                         cudaStream_t stream) {
    sched_kernel<<<1, 32, 0, stream>>>(seqlens, batch, R, num_parts, n_mtiles, fixed_overhead,
                                       meta, num_splits);
    return cudaGetLastError();
}

}  // namespace mla
