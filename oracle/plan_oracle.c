/*
 * plan_oracle.c -- plain CPU restatement of the decode tile scheduler.
 *
 * TEST INFRASTRUCTURE ONLY (see mla_oracle.c).  Shares no code with the CUDA
 * library; the tests compare the device scheduler's output with this one
 * integer for integer, and check the plan's invariants separately.
 *
 * Source: "FlashMLA 新内核深度解析：Seesaw 调度、细粒度 TMA 流水线与 H800 上的
 * 660 TFlops MLA 解码", section "Tile Scheduler：跨 SM 的负载均衡":
 *   1. count the KV blocks of every request from its sequence length;
 *   2. payload = ceil_div(total, num_sm_parts) + fixed_overhead_num_blocks
 *      is the work cap of one SM part;
 *   3. walk the requests in order, greedily filling each part up to the cap
 *      and splitting a request over several parts when it does not fit;
 *   4. record, per request, how many pieces it was cut into (num_splits, as a
 *      prefix sum) so the combine step can find them.
 *   The per-part record has the fields of that section's DecodingSchedMeta.
 *
 * Readings of what the page leaves open (each also listed in the design doc):
 *   - "total" counts every request's blocks plus one fixed overhead per
 *     request: total = sum_i (n_i + c).  A piece of a request costs its blocks
 *     plus c, so a request cut in two pays c twice.
 *   - a part that cannot fit the rest of the current request takes
 *     (remaining - c) blocks of it when that is at least one block, else it
 *     closes; the last part takes everything still unassigned, so the plan
 *     always covers every block.
 *   - begin/end request indices are inclusive, the begin block is inclusive and
 *     the end block exclusive (as the struct's comments on that page say);
 *     an empty part has begin_req = b, end_req = b - 1, blocks 0..0.
 *   - is_first_req_splitted / is_last_req_splitted are 1 when that request is
 *     cut into more than one piece; begin_split_idx is the global index of the
 *     piece this part computes for its first request, pieces being numbered
 *     request by request (num_splits[i] is the first piece of request i).
 */
#include <stdint.h>
#include <stdlib.h>

enum { F_BEGIN_REQ, F_END_REQ, F_BEGIN_BLOCK, F_END_BLOCK, F_BEGIN_SPLIT, F_FIRST_SPLIT,
       F_LAST_SPLIT, F_PAD, F_COUNT };

/*
 * oracle_plan: seqlens[b] -> parts[num_parts][8], num_splits[b + 1].
 * page is the KV page size in tokens; fixed_overhead >= 0.
 * Returns 0, or -3 on bad sizes, -2 out of memory.
 */
int oracle_plan(const int32_t *seqlens, int b, int page, int num_parts, int fixed_overhead,
                int32_t *parts, int32_t *num_splits) {
    if (b < 0 || page <= 0 || num_parts <= 0 || fixed_overhead < 0) return -3;
    int64_t *nblk = (int64_t *)malloc(sizeof(int64_t) * (size_t)(b > 0 ? b : 1));
    int32_t *pieces = (int32_t *)calloc((size_t)(b > 0 ? b : 1), sizeof(int32_t));
    int32_t *first_piece_of_part = (int32_t *)malloc(sizeof(int32_t) * (size_t)num_parts);
    if (!nblk || !pieces || !first_piece_of_part) {
        free(nblk);
        free(pieces);
        free(first_piece_of_part);
        return -2;
    }
    /* step 1: blocks per request */
    int64_t total = 0;
    for (int i = 0; i < b; ++i) {
        int64_t L = seqlens[i] > 0 ? seqlens[i] : 0;
        nblk[i] = (L + page - 1) / page;
        total += nblk[i] + fixed_overhead;
    }
    /* step 2: the cap */
    int64_t payload = (total + num_parts - 1) / num_parts + fixed_overhead;

    /* step 3: greedy walk */
    int now_req = 0;
    int64_t now_block = 0;
    for (int p = 0; p < num_parts; ++p) {
        int32_t *rec = parts + (int64_t)p * F_COUNT;
        for (int f = 0; f < F_COUNT; ++f) rec[f] = 0;
        if (now_req >= b) { /* nothing left: empty part */
            rec[F_BEGIN_REQ] = b;
            rec[F_END_REQ] = b - 1;
            first_piece_of_part[p] = -1;
            continue;
        }
        rec[F_BEGIN_REQ] = now_req;
        rec[F_BEGIN_BLOCK] = (int32_t)now_block;
        first_piece_of_part[p] = pieces[now_req]; /* pieces of now_req before this one */
        int64_t remain = payload;
        int end_req = now_req;
        int64_t end_block = 0;
        while (now_req < b) {
            int64_t rest = nblk[now_req] - now_block;
            int64_t cost = rest + fixed_overhead;
            if (p == num_parts - 1 || cost <= remain) {
                /* the rest of this request fits (or this is the last part) */
                pieces[now_req] += 1;
                remain -= cost;
                end_req = now_req;
                end_block = nblk[now_req];
                now_req += 1;
                now_block = 0;
            } else if (remain > fixed_overhead) {
                /* take what fits; the request continues in the next part */
                int64_t take = remain - fixed_overhead;
                pieces[now_req] += 1;
                now_block += take;
                end_req = now_req;
                end_block = now_block;
                remain = 0;
                break;
            } else {
                break;
            }
        }
        rec[F_END_REQ] = end_req;
        rec[F_END_BLOCK] = (int32_t)end_block;
    }

    /* step 4: prefix sum of pieces per request */
    num_splits[0] = 0;
    for (int i = 0; i < b; ++i) num_splits[i + 1] = num_splits[i] + pieces[i];
    for (int p = 0; p < num_parts; ++p) {
        int32_t *rec = parts + (int64_t)p * F_COUNT;
        if (first_piece_of_part[p] < 0) {
            rec[F_BEGIN_SPLIT] = num_splits[b];
            continue;
        }
        int br = rec[F_BEGIN_REQ], er = rec[F_END_REQ];
        rec[F_BEGIN_SPLIT] = num_splits[br] + first_piece_of_part[p];
        rec[F_FIRST_SPLIT] = pieces[br] > 1;
        rec[F_LAST_SPLIT] = pieces[er] > 1;
    }
    free(nblk);
    free(pieces);
    free(first_piece_of_part);
    return 0;
}
