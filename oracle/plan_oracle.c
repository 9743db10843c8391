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
 *   3. fill the parts request by request, in order, cutting a request into
 *      pieces over several parts when it does not fit in one;
 *   4. record, per request, how many pieces it was cut into (num_splits, as a
 *      prefix sum) so the combine step can find them.
 *   The per-part record has the fields of that section's DecodingSchedMeta.
 *
 * Readings of what the page leaves open:
 *   - total_num_blocks counts every request's blocks plus one fixed overhead
 *     c (c >= 1): total = sum_i (n_i + c).  With blocks alone the cap could
 *     not hold the overheads of a batch of many short requests.
 *   - Every piece of a request costs its blocks plus c: a request continued
 *     in a new part pays the overhead again there.
 *   - The greedy walk, part by part with remain = payload: while requests are
 *     left, if the rest of the current request (its unplaced blocks plus c)
 *     fits in remain, the part takes it whole and moves to the next request;
 *     otherwise the part takes remain - c blocks of it when that is at least
 *     one block (the request continues in the next part) and the part is
 *     closed.  Parts after the last request are empty.
 *   - begin/end request indices are inclusive, the begin block inclusive and
 *     the end block exclusive (the struct's comments on that page); an empty
 *     part has begin_req = b, end_req = b - 1, blocks 0..0.
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
 * page is the KV page size in tokens; fixed_overhead >= 1.
 * Returns 0, or -3 on bad sizes, -2 out of memory, -4 if the walk left work
 * unplaced (the cap rules that out).
 */
int oracle_plan(const int32_t *seqlens, int b, int page, int num_parts, int fixed_overhead,
                int32_t *parts, int32_t *num_splits) {
    if (b < 1 || page <= 0 || num_parts <= 0 || fixed_overhead < 1) return -3;
    const int64_t c = fixed_overhead;
    int64_t *nblk = (int64_t *)malloc(sizeof(int64_t) * (size_t)b);
    int32_t *pieces = (int32_t *)calloc((size_t)b, sizeof(int32_t));
    int32_t *first_piece_of_part = (int32_t *)malloc(sizeof(int32_t) * (size_t)num_parts);
    if (!nblk || !pieces || !first_piece_of_part) {
        free(nblk);
        free(pieces);
        free(first_piece_of_part);
        return -2;
    }
    /* step 1: blocks per request, and the total they cost */
    int64_t total = 0;
    for (int i = 0; i < b; ++i) {
        int64_t L = seqlens[i] > 0 ? seqlens[i] : 0;
        nblk[i] = (L + page - 1) / page;
        total += nblk[i] + c;
    }
    /* step 2: the cap of one part */
    const int64_t payload = (total + num_parts - 1) / num_parts + c;

    /* step 3: the greedy walk, request by request */
    int req = 0;     /* first request not yet fully placed */
    int64_t blk = 0; /* its first unplaced block */
    for (int p = 0; p < num_parts; ++p) {
        int32_t *rec = parts + (int64_t)p * F_COUNT;
        for (int f = 0; f < F_COUNT; ++f) rec[f] = 0;
        if (req >= b) {
            rec[F_BEGIN_REQ] = b;
            rec[F_END_REQ] = b - 1;
            first_piece_of_part[p] = -1;
            continue;
        }
        rec[F_BEGIN_REQ] = req;
        rec[F_BEGIN_BLOCK] = (int32_t)blk;
        first_piece_of_part[p] = pieces[req];
        int64_t remain = payload;
        while (req < b) {
            const int64_t rest = nblk[req] - blk;
            if (remain >= rest + c) { /* the rest fits: take it whole */
                remain -= rest + c;
                pieces[req] += 1;
                rec[F_END_REQ] = req;
                rec[F_END_BLOCK] = (int32_t)nblk[req];
                req += 1;
                blk = 0;
                continue;
            }
            const int64_t take = remain - c; /* cut: as many blocks as fit */
            if (take > 0) {
                pieces[req] += 1;
                rec[F_END_REQ] = req;
                blk += take;
                rec[F_END_BLOCK] = (int32_t)blk;
            }
            break;
        }
    }
    if (req < b) { /* cannot happen: parts * payload covers every overhead paid */
        free(nblk);
        free(pieces);
        free(first_piece_of_part);
        return -4;
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
