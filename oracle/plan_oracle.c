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
 *   - Every request costs its blocks plus one fixed overhead c (c >= 1), so
 *     total = sum_i (n_i + c).  Lay the requests out in order on a line of
 *     cost units: request i owns c overhead units followed by its n_i block
 *     units.  Part p takes the next ceil(total / parts) units, the range
 *     [p * q, (p + 1) * q) with q = ceil(total / parts).
 *   - A request belongs to a part when the part's range holds at least one of
 *     its blocks; a request with no blocks belongs to the part holding its
 *     first overhead unit.  A part's record lists its first and last request
 *     and the block range it covers in each.
 *   - Cost of a part = sum over its pieces of (blocks + c) <= q + c = payload:
 *     the page's "+ fixed_overhead" is the room for the overhead a split
 *     request pays again in the part that continues it.
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
 * Returns 0, or -3 on bad sizes, -2 out of memory.
 */
int oracle_plan(const int32_t *seqlens, int b, int page, int num_parts, int fixed_overhead,
                int32_t *parts, int32_t *num_splits) {
    if (b < 1 || page <= 0 || num_parts <= 0 || fixed_overhead < 1) return -3;
    const int64_t c = fixed_overhead;
    int64_t *nblk = (int64_t *)malloc(sizeof(int64_t) * (size_t)b);
    int64_t *start = (int64_t *)malloc(sizeof(int64_t) * (size_t)(b + 1));
    int32_t *pieces = (int32_t *)calloc((size_t)b, sizeof(int32_t));
    int32_t *first_piece_of_part = (int32_t *)malloc(sizeof(int32_t) * (size_t)num_parts);
    if (!nblk || !start || !pieces || !first_piece_of_part) {
        free(nblk);
        free(start);
        free(pieces);
        free(first_piece_of_part);
        return -2;
    }
    /* step 1: blocks per request, and each request's place on the cost line */
    start[0] = 0;
    for (int i = 0; i < b; ++i) {
        int64_t L = seqlens[i] > 0 ? seqlens[i] : 0;
        nblk[i] = (L + page - 1) / page;
        start[i + 1] = start[i] + c + nblk[i];
    }
    /* step 2: the share of one part */
    const int64_t total = start[b];
    const int64_t q = (total + num_parts - 1) / num_parts;

    /* step 3: each part takes the next q units; requests in order */
    for (int p = 0; p < num_parts; ++p) {
        int32_t *rec = parts + (int64_t)p * F_COUNT;
        for (int f = 0; f < F_COUNT; ++f) rec[f] = 0;
        const int64_t a = (int64_t)p * q;
        int64_t e = a + q;
        if (e > total) e = total;
        int first = -1, last = -1;
        int64_t first_b0 = 0, last_b1 = 0;
        for (int i = 0; i < b; ++i) {
            const int64_t blk_lo = start[i] + c; /* line position of block 0 */
            int in;
            int64_t j0 = 0, j1 = 0;
            if (nblk[i] > 0) {
                j0 = a - blk_lo;
                if (j0 < 0) j0 = 0;
                j1 = e - blk_lo;
                if (j1 > nblk[i]) j1 = nblk[i];
                in = j1 > j0;
            } else {
                in = start[i] >= a && start[i] < e;
            }
            if (!in) continue;
            if (first < 0) {
                first = i;
                first_b0 = j0;
                first_piece_of_part[p] = pieces[i];
            }
            last = i;
            last_b1 = j1;
            pieces[i] += 1;
        }
        if (first < 0) {
            rec[F_BEGIN_REQ] = b;
            rec[F_END_REQ] = b - 1;
            first_piece_of_part[p] = -1;
            continue;
        }
        rec[F_BEGIN_REQ] = first;
        rec[F_END_REQ] = last;
        rec[F_BEGIN_BLOCK] = (int32_t)first_b0;
        rec[F_END_BLOCK] = (int32_t)last_b1;
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
    free(start);
    free(pieces);
    free(first_piece_of_part);
    return 0;
}
