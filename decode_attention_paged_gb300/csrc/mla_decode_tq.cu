// mla_decode_tq.cu -- split-KV paged MLA decode for sm_103a with most of the
// query tile in tensor memory, so that three KV pages fit in shared memory.
//
// Sources (web pages, cited by title and section):
//   [Overview] "[DeepSeek-3] FlashMLA：把 MLA 的 KV Cache 优势变成 GPU 吞吐":
//       sec. 3 (one 576-dim cache row is K; its first 512 dims are V),
//       sec. 4 (paged KV through block_table), sec. 6 (split-KV partials),
//       sec. 7 (online softmax makes the partials mergeable).
//   [Rails] "Blackwell 多轨矩乘(multi-rail GEMM):FlashMLA 如何用一条 MMA 算完两路
//       QK", sec. 1.2-1.5 (M=64 .ws: each lane group reads its own copy of an
//       A operand held in tensor memory), sec. 1.5 (that copy's cost in TMEM
//       columns is what limits how much of Q fits).
//   [DeepDive] "FlashMLA 新内核深度解析：Seesaw 调度、细粒度 TMA 流水线与 H800
//       上的 660 TFlops MLA 解码": "细粒度 TMA copy-GEMM 流水线" (a 64x576 K
//       tile moves as 64x64 TMA copies), "缓存提示" (EVICT_FIRST), the exp ->
//       exp2 rewrite (end of the Seesaw section), "Programmatic Dependent
//       Launch", "Tile Scheduler" (each SM part walks its DecodingSchedMeta).
//   [AttnBook] "3.4 Attention kernel": "在线 softmax", 代码 (causal mask).
//
// Why this shape.  On GB300 one SM must take in a 72 KB page about every
// 1.6 us to keep HBM busy, and a page stays in shared memory from its TMA
// landing until PV has read it: QK^T, softmax and PV in a row, about 2 us.
// With the 72 KB Q tile in shared memory only two pages fit, so loads stall.
// Here Q's dims 0..447 live in tensor memory as the A operand of QK^T (the
// weight-stationary TS form reads a copy per lane group, so the copy takes
// 224 columns next to O's 256 and S's 32), and only dims 448..575 (two 64-dim
// chunks) stay in shared memory, packed to the rows the tile has.  For tiles
// of at most 32 rows that leaves room for three pages; larger tiles keep two.
// P goes into each page's RoPE chunk, which QK^T is done with, so P has one
// buffer per stage.
//
// Tensor memory (512 columns): O [64 x 512] fp32 as two weight-stationary
// N=256 halves at columns 0 and 128 (lanes 0..63 dims 256h + [0,128), lanes
// 64..127 dims 256h + [128,256)); Q dims 0..447 at 256..479 (28 k-steps x 8
// columns of bf16 pairs, the same rows in both lane groups); S [64 x 64] at
// 480..511 (lanes 0..63 tokens 0..31 of their row, lanes 64..127 tokens
// 32..63).
//
// The query tile arrives through the KV ring as a pseudo page ahead of its
// request's pages; the softmax threads move it into tensor memory (dims
// 0..447) and into the packed shared-memory chunks (dims 448..575).
//
// Warp roles (warp w runs on SM sub-partition w % 4 and reaches TMEM lanes
// 32 (w % 4) .. + 31): warps 0..3 softmax / correction / epilogue / Q copy
// (one thread per TMEM lane; for tiles of at most 32 valid rows only warps 0
// and 2 take part), warp 4 TMA producer, warp 5 TMEM owner and QK^T issuer,
// warp 7 PV issuer.  The two warps that hold the halves of the same rows
// exchange row maxima at a named barrier of their own and agree on every
// early exit through a barrier reduction, so they always pass the same
// barriers.  Every wait is bounded; a timeout records MLA_ERR_DEVICE_TIMEOUT,
// drains the CTA's own copies and MMAs, frees TMEM and returns.
#include "mla_fp8.cuh"
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

namespace {

constexpr int kProducerWarp = 4;
constexpr int kQkWarp = 5;
constexpr int kPvWarp = 7;
constexpr int kDequantWarp0 = 8;  // FP8 cache: warps 8..15 dequantise each page
constexpr int kThreads = 256;
constexpr int kThreadsFp8 = 512;
constexpr uint32_t kDequantBar = 3;  // named barrier of the eight dequant warps

constexpr int kMaxStages = 3;
constexpr uint32_t kStageBytes = kChunks * kChunkBytes;  // 73728
constexpr uint32_t kSmemMax = 232448;                    // 227 KB per CTA
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;    // two PV halves of 128 columns
constexpr uint32_t kColQ = 256;  // Q dims 0..447: 28 k-steps x 8 columns
constexpr uint32_t kColS = 480;  // S: 32 columns
constexpr int kTmemChunks = 7;   // 64-dim chunks of Q held in tensor memory
constexpr float kLazyThreshold = 8.0f;  // log2 units (factor 256)
constexpr uint64_t kDrainBudgetNs = 2000000000ull;

struct Barriers {
    uint64_t kv_full[kMaxStages];
    uint64_t kv_empty[kMaxStages];
    uint64_t q_ready;  // this request's Q tile is in TMEM and in the packed chunks
    uint64_t s_full, s_empty;
    uint64_t p_full[2], pv_done[2];  // by page parity
    uint64_t o_free;
    uint64_t drain_qk, drain_pv;
    uint64_t raw_full[kMaxStages];  // FP8: a ring entry's raw rows landed (Q entries: at issue)
};
static_assert(sizeof(Barriers) <= 256, "barrier block");

// Shared-memory layout as a function of the rows one Q tile load brings: the
// two packed Q chunks (q_rows rows each; the M=64 MMA still reads 64 rows per
// chunk, and the rows past q_rows -- the next chunk's, or the first stage's --
// are padding rows whose scores the softmax masks), then the KV stages.
struct TqLayout {
    uint32_t q_rows, n_stages;
    uint32_t off_kv, off_v, off_bar, off_misc, off_bt, bytes;
};
__host__ __device__ constexpr TqLayout tq_layout(int q_box_rows) {
    TqLayout l{};
    l.q_rows = q_box_rows <= 16 ? 16u : (q_box_rows <= 32 ? 32u : 64u);
    l.n_stages = l.q_rows <= 32 ? 3u : 2u;
    l.off_kv = 2u * l.q_rows * 128u;  // a multiple of 1024
    l.off_v = l.off_kv + l.n_stages * kStageBytes;  // row max / row sum swap: float[128]
    l.off_bar = l.off_v + 512u;
    l.off_misc = l.off_bar + 256u;  // tmem base, abort flag, FP8 out-of-cache flags
    l.off_bt = l.off_misc + 64u;    // block-table windows: int32 [2][32]
    l.bytes = l.off_bt + 256u;
    return l;
}
static_assert(tq_layout(32).n_stages == 3 && tq_layout(64).n_stages == 2, "stage counts");
static_assert(tq_layout(16).bytes <= kSmemMax && tq_layout(32).bytes <= kSmemMax &&
                  tq_layout(64).bytes <= kSmemMax,
              "exceeds the 227 KB per-CTA shared memory limit");
static_assert(kSmemMax < (1u << 18), "descriptor address arithmetic assumes < 256 KB");

struct Part {
    int begin_req, end_req, begin_block, end_block, begin_split;
};

__device__ __forceinline__ int blocks_of(int L) { return L > 0 ? (L + kPage - 1) / kPage : 0; }

__device__ __forceinline__ void item_range(const DecodeParams& p, const Part& part, int req,
                                           int& L, int& nb, int& b0, int& b1) {
    L = p.seqlens[req];
    if (L < 0) L = 0;
    nb = blocks_of(L);
    if (nb > p.max_blocks) nb = p.max_blocks;  // reported as MLA_ERR_SEQ_TOO_LONG
    if (L > nb * kPage) L = nb * kPage;
    b0 = (req == part.begin_req) ? part.begin_block : 0;
    b1 = (req == part.end_req) ? part.end_block : nb;
    if (b1 > nb) b1 = nb;
    if (b0 < 0) b0 = 0;
    if (b0 > b1) b0 = b1;
}

// Walk over the non-empty (request, block) pairs of a part.  g counts pages,
// item counts requests with at least one block; the ring holds each such
// request's Q tile followed by its pages, so page g of item i sits at ring
// index g + i + 1 and the item's Q tile at g_first + i.
struct Cursor {
    int req, blk, b0, b1, L, nb;
    uint32_t g;
    uint32_t item;
    bool valid;
    __device__ __forceinline__ uint32_t ring() const { return g + item + 1; }
};
__device__ __forceinline__ void cursor_seek(const DecodeParams& p, const Part& part, Cursor& c,
                                            int req) {
    for (; req <= part.end_req; ++req) {
        item_range(p, part, req, c.L, c.nb, c.b0, c.b1);
        if (c.b1 > c.b0) {
            c.req = req;
            c.blk = c.b0;
            c.valid = true;
            return;
        }
    }
    c.valid = false;
}
__device__ __forceinline__ Cursor cursor_begin(const DecodeParams& p, const Part& part) {
    Cursor c;
    c.g = 0;
    c.item = 0;
    cursor_seek(p, part, c, part.begin_req);
    return c;
}
__device__ __forceinline__ void cursor_next(const DecodeParams& p, const Part& part, Cursor& c) {
    ++c.g;
    if (++c.blk < c.b1) return;
    ++c.item;
    cursor_seek(p, part, c, c.req + 1);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& wc) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, wc, MLA_ERR_DEVICE_TIMEOUT);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}
// The arrive releases (CTA scope) what lane 0 has seen, and the warp barrier
// orders the other lanes' writes before it.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c,
                                             uint32_t& d) {
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr)
                 : "memory");
}

}  // namespace

// kFp8: the cache is in the FP8 layout ("[DeepSeek-3] FlashMLA", sec. 12).
// Each page's raw rows (one bulk copy) land at the top of its stage and eight
// more warps dequantise them in place into the bf16 page the MMAs read
// (mla_fp8.cuh, four threads per row); Q entries are bf16 as always.
template <bool kFp8>
__global__ void __launch_bounds__(kFp8 ? kThreadsFp8 : kThreads, 1)
    decode_tq_kernel(const __grid_constant__ DecodeParams p,
                     const __grid_constant__ CUtensorMap q_map,
                     const __grid_constant__ CUtensorMap kv_map) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int mtile = blockIdx.x, part_idx = blockIdx.y;
    const TqLayout lay = tq_layout(p.q_box_rows);
    const uint32_t n_stages = lay.n_stages;
    int rows_valid = p.R - mtile * kTileM;
    rows_valid = rows_valid > kTileM ? kTileM : rows_valid;
    // Softmax warps 1 and 3 hold rows 32..63 only; they sit out when those
    // rows do not exist.
    const uint32_t n_active = rows_valid > 32 ? 4u : 2u;
    const bool softmax_warp = warp < 4 && (n_active == 4 || (warp & 1) == 0);

    uint8_t* sQr = smem;  // packed Q chunks 7 and 8
    uint8_t* sKV = smem + lay.off_kv;
    Barriers* bars = reinterpret_cast<Barriers*>(smem + lay.off_bar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + lay.off_misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.off_misc + 4);
    volatile int* raw_bad = reinterpret_cast<volatile int*>(smem + lay.off_misc + 8);  // [3]
    WaitCtx wc{abort_flag, p.error_word, p.budget_ns};

    // ------------------------------------------------------------ prologue
    if (tid == 0) {
        *abort_flag = 0;
        for (uint32_t s = 0; s < n_stages; ++s) {
            // FP8: a page is full when the eight dequant warps arrived; a Q
            // entry gets its eight arrivals from the producer.
            mbar_init(&bars->kv_full[s], kFp8 ? 8 : 1);
            mbar_init(&bars->kv_empty[s], 1);
            mbar_init(&bars->raw_full[s], 1);
        }
        mbar_init(&bars->q_ready, n_active);
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->s_empty, n_active);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->p_full[b], n_active);
            mbar_init(&bars->pv_done[b], 1);
        }
        mbar_init(&bars->o_free, n_active);
        mbar_init(&bars->drain_qk, 1);
        mbar_init(&bars->drain_pv, 1);
        fence_barrier_init();
        prefetch_tensormap(&q_map);
        prefetch_tensormap(&kv_map);
    }
    if (warp == kQkWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait_primary();
    // The dependent (combine) grid may launch now.  It waits for this grid's
    // completion before it reads the partials; the plan, final once the wait
    // above returned, it may read at once.
    pdl_launch_dependents();

    bool ok = (smem_u32(smem) & 1023u) == 0;
    const int32_t* hdr = p.meta;
    // The part record is read beside the header: every metadata buffer has
    // room for kMetaMinParts records, and the record is used only once the
    // header matches this call.
    static_assert(kBeginReq == 0 && kEndReq == 1 && kBeginBlock == 2 && kEndBlock == 3 &&
                      kBeginSplit == 4,
                  "record fields 0..4");
    const int32_t* rec = hdr + kMetaHeader + part_idx * kMetaFields;
    int32_t rv[5] = {0, 0, 0, 0, 0};
    if (part_idx < kMetaMinParts) {
#pragma unroll
        for (int f = 0; f < 5; ++f) rv[f] = rec[f];
    }
    if (ok && (hdr[kHMagic] != kMetaMagic || hdr[kHBatch] != p.batch || hdr[kHRows] != p.R ||
               hdr[kHParts] != p.num_parts || hdr[kHPage] != kPage))
        ok = false;
    Part part{};
    if (ok) {
        if (part_idx >= kMetaMinParts) {
#pragma unroll
            for (int f = 0; f < 5; ++f) rv[f] = rec[f];
        }
        part.begin_req = rv[kBeginReq];
        part.end_req = rv[kEndReq];
        part.begin_block = rv[kBeginBlock];
        part.end_block = rv[kEndBlock];
        part.begin_split = rv[kBeginSplit];
        if (part.begin_req < p.batch &&
            (part.begin_req < 0 || part.end_req >= p.batch || part.end_req < part.begin_req))
            ok = false;
        if (part.begin_req >= p.batch) part.end_req = part.begin_req - 1;
    }
    if (!ok) {
        if (tid == 0) raise_error(wc, MLA_ERR_METADATA_MISMATCH);
        part.begin_req = 0;
        part.end_req = -1;
    }
    if (tid == 0) {
        for (int req = part.begin_req; req <= part.end_req; ++req) {
            const int L = p.seqlens[req];
            if (L > 0 && blocks_of(L) > p.max_blocks) raise_error(wc, MLA_ERR_SEQ_TOO_LONG);
        }
    }

    if (warp == kProducerWarp) {
        // ------------------------------------------------------ TMA producer
        // The whole warp walks the ring; lane 0 waits and issues the copies.
        // Block-table entries come through two 32-page windows in shared
        // memory: window w (pages 32w .. 32w + 31, page 32w + i copied by
        // lane i with cp.async) is fetched while window w - 1 is in use, so
        // no page waits for a global load (a load per page into a register
        // would make the next page's read wait for it).
        const uint64_t policy = policy_evict_first();
        const uint32_t q_bytes = kChunks * p.q_box_rows * 128;
        int32_t* bt_win = reinterpret_cast<int32_t*>(smem + lay.off_bt);
        // The part's first page: its block-table entry is read at once, beside
        // the first request's length, so page 0 waits for one load instead of
        // the first window's walk (which reads the lengths of the requests it
        // crosses) and its copy.  Used when the cursor does start there (a
        // part may begin on a request with no blocks, which it skips).
        const bool bt0_ok = part.begin_req <= part.end_req && part.begin_block >= 0 &&
                            part.begin_block < p.max_blocks;
        const int bt0 = bt0_ok ? p.block_table[static_cast<int64_t>(part.begin_req) * p.bt_stride +
                                               part.begin_block]
                               : 0;
        Cursor ld = cursor_begin(p, part), ahead = ld;
        const bool direct0 = bt0_ok && ld.valid && ld.req == part.begin_req && ld.blk == part.begin_block;
        auto fetch_window = [&](uint32_t slot) {
            int rq = -1, bk = 0;
            for (int i = 0; i < 32 && ahead.valid; ++i) {
                if (lane == i) {
                    rq = ahead.req;
                    bk = ahead.blk;
                }
                cursor_next(p, part, ahead);
            }
            if (rq >= 0)
                cp_async_4(smem_u32(bt_win + 32 * slot + lane),
                           p.block_table + static_cast<int64_t>(rq) * p.bt_stride + bk);
            cp_async_commit();
        };
        uint32_t n_issued = 0;  // ring entries issued
        uint32_t page_bits = 0;  // bit s: stage s's last entry was a page
        // Q tile of request req into stage st.  (FP8: the producer also makes
        // the dequant warps' seven other arrivals and completes the entry's
        // raw_full phase, which keeps that barrier's phases in ring order.)
        auto issue_q = [&](uint32_t st, int req) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->kv_full[st], q_bytes);
                for (int c = 0; c < kChunks; ++c)
                    tma_load_3d(&q_map, &bars->kv_full[st], sKV + st * kStageBytes + c * kChunkBytes,
                                64 * c, mtile * kTileM, req, policy);
                if (kFp8) {
                    for (int k = 0; k < 7; ++k) mbar_arrive(&bars->kv_full[st]);
                    mbar_arrive(&bars->raw_full[st]);
                }
            }
            __syncwarp();
            page_bits &= ~(1u << st);
        };
        // The first request's Q tile (ring entry 0) needs no block-table entry:
        // it goes out before the look-ahead loads.
        if (ld.valid) {
            issue_q(0, ld.req);
            n_issued = 1;
        }
        if (!direct0) fetch_window(0);
        bool stop = false;
        while (ld.valid && !stop) {
            // First block of a request: its Q tile goes into the ring first
            // (already out for the part's first request).
            for (int entry = (ld.blk == ld.b0 && ld.g > 0) ? 0 : 1; entry < 2; ++entry) {
                const uint32_t n = ld.ring() - 1 + entry;
                const uint32_t st = n % n_stages;
                if (n >= n_stages && !warp_wait(&bars->kv_empty[st], ((n / n_stages) + 1) & 1, wc)) {
                    stop = true;
                    break;
                }
                int page = 0;
                if (entry == 1) {
                    if (direct0 && ld.g == 0) {
                        page = bt0;
                    } else {
                        // Window (g / 32) has landed: the first waits for its
                        // only group (for both windows' groups, minus the
                        // second, when page 0 came direct); later ones leave
                        // the next window's group pending.
                        if (ld.g == 0)
                            cp_async_wait_group<0>();
                        else if ((ld.g & 31) == 0 || (direct0 && ld.g == 1))
                            cp_async_wait_group<1>();
                        __syncwarp();
                        page = bt_win[32 * ((ld.g >> 5) & 1) + (ld.g & 31)];
                    }
                }
                if (entry == 0) {
                    issue_q(st, ld.req);
                } else {
                    if (lane == 0) {
                        uint8_t* dst = sKV + st * kStageBytes;
                        if (kFp8) {
                            // One copy of the page's raw rows; a page outside
                            // the cache is not read and dequantises to zeros
                            // (as the bf16 tile reads zeros out of range).
                            const bool in =
                                page >= 0 && static_cast<int64_t>(page) * kPage < p.num_tokens;
                            raw_bad[st] = in ? 0 : 1;
                            if (in) {
                                mbar_arrive_expect_tx(&bars->raw_full[st], kFp8PageBytes);
                                bulk_load(dst + kFp8RawOff,
                                          p.kv_bytes + static_cast<int64_t>(page) * p.kv_page_bytes,
                                          kFp8PageBytes, &bars->raw_full[st], policy);
                            } else {
                                mbar_arrive(&bars->raw_full[st]);
                            }
                        } else {
                            mbar_arrive_expect_tx(&bars->kv_full[st], kStageBytes);
                            for (int c = 0; c < kChunks; ++c)
                                tma_load_3d(&kv_map, &bars->kv_full[st], dst + c * kChunkBytes,
                                            64 * c, 0, page, policy);
                        }
                    }
                    __syncwarp();
                    page_bits |= 1u << st;
                    // First page of a request: ask L2 for the next request's
                    // Q tile, which its ring entry will load after this
                    // request's last page.
                    if (ld.blk == ld.b0 && ld.req < part.end_req && lane == 0)
                        for (int c = 0; c < kChunks; ++c)
                            tma_prefetch_l2_3d(&q_map, 64 * c, mtile * kTileM, ld.req + 1);
                }
                n_issued = n + 1;
            }
            if (stop) break;
            // After page 0: the first window (when page 0 came direct) and the
            // second; after the last page of window w: window w + 2 into w's
            // slot (every lane has read its entry).
            if (ld.g == 0) {
                if (direct0) fetch_window(0);
                fetch_window(1);
            }
            else if ((ld.g & 31) == 31)
                fetch_window((ld.g >> 5) & 1);
            cursor_next(p, part, ld);
        }
        cp_async_wait_all();
        // Drain: no copy may still be landing when the CTA leaves (an FP8
        // page's copy completes raw_full; everything else kv_full).
        if (lane == 0)
            for (uint32_t k = (n_issued >= n_stages ? n_issued - n_stages : 0); k < n_issued; ++k) {
                const uint32_t st = k % n_stages;
                const bool raw = kFp8 && ((page_bits >> st) & 1u);
                mbar_drain(raw ? &bars->raw_full[st] : &bars->kv_full[st], (k / n_stages) & 1,
                           kDrainBudgetNs);
            }
        __syncwarp();
    } else if (warp == kQkWarp) {
        // ------------------------------------------------------ QK^T issuer
        // Page g needs its stage, its request's Q tile and a free S buffer.
        // 28 TS MMAs over dims 0..447 (A from TMEM), 8 SS MMAs over 448..575
        // (A from the packed chunks), all N = 64 into S.
        constexpr uint32_t idesc_qk = idesc_bf16_f32(64, 64, false, false);
        const uint64_t dK0 = smem_desc(smem_u32(sKV), 16, 1024);
        const uint64_t dQr = smem_desc(smem_u32(sQr), 16, 1024);
        constexpr uint64_t kStageUnits = kStageBytes >> 4;
        constexpr uint64_t kChunkUnits = kChunkBytes >> 4;
        const uint64_t q_chunk_units = (lay.q_rows * 128u) >> 4;
        const uint32_t tS = tmem + kColS, tQ = tmem + kColQ;
        for (Cursor qk = cursor_begin(p, part); qk.valid; cursor_next(p, part, qk)) {
            const uint32_t n = qk.ring();
            const uint32_t st = n % n_stages;
            if (qk.blk == qk.b0) {
                // The softmax warps copied this request's Q tile; its ring
                // stage (the entry before this page) is free.
                if (!warp_wait(&bars->q_ready, qk.item & 1, wc)) break;
                if (lane == 0) mbar_arrive(&bars->kv_empty[(n - 1) % n_stages]);
            }
            if (!warp_wait(&bars->kv_full[st], (n / n_stages) & 1, wc)) break;
            if (qk.g >= 1 && !warp_wait(&bars->s_empty, (qk.g - 1) & 1, wc)) break;
            tc_fence_after();
            const uint64_t bK = dK0 + st * kStageUnits;
            // One elected thread issues the whole burst and commits it.
            if (elect_one()) {
#pragma unroll
                for (int j = 0; j < 4 * kTmemChunks; ++j)
                    mma_ws_ts(tS, tQ + 8 * j, bK + (j / 4) * kChunkUnits + 2 * (j & 3), idesc_qk,
                              j ? 1u : 0u);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int c = kTmemChunks + j / 4;  // 7, 8
                    mma_ws_ss(tS, dQr + (j / 4) * q_chunk_units + 2 * (j & 3),
                              bK + c * kChunkUnits + 2 * (j & 3), idesc_qk, 1u);
                }
                mma_commit(&bars->s_full);
            }
            __syncwarp();
        }
        if (elect_one()) mma_commit(&bars->drain_qk);
        __syncwarp();
        if (lane == 0) mbar_drain(&bars->drain_qk, 0, kDrainBudgetNs);
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------ PV issuer
        // Page g needs P(g) (in its stage's RoPE chunk) and, on a request's
        // first block, O released by the previous request's epilogue.
        constexpr uint32_t idesc_pv = idesc_bf16_f32(64, 256, false, true);
        const uint64_t dV0 = smem_desc(smem_u32(sKV), kChunkBytes, 1024);
        const uint64_t dP0 = smem_desc(smem_u32(sKV + 8 * kChunkBytes), 16, 1024);
        constexpr uint64_t kStageUnits = kStageBytes >> 4;
        constexpr uint64_t kHalfUnits = (4 * kChunkBytes) >> 4;
        for (Cursor pv = cursor_begin(p, part); pv.valid; cursor_next(p, part, pv)) {
            const bool first = pv.blk == pv.b0;
            const uint32_t st = pv.ring() % n_stages;
            if (!warp_wait(&bars->p_full[pv.g & 1], (pv.g >> 1) & 1, wc)) break;
            if (first && pv.item > 0 && !warp_wait(&bars->o_free, (pv.item - 1) & 1, wc)) break;
            tc_fence_after();
            const uint64_t bV = dV0 + st * kStageUnits;
            const uint64_t dP = dP0 + st * kStageUnits;
            // One elected thread issues the whole burst and commits it.
            if (elect_one()) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ws_ss(tmem + kColO + 128 * h, dP + 2 * kk,
                                  bV + h * kHalfUnits + 128 * kk, idesc_pv,
                                  (first && kk == 0) ? 0u : 1u);
                mma_commit(&bars->pv_done[pv.g & 1]);
                mma_commit(&bars->kv_empty[st]);
            }
            __syncwarp();
        }
        if (elect_one()) mma_commit(&bars->drain_pv);
        __syncwarp();
        if (lane == 0) mbar_drain(&bars->drain_pv, 0, kDrainBudgetNs);
        __syncwarp();
    } else if (kFp8 && warp >= kDequantWarp0) {
        // ---------------------------------------- FP8 page dequantisation
        // In place, four threads per row (mla_fp8.cuh); the eight warps agree
        // on every exit through bar.red.and before the named barrier inside
        // the routine.  A page's raw_full phase is unambiguous: the stage's
        // previous entry completed its phase before this page was issued
        // into the stage, and the next cannot start before this page's PV.
        const int dt = tid - 32 * kDequantWarp0;
        for (Cursor c = cursor_begin(p, part); c.valid; cursor_next(p, part, c)) {
            const uint32_t n = c.ring(), st = n % n_stages;
            const bool ok = warp_wait(&bars->raw_full[st], (n / n_stages) & 1, wc);
            if (!named_bar_and(kDequantBar, 256, ok)) break;
            fp8_dequant_page_x4(sKV + st * kStageBytes, dt, raw_bad[st] != 0, kDequantBar);
            fence_proxy_async_smem();
            warp_arrive(&bars->kv_full[st]);
        }
    } else if (softmax_warp) {
        // ---------------- softmax / correction / epilogue / Q copy
        const int q4 = warp;              // TMEM lane quadrant
        const int Lrow = 32 * q4 + lane;  // TMEM lane
        const int r = Lrow & 63, half = Lrow >> 6;
        const int row = mtile * kTileM + r;
        const bool row_valid = r < rows_valid;
        const int s_idx = row / p.h_q, h_idx = row % p.h_q;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
        const uint32_t pair_bar = 1 + (q4 & 1);  // warps q4 and q4 ^ 2: the two halves of a row
        const int me = n_active == 4 ? tid : (32 * (warp >> 1) + lane);  // among active threads
        float* v_slot = reinterpret_cast<float*>(smem + lay.off_v);  // [128] row max / row sum
        uint32_t gblk = 0, item = 0;
        bool alive = true;
        // Q tile of a request, from its ring stage (ring entry nq): dims
        // 0..447 into this lane's TMEM copy, dims 448..575 into the packed
        // chunks (by the lane group 0 threads; both groups hold the same rows).
        // Needs only the previous request's QK^T to be complete, so it runs
        // before that request's epilogue and the next QK^T overlaps the
        // epilogue.
        auto q_copy = [&](uint32_t nq) -> bool {
            const uint32_t stq = nq % n_stages;
            if (!named_bar_and(pair_bar, 64, warp_wait(&bars->kv_full[stq], (nq / n_stages) & 1, wc)))
                return false;
            const uint8_t* sq = sKV + stq * kStageBytes;
            const bool have = r < p.q_box_rows;
#pragma unroll 1
            for (int c = 0; c < kTmemChunks; ++c) {
                uint32_t w[32];
                if (have) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        ld_shared_v4(smem_u32(sq + c * kChunkBytes + sw128_offset(r, u)), w[4 * u],
                                     w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) w[i] = 0u;
                }
                tmem_st32(tl + kColQ + 32 * c, w);
            }
            if (half == 0 && r < static_cast<int>(lay.q_rows)) {
                // rows keep their 128-byte swizzle: both bases are 1024-aligned
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint4 v = *reinterpret_cast<const uint4*>(
                            sq + (kTmemChunks + i) * kChunkBytes + r * 128 + u * 16);
                        *reinterpret_cast<uint4*>(sQr + i * lay.q_rows * 128 + r * 128 + u * 16) = v;
                    }
            }
            fence_proxy_async_smem();
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(&bars->q_ready);
            return true;
        };
        int q_done = -1;  // request whose Q tile is already in place
        for (int req = part.begin_req; req <= part.end_req && alive; ++req) {
            int L, nb, b0, b1;
            item_range(p, part, req, L, nb, b0, b1);
            int lim = L;
            if (p.causal) {
                lim = L - p.s_q + s_idx + 1;
                lim = lim < 0 ? 0 : (lim > L ? L : lim);
            }
            const int first_piece = p.num_splits[req];
            const bool split = (p.num_splits[req + 1] - first_piece) > 1;
            const int slot = (req == part.begin_req) ? part.begin_split : first_piece;
            const bool has_blocks = b1 > b0;
            if (has_blocks && q_done != req) {
                if (!q_copy(gblk + item)) {
                    alive = false;
                    break;
                }
            }
            float m_used = -INFINITY, l_part = 0.f;
            for (int blk = b0; blk < b1; ++blk, ++gblk) {
                const uint32_t n = gblk + item + 1;
                const uint32_t st = n % n_stages;
                uint8_t* stage = sKV + st * kStageBytes;
                if (!named_bar_and(pair_bar, 64, warp_wait(&bars->s_full, gblk & 1, wc))) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                uint32_t sv[32];
                tmem_ld32(tl + kColS, sv);
                tmem_ld_wait();
                tc_fence_before();
                warp_arrive(&bars->s_empty);

                const int t0 = blk * kPage + 32 * half;
                float x[32];
                float hmax = -INFINITY;
                const int nvis = row_valid ? lim - t0 : 0;  // columns c < nvis are visible
                const uint64_t sc2 = f32x2_splat(p.scale_log2);
                // Pages every valid row of the warp sees whole skip the masking.
                // (Rows past the tile then hold scores of padding query rows:
                // they only feed their own output rows, which are never
                // written, and are left out of the rescale vote.)
                if (__all_sync(0xffffffffu, !row_valid || nvis >= 32)) {
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        f32x2_mul(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), sc2, x[c],
                                  x[c + 1]);
                        hmax = fmaxf(hmax, fmaxf(x[c], x[c + 1]));
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        float a0, a1;
                        f32x2_mul(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), sc2, a0, a1);
                        x[c] = c < nvis ? a0 : -INFINITY;
                        x[c + 1] = c + 1 < nvis ? a1 : -INFINITY;
                        hmax = fmaxf(hmax, fmaxf(x[c], x[c + 1]));
                    }
                }
                // Row max over both halves (the slot is rewritten only after
                // the next barrier, which the partner passes after reading it).
                v_slot[Lrow] = hmax;
                named_bar_sync(pair_bar, 64);
                const float tmax = fmaxf(hmax, v_slot[Lrow ^ 64]);
                float alpha = 1.f;
                bool need = false;
                if (tmax > m_used + kLazyThreshold) {
                    alpha = (m_used == -INFINITY) ? 0.f : fast_exp2(m_used - tmax);
                    m_used = tmax;
                    need = true;
                }
                if (need) l_part *= alpha;
                uint32_t pk[16];
                // A row with no visible key yet has only -inf scores: with 0
                // in place of the -inf max every exp2 is exactly 0.
                const uint64_t m2 = f32x2_splat(m_used == -INFINITY ? 0.f : m_used);
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    float d0, d1;
                    f32x2_sub(x[2 * c], x[2 * c + 1], m2, d0, d1);
                    const float p0 = fast_exp2(d0);
                    const float p1 = fast_exp2(d1);
                    f32x2_add(ps0, ps1, p0, p1, ps0, ps1);
                    pk[c] = pack_bf16x2(p0, p1);
                }
                l_part += ps0 + ps1;

                // O is rescaled after PV(g - 1).  P has a buffer per stage,
                // but PV may trail by at most two pages so that the parity
                // waits on the two p_full / pv_done barriers stay unambiguous.
                // (The two warps of a pair see the same rows, hence the same
                // rescale decision.)
                const bool rescale = __any_sync(0xffffffffu, need && row_valid && blk > b0);
                const uint32_t lag = rescale ? 1u : 2u;
                bool ok = true;
                if (gblk >= lag) {
                    const uint32_t w = gblk - lag;
                    ok = warp_wait(&bars->pv_done[w & 1], (w >> 1) & 1, wc);
                }
                if (!named_bar_and(pair_bar, 64, ok)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                if (rescale) {
                    const float a = (need && blk > b0) ? alpha : 1.f;
#pragma unroll 1
                    for (int cg = 0; cg < 8; ++cg) {
                        uint32_t o[32];
                        tmem_ld32(tl + kColO + 32 * cg, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                        tmem_st32(tl + kColO + 32 * cg, o);
                    }
                    tmem_st_wait();
                }
                // Last page of the sequence: zero the V rows past its length
                // (they may hold any bits, and 0 * NaN would poison the sum).
                if (blk == nb - 1 && (L & (kPage - 1)) != 0) {
                    const int tail0 = L & (kPage - 1);
                    const int per_chunk = (kPage - tail0) * 8;
                    for (int i = me; i < 8 * per_chunk; i += 32 * static_cast<int>(n_active)) {
                        const int c = i / per_chunk, u = i % per_chunk;
                        reinterpret_cast<uint4*>(stage + c * kChunkBytes + tail0 * 128)[u] =
                            make_uint4(0, 0, 0, 0);
                    }
                }
                // P into the page's RoPE chunk (QK^T is done with it).
                uint8_t* pbuf = stage + 8 * kChunkBytes;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t off = sw128_offset(r, 4 * half + k);
                    *reinterpret_cast<uint4*>(pbuf + off) =
                        make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                warp_arrive(&bars->p_full[gblk & 1]);
            }
            if (!alive) break;
            if (has_blocks) {
                // The next request with blocks: its Q tile (the ring entry
                // after this request's last page) goes in now.
                for (int nr = req + 1; nr <= part.end_req; ++nr) {
                    int L2, nb2, c0, c1;
                    item_range(p, part, nr, L2, nb2, c0, c1);
                    if (c1 > c0) {
                        if (!q_copy(gblk + item + 1)) alive = false;
                        q_done = nr;
                        break;
                    }
                }
                if (!alive) break;
            }

            // ---------------------------------------------------- epilogue
            float l_tot = 0.f;
            if (has_blocks) {
                if (!named_bar_and(pair_bar, 64,
                                   warp_wait(&bars->pv_done[(gblk - 1) & 1],
                                             ((gblk - 1) >> 1) & 1, wc))) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                v_slot[Lrow] = l_part;
                named_bar_sync(pair_bar, 64);
                l_tot = l_part + v_slot[Lrow ^ 64];
            }
            const bool empty = !(l_tot > 0.f);
            const float inv = empty ? 0.f : 1.f / l_tot;
            const float lse2 = empty ? -INFINITY : m_used + fast_log2(l_tot);
            const int64_t acc_row = static_cast<int64_t>(slot) * p.R + row;
            if (has_blocks) {
                // Column groups per TMEM wait: two with the FP8 cache (measured
                // faster there), one for bf16 (two slowed it).
                constexpr int kGroups = kFp8 ? 2 : 1;
                auto store_cg = [&](int cg, const uint32_t (&o)[32]) {
                    const int dv0 = 256 * (cg >> 2) + 128 * half + 32 * (cg & 3);
                    if (split) {
                        float4* dst = reinterpret_cast<float4*>(p.oaccum + acc_row * kDv + dv0);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv,
                                                 __uint_as_float(o[4 * v + 1]) * inv,
                                                 __uint_as_float(o[4 * v + 2]) * inv,
                                                 __uint_as_float(o[4 * v + 3]) * inv);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(
                            p.out + req * p.out_sb + s_idx * p.out_ss + h_idx * p.out_sh + dv0);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint32_t w[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                w[j] = pack_bf16x2(__uint_as_float(o[8 * v + 2 * j]) * inv,
                                                   __uint_as_float(o[8 * v + 2 * j + 1]) * inv);
                            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                };
#pragma unroll 1
                for (int cg = 0; cg < 8; cg += kGroups) {
                    uint32_t o[kGroups][32];
#pragma unroll
                    for (int k = 0; k < kGroups; ++k) tmem_ld32(tl + kColO + 32 * (cg + k), o[k]);
                    tmem_ld_wait();
                    if (!row_valid) continue;
#pragma unroll
                    for (int k = 0; k < kGroups; ++k) store_cg(cg + k, o[k]);
                }
                tc_fence_before();
                warp_arrive(&bars->o_free);
                ++item;
            } else if (row_valid) {
                for (int hh = 0; hh < 2; ++hh) {
                    const int dv0 = 256 * hh + 128 * half;
                    if (split) {
                        float4* dst = reinterpret_cast<float4*>(p.oaccum + acc_row * kDv + dv0);
                        for (int v = 0; v < 32; ++v) dst[v] = make_float4(0.f, 0.f, 0.f, 0.f);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(
                            p.out + req * p.out_sb + s_idx * p.out_ss + h_idx * p.out_sh + dv0);
                        for (int v = 0; v < 16; ++v) dst[v] = make_uint4(0, 0, 0, 0);
                    }
                }
            }
            if (row_valid && half == 0) {
                if (split)
                    p.lseaccum[acc_row] = lse2;
                else
                    p.lse[(static_cast<int64_t>(req) * p.h_q + h_idx) * p.s_q + s_idx] =
                        empty ? -INFINITY : lse2 * 0.69314718055994531f;
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kQkWarp) tmem_dealloc(tmem, kTmemCols);
}

template <bool kFp8>
static cudaError_t tq_set_smem() {
    static int configured_mask = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 31 || !(__atomic_load_n(&configured_mask, __ATOMIC_RELAXED) & (1 << dev))) {
        e = cudaFuncSetAttribute(decode_tq_kernel<kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemMax));
        if (e != cudaSuccess) return e;
        if (dev < 31) __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_RELAXED);
    }
    return cudaSuccess;
}

cudaError_t launch_decode_tq(const DecodeParams& p, const CUtensorMap& q_map,
                             const CUtensorMap& kv_map, cudaStream_t stream) {
    const bool fp8 = p.fp8 != 0;
    cudaError_t e = fp8 ? tq_set_smem<true>() : tq_set_smem<false>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_mtiles, p.num_parts, 1);
    cfg.blockDim = dim3(fp8 ? kThreadsFp8 : kThreads, 1, 1);
    cfg.dynamicSmemBytes = tq_layout(p.q_box_rows).bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return fp8 ? cudaLaunchKernelEx(&cfg, decode_tq_kernel<true>, p, q_map, kv_map)
               : cudaLaunchKernelEx(&cfg, decode_tq_kernel<false>, p, q_map, kv_map);
}

}  // namespace mla
