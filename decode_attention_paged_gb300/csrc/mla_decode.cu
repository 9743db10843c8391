// mla_decode.cu -- persistent split-KV paged MLA decode kernel for sm_103a.
//
// Sources (web pages, cited by title and section):
//   [Overview] "[DeepSeek-3] FlashMLA：把 MLA 的 KV Cache 优势变成 GPU 吞吐":
//       sec. 3 (one 576-dim cache row is K; its first 512 dims are V),
//       sec. 4 (paged KV through block_table), sec. 6 (split-KV partials),
//       sec. 7 (online softmax makes the partials mergeable).
//   [DeepDive] "FlashMLA 新内核深度解析：Seesaw 调度、细粒度 TMA 流水线与 H800
//       上的 660 TFlops MLA 解码": "细粒度 TMA copy-GEMM 流水线" (a 64x576 K
//       tile moves as 9 TMA copies of 64x64), "缓存提示" (EVICT_FIRST on the
//       streamed KV and on Q), exp -> exp2 with the scale folded in (the Seesaw
//       section's closing note), "Programmatic Dependent Launch", "Tile
//       Scheduler" (one CTA group per SM part walks its DecodingSchedMeta).
//   [AttnBook] "3.4 Attention kernel": "在线 softmax" (m, l, o~ with the
//       e^(m - m') rescale), 代码 (bottom-right causal mask).
//
// Design for sm_103a (what differs from the Hopper kernel on those pages):
//   - One CTA per SM part and 64-query-row tile ("m-tile"); grid =
//     (ceil(R / 64), num_sm_parts), at most one CTA per SM (227 KB smem).
//   - The output tile O [64 x 512] fp32 lives in tensor memory, not registers:
//     weight-stationary MMAs with M = 64 use the 2x2 datapath, so O takes 256
//     of the 512 TMEM columns (lanes 0..63 hold dims [0,128) and [256,384),
//     lanes 64..127 dims [128,256) and [384,512)).  This removes the register
//     pressure that motivated the Seesaw schedule, so there is one output
//     tile and no seesaw.
//   - S = Q K^T [64 x 64] goes to TMEM too (32 columns per buffer, two
//     buffers): lanes 0..63 hold tokens 0..31 of each row, lanes 64..127
//     tokens 32..63, so a row's max is combined from two threads.
//   - Warp roles: warp 0 = TMA producer (lane 0 issues; the warp's lanes
//     keep block-table entries loaded 32 pages ahead), warp 1 = TMEM owner
//     and MMA issuer (converged warp, one elected thread per burst), warps 2..5 = softmax /
//     correction / epilogue (one thread per TMEM lane), warps 6..9 = row
//     gather for sparse decode (idle in dense decode).
//   - P of a page goes either into that page's RoPE chunk, dead once its
//     QK^T is done (the softmax of page g + 1 then waits for PV(g) only when
//     O must be rescaled), or into one P buffer placed after everything else,
//     which costs 8 KB more shared memory.  The host picks the first for
//     single-tile problems: the smaller footprint measured 18% faster on a
//     long ragged batch (the 8 KB alone made that difference).  With two or
//     more tiles the P buffer measured 2-5% faster: the PV then does not read
//     P and V from the same stage.
//   - Sparse decode ("[DeepSeek-3] FlashMLA", sec. 11) gathers each key row
//     with 16-byte cp.async copies, eight threads per row: measured on GB300
//     at the rate of the tiled TMA page load, while row-gather TMA copies
//     (four rows per instruction) reached under a quarter of it.
//   - Q and each 64-token page are TMA-loaded as 9 chunks of [64 x 64] bf16
//     with 128-byte swizzle; V is the first 8 chunks of the same page, read by
//     the PV MMA as an MN-major operand, so the page is loaded once.
//   - Lazy rescaling: the running max used for exponentiation only moves when
//     a tile's max exceeds it by more than 8 (log2 units); otherwise O and l
//     keep their scale.  Exact up to rounding: the final lse uses the max that
//     was actually used.
//   - Every wait is bounded (wall clock); on a timeout the CTA records
//     MLA_ERR_DEVICE_TIMEOUT, drains its own copies and MMAs, frees TMEM and
//     returns.  Waits in the softmax warps are taken by lane 0 and broadcast,
//     so control flow stays warp-uniform.
#include "mla_fp8.cuh"
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

namespace {

constexpr int kStages = 2;
constexpr int kThreads = 320;
constexpr int kGatherWarp0 = 6;  // warps 6..9: sparse-decode row gather
constexpr uint32_t kQBytes = kChunks * kChunkBytes;      // 73728
constexpr uint32_t kStageBytes = kChunks * kChunkBytes;  // 73728
constexpr uint32_t kPBytes = 64 * 128;                   // P [64 rows x 64 tokens] bf16
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;    // O: two PV halves of 128 columns
constexpr uint32_t kColS = 256;  // S: two buffers of 32 columns
constexpr float kLazyThreshold = 8.0f;  // log2 units (factor 256)
// Draining waits for copies/MMAs this CTA issued itself; they finish on their
// own, so the drain has its own budget, independent of the (possibly tiny)
// wait budget a caller set.
constexpr uint64_t kDrainBudgetNs = 2000000000ull;
#ifndef MLA_IDLE_SLEEP_NS
#define MLA_IDLE_SLEEP_NS 32
#endif
constexpr unsigned kIdleSleepNs = MLA_IDLE_SLEEP_NS;  // MMA issuer back-off when idle
#ifndef MLA_XCH_SLEEP_NS
#define MLA_XCH_SLEEP_NS 32
#endif
constexpr unsigned kXchSleepNs = MLA_XCH_SLEEP_NS;  // pair-exchange back-off

struct Barriers {
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t q_full, q_empty;
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full[2], pv_done[2];
    uint64_t o_free, drain;
    uint64_t raw_full[kStages];  // FP8: a page's raw rows have landed
};

// FP8 cache: a page's 64 raw rows of 656 bytes land at the top of its stage
// and are dequantised in place into the bf16 layout below them (mla_fp8.cuh).
static_assert(kFp8RawOff + kFp8PageBytes == kStageBytes, "raw rows at the top of a stage");
constexpr uint32_t kDequantBar = 1;  // named barrier of the four dequant warps
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + kQBytes;
// After the KV ring: the one P buffer (only in launches that use it), then
// the barriers, the pair-exchange slots (uint2 [2][128]) and the misc words
// (tmem base, abort flag, key masks).  The P buffer sits 8 KB-aligned right
// after the ring: placed elsewhere the PV MMAs measured a few percent slower.
constexpr uint32_t kOffP = kOffKV + kStages * kStageBytes;
constexpr uint32_t kTailBytes = 256 + 2 * 128 * 8 + 64 + 256;  // ..., block-table windows
constexpr uint32_t kSmemBytes = kOffP + kTailBytes;             // P in each page's RoPE chunk
constexpr uint32_t kSmemBytesP = kOffP + kPBytes + kTailBytes;  // with the P buffer
static_assert(sizeof(Barriers) <= 256, "barrier block");
static_assert(kChunks % 3 == 0, "QK^T is issued three chunks per turn");
static_assert(kSmemBytesP < (1u << 18), "descriptor address arithmetic assumes < 256 KB");
static_assert(kSmemBytesP <= 232448, "exceeds the 227 KB per-CTA shared memory limit");

struct Part {
    int begin_req, end_req, begin_block, end_block, begin_split;
};

__device__ __forceinline__ int blocks_of(int L) { return L > 0 ? (L + kPage - 1) / kPage : 0; }

// Blocks [b0, b1) of request `req` that this part owns, clamped to the
// sequence.  Every role calls this with the same inputs, so all roles see the
// same list of work items.
template <bool kHeads>
__device__ __forceinline__ void item_range(const DecodeParams& p, const Part& part, int req,
                                           int& L, int& nb, int& b0, int& b1) {
    L = p.sparse ? p.topk : p.seqlens[kHeads ? req / p.kvh : req];
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

// A walk over the (request, block) work items of one part, in order.  Each
// role keeps its own cursors; all walk the same sequence.
struct Cursor {
    int req, blk, b0, b1, L, nb;
    uint32_t g;     // block index within the part's work
    uint32_t item;  // index of the current request among those with blocks
    bool valid;
};
template <bool kHeads>
__device__ __forceinline__ void cursor_seek(const DecodeParams& p, const Part& part, Cursor& c,
                                            int req) {
    for (; req <= part.end_req; ++req) {
        item_range<kHeads>(p, part, req, c.L, c.nb, c.b0, c.b1);
        if (c.b1 > c.b0) {
            c.req = req;
            c.blk = c.b0;
            c.valid = true;
            return;
        }
    }
    c.valid = false;
}
template <bool kHeads>
__device__ __forceinline__ Cursor cursor_begin(const DecodeParams& p, const Part& part) {
    Cursor c;
    c.g = 0;
    c.item = 0;
    cursor_seek<kHeads>(p, part, c, part.begin_req);
    return c;
}
template <bool kHeads>
__device__ __forceinline__ void cursor_next(const DecodeParams& p, const Part& part, Cursor& c) {
    ++c.g;
    if (++c.blk < c.b1) return;
    ++c.item;
    cursor_seek<kHeads>(p, part, c, c.req + 1);
}

// Warp-uniform bounded wait: lane 0 polls, the verdict is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& wc) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, wc, MLA_ERR_DEVICE_TIMEOUT);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}
// One arrival per warp, after every lane's prior writes.
// The arrive releases (CTA scope) what lane 0 has seen, and the warp barrier
// orders the other lanes' writes before it.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Exchange one float with the partner thread that holds the other half of
// the same query row (TMEM lane L <-> L ^ 64).  Each side publishes (value,
// tag) with one 64-bit store and spins, with a bounded wait, until the
// partner's slot carries the same tag.  Two slots alternate: a thread can be at
// most one exchange ahead of its partner, because it cannot finish exchange
// n + 1 before the partner has published it.  The verdict is made uniform
// across the warp, so warp-collective instructions stay convergent.
__device__ __forceinline__ bool pair_exchange(uint2* xch, int lrow, uint32_t& seq, float v,
                                              float& partner, const WaitCtx& wc) {
    const uint32_t tag = ++seq;
    uint2* slots = xch + (tag & 1) * 128;
    asm volatile("st.volatile.shared.v2.u32 [%0], {%1, %2};" ::"r"(smem_u32(slots + lrow)),
                 "r"(__float_as_uint(v)), "r"(tag)
                 : "memory");
    const uint32_t src = smem_u32(slots + (lrow ^ 64));
    auto load = [&]() {
        uint2 r;
        asm volatile("ld.volatile.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(src)
                     : "memory");
        return r;
    };
    bool ok = true;
    uint2 got = load();
    if (got.y != tag) {
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t spin = 1;; ++spin) {
            // Back off: a hot spin of 32 lanes on shared memory would eat the
            // bandwidth the tensor core needs to read its operands.
            __nanosleep(kXchSleepNs);
            got = load();
            if (got.y == tag) break;
            if ((spin & 255) == 0) {
                if (*wc.abort_flag) {
                    ok = false;
                    break;
                }
                if (globaltimer_ns() - t0 > wc.budget_ns) {
                    raise_error(wc, MLA_ERR_DEVICE_TIMEOUT);
                    ok = false;
                    break;
                }
            }
        }
    }
    partner = __uint_as_float(got.x);
    return __all_sync(0xffffffffu, ok);
}

// Chunks [C0, C0 + 3) of S = Q K^T for one page: 12 MMAs, issued by the one
// elected thread that issues the whole burst, operand offsets known at compile
// time.
template <int C0>
__device__ __forceinline__ void issue_qk_turn(uint64_t dQ, uint64_t bK, uint32_t d) {
    constexpr uint32_t idesc_qk = idesc_bf16_f32(64, 64, false, false);
    constexpr uint64_t kChunkUnits = kChunkBytes >> 4;
#pragma unroll
    for (int cc = 0; cc < 3; ++cc) {
        const uint64_t a = dQ + (C0 + cc) * kChunkUnits, b = bK + (C0 + cc) * kChunkUnits;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_ws_ss(d, a + 2 * kk, b + 2 * kk, idesc_qk, (C0 + cc + kk) ? 1u : 0u);
    }
}

}  // namespace

// kStageP: P of each page in that page's RoPE chunk (else the one P buffer).
// kFp8: the cache is in the FP8 layout (its own instantiation: the dequant
// registers would otherwise raise every launch's register count).
// kHeads: several cache heads (p.kvh > 1); with one head the request and
// head arithmetic folds away (measured 5% on the h_q = 128 workloads).
// kGen: other head sizes (p.nc, p.nv chunks of 64 dims for d and dv; bf16,
// one cache head), with the 576 / 512 instantiations left as they are.
template <bool kStageP, bool kFp8, bool kHeads, bool kGen = false>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap q_map,
                  const __grid_constant__ CUtensorMap kv_map) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int mtile = blockIdx.x, part_idx = blockIdx.y;
    const int kvh = kHeads ? p.kvh : 1;     // cache heads
    const int grp = kHeads ? p.grp : p.h_q;  // query heads per cache head
    const int nc = kGen ? p.nc : kChunks;   // 64-dim chunks of a K / Q row
    const int nv = kGen ? p.nv : kDv / 64;  // 64-dim chunks of a V row
    const int dv = 64 * nv;

    uint8_t* sQ = smem + kOffQ;
    uint8_t* sKV = smem + kOffKV;
    uint8_t* sP = smem + kOffP;
    uint8_t* tail = smem + kOffP + (kStageP ? 0u : kPBytes);
    Barriers* bars = reinterpret_cast<Barriers*>(tail);
    uint2* xch = reinterpret_cast<uint2*>(tail + 256);
    uint8_t* misc = tail + 256 + 2 * 128 * 8;
    int32_t* bt_win = reinterpret_cast<int32_t*>(misc + 64);  // int32 [2][32]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
    // Sparse decode: key_part[2 * stage + w] has bit t set when stage row t
    // holds a key; the two gather warps of a stage own disjoint bits (written
    // before their kv_full arrivals).
    volatile uint64_t* key_part = reinterpret_cast<volatile uint64_t*>(misc + 8);
    // FP8: raw_bad[stage] = 1 when that page lies outside the cache.
    volatile int* raw_bad = reinterpret_cast<volatile int*>(misc + 40);
    WaitCtx wc{abort_flag, p.error_word, p.budget_ns};

    // ------------------------------------------------------------ prologue
    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->kv_full[s], kFp8 ? 4 : (p.sparse ? 2 : 1));
            mbar_init(&bars->raw_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->s_empty[s], 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->p_full[b], 4);
            mbar_init(&bars->pv_done[b], 1);
        }
        mbar_init(&bars->o_free, 4);
        mbar_init(&bars->drain, 1);
        fence_barrier_init();
        prefetch_tensormap(&q_map);
        prefetch_tensormap(&kv_map);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    // Pair-exchange slots start with tag 0, which no exchange uses.
    for (int i = tid; i < 2 * 128; i += kThreads) xch[i] = make_uint2(0u, 0u);
    // Query rows a partial Q tile load does not bring must read as zeros.
    if (p.q_box_rows < kTileM) {
        for (int i = tid; i < kChunks * kTileM * 8; i += kThreads) {
            const int c = i / (kTileM * 8), rem = i % (kTileM * 8), r = rem / 8;
            if (r >= p.q_box_rows)
                reinterpret_cast<uint4*>(sQ + c * kChunkBytes)[rem] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Everything above touched only on-chip state; global inputs may be
    // written by the preceding kernel on the stream (programmatic launch).
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
        if (part.begin_req >= p.batch) part.end_req = part.begin_req - 1;  // empty part
    }
    if (!ok) {
        if (tid == 0) raise_error(wc, MLA_ERR_METADATA_MISMATCH);
        part.begin_req = 0;
        part.end_req = -1;
    }
    if (tid == 0 && !p.sparse) {
        for (int req = part.begin_req; req <= part.end_req; ++req) {
            const int L = p.seqlens[req / kvh];
            if (L > 0 && blocks_of(L) > p.max_blocks) raise_error(wc, MLA_ERR_SEQ_TOO_LONG);
        }
    }

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // Loads run through a two-page ring.  The whole warp walks it (lane 0
        // waits and issues the copies).  Block-table entries come through two
        // 32-page windows in shared memory: window w (pages 32w .. 32w + 31,
        // page 32w + i copied by lane i with cp.async) is fetched while window
        // w - 1 is in use, so no page waits for a global load (a load per page
        // into a register would make the next page's read wait for it).
        //
        // Sparse decode: the gather warps fill the KV ring; this warp only
        // loads each request's Q tile.
        const uint64_t policy = policy_evict_first();
        const uint32_t q_bytes = nc * p.q_box_rows * 128;
        const bool sparse = p.sparse != 0;
        // Dense: the part's first page's block-table entry is read at once,
        // beside the first request's length, so page 0 waits for one load
        // instead of the first window's walk and its copy.  Used when the
        // cursor does start there (a part may begin on a request with no
        // blocks).
        const bool bt0_ok = !p.sparse && part.begin_req <= part.end_req &&
                            part.begin_block >= 0 && part.begin_block < p.max_blocks;
        const int bt0 = bt0_ok ? p.block_table[static_cast<int64_t>(part.begin_req / kvh) * p.bt_stride +
                                               part.begin_block]
                               : 0;
        Cursor ld = cursor_begin<kHeads>(p, part), ahead = ld;
        const bool direct0 = bt0_ok && ld.valid && ld.req == part.begin_req && ld.blk == part.begin_block;
        auto fetch_window = [&](uint32_t slot) {
            int rq = -1, bk = 0;
            for (int i = 0; i < 32 && ahead.valid; ++i) {
                if (lane == i) {
                    rq = ahead.req;
                    bk = ahead.blk;
                }
                cursor_next<kHeads>(p, part, ahead);
            }
            if (rq >= 0)
                cp_async_4(smem_u32(bt_win + 32 * slot + lane),
                           p.block_table + static_cast<int64_t>(rq / kvh) * p.bt_stride + bk);
            cp_async_commit();
        };
        uint32_t n_kv = 0, n_q = 0;
        // Q tile of request req (the whole tile, or its head-group slice).
        auto issue_q = [&](int req) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->q_full, q_bytes);
                if (!kHeads) {
                    for (int c = 0; c < nc; ++c)
                        tma_load_3d(&q_map, &bars->q_full, sQ + c * kChunkBytes, 64 * c,
                                    mtile * kTileM, req, policy);
                } else {
                    // map (576, grp, h_kv, s_q, b): the tile's rows s * grp + hh of
                    // head group j; a tile spans 64 / grp tokens, or one token's
                    // 64-head slice when grp > 64.
                    const int per_s = grp > kTileM ? grp / kTileM : 1;
                    const int hh0 = grp > kTileM ? (mtile % per_s) * kTileM : 0;
                    const int s0 = grp > kTileM ? mtile / per_s : mtile * (kTileM / grp);
                    for (int c = 0; c < kChunks; ++c)
                        tma_load_5d(&q_map, &bars->q_full, sQ + c * kChunkBytes, 64 * c, hh0,
                                    req % kvh, s0, req / kvh, policy);
                }
            }
            __syncwarp();
            ++n_q;
        };
        if (ld.valid) issue_q(ld.req);
        if (!sparse && !direct0) fetch_window(0);
        while (ld.valid) {
            if (!sparse) {
                // Window (g / 32) has landed: the first waits for its only
                // group (for both windows' groups, minus the second, when page
                // 0 came direct), later ones leave the next window's group
                // pending.
                int page = bt0;
                if (!(direct0 && ld.g == 0)) {
                    if (ld.g == 0)
                        cp_async_wait_group<0>();
                    else if ((ld.g & 31) == 0 || (direct0 && ld.g == 1))
                        cp_async_wait_group<1>();
                    __syncwarp();
                    page = bt_win[32 * ((ld.g >> 5) & 1) + (ld.g & 31)];
                }
                const int st = ld.g & 1;
                if (ld.g >= 2 && !warp_wait(&bars->kv_empty[st], ((ld.g >> 1) + 1) & 1, wc)) break;
                if (lane == 0) {
                    uint8_t* dst = sKV + st * kStageBytes;
                    if (kFp8) {
                        // One copy of the page's raw rows; a page outside the
                        // cache is not read and dequantises to zeros (as the
                        // bf16 path's out-of-range tile reads zeros).
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
                        mbar_arrive_expect_tx(&bars->kv_full[st], nc * kChunkBytes);
                        if (!kHeads) {
                            for (int c = 0; c < nc; ++c)
                                tma_load_3d(&kv_map, &bars->kv_full[st], dst + c * kChunkBytes,
                                            64 * c, 0, page, policy);
                        } else {  // map (576, h_kv, 64, pages): this request's cache head
                            for (int c = 0; c < kChunks; ++c)
                                tma_load_4d(&kv_map, &bars->kv_full[st], dst + c * kChunkBytes,
                                            64 * c, ld.req % kvh, 0, page, policy);
                        }
                    }
                }
                __syncwarp();
                ++n_kv;
            }
            // First block of a request: its Q tile (the part's first one went
            // out before the loop).
            if (ld.blk == ld.b0 && ld.g > 0) {
                if (!warp_wait(&bars->q_empty, (ld.item - 1) & 1, wc)) break;
                issue_q(ld.req);
            }
            // After page 0: the first window (when page 0 came direct) and the
            // second; after the last page of window w: window w + 2 into w's
            // slot (every lane has read its entry).
            if (!sparse) {
                if (ld.g == 0) {
                    if (direct0) fetch_window(0);
                    fetch_window(1);
                }
                else if ((ld.g & 31) == 31)
                    fetch_window((ld.g >> 5) & 1);
            }
            cursor_next<kHeads>(p, part, ld);
        }
        cp_async_wait_all();
        // Drain: never leave the CTA with copies still landing in its smem.
        if (lane == 0) {
            for (uint32_t k = (n_kv >= 2 ? n_kv - 2 : 0); k < n_kv; ++k)
                mbar_drain(kFp8 ? &bars->raw_full[k & 1] : &bars->kv_full[k & 1], (k >> 1) & 1,
                           kDrainBudgetNs);
            if (n_q > 0) mbar_drain(&bars->q_full, (n_q - 1) & 1, kDrainBudgetNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        // Two cursors: QK^T of block g needs its page, its request's Q tile
        // and a free S buffer; PV of block g needs P(g) from the softmax warps
        // (and, on a request's first block, O released by the previous
        // request's epilogue).  The whole warp runs this loop in step: lane 0
        // probes the barriers without blocking and broadcasts what it saw, and
        // one elected thread issues each burst and its commits.  (An isolated
        // probe had found single-thread issue ~1.5x slower per MMA than one
        // elect.sync per MMA; in the kernel, one elect per burst together with
        // fence-free barrier arrivals measured 4-12% faster.)
        // QK^T goes out in one burst of 36 MMAs once its page is in: splitting
        // it into turns with a check for a ready PV between them (so that a
        // PV never waits behind a whole QK^T) measured 4-19% slower, because
        // the checks stretched how long each stage is held.
        constexpr uint32_t idesc_pv = idesc_bf16_f32(64, 256, false, true);
        // Descriptors are built once; an MMA's operand then differs only in
        // the start-address field (bits 0..13, 16-byte units), which a plain
        // add moves without carrying into the next field (every address here
        // is below 256 KB).
        const uint64_t dQ = smem_desc(smem_u32(sQ), 16, 1024);
        const uint64_t dK0 = smem_desc(smem_u32(sKV), 16, 1024);
        const uint64_t dK1 = smem_desc(smem_u32(sKV + kStageBytes), 16, 1024);
        const uint64_t dV0 = smem_desc(smem_u32(sKV), kChunkBytes, 1024);
        const uint64_t dV1 = smem_desc(smem_u32(sKV + kStageBytes), kChunkBytes, 1024);
        // P(g): page g's RoPE chunk (dead once QK^T(g) is done) when
        // kStageP, else the one P buffer.
        const uint64_t dP0 = smem_desc(smem_u32(kStageP ? sKV + 8 * kChunkBytes : sP), 16, 1024);
        const uint64_t dP1 =
            smem_desc(smem_u32(kStageP ? sKV + kStageBytes + 8 * kChunkBytes : sP), 16, 1024);
        const uint32_t tS0 = tmem + kColS, tS1 = tmem + kColS + 32;
        const uint32_t tO0 = tmem + kColO, tO1 = tmem + kColO + 128;
        constexpr uint64_t kChunkUnits = kChunkBytes >> 4;
        Cursor qk = cursor_begin<kHeads>(p, part), pv = qk;
        uint64_t idle_since = 0;
        uint32_t idle_spins = 0;
        const bool leader = lane == 0;
        while (pv.valid) {
            bool did = false;
            if (pv.g < qk.g) {
                const bool first = pv.blk == pv.b0;
                bool ready = false;
                if (leader) {
                    ready = mbar_test_wait(&bars->p_full[pv.g & 1], (pv.g >> 1) & 1);
                    if (ready && first && pv.item > 0)
                        ready = mbar_test_wait(&bars->o_free, (pv.item - 1) & 1);
                }
                ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
                if (ready) {
                    tc_fence_after();
                    const uint64_t bV = (pv.g & 1) ? dV1 : dV0;
                    const uint64_t dP = (pv.g & 1) ? dP1 : dP0;
                    const uint32_t acc0 = first ? 0u : 1u;
                    // One elected thread issues the burst and commits it.
                    if (elect_one()) {
                        if (!kGen) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint32_t acc = kk ? 1u : acc0;
                                mma_ws_ss(tO0, dP + 2 * kk, bV + 128 * kk, idesc_pv, acc);
                                mma_ws_ss(tO1, dP + 2 * kk, bV + 4 * kChunkUnits + 128 * kk,
                                          idesc_pv, acc);
                            }
                        } else {
                            // V chunks in groups of 4, 2 or 1 (N = 256, 128,
                            // 64): group [cs, cs + n) writes TMEM columns
                            // 32 cs .. 32 (cs + n) (dims 64 cs + [0, 32 n) in
                            // lanes 0..63, 64 cs + [32 n, 64 n) in 64..127).
                            for (int cs = 0; cs < nv;) {
                                const int n = nv - cs >= 4 ? 4 : (nv - cs >= 2 ? 2 : 1);
                                const uint32_t idesc_g = idesc_bf16_f32(64, 64 * n, false, true);
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    mma_ws_ss(tmem + kColO + 32 * cs, dP + 2 * kk,
                                              bV + cs * kChunkUnits + 128 * kk, idesc_g,
                                              kk ? 1u : acc0);
                                cs += n;
                            }
                        }
                        mma_commit(&bars->pv_done[pv.g & 1]);
                        mma_commit(&bars->kv_empty[pv.g & 1]);
                    }
                    __syncwarp();
                    cursor_next<kHeads>(p, part, pv);
                    did = true;
                }
            }
            if (qk.valid) {
                const int st = qk.g & 1;
                bool ready = true;
                if (leader) {
                    if (qk.blk == qk.b0) ready = mbar_test_wait(&bars->q_full, qk.item & 1);
                    ready = ready && mbar_test_wait(&bars->kv_full[st], (qk.g >> 1) & 1);
                    if (ready && qk.g >= 2)
                        ready = mbar_test_wait(&bars->s_empty[st], ((qk.g >> 1) + 1) & 1);
                }
                ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
                if (ready) {
                    tc_fence_after();
                    const uint64_t bK = st ? dK1 : dK0;
                    const uint32_t d = st ? tS1 : tS0;
                    if (elect_one()) {
                        if (!kGen) {
                            issue_qk_turn<0>(dQ, bK, d);
                            issue_qk_turn<3>(dQ, bK, d);
                            issue_qk_turn<6>(dQ, bK, d);
                        } else {
                            constexpr uint32_t idesc_qk = idesc_bf16_f32(64, 64, false, false);
                            for (int c = 0; c < nc; ++c)
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    mma_ws_ss(d, dQ + c * kChunkUnits + 2 * kk,
                                              bK + c * kChunkUnits + 2 * kk, idesc_qk,
                                              (c + kk) ? 1u : 0u);
                        }
                        mma_commit(&bars->s_full[st]);
                        if (qk.blk == qk.b1 - 1) mma_commit(&bars->q_empty);
                    }
                    __syncwarp();
                    cursor_next<kHeads>(p, part, qk);
                    did = true;
                }
            }
            if (did) {
                idle_since = 0;
                idle_spins = 0;
                continue;
            }
            // Nothing ready: back off briefly.  This warp shares its SM
            // sub-partition with a softmax warp, and a hot polling loop would
            // take that warp's issue slots.
            if (kIdleSleepNs > 0) __nanosleep(kIdleSleepNs);
            if ((++idle_spins & 63) == 0) {
                bool stop = false;
                if (leader) {
                    if (*abort_flag) {
                        stop = true;
                    } else {
                        const uint64_t now = globaltimer_ns();
                        if (idle_since == 0) {
                            idle_since = now;
                        } else if (now - idle_since > p.budget_ns) {
                            raise_error(wc, MLA_ERR_DEVICE_TIMEOUT);
                            stop = true;
                        }
                    }
                }
                if (__shfl_sync(0xffffffffu, stop ? 1 : 0, 0)) break;
            }
        }
        // Drain: all MMAs finished before TMEM is released.
        if (elect_one()) mma_commit(&bars->drain);
        __syncwarp();
        if (leader) mbar_drain(&bars->drain, 0, kDrainBudgetNs);
        __syncwarp();
    } else if (warp >= kGatherWarp0) {
        // ------------------------------------------- sparse-decode row gather
        // Warps 6, 7 fill the stage of even pages, warps 8, 9 that of odd
        // pages, so two pages are in flight.  A page is the next 64 entries of
        // the request's key list; eight threads copy one cache row (nine
        // 128-byte lines, one 16-byte piece of each per thread) into the
        // page's row of every 64-dim chunk, in the 128-byte-swizzled layout
        // the MMAs read.  Entries that are padding, past the list or outside
        // the cache fill their row with zeros and lose their bit in the key
        // mask.  Each thread waits for its own copies and fences them for the
        // tensor core before its warp arrives on kv_full.
        if (p.sparse) {
            const int gw = warp - kGatherWarp0;
            const int grp = gw >> 1, wl = gw & 1;
            const int tl = 32 * wl + lane;
            const int uu = tl & 7, tb = tl >> 3;  // 16-byte piece; rows tb + 8 j
            const int64_t tok_bytes = p.kv_token_bytes;
            int cur[8], nxt[8];
            auto load_rows = [&](int (&d)[8], const Cursor& c) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = c.blk * kPage + tb + 8 * j;
                    d[j] = (c.valid && t < c.L) ? p.indices[static_cast<int64_t>(c.req) * p.topk + t]
                                                : -1;
                }
            };
            auto skip2 = [&](Cursor& c) {
                if (c.valid) cursor_next<kHeads>(p, part, c);
                if (c.valid) cursor_next<kHeads>(p, part, c);
            };
            Cursor c = cursor_begin<kHeads>(p, part);
            if (grp == 1 && c.valid) cursor_next<kHeads>(p, part, c);
            load_rows(cur, c);
            while (c.valid) {
                const int st = c.g & 1;  // == grp
                Cursor n2 = c;
                skip2(n2);
                load_rows(nxt, n2);  // this group's next page, used one turn later
                if (c.g >= 2 && !warp_wait(&bars->kv_empty[st], ((c.g >> 1) + 1) & 1, wc)) break;
                uint8_t* stage = sKV + st * kStageBytes;
                uint64_t mask = 0;
                bool bad = false;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int ix = cur[j];
                    const bool v = ix >= 0 && static_cast<int64_t>(ix) < p.num_tokens;
                    bad |= static_cast<int64_t>(ix) >= p.num_tokens;
                    const uint8_t* src =
                        p.kv_bytes + (v ? static_cast<int64_t>(ix) * tok_bytes : 0) + uu * 16;
                    const uint32_t dst = smem_u32(stage + sw128_offset(tb + 8 * j, uu));
                    const uint32_t n = v ? 16u : 0u;
#pragma unroll
                    for (int ch = 0; ch < kChunks; ++ch)
                        cp_async_16(dst + ch * kChunkBytes, src + ch * 128, n);
                    // rows 4 wl + q + 8 j (q = lane / 8) of this warp
                    const uint32_t b = __ballot_sync(0xffffffffu, v);
                    const uint64_t bits = (b & 1u) | ((b >> 7) & 2u) | ((b >> 14) & 4u) | ((b >> 21) & 8u);
                    mask |= bits << (4 * wl + 8 * j);
                }
                if (bad) atomicCAS(p.error_word, 0, MLA_ERR_BAD_INDEX);
                cp_async_wait_all();
                fence_proxy_async_smem();
                if (lane == 0) key_part[2 * st + wl] = mask;
                warp_arrive(&bars->kv_full[st]);
#pragma unroll
                for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
                skip2(c);
            }
        } else if (kFp8) {
            // ---------------------------------------- FP8 page dequantisation
            // In place, two threads per row (mla_fp8.cuh); the four warps
            // agree on every exit through bar.red.and before the named
            // barrier inside the routine.
            const int dt = tid - 32 * kGatherWarp0;
            for (Cursor c = cursor_begin<kHeads>(p, part); c.valid; cursor_next<kHeads>(p, part, c)) {
                const int st = c.g & 1;
                const bool ok = warp_wait(&bars->raw_full[st], (c.g >> 1) & 1, wc);
                if (!named_bar_and(kDequantBar, 128, ok)) break;
                fp8_dequant_page(sKV + st * kStageBytes, dt, raw_bad[st] != 0, kDequantBar);
                fence_proxy_async_smem();
                warp_arrive(&bars->kv_full[st]);
            }
        }
    } else if (warp >= 2) {
        // ------------------------------------- softmax / correction / epilogue
        const int q4 = warp & 3;
        const int Lrow = 32 * q4 + lane;  // TMEM lane
        const int r = Lrow & 63, half = Lrow >> 6;
        const int row = mtile * kTileM + r;
        const bool row_valid = row < p.R;
        const int s_idx = row / grp;  // query token (dense; causal limit)
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
        uint32_t gblk = 0, n_items = 0, xseq = 0;
        bool alive = true;
        for (int req = part.begin_req; req <= part.end_req && alive; ++req) {
            int L, nb, b0, b1;
            item_range<kHeads>(p, part, req, L, nb, b0, b1);
            int lim = L;
            if (p.causal) {
                lim = L - p.s_q + s_idx + 1;
                lim = lim < 0 ? 0 : (lim > L ? L : lim);
            }
            const int first_piece = p.num_splits[req];
            const bool split = (p.num_splits[req + 1] - first_piece) > 1;
            const int slot = (req == part.begin_req) ? part.begin_split : first_piece;
            float m_used = -INFINITY, l_part = 0.f;
            for (int blk = b0; blk < b1; ++blk, ++gblk) {
                const int st = gblk & 1;
                if (!warp_wait(&bars->s_full[st], (gblk >> 1) & 1, wc)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                uint32_t sv[32];
                tmem_ld32(tl + kColS + 32 * st, sv);
                tmem_ld_wait();
                tc_fence_before();
                warp_arrive(&bars->s_empty[st]);

                // Keys of this thread's 32 columns: the first lim - t0 of
                // them (dense), or the stage's key mask (sparse; the page's
                // kv_full phase completed before its S, so the wait is a
                // formality that orders the mask read).
                uint32_t keys;
                if (p.sparse) {
                    if (!warp_wait(&bars->kv_full[st], (gblk >> 1) & 1, wc)) {
                        alive = false;
                        break;
                    }
                    keys = static_cast<uint32_t>((key_part[2 * st] | key_part[2 * st + 1]) >>
                                                 (32 * half));
                } else {
                    const int n = lim - (blk * kPage + 32 * half);
                    keys = n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : (1u << n) - 1u);
                }
                float x[32];
                float hmax = -INFINITY;
                const uint64_t sc2 = f32x2_splat(p.scale_log2);
                // Pages every valid row of the warp sees whole skip the masking.
                // (Rows past the tile then hold scores of padding query rows:
                // they only feed their own output rows, which are never
                // written, and are left out of the rescale vote.)
                if (__all_sync(0xffffffffu, !row_valid || keys == 0xffffffffu)) {
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
                        x[c] = ((keys >> c) & 1u) ? a0 : -INFINITY;
                        x[c + 1] = ((keys >> (c + 1)) & 1u) ? a1 : -INFINITY;
                        hmax = fmaxf(hmax, fmaxf(x[c], x[c + 1]));
                    }
                }
                float pmax;
                if (!pair_exchange(xch, Lrow, xseq, hmax, pmax, wc)) {
                    alive = false;
                    break;
                }
                const float tmax = fmaxf(hmax, pmax);
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

                // With P in page g's own RoPE chunk (kStageP), only a
                // rescale of O has to wait for PV(g - 1); otherwise the wait
                // is for PV(g - 2): PV may trail by at most two pages, which
                // keeps the parity waits on the two pv_done barriers
                // unambiguous.  With the one P buffer, P(g) waits for PV(g - 1).
                const bool rescale = __any_sync(0xffffffffu, need && row_valid && blk > b0);
                const uint32_t lag = (kStageP && !rescale) ? 2u : 1u;
                if (gblk >= lag) {
                    const uint32_t w = gblk - lag;
                    if (!warp_wait(&bars->pv_done[w & 1], (w >> 1) & 1, wc)) {
                        alive = false;
                        break;
                    }
                }
                tc_fence_after();
                if (rescale) {
                    const float a = (need && blk > b0) ? alpha : 1.f;
#pragma unroll 1
                    for (int cg = 0; cg < nv; ++cg) {
                        uint32_t o[32];
                        tmem_ld32(tl + kColO + 32 * cg, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                        tmem_st32(tl + kColO + 32 * cg, o);
                    }
                    tmem_st_wait();
                }
                // Last page of the sequence: zero the V rows past its length so
                // stale slots (even NaN) cannot reach P.V through 0 * x.
                // (Sparse pages: rows without a key were filled with zeros.)
                if (!p.sparse && blk == nb - 1 && (L & (kPage - 1)) != 0) {
                    const int tail0 = L & (kPage - 1);
                    const int per_chunk = (kPage - tail0) * 8;  // 16-byte units
                    uint8_t* stage = sKV + st * kStageBytes;
                    for (int i = tid - 64; i < nv * per_chunk; i += 128) {
                        const int c = i / per_chunk, u = i % per_chunk;
                        reinterpret_cast<uint4*>(stage + c * kChunkBytes + tail0 * 128)[u] =
                            make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t off = sw128_offset(r, 4 * half + k);
                    *reinterpret_cast<uint4*>(
                        (kStageP ? sKV + st * kStageBytes + 8 * kChunkBytes : sP) + off) =
                        make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                warp_arrive(&bars->p_full[st]);
            }
            if (!alive) break;

            // ---------------------------------------------------- epilogue
            const bool has_blocks = b1 > b0;
            float l_tot = 0.f;
            if (has_blocks) {
                const uint32_t w = gblk - 1;
                if (!warp_wait(&bars->pv_done[w & 1], (w >> 1) & 1, wc)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                float l_other;
                if (!pair_exchange(xch, Lrow, xseq, l_part, l_other, wc)) {
                    alive = false;
                    break;
                }
                l_tot = l_part + l_other;
            }
            const bool empty = !(l_tot > 0.f);
            const float inv = empty ? 0.f : 1.f / l_tot;
            const float lse2 = empty ? -INFINITY : m_used + fast_log2(l_tot);
            const int64_t acc_row = static_cast<int64_t>(slot) * p.R + row;
            const OutMap om = out_map(req, row, p.h_q, p.s_q, p.fold, kvh, grp, p.out_sb,
                                      p.out_ss, p.out_sh);
            if (has_blocks) {
#pragma unroll 1
                for (int cg = 0; cg < nv; ++cg) {
                    uint32_t o[32];
                    tmem_ld32(tl + kColO + 32 * cg, o);
                    tmem_ld_wait();
                    // This thread's 32 dims of TMEM columns 32 cg .. 32 cg + 31
                    // (the PV groups of the MMA issuer: 4, 4 chunks for 512).
                    int dv0 = 256 * (cg >> 2) + 128 * half + 32 * (cg & 3);
                    if (kGen) {
                        for (int cs = 0;;) {
                            const int n = nv - cs >= 4 ? 4 : (nv - cs >= 2 ? 2 : 1);
                            if (cg < cs + n) {
                                dv0 = 64 * cs + 32 * n * half + 32 * (cg - cs);
                                break;
                            }
                            cs += n;
                        }
                    }
                    if (!row_valid) continue;
                    if (split) {
                        float4* dst = reinterpret_cast<float4*>(p.oaccum + acc_row * dv + dv0);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv,
                                                 __uint_as_float(o[4 * v + 1]) * inv,
                                                 __uint_as_float(o[4 * v + 2]) * inv,
                                                 __uint_as_float(o[4 * v + 3]) * inv);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(p.out + om.out_off + dv0);
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
                }
                tc_fence_before();
                warp_arrive(&bars->o_free);
                ++n_items;
            } else if (row_valid) {
                if (split) {
                    float4* dst = reinterpret_cast<float4*>(p.oaccum + acc_row * dv);
                    for (int v = 0; v < dv / 8; ++v) dst[v * 2 + half] = make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + om.out_off);
                    for (int v = 0; v < dv / 16; ++v) dst[v * 2 + half] = make_uint4(0, 0, 0, 0);
                }
            }
            if (row_valid && half == 0) {
                if (split)
                    p.lseaccum[acc_row] = lse2;
                else
                    p.lse[om.lse_idx] = empty ? -INFINITY : lse2 * 0.69314718055994531f;
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& q_map,
                          const CUtensorMap& kv_map, cudaStream_t stream) {
    // The instantiations a launch can pick: P placement x {bf16, FP8, bf16
    // with several cache heads, bf16 with other head sizes} (FP8 and other
    // head sizes have one cache head).
    using Kernel = void (*)(DecodeParams, CUtensorMap, CUtensorMap);
    static const Kernel kernels[2][4] = {
        {decode_kernel<false, false, false>, decode_kernel<false, true, false>,
         decode_kernel<false, false, true>, decode_kernel<false, false, false, true>},
        {decode_kernel<true, false, false>, decode_kernel<true, true, false>,
         decode_kernel<true, false, true>, decode_kernel<true, false, false, true>}};
    static int configured_mask = 0;  // per-device "smem attribute set" bits (first 31 devices)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 31 || !(configured_mask & (1 << dev))) {
        for (int sp = 0; sp < 2; ++sp)
            for (int m = 0; m < 4; ++m) {
                e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kernels[sp][m]),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sp ? kSmemBytes : kSmemBytesP));
                if (e != cudaSuccess) return e;
            }
        if (dev < 31) __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_RELAXED);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_mtiles, p.num_parts, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = p.stage_p ? kSmemBytes : kSmemBytesP;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // (nc = nv = 0: the 576 / 512 sizes every other call uses.)
    const bool general = (p.nc != 0 && p.nc != kChunks) || (p.nv != 0 && p.nv != kDv / 64);
    const int mode = p.fp8 ? 1 : (p.kvh > 1 ? 2 : (general ? 3 : 0));
    return cudaLaunchKernelEx(&cfg, kernels[p.stage_p ? 1 : 0][mode], p, q_map, kv_map);
}

}  // namespace mla
