// mla_decode_duo.cu -- split-KV paged MLA decode for query tiles of 128 rows on
// a CTA pair (2-CTA cluster, tcgen05 cta_group::2), for sm_103a.
//
// Sources (web pages, cited by title and section):
//   [Overview] "[DeepSeek-3] FlashMLA：把 MLA 的 KV Cache 优势变成 GPU 吞吐":
//       sec. 3 (one 576-dim cache row is K; its first 512 dims are V),
//       sec. 4 (paged KV through block_table), sec. 6 (split-KV partials),
//       sec. 7 (online softmax makes the partials mergeable).
//   [Rails] "Blackwell 多轨矩乘(multi-rail GEMM):FlashMLA 如何用一条 MMA 算完两路
//       QK": sec. 2.1-2.3 (the two lane groups hold different feature dims of
//       Q, each multiplies its own half of B, and the partial scores are added
//       after the MMA), sec. 4.3 (the 128-head configuration runs the same
//       idea on the 2-CTA form, whose M=128 layout is also a 2x2 datapath).
//   [DeepDive] "FlashMLA 新内核深度解析：Seesaw 调度、细粒度 TMA 流水线与 H800
//       上的 660 TFlops MLA 解码": 64x64 TMA copies of a K tile, EVICT_FIRST,
//       the exp -> exp2 rewrite, "Programmatic Dependent Launch", "Tile
//       Scheduler" (each SM part walks its DecodingSchedMeta).
//   [AttnBook] "3.4 Attention kernel": "在线 softmax", 代码 (causal mask).
//
// Why a pair.  A 64-row tile reads every K/V byte out of shared memory once
// per 64 query rows; at the tensor core's 128 bytes per clock of operand
// fetch that is exactly the MMA rate, with nothing left for Q, so QK^T runs
// near half rate.  With cta_group::2 and M = 128 one MMA feeds 128 rows (64
// per CTA) from each K/V byte, and each CTA loads only half of every page.
//
// How the page is split.  Both CTAs hold the same 64 tokens of a page, split
// by head dims into 64-dim chunks: the leader (rank 0) chunks 0, 1, 4, 5 and
// the RoPE chunk 8, the peer (rank 1) chunks 2, 3, 6, 7, each in slots 0..3 of
// the same stage offset (slot 4: the leader's RoPE chunk; zeros in the peer).
//   - PV (N = 256 per MMA, V MN-major): TMEM lanes 0..63 receive the columns
//     computed from the leader's slots, lanes 64..127 those from the peer's,
//     so with slots {2h, 2h+1} the two MMAs write O[rows, 256h + (0..127)] to
//     lanes 0..63 and O[rows, 256h + 128 + (0..127)] to lanes 64..127 -- O
//     [64 x 512] fp32 per CTA in 256 columns.
//   - QK^T (N = 128): Q's chunks 0, 1, 4, 5 sit in TMEM lanes 0..63 and its
//     chunks 2, 3, 6, 7 in lanes 64..127 (A read from TMEM, 128 columns); one
//     TS MMA per 16 dims gives lanes 0..63 the partial scores over the
//     leader's dims and lanes 64..127 those over the peer's dims, for all 64
//     tokens (the multi-rail form of [Rails] sec. 2).  The RoPE dims are four
//     SS MMAs with Q's RoPE chunk from shared memory against slot 4: the
//     peer's zeros leave lanes 64..127 unchanged.  The softmax adds the two
//     partial scores of each (row, token).
// Tensor memory: O 0..255, Q 256..383, S 384..511 (two buffers of 64).
//
// Pipeline.  Each CTA's producer loads its half of every page into a ring of
// five 40 KB stages, preceded by two pseudo-pages per request that carry its
// 64 query rows (chunks 0, 1, 4, 5, 8 and 2, 3, 6, 7).  The peer's otherwise
// idle MMA warp forwards "my half has landed" to the leader (a remote
// mbarrier arrive); the leader's QK^T and PV warps issue the MMAs for both
// CTAs and commit to barriers in both.  Eight softmax warps per CTA (two per SM
// sub-partition) each take 16 tokens of a row: warp w reads TMEM lane quadrant
// w % 4 (rows and rail) and token half w / 4.  P goes into slot 4 of the
// page's stage, which QK^T is done with (the peer's producer zeroes it again
// before the stage's next page).  The peer's softmax warps signal the leader's
// issuers with relaxed remote arrivals, one per warp and page (measured: a
// relay warp forwarding one arrival per page made the MTP step 12% and the
// ragged h_q 128 step 7% slower).  Every wait is
// bounded; after a timeout the softmax warps still pass every named barrier,
// and the two CTAs meet at a cluster barrier before tensor memory is freed.
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

namespace {

constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kPvWarp = 10;  // the leader's PV issuer (idle in the peer)
constexpr int kThreads = 352;
constexpr int kGatherWarp0 = 11;      // sparse decode: warps 11..14 gather rows
constexpr int kThreadsSparse = 480;
constexpr int kPairRows = 128;  // query rows of one CTA pair
constexpr int kCtaRows = 64;    // rows of one CTA
constexpr int kStages = 5;
constexpr int kSlots = 5;  // four latent chunks and the RoPE / P slot
constexpr uint32_t kSlotBytes = kChunkBytes;           // [64 rows][64 dims] bf16
constexpr uint32_t kStageBytes = kSlots * kSlotBytes;  // 40960
constexpr uint32_t kOffRing = 0;
constexpr uint32_t kOffQr = kOffRing + kStages * kStageBytes;  // Q's RoPE chunk (SS A operand)
constexpr uint32_t kOffX = kOffQr + kSlotBytes;  // partial-score exchange: float4 [2][2][4][64]
constexpr uint32_t kXBytes = 2 * 2 * 4 * 64 * 16;
constexpr uint32_t kOffM = kOffX + kXBytes;  // row max / row sum exchange: float [2][4][64]
constexpr uint32_t kMBytes = 2 * 4 * 64 * 4;
constexpr uint32_t kOffBar = kOffM + kMBytes;
constexpr uint32_t kOffMisc = kOffBar + 256;
constexpr uint32_t kOffBt = kOffMisc + 64;  // block-table windows: int32 [2][32]
constexpr uint32_t kSmemBytes = kOffBt + 256;
static_assert(kOffQr % 1024 == 0 && kOffX % 16 == 0, "operand alignment");
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
static_assert(kSmemBytes < (1u << 18), "descriptor address arithmetic assumes < 256 KB");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColQ = 256;
constexpr uint32_t kColS = 384;
constexpr float kLazyThreshold = 8.0f;  // log2 units (factor 256)
constexpr uint64_t kDrainBudgetNs = 2000000000ull;
constexpr uint16_t kBothCtas = 3;
constexpr uint16_t kLeaderCta = 1;
constexpr int kRopeChunk = 8;
// Named barriers of the softmax warps (0 is __syncthreads).
constexpr uint32_t kBarRowGroup0 = 1;  // +0 / +1: the four warps of rows 0..31 / 32..63
constexpr uint32_t kBarSoftmax = 3;    // all eight softmax warps
constexpr uint32_t kBarPair0 = 4;      // +0..3: the two warps of the same rows and token half
constexpr uint32_t kSoftmaxThreads = 256;

// 64-dim chunk of a 576-dim row in slot s (0..3) of the given rail: rail 0
// (the leader's half, TMEM lanes 0..63) 0, 1, 4, 5; rail 1 2, 3, 6, 7.
__device__ __forceinline__ int rail_chunk(int rail, int s) { return (s >> 1) * 4 + rail * 2 + (s & 1); }

struct Barriers {
    uint64_t kv_full[kStages];   // this CTA's copies of a ring entry landed
    uint64_t kv_peer[kStages];   // leader: the peer's half of a page landed
    uint64_t kv_empty[kStages];  // this CTA's stage may be refilled
    uint64_t s_full[2];          // S of a page is in this CTA's TMEM
    uint64_t s_empty[2];         // leader: all 16 softmax warps have read S
    uint64_t p_full[2];          // leader: all 16 softmax warps wrote P (and rescaled O)
    uint64_t pv_done[2];         // PV of a page finished (both CTAs)
    uint64_t q_ready;            // leader: both CTAs copied a request's Q
    uint64_t o_free;             // leader: all 16 softmax warps read O in the epilogue
    uint64_t drain;              // leader: every MMA of both issuers finished
    uint64_t q_copied;           // peer: its softmax warps copied a request's Q (entries landed)
};
static_assert(sizeof(Barriers) <= 256, "barrier block");

struct Part {
    int begin_req, end_req, begin_block, end_block, begin_split;
};

__device__ __forceinline__ int blocks_of(int L) { return L > 0 ? (L + kPage - 1) / kPage : 0; }

template <bool kSparse>
__device__ __forceinline__ void item_range(const DecodeParams& p, const Part& part, int req,
                                           int& L, int& nb, int& b0, int& b1) {
    L = kSparse ? p.topk : p.seqlens[req];
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

// Walk over the non-empty (request, block) pairs of a part.  The ring holds,
// for each request with blocks (item i), its two query pseudo-pages followed
// by its pages: page g of item i is ring entry g + 2 i + 2, the item's query
// entries g_first + 2 i and g_first + 2 i + 1.
struct Cursor {
    int req, blk, b0, b1, L, nb;
    uint32_t g, item;
    bool valid;
    __device__ __forceinline__ uint32_t ring() const { return g + 2 * item + 2; }
};
template <bool kSparse>
__device__ __forceinline__ void cursor_seek(const DecodeParams& p, const Part& part, Cursor& c,
                                            int req) {
    for (; req <= part.end_req; ++req) {
        item_range<kSparse>(p, part, req, c.L, c.nb, c.b0, c.b1);
        if (c.b1 > c.b0) {
            c.req = req;
            c.blk = c.b0;
            c.valid = true;
            return;
        }
    }
    c.valid = false;
}
template <bool kSparse>
__device__ __forceinline__ Cursor cursor_begin(const DecodeParams& p, const Part& part) {
    Cursor c;
    c.g = 0;
    c.item = 0;
    cursor_seek<kSparse>(p, part, c, part.begin_req);
    return c;
}
template <bool kSparse>
__device__ __forceinline__ void cursor_next(const DecodeParams& p, const Part& part, Cursor& c) {
    ++c.g;
    if (++c.blk < c.b1) return;
    ++c.item;
    cursor_seek<kSparse>(p, part, c, c.req + 1);
}

// Warp-uniform bounded wait (lane 0 polls; cluster-scope acquire, since some
// phases complete by arrivals from the other CTA).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& wc) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_cluster(bar, parity, wc, MLA_ERR_DEVICE_TIMEOUT);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}
// Warp-uniform bounded wait of the leader's issuer warps on barriers whose
// phases complete by remote arrivals from the peer.  It polls with the
// non-suspending test_wait and a short sleep: measured against the suspending
// try_wait on these barriers, the MTP step (batch 128, s_q 2, h_q 128, 4096
// tokens) took 320 instead of 343 us and the ragged h_q 128 step 104 instead
// of 108 us.
__device__ __forceinline__ bool warp_poll(uint64_t* bar, uint32_t parity, const WaitCtx& wc) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) {
        if (!mbar_test_wait_cluster(bar, parity)) {
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t spin = 1;; ++spin) {
                __nanosleep(32);
                if (mbar_test_wait_cluster(bar, parity)) break;
                if ((spin & 63) == 0) {
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
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}
// One arrival per warp on a barrier of the leader CTA (a remote arrival from
// the peer).  Relaxed: what the leader acts on is already complete (TMEM
// reads and stores waited for, shared-memory operands fenced for the tensor
// core by their writers).
__device__ __forceinline__ void warp_arrive_leader(uint64_t* bar, bool leader) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        if (leader)
            mbar_arrive(bar);
        else
            mbar_arrive_remote_relaxed(mapa_shared(smem_u32(bar), 0));
    }
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c,
                                             uint32_t& d) {
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr)
                 : "memory");
}

}  // namespace

template <bool kSparse>
__global__ void __launch_bounds__(kSparse ? kThreadsSparse : kThreads, 1)
    decode_duo_kernel(const __grid_constant__ DecodeParams p,
                      const __grid_constant__ CUtensorMap q_map,
                      const __grid_constant__ CUtensorMap kv_map) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int tile = blockIdx.x >> 1, part_idx = blockIdx.y;

    uint8_t* ring = smem + kOffRing;
    uint8_t* sQr = smem + kOffQr;
    float4* X = reinterpret_cast<float4*>(smem + kOffX);
    float* M = reinterpret_cast<float*>(smem + kOffM);
    Barriers* bars = reinterpret_cast<Barriers*>(smem + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    // Sparse decode: key_mask[stage] has bit t set when stage row t holds a
    // key (16 bits from each gather warp, written before its kv_full arrival).
    volatile uint64_t* key_mask = reinterpret_cast<volatile uint64_t*>(smem + kOffMisc + 16);
    volatile uint16_t* key_mask16 = reinterpret_cast<volatile uint16_t*>(smem + kOffMisc + 16);
    WaitCtx wc{abort_flag, p.error_word, p.budget_ns};

    // ------------------------------------------------------------ prologue
    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->kv_full[s], kSparse ? 4 : 1);
            mbar_init(&bars->kv_peer[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->s_full[b], 1);
            mbar_init(&bars->s_empty[b], 16);  // the softmax warps of both CTAs
            mbar_init(&bars->p_full[b], 16);
            mbar_init(&bars->pv_done[b], 1);
        }
        mbar_init(&bars->q_ready, 2);
        mbar_init(&bars->o_free, 16);
        mbar_init(&bars->drain, 2);  // the QK^T and PV issuers
        mbar_init(&bars->q_copied, 1);
        fence_barrier_init();
        prefetch_tensormap(&q_map);
        prefetch_tensormap(&kv_map);
    }
    // Tensor memory of both CTAs, allocated collectively (one warp of each).
    if (warp == kMmaWarp) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    // Both CTAs' barriers exist before any remote arrival or multicast commit.
    tc_fence_before();
    cluster_sync();
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
    if (tid == 0 && leader && !kSparse) {
        for (int req = part.begin_req; req <= part.end_req; ++req) {
            const int L = p.seqlens[req];
            if (L > 0 && blocks_of(L) > p.max_blocks) raise_error(wc, MLA_ERR_SEQ_TOO_LONG);
        }
    }

    if (kSparse && warp >= kGatherWarp0) {
        // ------------------------------------------- sparse: row gather
        // A page is the next 64 entries of a (request, query token)'s key
        // list.  Four warps, one on each SM sub-partition, gather this CTA's
        // chunks of the listed rows: warp gw takes rows 16 gw .. 16 gw + 15,
        // eight lanes per row, one 16-byte cp.async per chunk and lane, into
        // the page's stage in the 128-byte-swizzled layout the MMAs read.  A
        // warp waits for its own copies, fences them for the tensor core,
        // writes its 16 bits of the key mask and arrives on kv_full (four
        // arrivals a page).  Padding, entries past the list and positions
        // outside the cache read nothing (the row is zeros) and lose their
        // bit.  A page's list entries are fetched two pages ahead.  The query
        // pseudo-pages come by TMA, issued by warp 0 with the byte count; the
        // other warps arrive on them plainly.  Every warp takes the stages in
        // ring order, so each of its parity waits stays unambiguous, and
        // holds no unsignalled page while it waits.  (More pages in flight
        // per warp only lengthened each page's landing: random row reads
        // saturate the memory system first.)
        const int gw = warp - kGatherWarp0;
        const uint64_t policy = policy_evict_first();
        const int qrow0 = tile * kPairRows + static_cast<int>(rank) * kCtaRows;
        const int uu = lane & 7, rq = lane >> 3;
        const int n_ch = leader ? 5 : 4;
        const int64_t tok_bytes = p.kv_token_bytes;
        auto load_ix = [&](const Cursor& c) -> int {
            const int t = c.blk * kPage + 16 * gw + (lane & 15);
            return (c.valid && t < c.L) ? p.indices[static_cast<int64_t>(c.req) * p.topk + t] : -1;
        };
        auto acquire = [&](uint32_t n) -> bool {
            return n < kStages ||
                   warp_wait(&bars->kv_empty[n % kStages], ((n / kStages) + 1) & 1, wc);
        };
        Cursor ld = cursor_begin<true>(p, part);
        Cursor pf = ld;
        int ix_cur = load_ix(pf);
        if (pf.valid) cursor_next<true>(p, part, pf);
        int ix_next = load_ix(pf);
        uint32_t n_issued = 0;
        bool stop = false;
        while (ld.valid && !stop) {
            if (ld.blk == ld.b0) {
                for (int e = 0; e < 2; ++e) {
                    const uint32_t n = ld.ring() - 2 + e;
                    const uint32_t st = n % kStages;
                    if (!acquire(n)) {
                        stop = true;
                        break;
                    }
                    if (lane == 0) {
                        if (gw == 0) {
                            uint8_t* dst = ring + st * kStageBytes;
                            const int nl = e == 0 ? 5 : 4;
                            mbar_arrive_expect_tx(&bars->kv_full[st], nl * kSlotBytes);
                            for (int s = 0; s < nl; ++s)
                                tma_load_3d(&q_map, &bars->kv_full[st], dst + s * kSlotBytes,
                                            64 * (s == 4 ? kRopeChunk : rail_chunk(e, s)), qrow0,
                                            ld.req, policy);
                        } else {
                            mbar_arrive(&bars->kv_full[st]);
                        }
                    }
                    __syncwarp();
                    n_issued = n + 1;
                }
                if (stop) break;
            }
            const uint32_t n = ld.ring();
            const uint32_t st = n % kStages;
            if (!acquire(n)) break;
            uint8_t* stage = ring + st * kStageBytes;
            if (!leader) {
                // The peer's RoPE slot is zeros under a page (it held P or a
                // query entry before).
                uint4* z = reinterpret_cast<uint4*>(stage + 4 * kSlotBytes + 16 * gw * 128);
#pragma unroll
                for (int i = 0; i < 4; ++i) z[lane + 32 * i] = make_uint4(0u, 0u, 0u, 0u);
            }
            uint32_t mask = 0;
            bool bad = false;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // row 4 j + rq of this warp's rows: the entry of lane 4 j + rq
                const int ix = __shfl_sync(0xffffffffu, ix_cur, 4 * j + rq);
                const bool v = ix >= 0 && static_cast<int64_t>(ix) < p.num_tokens;
                bad |= static_cast<int64_t>(ix) >= p.num_tokens;
                const uint8_t* src = p.kv_bytes + (v ? static_cast<int64_t>(ix) * tok_bytes : 0) + uu * 16;
                const uint32_t dst = smem_u32(stage + sw128_offset(16 * gw + 4 * j + rq, uu));
                const uint32_t nbytes = v ? 16u : 0u;
                for (int s = 0; s < n_ch; ++s)
                    cp_async_16(dst + s * kSlotBytes,
                                src + 128 * (s == 4 ? kRopeChunk : rail_chunk(static_cast<int>(rank), s)),
                                nbytes);
                // rows 4 j .. 4 j + 3: the validity of lanes 0, 8, 16, 24
                const uint32_t b = __ballot_sync(0xffffffffu, v);
                mask |= ((b & 1u) | ((b >> 7) & 2u) | ((b >> 14) & 4u) | ((b >> 21) & 8u)) << (4 * j);
            }
            if (bad) atomicCAS(p.error_word, 0, MLA_ERR_BAD_INDEX);
            n_issued = n + 1;
            // The next page's entries are here; fetch the one after it.
            ix_cur = ix_next;
            if (pf.valid) cursor_next<true>(p, part, pf);
            ix_next = load_ix(pf);
            cursor_next<true>(p, part, ld);
            cp_async_wait_all();
            __syncwarp();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                key_mask16[4 * st + gw] = static_cast<uint16_t>(mask);
                mbar_arrive(&bars->kv_full[st]);
            }
            __syncwarp();
        }
        // Drain: the query entries' copies have landed before warp 0 leaves.
        if (gw == 0 && lane == 0)
            for (uint32_t k = (n_issued >= kStages ? n_issued - kStages : 0); k < n_issued; ++k)
                mbar_drain(&bars->kv_full[k % kStages], (k / kStages) & 1, kDrainBudgetNs);
        __syncwarp();
    } else if (warp == kProducerWarp) {
      if constexpr (!kSparse) {
        // ------------------------------------------------------ TMA producer
        // The whole warp walks the ring; lane 0 waits and issues the copies.
        // Block-table entries come through two 32-page windows in shared
        // memory: window w (pages 32w .. 32w + 31, page 32w + i copied by
        // lane i with cp.async) is fetched while window w - 1 is in use, so
        // no page waits for a global load (a load per page into a register
        // would make the next page's read wait for it).
        const uint64_t policy = policy_evict_first();
        const int qrow0 = tile * kPairRows + static_cast<int>(rank) * kCtaRows;
        const int n_kv = leader ? 5 : 4;
        int32_t* bt_win = reinterpret_cast<int32_t*>(smem + kOffBt);
        Cursor ld = cursor_begin<kSparse>(p, part), ahead = ld;
        auto fetch_window = [&](uint32_t slot) {
            int rq = -1, bk = 0;
            for (int i = 0; i < 32 && ahead.valid; ++i) {
                if (lane == i) {
                    rq = ahead.req;
                    bk = ahead.blk;
                }
                cursor_next<kSparse>(p, part, ahead);
            }
            if (rq >= 0)
                cp_async_4(smem_u32(bt_win + 32 * slot + lane),
                           p.block_table + static_cast<int64_t>(rq) * p.bt_stride + bk);
            cp_async_commit();
        };
        fetch_window(0);
        uint32_t n_issued = 0;
        bool stop = false;
        auto acquire = [&](uint32_t n) -> bool {
            return n < kStages ||
                   warp_wait(&bars->kv_empty[n % kStages], ((n / kStages) + 1) & 1, wc);
        };
        while (ld.valid && !stop) {
            if (ld.blk == ld.b0) {
                // The request's 64 query rows of this CTA: chunks 0, 1, 4, 5 and
                // the RoPE chunk, then chunks 2, 3, 6, 7.
                for (int e = 0; e < 2; ++e) {
                    const uint32_t n = ld.ring() - 2 + e;
                    const uint32_t st = n % kStages;
                    if (!acquire(n)) {
                        stop = true;
                        break;
                    }
                    if (lane == 0) {
                        uint8_t* dst = ring + st * kStageBytes;
                        const int nl = e == 0 ? 5 : 4;
                        mbar_arrive_expect_tx(&bars->kv_full[st], nl * kSlotBytes);
                        for (int s = 0; s < nl; ++s)
                            tma_load_3d(&q_map, &bars->kv_full[st], dst + s * kSlotBytes,
                                        64 * (s == 4 ? kRopeChunk : rail_chunk(e, s)), qrow0,
                                        ld.req, policy);
                    }
                    __syncwarp();
                    n_issued = n + 1;
                }
                if (stop) break;
            }
            // Window (g / 32) has landed: the first waits for its only group,
            // later ones leave the next window's group pending.
            if (ld.g == 0)
                cp_async_wait_group<0>();
            else if ((ld.g & 31) == 0)
                cp_async_wait_group<1>();
            __syncwarp();
            const int page = bt_win[32 * ((ld.g >> 5) & 1) + (ld.g & 31)];
            const uint32_t n = ld.ring();
            const uint32_t st = n % kStages;
            if (!acquire(n)) break;
            uint8_t* dst = ring + st * kStageBytes;
            if (!leader) {
                // The peer holds no RoPE dims: slot 4 must read as zeros in the
                // RoPE MMAs, whatever the stage's previous entry left there.
                uint4* z = reinterpret_cast<uint4*>(dst + 4 * kSlotBytes);
                for (int i = lane; i < static_cast<int>(kSlotBytes / 16); i += 32)
                    z[i] = make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->kv_full[st], n_kv * kSlotBytes);
                for (int s = 0; s < n_kv; ++s)
                    tma_load_3d(&kv_map, &bars->kv_full[st], dst + s * kSlotBytes,
                                64 * (s == 4 ? kRopeChunk : rail_chunk(static_cast<int>(rank), s)),
                                0, page, policy);
            }
            __syncwarp();
            n_issued = n + 1;
            // After page 0: the second window; after the last page of window
            // w: window w + 2 into w's slot (every lane has read its entry).
            if (ld.g == 0)
                fetch_window(1);
            else if ((ld.g & 31) == 31)
                fetch_window((ld.g >> 5) & 1);
            cursor_next<kSparse>(p, part, ld);
        }
        // Drain: no copy may still be landing when the CTA leaves.
        cp_async_wait_all();
        if (lane == 0)
            for (uint32_t k = (n_issued >= kStages ? n_issued - kStages : 0); k < n_issued; ++k)
                mbar_drain(&bars->kv_full[k % kStages], (k / kStages) & 1, kDrainBudgetNs);
        __syncwarp();
      }
    } else if (warp == kMmaWarp && !leader) {
        // ------------------------------------------- peer: landing forwarder
        // For every page the leader's MMAs will read, tell the leader that this
        // CTA's half has landed.  (Only pages: the query pseudo-pages are read
        // by this CTA's own softmax warps.)  A parity wait on a stage is
        // unambiguous only when the stage's previous entry is known to have
        // landed and its next one cannot have: a previous page was forwarded
        // here, and the query entries of a request are known to have landed
        // once the softmax warps copied them (q_copied, waited for before the
        // request's first page).  The next entry of a page's stage waits for
        // that page's PV, hence for this forwarding.
        for (Cursor c = cursor_begin<kSparse>(p, part); c.valid; cursor_next<kSparse>(p, part, c)) {
            const uint32_t n = c.ring();
            if (c.blk == c.b0 && !warp_wait(&bars->q_copied, c.item & 1, wc)) break;
            if (!warp_wait(&bars->kv_full[n % kStages], (n / kStages) & 1, wc)) break;
            if (lane == 0) mbar_arrive_remote_relaxed(mapa_shared(smem_u32(&bars->kv_peer[n % kStages]), 0));
            __syncwarp();
        }
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------- leader: QK^T issuer
        // QK^T of page g needs both halves of its page, the request's Q in
        // both CTAs and a free S buffer (both CTAs' softmax warps read S of
        // page g - 2).  One wait after another (a loop probing several
        // barriers in turn answered late); the barriers the peer completes are
        // polled (warp_poll).  One elected thread issues the burst and its
        // commit.
        constexpr uint32_t idesc_qk = idesc_bf16_f32(kPairRows, 128, false, false);
        constexpr uint64_t kStageUnits = kStageBytes >> 4, kSlotUnits = kSlotBytes >> 4;
        const uint64_t dK0 = smem_desc(smem_u32(ring), 16, 1024);
        const uint64_t dQr = smem_desc(smem_u32(sQr), 16, 1024);
        const uint32_t tQ = tmem + kColQ, tS = tmem + kColS;
        uint32_t peer_par = 0;  // bit s: parity of the next kv_peer[s] phase
        for (Cursor qk = cursor_begin<kSparse>(p, part); qk.valid; cursor_next<kSparse>(p, part, qk)) {
            const uint32_t n = qk.ring(), st = n % kStages;
            // (q_ready first: it also covers the landing of the request's
            // query entries, which share stages with its pages.)
            if (qk.blk == qk.b0 && !warp_poll(&bars->q_ready, qk.item & 1, wc)) break;
            if (!warp_wait(&bars->kv_full[st], (n / kStages) & 1, wc)) break;
            if (!warp_poll(&bars->kv_peer[st], (peer_par >> st) & 1, wc)) break;
            if (qk.g >= 2 && !warp_poll(&bars->s_empty[qk.g & 1], ((qk.g >> 1) + 1) & 1, wc)) break;
            tc_fence_after();
            const uint64_t bK = dK0 + st * kStageUnits;
            const uint32_t d = tS + 64 * (qk.g & 1);
            if (elect_one()) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    mma_pair_ts(d, tQ + 8 * j, bK + (j >> 2) * kSlotUnits + 2 * (j & 3), idesc_qk,
                                j ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_pair_ss(d, dQr + 2 * kk, bK + 4 * kSlotUnits + 2 * kk, idesc_qk, 1u);
                mma_commit_pair(&bars->s_full[qk.g & 1], kBothCtas);
            }
            __syncwarp();
            peer_par ^= 1u << st;
        }
        // Drain: every MMA finished before the CTAs meet at the final barrier.
        if (elect_one()) mma_commit_pair(&bars->drain, kLeaderCta);
        __syncwarp();
        if (lane == 0) mbar_drain(&bars->drain, 0, kDrainBudgetNs);
        __syncwarp();
    } else if (leader && warp == kPvWarp) {
        // ------------------------------------------------- leader: PV issuer
        // PV of page g needs P(g) from both CTAs' softmax warps (and, on a
        // request's first page, O released by the previous epilogue).  Its
        // commits free the page's stage in both CTAs (PV(g) finishes after
        // QK^T(g), issued earlier into the same tensor pipe).
        constexpr uint32_t idesc_pv = idesc_bf16_f32(kPairRows, 256, false, true);
        constexpr uint64_t kStageUnits = kStageBytes >> 4, kSlotUnits = kSlotBytes >> 4;
        const uint64_t dV0 = smem_desc(smem_u32(ring), kSlotBytes, 1024);
        const uint64_t dP0 = smem_desc(smem_u32(ring + 4 * kSlotBytes), 16, 1024);
        const uint32_t tO = tmem + kColO;
        for (Cursor pv = cursor_begin<kSparse>(p, part); pv.valid; cursor_next<kSparse>(p, part, pv)) {
            const bool first = pv.blk == pv.b0;
            if (!warp_poll(&bars->p_full[pv.g & 1], (pv.g >> 1) & 1, wc)) break;
            if (first && pv.item > 0 && !warp_poll(&bars->o_free, (pv.item - 1) & 1, wc)) break;
            tc_fence_after();
            const uint32_t st = pv.ring() % kStages;
            const uint64_t aP = dP0 + st * kStageUnits, bV = dV0 + st * kStageUnits;
            if (elect_one()) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_pair_ss(tO + 128 * hh, aP + 2 * kk, bV + 2 * hh * kSlotUnits + 128 * kk,
                                    idesc_pv, (first && kk == 0) ? 0u : 1u);
                mma_commit_pair(&bars->pv_done[pv.g & 1], kBothCtas);
                mma_commit_pair(&bars->kv_empty[st], kBothCtas);
            }
            __syncwarp();
        }
        if (elect_one()) mma_commit_pair(&bars->drain, kLeaderCta);
        __syncwarp();
        if (lane == 0) mbar_drain(&bars->drain, 0, kDrainBudgetNs);
        __syncwarp();
    } else if (warp < kProducerWarp) {
        // ------------------------------- softmax / correction / epilogue / Q copy
        // Every softmax warp runs the same sequence of named barriers whatever
        // happens: a wait that runs out (the CTA's abort flag is then set)
        // only marks the warp dead, after which it skips its waits and its
        // work but still passes every barrier, so no partner is left waiting.
        const int qd = warp & 3, h = warp >> 2;
        const int Lr = 32 * qd + lane;  // TMEM lane
        const int rho = Lr >> 6, r = Lr & 63;
        const int row = tile * kPairRows + static_cast<int>(rank) * kCtaRows + r;
        const bool row_valid = row < p.R;
        const int s_idx = row / p.h_q;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qd) << 16);
        const uint32_t row_bar = kBarRowGroup0 + (qd & 1);         // rows of this warp, 4 warps
        const uint32_t pair_bar = kBarPair0 + (qd & 1) + 2 * h;    // same rows and h, 2 warps
        const int stid = 32 * warp + lane;  // 0..255 among the softmax threads
        uint32_t gblk = 0, item = 0;
        bool alive = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (alive) alive = warp_wait(bar, parity, wc);
            return alive;
        };
        // Per-page signals to the leader's issuers: one arrival per warp,
        // remote (relaxed) from the peer.
        auto signal = [&](uint64_t* leader_bar) { warp_arrive_leader(leader_bar, leader); };
        // PV completions are observed in page order, and before P(g) is written
        // PV(g - 2) must be complete: a parity wait on pv_done[g & 1] is only
        // unambiguous when PV(g - 2) is known complete and PV(g + 2) cannot be
        // (it needs this warp's P(g + 2)).  This also keeps the softmax at
        // most two pages ahead of PV.
        uint32_t pv_seen = 0;  // PVs of pages < pv_seen observed complete
        auto wait_pv = [&](uint32_t upto) {
            for (; pv_seen < upto; ++pv_seen) wait(&bars->pv_done[pv_seen & 1], (pv_seen >> 1) & 1);
        };

        // Q of the request whose query entries start at ring entry nq: this
        // lane's rail chunks into its TMEM columns (two slots per warp half),
        // the RoPE chunk into its shared buffer.
        auto q_copy = [&](uint32_t nq) {
            const uint32_t sa = nq % kStages, sb = (nq + 1) % kStages;
            wait(&bars->kv_full[sa], (nq / kStages) & 1);
            wait(&bars->kv_full[sb], ((nq + 1) / kStages) & 1);
            // (Both waits are for all eight warps' copies: the barrier below
            // orders every warp's reads before the stages are released.)
            if (alive) {
                const uint8_t* src = ring + (rho ? sb : sa) * kStageBytes;
#pragma unroll 1
                for (int s = 2 * h; s < 2 * h + 2; ++s) {
                    uint32_t w[32];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        ld_shared_v4(smem_u32(src + s * kSlotBytes + sw128_offset(r, u)), w[4 * u],
                                     w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                    tmem_st32(tl + kColQ + 32 * s, w);
                }
                const uint4* rope =
                    reinterpret_cast<const uint4*>(ring + sa * kStageBytes + 4 * kSlotBytes);
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    reinterpret_cast<uint4*>(sQr)[2 * stid + k] = rope[2 * stid + k];
                tmem_st_wait();
                fence_proxy_async_smem();
            }
            tc_fence_before();
            named_bar_sync(kBarSoftmax, kSoftmaxThreads);
            if (stid == 0) {
                mbar_arrive(&bars->kv_empty[sa]);
                mbar_arrive(&bars->kv_empty[sb]);
                if (leader) {
                    mbar_arrive(&bars->q_ready);
                } else {
                    mbar_arrive_remote_relaxed(mapa_shared(smem_u32(&bars->q_ready), 0));
                    mbar_arrive(&bars->q_copied);
                }
            }
        };

        int q_done = -1;
        for (int req = part.begin_req; req <= part.end_req; ++req) {
            int L, nb, b0, b1;
            item_range<kSparse>(p, part, req, L, nb, b0, b1);
            int lim = L;
            if (p.causal) {
                lim = L - p.s_q + s_idx + 1;
                lim = lim < 0 ? 0 : (lim > L ? L : lim);
            }
            const int first_piece = p.num_splits[req];
            const bool split = (p.num_splits[req + 1] - first_piece) > 1;
            const int slot = (req == part.begin_req) ? part.begin_split : first_piece;
            const bool has_blocks = b1 > b0;
            if (has_blocks && q_done != req) q_copy(gblk + 2 * item);
            float m_used = -INFINITY, l_part = 0.f;
            for (int blk = b0; blk < b1; ++blk, ++gblk) {
                const uint32_t sbuf = gblk & 1;
                const uint32_t st = (gblk + 2 * item + 2) % kStages;
                uint8_t* stage = ring + st * kStageBytes;
                // Partial scores of tokens [32h, 32h + 32) over this lane's rail.
                uint32_t sv[32];
                if (wait(&bars->s_full[sbuf], (gblk >> 1) & 1)) {
                    tc_fence_after();
                    tmem_ld32(tl + kColS + 64 * sbuf + 32 * h, sv);
                    tmem_ld_wait();
                    tc_fence_before();
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) sv[c] = 0u;
                }
                signal(&bars->s_empty[sbuf]);
                // Keep tokens [32h + 16 rho, +16); hand the other 16 to the
                // thread of the other rail (lane Lr ^ 64, same h).  rho is
                // uniform over the warp, so each branch indexes statically.
                const int keep = 16 * rho;
                float kept[16];
                {
                    float4* xo = X + ((h * 2 + (1 - rho)) * 4) * 64 + r;
                    auto hand_over = [&](const uint32_t* mine, const uint32_t* theirs) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) kept[c] = __uint_as_float(mine[c]);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            xo[64 * k] = make_float4(
                                __uint_as_float(theirs[4 * k]), __uint_as_float(theirs[4 * k + 1]),
                                __uint_as_float(theirs[4 * k + 2]), __uint_as_float(theirs[4 * k + 3]));
                    };
                    if (rho == 0)
                        hand_over(sv, sv + 16);
                    else
                        hand_over(sv + 16, sv);
                }
                // The partner rewrites this thread's slot only after the row
                // barrier below, which this thread passes after reading it.
                named_bar_sync(pair_bar, 64);
                const float4* xi = X + ((h * 2 + rho) * 4) * 64 + r;
                float x[16];
                // Column c (token 32 h + keep + c of the page) is visible when
                // c < nvis (dense), or when bit c of keys, from the stage's
                // key mask, is set (sparse; the page's kv_full phase completed
                // before its S, so the wait only orders the mask read).
                int nvis = 16;
                uint32_t keys = 0xFFFFu;
                if constexpr (kSparse) {
                    wait(&bars->kv_full[st], ((gblk + 2 * item + 2) / kStages) & 1);
                    keys = static_cast<uint32_t>(key_mask[st] >> (32 * h + keep)) & 0xFFFFu;
                } else {
                    const int t0 = blk * kPage + 32 * h + keep;
                    nvis = row_valid ? lim - t0 : 0;
                }
                const bool whole = kSparse ? keys == 0xFFFFu : nvis >= 16;
                const uint64_t sc2 = f32x2_splat(p.scale_log2);
                float hmax = -INFINITY;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 v = xi[64 * k];
                    float a0, a1, a2, a3;
                    f32x2_add(kept[4 * k], kept[4 * k + 1], v.x, v.y, a0, a1);
                    f32x2_add(kept[4 * k + 2], kept[4 * k + 3], v.z, v.w, a2, a3);
                    f32x2_mul(a0, a1, sc2, x[4 * k], x[4 * k + 1]);
                    f32x2_mul(a2, a3, sc2, x[4 * k + 2], x[4 * k + 3]);
                }
                // Pages every valid row sees whole skip the masking (rows past
                // the tile only feed their own, never written, output rows).
                if (__all_sync(0xffffffffu, !row_valid || whole)) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) hmax = fmaxf(hmax, x[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        x[c] = (kSparse ? ((keys >> c) & 1u) != 0 : c < nvis) ? x[c] : -INFINITY;
                        hmax = fmaxf(hmax, x[c]);
                    }
                }
                // Row max over the four threads of the row (two exchange
                // buffers by page parity: a buffer is rewritten two pages later,
                // after everyone passed the next page's row barrier).
                float* mrow = M + sbuf * 256;
                mrow[(2 * h + rho) * 64 + r] = hmax;
                named_bar_sync(row_bar, 128);
                const float tmax = fmaxf(fmaxf(mrow[r], mrow[64 + r]), fmaxf(mrow[128 + r], mrow[192 + r]));
                float alpha = 1.f;
                bool need = false;
                if (tmax > m_used + kLazyThreshold) {
                    alpha = (m_used == -INFINITY) ? 0.f : fast_exp2(m_used - tmax);
                    m_used = tmax;
                    need = true;
                }
                if (need) l_part *= alpha;
                uint32_t pk[8];
                // A row with no visible key yet has only -inf scores: with 0 in
                // place of the -inf max every exp2 is exactly 0.
                const uint64_t m2 = f32x2_splat(m_used == -INFINITY ? 0.f : m_used);
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float d0, d1;
                    f32x2_sub(x[2 * c], x[2 * c + 1], m2, d0, d1);
                    const float p0 = fast_exp2(d0);
                    const float p1 = fast_exp2(d1);
                    f32x2_add(ps0, ps1, p0, p1, ps0, ps1);
                    pk[c] = pack_bf16x2(p0, p1);
                }
                l_part += ps0 + ps1;
                // O is rescaled after PV(g - 1); the four warps of a row group
                // see the same rows, hence the same decision.
                const bool rescale = __any_sync(0xffffffffu, need && row_valid && blk > b0);
                wait_pv(rescale ? gblk : (gblk > 0 ? gblk - 1 : 0));
                if (rescale && alive) {
                    tc_fence_after();
                    const float a = (need && blk > b0) ? alpha : 1.f;
#pragma unroll 1
                    for (int cg = 0; cg < 4; ++cg) {
                        uint32_t o[32];
                        tmem_ld32(tl + kColO + 128 * h + 32 * cg, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                        tmem_st32(tl + kColO + 128 * h + 32 * cg, o);
                    }
                    tmem_st_wait();
                }
                // Last page of the sequence: zero this CTA's V rows past its
                // length (they may hold any bits, and 0 * NaN would poison PV).
                if (!kSparse && blk == nb - 1 && (L & (kPage - 1)) != 0) {
                    const int tail0 = L & (kPage - 1);
                    const int per_slot = (kPage - tail0) * 8;  // 16-byte units
                    for (int i = stid; i < 4 * per_slot; i += kSoftmaxThreads) {
                        const int s = i / per_slot, u = i % per_slot;
                        reinterpret_cast<uint4*>(stage + s * kSlotBytes + tail0 * 128)[u] =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                // P of tokens [32h + 16 rho, +16) into slot 4 (QK^T is done with it).
                uint8_t* pbuf = stage + 4 * kSlotBytes;
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    *reinterpret_cast<uint4*>(pbuf + sw128_offset(r, 4 * h + 2 * rho + k)) =
                        make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                fence_proxy_async_smem();
                tc_fence_before();
                signal(&bars->p_full[sbuf]);
            }
            if (has_blocks) {
                // The next request with blocks: its query entries follow this
                // request's last page; copy them now, so that its QK^T overlaps
                // this epilogue (this request's last QK^T is complete).
                for (int nr = req + 1; nr <= part.end_req; ++nr) {
                    int L2, nb2, c0, c1;
                    item_range<kSparse>(p, part, nr, L2, nb2, c0, c1);
                    if (c1 > c0) {
                        q_copy(gblk + 2 * (item + 1));
                        q_done = nr;
                        break;
                    }
                }
            }

            // ---------------------------------------------------- epilogue
            float l_tot = 0.f;
            if (has_blocks) {
                wait_pv(gblk);
                tc_fence_after();
                // Row sum over the four threads, through the exchange buffer of
                // the next page's parity; the second row barrier keeps it from
                // being rewritten (by the next page's row max) before all four
                // have read it.
                float* lrow = M + (gblk & 1) * 256;
                lrow[(2 * h + rho) * 64 + r] = l_part;
                named_bar_sync(row_bar, 128);
                l_tot = (lrow[r] + lrow[64 + r]) + (lrow[128 + r] + lrow[192 + r]);
                named_bar_sync(row_bar, 128);
            }
            const bool empty = !(l_tot > 0.f);
            const float inv = empty ? 0.f : 1.f / l_tot;
            const float lse2 = empty ? -INFINITY : m_used + fast_log2(l_tot);
            const int64_t acc_row = static_cast<int64_t>(slot) * p.R + row;
            const OutMap om = out_map(req, row, p.h_q, p.s_q, kSparse ? p.fold : 0, 1, p.h_q, p.out_sb, p.out_ss,
                                      p.out_sh);
            const int dvb = 256 * h + 128 * rho;  // this thread's 128 output dims
            const bool write = row_valid && alive;
            if (has_blocks) {
                // Two 32-column groups per TMEM wait (one per wait was slower:
                // MTP decode 282 against 277 us).
#pragma unroll 1
                for (int cp = 0; cp < 4; cp += 2) {
                  uint32_t oo[2][32];
                  tmem_ld32(tl + kColO + 128 * h + 32 * cp, oo[0]);
                  tmem_ld32(tl + kColO + 128 * h + 32 * (cp + 1), oo[1]);
                  tmem_ld_wait();
                  if (!write) continue;
#pragma unroll
                  for (int k = 0; k < 2; ++k) {
                    const int cg = cp + k;
                    const uint32_t (&o)[32] = oo[k];
                    const int dv0 = dvb + 32 * cg;
                    if (split) {
                        float4* dst = reinterpret_cast<float4*>(p.oaccum + acc_row * kDv + dv0);
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
                            uint32_t wv[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                wv[j] = pack_bf16x2(__uint_as_float(o[8 * v + 2 * j]) * inv,
                                                    __uint_as_float(o[8 * v + 2 * j + 1]) * inv);
                            dst[v] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                        }
                    }
                  }
                }
                tc_fence_before();
                warp_arrive_leader(&bars->o_free, leader);
                ++item;
            } else if (write) {
                if (split) {
                    float4* dst = reinterpret_cast<float4*>(p.oaccum + acc_row * kDv + dvb);
                    for (int v = 0; v < 32; ++v) dst[v] = make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + om.out_off + dvb);
                    for (int v = 0; v < 16; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if (write && h == 0 && rho == 0) {
                if (split)
                    p.lseaccum[acc_row] = lse2;
                else
                    p.lse[om.lse_idx] = empty ? -INFINITY : lse2 * 0.69314718055994531f;
            }
        }
    }

    // ------------------------------------------------------------ teardown
    // Both CTAs meet here once their roles are done (every wait above is
    // bounded, the leader's MMAs and each CTA's copies are drained), so no
    // MMA, copy or remote arrival can still touch either CTA's memory when
    // tensor memory is freed and the CTAs exit.
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc_pair(tmem, kTmemCols);
}

namespace {

cudaError_t duo_set_attributes() {
    static int configured_mask = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 31 || !(__atomic_load_n(&configured_mask, __ATOMIC_RELAXED) & (1 << dev))) {
        e = cudaFuncSetAttribute(decode_duo_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(decode_duo_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        if (dev < 31) __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_RELAXED);
    }
    return cudaSuccess;
}

void duo_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, dim3 grid, int threads,
                cudaStream_t s) {
    cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
}

}  // namespace

int duo_max_active_clusters() {
    if (duo_set_attributes() != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    duo_config(cfg, attr, dim3(2, 1, 1), kThreads, nullptr);
    cfg.numAttrs = 1;  // the cluster shape only
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_duo_kernel<false>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_decode_duo(const DecodeParams& p, const CUtensorMap& q_map,
                              const CUtensorMap& kv_map, cudaStream_t stream) {
    cudaError_t e = duo_set_attributes();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    // (The sparse instantiation has four more warps; one CTA per SM either way.)
    duo_config(cfg, attr, dim3(2 * p.n_mtiles, p.num_parts, 1),
               p.sparse ? kThreadsSparse : kThreads, stream);
    return p.sparse ? cudaLaunchKernelEx(&cfg, decode_duo_kernel<true>, p, q_map, kv_map)
                    : cudaLaunchKernelEx(&cfg, decode_duo_kernel<false>, p, q_map, kv_map);
}

}  // namespace mla
