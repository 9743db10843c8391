// mla_decode_pair.cu -- split-KV paged MLA decode, one 2-CTA cluster per
// (SM part, 64-row query tile), the 576 head dims split across the pair.
//
// Sources (web pages, cited by title and section):
//   [Overview] "[DeepSeek-3] FlashMLA：把 MLA 的 KV Cache 优势变成 GPU 吞吐":
//       sec. 3 (one 576-dim cache row is K; its first 512 dims are V),
//       sec. 4 (paged KV through block_table), sec. 6 (split-KV partials),
//       sec. 7 (online softmax makes the partials mergeable), sec. 13 (two
//       CTAs of a cluster each take half of the work and exchange results
//       through distributed shared memory).
//   [DeepDive] "FlashMLA 新内核深度解析：Seesaw 调度、细粒度 TMA 流水线与 H800
//       上的 660 TFlops MLA 解码": "细粒度 TMA copy-GEMM 流水线" (a 64x576 K
//       tile moves as 64x64 TMA copies), "缓存提示" (EVICT_FIRST), the exp ->
//       exp2 rewrite (end of the Seesaw section), "Programmatic Dependent
//       Launch", "Tile Scheduler" (each SM part walks its DecodingSchedMeta).
//   [AttnBook] "3.4 Attention kernel": "在线 softmax", 代码 (causal mask).
//
// Why a pair.  On sm_103a the 64 x 512 fp32 output tile lives in tensor
// memory, so registers no longer limit the design -- shared memory does: a
// whole 64 x 576 Q tile (72 KB) plus whole 72 KB pages leaves room for only
// two pages in flight, and every page then waits out an HBM round trip plus
// QK^T -> softmax -> PV before its buffer can be refilled.  The pair splits
// the head dims instead: rank 0 owns the 64-dim chunks 0..3 (dims 0..255),
// rank 1 owns chunks 4..8 (dims 256..575, the last one the RoPE part).
// Each CTA loads only its chunks of Q and of every page (32 or 40 KB), so
// three or four pages are in flight per CTA (four when the query tile has at
// most 32 rows and Q takes less room) and P and the exchange buffer are double
// buffered; QK^T over its chunks gives a partial score tile; the two partials
// are swapped through distributed shared memory and summed in the same order
// on both sides, so both CTAs run the identical softmax and hold the identical
// P.  PV then needs only V's dims that the CTA already has: rank 0 computes
// output dims 0..255 from its chunks 0..3, rank 1 dims 256..511 from its
// chunks 4..7.  No byte of KV is loaded twice.
//
// The score swap uses asynchronous remote stores that complete transaction
// bytes on the receiver's barrier (no fences, no remote arrivals).  With two
// exchange buffers the sender needs no "buffer free" signal: thread T writes
// page g + 2 into the peer's slot T only after receiving the peer's page g + 1,
// which the peer's thread T sent after it had consumed page g from that slot.
//
// Per CTA: warp 0 = TMA producer (one thread), warp 1 = TMEM owner and QK^T
// issuer, warp 6 = PV issuer (both converged warps issuing through
// elect.sync, so P -> PV never waits behind a batch of QK^T MMAs), warps 2..5
// = score exchange, softmax, correction and epilogue (one thread per TMEM
// lane; when the query tile has at most 32 valid rows only the two warps that
// hold them take part).  Tensor
// memory: O half [64 x 256] fp32 through weight-stationary M=64 MMAs = 128
// columns (lanes 0..63 hold dims 0..127 of the half, lanes 64..127 dims
// 128..255); S partial [64 x 64] = 32 columns, two buffers.
//
// Every wait is bounded; a timeout records MLA_ERR_DEVICE_TIMEOUT, drains the
// CTA's own copies and MMAs, and both CTAs meet at a cluster barrier before
// releasing tensor memory.  A CTA that aborted also waits a short bounded
// while after that barrier, so that a score store its peer issued before the
// barrier has landed before the CTA's shared memory is released.
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

namespace {

// Tuning knobs (compile time).  The producer and the two MMA issuers are
// placed by warp index: warp w runs on SM sub-partition w % 4, and the
// softmax warps 2..5 must cover the four TMEM lane quadrants.
#ifndef MLA_PAIR_PRODUCER_WARP
#define MLA_PAIR_PRODUCER_WARP 0
#endif
#ifndef MLA_PAIR_PV_WARP
#define MLA_PAIR_PV_WARP 6
#endif
#ifndef MLA_PAIR_CTRL_SLEEP_NS  // back-off of the producer / MMA-issuer waits
#define MLA_PAIR_CTRL_SLEEP_NS 0
#endif
#ifndef MLA_PAIR_MAX_STAGES
#define MLA_PAIR_MAX_STAGES 5
#endif
#ifndef MLA_PAIR_COMPACT_Q
#define MLA_PAIR_COMPACT_Q 1
#endif
constexpr int kProducerWarp = MLA_PAIR_PRODUCER_WARP;
constexpr int kPvWarp = MLA_PAIR_PV_WARP;
constexpr int kThreads = 32 * ((kPvWarp > kProducerWarp ? kPvWarp : kProducerWarp) > 6
                                   ? ((kPvWarp > kProducerWarp ? kPvWarp : kProducerWarp) + 1)
                                   : 7);
static_assert(kProducerWarp != 1 && (kProducerWarp < 2 || kProducerWarp > 5) &&
                  kPvWarp != 1 && (kPvWarp < 2 || kPvWarp > 5) && kPvWarp != kProducerWarp,
              "warp roles overlap");
constexpr int kMaxStages = MLA_PAIR_MAX_STAGES;
constexpr int kMaxChunks = 5;                               // rank 1: chunks 4..8
constexpr uint32_t kUnitBytes = kMaxChunks * kChunkBytes;   // one KV stage, 40 KB
constexpr uint32_t kPBytes = 64 * 128;                      // P [64 rows x 64 tokens] bf16
constexpr uint32_t kSmemMax = 232448;                       // 227 KB per CTA
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 0;    // O half: 128 columns
constexpr uint32_t kColS = 128;  // S partial: two buffers of 32 columns
constexpr float kLazyThreshold = 8.0f;           // log2 units (factor 256)
constexpr uint64_t kDrainBudgetNs = 2000000000ull;
constexpr uint64_t kQuiesceNs = 100000ull;       // error path only
constexpr uint32_t kReadAhead = 8;               // block-table entries read ahead
constexpr int kPageRing = 16;

struct Barriers {
    uint64_t kv_full[kMaxStages];
    uint64_t kv_empty[kMaxStages];
    uint64_t q_full, q_empty;
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full[2], pv_done[2];
    uint64_t o_free, drain_qk, drain_pv;
    uint64_t xs_full[2];  // the peer's partial scores of a page landed in sX[b]
};
static_assert(sizeof(Barriers) <= 256, "barrier block");

// Shared-memory layout, a function of the rows one Q tile load brings (the
// same for every CTA of a launch).  Q chunks are packed q_rows * 128 bytes
// apart: the M=64 MMA still reads 64 rows per chunk, and the rows past q_rows
// (the next chunk's, or the next region's) are padding rows whose scores the
// softmax masks.  The exchange buffers hold one 128-byte slot per TMEM lane
// that can carry a valid row.  What remains holds as many 40 KB KV stages as
// fit.
struct PairLayout {
    uint32_t q_rows, x_slots, n_stages;
    uint32_t off_kv, off_p, off_x, off_bar, off_xch, off_misc, bytes;
};
__host__ __device__ constexpr PairLayout pair_layout(int q_box_rows) {
    PairLayout l{};
    l.q_rows = !MLA_PAIR_COMPACT_Q ? 64u : (q_box_rows <= 16 ? 16u : (q_box_rows <= 32 ? 32u : 64u));
    l.x_slots = l.q_rows <= 32 ? 64u : 128u;
    const uint32_t q_bytes = kMaxChunks * l.q_rows * 128u;
    const uint32_t fixed = q_bytes + 2 * kPBytes + 2 * l.x_slots * 128u + 256u + 2048u + 64u;
    uint32_t st = (kSmemMax - fixed) / kUnitBytes;
    l.n_stages = st > kMaxStages ? kMaxStages : st;
    l.off_kv = q_bytes;
    l.off_p = l.off_kv + l.n_stages * kUnitBytes;
    l.off_x = l.off_p + 2 * kPBytes;
    l.off_bar = l.off_x + 2 * l.x_slots * 128u;
    l.off_xch = l.off_bar + 256u;     // uint2 [2][128]: in-CTA pair exchange
    l.off_misc = l.off_xch + 2048u;   // tmem base, abort flag
    l.bytes = l.off_misc + 64u;
    return l;
}
static_assert(pair_layout(16).bytes <= kSmemMax && pair_layout(32).bytes <= kSmemMax &&
                  pair_layout(64).bytes <= kSmemMax,
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

struct Cursor {
    int req, blk, b0, b1, L, nb;
    uint32_t g;
    uint32_t item;
    bool valid;
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
// Wait of the producer and MMA-issuer warps: optionally backs off between
// probes so that a waiting control warp leaves issue slots to the softmax
// warp sharing its SM sub-partition.
__device__ __forceinline__ bool ctrl_wait(uint64_t* bar, uint32_t parity, const WaitCtx& c) {
    if (MLA_PAIR_CTRL_SLEEP_NS == 0) return mbar_wait(bar, parity, c, MLA_ERR_DEVICE_TIMEOUT);
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(MLA_PAIR_CTRL_SLEEP_NS);
        if (mbar_try_wait(bar, parity)) return true;
        if (*c.abort_flag) return false;
        if (globaltimer_ns() - t0 > c.budget_ns) {
            raise_error(c, MLA_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
}
__device__ __forceinline__ bool warp_wait_ctrl(uint64_t* bar, uint32_t parity, const WaitCtx& wc) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = ctrl_wait(bar, parity, wc);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  const WaitCtx& wc) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_cluster(bar, parity, wc, MLA_ERR_DEVICE_TIMEOUT);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        __threadfence_block();
        mbar_arrive(bar);
    }
}

// Exchange one float with the thread holding the other half of the same
// query row in this CTA (TMEM lane L <-> L ^ 64): tagged slots in two
// alternating buffers, a bounded spin, and a warp-uniform verdict.
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

// Chunks [0, NCH) of this CTA's partial S = Q K^T for one page, each MMA issued
// by one elected lane of the converged warp.
template <int NCH>
__device__ __forceinline__ void issue_qk(uint64_t dQ, uint64_t q_chunk_units, uint64_t bK,
                                         uint32_t d) {
    constexpr uint32_t idesc_qk = idesc_bf16_f32(64, 64, false, false);
    constexpr uint64_t kChunkUnits = kChunkBytes >> 4;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const uint64_t a = dQ + c * q_chunk_units, b = bK + c * kChunkUnits;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            if (elect_one()) mma_ws_ss(d, a + 2 * kk, b + 2 * kk, idesc_qk, (c + kk) ? 1u : 0u);
    }
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    decode_pair_kernel(const __grid_constant__ DecodeParams p,
                       const __grid_constant__ CUtensorMap q_map,
                       const __grid_constant__ CUtensorMap kv_map) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const uint32_t rank = cluster_ctarank();  // 0: dims 0..255, 1: dims 256..575
    const uint32_t peer = rank ^ 1u;
    const int mtile = blockIdx.y, part_idx = blockIdx.z;
    const int chunk0 = rank ? 4 : 0;
    const int nch = rank ? 5 : 4;
    const PairLayout lay = pair_layout(p.q_box_rows);
    const uint32_t n_stages = lay.n_stages;
    const uint32_t q_chunk_bytes = lay.q_rows * 128u;
    // Query rows of this tile that exist; the softmax warps whose TMEM lanes
    // hold only padding rows (q4 = warp & 3 odd: rows 32..63) sit out when
    // there are at most 32.
    int rows_valid = p.R - mtile * kTileM;
    rows_valid = rows_valid > kTileM ? kTileM : rows_valid;
    const uint32_t n_active = rows_valid > 32 ? 4u : 2u;
    const uint32_t x_bytes = static_cast<uint32_t>(rows_valid) * 2u * 128u;
    const uint32_t x_buf_bytes = lay.x_slots * 128u;
    const bool softmax_warp =
        warp >= 2 && warp <= 5 && (n_active == 4 || ((warp & 3) & 1) == 0);

    uint8_t* sQ = smem;
    uint8_t* sKV = smem + lay.off_kv;
    uint8_t* sP = smem + lay.off_p;
    uint8_t* sX = smem + lay.off_x;
    Barriers* bars = reinterpret_cast<Barriers*>(smem + lay.off_bar);
    uint2* xch = reinterpret_cast<uint2*>(smem + lay.off_xch);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + lay.off_misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.off_misc + 4);
    WaitCtx wc{abort_flag, p.error_word, p.budget_ns};

    // ------------------------------------------------------------ prologue
    if (tid == 0) {
        *abort_flag = 0;
        for (uint32_t s = 0; s < n_stages; ++s) {
            mbar_init(&bars->kv_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->s_empty[s], n_active);
            mbar_init(&bars->p_full[s], n_active);
            mbar_init(&bars->pv_done[s], 1);
            mbar_init(&bars->xs_full[s], 1);
        }
        mbar_init(&bars->o_free, n_active);
        mbar_init(&bars->drain_qk, 1);
        mbar_init(&bars->drain_pv, 1);
        fence_barrier_init();
        // First phase of both exchange buffers: expect the peer's bytes.
        mbar_arrive_expect_tx(&bars->xs_full[0], x_bytes);
        mbar_arrive_expect_tx(&bars->xs_full[1], x_bytes);
        prefetch_tensormap(&q_map);
        prefetch_tensormap(&kv_map);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    for (int i = tid; i < 2 * 128; i += kThreads) xch[i] = make_uint2(0u, 0u);
    tc_fence_before();
    // Both CTAs' barriers exist (and are armed) before either writes to the other.
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    pdl_wait_primary();

    bool ok = (smem_u32(smem) & 1023u) == 0;
    const int32_t* hdr = p.meta;
    if (ok && (hdr[kHMagic] != kMetaMagic || hdr[kHBatch] != p.batch || hdr[kHRows] != p.R ||
               hdr[kHParts] != p.num_parts || hdr[kHMTiles] != p.n_mtiles ||
               hdr[kHPage] != kPage))
        ok = false;
    Part part{};
    if (ok) {
        const int32_t* rec = hdr + kMetaHeader + part_idx * kMetaFields;
        part.begin_req = rec[kBeginReq];
        part.end_req = rec[kEndReq];
        part.begin_block = rec[kBeginBlock];
        part.end_block = rec[kEndBlock];
        part.begin_split = rec[kBeginSplit];
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
    if (tid == 0 && rank == 0) {
        for (int req = part.begin_req; req <= part.end_req; ++req) {
            const int L = p.seqlens[req];
            if (L > 0 && blocks_of(L) > p.max_blocks) raise_error(wc, MLA_ERR_SEQ_TOO_LONG);
        }
    }

    if (warp == kProducerWarp && lane == 0) {
        // ------------------------------------------------------ TMA producer
        const uint64_t policy = policy_evict_first();
        const uint32_t q_bytes = nch * p.q_box_rows * 128;  // TMA box: q_box_rows rows
        const uint32_t kv_bytes = nch * kChunkBytes;
        Cursor ld = cursor_begin(p, part), pf = ld;
        int ring[kPageRing];
        uint32_t n_kv = 0, n_q = 0;
        while (ld.valid) {
            while (pf.valid && pf.g <= ld.g + kReadAhead) {
                ring[pf.g % kPageRing] =
                    p.block_table[static_cast<int64_t>(pf.req) * p.bt_stride + pf.blk];
                cursor_next(p, part, pf);
            }
            const uint32_t st = ld.g % n_stages;
            if (ld.g >= n_stages &&
                !ctrl_wait(&bars->kv_empty[st], ((ld.g / n_stages) + 1) & 1, wc))
                break;
            const int page = ring[ld.g % kPageRing];
            mbar_arrive_expect_tx(&bars->kv_full[st], kv_bytes);
            uint8_t* dst = sKV + st * kUnitBytes;
            for (int c = 0; c < nch; ++c)
                tma_load_3d(&kv_map, &bars->kv_full[st], dst + c * kChunkBytes, 64 * (chunk0 + c),
                            0, page, policy);
            ++n_kv;
            if (ld.blk == ld.b0) {  // first block of a request: its Q tile
                if (ld.item > 0 &&
                    !ctrl_wait(&bars->q_empty, (ld.item - 1) & 1, wc))
                    break;
                mbar_arrive_expect_tx(&bars->q_full, q_bytes);
                for (int c = 0; c < nch; ++c)
                    tma_load_3d(&q_map, &bars->q_full, sQ + c * q_chunk_bytes, 64 * (chunk0 + c),
                                mtile * kTileM, ld.req, policy);
                ++n_q;
            }
            cursor_next(p, part, ld);
        }
        for (uint32_t k = (n_kv >= n_stages ? n_kv - n_stages : 0); k < n_kv; ++k)
            mbar_drain(&bars->kv_full[k % n_stages], (k / n_stages) & 1, kDrainBudgetNs);
        if (n_q > 0) mbar_drain(&bars->q_full, (n_q - 1) & 1, kDrainBudgetNs);
    } else if (warp == 1) {
        // ------------------------------------------------------ QK^T issuer
        // Block g needs its page, its request's Q tile and a free S buffer.
        const uint64_t dQ = smem_desc(smem_u32(sQ), 16, 1024);
        const uint64_t dK0 = smem_desc(smem_u32(sKV), 16, 1024);
        constexpr uint64_t kUnitUnits = kUnitBytes >> 4;
        const uint64_t q_chunk_units = q_chunk_bytes >> 4;
        for (Cursor qk = cursor_begin(p, part); qk.valid; cursor_next(p, part, qk)) {
            const uint32_t st = qk.g % n_stages;
            const int sb = qk.g & 1;
            if (qk.blk == qk.b0 && !warp_wait_ctrl(&bars->q_full, qk.item & 1, wc)) break;
            if (!warp_wait_ctrl(&bars->kv_full[st], (qk.g / n_stages) & 1, wc)) break;
            if (qk.g >= 2 && !warp_wait_ctrl(&bars->s_empty[sb], ((qk.g >> 1) + 1) & 1, wc))
                break;
            tc_fence_after();
            const uint64_t bK = dK0 + st * kUnitUnits;
            const uint32_t d = tmem + kColS + 32 * sb;
            if (nch == 4)
                issue_qk<4>(dQ, q_chunk_units, bK, d);
            else
                issue_qk<5>(dQ, q_chunk_units, bK, d);
            if (elect_one()) {
                mma_commit(&bars->s_full[sb]);
                if (qk.blk == qk.b1 - 1) mma_commit(&bars->q_empty);
            }
            __syncwarp();
        }
        if (elect_one()) mma_commit(&bars->drain_qk);
        __syncwarp();
        if (lane == 0) mbar_drain(&bars->drain_qk, 0, kDrainBudgetNs);
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------ PV issuer
        // Block g needs P(g) and, on a request's first block, O released by
        // the previous request's epilogue.
        constexpr uint32_t idesc_pv = idesc_bf16_f32(64, 256, false, true);
        const uint64_t dV0 = smem_desc(smem_u32(sKV), kChunkBytes, 1024);
        const uint64_t dP0 = smem_desc(smem_u32(sP), 16, 1024);
        constexpr uint64_t kUnitUnits = kUnitBytes >> 4;
        constexpr uint64_t kPUnits = kPBytes >> 4;
        const uint32_t tO = tmem + kColO;
        for (Cursor pv = cursor_begin(p, part); pv.valid; cursor_next(p, part, pv)) {
            const bool first = pv.blk == pv.b0;
            const int pb = pv.g & 1;
            if (!warp_wait_ctrl(&bars->p_full[pb], (pv.g >> 1) & 1, wc)) break;
            if (first && pv.item > 0 && !warp_wait_ctrl(&bars->o_free, (pv.item - 1) & 1, wc))
                break;
            tc_fence_after();
            const uint64_t bV = dV0 + (pv.g % n_stages) * kUnitUnits;
            const uint64_t aP = dP0 + pb * kPUnits;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                if (elect_one())
                    mma_ws_ss(tO, aP + 2 * kk, bV + 128 * kk, idesc_pv,
                              (first && kk == 0) ? 0u : 1u);
            if (elect_one()) {
                mma_commit(&bars->pv_done[pb]);
                mma_commit(&bars->kv_empty[pv.g % n_stages]);
            }
            __syncwarp();
        }
        if (elect_one()) mma_commit(&bars->drain_pv);
        __syncwarp();
        if (lane == 0) mbar_drain(&bars->drain_pv, 0, kDrainBudgetNs);
        __syncwarp();
    } else if (softmax_warp) {
        // -------------------- score exchange / softmax / correction / epilogue
        const int q4 = warp & 3;
        const int Lrow = 32 * q4 + lane;  // TMEM lane
        const int r = Lrow & 63, half = Lrow >> 6;
        const int row = mtile * kTileM + r;
        const bool row_valid = r < rows_valid;
        const int s_idx = row / p.h_q, h_idx = row % p.h_q;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
        // Index of this thread among the active softmax threads.
        const int me = n_active == 4 ? (tid - 64) : ((warp == 4 ? 0 : 32) + lane);
        // This thread's 128-byte slot in both exchange buffers; 16-byte units
        // are rotated by lane so a warp's accesses spread over all banks.
        const int x_slot = lay.x_slots == 64 ? ((Lrow & 31) + 32 * half) : Lrow;
        const uint32_t x_own = smem_u32(sX) + x_slot * 128;
        const uint32_t x_peer = mapa_shared(x_own, peer);
        const uint32_t xs_full_peer = mapa_shared(smem_u32(&bars->xs_full[0]), peer);
        const bool arm_thread = (warp == 2 && lane == 0);
        uint32_t gblk = 0, xseq = 0;
        bool alive = true;
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
            float m_used = -INFINITY, l_part = 0.f;
            for (int blk = b0; blk < b1; ++blk, ++gblk) {
                const int sb = gblk & 1;
                if (!warp_wait(&bars->s_full[sb], (gblk >> 1) & 1, wc)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                uint32_t sv[32];
                tmem_ld32(tl + kColS + 32 * sb, sv);
                tmem_ld_wait();
                tc_fence_before();
                warp_arrive(&bars->s_empty[sb]);

                // Swap partial scores with the peer (same lane, buffer sb).
                if (row_valid) {
                    const uint32_t dst = x_peer + sb * x_buf_bytes;
                    const uint32_t bar = xs_full_peer + sb * 8;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t u = (k ^ (lane & 7)) * 16;
                        st_async_v4(dst + u, sv[4 * k], sv[4 * k + 1], sv[4 * k + 2],
                                    sv[4 * k + 3], bar);
                    }
                }
                if (!warp_wait_cluster(&bars->xs_full[sb], (gblk >> 1) & 1, wc)) {
                    alive = false;
                    break;
                }
                // Re-arm this buffer for the page after next.
                if (arm_thread) mbar_arrive_expect_tx(&bars->xs_full[sb], x_bytes);
                uint32_t pv_[32];
                if (row_valid) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t u = (k ^ (lane & 7)) * 16;
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(pv_[4 * k]), "=r"(pv_[4 * k + 1]), "=r"(pv_[4 * k + 2]),
                                       "=r"(pv_[4 * k + 3])
                                     : "r"(x_own + sb * x_buf_bytes + u)
                                     : "memory");
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) pv_[c] = 0u;
                }

                const int t0 = blk * kPage + 32 * half;
                float x[32];
                float hmax = -INFINITY;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    // Same summation order on both CTAs: rank 0's partial first.
                    const float a = __uint_as_float(rank ? pv_[c] : sv[c]);
                    const float b = __uint_as_float(rank ? sv[c] : pv_[c]);
                    x[c] = (row_valid && t0 + c < lim) ? (a + b) * p.scale_log2 : -INFINITY;
                    hmax = fmaxf(hmax, x[c]);
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
                float psum = 0.f;
                const bool none = (m_used == -INFINITY);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float p0 = none ? 0.f : fast_exp2(x[2 * c] - m_used);
                    const float p1 = none ? 0.f : fast_exp2(x[2 * c + 1] - m_used);
                    psum += p0 + p1;
                    pk[c] = pack_bf16x2(p0, p1);
                }
                l_part += psum;

                // O must hold PV(g - 1) before it is rescaled for page g.
                if (__any_sync(0xffffffffu, need && blk > b0)) {
                    if (!warp_wait(&bars->pv_done[(gblk - 1) & 1], ((gblk - 1) >> 1) & 1, wc)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    const float a = (need && blk > b0) ? alpha : 1.f;
#pragma unroll 1
                    for (int cg = 0; cg < 4; ++cg) {
                        uint32_t o[32];
                        tmem_ld32(tl + kColO + 32 * cg, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                        tmem_st32(tl + kColO + 32 * cg, o);
                    }
                    tmem_st_wait();
                }
                // P buffer sb was last read by PV(g - 2).
                if (gblk >= 2 && !warp_wait(&bars->pv_done[sb], ((gblk - 2) >> 1) & 1, wc)) {
                    alive = false;
                    break;
                }
                // Last page of the sequence: zero the V rows past its length
                // in the chunks this CTA multiplies by P (they may hold any
                // bits, and 0 * NaN would poison the sum).
                if (blk == nb - 1 && (L & (kPage - 1)) != 0) {
                    const int tail0 = L & (kPage - 1);
                    const int per_chunk = (kPage - tail0) * 8;
                    uint8_t* stage = sKV + (gblk % n_stages) * kUnitBytes;
                    for (int i = me; i < 4 * per_chunk; i += 32 * static_cast<int>(n_active)) {
                        const int c = i / per_chunk, u = i % per_chunk;
                        reinterpret_cast<uint4*>(stage + c * kChunkBytes + tail0 * 128)[u] =
                            make_uint4(0, 0, 0, 0);
                    }
                }
                uint8_t* pbuf = sP + sb * kPBytes;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t off = sw128_offset(r, 4 * half + k);
                    *reinterpret_cast<uint4*>(pbuf + off) =
                        make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                warp_arrive(&bars->p_full[sb]);
            }
            if (!alive) break;

            // ---------------------------------------------------- epilogue
            const bool has_blocks = b1 > b0;
            float l_tot = 0.f;
            if (has_blocks) {
                if (!warp_wait(&bars->pv_done[(gblk - 1) & 1], ((gblk - 1) >> 1) & 1, wc)) {
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
            const int dv_base = 256 * rank + 128 * half;
            if (has_blocks) {
#pragma unroll 1
                for (int cg = 0; cg < 4; ++cg) {
                    uint32_t o[32];
                    tmem_ld32(tl + kColO + 32 * cg, o);
                    tmem_ld_wait();
                    const int dv0 = dv_base + 32 * cg;
                    if (!row_valid) continue;
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
                }
                tc_fence_before();
                warp_arrive(&bars->o_free);
            } else if (row_valid) {
                if (split) {
                    float4* dst = reinterpret_cast<float4*>(p.oaccum + acc_row * kDv + dv_base);
                    for (int v = 0; v < 32; ++v) dst[v] = make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + req * p.out_sb + s_idx * p.out_ss +
                                                          h_idx * p.out_sh + dv_base);
                    for (int v = 0; v < 16; ++v) dst[v] = make_uint4(0, 0, 0, 0);
                }
            }
            if (row_valid && half == 0 && rank == 0) {
                if (split)
                    p.lseaccum[acc_row] = lse2;
                else
                    p.lse[(static_cast<int64_t>(req) * p.h_q + h_idx) * p.s_q + s_idx] =
                        empty ? -INFINITY : lse2 * 0.69314718055994531f;
            }
        }
    }

    // ------------------------------------------------------------ teardown
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    // Neither CTA leaves while the other may still write into its memory.
    cluster_sync();
    if (*abort_flag) {
        // Error path only: let any score store the peer issued before the
        // barrier land before this CTA's shared memory is released.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < kQuiesceNs) {
        }
    }
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

static cudaLaunchConfig_t pair_config(const DecodeParams& p, cudaStream_t stream,
                                      cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, p.n_mtiles, p.num_parts);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = pair_layout(p.q_box_rows).bytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cfg;
}

static cudaError_t pair_set_smem() {
    static int configured_mask = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 31 || !(__atomic_load_n(&configured_mask, __ATOMIC_RELAXED) & (1 << dev))) {
        e = cudaFuncSetAttribute(decode_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemMax));
        if (e != cudaSuccess) return e;
        if (dev < 31) __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_RELAXED);
    }
    return cudaSuccess;
}

int pair_max_active_clusters() {
    if (pair_set_smem() != cudaSuccess) return 0;
    DecodeParams p{};
    p.n_mtiles = 1;
    p.num_parts = 1;
    p.q_box_rows = kTileM;  // the largest layout
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config(p, nullptr, attr);
    cfg.numAttrs = 1;  // cluster shape only
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_pair_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_decode_pair(const DecodeParams& p, const CUtensorMap& q_map,
                               const CUtensorMap& kv_map, cudaStream_t stream) {
    cudaError_t e = pair_set_smem();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config(p, stream, attr);
    return cudaLaunchKernelEx(&cfg, decode_pair_kernel, p, q_map, kv_map);
}

}  // namespace mla
