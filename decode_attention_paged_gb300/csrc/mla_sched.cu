// mla_sched.cu -- device tile scheduler: builds the split-KV plan from the
// sequence lengths.
//
// Source: "FlashMLA 新内核深度解析：Seesaw 调度、细粒度 TMA 流水线与 H800 上的 660
// TFlops MLA 解码", section "Tile Scheduler：跨 SM 的负载均衡".  One warp counts
// the 64-token blocks of every request, sets the per-part cap
//     payload = ceil(total / num_sm_parts) + fixed_overhead,
// and fills the SM parts request by request, cutting a request into several
// pieces when it does not fit.  It records one DecodingSchedMeta record per
// part and num_splits, the prefix sum of pieces per request, for the combine.
//
// Readings: total counts every request's blocks plus the fixed overhead c
// (c >= 1); every piece of a request pays c, so a request continued in a new
// part pays it again; a part takes the rest of the current request whole when
// it fits in what is left of the cap, else as many blocks as fit (cap left
// minus c, when that is at least one) and closes.
//
// How the warp computes that walk.  Lay the requests out in order on a line
// of cost units (request i: c overhead units from C[i], then one unit per
// block; C[b] = total) and let q = ceil(total / parts).  A part that starts
// at a request boundary x can reach x + q + c; one that starts inside a
// request's blocks pays c again and reaches x + q.  If that reach E falls
// inside the blocks of a request (more than c units past its start), the
// part takes blocks up to E and the next part starts there, mid-request;
// otherwise (E within the c overhead units of request k) not one block of k
// fits and the next part starts at k's boundary C[k].  Each reach is at
// least q past the previous one and the first is q + c, so the parts hold
// all the work.  Reaches that fall inside blocks just add q, so the warp
// tests 32 consecutive reaches at once (a binary search per lane) and moves
// to the first that falls into overhead units.  A request's pieces are one
// plus the cuts inside its blocks; numbered in part order they are numbered
// request by request, so a part's first piece index is a prefix sum over
// parts.
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

__device__ __forceinline__ int64_t blocks_of(int32_t L) {
    return L > 0 ? (static_cast<int64_t>(L) + kPage - 1) / kPage : 0;
}

// Requests and parts the warp can plan: three int32 arrays of about batch
// entries and two of parts + 1 live in shared memory (opt-in size).
constexpr int kSchedMaxBatch = 16384;
constexpr int kSchedMaxParts = 1024;
constexpr size_t sched_smem_bytes(int batch, int parts) {
    return sizeof(int32_t) * (3 * (static_cast<size_t>(batch) + 1) + 2 * (static_cast<size_t>(parts) + 1));
}

__device__ __forceinline__ int warp_inclusive_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Largest i in [0, n) with C[i] <= x (C nondecreasing, C[0] = 0 <= x).
__device__ __forceinline__ int last_le(const int32_t* C, int n, int x) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (C[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(32) sched_kernel(const int32_t* __restrict__ seqlens,
                                                   int seq_div, int uniform_len, int batch, int R,
                                                   int num_parts, int n_mtiles, int fixed,
                                                   int32_t* meta, int32_t* num_splits) {
    // Let the decode kernel (programmatically dependent) run its prologue now;
    // it waits for this grid's completion before reading the plan.
    pdl_launch_dependents();
    extern __shared__ int32_t s_buf[];
    int32_t* C = s_buf;                  // C[i]: first cost unit of request i; C[batch] = total
    int32_t* S = C + batch + 1;          // S[i]: index of request i's first piece; S[batch] = pieces
    int32_t* PC = S + batch + 1;         // PC[i]: pieces of request i
    int32_t* X = PC + batch + 1;         // X[p]: first cost unit of part p; total past the last
    int32_t* K = X + num_parts + 1;      // K[p]: request holding X[p]; batch at the end
    const int lane = threadIdx.x;
    const int c = fixed;
    const int64_t cap_blocks = (1 << 30) / batch - c;

    // 1. Place the requests on the cost line.
    int carry = 0;
    for (int base = 0; base < batch; base += 32) {
        const int i = base + lane;
        const int32_t L = seqlens ? (i < batch ? seqlens[i / seq_div] : 0) : uniform_len;
        // Cost units stay below 2^30 in total (a cap no real cache reaches:
        // 2^30 / batch blocks of 64 tokens per request), so that every
        // position and reach below fits an int.
        const int64_t nb = blocks_of(L) < cap_blocks ? blocks_of(L) : cap_blocks;
        const int v = i < batch ? static_cast<int>(nb) + c : 0;
        const int incl = warp_inclusive_scan(v);
        if (i < batch) {
            C[i + 1] = carry + incl;
            PC[i] = 1;
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
        C[0] = 0;
        X[0] = 0;
        K[0] = 0;
    }
    __syncwarp();
    const int total = C[batch];
    const int q = (total + num_parts - 1) / num_parts;
    auto nblk = [&](int i) { return C[i + 1] - C[i] - c; };

    // 2. The parts' starts, 32 reaches per round.  Part p + m reaches
    // E + m q as long as parts p .. p + m - 1 all end inside blocks.
    {
        int p = 0;
        int64_t E = static_cast<int64_t>(q) + c;  // part 0 starts at request 0's boundary
        for (;;) {
            const int64_t Em = E + static_cast<int64_t>(lane) * q;
            const bool live = p + lane < num_parts && Em < total;
            int km = 0;
            bool snap = false;
            if (live) {
                km = last_le(C, batch, static_cast<int>(Em));
                snap = Em - C[km] <= c;
            }
            const unsigned ev = __ballot_sync(0xffffffffu, snap || !live);
            const int f = ev ? __ffs(ev) - 1 : 32;
            if (lane < f) {  // part p + lane ends inside request km's blocks
                X[p + lane + 1] = static_cast<int>(Em);
                K[p + lane + 1] = km;
                atomicAdd(&PC[km], 1);
            }
            if (f == 32) {
                p += 32;
                E += static_cast<int64_t>(32) * q;
                continue;
            }
            const int kf = __shfl_sync(0xffffffffu, km, f);
            const bool snapped = __shfl_sync(0xffffffffu, snap ? 1 : 0, f) != 0;
            if (snapped) {  // part p + f closes at request kf's boundary
                const int xs = C[kf];
                if (lane == 0) {
                    X[p + f + 1] = xs;
                    K[p + f + 1] = kf;
                }
                p += f + 1;
                E = static_cast<int64_t>(xs) + q + c;
                continue;
            }
            // Part p + f (if it exists) takes the rest; later parts are empty.
            for (int r = p + f + 1 + lane; r <= num_parts; r += 32) {
                X[r] = total;
                K[r] = batch;
            }
            break;
        }
    }
    __syncwarp();

    // 3. num_splits: prefix sums of the pieces per request.
    carry = 0;
    for (int base = 0; base < batch; base += 32) {
        const int i = base + lane;
        const int incl = warp_inclusive_scan(i < batch ? PC[i] : 0);
        if (i < batch) S[i + 1] = carry + incl;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) S[0] = 0;
    __syncwarp();
    const int pieces_total = S[batch];

    // 4. One record per part: first and last requests from the starts of the
    // part and of the next one, first piece index by a prefix sum over parts.
    int4* rec_out = reinterpret_cast<int4*>(meta + kMetaHeader);
    carry = 0;
    for (int base = 0; base < num_parts; base += 32) {
        const int p = base + lane;
        int bq = 0, er = -1, b0 = 0, b1 = 0;
        const bool used = p < num_parts && X[p] < X[p + 1];
        if (used) {
            const int a = X[p], e = X[p + 1];
            bq = K[p];
            b0 = a > C[bq] ? a - C[bq] - c : 0;
            const int kn = K[p + 1];
            if (kn < batch && e > C[kn]) {  // the next part continues request kn
                er = kn;
                b1 = e - C[kn] - c;
            } else {
                er = kn - 1;
                b1 = nblk(er);
            }
        }
        const int np = used ? er - bq + 1 : 0;
        const int incl = warp_inclusive_scan(np);
        const int first_piece = carry + incl - np;
        carry += __shfl_sync(0xffffffffu, incl, 31);
        if (p >= num_parts) continue;
        if (!used) {
            rec_out[2 * p] = make_int4(batch, batch - 1, 0, 0);
            rec_out[2 * p + 1] = make_int4(pieces_total, 0, 0, 0);
            continue;
        }
        const int first_split = (S[bq + 1] - S[bq]) > 1;
        const int last_split = (S[er + 1] - S[er]) > 1;
        rec_out[2 * p] = make_int4(bq, er, b0, b1);
        rec_out[2 * p + 1] = make_int4(first_piece, first_split, last_split, 0);
    }
    for (int i = lane; i <= batch; i += 32) num_splits[i] = S[i];
    if (lane == 0) {
        reinterpret_cast<int4*>(meta)[0] = make_int4(kMetaMagic, batch, R, num_parts);
        reinterpret_cast<int4*>(meta)[1] = make_int4(n_mtiles, fixed, kPage, pieces_total);
    }
}

int sched_max_batch() { return kSchedMaxBatch; }

cudaError_t launch_sched(const int32_t* seqlens, int seq_div, int uniform_len, int batch, int R,
                         int num_parts, int n_mtiles, int fixed_overhead, int32_t* meta,
                         int32_t* num_splits, cudaStream_t stream) {
    if (num_parts < 1 || num_parts > kSchedMaxParts || batch < 1 || batch > kSchedMaxBatch ||
        fixed_overhead < 1 || fixed_overhead > (1 << 16))
        return cudaErrorInvalidValue;
    const size_t smem = sched_smem_bytes(batch, num_parts);
    // Same shared-memory carveout as the decode kernels, so that a step's
    // kernels follow one another without reconfiguring the SMs.
    static int carveout_mask = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
    if (dev >= 31 || !(__atomic_load_n(&carveout_mask, __ATOMIC_RELAXED) & (1 << dev))) {
        cudaError_t e = cudaFuncSetAttribute(sched_kernel,
                                             cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        if (dev < 31) __atomic_fetch_or(&carveout_mask, 1 << dev, __ATOMIC_RELAXED);
    }
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(sched_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(sched_smem_bytes(kSchedMaxBatch, kSchedMaxParts)));
        if (e != cudaSuccess) return e;
    }
    sched_kernel<<<1, 32, smem, stream>>>(seqlens, seq_div < 1 ? 1 : seq_div, uniform_len, batch, R,
                                          num_parts, n_mtiles, fixed_overhead, meta, num_splits);
    return cudaGetLastError();
}

}  // namespace mla
