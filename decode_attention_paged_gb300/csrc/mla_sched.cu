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
// fits and the next part starts at k's boundary C[k].  So the parts' starts
// follow one another by a single search each, and every record, piece count
// and split index follows from those starts with prefix sums and binary
// searches.  Each reach is at least q past the previous one and the first is
// q + c, so the parts hold all the work.
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

__device__ __forceinline__ int64_t blocks_of(int32_t L) {
    return L > 0 ? (static_cast<int64_t>(L) + kPage - 1) / kPage : 0;
}

// Requests and parts the warp can plan: two int32 arrays of batch + 1 entries
// and one of parts + 1 live in shared memory (opt-in size).
constexpr int kSchedMaxBatch = 16384;
constexpr int kSchedMaxParts = 1024;
constexpr size_t sched_smem_bytes(int batch, int parts) {
    return sizeof(int32_t) * (2 * (static_cast<size_t>(batch) + 1) + static_cast<size_t>(parts) + 1);
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
    int32_t* S = s_buf + batch + 1;      // S[i]: index of request i's first piece; S[batch] = pieces
    int32_t* X = s_buf + 2 * batch + 2;  // X[p]: first cost unit of part p; X[num_parts] = total
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
        if (i < batch) C[i + 1] = carry + incl;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) C[0] = 0;
    __syncwarp();
    const int total = C[batch];
    const int q = (total + num_parts - 1) / num_parts;

    // 2. The parts' starts, one after another.  k: the request holding the
    // current start; the next request holding a reach is found 32 requests
    // at a time (C increases, so the lanes with C[k + 1 + lane] <= E form a
    // prefix of the warp).
    {
        int x = 0, k = 0;
        bool boundary = true;
        int p = 0;
        for (; p < num_parts && x < total; ++p) {
            if (lane == 0) X[p] = x;
            const int E = x + q + (boundary ? c : 0);
            if (E >= total) {
                x = total;
                continue;
            }
            for (;;) {
                const int j = k + 1 + lane;
                const unsigned ok = __ballot_sync(0xffffffffu, j < batch && C[j] <= E);
                const int n_ok = __popc(ok);
                k += n_ok;
                if (n_ok < 32) break;
            }
            if (E - C[k] <= c) {
                x = C[k];
                boundary = true;
            } else {
                x = E;
                boundary = false;
            }
        }
        for (int r = p + lane; r <= num_parts; r += 32) X[r] = total;
    }
    __syncwarp();

    // 3. Pieces per request: the parts holding its first and last block
    // units (a request without blocks: its first overhead unit).
    auto nblk = [&](int i) { return C[i + 1] - C[i] - c; };
    auto part_of = [&](int pos) { return last_le(X, num_parts, pos); };
    auto first_part = [&](int i) { return part_of(nblk(i) > 0 ? C[i] + c : C[i]); };
    carry = 0;
    for (int base = 0; base < batch; base += 32) {
        const int i = base + lane;
        int pc = 0;
        if (i < batch) pc = nblk(i) > 0 ? part_of(C[i + 1] - 1) - first_part(i) + 1 : 1;
        const int incl = warp_inclusive_scan(pc);
        if (i < batch) S[i + 1] = carry + incl;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) S[0] = 0;
    __syncwarp();
    const int pieces_total = S[batch];

    // 4. One record per part: the requests holding its first and last units.
    int4* rec_out = reinterpret_cast<int4*>(meta + kMetaHeader);
    for (int p = lane; p < num_parts; p += 32) {
        const int a = X[p], e = X[p + 1];
        if (a >= e) {
            rec_out[2 * p] = make_int4(batch, batch - 1, 0, 0);
            rec_out[2 * p + 1] = make_int4(pieces_total, 0, 0, 0);
            continue;
        }
        const int bq = last_le(C, batch, a);
        const int er = last_le(C, batch, e - 1);
        const int b0 = a > C[bq] ? a - C[bq] - c : 0;
        const int b1 = e - C[er] - c > 0 ? e - C[er] - c : 0;
        const int begin_split = S[bq] + (p - first_part(bq));
        const int first_split = (S[bq + 1] - S[bq]) > 1;
        const int last_split = (S[er + 1] - S[er]) > 1;
        rec_out[2 * p] = make_int4(bq, er, b0, b1);
        rec_out[2 * p + 1] = make_int4(begin_split, first_split, last_split, 0);
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
