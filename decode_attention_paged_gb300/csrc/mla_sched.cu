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
// Reading of how the parts are filled (the page gives the cap, not the walk):
// every request costs its blocks plus the fixed overhead c (c >= 1); laid out
// in order on a line of cost units (c overhead units, then one unit per
// block), the requests cover total = sum_i (n_i + c) units, and part p takes
// the units [p*q, (p+1)*q), q = ceil(total / parts).  A request belongs to a
// part when that range holds one of its blocks (a request without blocks: its
// first unit).  A part then costs at most q + c = payload -- the "+ fixed
// overhead" is the room for the overhead a split request pays again in the
// part that continues it.  This fill is the same for every part's view, so
// the warp computes all parts at once: prefix sums place the requests on the
// line, and each lane binary-searches the requests at its parts' two ends.
// The plan only balances work: any valid plan gives the same attention result.
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

__device__ __forceinline__ int64_t blocks_of(int32_t L) {
    return L > 0 ? (static_cast<int64_t>(L) + kPage - 1) / kPage : 0;
}

// Requests the warp can plan: two int32 arrays of batch + 1 entries live in
// shared memory (opt-in size).
constexpr int kSchedMaxBatch = 16384;

__device__ __forceinline__ int warp_inclusive_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Largest i in [0, n) with C[i] <= x (C strictly increasing, C[0] = 0 <= x).
__device__ __forceinline__ int last_le(const int32_t* C, int n, int64_t x) {
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
    int32_t* C = s_buf;              // C[i]: first cost unit of request i; C[batch] = total
    int32_t* S = s_buf + batch + 1;  // S[i]: index of request i's first piece; S[batch] = pieces
    const int lane = threadIdx.x;
    const int c = fixed;

    // 1. Place the requests on the cost line.
    int carry = 0;
    for (int base = 0; base < batch; base += 32) {
        const int i = base + lane;
        const int32_t L = seqlens ? (i < batch ? seqlens[i / seq_div] : 0) : uniform_len;
        const int v = i < batch ? static_cast<int>(blocks_of(L)) + c : 0;
        const int incl = warp_inclusive_scan(v);
        if (i < batch) C[i + 1] = carry + incl;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) C[0] = 0;
    __syncwarp();
    const int64_t total = C[batch];
    const int64_t q = (total + num_parts - 1) / num_parts;

    // 2. Pieces per request: the parts its blocks' units fall in.
    auto nblk = [&](int i) { return C[i + 1] - C[i] - c; };
    auto first_part = [&](int i) -> int64_t {
        return nblk(i) > 0 ? (C[i] + c) / q : C[i] / q;
    };
    carry = 0;
    for (int base = 0; base < batch; base += 32) {
        const int i = base + lane;
        int pc = 0;
        if (i < batch) {
            const int n = nblk(i);
            pc = n > 0 ? static_cast<int>((C[i] + c + n - 1) / q - (C[i] + c) / q + 1) : 1;
        }
        const int incl = warp_inclusive_scan(pc);
        if (i < batch) S[i + 1] = carry + incl;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) S[0] = 0;
    __syncwarp();
    const int pieces_total = S[batch];

    // 3. One record per part.
    auto contained = [&](int i, int64_t a, int64_t e) -> bool {
        const int n = nblk(i);
        if (n > 0) {
            const int64_t lo = static_cast<int64_t>(C[i]) + c;
            return lo < e && lo + n > a;
        }
        return C[i] >= a && C[i] < e;
    };
    int4* rec_out = reinterpret_cast<int4*>(meta + kMetaHeader);
    for (int p = lane; p < num_parts; p += 32) {
        const int64_t a = static_cast<int64_t>(p) * q;
        const int64_t e = a + q < total ? a + q : total;
        int bq = -1, er = -1;
        if (a < total) {
            const int i0 = last_le(C, batch, a);
            if (contained(i0, a, e)) bq = i0;
            else if (i0 + 1 < batch && contained(i0 + 1, a, e)) bq = i0 + 1;
            if (bq >= 0) {
                const int j0 = last_le(C, batch, e - 1);
                er = contained(j0, a, e) ? j0 : j0 - 1;
            }
        }
        if (bq < 0) {
            rec_out[2 * p] = make_int4(batch, batch - 1, 0, 0);
            rec_out[2 * p + 1] = make_int4(pieces_total, 0, 0, 0);
            continue;
        }
        const int nb = nblk(bq), ne = nblk(er);
        int64_t b0 = nb > 0 ? a - C[bq] - c : 0;
        if (b0 < 0) b0 = 0;
        int64_t b1 = ne > 0 ? e - C[er] - c : 0;
        if (b1 > ne) b1 = ne;
        const int begin_split = S[bq] + static_cast<int>(p - first_part(bq));
        const int first_split = (S[bq + 1] - S[bq]) > 1;
        const int last_split = (S[er + 1] - S[er]) > 1;
        rec_out[2 * p] = make_int4(bq, er, static_cast<int>(b0), static_cast<int>(b1));
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
    const size_t smem = 2 * sizeof(int32_t) * (static_cast<size_t>(batch) + 1);
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
                                             static_cast<int>(2 * sizeof(int32_t) * (kSchedMaxBatch + 1)));
        if (e != cudaSuccess) return e;
    }
    sched_kernel<<<1, 32, smem, stream>>>(seqlens, seq_div < 1 ? 1 : seq_div, uniform_len, batch, R,
                                          num_parts, n_mtiles, fixed_overhead, meta, num_splits);
    return cudaGetLastError();
}

}  // namespace mla
