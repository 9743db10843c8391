// mla_combine.cu -- merges the split-KV partial results of every request that
// the tile scheduler cut into more than one piece.
//
// Source: "FlashMLA 新内核深度解析", section "Programmatic Dependent Launch": one
// warp per query row takes the max of the pieces' log-sum-exps, weights each
// partial output by exp2(lse_k - max), sums, and forms the final lse in the
// log2 domain; the kernel waits for the decode grid with
// cudaGridDependencySynchronize (griddepcontrol.wait) and reads the partials
// with ordinary loads (not the read-only path, which does not see the
// producer's writes under programmatic launch).  Pieces whose lse is -inf
// (nothing visible) get weight 0 (their partial rows are written as zeros);
// if every piece is empty the row is 0 and lse -inf ("CUTLASS 从零重写
// FlashAttention：Split KV 并行优化实战", sec. 3.3).
//
// Layout: oaccum [pieces][R][512] fp32 holds each piece's normalised output,
// lseaccum [pieces][R] its log2-domain log-sum-exp (m + log2 l, with scores
// already multiplied by softmax_scale * log2 e).  A warp works on one row:
// lane l owns dims [16 l, 16 l + 16), so each piece is read as one contiguous
// 2 KB burst per warp with 16-byte vector loads.  Rows cut into many pieces get
// several warps each, which split the pieces and add their partial sums.
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

__device__ __forceinline__ float4 ld_f4(const float* p) {
    // Plain (coherent) global load; see the note on programmatic launch above.
    float4 v;
    asm volatile("ld.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_f(const float* p) {
    float v;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ int ld_i(const int32_t* p) {
    int v;
    asm volatile("ld.global.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// kW warps per query row (kWarps / kW rows per CTA): warp j of a row takes
// the pieces k = j, j + kW, ..., so a row cut into many pieces streams them
// from several warps at once; the kW partial sums meet in shared memory.
template <int kW, int kWarps>
__global__ void __launch_bounds__(32 * kWarps) combine_kernel(CombineParams p) {
    constexpr int kCombineWarps = kWarps;
    constexpr int kRowsPerCta = kCombineWarps / kW;
    __shared__ float4 s_acc[kW > 1 ? kCombineWarps : 1][32][4];
    __shared__ float s_w[kW > 1 ? kCombineWarps : 1];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int req = blockIdx.y;
    const int row = blockIdx.x * kRowsPerCta + warp / kW;
    const int j = warp % kW;
    // The next decode grid may launch now: it waits for this grid's completion
    // before it reads its plan or writes anything.
    pdl_launch_dependents();
    // The plan is read before the wait: the decode grid lets this grid launch
    // only after its own wait, when the plan was already complete.  Metadata
    // built for another shape: the decode kernel has already recorded
    // MLA_ERR_METADATA_MISMATCH; num_splits may be too short to index.  (Every
    // condition below is the same for all warps of a CTA, or for all warps of
    // a row: no warp leaves while its row's partners still need the barrier.)
    const bool plan_ok = ld_i(p.meta + kHMagic) == kMetaMagic &&
                         ld_i(p.meta + kHBatch) == p.batch && ld_i(p.meta + kHRows) == p.R;
    int first = 0, n = 0;
    if (plan_ok) {
        first = ld_i(p.num_splits + req);
        n = ld_i(p.num_splits + req + 1) - first;
    }
    pdl_wait_primary();
    // A request cut into one piece was written by the decode kernel directly.
    if (n <= 1) return;
    const bool row_ok = row < p.R;
    const float* o_base = p.oaccum + (static_cast<int64_t>(first) * p.R + row) * kDv + lane * 16;
    const int64_t piece_stride = static_cast<int64_t>(p.R) * kDv;
    const int mine = n > j ? (n - j + kW - 1) / kW : 0;  // pieces of this warp
    // Partial rows of this warp's pieces base + u (u < 4), 16 floats per lane.
    float4 x[4][4];
    auto load_group = [&](int base) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (base + u < mine) {
                const float* src = o_base + static_cast<int64_t>(j + kW * (base + u)) * piece_stride;
#pragma unroll
                for (int v = 0; v < 4; ++v) x[u][v] = ld_f4(src + 4 * v);
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v) x[u][v] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    };
    // The first group's loads go out with the lse loads below.
    if (row_ok) load_group(0);

    // The largest piece lse of the row (every warp of the row computes it).
    const float* lse_base = p.lseaccum + static_cast<int64_t>(first) * p.R + row;
    float mx = -INFINITY;
    if (row_ok)
        for (int k = lane; k < n; k += 32) mx = fmaxf(mx, ld_f(lse_base + static_cast<int64_t>(k) * p.R));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));

    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    float wsum = 0.f;
    if (row_ok && mx != -INFINITY) {
        // Pieces j, j + kW, ...: lane t of each group of 32 holds piece
        // j + kW (base + t)'s weight; the partial rows are streamed with four
        // pieces' loads in flight.  An empty piece (lse = -inf) has weight 0
        // and an all-zero partial row.
        for (int base = 0; base < mine; base += 32) {
            const int t = base + lane;
            const float lk = t < mine ? ld_f(lse_base + static_cast<int64_t>(j + kW * t) * p.R) : -INFINITY;
            const float wl = (lk == -INFINITY) ? 0.f : fast_exp2(lk - mx);
            float ws = wl;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
            wsum += ws;
            const int m = min(32, mine - base);
            for (int j0 = 0; j0 < m; j0 += 4) {
                float w[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    w[u] = __shfl_sync(0xffffffffu, wl, (j0 + u) & 31);
                    if (j0 + u >= m) w[u] = 0.f;
                }
                if (base + j0 > 0) load_group(base + j0);
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        acc[4 * v + 0] += w[u] * x[u][v].x;
                        acc[4 * v + 1] += w[u] * x[u][v].y;
                        acc[4 * v + 2] += w[u] * x[u][v].z;
                        acc[4 * v + 3] += w[u] * x[u][v].w;
                    }
            }
        }
    }
    if (kW > 1) {
        // The row's kW partial sums meet in shared memory; its first warp adds
        // them in a fixed order.
#pragma unroll
        for (int v = 0; v < 4; ++v)
            s_acc[warp][lane][v] = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
        if (lane == 0) s_w[warp] = wsum;
        __syncthreads();
        if (j != 0) return;
        for (int q = 1; q < kW; ++q) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const float4 o = s_acc[warp + q][lane][v];
                acc[4 * v] += o.x;
                acc[4 * v + 1] += o.y;
                acc[4 * v + 2] += o.z;
                acc[4 * v + 3] += o.w;
            }
            wsum += s_w[warp + q];
        }
    }
    if (!row_ok) return;
    const OutMap om =
        out_map(req, row, p.h_q, p.s_q, p.fold, p.kvh, p.grp, p.out_sb, p.out_ss, p.out_sh);
    __nv_bfloat16* orow = p.out + om.out_off + lane * 16;
    float* lse_out = p.lse + om.lse_idx;
    if (mx == -INFINITY) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(orow)[0] = z;
        reinterpret_cast<uint4*>(orow)[1] = z;
        if (lane == 0) *lse_out = -INFINITY;
        return;
    }
    const float inv = 1.f / wsum;
    uint32_t packed[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) packed[i] = pack_bf16x2(acc[2 * i] * inv, acc[2 * i + 1] * inv);
    reinterpret_cast<uint4*>(orow)[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    reinterpret_cast<uint4*>(orow)[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    if (lane == 0) *lse_out = (mx + fast_log2(wsum)) * 0.69314718055994531f;
}

// Rows of dv != 512 floats (mla_decode_fwd_dims): the same merge, one warp
// per row, four rows per CTA; lane l owns dims [l nd, l nd + nd), nd = dv / 32
// (even), read as float2.
__global__ void __launch_bounds__(128) combine_dims_kernel(CombineParams p) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int req = blockIdx.y, row = blockIdx.x * 4 + warp;
    pdl_launch_dependents();
    // The plan is read before the wait (see combine_kernel).
    const bool plan_ok = ld_i(p.meta + kHMagic) == kMetaMagic &&
                         ld_i(p.meta + kHBatch) == p.batch && ld_i(p.meta + kHRows) == p.R;
    int first = 0, n = 0;
    if (plan_ok) {
        first = ld_i(p.num_splits + req);
        n = ld_i(p.num_splits + req + 1) - first;
    }
    pdl_wait_primary();
    if (row >= p.R || n <= 1) return;
    const int dv = p.dv, nd = dv / 32;
    const float* lse_base = p.lseaccum + static_cast<int64_t>(first) * p.R + row;
    float mx = -INFINITY;
    for (int k = lane; k < n; k += 32) mx = fmaxf(mx, ld_f(lse_base + static_cast<int64_t>(k) * p.R));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const OutMap om =
        out_map(req, row, p.h_q, p.s_q, p.fold, p.kvh, p.grp, p.out_sb, p.out_ss, p.out_sh);
    __nv_bfloat16* orow = p.out + om.out_off + lane * nd;
    if (mx == -INFINITY) {
        for (int i = 0; i < nd; i += 2) *reinterpret_cast<uint32_t*>(orow + i) = 0u;
        if (lane == 0) p.lse[om.lse_idx] = -INFINITY;
        return;
    }
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    float wsum = 0.f;
    const float* o_base = p.oaccum + (static_cast<int64_t>(first) * p.R + row) * dv + lane * nd;
    for (int k = 0; k < n; ++k) {
        const float lk = ld_f(lse_base + static_cast<int64_t>(k) * p.R);
        const float w = (lk == -INFINITY) ? 0.f : fast_exp2(lk - mx);
        wsum += w;
        const float* src = o_base + static_cast<int64_t>(k) * p.R * dv;
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            if (i < nd) {
                float2 v;
                asm volatile("ld.global.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(src + i));
                acc[i] += w * v.x;
                acc[i + 1] += w * v.y;
            }
        }
    }
    const float inv = 1.f / wsum;
#pragma unroll
    for (int i = 0; i < 16; i += 2)
        if (i < nd) *reinterpret_cast<uint32_t*>(orow + i) = pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
    if (lane == 0) p.lse[om.lse_idx] = (mx + fast_log2(wsum)) * 0.69314718055994531f;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool pdl) {
    if (p.dv != 0 && p.dv != kDv) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((p.R + 3) / 4, p.batch, 1);
        cfg.blockDim = dim3(128, 1, 1);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        return cudaLaunchKernelEx(&cfg, combine_dims_kernel, p);
    }
    // Warps per row from the average number of pieces per request (the plan
    // has at most batch + parts pieces): when requests average eight pieces or
    // more (few long sequences spread over many SM parts) eight warps share
    // each row; otherwise one warp per row, four rows per CTA (measured: the
    // wider form slowed steps whose requests have few pieces, its CTAs
    // launching early beside the decode kernel).
    const int parts = p.num_parts > 0 ? p.num_parts : 1;
    const int avg = (p.batch + parts + p.batch - 1) / p.batch;
    const int ki = avg >= 8 ? 1 : 0;
    const int w = ki ? 8 : 1, warps = ki ? 8 : 4;
    using Kernel = void (*)(CombineParams);
    const Kernel kernels[2] = {combine_kernel<1, 4>, combine_kernel<8, 8>};
    // Same shared-memory carveout as the decode kernels (no SM reconfiguration
    // between the kernels of one step).
    static int carveout_mask[2] = {0, 0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 31 || !(__atomic_load_n(&carveout_mask[ki], __ATOMIC_RELAXED) & (1 << dev))) {
        e = cudaFuncSetAttribute(kernels[ki], cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        if (dev < 31) __atomic_fetch_or(&carveout_mask[ki], 1 << dev, __ATOMIC_RELAXED);
    }
    const int rows_per_cta = warps / w;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.R + rows_per_cta - 1) / rows_per_cta, p.batch, 1);
    cfg.blockDim = dim3(32 * warps, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernels[ki], p);
}

}  // namespace mla
