// mla_fp8.cuh -- in-place dequantisation of one page of the FP8 cache layout
// ("[DeepSeek-3] FlashMLA：把 MLA 的 KV Cache 优势变成 GPU 吞吐", sec. 12: a row
// of 656 bytes = 512 float8_e4m3 latent values, 4 fp32 scales each shared by
// 128 of them, 64 bf16 RoPE values), used by the decode kernels that read it.
#pragma once

#include <cuda_fp8.h>

#include "sm103_ptx.cuh"

namespace mla {

constexpr uint32_t kFp8RowBytes = 656;
constexpr uint32_t kFp8PageBytes = 64 * kFp8RowBytes;  // 41984: one bulk copy
// The raw rows land at the top of a 72 KB stage and are rewritten below them.
constexpr uint32_t kFp8RawOff = 9 * 8192 - kFp8PageBytes;  // 31744, 16-byte aligned
static_assert(kFp8RawOff % 16 == 0 && kFp8PageBytes % 16 == 0, "bulk copy alignment");

// Four warps (dt = 0..127 among them) turn the page's raw rows at
// stage + kFp8RawOff into the bf16 page the MMAs read: 9 chunks of
// [64 rows x 64 dims], 128-byte swizzled, latent dims in chunks 0..7 and the
// RoPE in chunk 8.  Two threads per row: thread (t, hh) takes latent dims
// [256 hh, 256 hh + 256) with their two scales and RoPE dims
// [32 hh, 32 hh + 32).  The raw rows overlap the bf16 rows, so every thread
// reads all its raw bytes before any thread writes (named barrier bar_id of
// the four warps).  Each value becomes bf16(e4m3 * scale): e4m3 -> f16 is
// exact, the product is rounded to fp32, then to bf16 (nearest even).  A page
// outside the cache (bad) becomes zeros.  The caller fences the writes for
// the tensor core and signals the page.
// Two fp32 products in one instruction (each lane rounded to nearest, as the
// scalar multiply), packed to bf16x2.
__device__ __forceinline__ uint32_t mul2_pack_bf16x2(float x0, float x1, uint64_t s2) {
    uint64_t x, z;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(s2));
    float a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(z));
    return pack_bf16x2(a, b);
}

__device__ __forceinline__ void fp8_dequant_page(uint8_t* stage, int dt, bool bad,
                                                 uint32_t bar_id) {
    const int t = dt >> 1, hh = dt & 1;
    const uint8_t* raw = stage + kFp8RawOff + t * kFp8RowBytes;
    uint4 lat[16], rope[4];
    float sc[2];
#pragma unroll
    for (int u = 0; u < 16; ++u) lat[u] = *reinterpret_cast<const uint4*>(raw + 256 * hh + 16 * u);
#pragma unroll
    for (int u = 0; u < 4; ++u) rope[u] = *reinterpret_cast<const uint4*>(raw + 528 + 64 * hh + 16 * u);
    sc[0] = *reinterpret_cast<const float*>(raw + 512 + 8 * hh);
    sc[1] = *reinterpret_cast<const float*>(raw + 516 + 8 * hh);
    named_bar_sync(bar_id, 128);
    uint64_t s2[2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
        asm("mov.b64 %0, {%1, %1};" : "=l"(s2[h]) : "f"(sc[h]));
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const uint32_t in[4] = {lat[u].x, lat[u].y, lat[u].z, lat[u].w};
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const __nv_fp8x2_storage_t two =
                static_cast<__nv_fp8x2_storage_t>(in[j >> 1] >> (16 * (j & 1)));
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
            o[j] = bad ? 0u : mul2_pack_bf16x2(f.x, f.y, s2[u >> 3]);
        }
        const int dim0 = 256 * hh + 16 * u;  // 16 dims: two 16-byte units
        uint8_t* chunk = stage + (dim0 >> 6) * 8192;
        const uint32_t unit = (dim0 & 63) >> 3;
        *reinterpret_cast<uint4*>(chunk + sw128_offset(t, unit)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(chunk + sw128_offset(t, unit + 1)) =
            make_uint4(o[4], o[5], o[6], o[7]);
    }
    uint8_t* rchunk = stage + 8 * 8192;
#pragma unroll
    for (int u = 0; u < 4; ++u)
        *reinterpret_cast<uint4*>(rchunk + sw128_offset(t, 4 * hh + u)) =
            bad ? make_uint4(0, 0, 0, 0) : rope[u];
}

// The same page with 256 threads (dt = 0..255), four per row: thread (t, q)
// takes latent dims [128 q, 128 q + 128) with their scale and RoPE dims
// [16 q, 16 q + 16); the 16-byte reads of a row's four threads start at
// rotated units so that the eight threads of a quarter warp hit distinct
// bank groups.  Same rounding and the same barrier rule as above.  The unit
// loop is not unrolled (the staged units move down one register slot per
// turn): measured, the smaller code ran the page about 1% faster than the
// unrolled loop, and eight warps in place of four took the FP8 memory-bound
// step from 111 to 93 us.
__device__ __forceinline__ void fp8_dequant_page_x4(uint8_t* stage, int dt, bool bad,
                                                    uint32_t bar_id) {
    const int t = dt >> 2, q = dt & 3;
    const uint8_t* raw = stage + kFp8RawOff + t * kFp8RowBytes;
    uint4 lat[8], rope[2];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        lat[k] = *reinterpret_cast<const uint4*>(raw + 128 * q + 16 * ((k + 2 * q) & 7));
#pragma unroll
    for (int k = 0; k < 2; ++k) rope[k] = *reinterpret_cast<const uint4*>(raw + 528 + 32 * q + 16 * k);
    const float sc = *reinterpret_cast<const float*>(raw + 512 + 4 * q);
    named_bar_sync(bar_id, 256);
    uint64_t s2;
    asm("mov.b64 %0, {%1, %1};" : "=l"(s2) : "f"(sc));
#pragma unroll 1
    for (int k = 0; k < 8; ++k) {
        const int u = (k + 2 * q) & 7;  // 16-dim unit of this thread's 128 dims
        const uint32_t in[4] = {lat[0].x, lat[0].y, lat[0].z, lat[0].w};
#pragma unroll
        for (int i = 0; i < 7; ++i) lat[i] = lat[i + 1];
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const __nv_fp8x2_storage_t two =
                static_cast<__nv_fp8x2_storage_t>(in[j >> 1] >> (16 * (j & 1)));
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
            o[j] = bad ? 0u : mul2_pack_bf16x2(f.x, f.y, s2);
        }
        const int dim0 = 128 * q + 16 * u;
        uint8_t* chunk = stage + (dim0 >> 6) * 8192;
        const uint32_t unit = (dim0 & 63) >> 3;
        *reinterpret_cast<uint4*>(chunk + sw128_offset(t, unit)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(chunk + sw128_offset(t, unit + 1)) =
            make_uint4(o[4], o[5], o[6], o[7]);
    }
    uint8_t* rchunk = stage + 8 * 8192;
#pragma unroll
    for (int k = 0; k < 2; ++k)
        *reinterpret_cast<uint4*>(rchunk + sw128_offset(t, 2 * q + k)) =
            bad ? make_uint4(0, 0, 0, 0) : rope[k];
}

}  // namespace mla
