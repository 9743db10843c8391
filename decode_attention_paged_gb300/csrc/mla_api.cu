// mla_api.cu -- the C ABI of libmla.so (declared in include/mla_decode.h):
// argument checking, the split-plan geometry, TMA descriptor encoding and the
// kernel launches.  The library owns no device memory of its own apart from the
// per-device error word below (a module global, not an allocation).
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "mla_internal.h"

namespace mla {

// First device-side error since the last mla_last_device_error() call.
__device__ int g_mla_error_word = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultBudgetNs = 2000000000ull;
// The scheduler's fixed overhead per request piece, in 64-token blocks, by
// kernel: what a request boundary measured costs each kernel in pages of
// streaming (sweeps of 1..8 on GB300: the single-CTA kernel best at 2, the
// tensor-memory-Q kernel at 4, the CTA-pair kernel at 5-6).  A value set with
// mla_set_fixed_overhead overrides them.
int default_fixed_overhead(int kind) {
    return kind == MLA_KERNEL_DUO ? 5 : (kind == MLA_KERNEL_TQ ? 4 : 2);
}

std::atomic<uint64_t> g_budget_ns{kDefaultBudgetNs};
std::atomic<int> g_fixed_overhead{-1};  // -1: the kernel's default
std::atomic<int> g_kernel{MLA_KERNEL_AUTO};

int fixed_overhead_for(int kind) {
    const int v = g_fixed_overhead.load();
    return v >= 1 ? v : default_fixed_overhead(kind);
}

struct DeviceInfo {
    std::once_flag once;
    int sms = 0;
    int duo_clusters = 0;  // co-resident 2-CTA clusters of the CTA-pair kernel
    int major = 0, minor = 0;
    int* error_word = nullptr;
    cudaError_t status = cudaSuccess;
};
DeviceInfo g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_status = cudaSuccess;

int device_info(DeviceInfo** out) {
    int dev = 0;
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return MLA_ERR_NO_DEVICE;
    }
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
    DeviceInfo& d = g_dev[dev];
    std::call_once(d.once, [&] {
        d.status = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (d.status == cudaSuccess)
            d.status = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
        if (d.status == cudaSuccess)
            d.status = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (d.status == cudaSuccess)
            d.status = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.error_word), g_mla_error_word);
        if (d.status == cudaSuccess && d.major == 10 && d.minor == 3)
            d.duo_clusters = duo_max_active_clusters();
    });
    if (d.status != cudaSuccess) return MLA_ERR_CUDA;
    // The kernels are built for sm_103a only.
    if (d.major != 10 || d.minor != 3) return MLA_ERR_UNSUPPORTED;
    *out = &d;
    return MLA_OK;
}

int n_mtiles_of(int R) { return (R + kTileM - 1) / kTileM; }
constexpr int kPairTileM = 128;  // query rows of one CTA pair

// The decode kernel a dense call with R rows per request (h_kv cache heads)
// launches: the one mla_set_decode_kernel selected, or by tile height.
int kernel_for(int R, int h_kv, const DeviceInfo* d) {
    int kind = g_kernel.load();
    if (kind == MLA_KERNEL_AUTO)
        kind = R <= 32 ? MLA_KERNEL_TQ : (R >= kPairTileM ? MLA_KERNEL_DUO : MLA_KERNEL_SINGLE);
    // Several cache heads: the single-CTA kernel only.  The pair kernel loads
    // 64 query rows per CTA and needs its clusters to be resident.
    if (h_kv > 1) return MLA_KERNEL_SINGLE;
    if (kind == MLA_KERNEL_DUO && (R < kTileM || d->duo_clusters < 1)) return MLA_KERNEL_SINGLE;
    return kind;
}

// Query tiles of a request for a kernel (64 rows, or 128 for a CTA pair).
int tiles_of(int R, int kind) {
    return kind == MLA_KERNEL_DUO ? (R + kPairTileM - 1) / kPairTileM : n_mtiles_of(R);
}

// SM parts of the split plan: as many (part, query tile) work units as the
// kernel keeps resident at once -- one CTA per SM, or one cluster per SM pair.
int num_parts_of(int R, int h_kv, const DeviceInfo* d) {
    const int kind = kernel_for(R, h_kv, d);
    const int units = kind == MLA_KERNEL_DUO ? d->duo_clusters : d->sms;
    const int parts = units / tiles_of(R, kind);
    return parts > 0 ? parts : 1;
}

int num_parts_single(int R, const DeviceInfo* d) {
    const int parts = d->sms / n_mtiles_of(R);
    return parts > 0 ? parts : 1;
}

// Sparse decode: the CTA pair where the dense choice would take it (lists of
// at least 128 query rows), else the single-CTA kernel (the other kernel
// does no row gather).
int sparse_kind(int R, const DeviceInfo* d) {
    return kernel_for(R, 1, d) == MLA_KERNEL_DUO ? MLA_KERNEL_DUO : MLA_KERNEL_SINGLE;
}
int num_parts_sparse(int R, const DeviceInfo* d) {
    if (sparse_kind(R, d) != MLA_KERNEL_DUO) return num_parts_single(R, d);
    const int parts = d->duo_clusters / tiles_of(R, MLA_KERNEL_DUO);
    return parts > 0 ? parts : 1;
}

// Kernel geometry of a dense call: its requests are the (request i, cache
// head j) pairs, each with the s_q * grp rows of query heads j*grp..j*grp+grp-1.
struct Geo {
    int nreq, R, kvh, grp;
};
Geo geo_of(int batch, int h_q, int s_q, int h_kv) {
    return Geo{batch * h_kv, s_q * (h_q / h_kv), h_kv, h_q / h_kv};
}

int check_shape(int batch, int h_q, int s_q, int h_kv) {
    if (batch < 1 || h_q < 1 || s_q < 1 || h_kv < 1) return MLA_ERR_INVALID_ARGUMENT;
    if (h_q % h_kv != 0) return MLA_ERR_INVALID_ARGUMENT;
    if (static_cast<int64_t>(batch) * h_kv > sched_max_batch()) return MLA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(s_q) * h_q > (1 << 24)) return MLA_ERR_INVALID_ARGUMENT;
    if (h_kv > 1) {
        // A query tile covers whole head groups of 64 / grp tokens, or a
        // 64-head slice of one token.
        const int g = h_q / h_kv;
        if (g <= kTileM ? (kTileM % g != 0) : (g % kTileM != 0)) return MLA_ERR_UNSUPPORTED;
    }
    return MLA_OK;
}

// Sparse decode folds (request, query token) into the kernel's requests, each
// with the h_q rows of one token.
int check_shape_sparse(int batch, int h_q, int s_q, int h_kv, int topk) {
    if (batch < 1 || h_q < 1 || s_q < 1 || topk < 0) return MLA_ERR_INVALID_ARGUMENT;
    if (static_cast<int64_t>(batch) * s_q > sched_max_batch()) return MLA_ERR_UNSUPPORTED;
    if (h_q > (1 << 24) || topk > (1 << 24)) return MLA_ERR_INVALID_ARGUMENT;
    if (h_kv != 1) return MLA_ERR_UNSUPPORTED;
    return MLA_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace split: oaccum [pieces][R][512] fp32, then lseaccum [pieces][R].
void workspace_layout(int batch, int R, int parts, size_t* o_bytes, size_t* total) {
    const size_t pieces = static_cast<size_t>(batch) + parts;
    *o_bytes = align_up(pieces * R * kDv * sizeof(float), 256);
    *total = *o_bytes + align_up(pieces * R * sizeof(float), 256);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled through the runtime's driver entry point.
bool load_encode() {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        g_encode_status = cudaGetDriverEntryPointByVersion(
            "cuTensorMapEncodeTiled", reinterpret_cast<void**>(&g_encode), 12000,
            cudaEnableDefault, &q);
        if (g_encode_status == cudaSuccess && q != cudaDriverEntryPointSuccess)
            g_encode_status = cudaErrorNotSupported;
    });
    return g_encode_status == cudaSuccess && g_encode != nullptr;
}

// bf16 tensor map of any rank (2..5): dims[0] contiguous, strides_bytes[k]
// for dims[k + 1], 128-byte swizzle, zeros out of bounds.
int encode_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                const uint64_t* strides_bytes, const uint32_t* box) {
    if (!load_encode()) return MLA_ERR_CUDA;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], e[5];
    for (int k = 0; k < rank; ++k) {
        d[k] = dims[k];
        b[k] = box[k];
        e[k] = 1;
        if (k + 1 < rank) st[k] = strides_bytes[k];
    }
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                          const_cast<void*>(base), d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARGUMENT;
}

int encode_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box1) {
    if (!load_encode()) return MLA_ERR_CUDA;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {64, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARGUMENT;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_strerror(int code) {
    switch (code) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARGUMENT: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported configuration or device";
        case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MLA_ERR_CUDA: return "CUDA runtime error";
        case MLA_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
        case MLA_ERR_METADATA_MISMATCH: return "metadata was built for a different problem";
        case MLA_ERR_NO_DEVICE: return "no CUDA device";
        case MLA_ERR_SEQ_TOO_LONG: return "sequence longer than its block-table row";
        case MLA_ERR_BAD_ALIGNMENT: return "pointer or stride breaks the 16-byte alignment rule";
        case MLA_ERR_BAD_INDEX: return "a sparse key index points past the end of the cache";
        default: return "unknown error";
    }
}

int mla_version(void) { return 100; }

int mla_set_wait_budget_ns(uint64_t budget_ns) {
    g_budget_ns.store(budget_ns == 0 ? kDefaultBudgetNs : budget_ns);
    return MLA_OK;
}

int mla_set_decode_kernel(int kind) {
    if (kind != MLA_KERNEL_SINGLE && kind != MLA_KERNEL_TQ && kind != MLA_KERNEL_AUTO &&
        kind != MLA_KERNEL_DUO)
        return MLA_ERR_INVALID_ARGUMENT;
    g_kernel.store(kind);
    return MLA_OK;
}

int mla_get_decode_kernel(void) { return g_kernel.load(); }

int mla_set_fixed_overhead(int blocks) {
    g_fixed_overhead.store(blocks < 0 ? -1 : (blocks < 1 ? 1 : (blocks > 4096 ? 4096 : blocks)));
    return MLA_OK;
}

int mla_metadata_size(int batch, int h_q, int s_q, int h_kv, size_t* meta_bytes,
                      size_t* num_splits_bytes) {
    int st = check_shape(batch, h_q, s_q, h_kv);
    if (st) return st;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d))) return st;
    const Geo g = geo_of(batch, h_q, s_q, h_kv);
    const int parts = num_parts_of(g.R, h_kv, d);
    if (meta_bytes) *meta_bytes = sizeof(int32_t) * (kMetaHeader + static_cast<size_t>(parts > kMetaMinParts ? parts : kMetaMinParts) * kMetaFields);
    if (num_splits_bytes) *num_splits_bytes = sizeof(int32_t) * (static_cast<size_t>(g.nreq) + 1);
    return MLA_OK;
}

int mla_get_metadata(const int32_t* cache_seqlens_dev, int batch, int h_q, int s_q, int h_kv,
                     void* meta_dev, int32_t* num_splits_dev, mla_stream_t stream) {
    int st = check_shape(batch, h_q, s_q, h_kv);
    if (st) return st;
    if (!cache_seqlens_dev || !meta_dev || !num_splits_dev) return MLA_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(meta_dev) & 15u) || (reinterpret_cast<uintptr_t>(num_splits_dev) & 3u) ||
        (reinterpret_cast<uintptr_t>(cache_seqlens_dev) & 3u))
        return MLA_ERR_BAD_ALIGNMENT;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d))) return st;
    const Geo g = geo_of(batch, h_q, s_q, h_kv);
    const int parts = num_parts_of(g.R, h_kv, d);
    cudaError_t e = launch_sched(cache_seqlens_dev, h_kv, -1, g.nreq, g.R, parts,
                                 tiles_of(g.R, kernel_for(g.R, h_kv, d)),
                                 fixed_overhead_for(kernel_for(g.R, h_kv, d)),
                                 static_cast<int32_t*>(meta_dev), num_splits_dev,
                                 reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_workspace_size(int batch, int h_q, int s_q, int h_kv, size_t* bytes) {
    int st = check_shape(batch, h_q, s_q, h_kv);
    if (st) return st;
    if (!bytes) return MLA_ERR_INVALID_ARGUMENT;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d))) return st;
    const Geo g = geo_of(batch, h_q, s_q, h_kv);
    size_t ob = 0;
    workspace_layout(g.nreq, g.R, num_parts_of(g.R, h_kv, d), &ob, bytes);
    return MLA_OK;
}

}  // extern "C"

namespace {

int combine_core(const void* meta_dev, const int32_t* num_splits_dev, void* workspace_dev,
                 size_t workspace_bytes, int batch, int R, int parts, int s_q, int h_q, int fold,
                 int kvh, int grp, void* out_dev, int64_t out_batch_stride, int64_t out_s_stride,
                 int64_t out_h_stride, float* lse_dev, mla_stream_t stream, int dv = kDv);

int combine_only(const void* meta_dev, const int32_t* num_splits_dev, void* workspace_dev,
                 size_t workspace_bytes, int batch, int s_q, int h_q, int h_kv, void* out_dev,
                 int64_t out_batch_stride, int64_t out_s_stride, int64_t out_h_stride,
                 float* lse_dev, mla_stream_t stream) {
    int st = check_shape(batch, h_q, s_q, h_kv);
    if (st) return st;
    if (!meta_dev || !num_splits_dev || !out_dev || !lse_dev) return MLA_ERR_INVALID_ARGUMENT;
    if (out_h_stride < kDv || out_s_stride < out_h_stride * h_q ||
        out_batch_stride < out_s_stride * s_q)
        return MLA_ERR_INVALID_ARGUMENT;
    if (!aligned16(out_dev) || (out_batch_stride % 8) || (out_s_stride % 8) || (out_h_stride % 8) ||
        (reinterpret_cast<uintptr_t>(lse_dev) & 3u))
        return MLA_ERR_BAD_ALIGNMENT;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d))) return st;
    const Geo g = geo_of(batch, h_q, s_q, h_kv);
    return combine_core(meta_dev, num_splits_dev, workspace_dev, workspace_bytes, g.nreq, g.R,
                        num_parts_of(g.R, h_kv, d), s_q, h_q, 0, g.kvh, g.grp, out_dev,
                        out_batch_stride, out_s_stride, out_h_stride, lse_dev, stream);
}

// The combine launch for a plan of `batch` kernel requests of R rows each;
// fold > 0 for sparse decode (see DecodeParams::fold).
int combine_core(const void* meta_dev, const int32_t* num_splits_dev, void* workspace_dev,
                 size_t workspace_bytes, int batch, int R, int parts, int s_q, int h_q, int fold,
                 int kvh, int grp, void* out_dev, int64_t out_batch_stride, int64_t out_s_stride,
                 int64_t out_h_stride, float* lse_dev, mla_stream_t stream, int dv) {
    size_t o_bytes = 0, ws_need = 0;
    workspace_layout(batch, R, parts, &o_bytes, &ws_need);
    if (!workspace_dev || workspace_bytes < ws_need) return MLA_ERR_WORKSPACE_TOO_SMALL;
    if (reinterpret_cast<uintptr_t>(workspace_dev) & 255u) return MLA_ERR_BAD_ALIGNMENT;
    CombineParams c{};
    c.meta = static_cast<const int32_t*>(meta_dev);
    c.num_splits = num_splits_dev;
    c.oaccum = static_cast<const float*>(workspace_dev);
    c.lseaccum = reinterpret_cast<const float*>(static_cast<const char*>(workspace_dev) + o_bytes);
    c.out = static_cast<__nv_bfloat16*>(out_dev);
    c.out_sb = out_batch_stride;
    c.out_ss = out_s_stride;
    c.out_sh = out_h_stride;
    c.lse = lse_dev;
    c.batch = batch;
    c.s_q = s_q;
    c.h_q = h_q;
    c.R = R;
    c.num_parts = parts;
    c.fold = fold;
    c.kvh = kvh;
    c.grp = grp;
    c.dv = dv;
    cudaError_t e = launch_combine(c, reinterpret_cast<cudaStream_t>(stream), /*pdl=*/true);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int splitkv_only(const void* q_dev, int64_t q_batch_stride, const void* k_cache_dev,
                 int64_t k_page_stride, int64_t k_token_stride, int num_pages, int page_size,
                 const int32_t* block_table_dev, int64_t bt_batch_stride, int max_blocks_per_seq,
                 const int32_t* cache_seqlens_dev, int batch, int s_q, int h_q, int h_kv,
                 float softmax_scale, int causal, const void* meta_dev,
                 const int32_t* num_splits_dev, void* workspace_dev, size_t workspace_bytes,
                 void* out_dev, int64_t out_batch_stride, int64_t out_s_stride,
                 int64_t out_h_stride, float* lse_dev, mla_stream_t stream, int d_qk = kDqk,
                 int d_v = kDv) {
    int st = check_shape(batch, h_q, s_q, h_kv);
    if (st) return st;
    if (page_size != kPage) return MLA_ERR_UNSUPPORTED;
    // Other head sizes: 64-dim chunks, V the first d_v dims of each K row, one
    // cache head, on the single-CTA kernel.
    const bool general = d_qk != kDqk || d_v != kDv;
    if (general && (d_qk % 64 || d_qk < 64 || d_qk > kDqk || d_v % 64 || d_v < 64 ||
                    d_v > kDv || d_v > d_qk || h_kv != 1))
        return MLA_ERR_UNSUPPORTED;
    if (!q_dev || !k_cache_dev || !block_table_dev || !cache_seqlens_dev || !meta_dev ||
        !num_splits_dev || !out_dev || !lse_dev)
        return MLA_ERR_INVALID_ARGUMENT;
    if (num_pages < 1 || max_blocks_per_seq < 1 || bt_batch_stride < max_blocks_per_seq ||
        q_batch_stride < static_cast<int64_t>(s_q) * h_q * d_qk ||
        k_token_stride < static_cast<int64_t>(h_kv) * d_qk ||
        k_page_stride < k_token_stride * kPage || out_h_stride < d_v ||
        out_s_stride < out_h_stride * h_q || out_batch_stride < out_s_stride * s_q ||
        !std::isfinite(softmax_scale) || (causal != 0 && causal != 1))
        return MLA_ERR_INVALID_ARGUMENT;
    // TMA: 16-byte aligned bases and strides; vector stores: 16-byte aligned rows.
    if (!aligned16(q_dev) || !aligned16(k_cache_dev) || !aligned16(out_dev) ||
        (q_batch_stride % 8) || (k_page_stride % 8) || (k_token_stride % 8) ||
        (out_batch_stride % 8) || (out_s_stride % 8) || (out_h_stride % 8) ||
        (reinterpret_cast<uintptr_t>(lse_dev) & 3u))
        return MLA_ERR_BAD_ALIGNMENT;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d))) return st;
    const Geo g = geo_of(batch, h_q, s_q, h_kv);
    const int R = g.R;
    // (The plan's part count is mla_get_metadata's, for whichever kernel it
    // was made; the single-CTA kernel runs any part count.)
    const int parts = num_parts_of(R, h_kv, d);
    const int kind = general ? MLA_KERNEL_SINGLE : kernel_for(R, h_kv, d);
    size_t o_bytes = 0, ws_need = 0;
    workspace_layout(g.nreq, R, parts, &o_bytes, &ws_need);
    if (!workspace_dev || workspace_bytes < ws_need) return MLA_ERR_WORKSPACE_TOO_SMALL;
    if (reinterpret_cast<uintptr_t>(workspace_dev) & 255u) return MLA_ERR_BAD_ALIGNMENT;

    CUtensorMap q_map, kv_map;
    uint32_t q_box_rows = R < kTileM ? static_cast<uint32_t>(R) : kTileM;
    if (kind == MLA_KERNEL_DUO) q_box_rows = kTileM;  // each CTA of a pair loads 64 rows
    if (h_kv == 1) {
        st = encode_3d(&q_map, q_dev, d_qk, static_cast<uint64_t>(R), static_cast<uint64_t>(batch),
                       d_qk * 2, static_cast<uint64_t>(q_batch_stride) * 2, q_box_rows);
        if (st) return st;
        st = encode_3d(&kv_map, k_cache_dev, d_qk, kPage, static_cast<uint64_t>(num_pages),
                       static_cast<uint64_t>(k_token_stride) * 2,
                       static_cast<uint64_t>(k_page_stride) * 2, kPage);
        if (st) return st;
    } else {
        // Q as (576, grp, h_kv, s_q, b): a box brings a tile's rows s * grp + hh
        // of one head group (64 / grp tokens, or a 64-head slice of a token).
        const uint32_t gb = g.grp <= kTileM ? static_cast<uint32_t>(g.grp) : kTileM;
        const uint32_t sb = g.grp <= kTileM ? static_cast<uint32_t>(
                                                  s_q < kTileM / g.grp ? s_q : kTileM / g.grp)
                                            : 1u;
        q_box_rows = gb * sb;
        const uint64_t qd[5] = {kDqk, static_cast<uint64_t>(g.grp), static_cast<uint64_t>(h_kv),
                                static_cast<uint64_t>(s_q), static_cast<uint64_t>(batch)};
        const uint64_t qs[4] = {kDqk * 2, static_cast<uint64_t>(g.grp) * kDqk * 2,
                                static_cast<uint64_t>(h_q) * kDqk * 2,
                                static_cast<uint64_t>(q_batch_stride) * 2};
        const uint32_t qb[5] = {64, gb, 1, sb, 1};
        st = encode_bf16(&q_map, q_dev, 5, qd, qs, qb);
        if (st) return st;
        // Cache as (576, h_kv, 64, pages): the heads of a token adjacent.
        const uint64_t kd[4] = {kDqk, static_cast<uint64_t>(h_kv), kPage,
                                static_cast<uint64_t>(num_pages)};
        const uint64_t ks[3] = {kDqk * 2, static_cast<uint64_t>(k_token_stride) * 2,
                                static_cast<uint64_t>(k_page_stride) * 2};
        const uint32_t kb[4] = {64, 1, kPage, 1};
        st = encode_bf16(&kv_map, k_cache_dev, 4, kd, ks, kb);
        if (st) return st;
    }

    DecodeParams p{};
    p.block_table = block_table_dev;
    p.bt_stride = bt_batch_stride;
    p.max_blocks = max_blocks_per_seq;
    p.seqlens = cache_seqlens_dev;
    p.meta = static_cast<const int32_t*>(meta_dev);
    p.num_splits = num_splits_dev;
    p.out = static_cast<__nv_bfloat16*>(out_dev);
    p.out_sb = out_batch_stride;
    p.out_ss = out_s_stride;
    p.out_sh = out_h_stride;
    p.lse = lse_dev;
    p.oaccum = static_cast<float*>(workspace_dev);
    p.lseaccum = reinterpret_cast<float*>(static_cast<char*>(workspace_dev) + o_bytes);
    p.batch = g.nreq;
    p.s_q = s_q;
    p.h_q = h_q;
    p.R = R;
    p.n_mtiles = tiles_of(R, kind);
    p.num_parts = parts;
    p.q_box_rows = static_cast<int>(q_box_rows);
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.causal = causal;
    p.error_word = d->error_word;
    p.budget_ns = g_budget_ns.load();
    p.stage_p = p.n_mtiles == 1 ? 1 : 0;
    p.kvh = g.kvh;
    p.grp = g.grp;
    if (general) {
        p.nc = d_qk / 64;
        p.nv = d_v / 64;
    }

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = kind == MLA_KERNEL_TQ    ? launch_decode_tq(p, q_map, kv_map, s)
                    : kind == MLA_KERNEL_DUO ? launch_decode_duo(p, q_map, kv_map, s)
                                             : launch_decode(p, q_map, kv_map, s);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

extern "C" {

int mla_decode_splitkv(const void* q_dev, int64_t q_batch_stride, const void* k_cache_dev,
                       int64_t k_page_stride, int64_t k_token_stride, int num_pages, int page_size,
                       const int32_t* block_table_dev, int64_t bt_batch_stride,
                       int max_blocks_per_seq, const int32_t* cache_seqlens_dev, int batch,
                       int s_q, int h_q, int h_kv, float softmax_scale, int causal,
                       const void* meta_dev, const int32_t* num_splits_dev, void* workspace_dev,
                       size_t workspace_bytes, void* out_dev, int64_t out_batch_stride,
                       int64_t out_s_stride, int64_t out_h_stride, float* lse_dev,
                       mla_stream_t stream) {
    return splitkv_only(q_dev, q_batch_stride, k_cache_dev, k_page_stride, k_token_stride,
                        num_pages, page_size, block_table_dev, bt_batch_stride, max_blocks_per_seq,
                        cache_seqlens_dev, batch, s_q, h_q, h_kv, softmax_scale, causal, meta_dev,
                        num_splits_dev, workspace_dev, workspace_bytes, out_dev, out_batch_stride,
                        out_s_stride, out_h_stride, lse_dev, stream);
}

int mla_decode_combine(const void* meta_dev, const int32_t* num_splits_dev, void* workspace_dev,
                       size_t workspace_bytes, int batch, int s_q, int h_q, int h_kv,
                       void* out_dev, int64_t out_batch_stride, int64_t out_s_stride,
                       int64_t out_h_stride, float* lse_dev, mla_stream_t stream) {
    return combine_only(meta_dev, num_splits_dev, workspace_dev, workspace_bytes, batch, s_q, h_q,
                        h_kv, out_dev, out_batch_stride, out_s_stride, out_h_stride, lse_dev,
                        stream);
}

int mla_decode_fwd(const void* q_dev, int64_t q_batch_stride, const void* k_cache_dev,
                   int64_t k_page_stride, int64_t k_token_stride, int num_pages, int page_size,
                   const int32_t* block_table_dev, int64_t bt_batch_stride, int max_blocks_per_seq,
                   const int32_t* cache_seqlens_dev, int batch, int s_q, int h_q, int h_kv,
                   float softmax_scale, int causal, const void* meta_dev,
                   const int32_t* num_splits_dev, void* workspace_dev, size_t workspace_bytes,
                   void* out_dev, int64_t out_batch_stride, int64_t out_s_stride,
                   int64_t out_h_stride, float* lse_dev, mla_stream_t stream) {
    int st = splitkv_only(q_dev, q_batch_stride, k_cache_dev, k_page_stride, k_token_stride,
                          num_pages, page_size, block_table_dev, bt_batch_stride,
                          max_blocks_per_seq, cache_seqlens_dev, batch, s_q, h_q, h_kv,
                          softmax_scale, causal, meta_dev, num_splits_dev, workspace_dev,
                          workspace_bytes, out_dev, out_batch_stride, out_s_stride, out_h_stride,
                          lse_dev, stream);
    if (st) return st;
    return combine_only(meta_dev, num_splits_dev, workspace_dev, workspace_bytes, batch, s_q, h_q,
                        h_kv, out_dev, out_batch_stride, out_s_stride, out_h_stride, lse_dev,
                        stream);
}

int mla_decode_fwd_dims(const void* q_dev, int64_t q_batch_stride, const void* k_cache_dev,
                        int64_t k_page_stride, int64_t k_token_stride, int num_pages,
                        int page_size, const int32_t* block_table_dev, int64_t bt_batch_stride,
                        int max_blocks_per_seq, const int32_t* cache_seqlens_dev, int batch,
                        int s_q, int h_q, int h_kv, int d_qk, int d_v, float softmax_scale,
                        int causal, const void* meta_dev, const int32_t* num_splits_dev,
                        void* workspace_dev, size_t workspace_bytes, void* out_dev,
                        int64_t out_batch_stride, int64_t out_s_stride, int64_t out_h_stride,
                        float* lse_dev, mla_stream_t stream) {
    int st = splitkv_only(q_dev, q_batch_stride, k_cache_dev, k_page_stride, k_token_stride,
                          num_pages, page_size, block_table_dev, bt_batch_stride,
                          max_blocks_per_seq, cache_seqlens_dev, batch, s_q, h_q, h_kv,
                          softmax_scale, causal, meta_dev, num_splits_dev, workspace_dev,
                          workspace_bytes, out_dev, out_batch_stride, out_s_stride, out_h_stride,
                          lse_dev, stream, d_qk, d_v);
    if (st) return st;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d))) return st;
    const Geo g = geo_of(batch, h_q, s_q, h_kv);
    return combine_core(meta_dev, num_splits_dev, workspace_dev, workspace_bytes, g.nreq, g.R,
                        num_parts_of(g.R, h_kv, d), s_q, h_q, 0, g.kvh, g.grp, out_dev,
                        out_batch_stride, out_s_stride, out_h_stride, lse_dev, stream, d_v);
}

int mla_metadata_size_sparse(int batch, int h_q, int s_q, int h_kv, size_t* meta_bytes,
                             size_t* num_splits_bytes) {
    int st = check_shape_sparse(batch, h_q, s_q, h_kv, 0);
    if (st) return st;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d))) return st;
    const int parts = num_parts_sparse(h_q, d);
    if (meta_bytes)
        *meta_bytes = sizeof(int32_t) * (kMetaHeader + static_cast<size_t>(parts > kMetaMinParts ? parts : kMetaMinParts) * kMetaFields);
    if (num_splits_bytes)
        *num_splits_bytes = sizeof(int32_t) * (static_cast<size_t>(batch) * s_q + 1);
    return MLA_OK;
}

int mla_get_metadata_sparse(int topk, int batch, int h_q, int s_q, int h_kv, void* meta_dev,
                            int32_t* num_splits_dev, mla_stream_t stream) {
    int st = check_shape_sparse(batch, h_q, s_q, h_kv, topk);
    if (st) return st;
    if (!meta_dev || !num_splits_dev) return MLA_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(meta_dev) & 15u) ||
        (reinterpret_cast<uintptr_t>(num_splits_dev) & 3u))
        return MLA_ERR_BAD_ALIGNMENT;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d))) return st;
    const int kind = sparse_kind(h_q, d);
    cudaError_t e = launch_sched(nullptr, 1, topk, batch * s_q, h_q, num_parts_sparse(h_q, d),
                                 tiles_of(h_q, kind), fixed_overhead_for(kind),
                                 static_cast<int32_t*>(meta_dev), num_splits_dev,
                                 reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_workspace_size_sparse(int batch, int h_q, int s_q, int h_kv, size_t* bytes) {
    int st = check_shape_sparse(batch, h_q, s_q, h_kv, 0);
    if (st) return st;
    if (!bytes) return MLA_ERR_INVALID_ARGUMENT;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d))) return st;
    size_t ob = 0;
    workspace_layout(batch * s_q, h_q, num_parts_sparse(h_q, d), &ob, bytes);
    return MLA_OK;
}

int mla_decode_sparse_fwd(const void* q_dev, int64_t q_batch_stride, const void* k_cache_dev,
                          int64_t k_page_stride, int64_t k_token_stride, int num_pages,
                          int page_size, const int32_t* indices_dev, int topk, int batch, int s_q,
                          int h_q, int h_kv, float softmax_scale, const void* meta_dev,
                          const int32_t* num_splits_dev, void* workspace_dev,
                          size_t workspace_bytes, void* out_dev, int64_t out_batch_stride,
                          int64_t out_s_stride, int64_t out_h_stride, float* lse_dev,
                          mla_stream_t stream) {
    int st = check_shape_sparse(batch, h_q, s_q, h_kv, topk);
    if (st) return st;
    if (page_size != kPage) return MLA_ERR_UNSUPPORTED;
    if (!q_dev || !k_cache_dev || (!indices_dev && topk > 0) || !meta_dev || !num_splits_dev ||
        !out_dev || !lse_dev)
        return MLA_ERR_INVALID_ARGUMENT;
    const int64_t q_tok = static_cast<int64_t>(h_q) * kDqk;  // one query token's rows
    if (num_pages < 1 || static_cast<int64_t>(num_pages) * kPage > INT32_MAX ||
        q_batch_stride < s_q * q_tok || k_token_stride < kDqk ||
        k_page_stride < k_token_stride * kPage || out_h_stride < kDv ||
        out_s_stride < out_h_stride * h_q || out_batch_stride < out_s_stride * s_q ||
        !std::isfinite(softmax_scale))
        return MLA_ERR_INVALID_ARGUMENT;
    // The gather addresses the cache as one [num_pages * 64 x 576] row array,
    // and the Q map walks the (request, query token) pairs with one stride.
    if (k_page_stride != k_token_stride * kPage) return MLA_ERR_UNSUPPORTED;
    if (batch > 1 && s_q > 1 && q_batch_stride != s_q * q_tok) return MLA_ERR_UNSUPPORTED;
    if (!aligned16(q_dev) || !aligned16(k_cache_dev) || !aligned16(out_dev) ||
        (q_batch_stride % 8) || (k_token_stride % 8) || (out_batch_stride % 8) ||
        (out_s_stride % 8) || (out_h_stride % 8) ||
        (reinterpret_cast<uintptr_t>(lse_dev) & 3u) ||
        (reinterpret_cast<uintptr_t>(indices_dev) & 3u))
        return MLA_ERR_BAD_ALIGNMENT;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d))) return st;
    const int nreq = batch * s_q, R = h_q;
    const int kind = sparse_kind(R, d);
    const int parts = num_parts_sparse(R, d);
    size_t o_bytes = 0, ws_need = 0;
    workspace_layout(nreq, R, parts, &o_bytes, &ws_need);
    if (!workspace_dev || workspace_bytes < ws_need) return MLA_ERR_WORKSPACE_TOO_SMALL;
    if (reinterpret_cast<uintptr_t>(workspace_dev) & 255u) return MLA_ERR_BAD_ALIGNMENT;

    CUtensorMap q_map, kv_map;
    // (Each CTA of a pair loads 64 query rows.)
    const uint32_t q_box_rows = R < kTileM ? static_cast<uint32_t>(R) : kTileM;
    const int64_t q_req_stride = s_q == 1 ? q_batch_stride : q_tok;
    st = encode_3d(&q_map, q_dev, kDqk, static_cast<uint64_t>(R), static_cast<uint64_t>(nreq),
                   kDqk * 2, static_cast<uint64_t>(q_req_stride) * 2, q_box_rows);
    if (st) return st;
    const int64_t num_tokens = static_cast<int64_t>(num_pages) * kPage;
    // (The page map is not read in sparse mode; the kernel takes one.)
    st = encode_3d(&kv_map, k_cache_dev, kDqk, kPage, static_cast<uint64_t>(num_pages),
                   static_cast<uint64_t>(k_token_stride) * 2,
                   static_cast<uint64_t>(k_page_stride) * 2, kPage);
    if (st) return st;

    DecodeParams p{};
    p.max_blocks = topk > 0 ? (topk + kPage - 1) / kPage : 1;
    p.meta = static_cast<const int32_t*>(meta_dev);
    p.num_splits = num_splits_dev;
    p.out = static_cast<__nv_bfloat16*>(out_dev);
    p.out_sb = out_batch_stride;
    p.out_ss = out_s_stride;
    p.out_sh = out_h_stride;
    p.lse = lse_dev;
    p.oaccum = static_cast<float*>(workspace_dev);
    p.lseaccum = reinterpret_cast<float*>(static_cast<char*>(workspace_dev) + o_bytes);
    p.batch = nreq;
    p.s_q = s_q;
    p.h_q = h_q;
    p.R = R;
    p.n_mtiles = tiles_of(R, kind);
    p.num_parts = parts;
    p.q_box_rows = static_cast<int>(q_box_rows);
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.causal = 0;
    p.error_word = d->error_word;
    p.budget_ns = g_budget_ns.load();
    p.sparse = 1;
    p.indices = indices_dev;
    p.topk = topk;
    p.num_tokens = num_tokens;
    p.kv_bytes = static_cast<const uint8_t*>(k_cache_dev);
    p.kv_token_bytes = k_token_stride * 2;
    p.fold = s_q;
    p.stage_p = p.n_mtiles == 1 ? 1 : 0;
    p.kvh = 1;
    p.grp = h_q;
    cudaError_t e =
        kind == MLA_KERNEL_DUO
            ? launch_decode_duo(p, q_map, kv_map, reinterpret_cast<cudaStream_t>(stream))
            : launch_decode(p, q_map, kv_map, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    return combine_core(meta_dev, num_splits_dev, workspace_dev, workspace_bytes, nreq, R, parts,
                        s_q, h_q, s_q, 1, h_q, out_dev, out_batch_stride, out_s_stride,
                        out_h_stride, lse_dev, stream);
}

int mla_decode_fp8_fwd(const void* q_dev, int64_t q_batch_stride, const void* k_cache_dev,
                       int64_t k_page_stride_bytes, int num_pages, int page_size,
                       const int32_t* block_table_dev, int64_t bt_batch_stride,
                       int max_blocks_per_seq, const int32_t* cache_seqlens_dev, int batch,
                       int s_q, int h_q, int h_kv, float softmax_scale, int causal,
                       const void* meta_dev, const int32_t* num_splits_dev, void* workspace_dev,
                       size_t workspace_bytes, void* out_dev, int64_t out_batch_stride,
                       int64_t out_s_stride, int64_t out_h_stride, float* lse_dev,
                       mla_stream_t stream) {
    constexpr int64_t kRow = 656, kPageBytes = 64 * kRow;
    int st = check_shape(batch, h_q, s_q, h_kv);
    if (st) return st;
    if (h_kv != 1) return MLA_ERR_UNSUPPORTED;
    if (page_size != kPage) return MLA_ERR_UNSUPPORTED;
    if (!q_dev || !k_cache_dev || !block_table_dev || !cache_seqlens_dev || !meta_dev ||
        !num_splits_dev || !out_dev || !lse_dev)
        return MLA_ERR_INVALID_ARGUMENT;
    if (num_pages < 1 || static_cast<int64_t>(num_pages) * kPage > INT32_MAX ||
        max_blocks_per_seq < 1 || bt_batch_stride < max_blocks_per_seq ||
        q_batch_stride < static_cast<int64_t>(s_q) * h_q * kDqk ||
        k_page_stride_bytes < kPageBytes || out_h_stride < kDv ||
        out_s_stride < out_h_stride * h_q || out_batch_stride < out_s_stride * s_q ||
        !std::isfinite(softmax_scale) || (causal != 0 && causal != 1))
        return MLA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q_dev) || !aligned16(k_cache_dev) || !aligned16(out_dev) ||
        (q_batch_stride % 8) || (k_page_stride_bytes % 16) || (out_batch_stride % 8) ||
        (out_s_stride % 8) || (out_h_stride % 8) || (reinterpret_cast<uintptr_t>(lse_dev) & 3u))
        return MLA_ERR_BAD_ALIGNMENT;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d))) return st;
    const int R = s_q * h_q;
    // The plan is mla_get_metadata's (whatever kernel it was sized for); the
    // single-CTA kernel runs it with its own 64-row tiles.
    const int parts = num_parts_of(R, 1, d);
    size_t o_bytes = 0, ws_need = 0;
    workspace_layout(batch, R, parts, &o_bytes, &ws_need);
    if (!workspace_dev || workspace_bytes < ws_need) return MLA_ERR_WORKSPACE_TOO_SMALL;
    if (reinterpret_cast<uintptr_t>(workspace_dev) & 255u) return MLA_ERR_BAD_ALIGNMENT;

    CUtensorMap q_map;
    const uint32_t q_box_rows = R < kTileM ? static_cast<uint32_t>(R) : kTileM;
    st = encode_3d(&q_map, q_dev, kDqk, static_cast<uint64_t>(R), static_cast<uint64_t>(batch),
                   kDqk * 2, static_cast<uint64_t>(q_batch_stride) * 2, q_box_rows);
    if (st) return st;

    DecodeParams p{};
    p.block_table = block_table_dev;
    p.bt_stride = bt_batch_stride;
    p.max_blocks = max_blocks_per_seq;
    p.seqlens = cache_seqlens_dev;
    p.meta = static_cast<const int32_t*>(meta_dev);
    p.num_splits = num_splits_dev;
    p.out = static_cast<__nv_bfloat16*>(out_dev);
    p.out_sb = out_batch_stride;
    p.out_ss = out_s_stride;
    p.out_sh = out_h_stride;
    p.lse = lse_dev;
    p.oaccum = static_cast<float*>(workspace_dev);
    p.lseaccum = reinterpret_cast<float*>(static_cast<char*>(workspace_dev) + o_bytes);
    p.batch = batch;
    p.s_q = s_q;
    p.h_q = h_q;
    p.R = R;
    p.n_mtiles = n_mtiles_of(R);
    p.num_parts = parts;
    p.q_box_rows = static_cast<int>(q_box_rows);
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.causal = causal;
    p.error_word = d->error_word;
    p.budget_ns = g_budget_ns.load();
    p.fp8 = 1;
    p.kv_bytes = static_cast<const uint8_t*>(k_cache_dev);
    p.kv_page_bytes = k_page_stride_bytes;
    p.num_tokens = static_cast<int64_t>(num_pages) * kPage;
    p.stage_p = p.n_mtiles == 1 ? 1 : 0;
    p.kvh = 1;
    p.grp = h_q;
    // The kernel that keeps Q in tensor memory (three stages) where the dense
    // path would use it, else the single-CTA kernel.  (Both take a page
    // tensor map too; the FP8 path never reads it.)
    const bool tq = kernel_for(R, 1, d) == MLA_KERNEL_TQ;
    cudaError_t e = tq ? launch_decode_tq(p, q_map, q_map, reinterpret_cast<cudaStream_t>(stream))
                       : launch_decode(p, q_map, q_map, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    return combine_core(meta_dev, num_splits_dev, workspace_dev, workspace_bytes, batch, R, parts,
                        s_q, h_q, 0, 1, h_q, out_dev, out_batch_stride, out_s_stride,
                        out_h_stride, lse_dev, stream);
}

int mla_last_device_error(mla_stream_t stream, int* code) {
    if (!code) return MLA_ERR_INVALID_ARGUMENT;
    DeviceInfo* d = nullptr;
    int st = device_info(&d);
    if (st) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
    int v = 0, zero = 0;
    if (cudaMemcpy(&v, d->error_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (cudaMemcpy(d->error_word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
        return MLA_ERR_CUDA;
    *code = v;
    return MLA_OK;
}

}  // extern "C"
