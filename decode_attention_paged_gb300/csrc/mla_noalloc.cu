// mla_noalloc.cu -- mla_decode_fwd_noalloc: the decode call for callers that
// cannot allocate device memory (see include/mla_decode.h for who they are).
//
// The split-KV scratch that mla_decode_fwd otherwise takes from the caller
// lives here, in a file-scope device array of fixed size.  The array is part of
// the library's device image: every GPU that loads the library holds it until
// the process exits, whether or not this entry point is ever called.
//
// Host code must not use the array's name as a pointer: on the host it names a
// stand-in object, not device memory.  The device address is fetched once per
// device with cudaGetSymbolAddress (with that device current) and then passed
// to the kernels like any caller-provided workspace.
#include <mutex>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr size_t kNoAllocScratchBytes = MLA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxNoAllocDevices = 64;

// Partial outputs and log-sum-exps of split requests, shared by all calls.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array, per device.  Only a successful lookup is
// kept: a lookup that failed (for instance during a stream capture, where the
// runtime may refuse the call) is tried again on the next call.
struct ScratchAddress {
    std::mutex lock;
    void* ptr = nullptr;  // non-null once resolved
};
ScratchAddress g_scratch_address[kMaxNoAllocDevices];

void* scratch_address(int dev) {
    ScratchAddress& s = g_scratch_address[dev];
    std::lock_guard<std::mutex> guard(s.lock);
    if (s.ptr == nullptr) {
        // The current device is `dev`, so this resolves the array's copy on it.
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) == cudaSuccess) {
            s.ptr = p;
        } else {
            cudaGetLastError();  // clear the error state so that a later call can try again
        }
    }
    return s.ptr;
}

}  // namespace
}  // namespace mla

extern "C" int mla_decode_fwd_noalloc(
    const void* q_dev, int64_t q_batch_stride, const void* k_cache_dev, int64_t k_page_stride,
    int64_t k_token_stride, int num_pages, int page_size, const int32_t* block_table_dev,
    int64_t bt_batch_stride, int max_blocks_per_seq, const int32_t* cache_seqlens_dev, int batch,
    int s_q, int h_q, int h_kv, float softmax_scale, int causal, const void* meta_dev,
    const int32_t* num_splits_dev, void* out_dev, int64_t out_batch_stride, int64_t out_s_stride,
    int64_t out_h_stride, float* lse_dev, mla_stream_t stream) {
    using namespace mla;
    // Shape and device checks first (also reports a missing GPU).
    size_t need = 0;
    int st = mla_workspace_size(batch, h_q, s_q, h_kv, &need);
    if (st != MLA_OK) return st;
    if (need > kNoAllocScratchBytes) return MLA_ERR_WORKSPACE_TOO_SMALL;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxNoAllocDevices) return MLA_ERR_UNSUPPORTED;
    void* scratch = scratch_address(dev);
    if (scratch == nullptr) return MLA_ERR_CUDA;

    return mla_decode_fwd(q_dev, q_batch_stride, k_cache_dev, k_page_stride, k_token_stride,
                          num_pages, page_size, block_table_dev, bt_batch_stride,
                          max_blocks_per_seq, cache_seqlens_dev, batch, s_q, h_q, h_kv,
                          softmax_scale, causal, meta_dev, num_splits_dev, scratch,
                          kNoAllocScratchBytes, out_dev, out_batch_stride, out_s_stride,
                          out_h_stride, lse_dev, stream);
}
