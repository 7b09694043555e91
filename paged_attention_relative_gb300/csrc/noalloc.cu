// rel_attn_paged_varlen_noalloc: rel_attn_paged_varlen with its split-KV
// workspace taken from a fixed device array instead of a stream-ordered
// allocation.  For callers that must not allocate device memory: a framework
// that owns the device through its own memory pool (a second allocator behind
// its back can run out of memory while the pool holds nearly all of the
// device, or fragment it), or a program that allocates everything at start-up
// and forbids allocation afterwards.
//
// Everything but the workspace is the allocating entry point's own code
// (paged_varlen in api.cu): the same validation, status codes, kernels,
// REL_ATTN_CHECK device check, wait timeout and launch record.  The scratch
// array lives in this module, one copy per device that loads the library,
// held until the process exits.  Calls share it; see the header for the rules
// that follow from that.

#include <cstdio>
#include <mutex>

#include "kernels.h"
#include "rel_attn.h"

namespace relattn {

namespace {

constexpr size_t kScratchBytes = REL_ATTN_NOALLOC_SCRATCH_BYTES;

// File-scope scratch: split partials (fp32 O) followed by their log2-sum-exp.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Once per device, with that device current: the device address of the
// scratch array (in host code its name is only a host-side stand-in, not a
// device address).
rel_attn_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        char buf[256];
        snprintf(buf, sizeof buf, "noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        set_last_error_message(buf);
        return REL_ATTN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_last_error_message("noalloc: device ordinal too large");
        return REL_ATTN_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            char buf[256];
            snprintf(buf, sizeof buf, "noalloc: cudaGetSymbolAddress of the scratch array failed: %s",
                     cudaGetErrorString(e));
            set_last_error_message(buf);
            return REL_ATTN_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return REL_ATTN_OK;
}

}  // namespace
}  // namespace relattn

using namespace relattn;

extern "C" rel_attn_status rel_attn_paged_varlen_noalloc(
    const rel_attn_tensor* q, const rel_attn_tensor* key_cache, const rel_attn_tensor* value_cache,
    const rel_attn_tensor* block_table, const rel_attn_tensor* cache_seqlens, const rel_attn_tensor* cu_seqlens_q,
    int32_t max_seqlen_q, float softmax_scale, int32_t causal, int32_t window_left, int32_t window_right,
    int32_t rel_extent, const rel_attn_tensor* rel_logits, int32_t num_splits, rel_attn_tensor* out,
    rel_attn_stream stream) {
    const FixedWorkspace ws{scratch_address, kScratchBytes};
    return paged_varlen(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q, max_seqlen_q,
                        softmax_scale, causal, window_left, window_right, rel_extent, rel_logits, num_splits, out,
                        nullptr, stream, &ws);
}
