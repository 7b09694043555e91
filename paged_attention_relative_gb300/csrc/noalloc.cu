// rel_attn_paged_varlen_noalloc: the decode path of rel_attn_paged_varlen
// with its split-KV scratch taken from a fixed device array instead of a
// stream-ordered allocation.  For callers that must not allocate device
// memory: a framework that owns the device through its own memory pool (a
// second allocator behind its back can run out of memory while the pool
// holds nearly all of the device, or fragment it), or a program that
// allocates everything at start-up and forbids allocation afterwards.
//
// The scratch array lives in this module, one copy per device that loads the
// library, held until the process exits.  Calls share it; see the header for
// the rules that follow from that.

#include <cstdio>
#include <mutex>

#include "kernels.h"
#include "rel_attn.h"

namespace relattn {

void set_last_error_message(const char* msg);
int* device_error_word();

namespace {

constexpr size_t kScratchBytes = REL_ATTN_NOALLOC_SCRATCH_BYTES;

// File-scope scratch: split partials (fp32 O) followed by their log2-sum-exp.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchInfo {
    bool ready = false;
    void* ptr = nullptr;
    int major = 0, minor = 0, sms = 0;
};
ScratchInfo g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

rel_attn_status nfail(rel_attn_status st, const char* msg) {
    set_last_error_message(msg);
    return st;
}

// Once per device, with that device current: the device address of the
// scratch array (in host code its name is only a host-side stand-in).
rel_attn_status scratch_setup(ScratchInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nfail(REL_ATTN_ERR_CUDA, "noalloc: cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices) return nfail(REL_ATTN_ERR_UNSUPPORTED, "noalloc: device ordinal too large");
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchInfo& s = g_scratch[dev];
    if (!s.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
            return nfail(REL_ATTN_ERR_CUDA, "noalloc: cudaGetDeviceProperties failed");
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            char buf[256];
            snprintf(buf, sizeof buf, "noalloc: cudaGetSymbolAddress of the scratch array failed: %s",
                     cudaGetErrorString(e));
            return nfail(REL_ATTN_ERR_CUDA, buf);
        }
        s.ptr = p;
        s.major = prop.major;
        s.minor = prop.minor;
        s.sms = prop.multiProcessorCount;
        s.ready = true;
    }
    *out = &s;
    return REL_ATTN_OK;
}

bool is(const rel_attn_tensor* t, int dtype, int ndim) {
    if (!t || t->dtype != dtype || t->ndim != ndim) return false;
    int64_t n = 1;
    for (int i = 0; i < ndim; ++i) {
        if (t->shape[i] < 0) return false;
        n *= t->shape[i];
    }
    return n == 0 || t->data != nullptr;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace relattn

using namespace relattn;

extern "C" rel_attn_status rel_attn_paged_varlen_noalloc(
    const rel_attn_tensor* q, const rel_attn_tensor* key_cache, const rel_attn_tensor* value_cache,
    const rel_attn_tensor* block_table, const rel_attn_tensor* cache_seqlens, const rel_attn_tensor* cu_seqlens_q,
    int32_t max_seqlen_q, float softmax_scale, int32_t causal, int32_t window_left, int32_t window_right,
    int32_t rel_extent, const rel_attn_tensor* rel_logits, int32_t num_splits, rel_attn_tensor* out,
    rel_attn_stream stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const rel_attn_status bad = REL_ATTN_ERR_INVALID_ARGUMENT;
    if (!is(q, REL_ATTN_BF16, 3) || !is(key_cache, REL_ATTN_BF16, 4) || !is(value_cache, REL_ATTN_BF16, 4) ||
        !is(block_table, REL_ATTN_I32, 2) || !is(cache_seqlens, REL_ATTN_I32, 1) || !is(cu_seqlens_q, REL_ATTN_I32, 1) ||
        !out || !is(out, out->dtype == REL_ATTN_F32 ? REL_ATTN_F32 : REL_ATTN_BF16, 3))
        return nfail(bad, "noalloc: a tensor descriptor has the wrong dtype or rank, or NULL data");
    const int64_t T = q->shape[0], H = q->shape[1], D = q->shape[2];
    const int64_t NB = key_cache->shape[0], BS = key_cache->shape[1], Hk = key_cache->shape[2];
    const int64_t B = block_table->shape[0], MB = block_table->shape[1];
    const int out_elem = out->dtype == REL_ATTN_F32 ? 4 : 2;
    for (int i = 0; i < 4; ++i)
        if (value_cache->shape[i] != key_cache->shape[i] || value_cache->stride[i] != key_cache->stride[i])
            return nfail(bad, "noalloc: value_cache must have the shape and strides of key_cache");
    if (key_cache->shape[3] != D || out->shape[0] != T || out->shape[1] != H || out->shape[2] != D ||
        cache_seqlens->shape[0] != B || cu_seqlens_q->shape[0] != B + 1 || cache_seqlens->stride[0] != 1 ||
        cu_seqlens_q->stride[0] != 1 || (MB > 0 && block_table->stride[1] != 1) ||
        (B > 0 && block_table->stride[0] < MB))
        return nfail(bad, "noalloc: inconsistent shapes or strides");
    if (H <= 0 || Hk <= 0 || H % Hk != 0) return nfail(bad, "noalloc: num_heads must be a multiple of num_kv_heads");
    if (num_splits < 1 || rel_extent < 0 || max_seqlen_q < 0)
        return nfail(bad, "noalloc: num_splits >= 1, rel_extent >= 0 and max_seqlen_q >= 0 are required");
    if (rel_extent > 0 &&
        (!(is(rel_logits, REL_ATTN_BF16, 3) || is(rel_logits, REL_ATTN_F32, 3)) || rel_logits->shape[0] != T || rel_logits->shape[1] != H ||
         rel_logits->shape[2] != rel_extent || rel_logits->stride[2] != 1 || rel_logits->stride[1] != rel_extent ||
         rel_logits->stride[0] != H * rel_extent))
        return nfail(bad, "noalloc: rel_logits must be a contiguous (T, H, rel_extent) bf16 or fp32 tensor");
    if (q->stride[2] != 1 || out->stride[2] != 1 || key_cache->stride[3] != 1)
        return nfail(bad, "noalloc: the head_dim axis must be contiguous");
    if (D != 64 && D != 128) return nfail(REL_ATTN_ERR_UNSUPPORTED, "noalloc: head_dim must be 64 or 128");
    if (BS <= 0 || BS % 16 != 0) return nfail(REL_ATTN_ERR_UNSUPPORTED, "noalloc: block_size must be a multiple of 16");
    if (T > INT32_MAX / 2 || NB > INT32_MAX) return nfail(REL_ATTN_ERR_UNSUPPORTED, "noalloc: sizes beyond 32-bit indexing");
    if (T > 0 && max_seqlen_q < 1) return nfail(bad, "noalloc: max_seqlen_q must be >= 1 when T > 0");
    if (T == 0 || B == 0) return REL_ATTN_OK;
    const int64_t oal = 16 / out_elem;
    if (!al16(q->data) || q->stride[0] % 8 || q->stride[1] % 8 || !al16(out->data) || out->stride[0] % oal ||
        out->stride[1] % oal || !al16(key_cache->data) || !al16(value_cache->data) || key_cache->stride[0] % 8 ||
        key_cache->stride[1] % 8 || key_cache->stride[2] % 8)
        return nfail(REL_ATTN_ERR_UNSUPPORTED, "noalloc: tensors need 16-byte aligned bases and strides");
    const int64_t G = H / Hk;
    const int64_t rows = (int64_t)max_seqlen_q * G;
    if (rows > 64)
        return nfail(REL_ATTN_ERR_UNSUPPORTED,
                     "noalloc: covers the decode path only (max_seqlen_q * num_heads / num_kv_heads <= 64)");

    int64_t splits = num_splits;
    const int64_t slice_cap = (MB * BS + 15) / 16;
    if (splits > slice_cap) splits = slice_cap < 1 ? 1 : slice_cap;
    if (splits > 1024) splits = 1024;
    const size_t need = splits > 1 ? (size_t)splits * T * H * (D + 1) * sizeof(float) : 0;
    if (need > kScratchBytes) {
        char buf[256];
        snprintf(buf, sizeof buf,
                 "noalloc: the split workspace needs %zu bytes, more than the %zu-byte static scratch; "
                 "lower num_splits or use rel_attn_paged_varlen",
                 need, kScratchBytes);
        return nfail(bad, buf);
    }

    ScratchInfo* sc = nullptr;
    rel_attn_status st = scratch_setup(&sc);
    if (st != REL_ATTN_OK) return st;
    if (sc->major != 10 || sc->minor != 3) return nfail(REL_ATTN_ERR_UNSUPPORTED, "noalloc: device is not sm_103");
    int* err = device_error_word();
    if (!err) return nfail(REL_ATTN_ERR_CUDA, "noalloc: device error word unavailable");

    AttnParams p{};
    p.q = q->data;
    p.q_st = q->stride[0];
    p.q_sh = q->stride[1];
    p.k_cache = key_cache->data;
    p.v_cache = value_cache->data;
    p.c_s0 = key_cache->stride[0];
    p.c_s1 = key_cache->stride[1];
    p.c_s2 = key_cache->stride[2];
    p.NB = (int32_t)NB;
    p.block_table = static_cast<const int32_t*>(block_table->data);
    p.bt_stride = block_table->stride[0];
    p.max_blocks = (int32_t)MB;
    p.cache_seqlens = static_cast<const int32_t*>(cache_seqlens->data);
    p.cu_seqlens_q = static_cast<const int32_t*>(cu_seqlens_q->data);
    p.rel = rel_extent > 0 ? rel_logits->data : nullptr;
    p.bias_f32 = rel_extent > 0 && rel_logits->dtype == REL_ATTN_F32 ? 1 : 0;
    p.R = rel_extent;
    p.out = out->data;
    p.o_st = out->stride[0];
    p.o_sh = out->stride[1];
    p.out_f32 = out->dtype == REL_ATTN_F32 ? 1 : 0;
    p.B = (int32_t)B;
    p.T = (int32_t)T;
    p.H = (int32_t)H;
    p.Hk = (int32_t)Hk;
    p.G = (int32_t)G;
    p.BS = (int32_t)BS;
    p.D = (int32_t)D;
    p.max_rows = (int32_t)rows;
    p.max_seqlen_q = max_seqlen_q;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.causal = causal ? 1 : 0;
    p.wl = window_left;
    p.wr = window_right;
    p.timeout_ns = 2000ull * 1000000ull;
    p.err = err;
    p.num_splits = (int32_t)splits;
    if (splits > 1) {
        p.ws_o = static_cast<float*>(sc->ptr);
        p.ws_lse = p.ws_o + (size_t)splits * T * H * D;
    }
    const LaunchShape shape = decode_shape(p, sc->sms);
    p.nstage = shape.nstage;
    p.nprod = shape.nprod;
    cudaError_t e = launch_decode(p, shape, stream);
    if (e == cudaSuccess && splits > 1) e = launch_combine(p, stream);
    if (e != cudaSuccess) {
        char buf[256];
        snprintf(buf, sizeof buf, "noalloc: launch failed: %s", cudaGetErrorString(e));
        return nfail(REL_ATTN_ERR_CUDA, buf);
    }
    return REL_ATTN_OK;
}
