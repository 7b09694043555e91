// C ABI of the library: argument validation, TMA descriptors, kernel choice,
// stream-ordered split workspace, launch.  Declared in include/rel_attn.h and
// include/rel_attn_profile.h.
//
// The interface follows inkling_fa4_rel_attention and inkling_fa4_num_splits
// in the vLLM API docs for vllm.models.inkling.nvidia.ops.fa4_rel_attention.

#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "kernels.h"
#include "rel_attn.h"
#include "rel_attn_profile.h"

namespace relattn {

__device__ int g_device_error = 0;
__device__ int g_check_error = 0;

namespace {

thread_local std::string t_last_error;
thread_local rel_attn_launch_info t_launch = {};
thread_local cudaEvent_t t_ev_begin = nullptr;
thread_local cudaEvent_t t_ev_end = nullptr;

rel_attn_status fail(rel_attn_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
rel_attn_status fail(rel_attn_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

struct DeviceInfo {
    bool ready = false;
    int ordinal = 0;
    int major = 0, minor = 0, sms = 0;
    int* err = nullptr;
    int* check_err = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

rel_attn_status device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(REL_ATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(REL_ATTN_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) return fail(REL_ATTN_ERR_CUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
        d.ordinal = dev;
        d.major = prop.major;
        d.minor = prop.minor;
        d.sms = prop.multiProcessorCount;
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_error);
        if (e != cudaSuccess) return fail(REL_ATTN_ERR_CUDA, "error word: %s", cudaGetErrorString(e));
        d.err = static_cast<int*>(p);
        e = cudaGetSymbolAddress(&p, g_check_error);
        if (e != cudaSuccess) return fail(REL_ATTN_ERR_CUDA, "check word: %s", cudaGetErrorString(e));
        d.check_err = static_cast<int*>(p);
        d.ready = true;
    }
    *out = &d;
    return REL_ATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// rel_logits (T, H, R) as a 3-D TMA tensor, innermost first: (R, H, T), box
// (prefill_bias_window() distances, G heads, ts tokens), no swizzle; needs
// R % 8 == 0.
rel_attn_status make_rel_map(const rel_attn_tensor* t, int G, int ts, CUtensorMap* map) {
    auto enc = encode_fn();
    if (!enc) return fail(REL_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {(cuuint64_t)t->shape[2], (cuuint64_t)t->shape[1], (cuuint64_t)t->shape[0]};
    cuuint64_t strides[2] = {(cuuint64_t)t->stride[1] * 2, (cuuint64_t)t->stride[0] * 2};
    cuuint32_t box[3] = {(cuuint32_t)prefill_bias_window(), (cuuint32_t)G, (cuuint32_t)ts};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, t->data, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(REL_ATTN_ERR_UNSUPPORTED, "rel_logits: TMA descriptor rejected (CUresult %d)", (int)r);
    return REL_ATTN_OK;
}

// Paged cache (NB, BS, Hk, D) as a 5-D TMA view whose box is one 16-key page
// (or half of one) of one kv head with `dbox` 64-dim blocks, 128-byte swizzle.
// A box lands as [8-key half][64-dim block][8 keys][64 dims]: the halves, the
// blocks and the keys of a half are separate view dimensions (keys at the slot
// stride, blocks 128 bytes apart).  When pages are contiguous (block stride ==
// BS * slot stride) the half index runs across blocks, (64, 8, D / 64, NB * BS
// / 8, Hk) with a (64, 8, dbox, 2, 1) box: one box per page.  Otherwise (64,
// BS, D / 64, Hk, NB) with a (64, 8, dbox, 1, 1) box: one box per half.
rel_attn_status make_page_map(const rel_attn_tensor* t, int dbox, bool merged, CUtensorMap* map,
                              const char* name) {
    auto enc = encode_fn();
    if (!enc) return fail(REL_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t NB = (cuuint64_t)t->shape[0], BS = (cuuint64_t)t->shape[1], Hk = (cuuint64_t)t->shape[2],
                     D = (cuuint64_t)t->shape[3];
    const cuuint64_t s0 = (cuuint64_t)t->stride[0] * 2, s1 = (cuuint64_t)t->stride[1] * 2,
                     s2 = (cuuint64_t)t->stride[2] * 2;
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5];
    if (merged) {
        const cuuint64_t d[5] = {64, 8, D / 64, NB * BS / 8, Hk};
        const cuuint64_t st[4] = {s1, 128, 8 * s1, s2};
        const cuuint32_t bx[5] = {64, 8, (cuuint32_t)dbox, 2, 1};
        std::memcpy(dims, d, sizeof d);
        std::memcpy(strides, st, sizeof st);
        std::memcpy(box, bx, sizeof bx);
    } else {
        const cuuint64_t d[5] = {64, BS, D / 64, Hk, NB};
        const cuuint64_t st[4] = {s1, 128, s2, s0};
        const cuuint32_t bx[5] = {64, 8, (cuuint32_t)dbox, 1, 1};
        std::memcpy(dims, d, sizeof d);
        std::memcpy(strides, st, sizeof st);
        std::memcpy(box, bx, sizeof bx);
    }
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, t->data, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(REL_ATTN_ERR_UNSUPPORTED, "%s: TMA descriptor rejected (CUresult %d)", name, (int)r);
    return REL_ATTN_OK;
}

// q (T, H, D) as a 3-D TMA tensor, innermost first: (D, H, T), box (64 dims,
// G heads, 128 / G tokens) = one 64-dim block of a GQA-packed query tile,
// 128-byte swizzle.
rel_attn_status make_q_map(const rel_attn_tensor* t, int G, CUtensorMap* map) {
    auto enc = encode_fn();
    if (!enc) return fail(REL_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {(cuuint64_t)t->shape[2], (cuuint64_t)t->shape[1], (cuuint64_t)t->shape[0]};
    cuuint64_t strides[2] = {(cuuint64_t)t->stride[1] * 2, (cuuint64_t)t->stride[0] * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, t->data, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(REL_ATTN_ERR_UNSUPPORTED, "q: TMA descriptor rejected (CUresult %d)", (int)r);
    return REL_ATTN_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

rel_attn_status check_tensor(const rel_attn_tensor* t, const char* name, int dtype, int ndim) {
    if (!t) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "%s: descriptor is NULL", name);
    if (t->dtype != dtype) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "%s: dtype %d, expected %d", name, t->dtype, dtype);
    if (t->ndim != ndim) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "%s: rank %d, expected %d", name, t->ndim, ndim);
    int64_t n = 1;
    for (int i = 0; i < ndim; ++i) {
        if (t->shape[i] < 0) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "%s: negative extent", name);
        n *= t->shape[i];
    }
    if (n > 0 && !t->data) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "%s: NULL data with %lld elements", name, (long long)n);
    return REL_ATTN_OK;
}

int64_t span_bytes(const rel_attn_tensor* t, int elem) {
    int64_t last = 0;
    for (int i = 0; i < t->ndim; ++i) {
        if (t->shape[i] == 0) return 0;
        last += (t->shape[i] - 1) * t->stride[i];
    }
    return (last + 1) * elem;
}

bool overlaps(const rel_attn_tensor* a, int ea, const rel_attn_tensor* b, int eb) {
    if (!a || !b || !a->data || !b->data) return false;
    const int64_t na = span_bytes(a, ea), nb = span_bytes(b, eb);
    if (na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a->data), b0 = reinterpret_cast<uintptr_t>(b->data);
    return a0 < b0 + (uintptr_t)nb && b0 < a0 + (uintptr_t)na;
}

// Every tensor the kernels touch must be device memory of the current device:
// the tensor maps and the kernels' loads address it directly, so memory of
// another GPU or of the host is rejected before anything is encoded or
// launched.  `tma` tensors (read through tensor maps) must be plain device
// allocations; the others may also be managed memory.
rel_attn_status check_resident(const rel_attn_tensor* t, const char* name, int dev, bool tma) {
    if (!t || !t->data) return REL_ATTN_OK;
    cudaPointerAttributes a{};
    const cudaError_t e = cudaPointerGetAttributes(&a, t->data);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(REL_ATTN_ERR_UNSUPPORTED, "%s: not a CUDA allocation (%s)", name, cudaGetErrorString(e));
    }
    const bool on_dev = a.type == cudaMemoryTypeDevice && a.device == dev;
    if (!(on_dev || (!tma && a.type == cudaMemoryTypeManaged)))
        return fail(REL_ATTN_ERR_UNSUPPORTED, "%s is not device memory of the current device %d (memory type %d, device %d)",
                    name, dev, (int)a.type, a.device);
    return REL_ATTN_OK;
}

uint64_t wait_timeout_ns() {
    static uint64_t ns = [] {
        const char* s = std::getenv("REL_ATTN_WAIT_TIMEOUT_MS");
        long long ms = s ? std::atoll(s) : 0;
        if (ms <= 0) ms = 2000;
        return (uint64_t)ms * 1000000ull;
    }();
    return ns;
}

bool check_enabled() {
    const char* s = std::getenv("REL_ATTN_CHECK");
    return s && s[0] == '1';
}

// REL_ATTN_PREFILL_PAIR=1 sends head_dim-128 prefill calls with TMA-staged
// or no bias to the CTA-pair kernel instead of the one-CTA kernel (both
// compute the same attention; the one-CTA kernel is faster there).
bool prefill_pair_requested() {
    const char* s = std::getenv("REL_ATTN_PREFILL_PAIR");
    return s && s[0] == '1';
}

// Device-side precondition check (REL_ATTN_CHECK=1): one thread per request.
__global__ void check_kernel(const int32_t* cu, const int32_t* seqk, const int32_t* table, int64_t bt_stride, int B,
                             int T, int MB, int BS, int NB, int max_seqlen_q, int* err) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int code = 0;
    const int sq = cu[b + 1] - cu[b];
    if (b == 0 && cu[0] != 0) code = 1;
    if (b == B - 1 && cu[B] != T) code = 2;
    if (sq < 0) code = 3;
    if (sq > max_seqlen_q) code = 4;
    const int sk = seqk[b];
    if (sk < 0 || (long long)sk > (long long)MB * BS) code = 5;
    if (!code) {
        const int nblk = (sk + BS - 1) / BS;
        for (int n = 0; n < nblk; ++n) {
            const int blk = table[(size_t)b * bt_stride + n];
            if (blk < 0 || blk >= NB) {
                code = 6;
                break;
            }
        }
    }
    if (code) atomicCAS(err, 0, code);
}


// REL_ATTN_CHECK=1: run check_kernel on `stream`, wait for it, and turn a
// recorded violation into REL_ATTN_ERR_DEVICE_CHECK (no kernel runs after it).
rel_attn_status run_device_check(DeviceInfo* dev, cudaStream_t stream, const rel_attn_tensor* cu_seqlens_q,
                                 const rel_attn_tensor* cache_seqlens, const rel_attn_tensor* block_table,
                                 int64_t B, int64_t T, int64_t MB, int64_t BS, int64_t NB, int max_seqlen_q) {
    cudaError_t e = cudaMemsetAsync(dev->check_err, 0, sizeof(int), stream);
    if (e == cudaSuccess) {
        check_kernel<<<(unsigned)((B + 127) / 128), 128, 0, stream>>>(
            static_cast<const int32_t*>(cu_seqlens_q->data), static_cast<const int32_t*>(cache_seqlens->data),
            static_cast<const int32_t*>(block_table->data), block_table->stride[0], (int)B, (int)T, (int)MB,
            (int)BS, (int)NB, max_seqlen_q, dev->check_err);
        e = cudaGetLastError();
    }
    int code = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&code, dev->check_err, sizeof code, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(REL_ATTN_ERR_CUDA, "check kernel: %s", cudaGetErrorString(e));
    if (code)
        return fail(REL_ATTN_ERR_DEVICE_CHECK, "device-side precondition violated (code %d: %s)", code,
                    code == 1 ? "cu_seqlens_q[0] != 0" : code == 2 ? "cu_seqlens_q[B] != T"
                    : code == 3 ? "cu_seqlens_q decreasing" : code == 4 ? "a query length exceeds max_seqlen_q"
                    : code == 5 ? "cache_seqlens outside [0, MB*BS]" : "block id outside [0, NB)");
    return REL_ATTN_OK;
}
}  // namespace
}  // namespace relattn

using namespace relattn;

extern "C" const char* rel_attn_last_error(void) { return t_last_error.c_str(); }

extern "C" int32_t rel_attn_bucket_max_seqlen_q(int32_t max_seqlen_q) {
    if (max_seqlen_q < 0 || max_seqlen_q > (1 << 30)) {
        fail(REL_ATTN_ERR_INVALID_ARGUMENT, "rel_attn_bucket_max_seqlen_q: %d outside [0, 2^30]", max_seqlen_q);
        return -REL_ATTN_ERR_INVALID_ARGUMENT;
    }
    int32_t b = 1;
    while (b < max_seqlen_q) b <<= 1;
    return b;
}

extern "C" int32_t rel_attn_num_splits(int32_t is_local, int32_t batch_size, int32_t max_query_len,
                                       int32_t num_heads, int32_t num_kv_heads, int32_t max_kv_len) {
    if (batch_size < 1 || max_query_len < 1 || num_heads < 1 || num_kv_heads < 1 || num_heads % num_kv_heads != 0 ||
        max_kv_len < 0) {
        fail(REL_ATTN_ERR_INVALID_ARGUMENT, "rel_attn_num_splits: invalid sizes");
        return -REL_ATTN_ERR_INVALID_ARGUMENT;
    }
    if (is_local) return 1;
    const int64_t rows = (int64_t)max_query_len * (num_heads / num_kv_heads);
    const int64_t tiles = (rows + 255) / 256;
    const int64_t base = (int64_t)batch_size * num_kv_heads * tiles;
    const bool one_tile_b1 = tiles == 1 && batch_size == 1;
    const int64_t target = one_tile_b1 ? 256 : (tiles == 1 ? 128 : 64);
    int64_t cap = 128;
    if (one_tile_b1) {
        if (num_kv_heads == 8)
            cap = 16;
        else if (num_kv_heads == 4 || max_kv_len <= 8192)
            cap = 32;
        else if (max_kv_len <= 65536)
            cap = 64;
        else
            cap = 128;
    }
    const int64_t kv_blocks = ((int64_t)max_kv_len + 127) / 128;
    int64_t r = target / base;
    if (cap < r) r = cap;
    if (kv_blocks < r) r = kv_blocks;
    return (int32_t)(r < 1 ? 1 : r);
}

extern "C" rel_attn_status rel_attn_last_launch(rel_attn_launch_info* info) {
    if (!info) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "info is NULL");
    *info = t_launch;
    return REL_ATTN_OK;
}

extern "C" rel_attn_status rel_attn_set_kernel_events(void* begin, void* end) {
    if ((begin == nullptr) != (end == nullptr))
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "pass both events or neither");
    t_ev_begin = static_cast<cudaEvent_t>(begin);
    t_ev_end = static_cast<cudaEvent_t>(end);
    return REL_ATTN_OK;
}

extern "C" rel_attn_status rel_attn_device_error(int32_t* code) {
    if (!code) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "code is NULL");
    DeviceInfo* dev = nullptr;
    rel_attn_status st = device_info(&dev);
    if (st != REL_ATTN_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(REL_ATTN_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
    int v = 0;
    e = cudaMemcpy(&v, dev->err, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(dev->err, 0, sizeof v);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(REL_ATTN_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(e));
    *code = v;
    return REL_ATTN_OK;
}

namespace relattn {

// Body of rel_attn_paged_varlen, rel_attn_paged_varlen_lse (lse may be NULL)
// and rel_attn_paged_varlen_noalloc (fixed_ws non-NULL: the split workspace
// is that buffer, and a call needing more is rejected before any device work).
rel_attn_status paged_varlen(
    const rel_attn_tensor* q, const rel_attn_tensor* key_cache, const rel_attn_tensor* value_cache,
    const rel_attn_tensor* block_table, const rel_attn_tensor* cache_seqlens, const rel_attn_tensor* cu_seqlens_q,
    int32_t max_seqlen_q, float softmax_scale, int32_t causal, int32_t window_left, int32_t window_right,
    int32_t rel_extent, const rel_attn_tensor* rel_logits, int32_t num_splits, rel_attn_tensor* out,
    rel_attn_tensor* lse, rel_attn_stream stream_, const FixedWorkspace* fixed_ws) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    t_launch = rel_attn_launch_info{};
    rel_attn_status st;
    if ((st = check_tensor(q, "q", REL_ATTN_BF16, 3))) return st;
    if ((st = check_tensor(key_cache, "key_cache", REL_ATTN_BF16, 4))) return st;
    if ((st = check_tensor(value_cache, "value_cache", REL_ATTN_BF16, 4))) return st;
    if ((st = check_tensor(block_table, "block_table", REL_ATTN_I32, 2))) return st;
    if ((st = check_tensor(cache_seqlens, "cache_seqlens", REL_ATTN_I32, 1))) return st;
    if ((st = check_tensor(cu_seqlens_q, "cu_seqlens_q", REL_ATTN_I32, 1))) return st;
    if (!out) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "out: descriptor is NULL");
    if ((st = check_tensor(out, "out", out->dtype == REL_ATTN_F32 ? REL_ATTN_F32 : REL_ATTN_BF16, 3))) return st;
    const int out_elem = out->dtype == REL_ATTN_F32 ? 4 : 2;

    const int64_t T = q->shape[0], H = q->shape[1], D = q->shape[2];
    const int64_t NB = key_cache->shape[0], BS = key_cache->shape[1], Hk = key_cache->shape[2];
    const int64_t B = block_table->shape[0], MB = block_table->shape[1];
    for (int i = 0; i < 4; ++i)
        if (value_cache->shape[i] != key_cache->shape[i])
            return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "value_cache shape differs from key_cache");
    for (int i = 0; i < 4; ++i)
        if (value_cache->stride[i] != key_cache->stride[i])
            return fail(REL_ATTN_ERR_UNSUPPORTED, "value_cache strides must equal key_cache strides");
    if (key_cache->shape[3] != D) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "cache head_dim %lld != q head_dim %lld",
                                              (long long)key_cache->shape[3], (long long)D);
    if (out->shape[0] != T || out->shape[1] != H || out->shape[2] != D)
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "out shape must equal q shape");
    if (cache_seqlens->shape[0] != B) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "cache_seqlens must have B entries");
    if (cu_seqlens_q->shape[0] != B + 1) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "cu_seqlens_q must have B+1 entries");
    if (cache_seqlens->stride[0] != 1 || cu_seqlens_q->stride[0] != 1)
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "cache_seqlens and cu_seqlens_q must be contiguous");
    if (MB > 0 && block_table->stride[1] != 1)
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "block_table rows must be contiguous");
    if (B > 0 && block_table->stride[0] < MB)
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "block_table row stride smaller than its width");
    if (H <= 0 || Hk <= 0 || H % Hk != 0)
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "num_heads %lld must be a positive multiple of num_kv_heads %lld",
                    (long long)H, (long long)Hk);
    if (num_splits < 1) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "num_splits must be >= 1 (got %d)", num_splits);
    if (rel_extent < 0) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "rel_extent must be >= 0 (got %d)", rel_extent);
    if (max_seqlen_q < 0) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "max_seqlen_q must be >= 0");
    const bool rel_f32 = rel_extent > 0 && rel_logits && rel_logits->dtype == REL_ATTN_F32;
    const int rel_elem = rel_f32 ? 4 : 2;
    if (rel_extent > 0) {
        if ((st = check_tensor(rel_logits, "rel_logits", rel_f32 ? REL_ATTN_F32 : REL_ATTN_BF16, 3))) return st;
        if (rel_logits->shape[0] != T || rel_logits->shape[1] != H || rel_logits->shape[2] != rel_extent)
            return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "rel_logits must be (T, H, rel_extent)");
        if (rel_logits->stride[2] != 1 || rel_logits->stride[1] != rel_extent ||
            rel_logits->stride[0] != H * rel_extent)
            return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "rel_logits must be contiguous");
    }
    if (q->stride[2] != 1 || out->stride[2] != 1 || key_cache->stride[3] != 1 || value_cache->stride[3] != 1)
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "the head_dim axis must be contiguous");
    if (D != 64 && D != 128 && D != 256)
        return fail(REL_ATTN_ERR_UNSUPPORTED, "head_dim %lld unsupported (64, 128 or 256)", (long long)D);
    if (BS <= 0 || BS % 16 != 0)
        return fail(REL_ATTN_ERR_UNSUPPORTED, "block_size %lld unsupported (a multiple of 16)", (long long)BS);
    if (H / Hk > 128) return fail(REL_ATTN_ERR_UNSUPPORTED, "more than 128 query heads per kv head");
    if (T > INT32_MAX / 2 || NB > INT32_MAX || H * T > ((int64_t)1 << 40))
        return fail(REL_ATTN_ERR_UNSUPPORTED, "sizes beyond 32-bit indexing");
    if (T > 0 && max_seqlen_q < 1) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "max_seqlen_q must be >= 1 when T > 0");
    if (overlaps(out, out_elem, q, 2) || overlaps(out, out_elem, key_cache, 2) ||
        overlaps(out, out_elem, value_cache, 2) || (rel_extent > 0 && overlaps(out, out_elem, rel_logits, rel_elem)))
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "out aliases an input");
    if (lse) {
        if ((st = check_tensor(lse, "softmax_lse", REL_ATTN_F32, 2))) return st;
        if (lse->shape[0] != T || lse->shape[1] != H)
            return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "softmax_lse must be (T, H)");
        if (lse->stride[0] < 0 || lse->stride[1] < 0)
            return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "softmax_lse strides must be >= 0");
        if (overlaps(lse, 4, q, 2) || overlaps(lse, 4, key_cache, 2) || overlaps(lse, 4, value_cache, 2) ||
            overlaps(lse, 4, block_table, 4) || overlaps(lse, 4, cache_seqlens, 4) ||
            overlaps(lse, 4, cu_seqlens_q, 4) || overlaps(lse, 4, out, out_elem) ||
            (rel_extent > 0 && overlaps(lse, 4, rel_logits, rel_elem)))
            return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "softmax_lse aliases an input or out");
        if (!aligned(lse->data, 4)) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "softmax_lse is not 4-byte aligned");
    }
    if (T == 0 || B == 0) {
        t_launch.kernel = REL_ATTN_KERNEL_NONE;
        return REL_ATTN_OK;
    }
    // Alignment rules of the vector loads and TMA.
    const int64_t oal = 16 / out_elem;
    if (!aligned(q->data, 16) || q->stride[0] % 8 || q->stride[1] % 8 || !aligned(out->data, 16) ||
        out->stride[0] % oal || out->stride[1] % oal)
        return fail(REL_ATTN_ERR_UNSUPPORTED, "q/out need 16-byte aligned bases and strides");
    for (const rel_attn_tensor* c : {key_cache, value_cache})
        if (!aligned(c->data, 16) || c->stride[0] % 8 || c->stride[1] % 8 || c->stride[2] % 8)
            return fail(REL_ATTN_ERR_UNSUPPORTED, "caches need 16-byte aligned bases and strides");

    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev))) return st;
    if (dev->major != 10 || dev->minor != 3)
        return fail(REL_ATTN_ERR_UNSUPPORTED, "built for sm_103a; device is sm_%d%d", dev->major, dev->minor);
    if ((st = check_resident(q, "q", dev->ordinal, false)) ||
        (st = check_resident(key_cache, "key_cache", dev->ordinal, true)) ||
        (st = check_resident(value_cache, "value_cache", dev->ordinal, true)) ||
        (st = check_resident(block_table, "block_table", dev->ordinal, false)) ||
        (st = check_resident(cache_seqlens, "cache_seqlens", dev->ordinal, false)) ||
        (st = check_resident(cu_seqlens_q, "cu_seqlens_q", dev->ordinal, false)) ||
        (rel_extent > 0 && (st = check_resident(rel_logits, "rel_logits", dev->ordinal, true))) ||
        (st = check_resident(out, "out", dev->ordinal, false)) ||
        (lse && (st = check_resident(lse, "softmax_lse", dev->ordinal, false))))
        return st;

    const int64_t G = H / Hk;
    const int64_t rows = (int64_t)max_seqlen_q * G;
    const bool prefill = rows > 64;  // decode kernel up to 64 packed rows, tcgen05 tiles above

    // Splits: a cap, clamped to the 16-key slices a request can have.
    int64_t splits = num_splits;
    const int64_t slice_cap = (MB * BS + 15) / 16;
    if (splits > slice_cap) splits = slice_cap < 1 ? 1 : slice_cap;
    if (splits > 1024) splits = 1024;
    const size_t ws_bytes = splits > 1 ? (size_t)splits * T * H * (D + 1) * sizeof(float) : 0;
    if (fixed_ws && ws_bytes > fixed_ws->bytes)
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT,
                    "the split workspace needs %zu bytes, more than the %zu-byte static scratch; lower num_splits "
                    "or call rel_attn_paged_varlen",
                    ws_bytes, fixed_ws->bytes);
    // The fixed workspace's device address on this device (looked up once
    // per device, on the first call that gets this far).
    void* fixed_base = nullptr;
    if (fixed_ws && (st = fixed_ws->address(&fixed_base))) return st;

    if (check_enabled() && (st = run_device_check(dev, stream, cu_seqlens_q, cache_seqlens, block_table, B, T, MB,
                                                   BS, NB, max_seqlen_q)))
        return st;

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
    p.R = rel_extent;
    p.bias_f32 = rel_f32 ? 1 : 0;
    // bf16 bias windows are staged by TMA; fp32 rel_logits are read per element.
    p.vec_bias = (rel_extent > 0 && !rel_f32 && rel_extent % 8 == 0 && aligned(rel_logits->data, 16)) ? 1 : 0;
    p.out = out->data;
    p.o_st = out->stride[0];
    p.o_sh = out->stride[1];
    p.out_f32 = out->dtype == REL_ATTN_F32 ? 1 : 0;
    if (lse) {
        p.lse = static_cast<float*>(lse->data);
        p.lse_st = lse->stride[0];
        p.lse_sh = lse->stride[1];
    }
    p.B = (int32_t)B;
    p.T = (int32_t)T;
    p.H = (int32_t)H;
    p.Hk = (int32_t)Hk;
    p.G = (int32_t)G;
    p.BS = (int32_t)BS;
    p.D = (int32_t)D;
    p.max_rows = (int32_t)(rows > INT32_MAX ? INT32_MAX : rows);
    p.max_seqlen_q = max_seqlen_q;
    p.scale = softmax_scale;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.causal = causal ? 1 : 0;
    p.wl = window_left;
    p.wr = window_right;
    p.timeout_ns = wait_timeout_ns();
    p.err = dev->err;

    CUtensorMap maps[4];
    std::memset(maps, 0, sizeof maps);
    // The CTA-pair kernel (2-SM MMAs): head_dim 256 always (only it fits
    // that head size), head_dim 128 with TMA-staged or no bias on request.
    const bool pair =
        prefill && (D == 256 || (D == 128 && (rel_extent == 0 || p.vec_bias) && prefill_pair_requested()));
    if (prefill) {
        // Page views of the caches: one TMA box per 16-key page (two when the
        // pages are not contiguous).  K and V share strides, checked above.
        // The CTA-pair kernel stages half of every V tile's dims per CTA.
        p.kv_merged = p.c_s0 == (int64_t)BS * p.c_s1 ? 1 : 0;
        const int dbox = (int)(D / 64);
        if ((st = make_page_map(key_cache, dbox, p.kv_merged != 0, &maps[0], "key_cache"))) return st;
        if ((st = make_page_map(value_cache, pair ? dbox / 2 : dbox, p.kv_merged != 0, &maps[1], "value_cache")))
            return st;
        // Tokens per rel_logits box: the largest divisor of the tile's 128 / G
        // tokens that is at most 8 (a box then never crosses the tile).
        const int tpt = (int)(128 / G);
        int ts = 1;
        for (int d = 1; d <= 8 && d <= tpt; ++d)
            if (tpt % d == 0) ts = d;
        p.bias_ts = ts;
        if (p.vec_bias && (st = make_rel_map(rel_logits, (int)G, ts, &maps[2]))) return st;
        if (pair && (st = make_q_map(q, (int)G, &maps[3]))) return st;
    }

    p.num_splits = (int32_t)splits;

    // The split workspace: the caller's fixed buffer, else a stream-ordered
    // allocation freed after the combine.
    void* ws = nullptr;
    if (splits > 1) {
        void* base = nullptr;
        if (fixed_ws) {
            base = fixed_base;
        } else {
            cudaError_t e = cudaMallocAsync(&ws, ws_bytes, stream);
            if (e != cudaSuccess) {
                cudaGetLastError();
                return fail(e == cudaErrorMemoryAllocation ? REL_ATTN_ERR_OUT_OF_MEMORY : REL_ATTN_ERR_CUDA,
                            "split workspace of %zu bytes: %s", ws_bytes, cudaGetErrorString(e));
            }
            base = ws;
        }
        p.ws_o = static_cast<float*>(base);
        p.ws_lse = p.ws_o + (size_t)splits * T * H * D;
    }

    LaunchShape shape = pair ? prefill_pair_shape(p) : prefill ? prefill_shape(p) : decode_shape(p, dev->sms);
    p.nstage = shape.nstage;
    p.nprod = shape.nprod;
    if (t_ev_begin) cudaEventRecord(t_ev_begin, stream);
    cudaError_t e = pair      ? launch_prefill_pair(p, maps, shape, stream)
                    : prefill ? launch_prefill(p, maps, shape, stream)
                              : launch_decode(p, shape, stream);
    if (t_ev_end) cudaEventRecord(t_ev_end, stream);
    int launches = 1;
    if (e == cudaSuccess && splits > 1) {
        e = launch_combine(p, stream);
        ++launches;
    }
    if (ws) {
        cudaError_t e2 = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess) e = e2;
    }
    t_launch.kernel = pair ? REL_ATTN_KERNEL_PREFILL_PAIR : prefill ? REL_ATTN_KERNEL_PREFILL : REL_ATTN_KERNEL_DECODE;
    t_launch.num_splits = (int32_t)splits;
    t_launch.grid[0] = (int32_t)shape.grid.x;
    t_launch.grid[1] = (int32_t)shape.grid.y;
    t_launch.grid[2] = (int32_t)shape.grid.z;
    t_launch.block = shape.block;
    t_launch.smem_bytes = shape.smem;
    t_launch.launches = launches;
    t_launch.workspace_bytes = (int64_t)ws_bytes;
    if (e != cudaSuccess) return fail(REL_ATTN_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    return REL_ATTN_OK;
}

}  // namespace relattn

extern "C" rel_attn_status rel_attn_paged_varlen(
    const rel_attn_tensor* q, const rel_attn_tensor* key_cache, const rel_attn_tensor* value_cache,
    const rel_attn_tensor* block_table, const rel_attn_tensor* cache_seqlens, const rel_attn_tensor* cu_seqlens_q,
    int32_t max_seqlen_q, float softmax_scale, int32_t causal, int32_t window_left, int32_t window_right,
    int32_t rel_extent, const rel_attn_tensor* rel_logits, int32_t num_splits, rel_attn_tensor* out,
    rel_attn_stream stream) {
    return paged_varlen(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q, max_seqlen_q,
                        softmax_scale, causal, window_left, window_right, rel_extent, rel_logits, num_splits, out,
                        nullptr, stream, nullptr);
}

extern "C" rel_attn_status rel_attn_paged_varlen_lse(
    const rel_attn_tensor* q, const rel_attn_tensor* key_cache, const rel_attn_tensor* value_cache,
    const rel_attn_tensor* block_table, const rel_attn_tensor* cache_seqlens, const rel_attn_tensor* cu_seqlens_q,
    int32_t max_seqlen_q, float softmax_scale, int32_t causal, int32_t window_left, int32_t window_right,
    int32_t rel_extent, const rel_attn_tensor* rel_logits, int32_t num_splits, rel_attn_tensor* out,
    rel_attn_tensor* softmax_lse, rel_attn_stream stream) {
    return paged_varlen(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q, max_seqlen_q,
                        softmax_scale, causal, window_left, window_right, rel_extent, rel_logits, num_splits, out,
                        softmax_lse, stream, nullptr);
}

namespace relattn {

// Accessors for entry points defined in other files.
void set_last_error_message(const char* msg) { t_last_error = msg; }

int* device_error_word() {
    DeviceInfo* dev = nullptr;
    return device_info(&dev) == REL_ATTN_OK ? dev->err : nullptr;
}

}  // namespace relattn

extern "C" rel_attn_status rel_attn_cache_append(
    const rel_attn_tensor* key, const rel_attn_tensor* value, rel_attn_tensor* key_cache,
    rel_attn_tensor* value_cache, const rel_attn_tensor* block_table, const rel_attn_tensor* cache_seqlens,
    const rel_attn_tensor* cu_seqlens_q, rel_attn_stream stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    t_launch = rel_attn_launch_info{};
    rel_attn_status st;
    if ((st = check_tensor(key, "key", REL_ATTN_BF16, 3))) return st;
    if ((st = check_tensor(value, "value", REL_ATTN_BF16, 3))) return st;
    if ((st = check_tensor(key_cache, "key_cache", REL_ATTN_BF16, 4))) return st;
    if ((st = check_tensor(value_cache, "value_cache", REL_ATTN_BF16, 4))) return st;
    if ((st = check_tensor(block_table, "block_table", REL_ATTN_I32, 2))) return st;
    if ((st = check_tensor(cache_seqlens, "cache_seqlens", REL_ATTN_I32, 1))) return st;
    if ((st = check_tensor(cu_seqlens_q, "cu_seqlens_q", REL_ATTN_I32, 1))) return st;
    const int64_t T = key->shape[0], Hk = key->shape[1], D = key->shape[2];
    const int64_t NB = key_cache->shape[0], BS = key_cache->shape[1];
    const int64_t B = block_table->shape[0], MB = block_table->shape[1];
    for (int i = 0; i < 3; ++i)
        if (value->shape[i] != key->shape[i]) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "value shape differs from key");
    for (int i = 0; i < 4; ++i) {
        if (value_cache->shape[i] != key_cache->shape[i])
            return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "value_cache shape differs from key_cache");
        if (value_cache->stride[i] != key_cache->stride[i])
            return fail(REL_ATTN_ERR_UNSUPPORTED, "value_cache strides must equal key_cache strides");
    }
    if (key_cache->shape[2] != Hk || key_cache->shape[3] != D)
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "key is (T, Hk, D) with the caches' Hk and D");
    if (cache_seqlens->shape[0] != B) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "cache_seqlens must have B entries");
    if (cu_seqlens_q->shape[0] != B + 1) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "cu_seqlens_q must have B+1 entries");
    if (cache_seqlens->stride[0] != 1 || cu_seqlens_q->stride[0] != 1)
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "cache_seqlens and cu_seqlens_q must be contiguous");
    if (MB > 0 && block_table->stride[1] != 1)
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "block_table rows must be contiguous");
    if (B > 0 && block_table->stride[0] < MB)
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "block_table row stride smaller than its width");
    if (key->stride[2] != 1 || value->stride[2] != 1 || key_cache->stride[3] != 1)
        return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "the head_dim axis must be contiguous");
    if (D <= 0 || D % 8 != 0 || D > 512) return fail(REL_ATTN_ERR_UNSUPPORTED, "head_dim must be a multiple of 8 up to 512");
    if (BS <= 0) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "block_size must be positive");
    if (T > INT32_MAX / 2 || NB > INT32_MAX || B > INT32_MAX / 2)
        return fail(REL_ATTN_ERR_UNSUPPORTED, "sizes beyond 32-bit indexing");
    for (const rel_attn_tensor* src : {key, value})
        for (const rel_attn_tensor* dst : {key_cache, value_cache})
            if (overlaps(src, 2, dst, 2)) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "key/value alias a cache");
    if (overlaps(key_cache, 2, value_cache, 2)) return fail(REL_ATTN_ERR_INVALID_ARGUMENT, "key_cache aliases value_cache");
    if (T == 0 || B == 0) {
        t_launch.kernel = REL_ATTN_KERNEL_NONE;
        return REL_ATTN_OK;
    }
    for (const rel_attn_tensor* c : {key, value})
        if (!aligned(c->data, 16) || c->stride[0] % 8 || c->stride[1] % 8)
            return fail(REL_ATTN_ERR_UNSUPPORTED, "key/value need 16-byte aligned bases and strides");
    for (const rel_attn_tensor* c : {key_cache, value_cache})
        if (!aligned(c->data, 16) || c->stride[0] % 8 || c->stride[1] % 8 || c->stride[2] % 8)
            return fail(REL_ATTN_ERR_UNSUPPORTED, "caches need 16-byte aligned bases and strides");

    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev))) return st;
    if (dev->major != 10 || dev->minor != 3)
        return fail(REL_ATTN_ERR_UNSUPPORTED, "built for sm_103a; device is sm_%d%d", dev->major, dev->minor);
    if ((st = check_resident(key, "key", dev->ordinal, false)) ||
        (st = check_resident(value, "value", dev->ordinal, false)) ||
        (st = check_resident(key_cache, "key_cache", dev->ordinal, false)) ||
        (st = check_resident(value_cache, "value_cache", dev->ordinal, false)) ||
        (st = check_resident(block_table, "block_table", dev->ordinal, false)) ||
        (st = check_resident(cache_seqlens, "cache_seqlens", dev->ordinal, false)) ||
        (st = check_resident(cu_seqlens_q, "cu_seqlens_q", dev->ordinal, false)))
        return st;
    if (check_enabled() && (st = run_device_check(dev, stream, cu_seqlens_q, cache_seqlens, block_table, B, T, MB,
                                                   BS, NB, (int)T)))
        return st;
    AppendParams p{};
    p.key = key->data;
    p.value = value->data;
    p.k_st = key->stride[0];
    p.k_sh = key->stride[1];
    p.v_st = value->stride[0];
    p.v_sh = value->stride[1];
    p.k_cache = key_cache->data;
    p.v_cache = value_cache->data;
    p.c_s0 = key_cache->stride[0];
    p.c_s1 = key_cache->stride[1];
    p.c_s2 = key_cache->stride[2];
    p.block_table = static_cast<const int32_t*>(block_table->data);
    p.bt_stride = block_table->stride[0];
    p.cache_seqlens = static_cast<const int32_t*>(cache_seqlens->data);
    p.cu_seqlens_q = static_cast<const int32_t*>(cu_seqlens_q->data);
    p.B = (int32_t)B;
    p.T = (int32_t)T;
    p.Hk = (int32_t)Hk;
    p.BS = (int32_t)BS;
    p.D = (int32_t)D;
    p.MB = (int32_t)MB;
    p.NB = (int32_t)NB;
    p.err = dev->err;
    if (t_ev_begin) cudaEventRecord(t_ev_begin, stream);
    cudaError_t e = launch_append(p, stream);
    if (t_ev_end) cudaEventRecord(t_ev_end, stream);
    t_launch.kernel = REL_ATTN_KERNEL_APPEND;
    t_launch.num_splits = 0;
    t_launch.grid[0] = (int32_t)((T + 7) / 8);
    t_launch.grid[1] = 1;
    t_launch.grid[2] = 1;
    t_launch.block = 256;
    t_launch.launches = 1;
    if (e != cudaSuccess) return fail(REL_ATTN_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    return REL_ATTN_OK;
}
