// Host-side launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "rel_attn.h"

namespace relattn {

// Everything a kernel needs besides the tensor maps.  Strides in elements.
struct AttnParams {
    const void* q;             // (T, H, D) bf16
    int64_t q_st, q_sh;        // token / head strides
    const void* k_cache;       // (NB, BS, Hk, D) bf16
    const void* v_cache;
    int64_t c_s0, c_s1, c_s2;  // cache block / slot / head strides (shared by K and V)
    int32_t NB;
    const int32_t* block_table;
    int64_t bt_stride;         // MB
    int32_t max_blocks;        // MB
    const int32_t* cache_seqlens;
    const int32_t* cu_seqlens_q;
    const void* rel;           // (T, H, R) bf16 (or fp32 when bias_f32) contiguous, or null when R == 0
    int32_t R;
    int32_t bias_f32;          // rel_logits are fp32
    void* out;                 // (T, H, D) bf16, or fp32 when out_f32
    int64_t o_st, o_sh;
    int32_t out_f32;
    float* lse;                // (T, H) fp32 natural-log sum-exp of each row's scores, or null
    int64_t lse_st, lse_sh;    // token / head strides of lse
    float* ws_o;               // (S, T, H, D) fp32 partials when num_splits > 1
    float* ws_lse;             // (S, T, H) fp32 log2-sum-exp partials
    int32_t B, T, H, Hk, G, BS, D;
    int32_t num_splits;
    int32_t max_rows;          // max_seqlen_q * G (decode: <= 64)
    int32_t max_seqlen_q;
    float scale;               // softmax_scale
    float scale_log2;          // softmax_scale * log2(e)
    int32_t bias_ts;           // prefill: tokens per rel_logits TMA box (divides 128 / G, <= 8)
    int32_t causal, wl, wr;
    int32_t nstage;
    int32_t nprod;             // decode: producer warps
    int32_t vec_bias;          // rel_logits rows 16-byte aligned (R % 8 == 0): staged by 16-byte copies
    int32_t kv_merged;         // prefill: the caches' pages are contiguous (c_s0 == BS * c_s1), so one
                               // 5-D TMA box holds a whole 16-key page
    uint64_t timeout_ns;
    int* err;                  // device error word (bounded-wait timeouts)
};

struct LaunchShape {
    dim3 grid;
    int block = 0;
    int smem = 0;
    int nstage = 0;
    int mt = 0, ksl = 0;  // decode: 16-row tiles and 16-key slices per CTA
    int nprod = 1;        // decode: producer warps
};

// Split-KV decode kernel for <= 64 GQA-packed rows per (request, kv head).
LaunchShape decode_shape(const AttnParams& p, int num_sms);
cudaError_t launch_decode(const AttnParams& p, const LaunchShape& shape, cudaStream_t stream);

// tcgen05 prefill kernel for 128-row GQA-packed query tiles.  maps[0] / maps[1]
// describe key_cache / value_cache as 5-D TMA views with 128-byte swizzle
// (make_page_map): (64, 8, D / 64, NB * BS / 8, Hk) with a (64, 8, D / 64, 2, 1)
// box when kv_merged, else (64, BS, D / 64, Hk, NB) with a (64, 8, D / 64, 1, 1)
// box; maps[2] describes rel_logits as a
// 3-D tensor (R, H, T) with a (prefill_bias_window(), G, bias_ts) box (only
// read when vec_bias).
LaunchShape prefill_shape(const AttnParams& p);
// rel_logits values per staged bias row (the inner box extent of maps[2]).
int prefill_bias_window();
cudaError_t launch_prefill(const AttnParams& p, const CUtensorMap* maps, const LaunchShape& shape,
                           cudaStream_t stream);

// 2-SM tcgen05 prefill kernel (CTA pairs, cta_group::2) for head_dim 256, and
// 128 on request, with rel_logits staged by TMA (vec_bias) or no bias:
// clusters of two CTAs holding two 128-row query tiles.  maps[0] as for
// launch_prefill; maps[1] the same page view of value_cache with a box of
// D / 128 dim blocks (each CTA stages half of the dims); maps[2] as for
// launch_prefill; maps[3] describes q as a 3-D TMA tensor (D, H, T) with a
// (64, G, 128 / G) box and 128-byte swizzle.
LaunchShape prefill_pair_shape(const AttnParams& p);
cudaError_t launch_prefill_pair(const AttnParams& p, const CUtensorMap* maps, const LaunchShape& shape,
                                cudaStream_t stream);

// Paged KV-cache append (key/value rows of the new tokens into the caches).
struct AppendParams {
    const void* key;           // (T, Hk, D) bf16
    const void* value;
    int64_t k_st, k_sh, v_st, v_sh;  // token / head strides
    void* k_cache;             // (NB, BS, Hk, D) bf16
    void* v_cache;
    int64_t c_s0, c_s1, c_s2;  // cache block / slot / head strides (shared by K and V)
    const int32_t* block_table;
    int64_t bt_stride;
    const int32_t* cache_seqlens;
    const int32_t* cu_seqlens_q;
    int32_t B, T, Hk, BS, D;
    int32_t MB;                // block_table width
    int32_t NB;                // blocks in each cache
    int* err;                  // device error word: a token whose slot is outside the table or cache
};
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);

// LSE-weighted merge of split partials into out (and lse when requested).
cudaError_t launch_combine(const AttnParams& p, cudaStream_t stream);

// A fixed device buffer of `bytes` bytes that serves as the split workspace
// instead of a stream-ordered allocation (the allocation-free entry point).
// `address` returns its device address on the current device; the body calls
// it once host validation has passed, with the call's device current.
struct FixedWorkspace {
    rel_attn_status (*address)(void** ptr);
    size_t bytes;
};

// The attention entry points' common body (api.cu): validation, kernel
// choice, workspace, launches.  lse may be NULL; fixed_ws NULL allocates the
// split workspace on `stream`.
rel_attn_status paged_varlen(const rel_attn_tensor* q, const rel_attn_tensor* key_cache,
                             const rel_attn_tensor* value_cache, const rel_attn_tensor* block_table,
                             const rel_attn_tensor* cache_seqlens, const rel_attn_tensor* cu_seqlens_q,
                             int32_t max_seqlen_q, float softmax_scale, int32_t causal, int32_t window_left,
                             int32_t window_right, int32_t rel_extent, const rel_attn_tensor* rel_logits,
                             int32_t num_splits, rel_attn_tensor* out, rel_attn_tensor* lse, rel_attn_stream stream,
                             const FixedWorkspace* fixed_ws);

// Set the thread-local message rel_attn_last_error() returns.
void set_last_error_message(const char* msg);

}  // namespace relattn
