/*
 * rel_attn.h - paged, variable-length attention with an additive
 * relative-position bias (Inkling relative attention), for NVIDIA GB300
 * (sm_103a).  Plain C ABI: borrowed tensor descriptors, a CUDA stream, a
 * status code.  No exceptions, aborts or traps cross it.
 *
 * The operation follows the interface of inkling_fa4_rel_attention in the vLLM
 * API docs for vllm.models.inkling.nvidia.ops.fa4_rel_attention (signature and
 * docstring), with the bias rule of score_mod_rel_bias in the prhub report on
 * vLLM PR #48858 ("关键源码片段", the source excerpt).  For request b with
 * sq_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] query tokens and
 * sk_b = cache_seqlens[b] cached keys, query row i (global token
 * t = cu_seqlens_q[b] + i) and query head h:
 *
 *   g      = h / (H / Hk)                                (GQA map)
 *   K_j    = key_cache[block_table[b, j / BS], j % BS, g, :]   (V_j likewise)
 *   d_j    = (i + sk_b - sq_b) - j                       (relative distance)
 *   bias_j = rel_logits[t, h, d_j] if 0 <= d_j < rel_extent, else exactly 0
 *   s_j    = softmax_scale * q[t,h,:] . K_j + bias_j     (bias after the scale)
 *   allowed_j = j < sk_b  and (!causal || d_j >= 0)
 *               and (window_left  < 0 || d_j <=  window_left)
 *               and (window_right < 0 || d_j >= -window_right)
 *   out[t,h,:] = sum_allowed softmax(s)_j V_j ;  0 if no key is allowed.
 *
 * The causal mask is aligned bottom-right (row i sits at key position
 * i + sk_b - sq_b, the same offset the bias uses).
 */
#ifndef REL_ATTN_H
#define REL_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* A cudaStream_t.  NULL is the legacy default stream. */
typedef struct CUstream_st* rel_attn_stream;

typedef enum {
    REL_ATTN_BF16 = 0,
    REL_ATTN_F32 = 1,
    REL_ATTN_I32 = 2
} rel_attn_dtype;

/*
 * Borrowed view of one tensor.  data is a DEVICE pointer; shape and stride
 * are in elements (stride[k] is the element step of dimension k).  The
 * library never keeps the pointer past the stream work of the call.
 */
typedef struct {
    void* data;
    int32_t dtype;      /* rel_attn_dtype */
    int32_t ndim;
    int64_t shape[4];
    int64_t stride[4];
} rel_attn_tensor;

typedef enum {
    REL_ATTN_OK = 0,
    REL_ATTN_ERR_INVALID_ARGUMENT = 1,
    REL_ATTN_ERR_UNSUPPORTED = 2,
    REL_ATTN_ERR_CUDA = 3,
    REL_ATTN_ERR_OUT_OF_MEMORY = 4,
    REL_ATTN_ERR_DEVICE_CHECK = 5
} rel_attn_status;

/*
 * rel_attn_paged_varlen - the forward.  Defined by inkling_fa4_rel_attention
 * (vLLM API docs, fa4_rel_attention); bias rule from score_mod_rel_bias (prhub
 * report on PR #48858, source excerpt).
 *
 * Arguments (all tensors on the current CUDA device, sm_103):
 *   q              (T, H, D) bf16; last dim contiguous, strides 16-byte multiples
 *   key_cache      (NB, BS, Hk, D) bf16; last dim contiguous; base 16-byte aligned,
 *                  other strides 16-byte multiples
 *   value_cache    same shape and strides as key_cache
 *   block_table    (B, MB) int32, row-major contiguous: physical block of
 *                  request b's logical block n
 *   cache_seqlens  (B,) int32 = seqused_k, 0 <= sk_b <= MB * BS
 *   cu_seqlens_q   (B+1,) int32, cu[0] = 0, non-decreasing, cu[B] = T
 *   max_seqlen_q   >= every sq_b (the kernel choice and grid come from it)
 *   softmax_scale  multiplies q.k before the bias is added
 *   causal         nonzero: bottom-right aligned causal mask
 *   window_left, window_right
 *                  sliding window in keys; a negative side is unbounded;
 *                  (-1, -1) means no window
 *   rel_extent     R >= 0; R == 0 means no bias (rel_logits may then be NULL)
 *   rel_logits     (T, H, R) bf16 or fp32, fully contiguous (the pages make the
 *                  bias tensor contiguous before the call); bf16 rows with
 *                  R % 8 == 0 are staged by TMA on the prefill path, other
 *                  rows (fp32, or an R that is not a multiple of 8) are read
 *                  per element
 *   num_splits     >= 1: a cap on the number of KV splits per (request, kv head);
 *                  1 writes out directly, >1 writes fp32 partials and runs an
 *                  LSE-weighted combine.  Clamped to what the KV length allows.
 *   out            (T, H, D) bf16 (or fp32, which keeps the result before the
 *                  final bf16 rounding), caller-allocated; must not alias an input
 *   stream         the stream all work is ordered on
 *
 * Supported: D in {64, 128, 256}; BS a multiple of 16; H % Hk == 0;
 * H / Hk <= 128.  Above 64 GQA-packed rows, D = 256 runs the CTA-pair prefill
 * kernel (2-SM tcgen05 MMAs); D = 64 and 128 run the one-CTA prefill kernel
 * (D = 128 on the CTA-pair kernel when the environment variable
 * REL_ATTN_PREFILL_PAIR=1 is set and rel_logits are bf16 with R % 8 == 0 or
 * absent).
 *
 * Ownership: every tensor is caller-owned device memory, borrowed until the
 * stream work completes.  When num_splits > 1 the library allocates a
 * stream-ordered workspace (cudaMallocAsync / cudaFreeAsync on `stream`) of
 * num_splits * T * H * (D + 1) * 4 bytes.
 *
 * Errors: REL_ATTN_ERR_INVALID_ARGUMENT for a NULL pointer with a nonzero
 * size, a dtype/rank/shape/stride mismatch, H % Hk != 0, num_splits < 1 or
 * rel_extent < 0; REL_ATTN_ERR_UNSUPPORTED for another D or BS, a device that
 * is not sm_103, a layout TMA cannot address, or a tensor that is not device
 * memory of the current device (host memory, another GPU's memory; checked
 * with cudaPointerGetAttributes before any tensor map is encoded; q, out,
 * block_table, cache_seqlens, cu_seqlens_q and softmax_lse may also be
 * managed memory, the caches and rel_logits, read by TMA, may not);
 * REL_ATTN_ERR_OUT_OF_MEMORY
 * when the workspace cannot be allocated; REL_ATTN_ERR_CUDA for a launch
 * error.  rel_attn_last_error() then describes it.  T == 0 returns OK and
 * launches nothing.  Device-side preconditions (monotone cu_seqlens_q,
 * sq_b <= max_seqlen_q, block ids < NB, sk_b <= MB * BS) are documented, not
 * checked, unless the environment variable REL_ATTN_CHECK=1 is set, in which
 * case a check kernel runs first, the call synchronises `stream`, and a
 * violation returns REL_ATTN_ERR_DEVICE_CHECK without running the forward.
 * Without the check, a block id outside [0, NB) is clamped into the cache and
 * a key past the table's width reads no table entry, so a broken table gives
 * wrong values, never a read outside the caches.
 */
rel_attn_status rel_attn_paged_varlen(
    const rel_attn_tensor* q,
    const rel_attn_tensor* key_cache,
    const rel_attn_tensor* value_cache,
    const rel_attn_tensor* block_table,
    const rel_attn_tensor* cache_seqlens,
    const rel_attn_tensor* cu_seqlens_q,
    int32_t max_seqlen_q,
    float softmax_scale,
    int32_t causal,
    int32_t window_left,
    int32_t window_right,
    int32_t rel_extent,
    const rel_attn_tensor* rel_logits,
    int32_t num_splits,
    rel_attn_tensor* out,
    rel_attn_stream stream);

/*
 * rel_attn_paged_varlen_lse - rel_attn_paged_varlen that also writes the
 * log-sum-exp of each output row.  inkling_fa4_rel_attention (vLLM API docs,
 * fa4_rel_attention) calls the attention with return_lse=False; this entry
 * point is the return_lse=True form of the same call:
 *
 *   softmax_lse[t, h] = ln( sum_{allowed j} exp(s_j) ),  -inf if no key is allowed,
 *
 * with s_j the scaled, biased score defined above (natural logarithm, fp32).
 * With num_splits > 1 it is the merged value of all splits.
 *
 * Arguments are those of rel_attn_paged_varlen plus
 *   softmax_lse    (T, H) fp32, caller-allocated device memory, any strides >= 0
 *                  in elements (a transposed view of an (H, T) buffer gives the
 *                  FlashAttention layout); every (t, h) must address a distinct
 *                  element; must not alias out or an input; 4-byte aligned.
 *                  NULL makes the call identical to rel_attn_paged_varlen.
 *
 * Ownership and errors are those of rel_attn_paged_varlen, plus
 * REL_ATTN_ERR_INVALID_ARGUMENT for a softmax_lse of the wrong dtype, rank or
 * shape, a negative stride, misalignment, or overlap with out or an input.
 */
rel_attn_status rel_attn_paged_varlen_lse(
    const rel_attn_tensor* q,
    const rel_attn_tensor* key_cache,
    const rel_attn_tensor* value_cache,
    const rel_attn_tensor* block_table,
    const rel_attn_tensor* cache_seqlens,
    const rel_attn_tensor* cu_seqlens_q,
    int32_t max_seqlen_q,
    float softmax_scale,
    int32_t causal,
    int32_t window_left,
    int32_t window_right,
    int32_t rel_extent,
    const rel_attn_tensor* rel_logits,
    int32_t num_splits,
    rel_attn_tensor* out,
    rel_attn_tensor* softmax_lse,
    rel_attn_stream stream);

/*
 * rel_attn_paged_varlen_noalloc - rel_attn_paged_varlen that allocates no
 * device memory.  It has no counterpart on the pages that define the
 * attention; it exists for callers that cannot allocate: a framework that owns
 * the device through its own memory pool (a second allocator working behind
 * its back can run out of memory while the pool holds nearly all of the
 * device, or fragment it), or a program that allocates everything at start-up
 * and forbids allocation afterwards.
 *
 * Arguments, validation, status codes, kernels, the REL_ATTN_CHECK device
 * check, the wait timeout and the launch record are those of
 * rel_attn_paged_varlen (one shared implementation, decode and prefill path
 * alike).  The caller still provides every input and the output.  The only
 * difference is the split-KV workspace (num_splits * T * H * (D + 1) * 4
 * bytes, after num_splits is clamped; none with one split): it comes from a
 * fixed array of REL_ATTN_NOALLOC_SCRATCH_BYTES bytes inside the library, and
 * every GPU that loads the library holds one such array until the process
 * exits.  A call whose workspace would not fit returns
 * REL_ATTN_ERR_INVALID_ARGUMENT with a message naming both sizes, before any
 * device work.  It calls no cudaMalloc, cudaMallocAsync, cudaFree or other
 * allocating routine.
 *
 * The first call on each device that passes host validation looks up the
 * device address of the array (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture.  All calls share
 * the one array and it keeps the last call's contents; nothing in it needs to
 * start at zero, since every value the combine step reads is written earlier
 * in the same call.  Calls that use more than one split and overlap on the
 * GPU (other streams, other host threads) race on the array: order them on
 * one stream.
 */
#define REL_ATTN_NOALLOC_SCRATCH_BYTES (16u << 20)

rel_attn_status rel_attn_paged_varlen_noalloc(
    const rel_attn_tensor* q,
    const rel_attn_tensor* key_cache,
    const rel_attn_tensor* value_cache,
    const rel_attn_tensor* block_table,
    const rel_attn_tensor* cache_seqlens,
    const rel_attn_tensor* cu_seqlens_q,
    int32_t max_seqlen_q,
    float softmax_scale,
    int32_t causal,
    int32_t window_left,
    int32_t window_right,
    int32_t rel_extent,
    const rel_attn_tensor* rel_logits,
    int32_t num_splits,
    rel_attn_tensor* out,
    rel_attn_stream stream);

/*
 * rel_attn_cache_append - write the new tokens' keys and values into the paged
 * caches, the step before attending over them.  The attention of
 * inkling_fa4_rel_attention (vLLM API docs) reads cache_seqlens keys per
 * request and aligns query row i at key position i + cache_seqlens[b] - sq_b
 * (bottom-right), so the new tokens are the last sq_b keys of the cache and
 * must be in it before the call.  The pages show no interface for that write,
 * so this one reuses the attention's arguments: token i of
 * request b (row t = cu_seqlens_q[b] + i) is the key at logical position
 * pos = cache_seqlens[b] - sq_b + i, the bottom-right position the attention
 * gives it, and
 *
 *   key_cache[block_table[b, pos / BS], pos % BS, h, :] = key[t, h, :]
 *   value_cache[...same slot...]                        = value[t, h, :]
 *
 * for every kv head h.  A token with pos < 0 (cache_seqlens[b] < sq_b) has no
 * slot and is not written.  Bits are copied unchanged.
 *
 * Arguments (device tensors, current device, sm_103):
 *   key, value     (T, Hk, D) bf16; last dim contiguous, base and strides
 *                  16-byte multiples; read only
 *   key_cache, value_cache
 *                  (NB, BS, Hk, D) bf16 as for rel_attn_paged_varlen; written
 *   block_table, cache_seqlens, cu_seqlens_q
 *                  as for rel_attn_paged_varlen (cache_seqlens already counts
 *                  the new tokens)
 *   stream         the stream the copy is ordered on
 *
 * Supported: D a multiple of 8 up to 512; any BS > 0.
 * Ownership: all tensors caller-owned, borrowed until the stream work
 * completes; nothing is allocated.  The slots written must be distinct (block
 * tables of different requests must not share a slot in the written range);
 * otherwise which write lands is unspecified.
 * Errors: REL_ATTN_ERR_INVALID_ARGUMENT for a NULL pointer with a nonzero size,
 * a dtype/rank/shape/stride mismatch, or key/value overlapping a cache;
 * REL_ATTN_ERR_UNSUPPORTED for a D it cannot copy, misaligned data, a tensor
 * that is not device memory of the current device, or a device that is not
 * sm_103; REL_ATTN_ERR_CUDA for a launch error.  T == 0 is a no-op.
 * Device-side preconditions as for rel_attn_paged_varlen (checked when
 * REL_ATTN_CHECK=1).  Without the check, a token whose slot lies past the
 * table's width (pos / BS >= MB) or in a block id outside [0, NB) is not
 * written (a write is never clamped into another slot) and the device error
 * word (rel_attn_device_error, rel_attn_profile.h) records
 * REL_ATTN_CODE_APPEND_SLOT.
 */
rel_attn_status rel_attn_cache_append(
    const rel_attn_tensor* key,
    const rel_attn_tensor* value,
    rel_attn_tensor* key_cache,
    rel_attn_tensor* value_cache,
    const rel_attn_tensor* block_table,
    const rel_attn_tensor* cache_seqlens,
    const rel_attn_tensor* cu_seqlens_q,
    rel_attn_stream stream);

/*
 * rel_attn_num_splits - split-KV cap for this attention, defined by
 * inkling_fa4_num_splits (vLLM API docs, fa4_rel_attention) without its
 * Hopper branch (this library runs on sm_103 only).  Local (windowed)
 * attention gets 1.  Otherwise the GQA-packed query rows
 * max_query_len * (num_heads / num_kv_heads) are cut into 256-row tiles,
 * base = batch_size * num_kv_heads * tiles, target = 256 (one tile, batch 1),
 * 128 (one tile) or 64, a batch-1 single-tile cap of 16 (8 kv heads), 32
 * (4 kv heads or KV <= 8192), 64 (KV <= 65536) or 128, else a cap of 128;
 * the result is max(1, min(target / base, cap, ceil(max_kv_len / 128))).
 * Pure host integer logic; no device is touched.
 * Returns >= 1, or -REL_ATTN_ERR_INVALID_ARGUMENT when batch_size < 1,
 * max_query_len < 1, num_heads < 1, num_kv_heads < 1,
 * num_heads % num_kv_heads != 0 or max_kv_len < 0.
 */
int32_t rel_attn_num_splits(int32_t is_local, int32_t batch_size, int32_t max_query_len,
                            int32_t num_heads, int32_t num_kv_heads, int32_t max_kv_len);

/*
 * rel_attn_bucket_max_seqlen_q - the query-length bucket of
 * bucket_max_seqlen_q (vLLM API docs, fa4_rel_attention): the smallest power of
 * two >= max_seqlen_q (1 for 0 and 1).  A caller that captures calls in a
 * CUDA graph passes this bucket as max_seqlen_q, so one captured launch serves
 * every batch whose longest query fits the bucket (the kernels read the actual
 * lengths from cu_seqlens_q on the device).  Pure host integer logic.
 * Returns the bucket, or -REL_ATTN_ERR_INVALID_ARGUMENT when max_seqlen_q < 0
 * or the bucket would exceed 2^30.
 */
int32_t rel_attn_bucket_max_seqlen_q(int32_t max_seqlen_q);

/*
 * rel_attn_last_error - thread-local, NUL-terminated description of the last
 * non-OK status returned on this thread ("" if none).  Owned by the library;
 * valid until the next call on the same thread.
 */
const char* rel_attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* REL_ATTN_H */
