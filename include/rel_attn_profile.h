/*
 * rel_attn_profile.h - introspection hooks for rel_attn.h, used by tests and
 * benchmarks.  They have no counterpart on the pages that define the
 * attention (vLLM API docs for fa4_rel_attention; prhub report on PR #48858):
 * they only expose what the library launched and how long its main kernel ran.
 */
#ifndef REL_ATTN_PROFILE_H
#define REL_ATTN_PROFILE_H

#include <stdint.h>

#include "rel_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    REL_ATTN_KERNEL_NONE = 0,
    REL_ATTN_KERNEL_DECODE = 1,   /* split-KV decode kernel, <= 64 packed rows  */
    REL_ATTN_KERNEL_PREFILL = 2,  /* tcgen05 prefill kernel, 128-row tiles      */
    REL_ATTN_KERNEL_APPEND = 3,   /* paged KV-cache append (rel_attn_cache_append) */
    REL_ATTN_KERNEL_PREFILL_PAIR = 4  /* tcgen05 prefill kernel on CTA pairs (2-SM MMAs, cta_group::2);
                                         head_dim 128 calls use it only when the environment variable
                                         REL_ATTN_PREFILL_PAIR=1 is set (the one-CTA kernel is faster
                                         there) */
} rel_attn_kernel_kind;

/* What the last rel_attn_paged_varlen call on this thread launched. */
typedef struct {
    int32_t kernel;       /* rel_attn_kernel_kind of the main kernel          */
    int32_t num_splits;   /* splits after clamping (1 = no combine)           */
    int32_t grid[3];      /* main kernel grid                                 */
    int32_t block;        /* main kernel threads per block                    */
    int32_t smem_bytes;   /* main kernel dynamic shared memory                */
    int32_t launches;     /* kernels launched by the call (main + combine...) */
    int64_t workspace_bytes; /* stream-ordered workspace allocated            */
} rel_attn_launch_info;

/* Copy the last call's launch record (thread-local).  NULL -> INVALID_ARGUMENT. */
rel_attn_status rel_attn_last_launch(rel_attn_launch_info* info);

/*
 * Record `begin` just before and `end` just after the main kernel of every
 * following rel_attn_paged_varlen, rel_attn_paged_varlen_lse or
 * rel_attn_cache_append call on this thread, on that call's stream.  Both are cudaEvent_t handles owned by the caller; pass NULL, NULL
 * to stop.  Lets a benchmark time the dominant kernel alone with CUDA events.
 */
rel_attn_status rel_attn_set_kernel_events(void* begin, void* end);

/*
 * Synchronise the current device, then read and clear the device error word
 * that the kernels set when a bounded wait on an mbarrier runs out (0 = none;
 * otherwise a code naming the wait site) or when the cache append skips a
 * token without a valid slot (REL_ATTN_CODE_APPEND_SLOT).  Kernels that time out return early
 * instead of hanging; their outputs are then undefined.
 */
rel_attn_status rel_attn_device_error(int32_t* code);

/* Wait-site code that rel_attn_check_wait_timeout records. */
#define REL_ATTN_SITE_SELF_TEST 99
/* Code the cache append records when it skips a token whose slot lies
 * outside the block table or the cache. */
#define REL_ATTN_CODE_APPEND_SLOT 31

/*
 * Self-test of the bounded-wait path: launch on `stream` a one-thread kernel
 * whose single mbarrier wait is never satisfied; after timeout_ms (1..10000)
 * it records REL_ATTN_SITE_SELF_TEST in the device error word (unless a code
 * is already there) and returns, as the attention kernels do when a hand-off
 * never comes.  The device stays usable; read the word with
 * rel_attn_device_error.  Returns INVALID_ARGUMENT for a timeout outside the
 * range, CUDA for a launch error.
 */
rel_attn_status rel_attn_check_wait_timeout(int32_t timeout_ms, rel_attn_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* REL_ATTN_PROFILE_H */
