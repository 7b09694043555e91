// Paged KV-cache append: the new tokens' keys and values written into the
// paged caches ahead of the attention.  The chunked-prefill configuration
// attends over caches that already hold the new tokens ("appending" them);
// this kernel is that write.  Token i of request b (global row
// t = cu_seqlens_q[b] + i) is the (sk_b - sq_b + i)-th key of the request,
// the same bottom-right position the attention gives it, so
//
//   key_cache[block_table[b, pos / BS], pos % BS, h, :] = key[t, h, :]
//   (value likewise),  pos = cache_seqlens[b] - sq_b + i,
//
// and a token with pos < 0 (cache_seqlens[b] < sq_b) has no slot and is
// skipped; so is a token whose slot lies past the table's width or in a
// block outside the cache (recorded in the device error word).  One warp per token: it finds the token's request with one
// parallel read of cu_seqlens_q and cache_seqlens (32 requests per read) and
// a ballot, reads the block id, then moves all kv heads of K and V in
// 16-byte pieces.
// HBM-bound: every byte is read once and written once.

#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace relattn {

namespace {

__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
    const int lane = threadIdx.x & 31;
    const long long t = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= p.T) return;
    // Request of token t: the last b < B with cu_seqlens_q[b] <= t (empty
    // requests share their start with the next one, so take the last).  Lane
    // l reads cu_seqlens_q and cache_seqlens of request base + l; since
    // cu_seqlens_q is non-decreasing the lanes with cu <= t form a prefix.
    int b = 0, q0 = 0, q1 = 0, skb = 0;
    for (int base = 0; base < p.B; base += 32) {
        const int l = base + lane;
        const int cu_l = l <= p.B ? __ldg(p.cu_seqlens_q + l) : INT_MAX;
        const int sk_l = l < p.B ? __ldg(p.cache_seqlens + l) : 0;
        const unsigned m = __ballot_sync(0xffffffffu, l < p.B && cu_l <= t);
        if (m == 0) break;  // the prefix ended in the previous chunk
        const int top = 31 - __clz((int)m);
        b = base + top;
        q0 = __shfl_sync(0xffffffffu, cu_l, top);
        skb = __shfl_sync(0xffffffffu, sk_l, top);
        q1 = __shfl_sync(0xffffffffu, cu_l, top < 31 ? top + 1 : 31);
        if (top == 31) q1 = __ldg(p.cu_seqlens_q + b + 1);
        if (m != 0xffffffffu) break;
    }
    const int sq = q1 - q0;
    const int pos = skb - sq + (int)(t - q0);
    if (pos < 0) return;
    // A slot past the block table's width or a block id outside the cache
    // breaks the caller's contract: the token is not written (a write is
    // never clamped into another slot) and the device error word says so.
    const int n = pos / p.BS;
    if (n >= p.MB) {
        if (lane == 0) atomicCAS(p.err, 0, kCodeAppendSlot);
        return;
    }
    const int blk = __ldg(p.block_table + (size_t)b * p.bt_stride + n);
    if (blk < 0 || blk >= p.NB) {
        if (lane == 0) atomicCAS(p.err, 0, kCodeAppendSlot);
        return;
    }
    const long long dst_row = (long long)blk * p.c_s0 + (long long)(pos % p.BS) * p.c_s1;
    const int chunks = p.D / 8;  // 16-byte pieces per (token, head) row
    const int per_tensor = p.Hk * chunks;
    // Batches of kBatch pieces per lane: every load of a batch is in flight
    // before its stores.
    constexpr int kBatch = 8;
    for (int c0 = 0; c0 < 2 * per_tensor; c0 += 32 * kBatch) {
        uint4 v[kBatch];
        uint16_t* dst[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int c = c0 + u * 32 + lane;
            dst[u] = nullptr;
            if (c < 2 * per_tensor) {
                const bool is_v = c >= per_tensor;
                const int cc = is_v ? c - per_tensor : c;
                const int h = cc / chunks, k = cc % chunks;
                const uint16_t* src = static_cast<const uint16_t*>(is_v ? p.value : p.key) +
                                      t * (is_v ? p.v_st : p.k_st) + (long long)h * (is_v ? p.v_sh : p.k_sh) + k * 8;
                dst[u] = static_cast<uint16_t*>(is_v ? p.v_cache : p.k_cache) + dst_row + (long long)h * p.c_s2 + k * 8;
                v[u] = __ldg(reinterpret_cast<const uint4*>(src));
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (dst[u]) *reinterpret_cast<uint4*>(dst[u]) = v[u];
    }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
    if (p.T <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((p.T + 7) / 8);
    append_kernel<<<blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace relattn
