// Split-KV combine: out[t,h,:] = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),
// M = max_s lse_s, where o_s is split s's normalised partial output and lse_s
// its log2-sum-exp; a row whose every split is empty (all lse = -inf) gets 0.
// One warp per (token, head) row, D/32 contiguous dims per lane.
//
// The split count is the num_splits argument of inkling_fa4_rel_attention
// (vLLM API docs, fa4_rel_attention); the merge itself is the standard
// log-sum-exp rescaling of softmax partials.

#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace relattn {

namespace {

template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const AttnParams p) {
    constexpr int V = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long rows = (long long)p.T * p.H;
    const long long row = (long long)blockIdx.x * 8 + warp;
    if (row >= rows) return;
    const int S = p.num_splits;
    float mx = -CUDART_INF_F;
    for (int s = lane; s < S; s += 32) mx = fmaxf(mx, p.ws_lse[(size_t)s * rows + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    if (mx != -CUDART_INF_F) {
        float L = 0.f;
        for (int s = 0; s < S; ++s) {
            const float lse = p.ws_lse[(size_t)s * rows + row];
            if (lse == -CUDART_INF_F) continue;
            const float w = ex2(lse - mx);
            L += w;
            const float* src = p.ws_o + ((size_t)s * rows + row) * D + lane * V;
            if constexpr (V == 4) {
                const float4 v = *reinterpret_cast<const float4*>(src);
                acc[0] = fmaf(w, v.x, acc[0]);
                acc[1] = fmaf(w, v.y, acc[1]);
                acc[2] = fmaf(w, v.z, acc[2]);
                acc[3] = fmaf(w, v.w, acc[3]);
            } else {
                const float2 v = *reinterpret_cast<const float2*>(src);
                acc[0] = fmaf(w, v.x, acc[0]);
                acc[1] = fmaf(w, v.y, acc[1]);
            }
        }
        const float inv = 1.f / L;
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] *= inv;
    }
    const int t = (int)(row / p.H), h = (int)(row % p.H);
    const size_t oo = (size_t)t * p.o_st + (size_t)h * p.o_sh + lane * V;
    if (p.out_f32) {
        float* dst = reinterpret_cast<float*>(p.out) + oo;
        if constexpr (V == 4)
            *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        else
            *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
        return;
    }
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + oo;
    if constexpr (V == 4) {
        uint2 pk;
        pk.x = pack_bf16(acc[0], acc[1]);
        pk.y = pack_bf16(acc[2], acc[3]);
        *reinterpret_cast<uint2*>(dst) = pk;
    } else {
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0], acc[1]);
    }
}

}  // namespace

cudaError_t launch_combine(const AttnParams& p, cudaStream_t stream) {
    const long long rows = (long long)p.T * p.H;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    if (p.D == 128)
        combine_kernel<128><<<blocks, 256, 0, stream>>>(p);
    else if (p.D == 64)
        combine_kernel<64><<<blocks, 256, 0, stream>>>(p);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace relattn
