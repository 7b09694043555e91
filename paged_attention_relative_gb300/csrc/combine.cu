// Split-KV combine: out[t,h,:] = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),
// M = max_s lse_s, where o_s is split s's normalised partial output and lse_s
// its log2-sum-exp; a row whose every split is empty (all lse = -inf) gets 0.
// When requested, the row's natural-log sum-exp (M + log2 sum) * ln 2 goes to lse.
// One warp per (token, head) row, D/32 contiguous dims per lane (D = 64, 128, 256).
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
    // Launched as a programmatic dependent of the attention kernel: start up
    // while it finishes, read its partials only once it has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long rows = (long long)p.T * p.H;
    const long long row = (long long)blockIdx.x * 8 + warp;
    if (row >= rows) return;
    const int S = p.num_splits;
    // Lane l holds the log2-sum-exp of splits l, l+32, ... (all loads in flight at once).
    float lse_l[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int s = lane + 32 * k;
        lse_l[k] = s < S ? p.ws_lse[(size_t)s * rows + row] : -CUDART_INF_F;
    }
    float mx = fmaxf(fmaxf(lse_l[0], lse_l[1]), fmaxf(lse_l[2], lse_l[3]));
    for (int s = lane + 128; s < S; s += 32) mx = fmaxf(mx, p.ws_lse[(size_t)s * rows + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    float lse_row = -CUDART_INF_F;  // natural log of the merged sum-exp
    if (mx != -CUDART_INF_F) {
        float L = 0.f;
        const float* base = p.ws_o + (size_t)row * D + lane * V;
        const size_t split_stride = (size_t)rows * D;
        for (int s0 = 0; s0 < S; s0 += 32) {
            // weights of splits s0..s0+31, one per lane
            const int k = s0 >> 5;
            float lse;
            if (k == 0)
                lse = lse_l[0];
            else if (k == 1)
                lse = lse_l[1];
            else if (k == 2)
                lse = lse_l[2];
            else if (k == 3)
                lse = lse_l[3];
            else
                lse = s0 + lane < S ? p.ws_lse[(size_t)(s0 + lane) * rows + row] : -CUDART_INF_F;
            const float w_l = lse == -CUDART_INF_F ? 0.f : ex2(lse - mx);
            const int n = min(32, S - s0);
#pragma unroll 8
            for (int j = 0; j < n; ++j) {
                const float w = __shfl_sync(0xffffffffu, w_l, j);
                L += w;
                const float* src = base + (size_t)(s0 + j) * split_stride;
                if constexpr (V == 8) {
                    const float4 v = *reinterpret_cast<const float4*>(src);
                    const float4 u = *reinterpret_cast<const float4*>(src + 4);
                    acc[0] = fmaf(w, v.x, acc[0]);
                    acc[1] = fmaf(w, v.y, acc[1]);
                    acc[2] = fmaf(w, v.z, acc[2]);
                    acc[3] = fmaf(w, v.w, acc[3]);
                    acc[4] = fmaf(w, u.x, acc[4]);
                    acc[5] = fmaf(w, u.y, acc[5]);
                    acc[6] = fmaf(w, u.z, acc[6]);
                    acc[7] = fmaf(w, u.w, acc[7]);
                } else if constexpr (V == 4) {
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
        }
        const float inv = 1.f / L;
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] *= inv;
        lse_row = (mx + __log2f(L)) * kLn2;
    }
    const int t = (int)(row / p.H), h = (int)(row % p.H);
    if (p.lse && lane == 0) p.lse[(size_t)t * p.lse_st + (size_t)h * p.lse_sh] = lse_row;
    const size_t oo = (size_t)t * p.o_st + (size_t)h * p.o_sh + lane * V;
    if (p.out_f32) {
        float* dst = reinterpret_cast<float*>(p.out) + oo;
        if constexpr (V == 8) {
            *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        } else if constexpr (V == 4) {
            *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        } else {
            *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
        }
        return;
    }
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + oo;
    if constexpr (V == 8) {
        uint4 pk;
        pk.x = pack_bf16(acc[0], acc[1]);
        pk.y = pack_bf16(acc[2], acc[3]);
        pk.z = pack_bf16(acc[4], acc[5]);
        pk.w = pack_bf16(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(dst) = pk;
    } else if constexpr (V == 4) {
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (p.D == 256)
        e = cudaLaunchKernelEx(&cfg, combine_kernel<256>, p);
    else if (p.D == 128)
        e = cudaLaunchKernelEx(&cfg, combine_kernel<128>, p);
    else if (p.D == 64)
        e = cudaLaunchKernelEx(&cfg, combine_kernel<64>, p);
    else
        return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace relattn
