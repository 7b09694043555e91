// Split-KV decode kernel: one CTA per (split, kv head, request) over at most
// 64 GQA-packed query rows (query token i, head g*G + r packed as row i*G + r),
// so every K/V byte of a kv head is read from HBM once per split.
//
// Pipeline: one producer warp issues TMA tile loads of 16-key page slices
// (box 64 dims x 1 head x 16 slots x 1 block, 128-byte swizzle) into an
// nstage-deep ring of K/V stages; consumer warps wait on the stage's full
// mbarrier, run QK^T and PV on bf16 mma.sync (fp32 accumulate), apply the
// scale, the sheared relative bias and the mask per element, keep an fp32
// online softmax, and release the stage.  Warps split the stage's keys
// (KSL slices of 16) and the rows (MT tiles of 16); their partial (m, l, O)
// merge through shared memory at the end.  With one split the result is
// written as bf16; otherwise the fp32 O/l and log2-sum-exp go to the
// workspace for the combine kernel.
//
// Semantics: vLLM API docs, inkling_fa4_rel_attention (paged varlen forward);
// bias rule: prhub report on vLLM PR #48858, score_mod_rel_bias.

#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace relattn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D, int MT, int KSL>
struct DecodeCfg {
    static constexpr int kWarps = MT * KSL;              // consumer warps
    static constexpr int kThreads = (kWarps + 1) * 32;   // + one producer warp
    static constexpr int kStageKeys = 16 * KSL;
    static constexpr int kHalves = D / 64;               // 64-dim swizzled column blocks
    static constexpr int kHalfBytes = kStageKeys * 128;  // one column block of one operand
    static constexpr int kStageBytes = 2 * kHalves * kHalfBytes;
    static constexpr int kRedStride = D + 4;             // floats per row in the merge area
    static constexpr int kRedBytes = KSL * MT * 16 * (kRedStride + 2) * 4;
    static constexpr int kMaxStages = 16;
};

struct RowInfo {
    int valid;
    int pos;                   // key position of the query row
    const uint16_t* rel;       // rel_logits row (t, h, :)
};

template <int D, int MT, int KSL>
__global__ void __launch_bounds__(DecodeCfg<D, MT, KSL>::kThreads)
decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const AttnParams p) {
    using C = DecodeCfg<D, MT, KSL>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int nstage = p.nstage;
    const size_t body = (size_t)nstage * C::kStageBytes > (size_t)C::kRedBytes ? (size_t)nstage * C::kStageBytes
                                                                                : (size_t)C::kRedBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + body);
    uint64_t* empty = full + C::kMaxStages;
    int* abort_flag = reinterpret_cast<int*>(empty + C::kMaxStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = p.G;

    const int q0 = p.cu_seqlens_q[b];
    const int sq = p.cu_seqlens_q[b + 1] - q0;
    const int sk = p.cache_seqlens[b];
    const int n_rows = min(sq * G, p.max_rows);
    if (n_rows <= 0) return;
    const int off = sk - sq;

    // Keys any row of this request may see, cut into stage tiles and split.
    int khi = sk;
    if (p.causal) khi = min(khi, sq + off);
    if (p.wr >= 0) khi = min(khi, sq + off + p.wr);
    int klo = 0;
    if (p.wl >= 0) klo = max(0, off - p.wl);
    const int BN = C::kStageKeys;
    const int kstart = (klo / BN) * BN;
    const int n_tiles = khi > kstart ? (khi - kstart + BN - 1) / BN : 0;
    const int splits_eff = min(p.num_splits, n_tiles);
    int t_begin = 0, t_end = 0;
    if (split < splits_eff) {
        t_begin = (int)(((long long)split * n_tiles) / splits_eff);
        t_end = (int)(((long long)(split + 1) * n_tiles) / splits_eff);
    }
    const int n_it = t_end - t_begin;

    if (threadIdx.x == 0) {
        for (int i = 0; i < nstage; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], C::kWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    auto k_half = [&](int slot, int hh) { return smem + (size_t)slot * C::kStageBytes + hh * C::kHalfBytes; };
    auto v_half = [&](int slot, int hh) {
        return smem + (size_t)slot * C::kStageBytes + (C::kHalves + hh) * C::kHalfBytes;
    };

    if (warp == C::kWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        const uint64_t policy = l2_policy_evict_first();
        const int nblk_needed = min((khi + p.BS - 1) / p.BS, p.max_blocks);
        const int32_t* bt = p.block_table + (size_t)b * p.bt_stride;
        int cached_base = -(1 << 30);
        int my_blk = -1;
        for (int it = 0; it < n_it; ++it) {
            const int slot = it % nstage;
            const int round = it / nstage;
            const int k0 = kstart + (t_begin + it) * BN;
            bool ok = true;
            if (lane == 0) ok = mbar_wait(&empty[slot], (round & 1) ^ 1, p.timeout_ns, kSiteDecodeEmpty, p.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            int nvalid = 0;
#pragma unroll
            for (int u = 0; u < KSL; ++u) nvalid += (k0 + 16 * u < khi) ? 1 : 0;
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(nvalid * 2 * C::kHalves * 2048));
#pragma unroll
            for (int u = 0; u < KSL; ++u) {
                const int j = k0 + 16 * u;
                if (j >= khi) break;  // warp-uniform
                const int n = j / p.BS;
                if (n - cached_base >= 32 || n < cached_base) {
                    cached_base = n;
                    my_blk = (n + lane < nblk_needed) ? bt[n + lane] : -1;
                }
                const int blk = __shfl_sync(0xffffffffu, my_blk, n - cached_base);
                if (lane == 0) {
                    const int slot_in_blk = j - n * p.BS;
#pragma unroll
                    for (int hh = 0; hh < C::kHalves; ++hh) {
                        tma_load_4d_hint(k_half(slot, hh) + u * 2048, &tmK, &full[slot], hh * 64, g, slot_in_blk,
                                         blk, policy);
                        tma_load_4d_hint(v_half(slot, hh) + u * 2048, &tmV, &full[slot], hh * 64, g, slot_in_blk,
                                         blk, policy);
                    }
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int mt = warp % MT, ks = warp / MT;
    const int gq = lane >> 2, tig = lane & 3;
    const int rloc[2] = {mt * 16 + gq, mt * 16 + gq + 8};
    RowInfo ri[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int r = rloc[e];
        ri[e].valid = r < n_rows;
        const int qi = ri[e].valid ? r / G : 0;
        const int hh = ri[e].valid ? r % G : 0;
        ri[e].pos = qi + off;
        const int t = q0 + qi, h = g * G + hh;
        ri[e].rel = p.R > 0 ? reinterpret_cast<const uint16_t*>(p.rel) + ((size_t)t * p.H + h) * p.R : nullptr;
    }

    // Q fragments (A operand, rows x dims), loaded once.
    uint32_t qf[D / 16][4];
    {
        const uint16_t* qb = reinterpret_cast<const uint16_t*>(p.q);
        const uint32_t* rowp[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = ri[e].valid ? rloc[e] : 0;
            const int t = q0 + r / G, h = g * G + r % G;
            rowp[e] = reinterpret_cast<const uint32_t*>(qb + (size_t)t * p.q_st + (size_t)h * p.q_sh);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qf[kk][0] = ri[0].valid ? __ldg(rowp[0] + kk * 8 + tig) : 0u;
            qf[kk][1] = ri[1].valid ? __ldg(rowp[1] + kk * 8 + tig) : 0u;
            qf[kk][2] = ri[0].valid ? __ldg(rowp[0] + kk * 8 + 4 + tig) : 0u;
            qf[kk][3] = ri[1].valid ? __ldg(rowp[1] + kk * 8 + 4 + tig) : 0u;
        }
    }

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
    float l_run[2] = {0.f, 0.f};
    const float sl2 = p.scale_log2;
    const int R = p.R, wl = p.wl, wr = p.wr, causal = p.causal;

    for (int it = 0; it < n_it; ++it) {
        const int slot = it % nstage;
        const int round = it / nstage;
        const int jb = kstart + (t_begin + it) * BN + ks * 16;  // this warp's first key
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&full[slot], round & 1, p.timeout_ns, kSiteDecodeFull, p.err);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0) *abort_flag = 1;
            break;
        }
        // Keys at or past khi hold stale or unloaded data: zero their V rows so
        // that p = 0 times them stays 0.
        if (jb + 16 > khi) {
            const int first = max(0, khi - jb);
            for (int idx = lane; idx < (16 - first) * 8 * C::kHalves; idx += 32) {
                const int row = first + idx / (8 * C::kHalves);
                const int rem = idx % (8 * C::kHalves);
                uint8_t* base = v_half(slot, rem / 8) + (ks * 16 + row) * 128 + (rem % 8) * 16;
                *reinterpret_cast<uint4*>(base) = make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }

        // S = Q K^T over this warp's 16 keys: two n-tiles of 8 keys.
        float sacc[2][4];
#pragma unroll
        for (int i = 0; i < 2; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
        {
            const int krow = ks * 16 + (lane >> 4) * 8 + (lane & 7);
            const int csel = (lane >> 3) & 1;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t addr =
                    smem_u32(k_half(slot, kk >> 2)) + sw128_offset(krow, (kk & 3) * 2 + csel);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(addr, b0, b1, b2, b3);
                mma_bf16_16816(sacc[0], qf[kk], b0, b1);
                mma_bf16_16816(sacc[1], qf[kk], b2, b3);
            }
        }

        // Scale, sheared bias, mask.
        float s[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const RowInfo& rr = ri[e >> 1];
                const int j = jb + nt * 8 + 2 * tig + (e & 1);
                const int d = rr.pos - j;
                bool allowed = rr.valid && j < khi;
                if (causal) allowed = allowed && d >= 0;
                if (wl >= 0) allowed = allowed && d <= wl;
                if (wr >= 0) allowed = allowed && d >= -wr;
                float bias = 0.f;
                if (allowed && d >= 0 && d < R) bias = bf16_bits_to_f32(__ldg(rr.rel + d));
                s[nt][e] = allowed ? fmaf(sacc[nt][e], sl2, bias * kLog2e) : -CUDART_INF_F;
            }
        }

        // Online softmax (base 2).  Rows gq (e = 0,1) and gq + 8 (e = 2,3).
        float alpha[2];
#pragma unroll
        for (int rsel = 0; rsel < 2; ++rsel) {
            float mx = fmaxf(fmaxf(s[0][2 * rsel], s[0][2 * rsel + 1]), fmaxf(s[1][2 * rsel], s[1][2 * rsel + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run[rsel], mx);
            const float mu = m_new == -CUDART_INF_F ? 0.f : m_new;
            alpha[rsel] = ex2(m_run[rsel] - mu);
            float rs = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                s[nt][2 * rsel] = ex2(s[nt][2 * rsel] - mu);
                s[nt][2 * rsel + 1] = ex2(s[nt][2 * rsel + 1] - mu);
                rs += s[nt][2 * rsel] + s[nt][2 * rsel + 1];
            }
            l_run[rsel] = l_run[rsel] * alpha[rsel] + rs;
            m_run[rsel] = m_new;
        }
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            o[i][0] *= alpha[0];
            o[i][1] *= alpha[0];
            o[i][2] *= alpha[1];
            o[i][3] *= alpha[1];
        }

        // O += P V.
        uint32_t pa[4];
        pa[0] = pack_bf16(s[0][0], s[0][1]);
        pa[1] = pack_bf16(s[0][2], s[0][3]);
        pa[2] = pack_bf16(s[1][0], s[1][1]);
        pa[3] = pack_bf16(s[1][2], s[1][3]);
        {
            const int vrow = ks * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
            const int csel = lane >> 4;
#pragma unroll
            for (int n2 = 0; n2 < D / 16; ++n2) {
                const uint32_t addr =
                    smem_u32(v_half(slot, n2 >> 2)) + sw128_offset(vrow, (n2 & 3) * 2 + csel);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(addr, b0, b1, b2, b3);
                mma_bf16_16816(o[2 * n2], pa, b0, b1);
                mma_bf16_16816(o[2 * n2 + 1], pa, b2, b3);
            }
        }
        if (jb + 16 > khi) fence_proxy_async_smem();  // generic zeroing before the next TMA write
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // Quad-reduce the row sums (each thread summed its own columns).
#pragma unroll
    for (int rsel = 0; rsel < 2; ++rsel) {
        l_run[rsel] += __shfl_xor_sync(0xffffffffu, l_run[rsel], 1);
        l_run[rsel] += __shfl_xor_sync(0xffffffffu, l_run[rsel], 2);
    }

    // Merge the KSL key slices through shared memory (stage buffers are free:
    // every issued stage was waited on by every consumer warp).
    asm volatile("bar.sync 1, %0;" ::"r"(C::kWarps * 32) : "memory");
    if (*(volatile int*)abort_flag) return;  // CTA-uniform: every consumer warp sees it
    float* red_o = reinterpret_cast<float*>(smem);
    float* red_m = red_o + KSL * MT * 16 * C::kRedStride;
    float* red_l = red_m + KSL * MT * 16;
    const int rows_cta = MT * 16;
#pragma unroll
    for (int rsel = 0; rsel < 2; ++rsel) {
        const int r = rloc[rsel];
        float* dst = red_o + ((size_t)ks * rows_cta + r) * C::kRedStride;
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
            *reinterpret_cast<float2*>(dst + i * 8 + 2 * tig) = make_float2(o[i][2 * rsel], o[i][2 * rsel + 1]);
        if (tig == 0) {
            red_m[ks * rows_cta + r] = m_run[rsel];
            red_l[ks * rows_cta + r] = l_run[rsel];
        }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(C::kWarps * 32) : "memory");

    const bool partial = p.num_splits > 1;
    for (int idx = threadIdx.x; idx < rows_cta * (D / 4); idx += C::kWarps * 32) {
        const int r = idx / (D / 4), c4 = idx % (D / 4);
        if (r >= n_rows) continue;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < KSL; ++k) M = fmaxf(M, red_m[k * rows_cta + r]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int k = 0; k < KSL; ++k) {
                const float w = ex2(red_m[k * rows_cta + r] - M);
                L += w * red_l[k * rows_cta + r];
                const float4 v = *reinterpret_cast<const float4*>(red_o + ((size_t)k * rows_cta + r) * C::kRedStride + c4 * 4);
                acc.x += w * v.x;
                acc.y += w * v.y;
                acc.z += w * v.z;
                acc.w += w * v.w;
            }
            const float inv = 1.f / L;
            acc.x *= inv;
            acc.y *= inv;
            acc.z *= inv;
            acc.w *= inv;
        }
        const int qi = r / G, hh = r % G;
        const int t = q0 + qi, h = g * G + hh;
        if (!partial) {
            const size_t oo = (size_t)t * p.o_st + (size_t)h * p.o_sh + c4 * 4;
            if (p.out_f32) {
                *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + oo) = acc;
            } else {
                uint2 pk;
                pk.x = pack_bf16(acc.x, acc.y);
                pk.y = pack_bf16(acc.z, acc.w);
                *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.out) + oo) = pk;
            }
        } else {
            const size_t row = ((size_t)split * p.T + t) * p.H + h;
            *reinterpret_cast<float4*>(p.ws_o + row * D + c4 * 4) = acc;
            if (c4 == 0) p.ws_lse[row] = M == -CUDART_INF_F ? -CUDART_INF_F : M + __log2f(L);
        }
    }
}

template <int D, int MT, int KSL>
int decode_smem_bytes(int nstage) {
    using C = DecodeCfg<D, MT, KSL>;
    int body = nstage * C::kStageBytes;
    if (body < C::kRedBytes) body = C::kRedBytes;
    return 1024 + body + 2 * C::kMaxStages * 8 + 16;
}

template <int D, int MT, int KSL>
int pick_nstage(int ctas, int num_sms) {
    using C = DecodeCfg<D, MT, KSL>;
    // One CTA per SM when the grid fits in one wave, else two per SM.
    const int budget = (ctas <= num_sms) ? 200 * 1024 : 100 * 1024;
    int n = budget / C::kStageBytes;
    if (n > C::kMaxStages) n = C::kMaxStages;
    if (n < 2) n = 2;
    return n;
}

template <int D, int MT, int KSL>
cudaError_t launch_t(const AttnParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, const LaunchShape& s,
                     cudaStream_t stream) {
    auto kern = decode_kernel<D, MT, KSL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s.smem);
    if (e != cudaSuccess) return e;
    kern<<<s.grid, s.block, s.smem, stream>>>(tmK, tmV, p);
    return cudaGetLastError();
}

void tile_choice(int rows, int& mt, int& ksl) {
    if (rows <= 16) {
        mt = 1;
        ksl = 4;
    } else if (rows <= 32) {
        mt = 2;
        ksl = 4;
    } else {
        mt = 4;
        ksl = 2;
    }
}

}  // namespace

LaunchShape decode_shape(const AttnParams& p, int num_sms) {
    LaunchShape s;
    int mt, ksl;
    tile_choice(p.max_rows, mt, ksl);
    s.grid = dim3(p.num_splits, p.Hk, p.B);
    s.block = (mt * ksl + 1) * 32;
    const int ctas = p.num_splits * p.Hk * p.B;
    int nst = 2;
#define REL_ATTN_SHAPE(DD, M, K)                         \
    if (p.D == DD && mt == M && ksl == K) {             \
        nst = pick_nstage<DD, M, K>(ctas, num_sms);     \
        s.smem = decode_smem_bytes<DD, M, K>(nst);      \
    }
    REL_ATTN_SHAPE(64, 1, 4)
    REL_ATTN_SHAPE(64, 2, 4)
    REL_ATTN_SHAPE(64, 4, 2)
    REL_ATTN_SHAPE(128, 1, 4)
    REL_ATTN_SHAPE(128, 2, 4)
    REL_ATTN_SHAPE(128, 4, 2)
#undef REL_ATTN_SHAPE
    s.nstage = nst;
    return s;
}

cudaError_t launch_decode(const AttnParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const LaunchShape& s, cudaStream_t stream) {
    int mt, ksl;
    tile_choice(p.max_rows, mt, ksl);
#define REL_ATTN_LAUNCH(DD, M, K) \
    if (p.D == DD && mt == M && ksl == K) return launch_t<DD, M, K>(p, tmK, tmV, s, stream);
    REL_ATTN_LAUNCH(64, 1, 4)
    REL_ATTN_LAUNCH(64, 2, 4)
    REL_ATTN_LAUNCH(64, 4, 2)
    REL_ATTN_LAUNCH(128, 1, 4)
    REL_ATTN_LAUNCH(128, 2, 4)
    REL_ATTN_LAUNCH(128, 4, 2)
#undef REL_ATTN_LAUNCH
    return cudaErrorInvalidValue;
}

}  // namespace relattn
