// Prefill / chunked-prefill kernel on the 5th-generation tensor cores.
//
// One CTA per (128-row query tile, kv head, request, split).  Rows are
// GQA-packed token-major: row r of the tile is query token i0 + r / G of
// request b and query head g*G + r % G, so every K/V tile read for kv head g
// serves all G query heads.  The visible key range of the tile is cut into
// 128-key tiles, processed from the last to the first (the causal diagonal
// and the bias band come first, so the running maximum settles early).
//
// Warp roles (256 threads):
//   warps 0-2  producers: gather Q once and each K / V tile from the paged
//              cache with 16-byte cp.async (one block-table lookup per key,
//              zero-fill outside the visible range) into 128-byte-swizzled
//              K-major tiles; after their copies land they fence the async
//              proxy and arrive on the tile's full mbarrier.
//   warp 3     MMA issuer (one thread) and TMEM owner: S_j = Q K_j^T into one
//              of two TMEM buffers (M=128, N=128, K=head_dim), then
//              O += P_{j-1} V_{j-1} (P from shared memory, V read MN-major)
//              into a TMEM accumulator; tcgen05.commit signals completion.
//   warps 4-7  softmax: thread r owns row r (TMEM lane r).  It reads S_j,
//              applies scale, the sheared relative bias and the mask, keeps
//              the fp32 online softmax (base 2), writes P_j as bf16, rescales
//              its O row in TMEM when its maximum grew, and writes the output.
// Every mbarrier wait is bounded; on timeout the kernel records the site in
// the device error word and winds down.
//
// Semantics: vLLM API docs, inkling_fa4_rel_attention (paged varlen forward);
// bias rule: prhub report on vLLM PR #48858, score_mod_rel_bias.

#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace relattn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct PrefillCfg {
    static constexpr int BN = 128;  // keys per tile (query tiles are 128 rows)
    static constexpr int kDB = D / 64;              // 64-dim (128-byte) column blocks
    static constexpr int kBlk = 128 * 128;          // one 128-row x 128-byte block
    static constexpr int kTileBytes = kDB * kBlk;   // a Q, K or V tile
    static constexpr int kPBytes = 2 * kBlk;        // P: 128 rows x 128 keys, bf16
    static constexpr int kProdThreads = 96;         // warps 0-2
    static constexpr int kMmaWarp = 3;
    static constexpr int kStages = D == 128 ? 4 : 6;  // K/V ring slots (K even, V odd sequence numbers)
    static constexpr int kLag = 2;                    // copy groups in flight per producer thread
    static constexpr int kData = kTileBytes + kStages * kTileBytes + 2 * kPBytes;
    static constexpr int kTmemCols = 512;
    static constexpr int kOCol = 256;
};

struct PrefillBars {
    uint64_t q_full;
    uint64_t kv_full[8];
    uint64_t kv_empty[8];
    uint64_t s_full[2];
    uint64_t s_empty[2];
    uint64_t p_full[2];
    uint64_t p_free[2];
    uint64_t o_done;   // one phase per PV tile (rescale waits, never more than one phase behind)
    uint64_t o_final;  // single phase: every MMA of the CTA has completed
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ bool aborted(const PrefillBars* bars) {
    return *reinterpret_cast<const volatile int*>(&bars->abort) != 0;
}

template <int D>
__global__ void __launch_bounds__(256, 1) prefill_kernel(const AttnParams p) {
    using C = PrefillCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sKV = smem + C::kTileBytes;
    uint8_t* sP = sKV + C::kStages * C::kTileBytes;
    PrefillBars* bars = reinterpret_cast<PrefillBars*>(sP + 2 * C::kPBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G, TPT = 128 / G;
    const int qt = gridDim.x - 1 - blockIdx.x;  // longest tiles first
    const int g = blockIdx.y;
    const int S = p.num_splits;
    const int b = blockIdx.z / S, split = blockIdx.z % S;
    const int q0 = p.cu_seqlens_q[b];
    const int sq = p.cu_seqlens_q[b + 1] - q0;
    const int sk = p.cache_seqlens[b];
    const int i0 = qt * TPT;
    if (i0 >= sq) return;  // CTA-uniform, before any barrier
    const int i1 = min(sq, i0 + TPT);
    const int n_rows = (i1 - i0) * G;
    const int off = sk - sq;
    const int pos_min = i0 + off, pos_max = i1 - 1 + off;

    // Keys any row of the tile may see, as 128-key tiles, split contiguously.
    int hi = sk;
    if (p.causal) hi = min(hi, pos_max + 1);
    if (p.wr >= 0) hi = min(hi, pos_max + p.wr + 1);
    int lo = 0;
    if (p.wl >= 0) lo = max(0, pos_min - p.wl);
    int kb_first = 0, n_tiles = 0;
    if (hi > lo) {
        kb_first = lo / C::BN;
        n_tiles = (hi - 1) / C::BN - kb_first + 1;
    }
    const int s_eff = min(S, n_tiles);
    int t_begin = 0, t_end = 0;
    if (split < s_eff) {
        t_begin = (int)(((long long)split * n_tiles) / s_eff);
        t_end = (int)(((long long)(split + 1) * n_tiles) / s_eff);
    }
    const int n_it = t_end - t_begin;
    auto key_block = [&](int jj) { return kb_first + t_end - 1 - jj; };  // last tile first

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, C::kProdThreads);
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&bars->kv_full[i], C::kProdThreads);
            mbar_init(&bars->kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->s_empty[i], 128);
            mbar_init(&bars->p_full[i], 128);
            mbar_init(&bars->p_free[i], 1);
        }
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->o_final, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == C::kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars->tmem_base)),
                     "n"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp < 3) {
        // ------------------------------------------------------------ producers
        const int pt = threadIdx.x;
        const uint16_t* qg = reinterpret_cast<const uint16_t*>(p.q);
        const uint16_t* kc = reinterpret_cast<const uint16_t*>(p.k_cache);
        const uint16_t* vc = reinterpret_cast<const uint16_t*>(p.v_cache);
        const int32_t* bt = p.block_table + (size_t)b * p.bt_stride;
        const uint64_t pol_first = l2_policy_evict_first();
        const uint64_t pol_last = l2_policy_evict_last();
        constexpr int kChunks = C::kDB * 8;  // 16-byte chunks per 128-row tile row
        int issued = 0, done = 0;
        auto complete = [&](int k) {  // copy group k of this thread has landed
            fence_proxy_async_smem();
            if (k == 0)
                mbar_arrive(&bars->q_full);
            else
                mbar_arrive(&bars->kv_full[(k - 1) % C::kStages]);
        };
        // Q tile (group 0)
        for (int idx = pt; idx < 128 * kChunks; idx += C::kProdThreads) {
            const int r = idx / kChunks, c = idx % kChunks;
            const bool valid = r < n_rows;
            const int tok = i0 + r / G, hh = r % G;
            const uint16_t* src = qg + (size_t)(q0 + tok) * p.q_st + (size_t)(g * G + hh) * p.q_sh + c * 8;
            const uint32_t dst = smem_u32(sQ) + (c >> 3) * C::kBlk + sw128_offset(r, c & 7);
            cp_async_16(dst, valid ? src : qg, valid ? 16u : 0u, pol_first);
        }
        cp_async_commit();
        ++issued;
        for (int seq = 0; seq < 2 * n_it; ++seq) {
            const int slot = seq % C::kStages;
            const int round = seq / C::kStages;
            if (!mbar_wait(&bars->kv_empty[slot], (round & 1) ^ 1, p.timeout_ns, kSitePrefillKEmpty, p.err)) {
                bars->abort = 1;
                break;
            }
            if (aborted(bars)) break;
            const int j0 = key_block(seq >> 1) * C::BN;
            const uint16_t* cache = (seq & 1) ? vc : kc;
            const uint32_t dst0 = smem_u32(sKV + slot * C::kTileBytes);
            for (int idx = pt; idx < 128 * kChunks; idx += C::kProdThreads) {
                const int r = idx / kChunks, c = idx % kChunks;
                const int j = j0 + r;
                const bool valid = j >= lo && j < hi;
                const int n = j / p.BS;
                int blk = valid ? __ldg(bt + n) : 0;
                blk = min(max(blk, 0), p.NB - 1);  // an out-of-range id stays inside the cache
                const uint16_t* src =
                    cache + (size_t)blk * p.c_s0 + (size_t)(j - n * p.BS) * p.c_s1 + (size_t)g * p.c_s2 + c * 8;
                const uint32_t dst = dst0 + (c >> 3) * C::kBlk + sw128_offset(r, c & 7);
                cp_async_16(dst, valid ? src : cache, valid ? 16u : 0u, pol_last);
            }
            cp_async_commit();
            ++issued;
            if (issued - done > C::kLag) {
                cp_async_wait(C::kLag);
                complete(done++);
            }
        }
        while (done < issued) {
            cp_async_wait(issued - done - 1);
            complete(done++);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_it > 0) {
            constexpr uint32_t idS = umma_idesc_bf16(128, C::BN, false);
            constexpr uint32_t idPV = umma_idesc_bf16(128, D, true);
            const uint32_t aQ = smem_u32(sQ), aKV = smem_u32(sKV), aP = smem_u32(sP);
            bool ok = mbar_wait(&bars->q_full, 0, p.timeout_ns, kSitePrefillLoadQ, p.err);
            auto issue_pv = [&](int t) {
                const int pb = t & 1;
                const int seq = 2 * t + 1;
                const int slot = seq % C::kStages;
                ok = ok && mbar_wait(&bars->p_full[pb], (t >> 1) & 1, p.timeout_ns, kSitePrefillPFull, p.err);
                ok = ok && mbar_wait(&bars->kv_full[slot], (seq / C::kStages) & 1, p.timeout_ns, kSitePrefillVFull,
                                     p.err);
                if (!ok) return;
                tc_fence_after();
                const uint32_t pbase = aP + pb * C::kPBytes;
                const uint32_t vbase = aKV + slot * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk) {
                    const uint64_t da = umma_desc_sw128(pbase + (kk >> 2) * C::kBlk + (kk & 3) * 32, 16, 1024);
                    const uint64_t db = umma_desc_sw128(vbase + kk * 16 * 128, C::kBlk, 1024);
                    umma_bf16(tmem + C::kOCol, da, db, idPV, (t > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(&bars->o_done);
                umma_commit(&bars->kv_empty[slot]);
                umma_commit(&bars->p_free[pb]);
            };
            for (int jj = 0; jj < n_it && ok; ++jj) {
                const int sb = jj & 1;
                const int seq = 2 * jj;
                const int slot = seq % C::kStages;
                ok = ok && mbar_wait(&bars->kv_full[slot], (seq / C::kStages) & 1, p.timeout_ns, kSitePrefillKFull,
                                     p.err);
                ok = ok && mbar_wait(&bars->s_empty[sb], ((jj >> 1) & 1) ^ 1, p.timeout_ns, kSitePrefillSEmpty,
                                     p.err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t kbase = aKV + slot * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t da = umma_desc_sw128(aQ + (kk >> 2) * C::kBlk + (kk & 3) * 32, 16, 1024);
                    const uint64_t db = umma_desc_sw128(kbase + (kk >> 2) * C::kBlk + (kk & 3) * 32, 16, 1024);
                    umma_bf16(tmem + sb * C::BN, da, db, idS, kk > 0 ? 1u : 0u);
                }
                umma_commit(&bars->s_full[sb]);
                umma_commit(&bars->kv_empty[slot]);
                if (jj >= 1) issue_pv(jj - 1);
            }
            if (ok) issue_pv(n_it - 1);
            // The epilogue may be two or more o_done phases behind, where a
            // parity wait cannot tell phases apart: give it its own barrier.
            umma_commit(&bars->o_final);
            if (!ok) bars->abort = 1;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int r = threadIdx.x - 128;  // row == TMEM lane
        const bool valid = r < n_rows;
        const int tok = i0 + (valid ? r / G : 0);
        const int hh = valid ? r % G : 0;
        const int t = q0 + tok, h = g * G + hh;
        const int pos = tok + off;
        const uint16_t* relrow =
            p.R > 0 ? reinterpret_cast<const uint16_t*>(p.rel) + ((size_t)t * p.H + h) * p.R : nullptr;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float sl2 = p.scale_log2;
        const int R = p.R, wl = p.wl, wr = p.wr, causal = p.causal;
        float m_run = -CUDART_INF_F, l_run = 0.f;
        const uint32_t aP = smem_u32(sP);

        for (int jj = 0; jj < n_it; ++jj) {
            const int sb = jj & 1;
            const int j0 = key_block(jj) * C::BN;
            if (!mbar_wait(&bars->s_full[sb], (jj >> 1) & 1, p.timeout_ns, kSitePrefillSFull, p.err)) {
                bars->abort = 1;
            }
            if (__any_sync(0xffffffffu, aborted(bars))) break;  // warp-uniform: TMEM access is collective
            tc_fence_after();
            float s[C::BN];
#pragma unroll
            for (int c = 0; c < C::BN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(lane_base + sb * C::BN + c * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(v[e]);
            }
            tc_fence_before();
            mbar_arrive(&bars->s_empty[sb]);

            // Scale, sheared bias, mask.  Fast path: the whole key tile is
            // visible to this row and out of its bias band.
            const bool all_visible = !valid || ((j0 + C::BN <= sk) && (!causal || pos - (j0 + C::BN - 1) >= 0) &&
                                                (wl < 0 || pos - j0 <= wl) && (wr < 0 || pos - (j0 + C::BN - 1) >= -wr));
            const bool no_bias = !valid || R == 0 || pos - (j0 + C::BN - 1) >= R || pos - j0 < 0;
            float mx = -CUDART_INF_F;
            if (all_visible && no_bias) {
#pragma unroll
                for (int k = 0; k < C::BN; ++k) {
                    s[k] *= sl2;
                    mx = fmaxf(mx, s[k]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < C::BN; ++k) {
                    const int j = j0 + k;
                    const int d = pos - j;
                    bool allowed = j < sk;
                    if (causal) allowed = allowed && d >= 0;
                    if (wl >= 0) allowed = allowed && d <= wl;
                    if (wr >= 0) allowed = allowed && d >= -wr;
                    float bias = 0.f;
                    if (allowed && d >= 0 && d < R) bias = bf16_bits_to_f32(__ldg(relrow + d));
                    s[k] = allowed ? fmaf(s[k], sl2, bias * kLog2e) : -CUDART_INF_F;
                    mx = fmaxf(mx, s[k]);
                }
            }
            const float m_new = fmaxf(m_run, mx);
            const float mu = m_new == -CUDART_INF_F ? 0.f : m_new;
            const bool grow = m_run != -CUDART_INF_F && m_new > m_run;
            const float alpha = grow ? ex2(m_run - m_new) : 1.f;

            // P_j into shared buffer jj % 2 once PV_{j-2} has read it.
            if (!mbar_wait(&bars->p_free[sb], ((jj >> 1) & 1) ^ 1, p.timeout_ns, kSitePrefillPFull, p.err))
                bars->abort = 1;
            float rs = 0.f;
            const uint32_t prow = aP + sb * C::kPBytes;
#pragma unroll
            for (int c = 0; c < C::BN / 8; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = ex2(s[c * 8 + 2 * e] - mu), bq = ex2(s[c * 8 + 2 * e + 1] - mu);
                    rs += a + bq;
                    w[e] = pack_bf16(a, bq);
                }
                const uint32_t addr = prow + (c >> 3) * C::kBlk + sw128_offset(r, c & 7);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                             "r"(w[3])
                             : "memory");
            }
            l_run = l_run * alpha + rs;
            m_run = m_new;

            // Rescale the O row when its maximum grew (warp-collective TMEM access).
            if (jj >= 1 && __any_sync(0xffffffffu, grow)) {
                if (!mbar_wait(&bars->o_done, (jj - 1) & 1, p.timeout_ns, kSitePrefillOFull, p.err)) bars->abort = 1;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + C::kOCol + c * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tmem_st32(lane_base + C::kOCol + c * 32, v);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();  // P stores -> visible to the tensor core
            tc_fence_before();
            mbar_arrive(&bars->p_full[sb]);
        }

        // Epilogue: O / l.
        const bool have = __all_sync(0xffffffffu, n_it > 0 && !aborted(bars));
        if (have) {
            if (!mbar_wait(&bars->o_final, 0, p.timeout_ns, kSitePrefillOFull, p.err)) bars->abort = 1;
            tc_fence_after();
        }
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
        const bool partial = p.num_splits > 1;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            if (have) {
                tmem_ld32(lane_base + C::kOCol + c * 32, v);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
            if (!valid) continue;
            float o[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(v[e]) * inv_l;
            if (partial) {
                float* dst = p.ws_o + (((size_t)split * p.T + t) * p.H + h) * D + c * 32;
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
            } else if (p.out_f32) {
                float* dst = reinterpret_cast<float*>(p.out) + (size_t)t * p.o_st + (size_t)h * p.o_sh + c * 32;
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
            } else {
                uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + (size_t)t * p.o_st + (size_t)h * p.o_sh + c * 32;
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint4 pk;
                    pk.x = pack_bf16(o[e], o[e + 1]);
                    pk.y = pack_bf16(o[e + 2], o[e + 3]);
                    pk.z = pack_bf16(o[e + 4], o[e + 5]);
                    pk.w = pack_bf16(o[e + 6], o[e + 7]);
                    *reinterpret_cast<uint4*>(dst + e) = pk;
                }
            }
        }
        if (valid && partial)
            p.ws_lse[((size_t)split * p.T + t) * p.H + h] = l_run > 0.f ? m_run + __log2f(l_run) : -CUDART_INF_F;
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(C::kTmemCols)
                     : "memory");
}

template <int D>
int prefill_smem_bytes() {
    return 1024 + PrefillCfg<D>::kData + (int)sizeof(PrefillBars);
}

template <int D>
cudaError_t launch_t(const AttnParams& p, const LaunchShape& s, cudaStream_t stream) {
    auto kern = prefill_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s.smem);
    if (e != cudaSuccess) return e;
    kern<<<s.grid, s.block, s.smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

LaunchShape prefill_shape(const AttnParams& p) {
    LaunchShape s;
    const int tpt = 128 / p.G;
    const int qtiles = (p.max_seqlen_q + tpt - 1) / tpt;
    s.grid = dim3(qtiles, p.Hk, p.B * p.num_splits);
    s.block = 256;
    s.smem = p.D == 128 ? prefill_smem_bytes<128>() : prefill_smem_bytes<64>();
    s.nstage = p.D == 128 ? PrefillCfg<128>::kStages : PrefillCfg<64>::kStages;
    return s;
}

cudaError_t launch_prefill(const AttnParams& p, const LaunchShape& s, cudaStream_t stream) {
    if (p.D == 128) return launch_t<128>(p, s, stream);
    if (p.D == 64) return launch_t<64>(p, s, stream);
    return cudaErrorInvalidValue;
}

}  // namespace relattn
