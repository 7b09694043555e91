// Split-KV decode kernel: one CTA per (split, kv head, request) over at most
// 64 GQA-packed query rows (query token i, head g*G + r packed as row i*G + r),
// so every K/V byte of a kv head is read from HBM once per split.
//
// The CTA's key range (this split's share of the request's visible keys) is
// cut into stages of 16*KSL keys.  Producer warps gather each stage from
// the paged cache with 16-byte cp.async (one block-table lookup per 16-key
// page slice, keys past the visible range zero-filled) into a ring of NSTAGE
// slots whose rows are padded by 16 bytes, so the ldmatrix reads are
// conflict-free; completion is signalled on the slot's mbarrier by
// cp.async.mbarrier.arrive.  KSL x MT consumer warps (x 2 with head_dim 256,
// one per dim half, adding their partial scores through shared memory) each
// take one 16-key slice of a stage and one 16-row tile: QK^T and PV on bf16 mma.sync with
// fp32 accumulation, the scale, the sheared relative bias and the mask per
// element (skipped for slices wholly visible and outside the bias band), and
// an fp32 online softmax in base 2; then they release the slot.  The
// consumers' (m, l, O) merge through shared memory at the end.  With one
// split the result is written directly (bf16 or fp32); otherwise the
// normalised fp32 partial and its log2-sum-exp go to the workspace for the
// combine kernel.  Every mbarrier wait is bounded.
//
// Semantics: vLLM API docs, inkling_fa4_rel_attention (paged varlen forward);
// bias rule: prhub report on vLLM PR #48858, score_mod_rel_bias.

#include <math_constants.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace relattn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D, int MT, int KSL>
struct DecodeCfg {
    // head_dim 256: each 16-key slice goes to a pair of warps, each owning
    // half of the dims (a 16-row fragment of 256 fp32 accumulators per lane
    // would not fit in registers); they add their partial scores through
    // shared memory, so both hold the same softmax state.
    static constexpr int DS = D == 256 ? 2 : 1;       // dim halves per slice
    static constexpr int DW = D / DS;                 // dims one warp owns
    static constexpr int kConsumers = MT * KSL * DS;
    static constexpr int kMaxProducers = 4;
    static constexpr int kMaxThreads = (kConsumers + kMaxProducers) * 32;
    static constexpr int kStageKeys = 16 * KSL;
    // A stage holds kStageKeys K rows then as many V rows; each row is padded
    // by 16 bytes so the 8 rows an ldmatrix reads fall in distinct banks.
    static constexpr int kRowBytes = D * 2 + 16;
    static constexpr int kOperandBytes = kStageKeys * kRowBytes;
    static constexpr int kStageBytes = 2 * kOperandBytes;
    static constexpr int kChunks = D / 8;            // 16-byte chunks per key row
    static constexpr int kRowsPerCopy = 32 / kChunks;  // rows one warp-wide copy covers
    static constexpr int kRedStride = D + 4;         // floats per row in the merge area
    static constexpr int kRedBytes = KSL * MT * 16 * (kRedStride + 2) * 4;
    static constexpr int kMaxStages = 12;
    // Partial-score exchange (DS == 2): per warp pair, two tile-parity
    // buffers of 32 lanes x 8 floats per warp, and two mbarriers.
    static constexpr int kPairs = DS == 2 ? MT * KSL : 0;
    static constexpr int kXchBytes = kPairs * 2 * 2 * 32 * 8 * 4;
};

constexpr int kRankMax = 256;

__device__ __forceinline__ float bias_to_f32(uint16_t b) { return bf16_bits_to_f32(b); }
__device__ __forceinline__ float bias_to_f32(float b) { return b; }

// BF32: rel_logits are fp32 (else bf16).
template <int D, int MT, int KSL, bool BF32>
__global__ void __launch_bounds__(DecodeCfg<D, MT, KSL>::kMaxThreads) decode_kernel(const AttnParams p) {
    using C = DecodeCfg<D, MT, KSL>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int NST = p.nstage;
    const size_t body = (size_t)NST * C::kStageBytes > (size_t)C::kRedBytes ? (size_t)NST * C::kStageBytes
                                                                             : (size_t)C::kRedBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + body);
    uint64_t* empty = full + C::kMaxStages;
    uint64_t* xbar = empty + C::kMaxStages;  // [pair][tile parity], C::kPairs * 2
    int* abort_flag = reinterpret_cast<int*>(xbar + 2 * C::kPairs);
    float* xch = reinterpret_cast<float*>(abort_flag + 4);  // [pair][parity][dim half][32 lanes][8]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, g = blockIdx.y;
    const int G = p.G;

    // Longest requests first: grid index z takes the request of rank z in
    // decreasing cache length (ties by index), so the longest streams start
    // in the first wave and the short ones fill in behind them.  Ranking costs
    // B^2 comparisons per CTA, so only batches of up to kRankMax requests.
    int b = blockIdx.z;
    if (p.B > 1 && p.B <= kRankMax) {
        int* chosen = abort_flag + 1;
        const int target = blockIdx.z;
        for (int c = threadIdx.x; c < p.B; c += blockDim.x) {
            const int lc = p.cache_seqlens[c];
            int rank = 0;
            for (int o = 0; o < p.B; ++o) {
                const int lo_ = p.cache_seqlens[o];
                rank += (lo_ > lc) || (lo_ == lc && o < c);
            }
            if (rank == target) *chosen = c;
        }
        __syncthreads();
        b = *chosen;
    }

    const int q0 = p.cu_seqlens_q[b];
    const int sq = p.cu_seqlens_q[b + 1] - q0;
    const int sk = p.cache_seqlens[b];
    const int n_rows = min(sq * G, p.max_rows);
    if (n_rows <= 0) return;
    const int off = sk - sq;

    // Keys any row of this request may see, cut into stages and split.
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
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 32 * p.nprod);     // one arrival per producer lane
            mbar_init(&empty[i], C::kConsumers);  // one arrival per consumer warp
        }
        for (int i = 0; i < 2 * C::kPairs; ++i) mbar_init(&xbar[i], 2);  // both warps of the pair
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp >= C::kConsumers) {
        // ----------------------------------------------------------- producers
        // Producer warp pw gathers pages pw, pw + nprod, ... of every stage.
        const int pw = warp - C::kConsumers, nprod = p.nprod;
        const uint16_t* kc = reinterpret_cast<const uint16_t*>(p.k_cache);
        const uint16_t* vc = reinterpret_cast<const uint16_t*>(p.v_cache);
        const int32_t* bt = p.block_table + (size_t)b * p.bt_stride;
        const int nblk = min((khi + p.BS - 1) / p.BS, p.max_blocks);
        const uint64_t policy = l2_policy_evict_first();
        // This lane copies 16-byte chunk `cchunk` of rows crow, crow + kRowsPerCopy, ...
        const int crow = lane / C::kChunks, cchunk = lane % C::kChunks;
        const size_t lane_off = (size_t)crow * p.c_s1 + cchunk * 8 + (size_t)g * p.c_s2;
        const uint32_t lane_dst = crow * C::kRowBytes + cchunk * 16;
        int cached_base = -(1 << 30);
        int my_blk = 0;
        for (int it = 0; it < n_it; ++it) {
            const int slot = it % NST;
            const int round = it / NST;
            bool ok = true;
            if (lane == 0) ok = mbar_wait(&empty[slot], (round & 1) ^ 1, p.timeout_ns, kSiteDecodeEmpty, p.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const int k0 = kstart + (t_begin + it) * BN;
            const uint32_t dst_stage = smem_u32(smem + (size_t)slot * C::kStageBytes) + lane_dst;
            for (int pg = pw; pg < KSL; pg += nprod) {
                const int j0 = k0 + 16 * pg;
                const int n = j0 / p.BS;
                if (n - cached_base >= 32 || n < cached_base) {  // warp-uniform
                    cached_base = n;
                    my_blk = (n + lane < nblk) ? __ldg(bt + n + lane) : 0;
                }
                // A block id outside [0, NB) breaks the caller's contract; clamp
                // it so the gather stays inside the cache instead of faulting.
                const int blk = min(max(__shfl_sync(0xffffffffu, my_blk, n - cached_base), 0), p.NB - 1);
                const size_t page = (size_t)blk * p.c_s0 + (size_t)(j0 - n * p.BS) * p.c_s1 + lane_off;
                const bool full_pg = j0 + 16 <= khi;
#pragma unroll
                for (int r = 0; r < 16 / C::kRowsPerCopy; ++r) {
                    const int row = r * C::kRowsPerCopy;  // + crow
                    const bool okr = full_pg || j0 + row + crow < khi;
                    const size_t src = page + (size_t)row * p.c_s1;
                    const uint32_t dst = dst_stage + (16 * pg + row) * C::kRowBytes;
                    cp_async_16(dst, okr ? kc + src : kc, okr ? 16u : 0u, policy);
                    cp_async_16(dst + C::kOperandBytes, okr ? vc + src : vc, okr ? 16u : 0u, policy);
                }
            }
            cp_async_arrive_noinc(&full[slot]);
        }
        cp_async_wait(0);
        return;
    }

    // ---------------------------------------------------------------- consumers
    // row tile, 16-key slice of each stage, dim half (head_dim 256)
    const int mt = warp % MT, ks = (warp / MT) % KSL, dh = warp / (MT * KSL);

    // ------------------------------------------------------------- rows
    const int gq = lane >> 2, tig = lane & 3;
    const int r0 = mt * 16 + gq, r1 = r0 + 8;
    const bool valid0 = r0 < n_rows, valid1 = r1 < n_rows;
    const int qi0 = valid0 ? r0 / G : 0, qi1 = valid1 ? r1 / G : 0;
    const int pos0 = qi0 + off, pos1 = qi1 + off;  // key positions of the two rows
    const int h0 = g * G + (valid0 ? r0 % G : 0), h1 = g * G + (valid1 ? r1 % G : 0);
    // The two rows' rel_logits (bf16 bits or fp32 values).
    using BiasT = typename std::conditional<BF32, float, uint16_t>::type;
    const BiasT* rel0 = nullptr;
    const BiasT* rel1 = nullptr;
    if (p.R > 0) {
        rel0 = reinterpret_cast<const BiasT*>(p.rel) + ((size_t)(q0 + qi0) * p.H + h0) * p.R;
        rel1 = reinterpret_cast<const BiasT*>(p.rel) + ((size_t)(q0 + qi1) * p.H + h1) * p.R;
    }
    // Extreme key positions over the CTA's valid rows (rows are token-major).
    const int pos_lo = off, pos_hi = (n_rows - 1) / G + off;

    // Q fragments (A operand, rows x this warp's dims), loaded once.
    uint32_t qf[C::DW / 16][4];
    {
        const uint16_t* qb = reinterpret_cast<const uint16_t*>(p.q);
        const uint32_t* rowp0 =
            reinterpret_cast<const uint32_t*>(qb + (size_t)(q0 + qi0) * p.q_st + (size_t)h0 * p.q_sh);
        const uint32_t* rowp1 =
            reinterpret_cast<const uint32_t*>(qb + (size_t)(q0 + qi1) * p.q_st + (size_t)h1 * p.q_sh);
        const int w0 = dh * (C::DW / 2);  // first 32-bit word of this warp's dims
#pragma unroll
        for (int kk = 0; kk < C::DW / 16; ++kk) {
            qf[kk][0] = valid0 ? __ldg(rowp0 + w0 + kk * 8 + tig) : 0u;
            qf[kk][1] = valid1 ? __ldg(rowp1 + w0 + kk * 8 + tig) : 0u;
            qf[kk][2] = valid0 ? __ldg(rowp0 + w0 + kk * 8 + 4 + tig) : 0u;
            qf[kk][3] = valid1 ? __ldg(rowp1 + w0 + kk * 8 + 4 + tig) : 0u;
        }
    }

    float o[C::DW / 8][4];
#pragma unroll
    for (int a = 0; a < C::DW / 8; ++a) o[a][0] = o[a][1] = o[a][2] = o[a][3] = 0.f;
    // m_run: reference maximum of each row, an integer in log2 units (the
    // ceiling of the running maximum; see kQuantC: weights then do not
    // depend on the split partition).  O and l are rescaled, by an exact
    // power of two, only in slices where some row of the warp exceeded it.
    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
    float l_run[2] = {0.f, 0.f};
    const float sl2 = p.scale_log2;
    const int R = p.R, wl = p.wl, wr = p.wr, causal = p.causal;

    for (int it = 0; it < n_it; ++it) {
        const int slot = it % NST;
        const int round = it / NST;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&full[slot], round & 1, p.timeout_ns, kSiteDecodeFull, p.err);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0) *abort_flag = 1;
            break;
        }
        const uint8_t* kbuf = smem + (size_t)slot * C::kStageBytes + ks * 16 * C::kRowBytes;
        const uint8_t* vbuf = kbuf + C::kOperandBytes;
        const int jb = kstart + (t_begin + it) * BN + ks * 16;  // this warp's first key

        // S = Q K^T over the slice: two n-tiles of 8 keys, each accumulated in
        // two halves of the head dim to shorten the MMA chains.
        float sacc[2][4], sacc2[2][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[a][e] = sacc2[a][e] = 0.f;
        {
            const int krow = (lane >> 4) * 8 + (lane & 7);
            const int csel = (lane >> 3) & 1;
            const uint32_t kb = smem_u32(kbuf) + krow * C::kRowBytes + csel * 16 + dh * C::DW * 2;
#pragma unroll
            for (int kk = 0; kk < C::DW / 16; ++kk) {
                const uint32_t addr = kb + kk * 32;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(addr, b0, b1, b2, b3);
                if (kk & 1) {
                    mma_bf16_16816(sacc2[0], qf[kk], b0, b1);
                    mma_bf16_16816(sacc2[1], qf[kk], b2, b3);
                } else {
                    mma_bf16_16816(sacc[0], qf[kk], b0, b1);
                    mma_bf16_16816(sacc[1], qf[kk], b2, b3);
                }
            }
        }

        if constexpr (C::DS == 2) {
            // Add the partner warp's partial scores (its half of the dims).
            // Both warps form partial + partial in IEEE arithmetic, which is
            // commutative, so they hold bit-identical scores.
            const int pair = mt + MT * ks, par = it & 1;
            float* mine = xch + (((pair * 2 + par) * 2 + dh) * 32 + lane) * 8;
            const float* theirs = xch + (((pair * 2 + par) * 2 + (dh ^ 1)) * 32 + lane) * 8;
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int e = 0; e < 4; ++e) mine[a * 4 + e] = sacc[a][e] + sacc2[a][e];
            __syncwarp();
            if (lane == 0) mbar_arrive(&xbar[pair * 2 + par]);
            const bool xok = mbar_wait(&xbar[pair * 2 + par], (uint32_t)((it >> 1) & 1), p.timeout_ns,
                                       kSiteDecodeFull, p.err);
            if (!__all_sync(0xffffffffu, xok)) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    sacc[a][e] = mine[a * 4 + e] + theirs[a * 4 + e];
                    sacc2[a][e] = 0.f;
                }
        }

        // Scale, sheared bias, mask.  Warp-uniform fast path: every key of the
        // slice is visible to every row and no row's distance reaches the band.
        const bool all_visible = jb + 16 <= khi && (!causal || jb + 15 <= pos_lo) &&
                                 (wl < 0 || jb >= pos_hi - wl) && (wr < 0 || jb + 15 <= pos_lo + wr);
        const bool no_bias = R == 0 || pos_lo - (jb + 15) >= R || pos_hi - jb < 0;
        float s[2][4];
        if (all_visible && no_bias) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] = (sacc[nt][e] + sacc2[nt][e]) * sl2;
        } else {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const bool second = e >> 1;
                    const int pos = second ? pos1 : pos0;
                    const BiasT* relr = second ? rel1 : rel0;
                    const int j = jb + nt * 8 + 2 * tig + (e & 1);
                    const int d = pos - j;
                    bool allowed = (second ? valid1 : valid0) && j < khi;
                    if (causal) allowed = allowed && d >= 0;
                    if (wl >= 0) allowed = allowed && d <= wl;
                    if (wr >= 0) allowed = allowed && d >= -wr;
                    float bias = 0.f;
                    if (allowed && d >= 0 && d < R) bias = bias_to_f32(__ldg(relr + d));
                    s[nt][e] = allowed ? fmaf(sacc[nt][e] + sacc2[nt][e], sl2, bias * kLog2e) : -CUDART_INF_F;
                }
            }
        }

        // Online softmax (base 2).  Rows gq (e = 0,1) and gq + 8 (e = 2,3).
        float mx[2];
#pragma unroll
        for (int rsel = 0; rsel < 2; ++rsel) {
            float v = fmaxf(fmaxf(s[0][2 * rsel], s[0][2 * rsel + 1]), fmaxf(s[1][2 * rsel], s[1][2 * rsel + 1]));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
            mx[rsel] = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
        }
        const bool grow = mx[0] > m_run[0] || mx[1] > m_run[1];
        if (__any_sync(0xffffffffu, grow)) {
            float alpha[2];
#pragma unroll
            for (int rsel = 0; rsel < 2; ++rsel) {
                const float m_new = fmaxf(m_run[rsel], ref_max(mx[rsel]));
                alpha[rsel] = m_new == -CUDART_INF_F ? 1.f : exp2_int(m_run[rsel] - m_new);
                l_run[rsel] *= alpha[rsel];
                m_run[rsel] = m_new;
            }
#pragma unroll
            for (int a = 0; a < D / 8; ++a) {
                o[a][0] *= alpha[0];
                o[a][1] *= alpha[0];
                o[a][2] *= alpha[1];
                o[a][3] *= alpha[1];
            }
        }
#pragma unroll
        for (int rsel = 0; rsel < 2; ++rsel) {
            // 2^(q(s) - m): s quantised on the fixed grid, the subtraction exact.
            const float off = kQuantC + (m_run[rsel] == -CUDART_INF_F ? 0.f : m_run[rsel]);
            float rs = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                s[nt][2 * rsel] = ex2((s[nt][2 * rsel] + kQuantC) - off);
                s[nt][2 * rsel + 1] = ex2((s[nt][2 * rsel + 1] + kQuantC) - off);
                rs += s[nt][2 * rsel] + s[nt][2 * rsel + 1];
            }
            l_run[rsel] += rs;
        }

        // O += P V.  Keys past the visible range were zero-filled, so their
        // V rows contribute 0 * 0.
        uint32_t pa[4];
        pa[0] = pack_bf16(s[0][0], s[0][1]);
        pa[1] = pack_bf16(s[0][2], s[0][3]);
        pa[2] = pack_bf16(s[1][0], s[1][1]);
        pa[3] = pack_bf16(s[1][2], s[1][3]);
        {
            const int vrow = ((lane >> 3) & 1) * 8 + (lane & 7);
            const int csel = lane >> 4;
            const uint32_t vb = smem_u32(vbuf) + vrow * C::kRowBytes + csel * 16 + dh * C::DW * 2;
#pragma unroll
            for (int n2 = 0; n2 < C::DW / 16; ++n2) {
                const uint32_t addr = vb + n2 * 32;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(addr, b0, b1, b2, b3);
                mma_bf16_16816(o[2 * n2], pa, b0, b1);
                mma_bf16_16816(o[2 * n2 + 1], pa, b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // Quad-reduce the row sums (each thread summed its own columns).
#pragma unroll
    for (int rsel = 0; rsel < 2; ++rsel) {
        l_run[rsel] += __shfl_xor_sync(0xffffffffu, l_run[rsel], 1);
        l_run[rsel] += __shfl_xor_sync(0xffffffffu, l_run[rsel], 2);
    }

    // Merge the key slices through shared memory (every stage was waited on by
    // every consumer warp, so all copies into the ring have landed).
    asm volatile("bar.sync 1, %0;" ::"r"(C::kConsumers * 32) : "memory");
    if (*(volatile int*)abort_flag) return;  // CTA-uniform after the barrier
    float* red_o = reinterpret_cast<float*>(smem);
    float* red_m = red_o + KSL * MT * 16 * C::kRedStride;
    float* red_l = red_m + KSL * MT * 16;
    const int rows_cta = MT * 16;
#pragma unroll
    for (int rsel = 0; rsel < 2; ++rsel) {
        const int r = rsel ? r1 : r0;
        float* dst = red_o + ((size_t)ks * rows_cta + r) * C::kRedStride + dh * C::DW;
#pragma unroll
        for (int a = 0; a < C::DW / 8; ++a)
            *reinterpret_cast<float2*>(dst + a * 8 + 2 * tig) = make_float2(o[a][2 * rsel], o[a][2 * rsel + 1]);
        if (tig == 0 && dh == 0) {
            red_m[ks * rows_cta + r] = m_run[rsel];
            red_l[ks * rows_cta + r] = l_run[rsel];
        }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(C::kConsumers * 32) : "memory");

    const bool partial = p.num_splits > 1;
    for (int idx = threadIdx.x; idx < rows_cta * (D / 4); idx += C::kConsumers * 32) {
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
                const float w = exp2_int(red_m[k * rows_cta + r] - M);  // integers: an exact power of two
                L += w * red_l[k * rows_cta + r];
                const float4 v =
                    *reinterpret_cast<const float4*>(red_o + ((size_t)k * rows_cta + r) * C::kRedStride + c4 * 4);
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
            // natural-log sum-exp: M and log2 L are in base-2 units
            if (p.lse && c4 == 0)
                p.lse[(size_t)t * p.lse_st + (size_t)h * p.lse_sh] =
                    M == -CUDART_INF_F ? -CUDART_INF_F : (M + __log2f(L)) * kLn2;
        } else {
            const size_t row = ((size_t)split * p.T + t) * p.H + h;
            *reinterpret_cast<float4*>(p.ws_o + row * D + c4 * 4) = acc;
            if (c4 == 0) p.ws_lse[row] = M == -CUDART_INF_F ? -CUDART_INF_F : M + __log2f(L);
        }
    }
}

template <int D, int MT, int KSL>
int decode_smem_bytes(int nst) {
    using C = DecodeCfg<D, MT, KSL>;
    int body = nst * C::kStageBytes;
    if (body < C::kRedBytes) body = C::kRedBytes;
    return 128 + body + 2 * C::kMaxStages * 8 + 2 * C::kPairs * 8 + 16 + C::kXchBytes;
}

template <int D, int MT, int KSL>
int pick_stages(int ctas, int num_sms) {
    using C = DecodeCfg<D, MT, KSL>;
    // One CTA per SM when the grid fits in one wave or the CTA has eight
    // consumer warps, else two per SM; the ring takes what shared memory
    // allows so the producers run far ahead.
    const int budget = (ctas <= num_sms || C::kConsumers >= 8) ? 224 * 1024 : 111 * 1024;
    int n = (budget - 512) / C::kStageBytes;
    if (n > C::kMaxStages) n = C::kMaxStages;
    if (n < 2) n = 2;
    return n;
}

template <int D, int MT, int KSL, bool BF32>
cudaError_t launch_t(const AttnParams& p, const LaunchShape& s, cudaStream_t stream) {
    auto kern = decode_kernel<D, MT, KSL, BF32>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s.smem);
    if (e != cudaSuccess) return e;
    kern<<<s.grid, s.block, s.smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

// Tile shape: up to 16 packed rows use one 16-row MMA tile and 8 key groups
// (8 warps); 17-32 rows use 2 row tiles x 4 groups, 33-64 rows 4 x 2.  With
// head_dim 256 each group takes a pair of warps (one per dim half), so the
// groups halve: 4, 2 and 1.
LaunchShape decode_shape(const AttnParams& p, int num_sms) {
    LaunchShape s;
    const int ctas = p.num_splits * p.Hk * p.B;
    const int ds = p.D == 256 ? 2 : 1;
    if (p.max_rows <= 16) {
        s.mt = 1;
        // Eight consumer warps and four producers, one CTA per SM: one CTA
        // streams its (request, kv head) at close to an SM's share of HBM
        // bandwidth, and with the longest requests first the grid's tail is
        // the short ones.
        s.ksl = 8 / ds;
    } else if (p.max_rows <= 32) {
        s.mt = 2;
        s.ksl = 4 / ds;
    } else {
        s.mt = 4;
        s.ksl = 2 / ds;
    }
    s.grid = dim3(p.num_splits, p.Hk, p.B);
    // Four producer warps next to the eight consumers: a single issuing warp
    // cannot keep enough 16-byte gathers in flight.
    const int consumers = s.mt * s.ksl * ds;
    s.nprod = consumers >= 8 ? 4 : 2;
    s.block = (consumers + s.nprod) * 32;
#define REL_ATTN_SHAPE(DD, M, K)                         \
    if (p.D == DD && s.mt == M && s.ksl == K) {         \
        s.nstage = pick_stages<DD, M, K>(ctas, num_sms); \
        s.smem = decode_smem_bytes<DD, M, K>(s.nstage); \
    }
    REL_ATTN_SHAPE(64, 1, 8)
    REL_ATTN_SHAPE(64, 2, 4)
    REL_ATTN_SHAPE(64, 4, 2)
    REL_ATTN_SHAPE(128, 1, 8)
    REL_ATTN_SHAPE(128, 2, 4)
    REL_ATTN_SHAPE(128, 4, 2)
    REL_ATTN_SHAPE(256, 1, 4)
    REL_ATTN_SHAPE(256, 2, 2)
    REL_ATTN_SHAPE(256, 4, 1)
#undef REL_ATTN_SHAPE
    return s;
}

cudaError_t launch_decode(const AttnParams& p, const LaunchShape& s, cudaStream_t stream) {
#define REL_ATTN_LAUNCH(DD, M, K)                                                                      \
    if (p.D == DD && s.mt == M && s.ksl == K)                                                          \
        return p.bias_f32 ? launch_t<DD, M, K, true>(p, s, stream) : launch_t<DD, M, K, false>(p, s, stream);
    REL_ATTN_LAUNCH(64, 1, 8)
    REL_ATTN_LAUNCH(64, 2, 4)
    REL_ATTN_LAUNCH(64, 4, 2)
    REL_ATTN_LAUNCH(128, 1, 8)
    REL_ATTN_LAUNCH(128, 2, 4)
    REL_ATTN_LAUNCH(128, 4, 2)
    REL_ATTN_LAUNCH(256, 1, 4)
    REL_ATTN_LAUNCH(256, 2, 2)
    REL_ATTN_LAUNCH(256, 4, 1)
#undef REL_ATTN_LAUNCH
    return cudaErrorInvalidValue;
}

}  // namespace relattn
