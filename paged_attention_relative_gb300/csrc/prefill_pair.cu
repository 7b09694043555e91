// Prefill / chunked-prefill kernel on CTA pairs: 2-SM tcgen05 MMAs
// (cta_group::2), head_dim 128 or 256.
//
// One cluster of two CTAs per (pair of adjacent 128-row query tiles, kv
// head, request, split).  Rows are GQA-packed token-major as in the other
// kernels: row r of a tile is query token i0 + r / G of the request and
// query head g*G + r % G.  CTA rank r holds tile qt_top - r; one 2-SM MMA
// (M = 256) covers both tiles, issued by a single thread of the even CTA.
// The pair walks one sequence of 128-key tiles (the union of its tiles'
// visible ranges, last tile first); each CTA stages half of every tile,
// keys [64 r, 64 r + 64) of K (every 64-dim block) and dims
// [D/2 r, D/2 r + D/2) of V (all 128 keys): the split of the B operand that
// the 2-SM MMA reads from the two CTAs.  Halving K and V per CTA is what
// makes head_dim 256 fit: O takes TMEM columns [256, 512) and the 64 KB
// query tile, K and V halves and two bias windows stay within 227 KB.  No TMA multicast: every box is loaded once, by the CTA
// that holds it, and signals the even CTA's barrier.  A CTA whose tile lies
// past the request still takes part (its half of K/V, its softmax) and
// writes nothing.
//
// Per key tile j the MMA thread issues S_j = Q K_j^T (head_dim 128: per key
// half) and then O += P_{j-1} V_{j-1}, so S_{j+1} is computed while the
// softmax of tile j runs.  Its commits (multicast to both CTAs) also free the
// ring slots: the K slot of tile j once S_j completed, the V slot once PV_j
// completed.
//
// Warp roles (384 threads per CTA):
//   warp 0     the query tile (TMA, one box per 64-dim block), then this CTA's
//              half of every K tile into a ring (2 slots, 1 for head_dim
//              256): one TMA box per 16-key page with every dim block (two
//              8-key boxes when the cache's pages are not contiguous),
//              straight from the paged cache through a 5-D page view,
//              zero-filling cp.async only for the 16-key group that
//              straddles the cache length (keys inside the cache but outside
//              a row's window are finite and masked by the softmax).  The
//              TMA unit's cost is mostly per box, so page boxes (4 K and 8 V
//              boxes per tile instead of 2 KB boxes: 32 at head_dim 256) cut
//              the staging time per tile.
//   warp 1     bias windows: for each band tile one TMA box per 8-token
//              sub-box into one of three (head_dim 256: two) window buffers,
//              once the softmax has released that buffer's previous fill.
//   warp 2     this CTA's half of every V tile (its D/2 dims of every page:
//              one box per page) into a ring like K's.
//   warp 3     TMEM (512 columns, allocated by the pair) and, in the even
//              CTA, the MMA thread.
//   warps 4-11 softmax: thread (w, lane) owns keys [64 h, 64 h + 64) of row
//              32 * (w % 4) + lane, h = (w - 4) / 4; scale, sheared bias (read
//              reversed from the staged window), mask, exponentials against
//              an integer reference maximum that moves lazily (see kQuantC),
//              P into TMEM, a rare rescale of O, the epilogue.  head_dim 128:
//              as in the one-CTA kernel, each key half is an independent
//              stream (own S, P, O and reference maximum; S released as soon
//              as it is read; halves merged in the epilogue), the per-half S
//              MMA (N = 64) reading each CTA's 32 keys from K pages 2r, 2r + 1
//              (half 0) and 2r + 4, 2r + 5 (half 1).  head_dim 256: one O, the
//              two warps of a row exchange half-row maxima through shared
//              memory, and P is written over the S columns already read.
//
// TMEM columns (PairCfg): head_dim 128 O_0, O_1, S_0, S_1, P_0, P_1;
// head_dim 256 S_0 [0, 128), S_1 [128, 256), O [256, 512), P_j in S buffer
// j % 2 (keys [64 h, 64 h + 64) in columns [64 h, 64 h + 32)).
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
constexpr float kLazyRescale = 8.0f;  // log2 units

template <int D_>
struct PairCfg {
    static constexpr int D = D_;
    static constexpr int BN = 128;                    // keys per tile
    static constexpr int kDB = D / 64;                // 64-dim (128-byte) blocks
    static constexpr int kVB = D / 128;               // 64-dim blocks of this CTA's V half
    static constexpr int kQBytes = kDB * 128 * 128;   // the query tile: kDB blocks x 128 rows x 128 B
    // This CTA's halves of a K and a V tile, page by page (16 keys), each
    // page as one TMA box lands: [8-key half][64-dim block][8 keys][128 B].
    // K: 4 pages with every dim block; V: 8 pages with kVB dim blocks.
    static constexpr int kKHalf = kDB * 1024;
    static constexpr int kKPage = 2 * kKHalf;
    static constexpr int kVHalf = kVB * 1024;
    static constexpr int kVPage = 2 * kVHalf;
    static constexpr int kKBytes = 4 * kKPage;
    static constexpr int kVBytes = 8 * kVPage;
    static constexpr int kRing = D == 128 ? 2 : 1;    // K and V ring slots
    static constexpr int kBiasW = 152;                // rel_logits values per staged row
    static constexpr int kBiasBytes = 128 * kBiasW * 2 + 16 * 128;
    static constexpr int kBiasBufs = D == 128 ? 3 : 2;
    static constexpr int kXchBytes = 3 * 2 * 128 * 4;  // half-row maxima (2 tile buffers), half-row sums
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + kRing * kKBytes;
    static constexpr int kOffBias = kOffV + kRing * kVBytes;
    static constexpr int kOffXch = kOffBias + kBiasBufs * kBiasBytes;
    static constexpr int kData = kOffXch + kXchBytes;
    static constexpr int kThreads = 384;
    static constexpr int kTmemCols = 512;
    static constexpr int kSoftWarps = 8;
    // head_dim 128: the two key halves of every tile are independent softmax
    // streams, each with its own S, P and O in TMEM (O_0 [0,128), O_1
    // [128,256), S_0 [256,320), S_1 [320,384), P_0 [384,416), P_1 [416,448))
    // and its own reference maximum, merged in the epilogue.  head_dim 256:
    // no room for a second O, so S is double-buffered (S_0 [0,128), S_1
    // [128,256)), P is written over S and one O takes [256, 512).
    static constexpr bool kHalves = D == 128;
    static constexpr int kOCol = kHalves ? 0 : 256;
    static constexpr int kSCol = 256;
    static constexpr int kPCol = 384;
};

struct PairBars {
    uint64_t q_full;            // even CTA: both CTAs' query tiles have landed
    uint64_t k_full[2];         // even CTA: K slot filled in both CTAs (one phase per fill)
    uint64_t v_full[2];         // even CTA: V slot filled in both CTAs (one phase per fill)
    // head_dim 256: index = S buffer (one phase per use, every other tile);
    // head_dim 128: index = key half (one phase per tile).
    uint64_t p_full[2];         // even CTA: P written by both CTAs' softmax warps
    uint64_t s_full[2];         // both: S computed
    uint64_t o_done[2];         // both: PV completed
    uint64_t s_free[2];         // even CTA, head_dim 128: both CTAs' warps of key half h have read S_h
    uint64_t k_empty[2];        // both, head_dim 128: K slot's tile consumed by S_0 and S_1 (per use)
    uint64_t v_empty[2];        // both, head_dim 128: V slot's tile consumed by PV_0 and PV_1 (per use)
    uint64_t x_full[2];         // this CTA: per tile parity, every softmax warp published its half-row maxima
    uint64_t o_final;           // both: every MMA of the item completed
    uint64_t bias_full[3];      // this CTA: window buffer filled (one phase per fill)
    uint64_t bias_empty[3];     // this CTA: every softmax warp has read it
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ bool aborted(const PairBars* bars) {
    return *reinterpret_cast<const volatile int*>(&bars->abort) != 0;
}

constexpr int kCompactMaxB = 256;

// Cluster ci of a compact launch -> (request, top query tile of its pair), or
// request -1 past the last pair.  Requests in order; within a request the
// pairs go from the last (most keys) to the first.  Warp-collective.
__device__ __forceinline__ int2 compact_pair(const int32_t* cu, int B, int TPT, int ci) {
    const int lane = threadIdx.x & 31;
    int base = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
        const int bb = b0 + lane;
        int n = 0;
        if (bb < B) {
            const int nt = (__ldg(cu + bb + 1) - __ldg(cu + bb) + TPT - 1) / TPT;
            n = (nt + 1) / 2;
        }
        int inc = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        const int tot = __shfl_sync(0xffffffffu, inc, 31);
        if (ci < base + tot) {
            const int src = __ffs(__ballot_sync(0xffffffffu, base + inc > ci)) - 1;
            const int first = base + __shfl_sync(0xffffffffu, inc - n, src);
            const int nb = __shfl_sync(0xffffffffu, n, src);
            const int k = nb - 1 - (ci - first);
            return make_int2(b0 + src, 2 * k + 1);
        }
        base += tot;
    }
    return make_int2(-1, 0);
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    prefill_pair_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_rel,
                        const __grid_constant__ CUtensorMap tm_q) {
    using C = PairCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + C::kOffQ;
    uint8_t* sK = smem + C::kOffK;
    uint8_t* sV = smem + C::kOffV;
    uint8_t* sBias = smem + C::kOffBias;
    float* sXch = reinterpret_cast<float*>(smem + C::kOffXch);  // [3 bufs][2 halves][128 rows]
    PairBars* bars = reinterpret_cast<PairBars*>(smem + C::kData);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G, TPT = 128 / G;
    const int rank = (int)cluster_ctarank();
    const int g = blockIdx.y;
    const int S = p.num_splits;
    int qt_top, b, split;
    if (p.B <= kCompactMaxB) {
        const int2 ct = compact_pair(p.cu_seqlens_q, p.B, TPT, (int)(blockIdx.x / 2));
        if (ct.x < 0) return;  // past the last pair (the same in both CTAs)
        b = ct.x;
        qt_top = ct.y;
        split = blockIdx.z;
    } else {
        qt_top = (int)gridDim.x - 1 - 2 * (int)(blockIdx.x / 2);  // longest pairs first
        b = blockIdx.z / S;
        split = blockIdx.z % S;
    }
    const int q0 = p.cu_seqlens_q[b];
    const int sq = p.cu_seqlens_q[b + 1] - q0;
    const int sk = p.cache_seqlens[b];
    const int off = sk - sq;
    const int R = p.R;
    // A pair without rows (only past a request's last pair, in the
    // non-compact grid) leaves at once, in both CTAs.
    if ((qt_top - 1) * TPT >= sq) return;
    const int qt = qt_top - rank;  // this CTA's query tile
    const int i0 = qt * TPT;
    const int i1 = min(sq, i0 + TPT);
    const int n_rows = max(i1 - i0, 0) * G;
    const int pos_min = i0 + off, pos_max = i1 - 1 + off;

    // Keys any row of the pair may see, as 128-key tiles, split contiguously.
    const int u_pmin = (qt_top - 1) * TPT + off;
    const int u_pmax = min(sq, (qt_top + 1) * TPT) - 1 + off;
    int hi = sk, lo = 0;
    if (p.causal) hi = min(hi, u_pmax + 1);
    if (p.wr >= 0) hi = min(hi, u_pmax + p.wr + 1);
    if (p.wl >= 0) lo = max(0, u_pmin - p.wl);
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
    // Does key tile [j0, j0 + 128) reach this CTA's bias band 0 <= pos - j < R?
    auto band_tile = [&](int j0) {
        return R > 0 && n_rows > 0 && pos_max - j0 >= 0 && pos_min - (j0 + C::BN - 1) < R;
    };

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 2);  // one arrival per CTA
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->k_full[i], 2);
            mbar_init(&bars->v_full[i], 2);
            // one arrival per softmax warp of both CTAs (head_dim 128: per key half)
            mbar_init(&bars->p_full[i], C::kHalves ? C::kSoftWarps : 2 * C::kSoftWarps);
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->o_done[i], 1);
            mbar_init(&bars->x_full[i], C::kSoftWarps);
            mbar_init(&bars->s_free[i], C::kSoftWarps);
            mbar_init(&bars->k_empty[i], 1);
            mbar_init(&bars->v_empty[i], 1);
        }
        mbar_init(&bars->o_final, 1);
        for (int i = 0; i < C::kBiasBufs; ++i) {
            mbar_init(&bars->bias_full[i], 1);
            mbar_init(&bars->bias_empty[i], C::kSoftWarps);
        }
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 3) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars->tmem_base)),
                     "n"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    // The peer arrives on this CTA's barriers, and the MMAs signal both CTAs,
    // only after both have initialised them and allocated TMEM.
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------ Q, K and V producers
        const bool is_v = warp == 2;
        const uint16_t* cache = reinterpret_cast<const uint16_t*>(is_v ? p.v_cache : p.k_cache);
        const CUtensorMap* tmap = is_v ? &tm_v : &tm_k;
        const int32_t* bt = p.block_table + (size_t)b * p.bt_stride;
        const uint64_t pol_last = l2_policy_evict_last();
        if (lane == 0) tma_prefetch_desc(tmap);
        if (!is_v) {
            // The query tile: one box per 64-dim block (64 dims x G heads x TPT
            // tokens).  Rows past the request read other tokens or TMA's zero
            // fill and are never written out; when G does not divide 128 the
            // rows past G * TPT are zeroed once so that S stays finite there.
            const int q_rows = G * TPT;
            if (q_rows < 128) {
                for (int i = lane; i < C::kDB * (128 - q_rows) * 8; i += 32) {
                    const int chunk = i & 7, row = q_rows + ((i >> 3) % (128 - q_rows));
                    const int db = (i >> 3) / (128 - q_rows);
                    *reinterpret_cast<uint4*>(sQ + db * (128 * 128) +
                                              sw128_offset((uint32_t)row, (uint32_t)chunk)) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                const uint32_t qbar = mapa_shared(smem_u32(&bars->q_full), 0);
                tma_prefetch_desc(&tm_q);
                mbar_expect_tx_cluster(qbar, (uint32_t)(C::kDB * q_rows * 128));
                for (int db = 0; db < C::kDB; ++db)
                    tma_load_3d_pair(sQ + db * (128 * 128), &tm_q, qbar, 64 * db, g * G, q0 + i0, pol_last);
                mbar_arrive_cluster(qbar);
            }
            __syncwarp();
        }
        // 16-key pages of a tile this CTA stages: K pages 4 rank .. 4 rank + 3
        // (every dim block), V pages 0 .. 7 (dim blocks kVB rank .. kVB rank +
        // kVB - 1); local page i at i * page_bytes, laid out as its TMA box
        // lands: [8-key half][dim block][8 keys][128 B].
        // (head_dim 128: K pages 2 rank, 2 rank + 1, 2 rank + 4, 2 rank + 5,
        // so that each key half's S = Q K^T, N = 64, finds its 32 keys per
        // CTA in local pages 0-1 and 2-3.)
        const int g_first = is_v ? 0 : (C::kHalves ? 2 * rank : 4 * rank);
        auto page_of = [&](int li) { return g_first + li + (!is_v && C::kHalves ? 2 * (li >> 1) : 0); };
        const int n_groups = is_v ? 8 : 4;
        const int n_db = is_v ? C::kVB : C::kDB;       // dim blocks per page this CTA stages
        const int db_first = is_v ? C::kVB * rank : 0;
        const int page_bytes = is_v ? C::kVPage : C::kKPage;
        const int slot_bytes = is_v ? C::kVBytes : C::kKBytes;
        // One box per page when the cache's pages are contiguous, else one per 8-key half.
        const int nbox = p.kv_merged ? 1 : 2;
        uint8_t* ring = is_v ? sV : sK;
        uint32_t full_bar[2];
        for (int i = 0; i < 2; ++i)
            full_bar[i] = mapa_shared(smem_u32(is_v ? &bars->v_full[i] : &bars->k_full[i]), 0);
        // The slot of tile jj is free again once S (K) or PV (V) of tile
        // jj - kRing, the tile it held, has completed (barrier (jj - kRing) % 2).
        // (head_dim 128: the slot's own empty barrier, one phase per use.)
        uint64_t* free_bar[2] = {is_v ? &bars->o_done[0] : &bars->s_full[0], is_v ? &bars->o_done[1] : &bars->s_full[1]};
        if (C::kHalves) {
            free_bar[0] = is_v ? &bars->v_empty[0] : &bars->k_empty[0];
            free_bar[1] = is_v ? &bars->v_empty[1] : &bars->k_empty[1];
        }
        // At most one cp.async batch (the partial groups of a tile) is in
        // flight; it is retired (landed, proxy-fenced, one arrival with a
        // cluster-scope release on the even CTA's barrier, whose MMA reads
        // these bytes) after the next tile's boxes are issued, or before the
        // producer blocks on a slot.
        int pend = -1;
        auto retire = [&](int newer) {
            cp_async_wait(newer);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(full_bar[pend]);
            pend = -1;
        };
        // Block-table windows of 4 tiles: lane l holds the physical block of
        // 16-key group l % 8 of tile w0 + l / 8 (one coalesced load).
        auto load_win = [&](int w0) -> int {
            int v = 0;
            const int jw = w0 + (lane >> 3);
            if (jw < n_it) {
                const int jg = key_block(jw) * C::BN + 16 * (lane & 7);
                if (jg < sk && jg / p.BS < p.max_blocks) v = __ldg(bt + jg / p.BS);
            }
            return v;
        };
        int win_cur = load_win(0), win_nxt = load_win(4);
        for (int jj = 0; jj < n_it; ++jj) {
            const int slot = jj % C::kRing;
            if (jj >= C::kRing) {
                // The slot last held tile jj - kRing: use (jj - kRing) / 2 of barrier (jj - kRing) % 2.
                const int prev = jj - C::kRing;
                const uint32_t par = (uint32_t)((prev >> 1) & 1);
                if (!mbar_try_wait(free_bar[prev & 1], par)) {
                    if (pend >= 0) retire(0);
                    if (!mbar_wait(free_bar[prev & 1], par, p.timeout_ns, kSitePrefillKEmpty, p.err)) bars->abort = 1;
                }
            }
            if (__any_sync(0xffffffffu, aborted(bars))) break;
            if (jj >= 4 && (jj & 3) == 0) {
                win_cur = win_nxt;
                win_nxt = load_win(jj + 4);
            }
            const int wl = (jj & 3) * 8;
            const int j0 = key_block(jj) * C::BN;
            uint32_t full_mask = 0;  // bit i: local page i fully visible (whole-box TMA)
            for (int i = 0; i < n_groups; ++i) {
                const int jg = j0 + 16 * page_of(i);
                if (jg + 16 <= sk) full_mask |= 1u << i;
            }
            uint8_t* tile = ring + slot * slot_bytes;
            if (lane == 0) mbar_expect_tx_cluster(full_bar[jj & 1], (uint32_t)(__popc(full_mask) * page_bytes));
            __syncwarp();
            // TMA lanes: lane -> (local page lane / nbox, half lane % nbox),
            // through the page view of the cache (5-D; see make_page_map).
            {
                const int li = (lane / nbox) & (n_groups - 1);
                const int t_h = lane % nbox;
                const int pg = page_of(li);
                const int blk = min(max(__shfl_sync(0xffffffffu, win_cur, wl + pg), 0), p.NB - 1);
                if (lane < n_groups * nbox && ((full_mask >> li) & 1)) {
                    const int slot_in_blk = (j0 + 16 * pg) % p.BS;
                    // merged view (64, 8, D/64, NB * BS / 8, Hk): half-page blk * BS / 8 + slot / 8;
                    // split view (64, BS, D/64, Hk, NB): slot, head, block.
                    uint8_t* dst = tile + li * page_bytes + (p.kv_merged ? 0 : t_h * (page_bytes / 2));
                    const int c1 = p.kv_merged ? 0 : slot_in_blk + 8 * t_h;
                    const int c3 = p.kv_merged ? blk * (p.BS >> 3) + (slot_in_blk >> 3) : g;
                    const int c4 = p.kv_merged ? g : blk;
                    tma_load_5d_pair(dst, tmap, full_bar[jj & 1], 0, c1, db_first, c3, c4, pol_last);
                }
            }
            const bool part = full_mask != (1u << n_groups) - 1;
            if (part) {
                // Zero-filling cp.async of the groups not wholly visible:
                // n_db dim blocks x 16 keys x 8 chunks each.
                for (int i = 0; i < n_groups; ++i) {
                    if ((full_mask >> i) & 1) continue;
                    const int pg = page_of(i);
                    const int jg = j0 + 16 * pg;
                    const int blk = min(max(__shfl_sync(0xffffffffu, win_cur, wl + pg), 0), p.NB - 1);
                    const uint16_t* src0 =
                        cache + (long long)blk * p.c_s0 + (long long)(jg % p.BS) * p.c_s1 + (long long)g * p.c_s2;
                    for (int c = lane; c < n_db * 128; c += 32) {
                        const int dbl = c >> 7;
                        const int row = (c >> 3) & 15, chunk = c & 7;
                        const bool valid = jg + row < sk;
                        const uint16_t* src = src0 + (long long)row * p.c_s1 + 64 * (db_first + dbl) + chunk * 8;
                        const uint32_t dst = smem_u32(tile + i * page_bytes + (row >> 3) * (page_bytes / 2) +
                                                      dbl * 1024) +
                                             sw128_offset((uint32_t)(row & 7), (uint32_t)chunk);
                        cp_async_16(dst, valid ? src : cache, valid ? 16u : 0u, pol_last);
                    }
                }
                cp_async_commit();
            }
            if (pend >= 0) retire(part ? 1 : 0);
            if (part) {
                pend = jj & 1;
            } else {
                // Only TMA boxes: their bytes complete the phase, the arrival
                // needs no cluster-scope release (which costs ~1k cycles).
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(full_bar[jj & 1]);
            }
        }
        if (pend >= 0) retire(0);
    } else if (warp == 1) {
        // ------------------------------------------------------ bias windows
        // Band tile n's rel_logits into buffer n % 3, once every softmax warp
        // has finished reading fill n - 3: one TMA box per token sub-box of
        // TS tokens (all G heads), rows of kBiasW distances from the 16-byte
        // aligned distance below the sub-box's smallest one.
        if (p.vec_bias && lane == 0 && n_rows > 0) {
            const int TS = p.bias_ts, n_sub = TPT / TS;
            const int sub_bytes = (TS * G * C::kBiasW * 2 + 127) & ~127;
            const uint64_t pol = l2_policy_evict_first();
            int nbi = 0;
            for (int jj = 0; jj < n_it; ++jj) {
                const int j0 = key_block(jj) * C::BN;
                if (!band_tile(j0)) continue;
                const int bb = nbi % C::kBiasBufs, use = nbi / C::kBiasBufs;
                if (use > 0 && !mbar_wait(&bars->bias_empty[bb], (uint32_t)((use - 1) & 1), p.timeout_ns,
                                          kSitePrefillRelEmpty, p.err)) {
                    bars->abort = 1;
                    break;
                }
                if (aborted(bars)) break;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bars->bias_full[bb], (uint32_t)(n_sub * TS * G * C::kBiasW * 2));
                for (int sbx = 0; sbx < n_sub; ++sbx) {
                    const int ts = i0 + sbx * TS;
                    const int a = ts + off - j0 - 127;
                    tma_load_3d_hint(sBias + bb * C::kBiasBytes + sbx * sub_bytes, &tm_rel, &bars->bias_full[bb],
                                     a - (a & 7), g * G, q0 + ts, pol);
                }
                ++nbi;
            }
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------------------ MMA issuer (even CTA)
        // The whole warp runs the loop (converged); one elected lane issues.
        if (rank == 0 && n_it > 0) {
            constexpr uint32_t idS = umma_idesc_bf16(256, C::BN, false);
            constexpr uint32_t idPV = umma_idesc_bf16(256, C::D, true);
            constexpr int KS = C::D / 16;  // K-steps of S
            bool ok = mbar_wait_warp(&bars->q_full, 0, p.timeout_ns, kSitePrefillLoadQ, p.err);
            // Descriptors: Q (K-major, kDB dim blocks), K half (K-major), V half
            // (MN-major, kVB 64-dim blocks 16 KB apart).  A descriptor's low
            // bits hold address / 16, so a byte offset adds offset / 16.
            const uint64_t dQ = umma_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dK0 = umma_desc_sw128(smem_u32(sK), 16, C::kKHalf);
            const uint64_t dV0 = umma_desc_sw128(smem_u32(sV), 1024, C::kVHalf);
            uint64_t aQ[KS];
#pragma unroll
            for (int kk = 0; kk < KS; ++kk)
                aQ[kk] = dQ + (uint64_t)(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
            if constexpr (C::kHalves) {
                // Key half h of tile jj: S_h = Q K_jj[64h, 64h + 64)^T (N = 64:
                // each CTA's 32 keys in its local pages 2h, 2h + 1) once both
                // CTAs' warps of half h have read S_h(jj - 1) (s_free[h]); then
                // O_h += P_h V_jj[64h, 64h + 64) (4 K-steps) once both CTAs
                // wrote P_h (p_full[h]).  The slot's empty barrier follows the
                // second half.
                constexpr uint32_t idS2 = umma_idesc_bf16(256, 64, false);
                auto issue_s = [&](int jj) {
                    const int ks = jj % C::kRing;
                    uint64_t bK[KS];
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk)
                        bK[kk] = dK0 + (uint64_t)((ks * C::kKBytes + (kk >> 2) * 1024 + (kk & 3) * 32) >> 4);
                    ok = ok && mbar_wait_warp(&bars->k_full[jj & 1], (uint32_t)((jj >> 1) & 1), p.timeout_ns,
                                              kSitePrefillKFull, p.err);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        ok = ok && mbar_wait_warp(&bars->s_free[hh], (uint32_t)(jj & 1), p.timeout_ns,
                                                  kSitePrefillSFull, p.err);
                        if (!ok) return;
                        tc_fence_after();
                        const uint32_t sd = tmem + C::kSCol + 64 * hh;
                        const uint64_t ho = (uint64_t)((2 * hh * C::kKPage) >> 4);
                        umma2_ss<0>(sd, aQ[0], bK[0] + ho, idS2);
#pragma unroll
                        for (int kk = 1; kk < KS; ++kk) umma2_ss<1>(sd, aQ[kk], bK[kk] + ho, idS2);
                        umma2_commit_both(&bars->s_full[hh]);
                    }
                    umma2_commit_both(&bars->k_empty[ks]);
                };
                auto issue_pv = [&](int t) {
                    const int vs = t % C::kRing;
                    uint64_t bV[8];
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        bV[kk] = dV0 + (uint64_t)((vs * C::kVBytes + kk * C::kVPage) >> 4);
                    ok = ok && mbar_wait_warp(&bars->v_full[t & 1], (uint32_t)((t >> 1) & 1), p.timeout_ns,
                                              kSitePrefillVFull, p.err);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        ok = ok && mbar_wait_warp(&bars->p_full[hh], (uint32_t)(t & 1), p.timeout_ns,
                                                  kSitePrefillPFull, p.err);
                        if (!ok) return;
                        tc_fence_after();
                        const uint32_t od = tmem + C::kOCol + 128 * hh, pc = tmem + C::kPCol + 32 * hh;
                        if (t > 0)
                            umma2_ts<1>(od, pc, bV[4 * hh], idPV);
                        else
                            umma2_ts<0>(od, pc, bV[4 * hh], idPV);
#pragma unroll
                        for (int kk = 1; kk < 4; ++kk) umma2_ts<1>(od, pc + 8 * kk, bV[4 * hh + kk], idPV);
                        umma2_commit_both(&bars->o_done[hh]);
                    }
                    umma2_commit_both(&bars->v_empty[vs]);
                };
                for (int jj = 0; jj < n_it && ok; ++jj) {
                    issue_s(jj);
                    if (ok && jj >= 1) issue_pv(jj - 1);
                }
                if (ok) issue_pv(n_it - 1);
            } else {
                // S_jj = Q K^T into S buffer jj % 2, K from ring slot jj % kRing.
                auto issue_s = [&](int jj) {
                    const int sb = jj & 1, ks = jj % C::kRing;
                    uint64_t bK[KS];
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk)
                        bK[kk] = dK0 + (uint64_t)((ks * C::kKBytes + (kk >> 2) * 1024 + (kk & 3) * 32) >> 4);
                    ok = ok && mbar_wait_warp(&bars->k_full[jj & 1], (uint32_t)((jj >> 1) & 1), p.timeout_ns,
                                         kSitePrefillKFull, p.err);
                    if (!ok) return;
                    tc_fence_after();
                    const uint32_t sd = tmem + sb * C::BN;
                    umma2_ss<0>(sd, aQ[0], bK[0], idS);
#pragma unroll
                    for (int kk = 1; kk < KS; ++kk) umma2_ss<1>(sd, aQ[kk], bK[kk], idS);
                    umma2_commit_both(&bars->s_full[sb]);
                };
                // O += P_t V_t: P from S buffer t % 2 (keys [64 h, 64 h + 64) in
                // columns [64 h, 64 h + 32)), V from V slot t % 2.  The MMAs of
                // this warp (always its lowest lane, the one elect.sync picks)
                // run in issue order, so S_{t+2}, issued after PV_t, overwrites
                // the buffer only once PV_t has read P_t.
                auto issue_pv = [&](int t) {
                    const int pb = t & 1, vs = t % C::kRing;
                    uint64_t bV[8];
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) bV[kk] = dV0 + (uint64_t)((vs * C::kVBytes + kk * C::kVPage) >> 4);
                    ok = ok && mbar_wait_warp(&bars->p_full[pb], (uint32_t)((t >> 1) & 1), p.timeout_ns, kSitePrefillPFull,
                                         p.err);
                    ok = ok && mbar_wait_warp(&bars->v_full[t & 1], (uint32_t)((t >> 1) & 1), p.timeout_ns, kSitePrefillVFull,
                                         p.err);
                    if (!ok) return;
                    tc_fence_after();
                    const uint32_t pcol = tmem + pb * C::BN, od = tmem + C::kOCol;
                    if (t > 0)
                        umma2_ts<1>(od, pcol, bV[0], idPV);
                    else
                        umma2_ts<0>(od, pcol, bV[0], idPV);
#pragma unroll
                    for (int kk = 1; kk < 8; ++kk) umma2_ts<1>(od, pcol + 64 * (kk >> 2) + 8 * (kk & 3), bV[kk], idPV);
                    umma2_commit_both(&bars->o_done[pb]);
                };
                for (int jj = 0; jj < n_it && ok; ++jj) {
                    issue_s(jj);
                    if (ok && jj >= 1) issue_pv(jj - 1);
                }
                if (ok) issue_pv(n_it - 1);
            }
            // The epilogue may be two or more o_done phases behind, where a
            // parity wait cannot tell phases apart: it has its own barrier.
            umma2_commit_both(&bars->o_final);
            if (!ok) bars->abort = 1;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ softmax
        const int half = (warp - 4) >> 2;  // keys [64*half, 64*half + 64) of each tile
        const int r = (warp & 3) * 32 + lane;  // row == TMEM lane
        const bool valid = r < n_rows;
        const int i_rel = valid ? r / G : 0;  // token within the tile
        const int tok = i0 + i_rel;
        const int hh = valid ? r % G : 0;
        const int t = q0 + tok, h = g * G + hh;
        const int pos = tok + off;
        // Keys this row may see: [klo, khi).
        int khi = sk;
        if (p.causal) khi = min(khi, pos + 1);
        if (p.wr >= 0) khi = min(khi, pos + p.wr + 1);
        int klo = 0;
        if (p.wl >= 0) klo = max(0, pos - p.wl);
        const bool bias_f32 = p.bias_f32 != 0;
        const size_t rel_row = ((size_t)t * p.H + h) * (size_t)R;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float sc = p.scale;          // scores are kept in natural units: sc * q.k + bias
        const float sl2 = p.scale_log2;    // sc * log2(e)
        const bool pos_scale = sc > 0.f;
        const int kh = 64 * half;  // first key of this half within a tile
        float m_run = -CUDART_INF_F, l_half = 0.f;  // reference maximum (an integer in log2 units), half-row sum
        bool any_abort = false;
        const uint32_t p_bar[2] = {mapa_shared(smem_u32(&bars->p_full[0]), 0),
                                   mapa_shared(smem_u32(&bars->p_full[1]), 0)};

        // Bias windows: a band tile's rel_logits arrive by TMA as rows of
        // kBiasW values, one row per (token, head) of the tile, each starting
        // at the 16-byte aligned distance below the smallest distance its
        // token sub-box needs (zero-filled outside [0, R)).  Key k of the tile
        // reads element e_r + 127 - k of row r: this half's 64 keys the
        // 32-bit words W0 - 31 .. W0 + 1 (one byte permute per key pair).
        const int TS = p.bias_ts;
        const int sub_bytes = (TS * G * C::kBiasW * 2 + 127) & ~127;
        const int i_sub = (i_rel / TS) * TS;
        const int e_r = (i_rel - i_sub) + ((i0 + i_sub + off - 127) & 7);
        const int base_h = e_r + 127 - kh;
        const uint32_t* wrow = reinterpret_cast<const uint32_t*>(sBias + (i_rel / TS) * sub_bytes +
                                                                 (r - i_sub * G) * (C::kBiasW * 2)) +
                               (((base_h - 1) >> 1) - 31);
        const uint32_t psel = ((base_h - 1) & 1) ? 0x5432u : 0x3210u;
        int nb = 0;  // band tiles consumed

        if constexpr (C::kHalves) {
            // head_dim 128: key half `half` is its own softmax stream (S_h, P_h,
            // O_h, reference maximum); its S buffer is released to the MMA
            // thread (s_free, both CTAs' warps) as soon as it is read, so the
            // next S_h computes during this tile's exponentials.
            const uint32_t s_addr = lane_base + C::kSCol + 64 * half;
            const uint32_t p_addr = lane_base + C::kPCol + 32 * half;
            const uint32_t o_addr = lane_base + C::kOCol + 128 * half;
            const uint32_t sfree_bar = mapa_shared(smem_u32(&bars->s_free[half]), 0);
            bool s_ready = false;  // S_h of the next tile seen complete during this one
            // The first S_h needs no read: arrive for it now.
            if (n_it > 0 && lane == 0) mbar_arrive_remote(sfree_bar);
            for (int jj = 0; jj < n_it; ++jj) {
                const int j0 = key_block(jj) * C::BN;
                const int jh = j0 + kh;  // first key of this half
                const bool band = band_tile(j0);
                const bool my_abort = (!s_ready && !mbar_wait(&bars->s_full[half], (uint32_t)(jj & 1), p.timeout_ns,
                                                              kSitePrefillSFull, p.err)) ||
                                      aborted(bars);
                float2 s[32];  // keys (kh + 2e, kh + 2e + 1) of the tile
                float mx = -CUDART_INF_F;
                const bool raw = !band && pos_scale;
                {
                    tc_fence_after();
                    {
                        uint32_t v0[32], v1[32];
                        tmem_ld32(s_addr, v0);
                        tmem_ld32(s_addr + 32, v1);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            s[e] = make_float2(__uint_as_float(v0[2 * e]), __uint_as_float(v0[2 * e + 1]));
                            s[16 + e] = make_float2(__uint_as_float(v1[2 * e]), __uint_as_float(v1[2 * e + 1]));
                        }
                    }
                    tc_fence_before();
                    // S_h(jj) is in registers: the MMA thread may overwrite the buffer.
                    __syncwarp();
                    if (lane == 0 && jj + 1 < n_it) mbar_arrive_remote(sfree_bar);
                    if (!raw) {
                        const float2 sc2 = make_float2(sc, sc);
                        if (band && p.vec_bias) {
                            const int bb = nb % C::kBiasBufs;
                            if (!mbar_wait(&bars->bias_full[bb], (uint32_t)((nb / C::kBiasBufs) & 1), p.timeout_ns,
                                           kSitePrefillRelFull, p.err))
                                bars->abort = 1;
                            const uint32_t* wb = wrow + bb * (C::kBiasBytes / 4);
                            uint32_t wv[33];
#pragma unroll
                            for (int i = 0; i < 33; ++i) wv[i] = wb[i];
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const uint32_t pr = __byte_perm(wv[31 - e], wv[32 - e], psel);
                                s[e] = __ffma2_rn(
                                    s[e], sc2, make_float2(__uint_as_float(pr & 0xffff0000u), __uint_as_float(pr << 16)));
                            }
                            // Every read of this band tile's windows is done.
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&bars->bias_empty[bb]);
                        } else if (band) {
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const int d = pos - (jh + 2 * e);
                                const float b0 = valid && d >= 0 && d < R ? rel_at(p.rel, bias_f32, rel_row + d) : 0.f;
                                const float b1 =
                                    valid && d - 1 >= 0 && d - 1 < R ? rel_at(p.rel, bias_f32, rel_row + d - 1) : 0.f;
                                s[e] = __ffma2_rn(s[e], sc2, make_float2(b0, b1));
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) s[e] = __fmul2_rn(s[e], sc2);
                        }
                    }
                    // Mask (warp-uniform skip when every row of the warp sees the whole half tile).
                    const bool row_full = !valid || (jh >= klo && jh + 64 <= khi);
                    if (!__all_sync(0xffffffffu, row_full)) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int j = jh + 2 * e;
                            if (!row_full && !(j >= klo && j < khi)) s[e].x = -CUDART_INF_F;
                            if (!row_full && !(j + 1 >= klo && j + 1 < khi)) s[e].y = -CUDART_INF_F;
                        }
                    }
                    float mk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mk[i] = fmax3(s[i].x, s[i].y, s[8 + i].x);
#pragma unroll
                    for (int i = 0; i < 8; ++i) mk[i] = fmax3(mk[i], s[8 + i].y, s[16 + i].x);
#pragma unroll
                    for (int i = 0; i < 8; ++i) mk[i] = fmax3(mk[i], s[16 + i].y, s[24 + i].x);
#pragma unroll
                    for (int i = 0; i < 8; ++i) mk[i] = fmaxf(mk[i], s[24 + i].y);
                    mx = fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7]));
                    if (raw) mx *= sc;
                }
                if (band && p.vec_bias) ++nb;
                const float c1 = raw ? sl2 : kLog2e;
                uint32_t w[32];
                float rsum = 0.f;
                // This half of P (bf16 pairs) and its row sum against the
                // integer reference m: 2^(q(s * c1) - m), see kQuantC.
                auto exp_pass = [&](float m) {
                    const float offs = kQuantC + (m == -CUDART_INF_F ? 0.f : m);
                    const float2 c12 = make_float2(c1, c1), qc = make_float2(kQuantC, kQuantC),
                                 noff = make_float2(-offs, -offs);
                    float2 rs[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) rs[i] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float2 x = __fadd2_rn(__ffma2_rn(s[e], c12, qc), noff);
                        const float2 pe = make_float2(ex2(x.x), ex2(x.y));
                        rs[e & 3] = __fadd2_rn(rs[e & 3], pe);
                        w[e] = pack_bf16(pe.x, pe.y);
                    }
                    const float2 rs2 = __fadd2_rn(__fadd2_rn(rs[0], rs[1]), __fadd2_rn(rs[2], rs[3]));
                    rsum = rs2.x + rs2.y;
                };
                // This half's reference maximum moves lazily (only when its
                // maximum exceeds it by more than 8 in log2 units).
                float m_use = m_run;
                bool grow = false;
                const float hmx = mx * kLog2e;
                if (m_run == -CUDART_INF_F) {
                    m_use = ref_max(hmx);
                } else if (hmx > m_run + kLazyRescale) {
                    grow = true;
                    m_use = ref_max(hmx);
                }
                exp_pass(m_use);
                s_ready = jj + 1 < n_it && mbar_test_wait(&bars->s_full[half], (uint32_t)((jj + 1) & 1));
                if (__any_sync(0xffffffffu, my_abort)) {
                    any_abort = true;
                    bars->abort = 1;
                    break;
                }
                const float alpha = grow ? exp2_int(m_run - m_use) : 1.f;
                l_half = l_half * alpha + rsum;
                m_run = m_use;
                // P_h goes where P_h of the previous tile was: its PV_h must
                // have completed (and, for a rescale, finished adding into O_h).
                if (jj >= 1) {
                    if (!mbar_wait(&bars->o_done[half], (uint32_t)((jj - 1) & 1), p.timeout_ns, kSitePrefillOFull,
                                   p.err))
                        bars->abort = 1;
                    tc_fence_after();
                }
                if (jj >= 1 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t v[32];
                        tmem_ld32(o_addr + c * 32, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st32(o_addr + c * 32, v);
                    }
                }
                tmem_st32(p_addr, w);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(p_bar[half]);
            }

            // Epilogue: merge the halves, O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / l,
            // m = max(m_0, m_1), l the same combination of the sums (exact
            // powers of two); thread (row, half) writes dims [64 half, 64 half + 64).
            sXch[half * 128 + r] = m_run;
            sXch[(2 + half) * 128 + r] = l_half;
            const bool failed = bar_or(1, 256, any_abort || aborted(bars));
            const float m0 = sXch[r], m1 = sXch[128 + r];
            const float m_row = fmaxf(m0, m1);
            const float f0 = m0 == -CUDART_INF_F ? 0.f : exp2_int(m0 - m_row);
            const float f1 = m1 == -CUDART_INF_F ? 0.f : exp2_int(m1 - m_row);
            const float l_tot = sXch[2 * 128 + r] * f0 + sXch[3 * 128 + r] * f1;
            const bool have = n_it > 0 && !failed;
            if (have) {
                if (!mbar_wait(&bars->o_final, 0, p.timeout_ns, kSitePrefillOFull, p.err)) bars->abort = 1;
                tc_fence_after();
            }
            const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
            const float g0 = f0 * inv_l, g1 = f1 * inv_l;
            const bool partial = p.num_splits > 1;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int col = half * 64 + c * 32;  // output dims [col, col + 32)
                uint32_t v[32], u[32];
                if (have) {
                    tmem_ld32(lane_base + C::kOCol + col, v);
                    tmem_ld32(lane_base + C::kOCol + 128 + col, u);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = u[e] = 0u;
                }
                if (!valid) continue;
                float o[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(v[e]) * g0 + __uint_as_float(u[e]) * g1;
                if (partial) {
                    float* dst = p.ws_o + (((size_t)split * p.T + t) * p.H + h) * C::D + col;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                } else if (p.out_f32) {
                    float* dst = reinterpret_cast<float*>(p.out) + (size_t)t * p.o_st + (size_t)h * p.o_sh + col;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                } else {
                    uint16_t* dst =
                        reinterpret_cast<uint16_t*>(p.out) + (size_t)t * p.o_st + (size_t)h * p.o_sh + col;
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
            if (valid && partial && half == 0)
                p.ws_lse[((size_t)split * p.T + t) * p.H + h] = l_tot > 0.f ? m_row + __log2f(l_tot) : -CUDART_INF_F;
            if (valid && !partial && half == 0 && p.lse)
                p.lse[(size_t)t * p.lse_st + (size_t)h * p.lse_sh] =
                    l_tot > 0.f ? (m_row + __log2f(l_tot)) * kLn2 : -CUDART_INF_F;
        } else {

            for (int jj = 0; jj < n_it; ++jj) {
                const int sb = jj & 1;
                const int j0 = key_block(jj) * C::BN;
                const int jh = j0 + kh;  // first key of this half
                const bool band = band_tile(j0);
                bool my_abort = !mbar_wait(&bars->s_full[sb], (uint32_t)((jj >> 1) & 1), p.timeout_ns, kSitePrefillSFull,
                                           p.err);
                my_abort = __any_sync(0xffffffffu, my_abort || aborted(bars));
                float2 s[32];  // keys (kh + 2e, kh + 2e + 1) of the tile
                float mx = -CUDART_INF_F;
                // raw: s keeps q.k (no bias on this tile); the scale folds into
                // the exponent.  Otherwise s holds sc * q.k + bias.
                const bool raw = !band && pos_scale;
                if (!my_abort) {
                    tc_fence_after();
                    {
                        uint32_t v0[32], v1[32];
                        tmem_ld32(lane_base + sb * C::BN + kh, v0);
                        tmem_ld32(lane_base + sb * C::BN + kh + 32, v1);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            s[e] = make_float2(__uint_as_float(v0[2 * e]), __uint_as_float(v0[2 * e + 1]));
                            s[16 + e] = make_float2(__uint_as_float(v1[2 * e]), __uint_as_float(v1[2 * e + 1]));
                        }
                    }
                    tc_fence_before();
                    if (!raw) {
                        const float2 sc2 = make_float2(sc, sc);
                        if (band && p.vec_bias) {
                            const int bb = nb % C::kBiasBufs;
                            if (!mbar_wait(&bars->bias_full[bb], (uint32_t)((nb / C::kBiasBufs) & 1), p.timeout_ns,
                                           kSitePrefillRelFull, p.err))
                                bars->abort = 1;
                            const uint32_t* wb = wrow + bb * (C::kBiasBytes / 4);
                            uint32_t wv[33];
#pragma unroll
                            for (int i = 0; i < 33; ++i) wv[i] = wb[i];
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const uint32_t pr = __byte_perm(wv[31 - e], wv[32 - e], psel);
                                s[e] = __ffma2_rn(s[e], sc2,
                                                  make_float2(__uint_as_float(pr & 0xffff0000u), __uint_as_float(pr << 16)));
                            }
                            // Every read of this band tile's windows is done.
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&bars->bias_empty[bb]);
                        } else if (band) {
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const int d = pos - (jh + 2 * e);
                                const float b0 = valid && d >= 0 && d < R ? rel_at(p.rel, bias_f32, rel_row + d) : 0.f;
                                const float b1 =
                                    valid && d - 1 >= 0 && d - 1 < R ? rel_at(p.rel, bias_f32, rel_row + d - 1) : 0.f;
                                s[e] = __ffma2_rn(s[e], sc2, make_float2(b0, b1));
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) s[e] = __fmul2_rn(s[e], sc2);
                        }
                    }
                    // Mask (warp-uniform skip when every row of the warp sees the whole half tile).
                    const bool row_full = !valid || (jh >= klo && jh + 64 <= khi);
                    if (!__all_sync(0xffffffffu, row_full)) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int j = jh + 2 * e;
                            if (!row_full && !(j >= klo && j < khi)) s[e].x = -CUDART_INF_F;
                            if (!row_full && !(j + 1 >= klo && j + 1 < khi)) s[e].y = -CUDART_INF_F;
                        }
                    }
                    float mk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mk[i] = fmax3(s[i].x, s[i].y, s[8 + i].x);
#pragma unroll
                    for (int i = 0; i < 8; ++i) mk[i] = fmax3(mk[i], s[8 + i].y, s[16 + i].x);
#pragma unroll
                    for (int i = 0; i < 8; ++i) mk[i] = fmax3(mk[i], s[16 + i].y, s[24 + i].x);
#pragma unroll
                    for (int i = 0; i < 8; ++i) mk[i] = fmaxf(mk[i], s[24 + i].y);
                    mx = fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7]));
                    if (raw) mx *= sc;
                }
                if (my_abort) {
                    any_abort = true;
                    break;
                }
                if (band && p.vec_bias) ++nb;
                // Publish this half's maximum.  The partner's is needed only to
                // confirm the reference maximum (or, before the first visible
                // key, to set it), so the exponentials start from the current
                // reference and are redone in the rare case that it moves.
                const int xb = jj & 1;
                sXch[(xb * 2 + half) * 128 + r] = mx;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->x_full[xb]);
                auto row_max = [&]() -> float {
                    if (!mbar_wait(&bars->x_full[xb], (uint32_t)((jj >> 1) & 1), p.timeout_ns, kSitePrefillXchg, p.err))
                        bars->abort = 1;
                    return fmaxf(mx, sXch[(xb * 2 + (half ^ 1)) * 128 + r]);
                };
                const float c1 = raw ? sl2 : kLog2e;
                uint32_t w[32];
                float rsum = 0.f;
                // This half of P_j (bf16 pairs) and its row sum against the
                // integer reference m (log2 units): 2^(q(s * c1) - m), with the
                // score quantised on a fixed grid so that the subtraction is exact.
                auto exp_pass = [&](float m) {
                    const float offs = kQuantC + (m == -CUDART_INF_F ? 0.f : m);
                    const float2 c12 = make_float2(c1, c1), qc = make_float2(kQuantC, kQuantC),
                                 noff = make_float2(-offs, -offs);
                    float2 rs[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) rs[i] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float2 x = __fadd2_rn(__ffma2_rn(s[e], c12, qc), noff);
                        const float2 pe = make_float2(ex2(x.x), ex2(x.y));
                        rs[e & 3] = __fadd2_rn(rs[e & 3], pe);
                        w[e] = pack_bf16(pe.x, pe.y);
                    }
                    const float2 rs2 = __fadd2_rn(__fadd2_rn(rs[0], rs[1]), __fadd2_rn(rs[2], rs[3]));
                    rsum = rs2.x + rs2.y;
                };
                // Lazy rescaling: the reference maximum m_run (an integer in log2
                // units) only moves when the row maximum exceeds it by more than
                // 8, so P stays below 2^8 and O is rescaled rarely (by an exact
                // power of two); O / l is unchanged.
                float m_use = m_run;
                bool grow = false;
                if (m_run == -CUDART_INF_F) {
                    m_use = ref_max(row_max() * kLog2e);
                    exp_pass(m_use);
                } else {
                    exp_pass(m_run);
                    const float rmx = row_max() * kLog2e;
                    if (rmx > m_run + kLazyRescale) {
                        grow = true;
                        m_use = ref_max(rmx);
                        exp_pass(m_use);
                    }
                }
                const float alpha = grow ? exp2_int(m_run - m_use) : 1.f;
                // This half of P_j over the S columns this thread has already read
                // (PV_{j-2}, the last reader of the buffer, completed before S_j).
                tmem_st32(lane_base + sb * C::BN + kh, w);
                l_half = l_half * alpha + rsum;
                m_run = m_use;

                // Rescale this half of the O row when the reference maximum moved
                // (warp-collective TMEM access): PV_{j-1} must have completed.
                if (jj >= 1 && __any_sync(0xffffffffu, grow)) {
                    if (!mbar_wait(&bars->o_done[(jj - 1) & 1], (uint32_t)(((jj - 1) >> 1) & 1), p.timeout_ns,
                                   kSitePrefillOFull, p.err))
                        bars->abort = 1;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < C::D / 64; ++c) {
                        uint32_t v[32];
                        const uint32_t ta = lane_base + C::kOCol + half * (C::D / 2) + c * 32;
                        tmem_ld32(ta, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st32(ta, v);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(p_bar[sb]);
            }

            // Epilogue: O / l, with l the sum of the two halves' partial sums.
            // (buffer 2: the partner may still read buffer (n_it - 1) % 2 of the last tile)
            sXch[(4 + half) * 128 + r] = l_half;
            const bool failed = bar_or(1, 256, any_abort || aborted(bars));
            const float l_tot = sXch[4 * 128 + r] + sXch[5 * 128 + r];
            const bool have = n_it > 0 && !failed;
            if (have) {
                if (!mbar_wait(&bars->o_final, 0, p.timeout_ns, kSitePrefillOFull, p.err)) bars->abort = 1;
                tc_fence_after();
            }
            const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
            const bool partial = p.num_splits > 1;
#pragma unroll
            for (int c = 0; c < C::D / 64; ++c) {
                const int col = half * (C::D / 2) + c * 32;  // output dims [col, col + 32)
                uint32_t v[32];
                if (have) {
                    tmem_ld32(lane_base + C::kOCol + col, v);
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
                    float* dst = p.ws_o + (((size_t)split * p.T + t) * p.H + h) * C::D + col;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                } else if (p.out_f32) {
                    float* dst = reinterpret_cast<float*>(p.out) + (size_t)t * p.o_st + (size_t)h * p.o_sh + col;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                } else {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + (size_t)t * p.o_st + (size_t)h * p.o_sh + col;
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
            if (valid && partial && half == 0)
                p.ws_lse[((size_t)split * p.T + t) * p.H + h] = l_tot > 0.f ? m_run + __log2f(l_tot) : -CUDART_INF_F;
            if (valid && !partial && half == 0 && p.lse)
                p.lse[(size_t)t * p.lse_st + (size_t)h * p.lse_sh] =
                    l_tot > 0.f ? (m_run + __log2f(l_tot)) * kLn2 : -CUDART_INF_F;
        }
    }

    // Both CTAs are done with TMEM and with each other's barriers.
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 3)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(C::kTmemCols)
                     : "memory");
}

template <int D>
int prefill_pair_smem_bytes() {
    return 1024 + PairCfg<D>::kData + (int)sizeof(PairBars);
}

template <int D>
cudaError_t launch_pair_t(const AttnParams& p, const CUtensorMap* maps, const LaunchShape& s, cudaStream_t stream) {
    auto kern = prefill_pair_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = s.grid;
    cfg.blockDim = dim3((unsigned)s.block);
    cfg.dynamicSmemBytes = (size_t)s.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, maps[0], maps[1], maps[2], maps[3]);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

LaunchShape prefill_pair_shape(const AttnParams& p) {
    LaunchShape s;
    const int tpt = 128 / p.G;
    const int qtiles = (p.max_seqlen_q + tpt - 1) / tpt;
    if (p.B <= kCompactMaxB) {
        // Pairs with rows: at most ceil(qtiles / 2) per request, and at most
        // one partly filled pair per request beyond T / (2 * tpt) full ones.
        const long long per_req = (qtiles + 1) / 2;
        const long long by_rows = ((long long)p.T + 2 * tpt - 1) / (2 * tpt) + p.B;
        const long long n_cl = per_req * p.B < by_rows ? per_req * p.B : by_rows;
        s.grid = dim3((unsigned)(n_cl * 2), p.Hk, p.num_splits);
    } else {
        s.grid = dim3((unsigned)((qtiles + 1) / 2 * 2), p.Hk, p.B * p.num_splits);
    }
    s.block = 384;
    s.smem = p.D == 256 ? prefill_pair_smem_bytes<256>() : prefill_pair_smem_bytes<128>();
    s.nstage = p.D == 256 ? PairCfg<256>::kRing : PairCfg<128>::kRing;
    return s;
}

cudaError_t launch_prefill_pair(const AttnParams& p, const CUtensorMap* maps, const LaunchShape& s,
                                cudaStream_t stream) {
    if (p.D == 128) return launch_pair_t<128>(p, maps, s, stream);
    if (p.D == 256) return launch_pair_t<256>(p, maps, s, stream);
    return cudaErrorInvalidValue;
}

}  // namespace relattn
