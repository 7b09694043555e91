// Prefill / chunked-prefill kernel on the 5th-generation tensor cores.
//
// One CTA per (128-row query tile, kv head, request, split).  Rows are
// GQA-packed token-major: row r of the tile is query token i0 + r / G of
// request b and query head g*G + r % G, so every K/V tile read for kv head g
// serves all G query heads.  CTAs run in clusters of two adjacent query
// tiles that walk one sequence of 128-key tiles (the union of their visible
// ranges, processed from the last to the first: the causal diagonal and the
// bias band come first, so the running maximum settles early) and receive
// every K/V tile through TMA multicast.
//
// Warp roles (384 threads):
//   warps 0, 2 producers: warp 0 loads the K tiles, warp 2 the V tiles,
//              each into its own ring so K never waits behind a V slot.  A tile
//              arrives straight from the paged cache as TMA boxes of one
//              16-key page each (all 64-dim blocks of one kv head, through a
//              5-D view of the cache; two boxes of 8 keys when the cache's
//              pages are not contiguous), one per page wholly inside the
//              cache, multicast to the other CTA of the cluster (the two take
//              turns issuing), with block-table entries fetched a 4-tile
//              window ahead (one coalesced load per window).  The TMA unit's
//              cost is mostly per box (on GB300 about 50 cycles per box plus
//              1.5 per 128-byte row), so whole pages rather than 64-dim blocks
//              per box take it off the critical path.  Keys inside the
//              cache but outside a row's window are finite and the softmax
//              masks them, so only the one group that straddles the cache
//              length goes through zero-filling cp.async (proxy-fenced once
//              landed): keys past it may hold stale, non-finite data.  Tiles
//              are 128-byte swizzled; a slot's full mbarrier takes the TMA
//              bytes plus the producer's arrivals, its empty mbarrier one MMA
//              commit per CTA of the cluster.  The producer loop keeps
//              nothing else in it: no global loads, no divisions.
//   warp 1     bias windows: for each band tile (one that reaches some row's
//              bias band) it stages that tile's rel_logits by TMA into one of
//              two window buffers (one with D = 64) once the softmax warps
//              have released that buffer's previous fill (see below), so the
//              next band tile's windows load while the current one is read.
//   warp 3     MMA issuer (the whole warp runs the loop, one elected lane
//              issues) and TMEM owner.  Per tile and per key half h (keys
//              [64h, 64h + 64)): S_h = Q K_j[64h..]^T (M=128, N=64,
//              K=head_dim, Q read from TMEM) and O_h += P_h V_j[64h..] (P_h
//              read from TMEM, V from shared memory, MN-major); the two
//              halves are independent softmax streams, like two splits of
//              the key range merged at the end.  tcgen05.commit signals
//              completion.
//   warps 4-11 softmax: warps 4-7 take key half 0 of every tile and warps
//              8-11 half 1; warp w reads TMEM lanes 32*(w%4).. so thread
//              (w, lane) owns half h of row 32*(w%4) + lane.  Per tile it
//              reads S_h (and releases the buffer at once, so the next S_h
//              computes during this tile's exponentials), forms sc * q.k +
//              bias (natural units; tiles outside every row's bias band keep
//              the raw q.k and fold the scale into the exponent), masks only
//              when some row of the warp does not see the whole half tile,
//              computes P_h against its half's reference maximum, writes it
//              into TMEM as bf16 pairs and rescales its O_h row when the
//              reference moved.  Each half keeps its own reference maximum,
//              an integer in log2 units (so weights do not depend on the
//              split partition, see kQuantC) that moves lazily (only when the
//              half-row maximum exceeds it by more than 2^8), so no maxima
//              cross between warps during the tiles.  The epilogue merges the
//              halves by exact powers of two and writes the output.  The
//              bias of a band tile is staged by warp 1: one 152-value window
//              per (token, head) row, starting at the 16-byte aligned
//              distance below the row's token sub-box, zero outside [0, R),
//              so the sheared gather becomes a reversed shared-memory read.
// Every mbarrier wait is bounded; on timeout the kernel records the site in
// the device error word and winds down.
//
// TMEM columns: O_0 [0,D), O_1 [D,2D), S_0 and S_1 (64 each), P_0 and P_1
// (32 each: 64 keys as bf16 pairs), Q (D/2: bf16 pairs).  Warps 4-7 copy Q
// into TMEM at the start.
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
// Lazy rescaling threshold in log2 units.
constexpr float kLazyRescale = 8.0f;
// CTAs per cluster: adjacent query tiles that share (multicast) every K/V tile.
constexpr int kCluster = 2;

template <int D>
struct PrefillCfg {
    static constexpr int BN = 128;                  // keys per tile (query tiles are 128 rows)
    static constexpr int kDB = D / 64;              // 64-dim (128-byte) column blocks
    // A K or V tile in shared memory: 8 pages of 16 keys, each two halves of
    // 8 keys, each half kDB swizzle atoms (8 keys x 64 dims, 1 KB): key
    // 16 p + 8 h + r, dims [64 c, 64 c + 64) at p * kPage + h * kHalf + c * 1024
    // + r * 128.  This is the order a 5-D TMA box of one page lands in, and
    // a canonical 128-byte-swizzled operand: K-major (keys = N) with 8-key
    // groups kHalf apart, or MN-major (dims = N) with 64-dim blocks 1 KB apart.
    static constexpr int kHalf = kDB * 1024;
    static constexpr int kPage = 2 * kHalf;
    static constexpr int kTileBytes = 8 * kPage;
    static constexpr int kMmaWarp = 3;
    static constexpr int kSoftThreads = 256;        // warps 4-11
    static constexpr int kThreads = 384;
    static constexpr int kKRing = D == 128 ? 2 : 6;   // K tile slots
    static constexpr int kVRing = D == 128 ? 2 : 4;   // V tile slots (after the K ring)
    static constexpr int kStages = kKRing + kVRing;
    // rel_logits values per staged bias row: at least 128 + 14 (a tile plus the
    // shear of an 8-token sub-box and 16-byte alignment); 152 makes the row
    // pitch 76 words, so the 32 rows of a warp spread over the banks.
    static constexpr int kBiasW = 152;
    // 128 rows, plus up to 16 token sub-boxes each padded to a 128-byte boundary
    static constexpr int kBiasBytes = 128 * kBiasW * 2 + 16 * 128;
    // Band tiles' windows are double-buffered where shared memory allows.
    static constexpr int kBiasBufs = D == 128 ? 2 : 1;
    // Per half and row: the final reference maximum and sum (epilogue merge).
    static constexpr int kXchBytes = 2 * 2 * 128 * 4;
    static constexpr int kData = kStages * kTileBytes + kBiasBufs * kBiasBytes + kXchBytes;
    // TMEM columns: O_0, O_1 (D each), S_0, S_1 (64 each), P_0, P_1 (32 each:
    // 64 keys as bf16 pairs), Q (D / 2: bf16 pairs).  Half h of the softmax
    // (keys [64h, 64h + 64) of every tile) owns S_h, P_h and O_h.
    static constexpr int kTmemCols = 512;
    static constexpr int kOCol = 0;
    static constexpr int kSCol = 2 * D;
    static constexpr int kPCol = 2 * D + 128;
    static constexpr int kQCol = 2 * D + 192;
};

struct PrefillBars {
    uint64_t q_full;
    uint64_t kv_full[10];
    uint64_t kv_empty[10];   // this CTA's MMAs have read the slot's current use (a local commit)
    uint64_t kv_peer[10];    // the other CTA's MMAs have (its producer forwards its kv_empty)
    uint64_t s_full[2];  // per half, one phase per tile: S_h(jj) is in TMEM
    uint64_t s_free1;    // one phase per tile: warps 8-11 have read S_1 (warps 4-7 use the K slot's barrier)
    uint64_t p_full1;    // one phase per tile: P_1 is in TMEM (warps 4-7 use the V slot's barrier)
    uint64_t o_done[2];  // per half, one phase per PV tile: PV_h has read P_h and added into O_h
    uint64_t o_final;  // single phase: every MMA of the CTA has completed
    uint64_t bias_full[2];   // per window buffer, one phase per fill: its rel_logits windows have landed
    uint64_t bias_empty[2];  // per window buffer, one phase per fill: every softmax warp has read them
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ bool aborted(const PrefillBars* bars) {
    return *reinterpret_cast<const volatile int*>(&bars->abort) != 0;
}

// Batches up to this size launch one cluster per (request, pair of query
// tiles) that has rows, found by a scan over cu_seqlens_q; larger ones launch
// max_seqlen_q's tile count for every request and let empty clusters leave.
constexpr int kCompactMaxB = 256;

// A cluster's work: request b, the top query tile of its pair, the request's
// first query token q0, its query and cache lengths.
struct ClusterWork {
    int b, top, q0, sq, sk;
};

// Cluster ci of a compact launch -> its work, or request -1 past the last
// pair.  Requests in order; within a request the pairs go from the last (most
// keys) to the first.  The lengths come from the same scan (one round of
// independent loads: they are on the CTA's start-up path).  Warp-collective:
// every lane gets the same answer.
__device__ __forceinline__ ClusterWork compact_cluster_work(const int32_t* cu, const int32_t* seqk, int B, int TPT,
                                                            int ci) {
    const int lane = threadIdx.x & 31;
    int base = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
        const int bb = b0 + lane;
        int n = 0, c0 = 0, c1 = 0, kl = 0;
        if (bb < B) {
            c0 = __ldg(cu + bb);
            c1 = __ldg(cu + bb + 1);
            kl = __ldg(seqk + bb);
            const int nt = (c1 - c0 + TPT - 1) / TPT;
            n = (nt + kCluster - 1) / kCluster;
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
            ClusterWork w;
            w.b = b0 + src;
            w.top = k * kCluster + kCluster - 1;
            w.q0 = __shfl_sync(0xffffffffu, c0, src);
            w.sq = __shfl_sync(0xffffffffu, c1 - c0, src);
            w.sk = __shfl_sync(0xffffffffu, kl, src);
            return w;
        }
        base += tot;
    }
    ClusterWork none;
    none.b = -1;
    none.top = none.q0 = none.sq = none.sk = 0;
    return none;
}

// VEC: rel_logits rows are 16-byte aligned (R % 8 == 0), so bias windows are
// staged by 16-byte copies; otherwise the bias is read per element.
template <int D, bool VEC>
__global__ void __launch_bounds__(PrefillCfg<D>::kThreads, 1)
    prefill_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_rel) {
    using C = PrefillCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sKV = smem;
    uint8_t* sBias = sKV + C::kStages * C::kTileBytes;
    float* sM = reinterpret_cast<float*>(sBias + C::kBiasBufs * C::kBiasBytes);  // [2 halves][128 rows]
    float* sL = sM + 2 * 128;                                                      // [2 halves][128 rows]
    PrefillBars* bars = reinterpret_cast<PrefillBars*>(sBias + C::kBiasBufs * C::kBiasBytes + C::kXchBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G, TPT = 128 / G;
    const int crank = (int)cluster_ctarank();
    const int g = blockIdx.y;
    const int S = p.num_splits;
    int qt, b, split, q0, sq, sk;
    if (p.B <= kCompactMaxB) {
        const ClusterWork w =
            compact_cluster_work(p.cu_seqlens_q, p.cache_seqlens, p.B, TPT, (int)(blockIdx.x / kCluster));
        if (w.b < 0) return;  // past the last pair (the same in every CTA of the cluster)
        b = w.b;
        qt = w.top - crank;
        split = blockIdx.z;
        q0 = w.q0;
        sq = w.sq;
        sk = w.sk;
    } else {
        qt = gridDim.x - 1 - blockIdx.x;  // longest tiles first
        b = blockIdx.z / S;
        split = blockIdx.z % S;
        q0 = p.cu_seqlens_q[b];
        sq = p.cu_seqlens_q[b + 1] - q0;
        sk = p.cache_seqlens[b];
    }
    const int i0 = qt * TPT;
    const int i1 = min(sq, i0 + TPT);
    const int n_rows = max(i1 - i0, 0) * G;
    const int off = sk - sq;
    const int pos_min = i0 + off, pos_max = i1 - 1 + off;
    const int R = p.R;

    // The kCluster CTAs of a cluster hold adjacent query tiles of one (request,
    // kv head, split) and walk one shared sequence of K/V tiles: the union of
    // their visible ranges.  Rank r holds tile qt_top - r; CTAs whose tile is
    // past the request's end are inactive (no loads, no MMAs).
    const int qt_top = qt + crank;
    uint32_t active = 0;
#pragma unroll
    for (int r = 0; r < kCluster; ++r)
        if ((qt_top - r) * TPT < sq) active |= 1u << r;
    const bool me_active = (active >> crank) & 1;
    const int n_act = __popc(active);
    const int my_idx = __popc(active & ((1u << crank) - 1));
    const uint16_t mc_mask = (uint16_t)active;
    const int u_i0 = (qt_top - (kCluster - 1)) * TPT;                       // lowest tile of the cluster
    const int u_i1 = min(sq, (qt_top - (active ? __ffs(active) - 1 : 0) + 1) * TPT);  // end of the highest active one

    // Keys any row of the cluster's tiles may see, as 128-key tiles, split contiguously.
    int hi = sk, lo = 0;
    if (active) {
        const int u_pmin = u_i0 + off, u_pmax = u_i1 - 1 + off;
        if (p.causal) hi = min(hi, u_pmax + 1);
        if (p.wr >= 0) hi = min(hi, u_pmax + p.wr + 1);
        if (p.wl >= 0) lo = max(0, u_pmin - p.wl);
    }
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
    // Does key tile [j0, j0+128) reach the bias band 0 <= pos - j < R of some row?
    auto band_tile = [&](int j0) { return R > 0 && pos_max - j0 >= 0 && pos_min - (j0 + C::BN - 1) < R; };

    // A cluster with no rows at all touches no shared memory of another CTA:
    // both of its CTAs leave at once (the same test in both).
    if (active == 0) return;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, C::kSoftThreads / 2);
        for (int i = 0; i < C::kStages; ++i) {
            // producer lanes + the expect_tx arrival, plus one arrival per
            // warp of softmax half 0: a K slot's once that half has read the
            // previous tile's S_0 (its buffer may be overwritten), a V slot's
            // once P_0 of its tile is in TMEM.  The MMA thread then waits once
            // before S_0 and once before PV_0.
            mbar_init(&bars->kv_full[i], 33 + 4);
            mbar_init(&bars->kv_empty[i], 1);
            mbar_init(&bars->kv_peer[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->o_done[i], 1);
        }
        mbar_init(&bars->s_free1, 4);
        mbar_init(&bars->p_full1, 4);
        mbar_init(&bars->o_final, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->bias_full[i], 1);
            mbar_init(&bars->bias_empty[i], C::kSoftThreads / 32);
        }
        bars->abort = 0;
        fence_mbar_init();
    }
    // The producers load their first block-table windows now: the first K
    // and V boxes wait on them.  Block-table windows of 4 tiles: lane l holds
    // the physical block of 16-key group l % 8 of tile w0 + l / 8; the next
    // window is fetched one window ahead (32 consecutive entries when BS is 16).
    const int32_t* bt = p.block_table + (size_t)b * p.bt_stride;
    auto load_win = [&](int w0) -> int {
        int v = 0;
        const int jw = w0 + (lane >> 3);
        if (jw < n_it) {
            const int jg = key_block(jw) * C::BN + 16 * (lane & 7);
            // (a key past the table's width, i.e. cache_seqlens > MB * BS,
            // reads no entry: the clamp below then keeps block 0)
            if (jg < sk && jg / p.BS < p.max_blocks) v = __ldg(bt + jg / p.BS);
        }
        return v;
    };
    int win_cur = 0, win_nxt = 0;
    if (me_active && (warp == 0 || warp == 2)) {
        win_cur = load_win(0);
        win_nxt = load_win(4);
    }

    if (me_active && warp == C::kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars->tmem_base)),
                     "n"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // This CTA's barriers are initialised.  The other CTA multicasts into its
    // ring and arrives on its barriers only after its cluster_wait has seen
    // this arrival; until then each CTA works on its own (first fills of
    // every ring slot are loaded by each CTA for itself).
    cluster_arrive();
    if (!me_active) {
        cluster_wait();
        cluster_sync();
        return;
    }
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------ Q/K and V producers
        // Warp 0 loads the K ring, warp 2 the V ring, so a K tile never
        // queues behind a V slot the softmax still holds.  One TMA box per
        // 16-key page wholly inside the cache (both 8-key halves in one box
        // when the cache's pages are contiguous, else one box per half),
        // multicast to the cluster, the active CTAs taking turns; the group
        // that straddles the cache length goes through zero-filling
        // cp.async, so V rows past it hold zeros, never stale cache contents
        // (0 * NaN would poison the row).
        const bool is_v = warp == 2;
        constexpr int kChunks = D / 8;
        constexpr int kRows = 32 / kChunks;
        constexpr int kPerPage = 16 / kRows;
        const int lrow = lane / kChunks, lchunk = lane % kChunks;
        const uint16_t* cache = reinterpret_cast<const uint16_t*>(is_v ? p.v_cache : p.k_cache);
        const CUtensorMap* tmap = is_v ? &tm_v : &tm_k;
        const uint64_t pol_last = l2_policy_evict_last();
        const uint32_t col_off = (lchunk >> 3) * 1024;
        // Within a 16-row group, row (kk*kRows + lrow) & 7 == ((kk*kRows) & 7) | lrow,
        // so the 128-byte swizzle is the per-lane constant cx XOR a compile-time one.
        const long long lane_off = (long long)lrow * p.c_s1 + lchunk * 8;
        const long long row_step = (long long)kRows * p.c_s1;
        const uint32_t cx = (uint32_t)((lchunk & 7) ^ lrow);
        const uint32_t dst_lane = col_off + lrow * 128;
        if (lane == 0) tma_prefetch_desc(tmap);
        // At most one cp.async group (the partial groups of a tile) is in
        // flight; it is retired (landed, proxy-fenced, one arrival per lane)
        // after the next tile has been issued, or before the producer blocks
        // on a full ring.
        uint64_t* pend = nullptr;
        auto retire = [&](int newer) {
            cp_async_wait(newer);
            fence_proxy_async_smem();
            mbar_arrive(pend);
            pend = nullptr;
        };
        // TMA lanes: lane -> (16-key group lane / nbox, half lane % nbox),
        // nbox = 1 when a box holds the whole page.
        const int nbox = p.kv_merged ? 1 : 2;
        const int t_pg = lane / nbox, t_h = lane % nbox;
        const int ring0 = is_v ? C::kKRing : 0;
        const int ring = is_v ? C::kVRing : C::kKRing;
        int sidx = 0;
        uint32_t eph = 1;  // parity of the empty phase to wait for
        // The slot's previous use is released by this CTA's MMA commit
        // (kv_empty) and, with two active CTAs, by the other CTA's, which its
        // producer forwards here (kv_peer); this producer forwards its own in
        // turn.  (The MMA thread then only commits locally: a multicast
        // commit stalls the tensor pipe.)
        const uint32_t peer_bar0 = mapa_shared(smem_u32(&bars->kv_peer[ring0]), (uint32_t)crank ^ 1u);
        // Never block on a full ring while holding copies whose landing has
        // not been signalled: the consumer may be waiting for exactly those.
        auto wait_slot = [&](uint64_t* bar, uint32_t par, int site) {
            if (!mbar_try_wait(bar, par)) {
                if (pend) retire(0);
                if (!mbar_wait(bar, par, p.timeout_ns, site, p.err)) bars->abort = 1;
            }
        };
        auto release_to_peer = [&](int slot, uint32_t par) {
            if (lane == 0) mbar_arrive_remote(peer_bar0 + (uint32_t)(slot - ring0) * 8u);
            wait_slot(&bars->kv_peer[slot], par, kSitePrefillKEmpty);
        };
        bool waited = false;  // this thread's cluster_wait is done
        for (int jj = 0; jj < n_it; ++jj) {
            // Multicast loads and releases to the other CTA from the second
            // use of a slot on.
            if (jj == ring) {
                cluster_wait();
                waited = true;
            }
            const bool mc = jj >= ring;
            const int slot = ring0 + sidx;
            wait_slot(&bars->kv_empty[slot], eph, kSitePrefillKEmpty);
            if (jj >= ring && n_act == 2) release_to_peer(slot, eph);
            if (++sidx == ring) {
                sidx = 0;
                eph ^= 1;
            }
            if (__any_sync(0xffffffffu, aborted(bars))) break;
            if (jj >= 4 && (jj & 3) == 0) {
                win_cur = win_nxt;
                win_nxt = load_win(jj + 4);
            }
            const int wl = (jj & 3) * 8;
            const int j0 = key_block(jj) * C::BN;
            // Bit pg set: 16-key group pg is fully visible (whole-box TMA).
            uint32_t full_mask = 0;
#pragma unroll
            for (int pg = 0; pg < 8; ++pg) {
                const int jg = j0 + 16 * pg;
                if (jg + 16 <= sk) full_mask |= 1u << pg;
            }
            uint64_t* full_bar = &bars->kv_full[slot];
            uint8_t* tile = sKV + slot * C::kTileBytes;
            if (lane == 0) mbar_arrive_expect_tx(full_bar, (uint32_t)__popc(full_mask) * C::kDB * 2048u);
            __syncwarp();
            const int blk_t = min(max(__shfl_sync(0xffffffffu, win_cur, wl + (t_pg & 7)), 0), p.NB - 1);
            if (lane < 8 * nbox && ((full_mask >> t_pg) & 1) && (!mc || lane % n_act == my_idx)) {
                const int slot_in_blk = (j0 + 16 * t_pg) % p.BS;
                // merged view (64, 8, kDB, NB * BS / 8, Hk): half-page blk * BS / 8 + slot / 8;
                // split view (64, BS, kDB, Hk, NB): slot, head, block.
                uint8_t* dst = tile + t_pg * C::kPage + (p.kv_merged ? 0 : t_h * C::kHalf);
                const int c1 = p.kv_merged ? 0 : slot_in_blk + 8 * t_h;
                const int c3 = p.kv_merged ? blk_t * (p.BS >> 3) + (slot_in_blk >> 3) : g;
                const int c4 = p.kv_merged ? g : blk_t;
                if (mc)
                    tma_load_5d_mc(dst, tmap, full_bar, 0, c1, 0, c3, c4, mc_mask, pol_last);
                else
                    tma_load_5d(dst, tmap, full_bar, 0, c1, 0, c3, c4, pol_last);
            }
            const bool part = full_mask != 0xffu;
            if (part) {
                const uint32_t dst_tile = smem_u32(tile) + dst_lane;
                for (int pg = 0; pg < 8; ++pg) {
                    if ((full_mask >> pg) & 1) continue;
                    const int jg = j0 + 16 * pg;
                    const int blk = min(max(__shfl_sync(0xffffffffu, win_cur, wl + pg), 0), p.NB - 1);
                    const uint16_t* src = cache + (long long)blk * p.c_s0 + (long long)(jg % p.BS) * p.c_s1 +
                                          (long long)g * p.c_s2 + lane_off;
#pragma unroll
                    for (int kk = 0; kk < kPerPage; ++kk) {
                        const int row = kk * kRows + lrow;  // key jg + row
                        const bool valid = jg + row < sk;
                        const uint32_t dst = dst_tile + pg * C::kPage + ((kk * kRows) >> 3) * C::kHalf +
                                             ((kk * kRows) & 7) * 128 + ((cx ^ ((kk * kRows) & 7)) << 4);
                        cp_async_16(dst, valid ? src : cache, valid ? 16u : 0u, pol_last);
                        src += row_step;
                    }
                }
                cp_async_commit();
            }
            if (pend) retire(part ? 1 : 0);
            if (part) {
                pend = full_bar;
            } else {
                __syncwarp();
                if (lane == 0) mbar_arrive_cnt(full_bar, 32);
            }
        }
        if (pend) retire(0);
        // (also when the loop stopped early on an abort: every thread waits
        // once between its cluster arrivals)
        if (!waited) cluster_wait();
        // Wait until both CTAs have released each slot for the last time
        // (forwarding this CTA's release): afterwards no arrival from the
        // other CTA is still travelling to this one.
        if (!__any_sync(0xffffffffu, aborted(bars))) {
            for (int i = 0; i < min(ring, n_it); ++i) {
                const int last = i + ring * ((n_it - 1 - i) / ring);
                const uint32_t par = (uint32_t)(last / ring) & 1u;
                wait_slot(&bars->kv_empty[ring0 + i], par, kSitePrefillKEmpty);
                if (n_act == 2) release_to_peer(ring0 + i, par);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ bias windows
        cluster_wait();
        // Band tile n's rel_logits, once every softmax warp has finished
        // reading band tile n-1's: one TMA box per token sub-box of TS tokens
        // (all G heads), rows of kBiasW distances from the 16-byte aligned
        // distance below the sub-box's smallest one.
        if (VEC && lane == 0) {
            const int TS = p.bias_ts, n_sub = TPT / TS;
            const int sub_bytes = (TS * G * C::kBiasW * 2 + 127) & ~127;
            const uint64_t pol = l2_policy_evict_first();
            int nbi = 0;
            for (int jj = 0; jj < n_it; ++jj) {
                const int j0 = key_block(jj) * C::BN;
                if (!band_tile(j0)) continue;
                // Buffer bb's fill number `use` waits for the softmax to release fill use - 1.
                const int bb = nbi % C::kBiasBufs, use = nbi / C::kBiasBufs;
                if (use > 0 && !mbar_wait(&bars->bias_empty[bb], (use - 1) & 1, p.timeout_ns, kSitePrefillRelEmpty,
                                          p.err)) {
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
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------ MMA issuer
        cluster_wait();
        // The whole warp runs the loop (converged); one elected lane issues.
        if (n_it > 0) {
            constexpr uint32_t idS = umma_idesc_bf16(128, 64, false);
            constexpr uint32_t idPV = umma_idesc_bf16(128, D, true);
            const uint32_t aKV = smem_u32(sKV);
            bool ok = mbar_wait_warp(&bars->q_full, 0, p.timeout_ns, kSitePrefillLoadQ, p.err);
            // Descriptors are formed before each wait, so the MMAs of a group
            // issue back to back.  A descriptor's low bits hold address / 16,
            // so a byte offset inside shared memory adds offset / 16.  Keys
            // [64h, 64h + 64) of a tile are its pages 4h .. 4h + 3.
            const uint64_t dK0 = umma_desc_sw128(aKV, 16, C::kHalf);
            const uint64_t dV0 = umma_desc_sw128(aKV, 1024, C::kHalf);
            constexpr uint64_t kHalfK = (uint64_t)((4 * C::kPage) >> 4);
            const uint32_t aq = tmem + C::kQCol;
            // O_h += P_h(t) V_t[64h, 64h + 64): four K-steps of 16 keys.  Half
            // 0's P is covered by the V slot's full barrier (it also counts the
            // arrivals of warps 4-7), half 1's by p_full1.
            auto issue_pv = [&](int t) {
                const int slot = C::kKRing + t % C::kVRing;
                const uint64_t dv = dV0 + (uint64_t)((slot * C::kTileBytes) >> 4);
                uint64_t dV[C::BN / 16];
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk) dV[kk] = dv + (uint64_t)((kk * C::kPage) >> 4);
                const uint32_t o0 = tmem + C::kOCol, o1 = tmem + C::kOCol + D;
                const uint32_t p0 = tmem + C::kPCol, p1 = tmem + C::kPCol + 32;
                ok = ok && mbar_wait_warp(&bars->kv_full[slot], (t / C::kVRing) & 1, p.timeout_ns, kSitePrefillPFull,
                                          p.err);
                if (!ok) return;
                tc_fence_after();
                if (t > 0)
                    umma_ts<1>(o0, p0, dV[0], idPV);
                else
                    umma_ts<0>(o0, p0, dV[0], idPV);
#pragma unroll
                for (int kk = 1; kk < 4; ++kk) umma_ts<1>(o0, p0 + 8 * kk, dV[kk], idPV);
                umma_commit(&bars->o_done[0]);
                ok = mbar_wait_warp(&bars->p_full1, t & 1, p.timeout_ns, kSitePrefillPFull, p.err);
                if (!ok) return;
                tc_fence_after();
                if (t > 0)
                    umma_ts<1>(o1, p1, dV[4], idPV);
                else
                    umma_ts<0>(o1, p1, dV[4], idPV);
#pragma unroll
                for (int kk = 1; kk < 4; ++kk) umma_ts<1>(o1, p1 + 8 * kk, dV[4 + kk], idPV);
                umma_commit(&bars->o_done[1]);
                umma_commit(&bars->kv_empty[slot]);
            };
            // S_h(jj) = Q K_jj[64h, 64h + 64)^T (N = 64).  S_0 waits on the K
            // slot's full barrier, which also counts warps 4-7 having read
            // S_0(jj - 1); S_1 waits on s_free1.  Tile jj's K slot depends on
            // jj % 2 only when the K ring has two slots: unroll by two so the
            // descriptors are constants.
            auto issue_s = [&](int jj, auto par) {
                constexpr int P = decltype(par)::value;
                const int slot_rt = C::kKRing == 2 ? P : jj % C::kKRing;
                const uint64_t dk = dK0 + (uint64_t)((slot_rt * C::kTileBytes) >> 4);
                uint64_t dK[D / 16];
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) dK[kk] = dk + (uint64_t)((((kk >> 2) * 1024) + (kk & 3) * 32) >> 4);
                const uint32_t s0 = tmem + C::kSCol, s1 = tmem + C::kSCol + 64;
                ok = ok && mbar_wait_warp(&bars->kv_full[slot_rt], (jj / C::kKRing) & 1, p.timeout_ns,
                                          kSitePrefillKFull, p.err);
                if (!ok) return;
                tc_fence_after();
                umma_ts<0>(s0, aq, dK[0], idS);
#pragma unroll
                for (int kk = 1; kk < D / 16; ++kk) umma_ts<1>(s0, aq + 8 * kk, dK[kk], idS);
                umma_commit(&bars->s_full[0]);
                ok = mbar_wait_warp(&bars->s_free1, jj & 1, p.timeout_ns, kSitePrefillSFull, p.err);
                if (!ok) return;
                tc_fence_after();
                umma_ts<0>(s1, aq, dK[0] + kHalfK, idS);
#pragma unroll
                for (int kk = 1; kk < D / 16; ++kk) umma_ts<1>(s1, aq + 8 * kk, dK[kk] + kHalfK, idS);
                umma_commit(&bars->s_full[1]);
                umma_commit(&bars->kv_empty[slot_rt]);
            };
            using I0 = std::integral_constant<int, 0>;
            using I1 = std::integral_constant<int, 1>;
            for (int jj = 0; jj < n_it && ok; jj += 2) {
                issue_s(jj, I0{});
                if (!ok) break;
                if (jj >= 1) issue_pv(jj - 1);
                if (jj + 1 < n_it) {
                    issue_s(jj + 1, I1{});
                    if (!ok) break;
                    issue_pv(jj);
                }
            }
            // The last tile's PV follows.
            if (ok) issue_pv(n_it - 1);
            // The epilogue may be two or more o_done phases behind, where a
            // parity wait cannot tell phases apart: give it its own barrier.
            umma_commit(&bars->o_final);
            if (!ok) bars->abort = 1;
        }
        __syncwarp();
    } else if (warp >= 4) {
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

        // Warps 4-7 copy the Q tile into TMEM: row r to lane r, bf16 pairs per
        // column (zeros past the tile's rows).  The loads overlap the first K
        // tile's flight (issued before the barrier the other warps wait at).
        if (half == 0) {
            uint32_t qv[D / 64][32];
            const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.q) +
                                                              (size_t)t * p.q_st + (size_t)h * p.q_sh);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const uint4 v = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
                qv[c / 8][4 * (c % 8)] = v.x;
                qv[c / 8][4 * (c % 8) + 1] = v.y;
                qv[c / 8][4 * (c % 8) + 2] = v.z;
                qv[c / 8][4 * (c % 8) + 3] = v.w;
            }
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tmem_st32(lane_base + C::kQCol + 32 * c, qv[c]);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->q_full);
        }
        cluster_wait();

        // Bias windows (VEC): a band tile's rel_logits arrive by TMA as rows of
        // kBiasW values, one row per (token, head) of the tile, each starting at
        // the 16-byte aligned distance below the smallest distance its token
        // sub-box needs (zero-filled outside [0, R)).  Key k of the tile reads
        // element e_r + 127 - k of row r.
        const int TS = p.bias_ts;
        const int sub_bytes = (TS * G * C::kBiasW * 2 + 127) & ~127;  // TMA destinations are 128-byte aligned
        const int i_sub = (i_rel / TS) * TS;
        const int e_r = (i_rel - i_sub) + ((i0 + i_sub + off - 127) & 7);
        // This half's 64 keys read elements base_h - k (k = 0..63), i.e. the
        // 32-bit words W0 - 31 .. W0 + 1 of the row; key pair (2m, 2m+1) sits
        // in word W0 - m, or straddles words W0 - m and W0 - m + 1 when
        // base_h is even (one byte permute either way).
        const int base_h = e_r + 127 - kh;
        const uint32_t* wrow = reinterpret_cast<const uint32_t*>(sBias + (i_rel / TS) * sub_bytes +
                                                                 (r - i_sub * G) * (C::kBiasW * 2)) +
                               (((base_h - 1) >> 1) - 31);
        const uint32_t psel = ((base_h - 1) & 1) ? 0x5432u : 0x3210u;
        int nb = 0;  // band tiles consumed
        bool s_ready = false;  // S_h of the next tile seen complete during this one
        // This half's S, P and O in TMEM.  Its S buffer is free again once its
        // four warps have read it: warps 4-7 say so on the next tile's K slot
        // barrier (the MMA thread waits on that one before S_0 anyway), warps
        // 8-11 on s_free1.  The first S needs no read, so arrive for it now.
        const uint32_t s_addr = lane_base + C::kSCol + 64 * half;
        const uint32_t p_addr = lane_base + C::kPCol + 32 * half;
        const uint32_t o_addr = lane_base + C::kOCol + D * half;
        if (n_it > 0 && lane == 0) mbar_arrive(half == 0 ? &bars->kv_full[0] : &bars->s_free1);

        for (int jj = 0; jj < n_it; ++jj) {
            const int j0 = key_block(jj) * C::BN;
            const int jh = j0 + kh;  // first key of this half
            const bool band = band_tile(j0);
            // S_h(jj)'s barrier was usually seen complete already, tested
            // during the previous tile's exponentials (a wait on a completed
            // barrier still costs ~100 cycles).
            const bool my_abort =
                (!s_ready && !mbar_wait(&bars->s_full[half], jj & 1, p.timeout_ns, kSitePrefillSFull, p.err)) ||
                aborted(bars);
            float2 s[32];  // keys (kh + 2e, kh + 2e + 1) of the tile
            float mx = -CUDART_INF_F;
            // raw: s keeps q.k (no bias on this tile); the scale folds into
            // the exponent.  Otherwise s holds sc * q.k + bias.
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
                if (lane == 0 && jj + 1 < n_it)
                    mbar_arrive(half == 0 ? &bars->kv_full[(jj + 1) % C::kKRing] : &bars->s_free1);

                if (!raw) {
                    const float2 sc2 = make_float2(sc, sc);
                    if (band) {
                        if constexpr (VEC) {
                            const int bb = nb % C::kBiasBufs;
                            if (!mbar_wait(&bars->bias_full[bb], (nb / C::kBiasBufs) & 1, p.timeout_ns,
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
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const int d = pos - (jh + 2 * e);
                                const float b0 = valid && d >= 0 && d < R ? rel_at(p.rel, bias_f32, rel_row + d) : 0.f;
                                const float b1 =
                                    valid && d - 1 >= 0 && d - 1 < R ? rel_at(p.rel, bias_f32, rel_row + d - 1) : 0.f;
                                s[e] = __ffma2_rn(s[e], sc2, make_float2(b0, b1));
                            }
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
            if (band) ++nb;
            const float c1 = raw ? sl2 : kLog2e;
            uint32_t w[32];
            float rsum = 0.f;
            // This half of P_j (bf16 pairs) and its row sum against the
            // integer reference m (log2 units): 2^(q(s * c1) - m), with the
            // score quantised on a fixed grid so that the subtraction is exact.
            auto exp_pass = [&](float m) {
                const float off = kQuantC + (m == -CUDART_INF_F ? 0.f : m);
                const float2 c12 = make_float2(c1, c1), qc = make_float2(kQuantC, kQuantC),
                             noff = make_float2(-off, -off);
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
            // Each half keeps its own reference maximum m_run (an integer in
            // log2 units), so no maxima cross between warps.  It moves lazily:
            // only when this half-row's maximum exceeds it by more than 8, so
            // P stays below 2^8 and O_h is rescaled rarely (by an exact power
            // of two).  The halves are merged in the epilogue.
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
            s_ready = jj + 1 < n_it && mbar_test_wait(&bars->s_full[half], (jj + 1) & 1);
            if (__any_sync(0xffffffffu, my_abort)) {
                any_abort = true;
                bars->abort = 1;
                break;
            }
            const float alpha = grow ? exp2_int(m_run - m_use) : 1.f;
            l_half = l_half * alpha + rsum;
            m_run = m_use;
            // P_h(jj) goes where P_h(jj - 1) was: PV_h(jj - 1) must have read
            // it (and, for a rescale, finished adding into O_h).
            if (jj >= 1) {
                if (!mbar_wait(&bars->o_done[half], (jj - 1) & 1, p.timeout_ns, kSitePrefillOFull, p.err))
                    bars->abort = 1;
                tc_fence_after();
            }
            // Rescale this thread's O_h row when its reference moved
            // (warp-collective TMEM access).
            if (jj >= 1 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
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
            if (lane == 0) mbar_arrive(half == 0 ? &bars->kv_full[C::kKRing + jj % C::kVRing] : &bars->p_full1);
        }

        // Epilogue: merge the halves, O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / l
        // with m = max(m_0, m_1) and l the same combination of the half-row
        // sums (exact powers of two).  Thread (row, half) writes output dims
        // [half D/2, half D/2 + D/2).
        sM[half * 128 + r] = m_run;
        sL[half * 128 + r] = l_half;
        const bool failed = bar_or(1, C::kSoftThreads, any_abort || aborted(bars));
        const float m0 = sM[r], m1 = sM[128 + r];
        const float m_row = fmaxf(m0, m1);
        const float f0 = m0 == -CUDART_INF_F ? 0.f : exp2_int(m0 - m_row);
        const float f1 = m1 == -CUDART_INF_F ? 0.f : exp2_int(m1 - m_row);
        const float l_tot = sL[r] * f0 + sL[128 + r] * f1;
        const bool have = n_it > 0 && !failed;
        if (have) {
            if (!mbar_wait(&bars->o_final, 0, p.timeout_ns, kSitePrefillOFull, p.err)) bars->abort = 1;
            tc_fence_after();
        }
        const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
        const float g0 = f0 * inv_l, g1 = f1 * inv_l;
        const bool partial = p.num_splits > 1;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            const int col = half * (D / 2) + c * 32;  // output dims [col, col + 32)
            uint32_t v[32], u[32];
            if (have) {
                tmem_ld32(lane_base + C::kOCol + col, v);
                tmem_ld32(lane_base + C::kOCol + D + col, u);
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
                float* dst = p.ws_o + (((size_t)split * p.T + t) * p.H + h) * D + col;
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
            p.ws_lse[((size_t)split * p.T + t) * p.H + h] = l_tot > 0.f ? m_row + __log2f(l_tot) : -CUDART_INF_F;
        if (valid && !partial && half == 0 && p.lse)
            p.lse[(size_t)t * p.lse_st + (size_t)h * p.lse_sh] =
                l_tot > 0.f ? (m_row + __log2f(l_tot)) * kLn2 : -CUDART_INF_F;
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(C::kTmemCols)
                     : "memory");
    cluster_sync();
}

template <int D>
int prefill_smem_bytes() {
    return 1024 + PrefillCfg<D>::kData + (int)sizeof(PrefillBars);
}

template <int D, bool VEC>
cudaError_t launch_t(const AttnParams& p, const CUtensorMap* maps, const LaunchShape& s, cudaStream_t stream) {
    auto kern = prefill_kernel<D, VEC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = s.grid;
    cfg.blockDim = dim3((unsigned)s.block);
    cfg.dynamicSmemBytes = (size_t)s.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, maps[0], maps[1], maps[2]);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

int prefill_bias_window() { return PrefillCfg<128>::kBiasW; }

LaunchShape prefill_shape(const AttnParams& p) {
    LaunchShape s;
    const int tpt = 128 / p.G;
    const int qtiles = (p.max_seqlen_q + tpt - 1) / tpt;
    if (p.B <= kCompactMaxB) {
        // Pairs with rows: at most ceil(qtiles / 2) per request, and at most
        // one partly filled pair per request beyond T / (2 * tpt) full ones.
        const long long per_req = (qtiles + kCluster - 1) / kCluster;
        const long long by_rows = ((long long)p.T + kCluster * tpt - 1) / (kCluster * tpt) + p.B;
        const long long n_cl = per_req * p.B < by_rows ? per_req * p.B : by_rows;
        s.grid = dim3((unsigned)(n_cl * kCluster), p.Hk, p.num_splits);
    } else {
        s.grid = dim3((qtiles + kCluster - 1) / kCluster * kCluster, p.Hk, p.B * p.num_splits);
    }
    s.block = PrefillCfg<128>::kThreads;
    s.smem = p.D == 128 ? prefill_smem_bytes<128>() : prefill_smem_bytes<64>();
    s.nstage = p.D == 128 ? PrefillCfg<128>::kStages : PrefillCfg<64>::kStages;
    return s;
}

cudaError_t launch_prefill(const AttnParams& p, const CUtensorMap* maps, const LaunchShape& s,
                           cudaStream_t stream) {
    const bool vec = p.vec_bias != 0;
    if (p.D == 128) return vec ? launch_t<128, true>(p, maps, s, stream) : launch_t<128, false>(p, maps, s, stream);
    if (p.D == 64) return vec ? launch_t<64, true>(p, maps, s, stream) : launch_t<64, false>(p, maps, s, stream);
    return cudaErrorInvalidValue;
}

}  // namespace relattn
