// fwd.cu -- forward pass of the attention core on sm_103a.
//
// Computes, for every (query head, 128-query block) tile,
//     S = scale * Q K^T  (causal: key j visible to query i iff j <= i),
//     P = softmax(S) row-wise, P_d = P * M / (1 - p)  (softmax dropout),
//     O = P_d V,  LSE_i = ln sum_j exp(S_ij),
// and stores only O and LSE: the scores, probabilities and mask never reach
// global memory.  This is the attention core that selective activation
// recomputation discards after the forward pass ("Reducing Activation
// Recomputation in Large Transformer Models", Key takeaways, fourth bullet;
// "Recomputing Activations", "Memory for compute, selectively").
//
// Persistent: one CTA per SM walks its share of the tiles (sched.cuh), with
// one MMA stream across tile boundaries.  Structure of a CTA (384 threads):
//   warp 0  TMA: lane 0 the K ring over all blocks of all tiles, lane 1 each
//           tile's Q into the free one of two Q buffers (one for d = 160)
//   warp 2  TMA: V blocks into their own ring
//   warp 1  one thread issues tcgen05 MMAs: S_j = Q K_j^T into one of two
//           TMEM score buffers, then O += P_{j-1} V_{j-1} with P read from TMEM
//   warps 4-11  two warpgroups on the same 128 query rows (TMEM lanes), one
//           per half of the 128 keys of a block: online softmax in the log2
//           domain, dropout from Philox, P_d written back to TMEM as bf16
//           inside the half's own score columns; epilogue O / l -> bf16
//           staged in shared memory and written by one TMA store per tile
//           (d <= 128; d = 160 stores rows from registers)
// For d <= 128 the two halves of a row are independent online softmaxes: each
// keeps its own running maximum and sum, and its own O accumulator in TMEM
// (O_h += P_h V_h, V_h the half's 64 rows of the block), so neither waits on
// the other inside a tile; the epilogue merges them,
//     m = max(m_0, m_1),  l = sum_h l_h 2^(m_h - m),  O = sum_h O_h 2^(m_h - m) / l.
// For d = 160 TMEM has no room for a second accumulator: the halves share one
// O and swap their block maxima (and the final sums) through TMEM columns.
// The running maximum is only moved (and O rescaled in TMEM) when it grows by
// more than 2^8, so most blocks skip the rescale; O / l is exact either way.
#include "kernels.h"
#include "philox.cuh"
#include "ptx.cuh"
#include "sched.cuh"
#include "tile.cuh"

namespace ac {

namespace {

template <int D>
struct FwdCfg {
    using G = TileGeom<D>;
    static constexpr uint32_t TILE = G::template tile_bytes<128>();
    static constexpr uint32_t CHUNK = G::template chunk_bytes<128>();
    // K and V rings: a block's load is issued when the block ST earlier has
    // been consumed, so ST blocks of work must cover one TMA round trip.  Two Q
    // buffers (where they fit) let the next tile's Q land during this tile.
    // O is staged in shared memory and written by one coalesced TMA store per
    // tile where the stage fits (d <= 128); d = 160 stores rows from registers.
    static constexpr int NQ = (D <= 128) ? 2 : 1;
    static constexpr bool STAGE_O = (D <= 128);
    static constexpr int ST = (D <= 64) ? 5 : (D <= 96 ? 3 : 2);
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = NQ * TILE;
    static constexpr uint32_t OFF_V = OFF_K + ST * TILE;
    static constexpr uint32_t OFF_OST = OFF_V + ST * TILE;
    static constexpr uint32_t OFF_BAR = OFF_OST + (STAGE_O ? TILE : 0);
    static constexpr uint32_t BAR_BYTES = 512;
    // SPLIT (d <= 128): each column half of a row keeps its own running maximum,
    // sum and O accumulator, so the halves never wait on each other inside a
    // tile; the tile's epilogue merges the two (row statistics swapped through
    // XCH_BYTES of shared memory).  d = 160 has no TMEM for a second
    // accumulator: its halves share one O and swap their block maxima.
    static constexpr bool SPLIT = (D <= 128);
    static constexpr uint32_t OFF_XCH = OFF_BAR + BAR_BYTES;
    static constexpr uint32_t XCH_BYTES = SPLIT ? 128 * 8 : 0;
    static constexpr uint32_t SMEM = OFF_XCH + XCH_BYTES + 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    // TMEM columns: two score buffers, then the O accumulator of half 0 (T_O)
    // and of half 1 (T_O1) when SPLIT, else the shared O and six exchange
    // columns through which the two halves of a row swap their block maxima
    // (2 buffers x 2 halves) and row sums (2 halves).
    static constexpr uint32_t T_S0 = 0, T_S1 = 128, T_O = 256, T_O1 = 256 + D, T_X = 256 + D;
    static_assert(SPLIT ? (T_O1 + D <= 512) : (T_X + 6 <= 512), "TMEM budget");
};

struct FwdBars {
    uint64_t q_full[2], q_empty[2];
    uint64_t k_full[6], k_empty[6], v_full[6], v_empty[6];
    uint64_t s_full[2], p_full[2];
    uint64_t p_half[2][2];  // SPLIT: [score buffer][half] P_d of the half is in TMEM
    uint64_t o_half[2];     // SPLIT: the half's P.V of the block is done
    uint64_t xmax[2];       // row-max exchange between the two column halves
    uint64_t lsum, lsum2;   // row-statistics exchange at the end of a tile
    uint64_t o_done, o_free;
    uint64_t o_tile;        // a tile's last P.V product is done (its O is final)
    uint64_t drain;         // every MMA of this CTA is done (before TMEM is released)
    uint64_t ost_free;      // the O stage is free for this tile's rows (row threads)
    uint64_t ost_full;      // this tile's rows are in the O stage (row threads)
    uint64_t never;
    uint32_t tmem_base;
    int32_t abort_flag;
};
static_assert(sizeof(FwdBars) <= FwdCfg<64>::BAR_BYTES, "barrier block");

// Wait sites reported in bits 8.. of the status word on a timeout.
enum : int32_t {
    kSiteInject = 1, kSiteKEmpty, kSiteVEmpty, kSiteQFull, kSiteKFull, kSiteVFull, kSitePFull,
    kSiteSFull, kSiteODone, kSiteXmax, kSiteQEmpty, kSiteOFree, kSiteLsum, kSiteOTile, kSiteDrain, kSiteStage
};
__device__ __forceinline__ int32_t timeout_code(int32_t site) { return 6 | (site << 8); }

}  // namespace

template <int D, bool DROP, bool PACKED>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const FwdArgs args)
{
    using G = TileGeom<D>;
    using C = FwdCfg<D>;
    constexpr int ST = C::ST;
    const CommonArgs& a = args.c;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t sb = raw + pad;
    FwdBars* bars = reinterpret_cast<FwdBars*>(smem_raw + pad + C::OFF_BAR);
    auto bar = [](uint64_t& b) { return smem_u32(&b); };

    const TileSched sched{a.n_blk * a.n_bh, (int)gridDim.x, (int)blockIdx.x};
    const uint32_t warp = warp_id(), lane = lane_id();

    if (threadIdx.x == 0) {
        for (int qs = 0; qs < 2; ++qs) {
            mbar_init(bar(bars->q_full[qs]), 1);
            mbar_init(bar(bars->q_empty[qs]), 1);    // the tile's last S MMA is done
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(bars->s_full[b]), 1);
            mbar_init(bar(bars->p_full[b]), kRowThreads);
            mbar_init(bar(bars->xmax[b]), kRowThreads);
            mbar_init(bar(bars->p_half[b][0]), kRowThreads / 2);
            mbar_init(bar(bars->p_half[b][1]), kRowThreads / 2);
            mbar_init(bar(bars->o_half[b]), 1);
        }
        mbar_init(bar(bars->o_done), 1);
        mbar_init(bar(bars->o_free), kRowThreads);
        mbar_init(bar(bars->o_tile), 1);
        mbar_init(bar(bars->drain), 1);
        mbar_init(bar(bars->ost_free), kRowThreads);
        mbar_init(bar(bars->ost_full), kRowThreads);
        for (int st = 0; st < ST; ++st) {
            mbar_init(bar(bars->k_full[st]), 1);
            mbar_init(bar(bars->k_empty[st]), 1);
            mbar_init(bar(bars->v_full[st]), 1);
            mbar_init(bar(bars->v_empty[st]), 1);
        }
        mbar_init(bar(bars->lsum), kRowThreads);
        mbar_init(bar(bars->lsum2), kRowThreads);
        mbar_init(bar(bars->never), 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const WaitCtx wc{&bars->abort_flag, a.status, a.timeout_ns};

    bool alive = true;
    if (a.inject_timeout) alive = wait_bounded(wc, bar(bars->never), 0, timeout_code(kSiteInject));

    if (alive && warp == 0) {
        if (lane == 0) {
            // ---- TMA producer: the K ring over all blocks of all tiles
            int g = 0;
            bool ok = true;
            int vt = 0;
            QTile w;
            while (ok && next_qtile<PACKED>(sched, a, 128, vt, w)) {
                for (int j = 0; j < w.nk; ++j, ++g) {
                    const int st = g % ST;
                    ok = wait_bounded(wc, bar(bars->k_empty[st]), ((g / ST) & 1) ^ 1, timeout_code(kSiteKEmpty));
                    // At the start every CTA loads at once and HBM is the bottleneck:
                    // the ring's later stages wait until the block before has landed,
                    // so the first scores' operands are not queued behind them.
                    if (ok && g > 0 && g < ST)
                        ok = wait_bounded(wc, bar(bars->k_full[g - 1]), 0, timeout_code(kSiteKFull));
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(bars->k_full[st]), C::TILE);
                    for (int ch = 0; ch < G::NCH; ++ch)
                        tma_load_3d(sb + C::OFF_K + st * C::TILE + ch * C::CHUNK, &tm_k, ch * G::CW, w.yk + j * 128,
                                    w.zk, bar(bars->k_full[st]));
                }
            }
        } else if (lane == 1) {
            // ---- TMA producer: each tile's Q as soon as its buffer is free
            int vt = 0;
            QTile w;
            for (int u = 0; next_qtile<PACKED>(sched, a, 128, vt, w); ++u) {
                const int qs = u % C::NQ;
                if (!wait_bounded(wc, bar(bars->q_empty[qs]), ((u / C::NQ) & 1) ^ 1, timeout_code(kSiteQEmpty)))
                    break;
                // the second tile's Q only once the first has landed (see the K ring)
                if (u == 1 && C::NQ == 2 && !wait_bounded(wc, bar(bars->q_full[0]), 0, timeout_code(kSiteQFull)))
                    break;
                mbar_arrive_expect_tx(bar(bars->q_full[qs]), C::TILE);
                for (int ch = 0; ch < G::NCH; ++ch)
                    tma_load_3d(sb + C::OFF_Q + qs * C::TILE + ch * C::CHUNK, &tm_q, ch * G::CW, w.yq, w.zq,
                                bar(bars->q_full[qs]));
            }
        }
    } else if (alive && warp == 2) {
        if (lane == 0) {
            // ---- TMA producer: the V ring
            int g = 0;
            bool ok = true;
            int vt = 0;
            QTile w;
            while (ok && next_qtile<PACKED>(sched, a, 128, vt, w)) {
                for (int j = 0; j < w.nk; ++j, ++g) {
                    const int st = g % ST;
                    ok = wait_bounded(wc, bar(bars->v_empty[st]), ((g / ST) & 1) ^ 1, timeout_code(kSiteVEmpty));
                    // the first V block after the first K block, the ring's later
                    // stages after the block before (see the K ring)
                    if (ok && g < ST)
                        ok = wait_bounded(wc, bar(g == 0 ? bars->k_full[0] : bars->v_full[g - 1]), 0,
                                          timeout_code(g == 0 ? kSiteKFull : kSiteVFull));
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(bars->v_full[st]), C::TILE);
                    for (int ch = 0; ch < G::NCH; ++ch)
                        tma_load_3d(sb + C::OFF_V + st * C::TILE + ch * C::CHUNK, &tm_v, ch * G::CW, w.yk + j * 128,
                                    w.zk, bar(bars->v_full[st]));
                }
            }
        }
    } else if (alive && warp == 1) {
        {   // the whole warp issues (see mma_ss)
            // ---- MMA issuer.  One stream over all blocks of all tiles of this CTA:
            // S_g, then O += P_{g-1} V_{g-1} for the block before (which may belong to
            // the previous tile), so the next tile's first scores overlap the last
            // softmax of the current one.
            constexpr uint32_t IDS = idesc_bf16(128, 128, false, false);  // S = Q K^T
            constexpr uint32_t IDO = idesc_bf16(128, D, false, true);     // O += P V
            struct Blk {
                int g, j, nk, u;
            };
            auto issue_pv = [&](const Blk& k) -> bool {
                if (k.j == 0 && !wait_warp(wc, bar(bars->o_free), (k.u & 1) ^ 1, timeout_code(kSiteOFree)))
                    return false;
                const int st = k.g % ST;
                const uint32_t vbase = sb + C::OFF_V + st * C::TILE;
                const uint32_t tP = tmem + ((k.g & 1) ? C::T_S1 : C::T_S0);
                if constexpr (C::SPLIT) {
                    // O_h += P_h V_h for each half h of the block's keys (P_h in the
                    // half's first 32 score columns, V_h the half's 64 rows of V)
                    if (!wait_warp(wc, bar(bars->v_full[st]), (k.g / ST) & 1, timeout_code(kSiteVFull)))
                        return false;
                    for (int h = 0; h < 2; ++h) {
                        if (!wait_warp(wc, bar(bars->p_half[k.g & 1][h]), (k.g >> 1) & 1, timeout_code(kSitePFull)))
                            return false;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ts(tmem + (h ? C::T_O1 : C::T_O), tP + 64 * h + 8 * kk,
                                   G::template desc_mn<128>(vbase, 4 * h + kk), IDO, (k.j > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(bar(bars->o_half[h]));
                    }
                } else {
                    if (!wait_warp(wc, bar(bars->p_full[k.g & 1]), (k.g >> 1) & 1, timeout_code(kSitePFull)))
                        return false;
                    if (!wait_warp(wc, bar(bars->v_full[st]), (k.g / ST) & 1, timeout_code(kSiteVFull)))
                        return false;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tmem + C::T_O, tP + split_a_col(kk, 128), G::template desc_mn<128>(vbase, kk), IDO,
                               (k.j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(bars->o_done));
                }
                mma_commit(bar(bars->v_empty[st]));
                if (k.j == k.nk - 1) mma_commit(bar(bars->o_tile));
                return true;
            };
            Blk prev{-1, 0, 0, 0};
            int g = 0;
            bool ok = true;
            int vt = 0;
            QTile w;
            for (int u = 0; ok && next_qtile<PACKED>(sched, a, 128, vt, w); ++u) {
                // At a tile boundary the previous tile's last P.V goes first unless this
                // tile's Q and first K block are already resident: it must never wait on
                // this tile's loads.
                const int qs = u % C::NQ;
                if (prev.g >= 0 && (!test_wait_warp(bar(bars->q_full[qs]), (u / C::NQ) & 1) ||
                                    !test_wait_warp(bar(bars->k_full[g % ST]), (g / ST) & 1))) {
                    ok = issue_pv(prev);
                    prev.g = -1;
                    if (!ok) break;
                }
                ok = wait_warp(wc, bar(bars->q_full[qs]), (u / C::NQ) & 1, timeout_code(kSiteQFull));
                for (int j = 0; j < w.nk && ok; ++j, ++g) {
                    const int st = g % ST;
                    ok = wait_warp(wc, bar(bars->k_full[st]), (g / ST) & 1, timeout_code(kSiteKFull));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kbase = sb + C::OFF_K + st * C::TILE;
                    const uint32_t qbase = sb + C::OFF_Q + qs * C::TILE;
                    const uint32_t tS = tmem + ((g & 1) ? C::T_S1 : C::T_S0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tS, G::template desc_k<128>(qbase, kk), G::template desc_k<128>(kbase, kk), IDS,
                               kk > 0 ? 1u : 0u);
                    mma_commit(bar(bars->k_empty[st]));
                    mma_commit(bar(bars->s_full[g & 1]));
                    if (j == w.nk - 1) mma_commit(bar(bars->q_empty[qs]));
                    if (prev.g >= 0) ok = issue_pv(prev);
                    prev = Blk{g, j, w.nk, u};
                }
            }
            if (ok && prev.g >= 0) ok = issue_pv(prev);
            // every MMA must be complete before the CTA releases TMEM
            mma_commit(bar(bars->drain));
            wait_warp(wc, bar(bars->drain), 0, timeout_code(kSiteDrain));
        }
    } else if (alive && warp >= 4) {
        // ---- softmax / epilogue: row = TMEM lane, half = which 64 keys of a block
        const RowThread rt = row_thread();
        const int h = rt.half, r = rt.row;
        const uint32_t lane_off = rt.lane_off;
        const uint32_t tX = tmem + C::T_X + lane_off;   // exchange columns of this warp's rows (d = 160)
        float2* xch = reinterpret_cast<float2*>(smem_raw + pad + C::OFF_XCH);   // row statistics (SPLIT)
        int pv_done = 0;            // P.V products completed into O by earlier tiles
        int g0 = 0;
        bool ok = true;
        int vt = 0;
        QTile w;
        for (int u = 0; ok && next_qtile<PACKED>(sched, a, 128, vt, w); ++u) {
            const int qb = w.qb, bh = w.bh, nk = w.nk;
            const int i = qb * 128 + r;          // query of the sequence
            const bool live = i < w.lq;          // rows past the end are computed, not stored
            const uint32_t tO = tmem + C::T_O + lane_off;
            const uint32_t tO1 = tmem + C::T_O1 + lane_off;
            // this half's accumulator (SPLIT), else the shared one
            const uint32_t tOh = (C::SPLIT && h) ? tO1 : tO;
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < nk; ++j) {
                const int g = g0 + j;
                const uint32_t tS = tmem + ((g & 1) ? C::T_S1 : C::T_S0) + lane_off + 64 * h;
                ok = __all_sync(0xffffffffu,
                                wait_bounded(wc, bar(bars->s_full[g & 1]), (g >> 1) & 1, timeout_code(kSiteSFull)));
                if (!ok) break;
                tc_fence_after();
                float x[64];
                {
                    uint32_t rr[64];
                    tmem_ld64(tS, rr);
#pragma unroll
                    for (int e = 0; e < 64; ++e) x[e] = __uint_as_float(rr[e]);
                }
                const int key0 = j * 128 + 64 * h;
                if (a.causal && j == qb) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (64 * h + c > r) x[c] = -INFINITY;
                }
                if (key0 + 64 > w.lk) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (key0 + c >= w.lk) x[c] = -INFINITY;
                }
                float mx = fmax3(x[0], x[1], x[2]);
#pragma unroll
                for (int c = 3; c < 63; c += 2) mx = fmax3(mx, x[c], x[c + 1]);
                mx = fmaxf(mx, x[63]);
                if constexpr (!C::SPLIT) {
                    // swap block maxima with the other half of the row through TMEM
                    tmem_st1(tX + (g & 1) * 2 + h, __float_as_uint(mx));
                    tmem_st_wait();
                    tc_fence_before();
                    ok = __all_sync(0xffffffffu, row_barrier(wc, bar(bars->xmax[g & 1]), (g >> 1) & 1,
                                                             timeout_code(kSiteXmax)));
                    if (!ok) break;
                    tc_fence_after();
                    mx = fmaxf(mx, __uint_as_float(tmem_ld1(tX + (g & 1) * 2 + (h ^ 1))));
                }
                const float m_new = fmaxf(m_run, mx * a.scale_log2);
                if (__any_sync(0xffffffffu, m_new > m_run + 8.0f)) {
                    if (j > 0) {
                        // the accumulator's last P.V (block j - 1) must be done
                        ok = __all_sync(0xffffffffu,
                                        wait_bounded(wc, bar(C::SPLIT ? bars->o_half[h] : bars->o_done),
                                                     (pv_done + j - 1) & 1, timeout_code(kSiteODone)));
                        if (!ok) break;
                        tc_fence_after();
                        const float f = ex2_approx(m_run - m_new);
                        l_run *= f;
                        const uint64_t f2 = f2_pack(f, f);
                        // SPLIT: all of this half's accumulator; else this half's share
                        // of the columns of the shared one
                        constexpr int c_step = C::SPLIT ? 1 : 2;
#pragma unroll 1
                        for (int c32 = C::SPLIT ? 0 : h; c32 < D / 32; c32 += c_step) {
                            uint32_t rr[32];
                            tmem_ld32(tOh + c32 * 32, rr);
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const uint64_t o2 =
                                    f2_mul(f2_pack(__uint_as_float(rr[2 * e]), __uint_as_float(rr[2 * e + 1])), f2);
                                float lo, hi;
                                f2_unpack(o2, lo, hi);
                                rr[2 * e] = __float_as_uint(lo);
                                rr[2 * e + 1] = __float_as_uint(hi);
                            }
                            tmem_st32(tOh + c32 * 32, rr);
                        }
                        tmem_st_wait();
                    }
                    m_run = m_new;
                }
                // A SPLIT half whose keys have all been masked so far has m_run = -inf:
                // its exponent reference is then 0 (every p of the half is 0).
                const float m_ref = (C::SPLIT && m_run == -INFINITY) ? 0.f : m_run;
                // p = 2^(x * scale_log2 - m), two at a time, and the dropout mask, in four
                // independent units of 16 keys (one Philox call each) so that the exp2
                // (MUFU) and Philox (integer multiply) work of different units overlap;
                // the row sum is taken before dropout.  A unit's keep decisions come out
                // of one SWAR test per output word (four keys) as byte sign bits, which
                // mask the packed bf16 pairs directly.
                const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
                const uint64_t nm2 = f2_pack(-m_ref, -m_ref);
                const KeepSwar8 ks(a.thr);
                uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
                uint32_t pw[32];
                uint4 w4[4];
#pragma unroll
                for (int u16 = 0; u16 < 4; ++u16)
                    w4[u16] = DROP ? philox4x32_10_rk((uint32_t)(key0 >> 4) + u16, (uint32_t)i, (uint32_t)bh + a.bh0,
                                                    a.offset, a.rk)
                                 : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u16 = 0; u16 < 4; ++u16) {
                    const uint32_t wv[4] = {w4[u16].x, w4[u16].y, w4[u16].z, w4[u16].w};
#pragma unroll
                    for (int tt = 0; tt < 4; ++tt) {
                        const uint32_t keep = DROP ? ks(wv[tt]) : 0u;   // keys 16 u16 + 4 tt .. + 3
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const int e = 8 * u16 + 2 * tt + q;            // pair e: keys key0 + 2e, 2e + 1
                            float lo, hi;
                            f2_unpack(f2_fma(f2_pack(x[2 * e], x[2 * e + 1]), sc2, nm2), lo, hi);
                            lo = ex2_approx(lo);
                            hi = ex2_approx(hi);
                            acc2[q] = f2_add(acc2[q], f2_pack(lo, hi));
                            pw[e] = DROP ? pack_bf16x2(lo, hi) & keep_pair16(keep, q) : pack_bf16x2(lo, hi);
                        }
                    }
                }
                {
                    float lo, hi;
                    f2_unpack(f2_add(acc2[0], acc2[1]), lo, hi);
                    l_run += lo + hi;
                }
                tmem_st32(tS, pw);   // P_d of these 64 keys over the first 32 of the half's columns
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(C::SPLIT ? bars->p_half[g & 1][h] : bars->p_full[g & 1]));
            }
            if (!ok) break;
            // Final row statistics, and the factors that turn the accumulator(s) into
            // O: O = a0 * O_0 + a1 * O_1 (SPLIT), O = a0 * O (else).
            float a0 = 0.f, a1 = 0.f, lse_i = 0.f;
            if constexpr (C::SPLIT) {
                // half 1 hands its (m, l) to half 0, which merges them and hands back
                // the two factors
                if (h == 1) xch[r] = make_float2(m_run, l_run);
                ok = __all_sync(0xffffffffu, row_barrier(wc, bar(bars->lsum), u & 1, timeout_code(kSiteLsum)));
                if (!ok) break;
                if (h == 0) {
                    const float2 o1 = xch[r];
                    const float m = fmaxf(m_run, o1.x);
                    const float m_ref = (m == -INFINITY) ? 0.f : m;
                    const float f0 = ex2_approx(m_run - m_ref), f1 = ex2_approx(o1.x - m_ref);
                    const float l_tot = l_run * f0 + o1.y * f1;
                    const float inv = a.keep_scale / l_tot;
                    a0 = f0 * inv;
                    a1 = f1 * inv;
                    lse_i = (m_ref + log2f(l_tot)) * 0.693147180559945309f;
                    xch[r] = make_float2(a0, a1);
                }
                ok = __all_sync(0xffffffffu, row_barrier(wc, bar(bars->lsum2), u & 1, timeout_code(kSiteLsum)));
                if (!ok) break;
                if (h == 1) {
                    const float2 f = xch[r];
                    a0 = f.x;
                    a1 = f.y;
                }
            } else {
                // row sum over both halves, through TMEM
                tmem_st1(tX + 4 + h, __float_as_uint(l_run));
                tmem_st_wait();
                tc_fence_before();
                ok = __all_sync(0xffffffffu, row_barrier(wc, bar(bars->lsum), u & 1, timeout_code(kSiteLsum)));
                if (!ok) break;
                tc_fence_after();
                const float l_tot = l_run + __uint_as_float(tmem_ld1(tX + 4 + (h ^ 1)));
                a0 = a.keep_scale / l_tot;
                lse_i = (m_run + log2f(l_tot)) * 0.693147180559945309f;
            }
            // the tile's final P.V: a barrier of its own, completing once per tile (the
            // per-block barriers may still be two phases behind here)
            ok = __all_sync(0xffffffffu, wait_bounded(wc, bar(bars->o_tile), u & 1, timeout_code(kSiteOTile)));
            if (!ok) break;
            tc_fence_after();
            // 32 columns [32 c32, 32 c32 + 32) of this row of O, as fp32 bits
            auto o_chunk = [&](int c32, uint32_t (&rr)[32]) {
                tmem_ld32(tO + c32 * 32, rr);
                if constexpr (C::SPLIT) {
                    uint32_t r1[32];
                    tmem_ld32(tO1 + c32 * 32, r1);
                    const uint64_t a02 = f2_pack(a0, a0), a12 = f2_pack(a1, a1);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint64_t o2 =
                            f2_fma(f2_pack(__uint_as_float(rr[2 * e]), __uint_as_float(rr[2 * e + 1])), a02,
                                   f2_mul(f2_pack(__uint_as_float(r1[2 * e]), __uint_as_float(r1[2 * e + 1])), a12));
                        float lo, hi;
                        f2_unpack(o2, lo, hi);
                        rr[2 * e] = __float_as_uint(lo);
                        rr[2 * e + 1] = __float_as_uint(hi);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * a0);
                }
            };
            // O row i straight to global memory: 16-byte stores of this half's
            // 32-column chunks.  The TMEM loads are warp-collective, so every lane
            // takes them; only the stores are guarded (rows past the sequence's end).
            auto store_rows = [&]() {
                uint4* orow = reinterpret_cast<uint4*>(args.o + (size_t)w.zq * args.o_head_stride +
                                                       (size_t)(live ? w.yq + r : 0) * args.o_row_stride);
#pragma unroll 1
                for (int c32 = h; c32 < D / 32; c32 += 2) {
                    uint32_t rr[32];
                    o_chunk(c32, rr);
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4) {
                        uint32_t wv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            wv[e] = pack_bf16x2(__uint_as_float(rr[8 * u4 + 2 * e]),
                                                __uint_as_float(rr[8 * u4 + 2 * e + 1]));
                        if (live) orow[c32 * 4 + u4] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                }
            };
            if (live && h == 0) args.lse[(size_t)w.zq * a.lse_stride + w.yq + r] = lse_i;
            if constexpr (C::STAGE_O) {
                // O / l -> bf16 into the stage, then one TMA store of the tile (rows past
                // s are clipped by the tensor map).  The stage is reused only after the
                // previous tile's store has read it.  A packed batch's tail tile stores
                // its rows one by one instead: its tensor map runs on into the next
                // sequence.  Both take the stage barriers, which count tiles.
                if (h == 0 && r == 0) bulk_wait_read0();
                ok = __all_sync(0xffffffffu, row_barrier(wc, bar(bars->ost_free), u & 1, timeout_code(kSiteStage)));
                if (!ok) break;
                if (!w.tail) {
#pragma unroll 1
                    for (int c32 = h; c32 < D / 32; c32 += 2) {
                        uint32_t rr[32];
                        o_chunk(c32, rr);
                        stage_row32<D, 128>(sb + C::OFF_OST, r, c32 * 32, rr, 1.0f);
                    }
                } else {
                    store_rows();
                }
                fence_proxy_async_smem();
                ok = __all_sync(0xffffffffu, row_barrier(wc, bar(bars->ost_full), u & 1, timeout_code(kSiteStage)));
                if (!ok) break;
                if (!w.tail && h == 0 && r == 0 && !bars->abort_flag) {
                    for (int ch = 0; ch < G::NCH; ++ch)
                        tma_store_3d(&tm_o, sb + C::OFF_OST + ch * C::CHUNK, ch * G::CW, w.yq, w.zq);
                    bulk_commit();
                }
            } else {
                store_rows();
            }
            tc_fence_before();
            mbar_arrive(bar(bars->o_free));
            pv_done += nk;
            g0 += nk;
        }
        // the last tile's O store must have read the stage before the CTA exits
        if (C::STAGE_O && h == 0 && r == 0) bulk_wait_read0();
    }

    __syncthreads();
    if (bars->abort_flag) {
        // Let any copy or MMA issued before the abort land before TMEM and
        // shared memory are released.
        for (int k = 0; k < 20; ++k) __nanosleep(50000);
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool DROP, bool PACKED>
static int launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& to, const FwdArgs& a, cudaStream_t stream)
{
    constexpr uint32_t smem = FwdCfg<D>::SMEM;
    auto kern = attn_fwd_kernel<D, DROP, PACKED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    const unsigned tiles = (unsigned)a.c.n_blk * (unsigned)a.c.n_bh;
    const unsigned grid = tiles < (unsigned)a.num_sms ? tiles : (unsigned)a.num_sms;
    kern<<<grid, kThreads, smem, stream>>>(tq, tk, tv, to, a);
    return (int)cudaGetLastError();
}

int launch_fwd(int d, bool dropout, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& to, const FwdArgs& a, cudaStream_t stream)
{
#define AC_FWD_CASE(DD)                                                                             \
    case DD:                                                                                        \
        return a.c.cu_q ? (dropout ? launch_fwd_t<DD, true, true>(tq, tk, tv, to, a, stream)          \
                                   : launch_fwd_t<DD, false, true>(tq, tk, tv, to, a, stream))        \
                        : (dropout ? launch_fwd_t<DD, true, false>(tq, tk, tv, to, a, stream)         \
                                   : launch_fwd_t<DD, false, false>(tq, tk, tv, to, a, stream));
    switch (d) {
        AC_FWD_CASE(64)
        AC_FWD_CASE(96)
        AC_FWD_CASE(128)
        AC_FWD_CASE(160)
        default: return (int)cudaErrorInvalidValue;
    }
#undef AC_FWD_CASE
}

}  // namespace ac
