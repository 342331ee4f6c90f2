// bwd.cu -- recompute-backward of the attention core on sm_103a.
//
// Selective activation recomputation keeps only Q, K, V, O, the per-row LSE
// and the dropout seed/offset; the backward pass recomputes the scores,
// probabilities and dropout mask on chip ("Reducing Activation Recomputation
// in Large Transformer Models", Key takeaways, fourth bullet; "Recomputing
// Activations", second paragraph: the backward pass rebuilds the scores).
// With Z = M / (1 - p) the gradients are
//     dP_d = dO V^T,  dP = dP_d * Z,  dS = P * (dP - D),  D_i = rowsum(dO_i * O_i)
//     dV = (P * Z)^T dO,  dK = scale * dS^T Q,  dQ = scale * dS K
// (D_i equals sum_j P_ij dP_ij because O_i = sum_j P_ij Z_ij V_j).
//
// Two kernels, launched in this order:
//   bwd_dq    one (query head, 128-query block) per CTA; queries on TMEM
//             lanes; forms -LSE_i * log2(e) and a first estimate
//             D~_i = rowsum(dO_i * O_i) from the bf16 output, recomputes S and
//             dP per key block, accumulates dQ in TMEM with the exact
//             statistic D_i = sum_j P_ij dP_ij (see below) and writes both
//             row statistics to a padded workspace
//   bwd_dkdv  one (KV head, 128-key block) per CTA; keys on TMEM lanes; loops
//             over the query heads of the GQA group and their query tiles;
//             recomputes S^T and dP^T, accumulates dV and dK in TMEM
// The dropout mask is drawn once per backward where the workspace has room
// for it (d <= 128): bwd_dq stores its keep decisions as bits (one 32-bit
// word per query row and 32 keys), and bwd_dkdv loads them with its query
// tiles and transposes them to its key-major lanes (mask_pair_word gives the
// layout).  Otherwise bwd_dkdv draws the mask again, transposed.
// Neither gradient kernel writes a partial sum to global memory: each output
// tile is finished in TMEM and stored once.
#include "kernels.h"
#include "philox.cuh"
#include "ptx.cuh"
#include "sched.cuh"
#include "tile.cuh"

namespace ac {
// The backward kernels' waits do not suspend (they retry after the hardware's
// short try-wait limit): their row threads' dependency chains resume sooner, which
// outweighs the issue slots a retrying warp takes (mbar_try_wait).
constexpr bool kBwdSuspend = false;
}  // namespace ac

namespace ac {

namespace {

enum : int32_t {
    kSiteInject = 1, kSiteKvFull, kSiteQEmpty, kSiteQFull, kSitePFull, kSiteDsFull, kSiteSFull,
    kSiteDpFull, kSiteAcc, kSiteKEmpty, kSiteVEmpty, kSiteKFull, kSiteVFull, kSitePRead, kSiteOFull, kSiteStage, kSiteRng,
    kSiteX, kSiteDrain
};
__device__ __forceinline__ int32_t timeout_code(int32_t site) { return 6 | (site << 8); }

}  // namespace

// ============================================================ dK / dV ====
namespace {

template <int D>
struct DkdvCfg {
    using G = TileGeom<D>;
    static constexpr int BQ = dkdv_query_tile(D);
    static constexpr uint32_t KV_TILE = G::template tile_bytes<128>();
    static constexpr uint32_t KV_CHUNK = G::template chunk_bytes<128>();
    static constexpr uint32_t Q_TILE = G::template tile_bytes<BQ>();
    static constexpr uint32_t Q_CHUNK = G::template chunk_bytes<BQ>();
    static constexpr int ST = 2;
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = KV_TILE;
    static constexpr uint32_t OFF_Q = 2 * KV_TILE;
    static constexpr uint32_t OFF_DO = OFF_Q + ST * Q_TILE;
    static constexpr uint32_t OFF_LSE = OFF_DO + ST * Q_TILE;
    static constexpr uint32_t OFF_DEL = OFF_LSE + ST * BQ * 4;
    // keep bits of a query tile, when the dQ kernel handed them over: 4 key
    // quarters x BQ query rows (in 64-row units) of 32-bit words
    static constexpr uint32_t MSK_BYTES = BQ * 16;
    static constexpr uint32_t OFF_MSK = OFF_DEL + ST * BQ * 4;
    static constexpr uint32_t OFF_BAR = OFF_MSK + ST * MSK_BYTES;
    static constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    // TMEM columns
    static constexpr uint32_t T_DV = 0, T_DK = D, T_S = 2 * D, T_DP = 2 * D + BQ;
    static_assert(T_DP + BQ <= 512, "TMEM budget");
};

struct DkdvBars {
    uint64_t kv_full, kv_empty;        // a tile's K and V landed / free (its last S and dP done)
    uint64_t q_full[2], q_empty[2];
    uint64_t s_full, dp_full, p_full, ds_full;
    uint64_t acc_done, acc_free;       // a tile's accumulators complete / read out
    uint64_t out_staged;               // the tile's dK and dV staged (or stored row by row)
    uint64_t out_read;                 // the store lane has finished a tile
    uint64_t stage_free[2];            // the staged output in a query-ring slot has been read
    uint64_t kv_stage_free;            // the staged output in the K/V buffers has been read
    uint64_t drain, never;
    uint32_t tmem_base;
    int32_t abort_flag;
};
static_assert(sizeof(DkdvBars) <= 256, "barrier block");

// One work tile of the dK/dV kernel: a 128-key block of one KV head of one
// sequence (or batch element).  Tile t: key block t / n_bkv (small key blocks
// see the most queries under the causal mask: longest first) and flattened KV
// head bkv = t % n_bkv = sequence * h_kv + head.
struct KTile {
    int kb, bkv, seq, kvh;
    int bh0;              // the group's first flattened query head
    int q_first, k_first; // the sequence's first query and key rows (packed batch), or 0
    int lq, lk;           // its query and key counts
    int qt0, per_head, n_it;   // first query tile, tiles per query head, iterations
    int yk, zk;           // TMA coordinates of the key block
    bool empty;           // a packed batch's key block past its sequence's keys
    bool tail;            // a packed batch's key block holding rows past its end
};
template <bool PACKED>
__device__ __forceinline__ KTile k_tile(const CommonArgs& a, int t, int bq)
{
    KTile w;
    const int n_bkv = a.n_bh / a.h_q * a.h_kv;
    const int group = a.h_q / a.h_kv;
    w.kb = t / n_bkv;
    w.bkv = t % n_bkv;
    w.seq = w.bkv / a.h_kv;
    w.kvh = w.bkv % a.h_kv;
    w.bh0 = w.seq * a.h_q + w.kvh * group;
    if constexpr (PACKED) {
        w.q_first = a.cu_q[w.seq];
        w.k_first = a.cu_k[w.seq];
        w.lq = a.cu_q[w.seq + 1] - w.q_first;
        w.lk = a.cu_k[w.seq + 1] - w.k_first;
        w.zk = w.kvh;
    } else {
        w.q_first = w.k_first = 0;
        w.lq = a.s;
        w.lk = a.s_k;
        w.zk = w.bkv;
    }
    w.empty = w.kb * 128 >= w.lk;
    w.tail = PACKED && (w.kb + 1) * 128 > w.lk;
    const int n_qt = ((w.lq + 127) / 128) * 128 / bq;
    w.qt0 = a.causal ? (w.kb * 128) / bq : 0;
    // under a top-left causal mask a key block past the last query is seen by none
    w.per_head = n_qt > w.qt0 ? n_qt - w.qt0 : 0;
    w.n_it = w.empty ? 0 : group * w.per_head;
    w.yk = w.k_first + w.kb * 128;
    return w;
}
// The key blocks the kernel walks: under a causal mask the padded layout's key
// blocks past the last query block are seen by no query (the caller zeroes
// their gradients); a packed batch's sequences differ, so there every key block
// is a tile and such blocks store zeros.
template <bool PACKED>
__host__ __device__ inline int dkdv_key_blocks(const CommonArgs& a)
{
    return (!PACKED && a.causal && a.n_blk < a.n_blk_k) ? a.n_blk : a.n_blk_k;
}
template <bool PACKED>
__device__ __forceinline__ bool next_ktile(const TileSched& sched, const CommonArgs& a, int bq, int& v, KTile& w)
{
    for (;; ++v) {
        const int t = sched.tile(v);
        if (t < 0) return false;
        w = k_tile<PACKED>(a, t, bq);
        if (!w.empty) {
            ++v;
            return true;
        }
    }
}

}  // namespace

template <int D, bool DROP, bool MWS, bool PACKED>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                     const BwdArgs args)
{
    using G = TileGeom<D>;
    using C = DkdvCfg<D>;
    constexpr int BQ = C::BQ;
    constexpr int ST = C::ST;
    const CommonArgs& a = args.c;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t sb = raw + pad;
    uint8_t* smem = smem_raw + pad;
    DkdvBars* bars = reinterpret_cast<DkdvBars*>(smem + C::OFF_BAR);
    auto bar = [](uint64_t& b) { return smem_u32(&b); };

    const int group = a.h_q / a.h_kv;
    constexpr bool packed = PACKED;
    // Persistent: one CTA per SM walks its share of the key-block tiles, longest first.
    const TileSched sched{dkdv_key_blocks<PACKED>(a) * (a.n_bh / a.h_q * a.h_kv), (int)gridDim.x, (int)blockIdx.x};
    // Staging of dK and dV: where a query tile is 128 rows (d <= 128), a
    // tile's dK and dV are staged in the query-ring slot of its last iteration
    // (free once its last dK product is done), so the next tile's K and V can land
    // during this tile's epilogue; otherwise (d = 160) they are staged in the K and
    // V buffers and the next tile's K and V wait for their store.
    constexpr bool RING_STAGE = (BQ == 128);
    // TMA row / head coordinates and workspace row of query tile qt of head `hq` of the group
    auto q_coords = [&](const KTile& w, int hq, int qt, int& yq, int& zq, size_t& srow) {
        yq = w.q_first + qt * BQ;
        zq = packed ? w.kvh * group + hq : w.bh0 + hq;
        srow = packed ? (size_t)(w.kvh * group + hq) * a.ws_stride + packed_ws_row0(w.q_first, w.seq) + qt * BQ
                      : (size_t)(w.bh0 + hq) * a.ws_stride + qt * BQ;
    };
    const uint32_t warp = warp_id(), lane = lane_id();

    if (threadIdx.x == 0) {
        mbar_init(bar(bars->kv_full), 1);
        mbar_init(bar(bars->kv_empty), 1);
        for (int st = 0; st < ST; ++st) {
            mbar_init(bar(bars->q_full[st]), 1);
            mbar_init(bar(bars->q_empty[st]), 1);
            mbar_init(bar(bars->stage_free[st]), 1);
        }
        mbar_init(bar(bars->s_full), 1);
        mbar_init(bar(bars->dp_full), 1);
        mbar_init(bar(bars->p_full), kRowThreads);
        mbar_init(bar(bars->ds_full), kRowThreads);
        mbar_init(bar(bars->acc_done), 1);
        mbar_init(bar(bars->acc_free), kRowThreads);
        mbar_init(bar(bars->out_staged), kRowThreads);
        mbar_init(bar(bars->out_read), 1);
        mbar_init(bar(bars->kv_stage_free), 1);
        mbar_init(bar(bars->drain), 1);
        mbar_init(bar(bars->never), 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
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
    if (a.inject_timeout) alive = wait_bounded<kBwdSuspend>(wc, bar(bars->never), 0, timeout_code(kSiteInject));

    if (alive && warp == 0) {
        if (lane == 0) {
            // ---- TMA producer: per tile K and V (once its predecessor's last S and dP
            // products are done), then (Q, dO, LSE2, D and the keep bits) per query tile
            // through one ring over all tiles.  A ring slot that holds a tile's staged
            // output is refilled only after the store has read it.
            int g = 0, u = 0, vt = 0;
            bool ok = true;
            uint32_t pending = 0u;     // bit st: slot st holds staged output not yet read
            uint32_t sf_parity = 0u;   // bit st: phase parity of slot st's stage_free
            KTile w;
            while (ok && next_ktile<PACKED>(sched, a, BQ, vt, w)) {
                ok = wait_bounded<kBwdSuspend>(wc, bar(bars->kv_empty), (u & 1) ^ 1, timeout_code(kSiteKvFull));
                if (ok && !RING_STAGE && u > 0)
                    ok = wait_bounded<kBwdSuspend>(wc, bar(bars->kv_stage_free), (u - 1) & 1, timeout_code(kSiteStage));
                if (!ok) break;
                mbar_arrive_expect_tx(bar(bars->kv_full), 2 * C::KV_TILE);
                for (int ch = 0; ch < G::NCH; ++ch) {
                    tma_load_3d(sb + C::OFF_K + ch * C::KV_CHUNK, &tm_k, ch * G::CW, w.yk, w.zk, bar(bars->kv_full));
                    tma_load_3d(sb + C::OFF_V + ch * C::KV_CHUNK, &tm_v, ch * G::CW, w.yk, w.zk, bar(bars->kv_full));
                }
                for (int it = 0; it < w.n_it && ok; ++it, ++g) {
                    const int st = g % ST;
                    const int bh = w.bh0 + it / w.per_head;
                    const int qt = w.qt0 + it % w.per_head;
                    int yq, zq;
                    size_t srow;
                    q_coords(w, it / w.per_head, qt, yq, zq, srow);
                    ok = wait_bounded<kBwdSuspend>(wc, bar(bars->q_empty[st]), ((g / ST) & 1) ^ 1, timeout_code(kSiteQEmpty));
                    if (ok && RING_STAGE && ((pending >> st) & 1u)) {
                        ok = wait_bounded<kBwdSuspend>(wc, bar(bars->stage_free[st]), (sf_parity >> st) & 1u, timeout_code(kSiteStage));
                        sf_parity ^= 1u << st;
                        pending &= ~(1u << st);
                    }
                    if (!ok) break;
                    const uint32_t fb = bar(bars->q_full[st]);
                    mbar_arrive_expect_tx(fb, 2 * C::Q_TILE + 2 * BQ * 4 + (MWS ? C::MSK_BYTES : 0u));
                    for (int ch = 0; ch < G::NCH; ++ch) {
                        tma_load_3d(sb + C::OFF_Q + st * C::Q_TILE + ch * C::Q_CHUNK, &tm_q, ch * G::CW, yq, zq, fb);
                        tma_load_3d(sb + C::OFF_DO + st * C::Q_TILE + ch * C::Q_CHUNK, &tm_do, ch * G::CW, yq, zq,
                                    fb);
                    }
                    bulk_load_1d(sb + C::OFF_LSE + st * BQ * 4, args.lse2_ws + srow, BQ * 4, fb);
                    bulk_load_1d(sb + C::OFF_DEL + st * BQ * 4, args.delta_ws + srow, BQ * 4, fb);
                    if constexpr (MWS) {
                        // this tile's rows of the (qb, kb) keep bits: both 64-row units, or one
                        const size_t w0 =
                            mask_pair_word(a, bh, (qt * BQ) >> 7, w.kb) + (size_t)(((qt * BQ) & 127) >> 6) * 256;
                        bulk_load_1d(sb + C::OFF_MSK + st * C::MSK_BYTES, args.mask_ws + w0, C::MSK_BYTES, fb);
                    }
                }
                // the tile's last slot will hold its staged dK and dV
                if (RING_STAGE && w.n_it > 0 && !w.tail) pending |= 1u << ((g - 1) % ST);
                ++u;
            }
        } else if (lane == 1) {
            // ---- dK and dV out: once the row threads have staged a tile's rows, one
            // TMA store each, then the staging area is released (a tail tile's rows
            // and a tile without queries were stored by the row threads)
            int g = 0, u = 0, vt = 0;
            bool ok = true;
            KTile w;
            while (ok && next_ktile<PACKED>(sched, a, BQ, vt, w)) {
                g += w.n_it;
                ok = wait_bounded<kBwdSuspend>(wc, bar(bars->out_staged), u & 1, timeout_code(kSiteStage));
                if (!ok) break;
                const int slot = (g - 1 + 2 * ST) % ST;
                const bool staged = !w.tail && (!RING_STAGE || w.n_it > 0);
                if (staged) {
                    const uint32_t ok_off = RING_STAGE ? C::OFF_Q + slot * C::Q_TILE : C::OFF_K;
                    const uint32_t ov_off = RING_STAGE ? C::OFF_DO + slot * C::Q_TILE : C::OFF_V;
                    for (int ch = 0; ch < G::NCH; ++ch) {
                        tma_store_3d(&tm_dv, sb + ov_off + ch * C::KV_CHUNK, ch * G::CW, w.yk, w.zk);
                        tma_store_3d(&tm_dk, sb + ok_off + ch * C::KV_CHUNK, ch * G::CW, w.yk, w.zk);
                    }
                    bulk_commit();
                    bulk_wait_read0();
                }
                if (RING_STAGE) {
                    if (staged) mbar_arrive(bar(bars->stage_free[slot]));
                } else {
                    mbar_arrive(bar(bars->kv_stage_free));
                }
                mbar_arrive(bar(bars->out_read));
                ++u;
            }
        }
    } else if (alive && warp == 1) {
        {   // the whole warp issues (see mma_ss)
            // ---- MMA issuer.  Order: S0 dP0 | dV0 S1 dK0 dP1 | dV1 S2 dK1 dP2 | ...
            constexpr uint32_t IDS = idesc_bf16(128, BQ, false, false);  // S^T = K Q^T, dP^T = V dO^T
            constexpr uint32_t IDG = idesc_bf16(128, D, false, true);    // dV += P^T dO, dK += dS^T Q
            auto issue_s = [&](int it) {
                const uint32_t qbase = sb + C::OFF_Q + (it % ST) * C::Q_TILE;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + C::T_S, G::template desc_k<128>(sb + C::OFF_K, kk),
                           G::template desc_k<BQ>(qbase, kk), IDS, kk > 0 ? 1u : 0u);
                mma_commit(bar(bars->s_full));
            };
            auto issue_dp = [&](int it) {
                const uint32_t dobase = sb + C::OFF_DO + (it % ST) * C::Q_TILE;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + C::T_DP, G::template desc_k<128>(sb + C::OFF_V, kk),
                           G::template desc_k<BQ>(dobase, kk), IDS, kk > 0 ? 1u : 0u);
                mma_commit(bar(bars->dp_full));
            };
            int g = 0, u = 0, vt = 0;
            bool ok = true;
            KTile w;
            while (ok && next_ktile<PACKED>(sched, a, BQ, vt, w)) {
                const int n_it = w.n_it;
                ok = wait_warp<kBwdSuspend>(wc, bar(bars->kv_full), u & 1, timeout_code(kSiteKvFull));
                if (ok && n_it > 0) ok = wait_warp<kBwdSuspend>(wc, bar(bars->q_full[g % ST]), (g / ST) & 1, timeout_code(kSiteQFull));
                if (!ok) break;
                tc_fence_after();
                if (n_it > 0) {
                    issue_s(g);
                    issue_dp(g);
                }
                // K and V are free once the tile's last S and dP products are done
                if (n_it <= 1) mma_commit(bar(bars->kv_empty));
                for (int it = 0; it < n_it && ok; ++it, ++g) {
                    const int st = g % ST;
                    const uint32_t qbase = sb + C::OFF_Q + st * C::Q_TILE;
                    const uint32_t dobase = sb + C::OFF_DO + st * C::Q_TILE;
                    ok = wait_warp<kBwdSuspend>(wc, bar(bars->p_full), g & 1, timeout_code(kSitePFull));
                    // the first dV product of a tile overwrites the accumulators: the
                    // epilogue of the tile before must have read them
                    if (ok && it == 0) ok = wait_warp<kBwdSuspend>(wc, bar(bars->acc_free), (u & 1) ^ 1, timeout_code(kSiteAcc));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk)
                        mma_ts(tmem + C::T_DV, tmem + C::T_S + split_a_col(kk, BQ), G::template desc_mn<BQ>(dobase, kk),
                               IDG, (it > 0 || kk > 0) ? 1u : 0u);
                    if (it + 1 < n_it) {
                        const int st1 = (g + 1) % ST;
                        ok = wait_warp<kBwdSuspend>(wc, bar(bars->q_full[st1]), ((g + 1) / ST) & 1, timeout_code(kSiteQFull));
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(g + 1);
                    }
                    ok = wait_warp<kBwdSuspend>(wc, bar(bars->ds_full), g & 1, timeout_code(kSiteDsFull));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk)
                        mma_ts(tmem + C::T_DK, tmem + C::T_DP + split_a_col(kk, BQ), G::template desc_mn<BQ>(qbase, kk),
                               IDG, (it > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(bars->q_empty[st]));
                    if (it + 1 < n_it) {
                        issue_dp(g + 1);
                        if (it + 2 == n_it) mma_commit(bar(bars->kv_empty));
                    }
                }
                if (!ok) break;
                mma_commit(bar(bars->acc_done));
                ++u;
            }
            // every MMA must be complete before the CTA releases TMEM
            mma_commit(bar(bars->drain));
            wait_warp<kBwdSuspend>(wc, bar(bars->drain), 0, timeout_code(kSiteDrain));
        }
    } else if (alive && warp >= 4) {
        // ---- row threads: key = TMEM lane, half = which BQ/2 queries of a tile
        constexpr int HQ = BQ / 2;
        const RowThread rt = row_thread();
        const int h = rt.half, r = rt.row;
        const uint32_t lane_off = rt.lane_off;
        const float* lse2_s = reinterpret_cast<const float*>(smem + C::OFF_LSE);
        const KeepSwar8 ks(a.thr);
        const uint64_t zs2 = f2_pack(a.keep_scale, a.keep_scale);
        const float* del_s = reinterpret_cast<const float*>(smem + C::OFF_DEL);
        // Keep bytes of this lane's key over the half's queries (transposed draw).  Those
        // of tile it + 1 are drawn right after tile it's dS, while the tensor core forms
        // S_{it+1}: the draw needs no score.
        uint32_t kw[HQ / 16][4];
        auto draw_mask = [&](const KTile& w, int it) {
            const int bh = w.bh0 + it / w.per_head;
            const int q0 = (w.qt0 + it % w.per_head) * BQ + HQ * h;
            const uint32_t warp_key0 = (uint32_t)(w.kb * 128 + (int)(warp & 3u) * 32);
            const PhiloxKey pk{a.rk, (uint32_t)bh + a.bh0, a.offset};
            keep_bytes_col16<HQ>(pk, ks, warp_key0 / 16u + lane / 16u, (uint32_t)q0, kw);
        };
        // With the dQ kernel's keep bits (MWS): this key's bits over the half's
        // queries, transposed from the staged rows and spread to byte sign bits
        // (byte t of word n: query 4n + t of the half).
        uint32_t kbyte[HQ / 4] = {};
        // the keep word (byte sign bits of four consecutive queries) holding the
        // query pair (2e, 2e + 1) in its bytes 2 (e & 1) and 2 (e & 1) + 1
        auto keep_word = [&](int e) -> uint32_t {
            if constexpr (MWS) return kbyte[e >> 1];
            else return kw[e >> 3][(e & 7) >> 1];
        };
        // The dQ kernel's words hold key 4k + b of a warp's 32 keys at bit 8b + 7 - k;
        // after the transpose, lane p holds the queries of bit position p, so the lane
        // of key L reads it from lane keep_bit_position(L).
        const int src_lane = (int)keep_bit_position(lane);
        int g = 0, u = 0, vt = 0;
        bool ok = true;
        KTile w;
        while (ok && next_ktile<PACKED>(sched, a, BQ, vt, w)) {
        const int n_it = w.n_it, kb = w.kb;
        const int key = kb * 128 + r;
        if (DROP && !MWS && n_it > 0) draw_mask(w, 0);
        for (int it = 0; it < n_it; ++it, ++g) {
            const int st = g % ST;
            const int q0 = (w.qt0 + it % w.per_head) * BQ + HQ * h;     // this half's first query
            ok = __all_sync(0xffffffffu,
                            wait_bounded<kBwdSuspend>(wc, bar(bars->q_full[st]), (g / ST) & 1, timeout_code(kSiteQFull)));
            if (!ok) break;
            // The keep bits came with this query tile's stage: their transpose needs no
            // score, so it runs while the tensor core forms S^T.
            if constexpr (DROP && MWS) {
                const uint32_t* msk = reinterpret_cast<const uint32_t*>(smem + C::OFF_MSK + st * C::MSK_BYTES);
#pragma unroll
                for (int c = 0; c < HQ / 32; ++c) {
                    const int row = HQ * h + 32 * c + (int)lane;    // query row of the tile
                    const uint32_t col = __shfl_sync(
                        0xffffffffu, transpose32(msk[(row >> 6) * 256 + (int)(warp & 3u) * 64 + (row & 63)]), src_lane);
#pragma unroll
                    for (int n = 0; n < 8; ++n) kbyte[8 * c + n] = keep_nibble_bytes((col >> (4 * n)) & 0xFu);
                }
            }
            ok = __all_sync(0xffffffffu, wait_bounded<kBwdSuspend>(wc, bar(bars->s_full), g & 1, timeout_code(kSiteSFull)));
            if (!ok) break;
            tc_fence_after();
            // per-query row statistics of this half (-LSE log2(e) and -D), four at a time
            const float4* nl4 = reinterpret_cast<const float4*>(lse2_s + st * BQ + HQ * h);
            const float4* dl4 = reinterpret_cast<const float4*>(del_s + st * BQ + HQ * h);
            const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
            uint64_t pp[HQ / 2];
            uint32_t rs[HQ];
            if constexpr (HQ == 64) {
                tmem_ld64(tmem + C::T_S + lane_off + HQ * h, rs);
            } else {
                uint32_t r32[32];
                tmem_ld32(tmem + C::T_S + lane_off + HQ * h, r32);
#pragma unroll
                for (int e = 0; e < 32; ++e) rs[e] = r32[e];
            }
#pragma unroll
            for (int c32 = 0; c32 < HQ / 32; ++c32) {
                const uint32_t* rr = rs + 32 * c32;
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    const float4 l = nl4[c32 * 8 + e / 2];
                    float lo, hi;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[2 * e]), __uint_as_float(rr[2 * e + 1])), sc2,
                                     f2_pack(l.x, l.y)), lo, hi);
                    pp[c32 * 16 + e] = f2_pack(ex2_approx(lo), ex2_approx(hi));
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[2 * e + 2]), __uint_as_float(rr[2 * e + 3])), sc2,
                                     f2_pack(l.z, l.w)), lo, hi);
                    pp[c32 * 16 + e + 1] = f2_pack(ex2_approx(lo), ex2_approx(hi));
                }
            }
            if (a.causal && q0 < kb * 128 + 128) {
#pragma unroll
                for (int e = 0; e < HQ / 2; ++e) {
                    float lo, hi;
                    f2_unpack(pp[e], lo, hi);
                    if (q0 + 2 * e < key) lo = 0.f;
                    if (q0 + 2 * e + 1 < key) hi = 0.f;
                    pp[e] = f2_pack(lo, hi);
                }
            }
            // P^T masked by the keep mask (dropped entries +0) -> TMEM over the first HQ/2
            // of this half's S^T columns; the factor 1/(1-p) is applied to dV at the end
            {
                uint32_t pw[HQ / 2];
#pragma unroll
                for (int e = 0; e < HQ / 2; ++e)
                    pw[e] = DROP ? pack_bf16x2(pp[e]) & keep_pair16(keep_word(e), e & 1) : pack_bf16x2(pp[e]);
                if constexpr (HQ / 2 == 32) {
                    tmem_st32(tmem + C::T_S + lane_off + HQ * h, pw);
                } else {
                    tmem_st16(tmem + C::T_S + lane_off + HQ * h, pw);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(bars->p_full));

            ok = __all_sync(0xffffffffu, wait_bounded<kBwdSuspend>(wc, bar(bars->dp_full), g & 1, timeout_code(kSiteDpFull)));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int c32 = 0; c32 < HQ / 32; ++c32) {
                uint32_t rr[32];
                tmem_ld32(tmem + C::T_DP + lane_off + HQ * h + c32 * 32, rr);
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int ep = c32 * 16 + e;
                    uint32_t dlo = rr[2 * e], dhi = rr[2 * e + 1];
                    if (DROP) {
                        // dP = dP_d * Z: dropped elements' dP_d is cleared, kept ones carry
                        // 1/(1-p) in the FMA below
                        const uint32_t kwd = keep_word(ep);
                        dlo &= keep_mask32(kwd, 2 * (ep & 1));
                        dhi &= keep_mask32(kwd, 2 * (ep & 1) + 1);
                    }
                    const float4 dl = dl4[ep >> 1];
                    const uint64_t nd = (ep & 1) ? f2_pack(dl.z, dl.w) : f2_pack(dl.x, dl.y);   // -D
                    const uint64_t dp = f2_pack(__uint_as_float(dlo), __uint_as_float(dhi));
                    w[e] = pack_bf16x2(f2_mul(pp[ep], DROP ? f2_fma(dp, zs2, nd) : f2_add(dp, nd)));
                }
                tmem_st16(tmem + C::T_DP + lane_off + HQ * h + c32 * 16, w);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(bars->ds_full));
            if (DROP && !MWS && it + 1 < n_it) draw_mask(w, it + 1);
        }
        if (!ok) break;
        ok = __all_sync(0xffffffffu, wait_bounded<kBwdSuspend>(wc, bar(bars->acc_done), u & 1, timeout_code(kSiteAcc)));
        if (!ok) break;
        // dV and dK of this key row: staged for the TMA store of the tile (in the
        // query-ring slot of its last iteration, or the K and V buffers), or -- a
        // packed batch's tail block, whose tensor map runs on into the next
        // sequence, and a ring-staged tile without queries -- stored row by row;
        // zero when no query sees the block
        const int slot = (g - 1 + 2 * ST) % ST;
        const bool direct = w.tail || (RING_STAGE && n_it == 0);
        auto put_row = [&](uint16_t* base, uint32_t stage_off, int c32, uint32_t (&rr)[32], float mul) {
            if (!direct) {
                stage_row32<D, 128>(sb + stage_off, r, c32 * 32, rr, mul);
            } else if (kb * 128 + r < w.lk) {
                uint4* row = reinterpret_cast<uint4*>(base + (size_t)w.zk * args.kv_head_stride +
                                                      (size_t)(w.yk + r) * args.kv_row_stride) + c32 * 4;
#pragma unroll
                for (int u4 = 0; u4 < 4; ++u4) {
                    uint32_t wv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        wv[e] = pack_bf16x2(__uint_as_float(rr[8 * u4 + 2 * e]) * mul,
                                            __uint_as_float(rr[8 * u4 + 2 * e + 1]) * mul);
                    row[u4] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
        };
        const uint32_t stage_k = RING_STAGE ? C::OFF_Q + slot * C::Q_TILE : C::OFF_K;
        const uint32_t stage_v = RING_STAGE ? C::OFF_DO + slot * C::Q_TILE : C::OFF_V;
        tc_fence_after();
#pragma unroll 1
        for (int c32 = h; c32 < D / 32; c32 += 2) {
            uint32_t rr[32];
            tmem_ld32(tmem + C::T_DV + lane_off + c32 * 32, rr);
            if (n_it == 0) {
#pragma unroll
                for (int e = 0; e < 32; ++e) rr[e] = 0u;
            }
            put_row(args.dv, stage_v, c32, rr, DROP ? a.keep_scale : 1.0f);
            tmem_ld32(tmem + C::T_DK + lane_off + c32 * 32, rr);
            if (n_it == 0) {
#pragma unroll
                for (int e = 0; e < 32; ++e) rr[e] = 0u;
            }
            put_row(args.dk, stage_k, c32, rr, a.scale);
        }
        tc_fence_before();
        mbar_arrive(bar(bars->acc_free));   // the next tile's products may overwrite them
        fence_proxy_async_smem();
        // the store lane takes one tile at a time: a tile is handed over only after
        // the previous one is done (tiles without queries can follow one another fast)
        if (u > 0) ok = __all_sync(0xffffffffu, wait_bounded<kBwdSuspend>(wc, bar(bars->out_read), (u - 1) & 1, timeout_code(kSiteStage)));
        if (!ok) break;
        mbar_arrive(bar(bars->out_staged));
        ++u;
        }
    }

    __syncthreads();
    if (bars->abort_flag) {
        for (int k = 0; k < 20; ++k) __nanosleep(50000);
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// =============================================================== dQ ======
// Tiles are (query head, 128-query block) pairs, queries on TMEM lanes.  Per
// key block j: S = Q K_j^T and dP_d = dO V_j^T into TMEM; the row threads
// form P, the mask, dP = dP_d * Z and
//     dS~ = P (dP - D~),        D~ = rowsum(dO * O) from the bf16 output,
// and accumulate the exact row statistic D = sum_j P_ij dP_ij in fp32.  The
// tensor core accumulates dQ~ += dS~ K_j and PK += P K_j.  At the end
//     dQ = scale (dQ~ - (D - D~) PK),
// which equals scale * sum_j P_ij (dP_ij - D_i) K_j: the gradient with the
// exact statistic, not the one rounded through the stored bf16 output.  The
// exact D is written back to the workspace for the dK/dV kernel.
//
// Persistent: one CTA per SM walks its share of the tiles, longest first
// (sched.cuh).  Q and dO have a buffer of their own, so the next tile's are
// loaded while this one's epilogue runs (once its last S and dP products are
// done and its rows have formed D~); the K and V rings, the score buffers and
// the MMA stream run on across tiles, and the next tile's first P K product
// only waits until the epilogue has read the accumulators.  The O buffer
// serves twice per tile: O for D~, formed in the first block after the
// probabilities, then the staged dQ of the epilogue, which one TMA store
// writes out before the next tile's O comes in.  The row statistic -LSE is
// read a tile ahead, and the next tile's Q, dO and O are pulled into L2.
namespace {

template <int D>
struct DqCfg {
    using G = TileGeom<D>;
    static constexpr int BN = dq_key_tile(D);
    static constexpr uint32_t QT = G::template tile_bytes<128>();
    static constexpr uint32_t QCH = G::template chunk_bytes<128>();
    static constexpr uint32_t KT = G::template tile_bytes<BN>();
    static constexpr uint32_t KCH = G::template chunk_bytes<BN>();
    static constexpr uint32_t RED_BYTES = 2 * 128 * 4;       // [2 halves][128] partial row statistics
    // Keep bits of a key block, drawn by the RNG warps: [BN / 32][128 rows]
    // words, key 32 q + c of row r at bit keep_bit_position(c) of word [q][r];
    // a ring of RNG_ST blocks lets the RNG warps run ahead of the row threads.
    static constexpr int RNG_ST = 4;
    static constexpr uint32_t RNG_BYTES = (BN / 32) * 128 * 4;
    static constexpr uint32_t BAR_BYTES = 512;
    // A K tile is an operand of three products (S, P K and dQ), so its ring slot
    // frees only when the block's dQ product is done.  V is read by one
    // product, dP, issued about a block after its slot frees, so where two V
    // stages would leave the K ring short of four, V gets one; the K ring takes
    // every stage that fits beside Q, dO, O, V and the keep-bit ring, up to four.
    static constexpr uint32_t FIXED = 3u * QT + BAR_BYTES + RED_BYTES + RNG_ST * RNG_BYTES + 1024u;
    static constexpr int VST = (227u * 1024u - FIXED - 2u * KT) / KT >= 4 ? 2 : 1;
    static constexpr int KST_FIT = (int)((227u * 1024u - FIXED - (uint32_t)VST * KT) / KT);
    static constexpr int KST = KST_FIT < 4 ? KST_FIT : 4;
    static_assert(KST >= 2, "K ring");
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_DO = QT;
    static constexpr uint32_t OFF_O = 2 * QT;
    static constexpr uint32_t OFF_K = 3 * QT;
    static constexpr uint32_t OFF_V = OFF_K + KST * KT;
    static constexpr uint32_t OFF_BAR = OFF_V + VST * KT;
    static constexpr uint32_t OFF_RED = OFF_BAR + BAR_BYTES;
    static constexpr uint32_t OFF_RNG = OFF_RED + RED_BYTES;
    static constexpr uint32_t SMEM = OFF_RNG + RNG_ST * RNG_BYTES + 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    // TMEM: S (later P in the first half of each row half) | dP (later dS~) | dQ~ | PK
    static constexpr uint32_t T_S = 0, T_DP = BN, T_DQ = 2 * BN, T_PK = 2 * BN + D;
    static_assert(T_PK + D <= 512, "TMEM budget");
};

struct DqBars {
    uint64_t q_full, q_empty;          // Q and dO of a tile (freed by the products and the D~ reads)
    uint64_t o_full, dq_staged;        // O of a tile in the O buffer / the tile's dQ staged there
    uint64_t k_full[4], k_empty[4], v_full[2], v_empty[2];
    uint64_t s_full, p_full, dp_full, ds_full;
    uint64_t acc_done, acc_free;       // a tile's accumulators complete / read out
    uint64_t xbar;                     // exchange barrier of the 256 row threads
    uint64_t rng_full[4], rng_empty[4];  // keep-bit ring
    uint64_t drain, never;
    uint32_t tmem_base;
    int32_t abort_flag;
};
static_assert(sizeof(DqBars) <= DqCfg<64>::BAR_BYTES, "barrier block");

}  // namespace

template <int D, bool DROP, bool MWS, bool PACKED>
__global__ void __launch_bounds__(kThreadsRng, 1)
attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_dq,
                   const BwdArgs args)
{
    using G = TileGeom<D>;
    using C = DqCfg<D>;
    constexpr int BN = C::BN;
    constexpr int KST = C::KST, VST = C::VST;
    const CommonArgs& a = args.c;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t sb = raw + pad;
    DqBars* bars = reinterpret_cast<DqBars*>(smem_raw + pad + C::OFF_BAR);
    auto bar = [](uint64_t& b) { return smem_u32(&b); };

    const TileSched sched{a.n_blk * a.n_bh, (int)gridDim.x, (int)blockIdx.x};
    const uint32_t warp = warp_id(), lane = lane_id();

    if (threadIdx.x == 0) {
        mbar_init(bar(bars->q_full), 1);
        mbar_init(bar(bars->q_empty), 1 + kRowThreads);
        mbar_init(bar(bars->o_full), 1);
        mbar_init(bar(bars->dq_staged), kRowThreads);
        for (int st = 0; st < KST; ++st) {
            mbar_init(bar(bars->k_full[st]), 1);
            mbar_init(bar(bars->k_empty[st]), 1);
        }
        for (int st = 0; st < VST; ++st) {
            mbar_init(bar(bars->v_full[st]), 1);
            mbar_init(bar(bars->v_empty[st]), 1);
        }
        mbar_init(bar(bars->s_full), 1);
        mbar_init(bar(bars->p_full), kRowThreads);
        mbar_init(bar(bars->dp_full), 1);
        mbar_init(bar(bars->ds_full), kRowThreads);
        mbar_init(bar(bars->acc_done), 1);
        mbar_init(bar(bars->acc_free), kRowThreads);
        mbar_init(bar(bars->xbar), kRowThreads);
        for (int st = 0; st < C::RNG_ST; ++st) {
            mbar_init(bar(bars->rng_full[st]), kRngThreads);
            mbar_init(bar(bars->rng_empty[st]), kRowThreads);
        }
        mbar_init(bar(bars->drain), 1);
        mbar_init(bar(bars->never), 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_o);
        tma_prefetch_desc(&tm_dq);
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
    if (a.inject_timeout) alive = wait_bounded<kBwdSuspend>(wc, bar(bars->never), 0, timeout_code(kSiteInject));

    // Registers: the row warps raise their share to kDqRowRegs (176), every
    // other warp lowers its own to kDqOtherRegs (80); kernels.h checks the sum
    // against the launch.  Each role branch adjusts first thing, before any wait.
    if (alive && warp == 0) {
        regs_lower<kDqOtherRegs>();
        if (lane == 0) {
            // ---- TMA producer: the K ring over all blocks of all tiles
            int g = 0;
            bool ok = true;
            int vt = 0;
            QTile w;
            while (ok && next_qtile<PACKED>(sched, a, BN, vt, w)) {
                for (int j = 0; j < w.nk; ++j, ++g) {
                    const int st = g % KST;
                    ok = wait_bounded<kBwdSuspend>(wc, bar(bars->k_empty[st]), ((g / KST) & 1) ^ 1, timeout_code(kSiteKEmpty));
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(bars->k_full[st]), C::KT);
                    for (int ch = 0; ch < G::NCH; ++ch)
                        tma_load_3d(sb + C::OFF_K + st * C::KT + ch * C::KCH, &tm_k, ch * G::CW, w.yk + j * BN, w.zk,
                                    bar(bars->k_full[st]));
                }
            }
        } else if (lane == 1) {
            // ---- TMA producer and dQ store: per tile its Q and dO (once the previous
            // tile's last S and dP products are done and its rows have formed D~),
            // then the previous tile's dQ (staged by the row threads in the O
            // buffer) goes out by TMA, and once that store has read the buffer this
            // tile's O comes in.  The next tile's Q, dO and O are pulled into L2
            // meanwhile, so their loads at the tile boundary are short.
            // (A packed batch's tail tile stores its dQ rows itself: its tensor map
            // runs on into the next sequence.)
            QTile prev{}, w{}, wn{};
            int vt = 0;
            bool have = next_qtile<PACKED>(sched, a, BN, vt, w);
            for (int u = 0;; ++u) {
                if (have) {
                    if (!wait_bounded<kBwdSuspend>(wc, bar(bars->q_empty), (u & 1) ^ 1, timeout_code(kSiteQEmpty))) break;
                    mbar_arrive_expect_tx(bar(bars->q_full), 2 * C::QT);
                    for (int ch = 0; ch < G::NCH; ++ch) {
                        tma_load_3d(sb + C::OFF_Q + ch * C::QCH, &tm_q, ch * G::CW, w.yq, w.zq, bar(bars->q_full));
                        tma_load_3d(sb + C::OFF_DO + ch * C::QCH, &tm_do, ch * G::CW, w.yq, w.zq, bar(bars->q_full));
                    }
                }
                if (u > 0) {
                    if (!wait_bounded<kBwdSuspend>(wc, bar(bars->dq_staged), (u - 1) & 1, timeout_code(kSiteStage))) break;
                    if (!prev.tail) {
                        for (int ch = 0; ch < G::NCH; ++ch)
                            tma_store_3d(&tm_dq, sb + C::OFF_O + ch * C::QCH, ch * G::CW, prev.yq, prev.zq);
                        bulk_commit();
                        bulk_wait_read0();
                    }
                }
                if (!have) break;
                mbar_arrive_expect_tx(bar(bars->o_full), C::QT);
                for (int ch = 0; ch < G::NCH; ++ch)
                    tma_load_3d(sb + C::OFF_O + ch * C::QCH, &tm_o, ch * G::CW, w.yq, w.zq, bar(bars->o_full));
                const bool have_next = next_qtile<PACKED>(sched, a, BN, vt, wn);
                if (have_next) {
                    for (int ch = 0; ch < G::NCH; ++ch) {
                        tma_prefetch_3d(&tm_q, ch * G::CW, wn.yq, wn.zq);
                        tma_prefetch_3d(&tm_do, ch * G::CW, wn.yq, wn.zq);
                        tma_prefetch_3d(&tm_o, ch * G::CW, wn.yq, wn.zq);
                    }
                }
                prev = w;
                w = wn;
                have = have_next;
            }
        }
    } else if (alive && warp == 2) {
        regs_lower<kDqOtherRegs>();
        if (lane == 0) {
            // ---- TMA producer: the V ring over all blocks of all tiles
            int g = 0;
            bool ok = true;
            int vt = 0;
            QTile w;
            while (ok && next_qtile<PACKED>(sched, a, BN, vt, w)) {
                for (int j = 0; j < w.nk; ++j, ++g) {
                    const int st = g % VST;
                    ok = wait_bounded<kBwdSuspend>(wc, bar(bars->v_empty[st]), ((g / VST) & 1) ^ 1, timeout_code(kSiteVEmpty));
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(bars->v_full[st]), C::KT);
                    for (int ch = 0; ch < G::NCH; ++ch)
                        tma_load_3d(sb + C::OFF_V + st * C::KT + ch * C::KCH, &tm_v, ch * G::CW, w.yk + j * BN, w.zk,
                                    bar(bars->v_full[st]));
                }
            }
        }
    } else if (alive && warp == 1) {
        regs_lower<kDqOtherRegs>();
        {   // the whole warp issues (see mma_ss)
            // ---- MMA issuer.  Per tile: S0 dP0 | PK0 S1 dQ0 dP1 | PK1 S2 dQ1 dP2 | ...
            // PK_j reads P_j from the S columns as soon as the row threads have
            // stored it, so after dS_j only dQ_j and dP_{j+1} stand between the
            // row threads and their next dS.  g counts blocks over all tiles.
            constexpr uint32_t IDS = idesc_bf16(128, BN, false, false);  // S = Q K^T, dP_d = dO V^T
            constexpr uint32_t IDQ = idesc_bf16(128, D, false, true);    // dQ~ += dS~ K, PK += P K
            auto issue_s = [&](int g) -> bool {
                const int st = g % KST;
                if (!wait_warp<kBwdSuspend>(wc, bar(bars->k_full[st]), (g / KST) & 1, timeout_code(kSiteKFull))) return false;
                tc_fence_after();
                const uint32_t kbase = sb + C::OFF_K + st * C::KT;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + C::T_S, G::template desc_k<128>(sb + C::OFF_Q, kk), G::template desc_k<BN>(kbase, kk),
                           IDS, kk > 0 ? 1u : 0u);
                mma_commit(bar(bars->s_full));
                return true;
            };
            auto issue_dp = [&](int g) -> bool {
                const int st = g % VST;
                if (!wait_warp<kBwdSuspend>(wc, bar(bars->v_full[st]), (g / VST) & 1, timeout_code(kSiteVFull))) return false;
                tc_fence_after();
                const uint32_t vbase = sb + C::OFF_V + st * C::KT;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + C::T_DP, G::template desc_k<128>(sb + C::OFF_DO, kk),
                           G::template desc_k<BN>(vbase, kk), IDS, kk > 0 ? 1u : 0u);
                mma_commit(bar(bars->v_empty[st]));
                mma_commit(bar(bars->dp_full));
                return true;
            };
            int g = 0;
            bool ok = true;
            int vt = 0;
            QTile w;
            for (int u = 0; ok && next_qtile<PACKED>(sched, a, BN, vt, w); ++u) {
                const int g0 = g;
                ok = wait_warp<kBwdSuspend>(wc, bar(bars->q_full), u & 1, timeout_code(kSiteQFull));
                if (ok) ok = issue_s(g0);
                if (ok) ok = issue_dp(g0);
                // Q and dO are free once the tile's last S and dP products are done
                if (ok && w.nk == 1) mma_commit(bar(bars->q_empty));
                for (int j = 0; j < w.nk && ok; ++j, ++g) {
                    const int st = g % KST;
                    const uint32_t kbase = sb + C::OFF_K + st * C::KT;
                    ok = wait_warp<kBwdSuspend>(wc, bar(bars->p_full), g & 1, timeout_code(kSitePRead));
                    // the first P K of a tile overwrites PK: the epilogue of the tile
                    // before must have read the accumulators
                    if (ok && j == 0)
                        ok = wait_warp<kBwdSuspend>(wc, bar(bars->acc_free), (u & 1) ^ 1, timeout_code(kSiteAcc));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ts(tmem + C::T_PK, tmem + C::T_S + split_a_col(kk, BN), G::template desc_mn<BN>(kbase, kk),
                               IDQ, (j > 0 || kk > 0) ? 1u : 0u);
                    if (j + 1 < w.nk) {
                        ok = issue_s(g + 1);      // overwrites P_j: after PK_j in the tensor pipe
                        if (!ok) break;
                    }
                    ok = wait_warp<kBwdSuspend>(wc, bar(bars->ds_full), g & 1, timeout_code(kSiteDsFull));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ts(tmem + C::T_DQ, tmem + C::T_DP + split_a_col(kk, BN), G::template desc_mn<BN>(kbase, kk),
                               IDQ, (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(bars->k_empty[st]));
                    if (j + 1 < w.nk) {
                        ok = issue_dp(g + 1);
                        if (ok && j + 2 == w.nk) mma_commit(bar(bars->q_empty));
                    }
                }
                if (ok) mma_commit(bar(bars->acc_done));
            }
            // every MMA must be complete before the CTA releases TMEM
            mma_commit(bar(bars->drain));
            wait_warp<kBwdSuspend>(wc, bar(bars->drain), 0, timeout_code(kSiteDrain));
        }
    } else if (alive && warp >= 12 && DROP) {
        regs_lower<kDqOtherRegs>();
        // ---- RNG warps: the keep bits of every key block, drawn ahead of the
        // row threads into the ring (thread = query row of the tile; two Philox
        // calls of 16 keys per 32-key word, one SWAR test per output word), and
        // handed to the dK/dV kernel when it reads them instead of drawing.
        const int r = (int)threadIdx.x - 12 * 32;
        const KeepSwar8 ks(a.thr);
        int g = 0;
        bool ok = true;
        int vt = 0;
        QTile w;
        while (ok && next_qtile<PACKED>(sched, a, BN, vt, w)) {
            const uint32_t i = (uint32_t)(w.qb * 128 + r);
            const uint32_t bhc = (uint32_t)w.bh + a.bh0;
            for (int j = 0; j < w.nk; ++j, ++g) {
                const int rs = g % C::RNG_ST;
                ok = __all_sync(0xffffffffu, wait_bounded<kBwdSuspend>(wc, bar(bars->rng_empty[rs]), ((g / C::RNG_ST) & 1) ^ 1,
                                                          timeout_code(kSiteRng)));
                if (!ok) break;
                uint32_t* ring = reinterpret_cast<uint32_t*>(smem_raw + pad + C::OFF_RNG + rs * C::RNG_BYTES);
#pragma unroll
                for (int q = 0; q < BN / 32; ++q) {
                    const uint32_t grp = (uint32_t)((j * BN) >> 4) + 2u * (uint32_t)q;
                    const uint4 w0 = philox4x32_10_rk(grp, i, bhc, a.offset, a.rk);
                    const uint4 w1 = philox4x32_10_rk(grp + 1u, i, bhc, a.offset, a.rk);
                    const uint32_t k8[8] = {ks(w0.x), ks(w0.y), ks(w0.z), ks(w0.w),
                                            ks(w1.x), ks(w1.y), ks(w1.z), ks(w1.w)};
                    const uint32_t bits = keep_bits32(k8);
                    ring[q * 128 + r] = bits;
                    if constexpr (MWS) {
                        // key quarter of the 128-key block, query unit (rows 0-63 /
                        // 64-127) and row within it
                        const int kq = ((j * BN) & 127) + 32 * q;
                        const size_t word = mask_pair_word(a, w.bh, w.qb, (j * BN) >> 7) + (size_t)(r >> 6) * 256 +
                                            (size_t)(kq >> 5) * 64 + (size_t)(r & 63);
                        args.mask_ws[word] = bits;
                    }
                }
                mbar_arrive(bar(bars->rng_full[rs]));
            }
        }
    } else if (alive && warp >= 4 && warp < 12) {
        regs_raise<kDqRowRegs>();
        // ---- row threads: query row = TMEM lane, half = which BN/2 keys of a block
        constexpr int HK = BN / 2;
        const RowThread rt = row_thread();
        const int h = rt.half, r = rt.row;
        const uint32_t lane_off = rt.lane_off;
        float* dred = reinterpret_cast<float*>(smem_raw + pad + C::OFF_RED);   // [2 halves][128]
        const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
        const uint64_t zs2 = f2_pack(a.keep_scale, a.keep_scale);
        // -LSE * log2(e) of this thread's query in a tile (-inf past the sequence's
        // end, so its probabilities recompute to 0); the next tile's value is
        // loaded a whole tile ahead of its use.
        auto row_nl2 = [&](const QTile& x) -> float {
            return x.qb * 128 + r < x.lq ? -args.lse[(size_t)x.zq * a.lse_stride + x.yq + r] * 1.44269504088896340736f
                                         : -INFINITY;
        };
        int vt = 0;
        QTile w, wn;
        bool have = next_qtile<PACKED>(sched, a, BN, vt, w);
        float nl2_next = have ? row_nl2(w) : 0.f;
        int g = 0, nx = 0;
        bool ok = true;
        for (int u = 0; ok && have; ++u) {
            const int qb = w.qb, nk = w.nk;
            const int i = qb * 128 + r;              // query of the sequence
            const size_t srow = (size_t)w.ws0 + r;
            const float nl2 = nl2_next;
            const bool have_next = next_qtile<PACKED>(sched, a, BN, vt, wn);
            nl2_next = have_next ? row_nl2(wn) : 0.f;
            if (h == 0) args.lse2_ws[srow] = nl2;
            const uint64_t nl22 = f2_pack(nl2, nl2);
            // The first estimate D~ = rowsum(dO * O) comes from the staged bf16 O
            // and dO tiles (rows past s were filled with zeros by TMA), formed in
            // the first block after its probabilities, which hides the O load;
            // both halves sum the whole row.
            float d_tilde = 0.f;
            uint64_t dt2 = 0, ndt2 = 0;
            uint64_t dacc2 = f2_pack(0.f, 0.f);
            for (int j = 0; j < nk && ok; ++j, ++g) {
                // this block's keep bits from the RNG warps' ring: they need no score, so
                // they are taken (and the slot freed) while the tensor core forms S
                uint32_t kbits[HK / 32];
                if (DROP) {
                    const int rs = g % C::RNG_ST;
                    ok = __all_sync(0xffffffffu, wait_bounded<kBwdSuspend>(wc, bar(bars->rng_full[rs]), (g / C::RNG_ST) & 1,
                                                              timeout_code(kSiteRng)));
                    if (!ok) break;
                    const uint32_t* ring =
                        reinterpret_cast<const uint32_t*>(smem_raw + pad + C::OFF_RNG + rs * C::RNG_BYTES);
#pragma unroll
                    for (int c32 = 0; c32 < HK / 32; ++c32) kbits[c32] = ring[(h * (HK / 32) + c32) * 128 + r];
                    mbar_arrive(bar(bars->rng_empty[rs]));
                }
                ok = __all_sync(0xffffffffu, wait_bounded<kBwdSuspend>(wc, bar(bars->s_full), g & 1, timeout_code(kSiteSFull)));
                if (!ok) break;
                tc_fence_after();
                uint64_t pp[HK / 2];
                if constexpr (HK == 64) {
                    uint32_t rr[64];
                    tmem_ld64(tmem + C::T_S + lane_off + HK * h, rr);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        pp[e] = f2_pack(__uint_as_float(rr[2 * e]), __uint_as_float(rr[2 * e + 1]));
                } else {
                    uint32_t rr[32];
                    tmem_ld32(tmem + C::T_S + lane_off + HK * h, rr);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pp[e] = f2_pack(__uint_as_float(rr[2 * e]), __uint_as_float(rr[2 * e + 1]));
                }
                const int key0 = j * BN + HK * h;
                // Scores of keys this query does not see (past the diagonal, or past the
                // last key) become -inf before the exponential; only the blocks that
                // hold such keys run this (a uniform branch), the others go straight on.
                const int k_end = a.causal ? min(i + 1, w.lk) : w.lk;    // first key not seen
                if (key0 + HK > (a.causal ? min(qb * 128, w.lk) : w.lk)) {
#pragma unroll
                    for (int e = 0; e < HK / 2; ++e) {
                        float lo, hi;
                        f2_unpack(pp[e], lo, hi);
                        if (key0 + 2 * e >= k_end) lo = -INFINITY;
                        if (key0 + 2 * e + 1 >= k_end) hi = -INFINITY;
                        pp[e] = f2_pack(lo, hi);
                    }
                }
#pragma unroll
                for (int e = 0; e < HK / 2; ++e) {
                    float lo, hi;
                    f2_unpack(f2_fma(pp[e], sc2, nl22), lo, hi);
                    pp[e] = f2_pack(ex2_approx(lo), ex2_approx(hi));
                }
                // P (before dropout) over the first HK/2 of this half's S columns, for PK += P K
                {
                    uint32_t pw[HK / 2];
#pragma unroll
                    for (int e = 0; e < HK / 2; ++e) pw[e] = pack_bf16x2(pp[e]);
                    if constexpr (HK / 2 == 32) {
                        tmem_st32(tmem + C::T_S + lane_off + HK * h, pw);
                    } else {
                        tmem_st16(tmem + C::T_S + lane_off + HK * h, pw);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(bars->p_full));
                if (j == 0) {
                    ok = __all_sync(0xffffffffu, wait_bounded<kBwdSuspend>(wc, bar(bars->o_full), u & 1, timeout_code(kSiteOFull)));
                    if (ok)
                        ok = __all_sync(0xffffffffu,
                                        wait_bounded<kBwdSuspend>(wc, bar(bars->q_full), u & 1, timeout_code(kSiteQFull)));
                    if (!ok) break;
                    uint64_t acc2 = f2_pack(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < D / 8; ++c) {
                        const uint32_t off = G::template unit_offset<128>(r, 8 * c);
                        const uint4 ov = ld_shared_v4(sb + C::OFF_O + off);
                        const uint4 gv = ld_shared_v4(sb + C::OFF_DO + off);
                        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
                        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            acc2 = f2_fma(f2_pack(__uint_as_float(ow[e] << 16), __uint_as_float(ow[e] & 0xFFFF0000u)),
                                          f2_pack(__uint_as_float(gw[e] << 16), __uint_as_float(gw[e] & 0xFFFF0000u)),
                                          acc2);
                    }
                    mbar_arrive(bar(bars->q_empty));    // this thread has read dO
                    float lo, hi;
                    f2_unpack(acc2, lo, hi);
                    d_tilde = lo + hi;
                    dt2 = f2_pack(d_tilde, d_tilde);
                    ndt2 = f2_pack(-d_tilde, -d_tilde);
                }
                // The keep decisions of this half's keys, from the RNG warps' bits: keys
                // 4k .. 4k + 3 of each 32 as the byte sign bits of keep[k] (one shift
                // and one mask per word, the inverse of keep_bits32).
                uint32_t keep[HK / 4];
                if (DROP) {
#pragma unroll
                    for (int c32 = 0; c32 < HK / 32; ++c32) {
#pragma unroll
                        for (int k = 0; k < 8; ++k) keep[8 * c32 + k] = (kbits[c32] << k) & 0x80808080u;
                    }
                }
                ok = __all_sync(0xffffffffu, wait_bounded<kBwdSuspend>(wc, bar(bars->dp_full), g & 1, timeout_code(kSiteDpFull)));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c32 = 0; c32 < HK / 32; ++c32) {
                    uint32_t rr[32];
                    tmem_ld32(tmem + C::T_DP + lane_off + HK * h + c32 * 32, rr);
                    uint32_t wd[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {               // pair e: keys 2e, 2e + 1 of the chunk
                        const int ep = c32 * 16 + e;
                        uint32_t dlo = rr[2 * e], dhi = rr[2 * e + 1];
                        if (DROP) {
                            // dropped elements' dP_d is cleared; kept ones carry 1/(1-p) below
                            dlo &= keep_mask32(keep[8 * c32 + (e >> 1)], 2 * (e & 1));
                            dhi &= keep_mask32(keep[8 * c32 + (e >> 1)], 2 * (e & 1) + 1);
                        }
                        const uint64_t dp = f2_pack(__uint_as_float(dlo), __uint_as_float(dhi));
                        dacc2 = f2_fma(pp[ep], dp, dacc2);
                        wd[e] = pack_bf16x2(f2_mul(pp[ep], DROP ? f2_fma(dp, zs2, ndt2) : f2_sub(dp, dt2)));
                    }
                    tmem_st16(tmem + C::T_DP + lane_off + HK * h + c32 * 16, wd);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(bars->ds_full));
            }
            if (!ok) break;
            // ---- epilogue: the exact row statistic from both halves, then
            // dQ = scale (dQ~ - (D - D~) PK), staged in the O buffer (its O was
            // read for D~ before the exchange below) for the producer's TMA store
            float d_exact;
            {
                float lo, hi;
                f2_unpack(dacc2, lo, hi);
                d_exact = DROP ? (lo + hi) * a.keep_scale : lo + hi;   // dP = Z dP_d, Z = keep / (1 - p)
            }
            dred[h * 128 + r] = d_exact;
            ok = __all_sync(0xffffffffu, row_barrier<kBwdSuspend>(wc, bar(bars->xbar), nx++ & 1, timeout_code(kSiteX)));
            if (!ok) break;
            d_exact += dred[(h ^ 1) * 128 + r];
            // every row thread has read the region before anyone writes it again
            ok = __all_sync(0xffffffffu, row_barrier<kBwdSuspend>(wc, bar(bars->xbar), nx++ & 1, timeout_code(kSiteX)));
            if (!ok) break;
            ok = __all_sync(0xffffffffu, wait_bounded<kBwdSuspend>(wc, bar(bars->acc_done), u & 1, timeout_code(kSiteAcc)));
            if (!ok) break;
            tc_fence_after();
            const float eps = d_exact - d_tilde;
#pragma unroll 1
            for (int c32 = h; c32 < D / 32; c32 += 2) {
                uint32_t rq[32], rp[32];
                tmem_ld32(tmem + C::T_DQ + lane_off + c32 * 32, rq);
                tmem_ld32(tmem + C::T_PK + lane_off + c32 * 32, rp);
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    rq[c] = __float_as_uint(fmaf(-eps, __uint_as_float(rp[c]), __uint_as_float(rq[c])));
                if (!w.tail) {
                    stage_row32<D, 128>(sb + C::OFF_O, r, c32 * 32, rq, a.scale);
                } else if (i < w.lq) {
                    // a packed batch's tail tile: this row straight to global memory
                    uint4* qrow = reinterpret_cast<uint4*>(args.dq + (size_t)w.zq * args.q_head_stride +
                                                           (size_t)(w.yq + r) * args.q_row_stride) + c32 * 4;
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4) {
                        uint32_t wv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            wv[e] = pack_bf16x2(__uint_as_float(rq[8 * u4 + 2 * e]) * a.scale,
                                                __uint_as_float(rq[8 * u4 + 2 * e + 1]) * a.scale);
                        qrow[u4] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(bars->acc_free));   // the next tile's P K and dQ may overwrite them
            fence_proxy_async_smem();
            mbar_arrive(bar(bars->dq_staged));
            if (h == 0) args.delta_ws[srow] = -d_exact;    // the dK/dV kernel adds it
            w = wn;
            have = have_next;
        }
    } else if (alive) {
        regs_lower<kDqOtherRegs>();   // idle warps (and the RNG warps without dropout)
    }
    __syncthreads();
    if (bars->abort_flag) {
        for (int k = 0; k < 20; ++k) __nanosleep(50000);
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ========================================================== launchers ====

template <int D, bool DROP, bool MWS, bool PACKED>
static int launch_dkdv_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv, const BwdArgs& a,
                         cudaStream_t stream)
{
    constexpr uint32_t smem = DkdvCfg<D>::SMEM;
    auto kern = attn_bwd_dkdv_kernel<D, DROP, MWS, PACKED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    const unsigned n_bkv = (unsigned)(a.c.n_bh / a.c.h_q * a.c.h_kv);
    const unsigned tiles = (unsigned)dkdv_key_blocks<PACKED>(a.c) * n_bkv;
    const unsigned grid = tiles < (unsigned)a.num_sms ? tiles : (unsigned)a.num_sms;   // persistent
    kern<<<grid, kThreads, smem, stream>>>(tq, tk, tv, tdo, tdk, tdv, a);
    return (int)cudaGetLastError();
}

template <int D, bool DROP, bool MWS, bool PACKED>
static int launch_dq_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& to, const CUtensorMap& tdq, const BwdArgs& a, cudaStream_t stream)
{
    constexpr uint32_t smem = DqCfg<D>::SMEM;
    auto kern = attn_bwd_dq_kernel<D, DROP, MWS, PACKED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    // the row warps' register raise waits until the others' shares are free:
    // refuse a build whose register count cannot cover the shares
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return (int)e;
    if (fa.numRegs * kThreadsRng < reg_shares(kDqRowRegs, kDqOtherRegs, kThreadsRng))
        return (int)cudaErrorInvalidConfiguration;
    const unsigned tiles = (unsigned)a.c.n_blk * (unsigned)a.c.n_bh;
    const unsigned grid = tiles < (unsigned)a.num_sms ? tiles : (unsigned)a.num_sms;
    kern<<<grid, kThreadsRng, smem, stream>>>(tq, tk, tv, tdo, to, tdq, a);
    return (int)cudaGetLastError();
}

int launch_bwd_dkdv(int d, bool dropout, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                    const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv, const BwdArgs& a,
                    cudaStream_t stream)
{
#define AC_DKDV_CASE(DD)                                                                            \
    case DD:                                                                                        \
        return a.c.cu_q ? (!dropout ? launch_dkdv_t<DD, false, false, true>(tq, tk, tv, tdo, tdk, tdv, a, stream) \
                                    : launch_dkdv_t<DD, true, false, true>(tq, tk, tv, tdo, tdk, tdv, a, stream))  \
               : !dropout  ? launch_dkdv_t<DD, false, false, false>(tq, tk, tv, tdo, tdk, tdv, a, stream)          \
               : a.mask_ws ? launch_dkdv_t<DD, true, true, false>(tq, tk, tv, tdo, tdk, tdv, a, stream)            \
                           : launch_dkdv_t<DD, true, false, false>(tq, tk, tv, tdo, tdk, tdv, a, stream);
    switch (d) {
        AC_DKDV_CASE(64)
        AC_DKDV_CASE(96)
        AC_DKDV_CASE(128)
        AC_DKDV_CASE(160)
        default: return (int)cudaErrorInvalidValue;
    }
#undef AC_DKDV_CASE
}

int launch_bwd_dq(int d, bool dropout, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                  const CUtensorMap& tdo, const CUtensorMap& to, const CUtensorMap& tdq, const BwdArgs& a,
                  cudaStream_t stream)
{
#define AC_DQ_CASE(DD)                                                                              \
    case DD:                                                                                        \
        return a.c.cu_q ? (!dropout ? launch_dq_t<DD, false, false, true>(tq, tk, tv, tdo, to, tdq, a, stream) \
                                    : launch_dq_t<DD, true, false, true>(tq, tk, tv, tdo, to, tdq, a, stream))  \
               : !dropout  ? launch_dq_t<DD, false, false, false>(tq, tk, tv, tdo, to, tdq, a, stream)          \
               : a.mask_ws ? launch_dq_t<DD, true, true, false>(tq, tk, tv, tdo, to, tdq, a, stream)            \
                           : launch_dq_t<DD, true, false, false>(tq, tk, tv, tdo, to, tdq, a, stream);
    switch (d) {
        AC_DQ_CASE(64)
        AC_DQ_CASE(96)
        AC_DQ_CASE(128)
        AC_DQ_CASE(160)
        default: return (int)cudaErrorInvalidValue;
    }
#undef AC_DQ_CASE
}

}  // namespace ac
