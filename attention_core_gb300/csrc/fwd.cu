// fwd.cu -- forward pass of the attention core on sm_103a.
//
// Computes, for one (query head, 128-query block) per CTA,
//     S = scale * Q K^T  (causal: key j visible to query i iff j <= i),
//     P = softmax(S) row-wise, P_d = P * M / (1 - p)  (softmax dropout),
//     O = P_d V,  LSE_i = ln sum_j exp(S_ij),
// and stores only O and LSE: the scores, probabilities and mask never reach
// global memory.  This is the attention core that selective activation
// recomputation discards after the forward pass ("Reducing Activation
// Recomputation in Large Transformer Models", Key takeaways, fourth bullet;
// "Recomputing Activations", "Memory for compute, selectively").
//
// Structure of a CTA (384 threads):
//   warp 0  TMA: Q once, then K blocks into a ring of stages
//   warp 2  TMA: V blocks into their own ring
//   warp 1  one thread issues tcgen05 MMAs: S_j = Q K_j^T into one of two
//           TMEM score buffers, then O += P_{j-1} V_{j-1} with P read from TMEM
//   warps 4-11  two warpgroups on the same 128 query rows (TMEM lanes), one
//           per half of the 128 keys of a block: online softmax in the log2
//           domain (the halves swap their row maxima through shared memory),
//           dropout from Philox, P_d written back to TMEM as bf16 inside the
//           half's own score columns; epilogue O / l -> bf16 -> TMA store.
// The running maximum is only moved (and O rescaled in TMEM) when it grows by
// more than 2^8, so most blocks skip the rescale; O / l is exact either way.
#include "kernels.h"
#include "philox.cuh"
#include "ptx.cuh"
#include "tile.cuh"

namespace ac {

namespace {

template <int D>
struct FwdCfg {
    using G = TileGeom<D>;
    static constexpr uint32_t TILE = G::template tile_bytes<128>();
    static constexpr uint32_t CHUNK = G::template chunk_bytes<128>();
    static constexpr int ST = (D <= 96) ? 4 : 2;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = TILE;
    static constexpr uint32_t OFF_V = TILE * (1 + ST);
    static constexpr uint32_t OFF_BAR = TILE * (1 + 2 * ST);
    static constexpr uint32_t OFF_RED = OFF_BAR + 256;          // [2 buffers][2 halves][128] row maxima
    static constexpr uint32_t OFF_LRED = OFF_RED + 2 * 2 * 128 * 4;  // [2 halves][128] row sums
    static constexpr uint32_t SMEM = OFF_LRED + 2 * 128 * 4 + 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    // TMEM columns: two score buffers, then the O accumulator.
    static constexpr uint32_t T_S0 = 0, T_S1 = 128, T_O = 256;
    static_assert(T_O + D <= 512, "TMEM budget");
};

struct FwdBars {
    uint64_t q_full;
    uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
    uint64_t s_full[2], p_full[2];
    uint64_t o_done;
    uint64_t xmax[2];      // row-max exchange between the two column halves
    uint64_t never;
    uint32_t tmem_base;
    int32_t abort_flag;
};

// Wait sites reported in bits 8.. of the status word on a timeout.
enum : int32_t {
    kSiteInject = 1, kSiteKEmpty, kSiteVEmpty, kSiteQFull, kSiteKFull, kSiteVFull, kSitePFull,
    kSiteSFull, kSiteODone, kSiteXmax
};
__device__ __forceinline__ int32_t timeout_code(int32_t site) { return 6 | (site << 8); }

}  // namespace

template <int D, bool DROP>
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

    const int n_bh = a.n_bh;
    const int qb = a.n_blk - 1 - (int)(blockIdx.x / n_bh);   // longest causal rows first
    const int bh = (int)(blockIdx.x % n_bh);
    const int group = a.h_q / a.h_kv;
    const int bkv = (bh / a.h_q) * a.h_kv + (bh % a.h_q) / group;
    const int nk = a.causal ? (qb + 1) : a.n_blk;
    const uint32_t warp = warp_id(), lane = lane_id();

    if (threadIdx.x == 0) {
        mbar_init(bar(bars->q_full), 1);
        for (int st = 0; st < ST; ++st) {
            mbar_init(bar(bars->k_full[st]), 1);
            mbar_init(bar(bars->k_empty[st]), 1);
            mbar_init(bar(bars->v_full[st]), 1);
            mbar_init(bar(bars->v_empty[st]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(bars->s_full[b]), 1);
            mbar_init(bar(bars->p_full[b]), kRowThreads);
            mbar_init(bar(bars->xmax[b]), kRowThreads);
        }
        mbar_init(bar(bars->o_done), 1);
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
            // ---- TMA producer: Q, then the K ring
            mbar_arrive_expect_tx(bar(bars->q_full), C::TILE);
            for (int ch = 0; ch < G::NCH; ++ch)
                tma_load_3d(sb + C::OFF_Q + ch * C::CHUNK, &tm_q, ch * G::CW, qb * 128, bh, bar(bars->q_full));
            for (int j = 0; j < nk; ++j) {
                const int st = j % ST;
                if (!wait_bounded(wc, bar(bars->k_empty[st]), ((j / ST) & 1) ^ 1, timeout_code(kSiteKEmpty)))
                    break;
                mbar_arrive_expect_tx(bar(bars->k_full[st]), C::TILE);
                for (int ch = 0; ch < G::NCH; ++ch)
                    tma_load_3d(sb + C::OFF_K + st * C::TILE + ch * C::CHUNK, &tm_k, ch * G::CW, j * 128, bkv,
                                bar(bars->k_full[st]));
            }
        }
    } else if (alive && warp == 2) {
        if (lane == 0) {
            // ---- TMA producer: the V ring
            for (int j = 0; j < nk; ++j) {
                const int st = j % ST;
                if (!wait_bounded(wc, bar(bars->v_empty[st]), ((j / ST) & 1) ^ 1, timeout_code(kSiteVEmpty)))
                    break;
                mbar_arrive_expect_tx(bar(bars->v_full[st]), C::TILE);
                for (int ch = 0; ch < G::NCH; ++ch)
                    tma_load_3d(sb + C::OFF_V + st * C::TILE + ch * C::CHUNK, &tm_v, ch * G::CW, j * 128, bkv,
                                bar(bars->v_full[st]));
            }
        }
    } else if (alive && warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer
            constexpr uint32_t IDS = idesc_bf16(128, 128, false, false);  // S = Q K^T
            constexpr uint32_t IDO = idesc_bf16(128, D, false, true);     // O += P V
            bool ok = wait_bounded(wc, bar(bars->q_full), 0, timeout_code(kSiteQFull));
            auto issue_pv = [&](int i) -> bool {
                if (!wait_bounded(wc, bar(bars->p_full[i & 1]), (i >> 1) & 1, timeout_code(kSitePFull)))
                    return false;
                const int st = i % ST;
                if (!wait_bounded(wc, bar(bars->v_full[st]), (i / ST) & 1, timeout_code(kSiteVFull)))
                    return false;
                tc_fence_after();
                const uint32_t vbase = sb + C::OFF_V + st * C::TILE;
                const uint32_t tP = tmem + ((i & 1) ? C::T_S1 : C::T_S0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tmem + C::T_O, tP + split_a_col(kk, 128), G::template desc_mn<128>(vbase, kk), IDO,
                           (i > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(bars->v_empty[st]));
                mma_commit(bar(bars->o_done));
                return true;
            };
            for (int j = 0; j < nk && ok; ++j) {
                const int st = j % ST;
                ok = wait_bounded(wc, bar(bars->k_full[st]), (j / ST) & 1, timeout_code(kSiteKFull));
                if (!ok) break;
                tc_fence_after();
                const uint32_t kbase = sb + C::OFF_K + st * C::TILE;
                const uint32_t tS = tmem + ((j & 1) ? C::T_S1 : C::T_S0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tS, G::template desc_k<128>(sb + C::OFF_Q, kk), G::template desc_k<128>(kbase, kk),
                           IDS, kk > 0 ? 1u : 0u);
                mma_commit(bar(bars->k_empty[st]));
                mma_commit(bar(bars->s_full[j & 1]));
                if (j > 0) ok = issue_pv(j - 1);
            }
            if (ok) issue_pv(nk - 1);
        }
    } else if (alive && warp >= 4) {
        // ---- softmax / epilogue: row = TMEM lane, half = which 64 keys of a block
        const RowThread rt = row_thread();
        const int h = rt.half, r = rt.row;
        const uint32_t lane_off = rt.lane_off;
        const int i = qb * 128 + r;
        const uint32_t t16 = a.thr << 16;
        float* xmax = reinterpret_cast<float*>(smem_raw + pad + C::OFF_RED);
        float* lred = reinterpret_cast<float*>(smem_raw + pad + C::OFF_LRED);
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < nk; ++j) {
            const uint32_t tS = tmem + ((j & 1) ? C::T_S1 : C::T_S0) + lane_off + 64 * h;
            ok = __all_sync(0xffffffffu,
                            wait_bounded(wc, bar(bars->s_full[j & 1]), (j >> 1) & 1, timeout_code(kSiteSFull)));
            if (!ok) break;
            tc_fence_after();
            float x[64];
#pragma unroll
            for (int c32 = 0; c32 < 2; ++c32) {
                uint32_t rr[32];
                tmem_ld32(tS + c32 * 32, rr);
#pragma unroll
                for (int e = 0; e < 32; ++e) x[c32 * 32 + e] = __uint_as_float(rr[e]);
            }
            const int key0 = j * 128 + 64 * h;
            if (a.causal && j == qb) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (64 * h + c > r) x[c] = -INFINITY;
            }
            if (!a.causal && key0 + 64 > a.s) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (key0 + c >= a.s) x[c] = -INFINITY;
            }
            float mx = x[0];
#pragma unroll
            for (int c = 1; c < 64; ++c) mx = fmaxf(mx, x[c]);
            // swap block maxima with the other half of the row
            xmax[((j & 1) * 2 + h) * 128 + r] = mx;
            ok = __all_sync(0xffffffffu, row_barrier(wc, bar(bars->xmax[j & 1]), (j >> 1) & 1,
                                                     timeout_code(kSiteXmax)));
            if (!ok) break;
            mx = fmaxf(mx, xmax[((j & 1) * 2 + (h ^ 1)) * 128 + r]);
            const float m_new = fmaxf(m_run, mx * a.scale_log2);
            if (__any_sync(0xffffffffu, m_new > m_run + 8.0f)) {
                if (j > 0) {
                    ok = __all_sync(0xffffffffu, wait_bounded(wc, bar(bars->o_done), (j - 1) & 1,
                                                              timeout_code(kSiteODone)));
                    if (!ok) break;
                    tc_fence_after();
                    const float f = ex2_approx(m_run - m_new);
                    l_run *= f;
#pragma unroll 1
                    for (int c32 = h; c32 < D / 32; c32 += 2) {
                        uint32_t rr[32];
                        tmem_ld32(tmem + C::T_O + lane_off + c32 * 32, rr);
#pragma unroll
                        for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * f);
                        tmem_st32(tmem + C::T_O + lane_off + c32 * 32, rr);
                    }
                    tmem_st_wait();
                }
                m_run = m_new;
            }
            const float neg_m = -m_run;
            float lsum = 0.f;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float pv = ex2_approx(fmaf(x[c], a.scale_log2, neg_m));
                lsum += pv;
                x[c] = pv;
            }
            l_run += lsum;
            uint32_t pw[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) pw[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
            if (DROP) {
                // group g covers keys key0 + 8g .. +7: words 4g .. 4g+3 of pw
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const uint4 w4 = philox4x32_10((uint32_t)(key0 >> 3) + g, (uint32_t)i, (uint32_t)bh, a.offset,
                                                   a.seed_lo, a.seed_hi);
                    pw[4 * g + 0] &= keep_mask16x2(w4.x, t16);
                    pw[4 * g + 1] &= keep_mask16x2(w4.y, t16);
                    pw[4 * g + 2] &= keep_mask16x2(w4.z, t16);
                    pw[4 * g + 3] &= keep_mask16x2(w4.w, t16);
                }
            }
            tmem_st32(tS, pw);   // P_d of these 64 keys over the first 32 of the half's columns
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(bars->p_full[j & 1]));
        }
        // row sum over both halves (every row thread reaches this point once)
        lred[h * 128 + r] = l_run;
        named_barrier_sync(1, kRowThreads);
        const float l_tot = l_run + lred[(h ^ 1) * 128 + r];
        if (ok)
            ok = __all_sync(0xffffffffu,
                            wait_bounded(wc, bar(bars->o_done), (nk - 1) & 1, timeout_code(kSiteODone)));
        if (ok) {
            tc_fence_after();
            const float inv = a.keep_scale / l_tot;
#pragma unroll 1
            for (int c32 = h; c32 < D / 32; c32 += 2) {
                uint32_t rr[32];
                tmem_ld32(tmem + C::T_O + lane_off + c32 * 32, rr);
                stage_row32<D, 128>(sb + C::OFF_Q, r, c32 * 32, rr, inv);
            }
            if (h == 0 && i < a.s) args.lse[(size_t)bh * a.s + i] = (m_run + log2f(l_tot)) * 0.693147180559945309f;
        }
        fence_proxy_async_smem();
        named_barrier_sync(1, kRowThreads);
        if (h == 0 && r == 0 && !bars->abort_flag) {
            for (int ch = 0; ch < G::NCH; ++ch)
                tma_store_3d(&tm_o, sb + C::OFF_Q + ch * C::CHUNK, ch * G::CW, qb * 128, bh);
            bulk_commit();
            bulk_wait_read0();
        }
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

template <int D, bool DROP>
static int launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& to, const FwdArgs& a, cudaStream_t stream)
{
    constexpr uint32_t smem = FwdCfg<D>::SMEM;
    auto kern = attn_fwd_kernel<D, DROP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    const unsigned grid = (unsigned)a.c.n_blk * (unsigned)a.c.n_bh;
    kern<<<grid, kThreads, smem, stream>>>(tq, tk, tv, to, a);
    return (int)cudaGetLastError();
}

int launch_fwd(int d, bool dropout, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& to, const FwdArgs& a, cudaStream_t stream)
{
#define AC_FWD_CASE(DD)                                                                             \
    case DD:                                                                                        \
        return dropout ? launch_fwd_t<DD, true>(tq, tk, tv, to, a, stream)                          \
                       : launch_fwd_t<DD, false>(tq, tk, tv, to, a, stream);
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
