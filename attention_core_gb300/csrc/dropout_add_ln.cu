// dropout_add_ln.cu -- dropout, residual add and layer norm at a residual
// sub-layer boundary, on either side of the attention core:
//     z = residual + dropout(x),   y = gamma * (z - mean) * rstd + beta,
// per row (token) over the hidden size H, rstd = 1 / sqrt(var + eps) with the
// biased variance.  These are the layer norms and dropouts that tensor
// parallelism leaves replicated and that act on every position independently
// ("Reducing Activation Recomputation in Large Transformer Models", Key
// takeaways, first and second bullets).  As in the attention core, the
// backward redraws the dropout mask from (seed, offset) instead of reading a
// stored one: the block keeps z (bf16), mean and rstd.
//
// Mask: Philox-4x32-10 with key (seed lo, seed hi) and counter (col / 8, row,
// 0xFFFFFFFF, offset); column col takes the low (even) or high (odd) 16-bit
// half of word (col % 8) / 2 and is dropped iff that draw < thr.  Word 2 is a
// value no attention-core head index takes, so the two never share a counter.
//
// HBM-bound.  Each thread owns 8-column vectors (16-byte bf16 loads and
// stores; one Philox call per vector), a CTA walks rows with a grid stride.
#include "kernels.h"
#include "philox.cuh"
#include "tile.cuh"

namespace ac {

namespace {

constexpr uint32_t kDalStream = 0xFFFFFFFFu;   // Philox counter word 2 of this block's mask

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        f[2 * e] = __uint_as_float(w[e] << 16);
        f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8])
{
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// Keep flags of the 8 columns 8v .. 8v + 7 of one row (bit e: column 8v + e).
__device__ __forceinline__ uint32_t dal_keep8(const DalArgs& a, uint32_t v, uint32_t row)
{
    const uint4 w = philox4x32_10_rk(v, row, kDalStream, a.offset, a.rk);
    const uint32_t t16 = a.thr << 16;
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint32_t bits = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        bits |= ((ws[e] << 16) >= t16 ? 1u : 0u) << (2 * e);
        bits |= (ws[e] >= t16 ? 1u : 0u) << (2 * e + 1);
    }
    return bits;
}

// Sum over the CTA (every thread gets the result).  `red` holds one slot per warp.
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();                 // previous use of red is finished
    if (l == 0) red[w] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) s += red[i];
    return s;
}

constexpr int kFwdThreads = 256;

}  // namespace

// Bounded wait on an mbarrier phase: false if it did not complete in time.
__device__ __forceinline__ bool dal_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > limit_ns) return false;
    return true;
}

// Forward: NV 8-column vectors per thread (H <= 8 * kFwdThreads * NV).  Thread 0
// keeps the CTA's next two rows of x and the residual in flight: bulk copies
// into two shared-memory stages, each completing an mbarrier.  A stage is
// refilled as soon as every thread has read it (after the first reduction).
template <int NV, bool DROP>
__global__ void __launch_bounds__(kFwdThreads)
dal_fwd_kernel(const DalArgs a)
{
    extern __shared__ __align__(128) uint8_t stage_raw[];   // [2][x row | residual row] bf16
    __shared__ float red[kFwdThreads / 32];
    __shared__ __align__(8) uint64_t full[2];
    const int H = a.hidden;
    const uint32_t row_bytes = (uint32_t)H * 2u;
    const float inv_h = 1.0f / (float)H;
    const int G = gridDim.x;
    const uint32_t sbase = smem_u32(stage_raw);
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&full[0]), 1);
        mbar_init(smem_u32(&full[1]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int row, int st) {
        const uint32_t bar = smem_u32(&full[st]);
        mbar_arrive_expect_tx(bar, 2u * row_bytes);
        bulk_load_1d(sbase + (uint32_t)st * 2u * row_bytes, a.x + (size_t)row * H, row_bytes, bar);
        bulk_load_1d(sbase + (uint32_t)st * 2u * row_bytes + row_bytes, a.residual + (size_t)row * H, row_bytes,
                     bar);
    };
    if (threadIdx.x == 0) {
        if ((int)blockIdx.x < a.n_rows) issue(blockIdx.x, 0);
        if ((int)blockIdx.x + G < a.n_rows) issue(blockIdx.x + G, 1);
    }
    int it = 0;
    for (int row = blockIdx.x; row < a.n_rows; row += G, ++it) {
        const int st = it & 1;
        const bool ok = dal_wait(smem_u32(&full[st]), (uint32_t)(it >> 1) & 1u, a.timeout_ns);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0 && a.status) atomicCAS(a.status, 0, 6 | (1 << 8));
            __nanosleep(1000000);          // let copies already issued land before the CTA exits
            return;
        }
        const uint32_t xs = sbase + (uint32_t)st * 2u * row_bytes, rs = xs + row_bytes;
        const size_t base = (size_t)row * H;
        float zf[NV][8];
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = threadIdx.x + kFwdThreads * k;
            if (8 * v < H) {
                float xf[8], rf[8];
                bf16x8_to_f32(ld_shared_v4(xs + 16u * (uint32_t)v), xf);
                bf16x8_to_f32(ld_shared_v4(rs + 16u * (uint32_t)v), rf);
                const uint32_t keep = DROP ? dal_keep8(a, (uint32_t)v, (uint32_t)row) : 0xFFu;
#pragma unroll
                for (int e = 0; e < 8; ++e) zf[k][e] = ((keep >> e) & 1u) ? fmaf(xf[e], a.keep_scale, rf[e]) : rf[e];
                const uint4 zb = f32_to_bf16x8(zf[k]);
                *reinterpret_cast<uint4*>(a.z + base + 8 * v) = zb;
                bf16x8_to_f32(zb, zf[k]);          // the layer norm reads the stored z
#pragma unroll
                for (int e = 0; e < 8; ++e) s += zf[k][e];
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) zf[k][e] = 0.f;
            }
        }
        const float mean = block_sum<kFwdThreads>(s, red) * inv_h;
        // every thread has read this stage: refill it with the row after next
        if (threadIdx.x == 0 && row + 2 * G < a.n_rows) issue(row + 2 * G, st);
        float q = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (8 * (threadIdx.x + kFwdThreads * k) < H) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float d = zf[k][e] - mean;
                    q = fmaf(d, d, q);
                }
            }
        }
        const float rstd = rsqrtf(block_sum<kFwdThreads>(q, red) * inv_h + a.eps);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = threadIdx.x + kFwdThreads * k;
            if (8 * v < H) {
                const float4 g0 = *reinterpret_cast<const float4*>(a.gamma + 8 * v);
                const float4 g1 = *reinterpret_cast<const float4*>(a.gamma + 8 * v + 4);
                const float4 b0 = *reinterpret_cast<const float4*>(a.beta + 8 * v);
                const float4 b1 = *reinterpret_cast<const float4*>(a.beta + 8 * v + 4);
                const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                float yf[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) yf[e] = fmaf((zf[k][e] - mean) * rstd, g[e], b[e]);
                *reinterpret_cast<uint4*>(a.y + base + 8 * v) = f32_to_bf16x8(yf);
            }
        }
        if (threadIdx.x == 0) {
            a.mean[row] = mean;
            a.rstd[row] = rstd;
        }
    }
}

// Backward: NV 8-column vectors per thread (H <= 8 * NT * NV).  The
// per-column sums for dgamma and dbeta accumulate over the CTA's rows in
// shared memory ([2][H] fp32; each column belongs to one thread, so no
// synchronisation) and are written once, as this CTA's row of the partial-sum
// workspace.
// Up to 8192 columns, 256-thread CTAs (two or more per SM) overlap one CTA's
// reductions and stores with another's loads; above, 512 threads, one CTA per
// SM, which halves the partial-sum rows.
template <int NV, bool DROP, int NT>
__global__ void __launch_bounds__(NT, NT == 256 ? 2 : 1)
dal_bwd_kernel(const DalArgs a)
{
    extern __shared__ float4 acc4[];
    __shared__ float red[NT / 32];
    const int H = a.hidden;
    const float inv_h = 1.0f / (float)H;
    float* acc_g = reinterpret_cast<float*>(acc4);
    float* acc_b = acc_g + H;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int v = threadIdx.x + NT * k;
        if (8 * v < H) {
            const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
            reinterpret_cast<float4*>(acc_g)[2 * v] = z4;
            reinterpret_cast<float4*>(acc_g)[2 * v + 1] = z4;
            reinterpret_cast<float4*>(acc_b)[2 * v] = z4;
            reinterpret_cast<float4*>(acc_b)[2 * v + 1] = z4;
        }
    }

    for (int row = blockIdx.x; row < a.n_rows; row += gridDim.x) {
        const size_t base = (size_t)row * H;
        const float mean = a.mean[row], rstd = a.rstd[row];
        uint4 dyv[NV], zv[NV], nv4[NV];
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = threadIdx.x + NT * k;
            if (8 * v < H) {
                dyv[k] = *reinterpret_cast<const uint4*>(a.dy + base + 8 * v);
                zv[k] = *reinterpret_cast<const uint4*>(a.z + base + 8 * v);
                nv4[k] = a.dz_next ? *reinterpret_cast<const uint4*>(a.dz_next + base + 8 * v) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = threadIdx.x + NT * k;
            if (8 * v < H) {
                float dyf[8], zf[8];
                bf16x8_to_f32(dyv[k], dyf);
                bf16x8_to_f32(zv[k], zf);
                const float4 g0 = *reinterpret_cast<const float4*>(a.gamma + 8 * v);
                const float4 g1 = *reinterpret_cast<const float4*>(a.gamma + 8 * v + 4);
                const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                float4* ag = reinterpret_cast<float4*>(acc_g) + 2 * v;
                float4* ab = reinterpret_cast<float4*>(acc_b) + 2 * v;
                float4 ag0 = ag[0], ag1 = ag[1], ab0 = ab[0], ab1 = ab[1];
                float xh[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    xh[e] = (zf[e] - mean) * rstd;
                    const float gg = dyf[e] * g[e];
                    s1 += gg;
                    s2 = fmaf(gg, xh[e], s2);
                }
                ag0.x = fmaf(dyf[0], xh[0], ag0.x); ag0.y = fmaf(dyf[1], xh[1], ag0.y);
                ag0.z = fmaf(dyf[2], xh[2], ag0.z); ag0.w = fmaf(dyf[3], xh[3], ag0.w);
                ag1.x = fmaf(dyf[4], xh[4], ag1.x); ag1.y = fmaf(dyf[5], xh[5], ag1.y);
                ag1.z = fmaf(dyf[6], xh[6], ag1.z); ag1.w = fmaf(dyf[7], xh[7], ag1.w);
                ab0.x += dyf[0]; ab0.y += dyf[1]; ab0.z += dyf[2]; ab0.w += dyf[3];
                ab1.x += dyf[4]; ab1.y += dyf[5]; ab1.z += dyf[6]; ab1.w += dyf[7];
                ag[0] = ag0; ag[1] = ag1; ab[0] = ab0; ab[1] = ab1;
            }
        }
        const float m1 = block_sum<NT>(s1, red) * inv_h;
        const float m2 = block_sum<NT>(s2, red) * inv_h;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = threadIdx.x + NT * k;
            if (8 * v < H) {
                float dyf[8], zf[8], dz[8];
                bf16x8_to_f32(dyv[k], dyf);
                bf16x8_to_f32(zv[k], zf);
                const float4 g0 = *reinterpret_cast<const float4*>(a.gamma + 8 * v);
                const float4 g1 = *reinterpret_cast<const float4*>(a.gamma + 8 * v + 4);
                const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                float nf[8];
                bf16x8_to_f32(nv4[k], nf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float xh = (zf[e] - mean) * rstd;
                    dz[e] = fmaf(rstd, dyf[e] * g[e] - m1 - xh * m2, nf[e]);
                }
                *reinterpret_cast<uint4*>(a.d_residual + base + 8 * v) = f32_to_bf16x8(dz);
                const uint32_t keep = DROP ? dal_keep8(a, (uint32_t)v, (uint32_t)row) : 0xFFu;
                float dxf[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) dxf[e] = ((keep >> e) & 1u) ? dz[e] * a.keep_scale : 0.f;
                *reinterpret_cast<uint4*>(a.dx + base + 8 * v) = f32_to_bf16x8(dxf);
            }
        }
    }
    float4* pg = reinterpret_cast<float4*>(a.partial + (size_t)blockIdx.x * H);
    float4* pb = reinterpret_cast<float4*>(a.partial + (size_t)gridDim.x * H + (size_t)blockIdx.x * H);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int v = threadIdx.x + NT * k;
        if (8 * v < H) {
            pg[2 * v] = reinterpret_cast<const float4*>(acc_g)[2 * v];
            pg[2 * v + 1] = reinterpret_cast<const float4*>(acc_g)[2 * v + 1];
            pb[2 * v] = reinterpret_cast<const float4*>(acc_b)[2 * v];
            pb[2 * v + 1] = reinterpret_cast<const float4*>(acc_b)[2 * v + 1];
        }
    }
}

// dgamma and dbeta: column sums of the partial rows, in a fixed order
// (bit-reproducible).  A CTA of 256 threads owns 32 columns: warp w sums the
// partial rows w, w + 8, ... (lane = column; coalesced 128-byte loads), then
// the eight warp sums are added in warp order.
__global__ void __launch_bounds__(256)
dal_reduce_kernel(const DalArgs a, int n_part)
{
    __shared__ float sg[8][32], sb[8][32];
    const int H = a.hidden;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    float g = 0.f, b = 0.f;
    if (c < H) {
#pragma unroll 4
        for (int p = w; p < n_part; p += 8) {
            g += a.partial[(size_t)p * H + c];
            b += a.partial[(size_t)(n_part + p) * H + c];
        }
    }
    sg[w][lane] = g;
    sb[w][lane] = b;
    __syncthreads();
    if (w == 0 && c < H) {
        float tg = 0.f, tb = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            tg += sg[k][lane];
            tb += sb[k][lane];
        }
        a.dgamma[c] = tg;
        a.dbeta[c] = tb;
    }
}

namespace {

// Grids: as many CTAs as are resident at once (rows are grid-strided), so no
// CTA waits for another to finish before it starts.
template <typename K>
int resident_grid(K kern, int threads, int smem, int sms, int cap, int* grid)
{
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess) return (int)e;
    const int g = (per_sm > 0 ? per_sm : 1) * sms;
    *grid = g < cap ? g : cap;
    return 0;
}

template <int NV>
int launch_fwd_nv(bool drop, const DalArgs& a, int sms, cudaStream_t st)
{
    const int smem = 8 * a.hidden;     // two stages of an x row and a residual row (bf16)
    auto kern = drop ? dal_fwd_kernel<NV, true> : dal_fwd_kernel<NV, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    int grid = 0;
    if (int rc = resident_grid(kern, kFwdThreads, smem, sms, a.n_rows, &grid)) return rc;
    kern<<<grid, kFwdThreads, smem, st>>>(a);
    return (int)cudaGetLastError();
}

template <int NV, int NT>
int launch_bwd_nv(bool drop, const DalArgs& a, int sms, cudaStream_t st)
{
    const int smem = 8 * a.hidden;     // [2][hidden] fp32 column sums
    auto kern = drop ? dal_bwd_kernel<NV, true, NT> : dal_bwd_kernel<NV, false, NT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    const int cap = a.n_rows < kDalMaxPartial ? a.n_rows : kDalMaxPartial;
    int grid = 0;
    if (int rc = resident_grid(kern, NT, smem, sms, cap, &grid)) return rc;
    kern<<<grid, NT, smem, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return (int)cudaErrorLaunchFailure;
    dal_reduce_kernel<<<(a.hidden + 31) / 32, 256, 0, st>>>(a, grid);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_dal_fwd(const DalArgs& a, int sms, cudaStream_t st)
{
    const int nv = (a.hidden + 8 * kFwdThreads - 1) / (8 * kFwdThreads);
    const bool drop = a.thr != 0;
    if (nv <= 1) return launch_fwd_nv<1>(drop, a, sms, st);
    if (nv <= 2) return launch_fwd_nv<2>(drop, a, sms, st);
    if (nv <= 3) return launch_fwd_nv<3>(drop, a, sms, st);
    if (nv <= 4) return launch_fwd_nv<4>(drop, a, sms, st);
    if (nv <= 6) return launch_fwd_nv<6>(drop, a, sms, st);
    if (nv <= 8) return launch_fwd_nv<8>(drop, a, sms, st);
    if (nv <= 10) return launch_fwd_nv<10>(drop, a, sms, st);
    if (nv <= 12) return launch_fwd_nv<12>(drop, a, sms, st);
    if (nv <= 14) return launch_fwd_nv<14>(drop, a, sms, st);
    return (int)cudaErrorInvalidValue;
}

int launch_dal_bwd(const DalArgs& a, int sms, cudaStream_t st)
{
    const bool drop = a.thr != 0;
    if (a.hidden <= 8 * 256 * 4) {       // 256 threads, two or more CTAs per SM
        const int nv = (a.hidden + 8 * 256 - 1) / (8 * 256);
        if (nv <= 1) return launch_bwd_nv<1, 256>(drop, a, sms, st);
        if (nv <= 2) return launch_bwd_nv<2, 256>(drop, a, sms, st);
        if (nv <= 3) return launch_bwd_nv<3, 256>(drop, a, sms, st);
        return launch_bwd_nv<4, 256>(drop, a, sms, st);
    }
    // 512 threads, one CTA per SM: half the partial-sum rows of two 256-thread CTAs
    const int nv = (a.hidden + 8 * 512 - 1) / (8 * 512);
    if (nv <= 3) return launch_bwd_nv<3, 512>(drop, a, sms, st);
    if (nv <= 4) return launch_bwd_nv<4, 512>(drop, a, sms, st);
    if (nv <= 5) return launch_bwd_nv<5, 512>(drop, a, sms, st);
    if (nv <= 6) return launch_bwd_nv<6, 512>(drop, a, sms, st);
    if (nv <= 7) return launch_bwd_nv<7, 512>(drop, a, sms, st);
    return (int)cudaErrorInvalidValue;
}

}  // namespace ac
