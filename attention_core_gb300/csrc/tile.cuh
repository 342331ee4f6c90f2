// tile.cuh -- shared-memory tile geometry common to the kernels.
//
// A [rows x D] bf16 tile (rows are queries or keys, D the head dimension) is
// stored as D / CW column chunks, each chunk [rows x CW] with one row per CW*2
// bytes, written by TMA with the matching hardware swizzle: CW = 64 (128-byte
// rows, 128-byte swizzle) when D is a multiple of 64, else CW = 32 (64-byte
// rows, 64-byte swizzle).  The same bytes serve as a K-major operand (the
// head dimension is the reduction: Q.K^T, dO.V^T) and as an MN-major operand
// (the rows are the reduction: P.V, dS.K, P^T.dO, dS^T.Q).
#pragma once
#include <stdint.h>

#include "ptx.cuh"

namespace ac {

template <int D>
struct TileGeom {
    static_assert(D % 32 == 0 && D >= 32 && D <= 256, "head dimension must be a multiple of 32 in [32, 256]");
    static constexpr int CW = (D % 64 == 0) ? 64 : 32;
    static constexpr int NCH = D / CW;
    static constexpr uint32_t ROWB = CW * 2;                   // bytes per row of a chunk
    static constexpr uint32_t LAYOUT = (CW == 64) ? 2u : 4u;   // descriptor swizzle code
    static constexpr uint32_t SBO = 8 * ROWB;                  // stride of 8-row groups
    static constexpr CUtensorMapSwizzle TMA_SWIZZLE =
        (CW == 64) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    template <int ROWS>
    __host__ __device__ static constexpr uint32_t tile_bytes() { return (uint32_t)ROWS * D * 2; }
    template <int ROWS>
    __host__ __device__ static constexpr uint32_t chunk_bytes() { return (uint32_t)ROWS * ROWB; }

    // The descriptors of a tile's slices differ only in their start-address
    // field (address >> 4 in bits 0-13).  Tile bases and slice offsets are
    // multiples of 16 and every shared-memory address is below 256 KB, so the
    // descriptor of slice kk is that of slice 0 plus offset(kk) >> 4 in the low
    // word, with no carry out of the field: one 32-bit add per slice on the
    // MMA-issuing thread instead of rebuilding the descriptor.
    template <int ROWS>
    __host__ __device__ static constexpr uint32_t k_offset(int kk)
    {
        return (uint32_t)((kk * 16) / CW) * chunk_bytes<ROWS>() + (uint32_t)((kk * 16) % CW) * 2;
    }
    // K-major operand: the 16-wide slice kk of the head dimension.
    template <int ROWS>
    __device__ static __forceinline__ uint64_t desc_k(uint32_t base, int kk)
    {
        return desc_plus(smem_desc(base, 16, SBO, LAYOUT), k_offset<ROWS>(kk) >> 4);
    }
    // MN-major operand: rows [16 kk, 16 kk + 16) as the reduction slice,
    // the head dimension (D wide, chunk after chunk) as N.
    template <int ROWS>
    __device__ static __forceinline__ uint64_t desc_mn(uint32_t base, int kk)
    {
        return desc_plus(smem_desc(base, chunk_bytes<ROWS>(), SBO, LAYOUT), ((uint32_t)kk * 16 * ROWB) >> 4);
    }
    // Byte offset of the 16-byte unit holding columns [col, col + 8) of row r.
    template <int ROWS>
    __device__ static __forceinline__ uint32_t unit_offset(int r, int col)
    {
        const uint32_t unit = (uint32_t)(col % CW) / 8;
        const uint32_t sw = (CW == 64) ? (uint32_t)(r & 7) : (uint32_t)((r >> 1) & 3);
        return (uint32_t)(col / CW) * chunk_bytes<ROWS>() + (uint32_t)r * ROWB + ((unit ^ sw) << 4);
    }
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

// Scale 32 fp32 accumulator columns [c0, c0 + 32) of row r, round to bf16
// and write them into a staged [ROWS x D] output tile (TMA-store layout).
template <int D, int ROWS>
__device__ __forceinline__ void stage_row32(uint32_t tile_base, int r, int c0, const uint32_t (&acc)[32],
                                            float mul)
{
    using G = TileGeom<D>;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(acc[8 * u + 2 * e]) * mul;
            const float hi = __uint_as_float(acc[8 * u + 2 * e + 1]) * mul;
            w[e] = pack_bf16x2(lo, hi);
        }
        st_shared_v4(tile_base + G::template unit_offset<ROWS>(r, c0 + 8 * u), w[0], w[1], w[2], w[3]);
    }
}

}  // namespace ac
