// philox.cuh -- counter-based dropout mask for the softmax dropout of the
// attention core ("Reducing Activation Recomputation in Large Transformer
// Models", Key takeaways: the core is QK^T, softmax, softmax dropout,
// attention over V; the backward pass recomputes it, so forward and
// recompute must draw the identical mask).
//
// Generator: Philox-4x32-10 as defined by Salmon, Moraes, Dror and Shaw,
// "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), section 3.2.
// Mask reading (the pages fix none; the public header states it too):
//   counter = (key / 8, query, flattened query head, offset), key = seed;
//   one call yields eight 16-bit draws for keys 8*(key/8) .. +7, key e of the
//   group taking the low (e even) or high (e odd) half of word e / 2;
//   an element is dropped iff its draw < thr = round(p * 65536).
#pragma once
#include <stdint.h>

#include "ptx.cuh"

namespace ac {

struct PhiloxKey {
    uint32_t k0, k1;      // seed low / high word
    uint32_t bh;          // flattened query head (counter word 2)
    uint32_t offset;      // counter word 3
    uint32_t thr;         // drop iff draw < thr
};

__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint64_t pa = (uint64_t)0xD2511F53u * c0;   // one wide multiply: both halves
        const uint64_t pb = (uint64_t)0xCD9E8D57u * c2;
        c0 = (uint32_t)(pb >> 32) ^ c1 ^ k0;
        c1 = (uint32_t)pb;
        c2 = (uint32_t)(pa >> 32) ^ c3 ^ k1;
        c3 = (uint32_t)pa;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return make_uint4(c0, c1, c2, c3);
}

// Keep mask of the two keys a Philox output word decides (low half: the even
// key, high half: the odd key), as 16-bit lane masks: 0xffff where the draw
// is >= thr (kept), 0 where dropped.  t16 = thr << 16.  A high half is >= thr
// exactly when the whole word is >= thr << 16; a low half when the word
// shifted left by 16 is.
__device__ __forceinline__ uint32_t keep_mask16x2(uint32_t w, uint32_t t16)
{
    return (w >= t16 ? 0xffff0000u : 0u) | ((w << 16) >= t16 ? 0x0000ffffu : 0u);
}

// Dropout factors of the two keys a Philox output word decides: z = zs where
// the draw is >= thr (kept), 0 where dropped, packed (even key, odd key).
// t16 = thr << 16 (see keep_mask16x2).
__device__ __forceinline__ uint64_t keep_factor2(uint32_t w, uint32_t t16, float zs)
{
    return f2_pack((w << 16) >= t16 ? zs : 0.f, w >= t16 ? zs : 0.f);
}

// Keep bits of the eight keys 8*group .. 8*group+7 of one query row:
// bit e is 1 iff key 8*group + e survives.
__device__ __forceinline__ uint32_t keep_byte(const PhiloxKey& pk, uint32_t group, uint32_t query)
{
    const uint4 w = philox4x32_10(group, query, pk.bh, pk.offset, pk.k0, pk.k1);
    const uint32_t t = pk.thr;
    uint32_t b = 0;
    b |= (uint32_t)((w.x & 0xFFFFu) >= t) << 0;
    b |= (uint32_t)((w.x >> 16) >= t) << 1;
    b |= (uint32_t)((w.y & 0xFFFFu) >= t) << 2;
    b |= (uint32_t)((w.y >> 16) >= t) << 3;
    b |= (uint32_t)((w.z & 0xFFFFu) >= t) << 4;
    b |= (uint32_t)((w.z >> 16) >= t) << 5;
    b |= (uint32_t)((w.w & 0xFFFFu) >= t) << 6;
    b |= (uint32_t)((w.w >> 16) >= t) << 7;
    return b;
}

// Keep bits of 32 consecutive keys [32*blk32, 32*blk32 + 32) of one query
// row (lanes are queries): bit c is key 32*blk32 + c.
__device__ __forceinline__ uint32_t keep_word_row(const PhiloxKey& pk, uint32_t blk32, uint32_t query)
{
    uint32_t m = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) m |= keep_byte(pk, blk32 * 4 + g, query) << (8 * g);
    return m;
}

// Transposed orientation (lanes are keys).  The calling warp holds 32
// consecutive keys starting at a multiple of 8 (lane L is key key0 + L).
// Returns, for this lane's key, the keep bits of the 32 queries
// [q0, q0 + 32): bit c is query q0 + c.  Each lane of an 8-lane group draws
// the groups of four of the queries and the eight lanes swap bytes.
__device__ __forceinline__ uint32_t keep_word_col(const PhiloxKey& pk, uint32_t key0, uint32_t q0)
{
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t t = lane & 7;                   // this lane's key within its group of 8
    const uint32_t group = (key0 + lane) >> 3;     // same for the 8 lanes
    // byte u of w: keep bits (over the 8 keys) of query q0 + 8u + t
    uint32_t w = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) w |= keep_byte(pk, group, q0 + 8 * u + t) << (8 * u);
    uint32_t m = 0;
#pragma unroll
    for (int src = 0; src < 8; ++src) {
        const uint32_t x = __shfl_sync(0xffffffffu, w, (lane & ~7u) | (uint32_t)src);
        // bit 8u + t of x is query q0 + 8u + src for this lane's key
        m |= ((x >> t) & 0x01010101u) << src;
    }
    return m;
}

}  // namespace ac
