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

// Dropout factors of the two keys a Philox output word decides: z = zs where
// the draw is >= thr (kept), 0 where dropped, packed (even key, odd key).
// t16 = thr << 16: the high half is >= thr exactly when the whole word is
// >= thr << 16, the low half when the word shifted left by 16 is.
__device__ __forceinline__ uint64_t keep_factor2(uint32_t w, uint32_t t16, float zs)
{
    return f2_pack((w << 16) >= t16 ? zs : 0.f, w >= t16 ? zs : 0.f);
}

// Byte permute (PRMT): result byte i is byte sel_i & 7 of {b, a} (a holds
// bytes 0-3), or that byte's sign bit replicated when sel_i & 8.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Both draws of a Philox output word against thr at once (SWAR): returns a
// word whose bit 15 is "low draw kept" and bit 31 "high draw kept".  With
// low15 the draw's low 15 bits, adding k = 0x8000 - thr (thr <= 0x8000) to
// low15 carries into the half's top bit exactly when low15 >= thr, and a draw
// with its own top bit set is kept as well (OR); for thr > 0x8000,
// k = 0x10000 - thr and the draw's top bit is required (AND).  No half can
// carry into the next.  kk = k replicated in both halves; f = all ones for
// the OR case, 0 for the AND case (a bitwise majority picks between them).
__device__ __forceinline__ uint32_t keep_swar(uint32_t w, uint32_t kk, uint32_t f)
{
    const uint32_t d = (w & 0x7FFF7FFFu) + kk;
    return (d & w) | (f & (d | w));
}

struct KeepSwar {
    uint32_t kk, f;
    __device__ __forceinline__ explicit KeepSwar(uint32_t thr)
    {
        const uint32_t k = thr <= 0x8000u ? 0x8000u - thr : 0x10000u - thr;
        kk = k | (k << 16);
        f = thr <= 0x8000u ? 0xFFFFFFFFu : 0u;
    }
};

// Transposed orientation (lanes are keys).  The calling warp holds 32
// consecutive keys starting at a multiple of 8 (lane L is key 8*group + t,
// t = L & 7); the half-tile covers the HQ queries [q0, q0 + HQ).
//
// Lane t draws the Philox calls (group, q0 + 16*(u>>1) + 2t + (u&1)) for
// u = 0 .. HQ/8-1; each call decides the group's 8 keys for one query.  The
// keep decisions become byte sign bits (two words: keys 0-3, 4-7), and an
// 8-lane butterfly of byte permutes (three shuffles) transposes each 8x8
// block, so that afterwards, for this lane's key,
//     byte t of (lo[u], hi[u]) has its sign bit set iff query
//     q0 + 16*(u>>1) + 2t + (u&1) is kept.
// The queries 2e and 2e+1 of a bf16 pair thus sit in bytes t = e & 7 of
// blocks u = 2(e>>3) and u + 1 (see keep_pair_mask).
template <int HQ>
__device__ __forceinline__ void keep_bytes_col(const PhiloxKey& pk, const KeepSwar& ks, uint32_t group, uint32_t q0,
                                               uint32_t (&lo)[HQ / 8], uint32_t (&hi)[HQ / 8])
{
    static_assert(HQ % 16 == 0, "query half-tile must be a multiple of 16");
    const uint32_t t = threadIdx.x & 7;
    const bool b2 = t & 4, b1 = t & 2, b0 = t & 1;
    // stage selectors (swap bytes whose index differs from the lane in bit 1 / bit 0)
    const uint32_t s2_send = b1 ? 0x5410u : 0x7632u, s2_lo = b1 ? 0x3254u : 0x5410u, s2_hi = b1 ? 0x3276u : 0x7610u;
    const uint32_t s1_send = b0 ? 0x6420u : 0x7531u, s1_lo = b0 ? 0x3514u : 0x5240u, s1_hi = b0 ? 0x3716u : 0x7260u;
    // all Philox calls first (independent chains the scheduler can interleave)
    uint4 w[HQ / 8];
#pragma unroll
    for (int u = 0; u < HQ / 8; ++u) {
        const uint32_t q = q0 + 16u * (uint32_t)(u >> 1) + 2u * t + (uint32_t)(u & 1);
        w[u] = philox4x32_10(group, q, pk.bh, pk.offset, pk.k0, pk.k1);
    }
#pragma unroll
    for (int u = 0; u < HQ / 8; ++u) {
        uint32_t l = prmt(keep_swar(w[u].x, ks.kk, ks.f), keep_swar(w[u].y, ks.kk, ks.f), 0x7531u);
        uint32_t h = prmt(keep_swar(w[u].z, ks.kk, ks.f), keep_swar(w[u].w, ks.kk, ks.f), 0x7531u);
        // bit 2: whole words
        uint32_t r = __shfl_xor_sync(0xffffffffu, b2 ? l : h, 4);
        if (b2) l = r; else h = r;
        // bit 1: 16-bit halves
        r = __shfl_xor_sync(0xffffffffu, prmt(l, h, s2_send), 2);
        l = prmt(l, r, s2_lo);
        h = prmt(h, r, s2_hi);
        // bit 0: bytes
        r = __shfl_xor_sync(0xffffffffu, prmt(l, h, s1_send), 1);
        l = prmt(l, r, s1_lo);
        h = prmt(h, r, s1_hi);
        lo[u] = l;
        hi[u] = h;
    }
}

// 16-bit lane mask of the query pair (2e, 2e+1) of the half-tile, for this
// lane's key: low half 0xffff iff query 2e is kept, high half iff 2e+1 is.
template <int HQ>
__device__ __forceinline__ uint32_t keep_pair_mask(const uint32_t (&lo)[HQ / 8], const uint32_t (&hi)[HQ / 8], int e)
{
    const int a = e >> 3, t = e & 7, j = t & 3;
    const uint32_t sel = (uint32_t)((8 | j) | ((8 | j) << 4) | ((12 | j) << 8) | ((12 | j) << 12));
    return t < 4 ? prmt(lo[2 * a], lo[2 * a + 1], sel) : prmt(hi[2 * a], hi[2 * a + 1], sel);
}

// Keep bits of four consecutive queries (bit t = query t) as the sign bits of
// four bytes (bit t -> bit 8t + 7).  Multiplying by 2^7 + 2^14 + 2^21 + 2^28
// moves bit t up by 7t + 7; a cross term t + 7u + 7 (u != t) never lands on a
// position 8k + 7 and no two terms share a position, so nothing carries.
__device__ __forceinline__ uint32_t keep_nibble_bytes(uint32_t nibble)
{
    return (nibble * 0x10204080u) & 0x80808080u;
}

// The 16-bit lane mask of the query pair (2e, 2e+1) from such words (byte t
// of word n: query 4n + t): low half from query 2e's byte, high half from
// query 2e + 1's.
__device__ __forceinline__ uint32_t keep_pair_mask_nat(const uint32_t* kbyte, int e)
{
    return prmt(kbyte[e >> 1], 0u, (e & 1) ? 0xBBAAu : 0x9988u);
}

// 32 x 32 bit transpose across a warp: on entry lane L holds row L (bit k =
// element (L, k)); on return lane L holds column L (bit i = element (i, L)).
// Five exchange stages; at stage j lanes L and L ^ j swap the j-wide blocks
// that lie on the wrong side of the diagonal.
__device__ __forceinline__ uint32_t transpose32(uint32_t x)
{
    const uint32_t lane = threadIdx.x & 31u;
    constexpr uint32_t kMask[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        const uint32_t j = 16u >> s, m = kMask[s];
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
        x = (lane & j) ? (((y >> j) & m) | (x & ~m)) : ((x & m) | ((y << j) & ~m));
    }
    return x;
}

}  // namespace ac
