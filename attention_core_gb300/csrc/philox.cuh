// philox.cuh -- counter-based dropout mask for the softmax dropout of the
// attention core ("Reducing Activation Recomputation in Large Transformer
// Models", Key takeaways: the core is QK^T, softmax, softmax dropout,
// attention over V; the backward pass recomputes it, so forward and
// recompute must draw the identical mask).
//
// Generator: Philox-4x32-10 as defined by Salmon, Moraes, Dror and Shaw,
// "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), section 3.2.
// Mask reading of the attention core (the pages fix none; the public header
// states it too):
//   counter = (key / 16, query, flattened query head, offset), key = seed;
//   one call yields sixteen 8-bit draws for keys 16*(key/16) .. +15, key e of
//   the group taking byte e % 4 (bits 8(e%4) .. 8(e%4)+7) of word e / 4;
//   an element is dropped iff its draw < thr = round(p * 256) (at most 255).
// (The dropout + layer norm block beside the core reads 16-bit draws; its
// own file states that reading.)
#pragma once
#include <stdint.h>

#include "ptx.cuh"

namespace ac {

struct PhiloxKey {
    const uint32_t* rk;   // the key schedule (philox_round_keys)
    uint32_t bh;          // flattened query head (counter word 2)
    uint32_t offset;      // counter word 3
};

// The key schedule of Philox-4x32-10: round r (0..9) uses the key words
// rk[2r] = k0 + r * 0x9E3779B9 and rk[2r+1] = k1 + r * 0xBB67AE85 (the Weyl
// sequence of the SC'11 paper).  The schedule depends on the seed only, so the
// host computes it once per call and the kernels read it from their
// parameters.
__host__ __device__ inline void philox_round_keys(uint32_t k0, uint32_t k1, uint32_t (&rk)[20])
{
    for (int r = 0; r < 10; ++r) {
        rk[2 * r] = k0 + (uint32_t)r * 0x9E3779B9u;
        rk[2 * r + 1] = k1 + (uint32_t)r * 0xBB67AE85u;
    }
}

// Philox-4x32-10 of one counter under a precomputed key schedule.
__device__ __forceinline__ uint4 philox4x32_10_rk(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                  const uint32_t* rk)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint64_t pa = (uint64_t)0xD2511F53u * c0;   // one wide multiply: both halves
        const uint64_t pb = (uint64_t)0xCD9E8D57u * c2;
        c0 = (uint32_t)(pb >> 32) ^ c1 ^ rk[2 * round];
        c1 = (uint32_t)pb;
        c2 = (uint32_t)(pa >> 32) ^ c3 ^ rk[2 * round + 1];
        c3 = (uint32_t)pa;
    }
    return make_uint4(c0, c1, c2, c3);
}

// Byte permute (PRMT): result byte i is byte sel_i & 7 of {b, a} (a holds
// bytes 0-3), or that byte's sign bit replicated when sel_i & 8.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// The four 8-bit draws of a Philox output word against thr at once (SWAR):
// returns a word whose byte b has its sign bit set iff draw b >= thr.  With x
// the draw's low 7 bits, adding k = 0x80 - thr (thr <= 0x80) to x sets the
// byte's top bit exactly when x >= thr, and a draw with its own top bit set is
// kept as well (OR); for thr > 0x80, k = 0x100 - thr and the draw's top bit is
// required (AND).  No byte can carry into the next.  kk = k in every byte; f =
// all ones for the OR case, 0 for the AND case (a bitwise majority picks).
struct KeepSwar8 {
    uint32_t kk, f;
    __device__ __forceinline__ explicit KeepSwar8(uint32_t thr)
    {
        const uint32_t k = thr <= 0x80u ? 0x80u - thr : 0x100u - thr;
        kk = k * 0x01010101u;
        f = thr <= 0x80u ? 0xFFFFFFFFu : 0u;
    }
    __device__ __forceinline__ uint32_t operator()(uint32_t w) const
    {
        const uint32_t d = (w & 0x7F7F7F7Fu) + kk;
        return (d & w) | (f & (d | w));
    }
};

// From a keep word (byte sign bits, keys 4t .. 4t+3): the 16-bit lane mask of
// the bf16 pair of keys (4t, 4t+1) (q = 0) or (4t+2, 4t+3) (q = 1): low half
// 0xffff iff the even key is kept, high half iff the odd one is.
__device__ __forceinline__ uint32_t keep_pair16(uint32_t r, int q)
{
    return prmt(r, 0u, q ? 0xBBAAu : 0x9988u);
}
// The 32-bit mask (all ones iff kept) of key 4t + b of a keep word.
__device__ __forceinline__ uint32_t keep_mask32(uint32_t r, int b)
{
    return prmt(r, 0u, 0x8888u | (0x1111u * (uint32_t)b));
}

// Keep bits of 32 consecutive keys (eight keep words, keys 4k .. 4k+3 in word
// k) as one word: key 4k + b at bit 8b + 7 - k.  This is the layout the dQ
// kernel hands to the dK/dV kernel; keep_bit_position gives the bit of a key.
__device__ __forceinline__ uint32_t keep_bits32(const uint32_t (&r)[8])
{
    uint32_t bits = r[0] & 0x80808080u;
#pragma unroll
    for (int k = 1; k < 8; ++k) bits |= (r[k] >> k) & (0x80808080u >> k);
    return bits;
}
__host__ __device__ constexpr uint32_t keep_bit_position(uint32_t key32)
{
    return 8u * (key32 & 3u) + 7u - (key32 >> 2);
}

// Transposed orientation (lanes are keys).  The calling warp holds 32
// consecutive keys starting at a multiple of 16: lanes 0-15 the first group of
// 16, lanes 16-31 the second (lane L is key 16*group + t, t = L & 15).  The
// half-tile covers the HQ queries [q0, q0 + HQ).
//
// Lane t draws the Philox calls (group, q0 + 16u + t) for u = 0 .. HQ/16 - 1;
// each call decides the group's 16 keys for one query.  The keep decisions
// become byte sign bits (four words: keys 0-3, 4-7, 8-11, 12-15), and a
// 16-lane butterfly (four stages of two shuffles) transposes each 16 x 16 byte
// block, so that afterwards, for this lane's key, byte i of the four words
// kw[u][0..3] (byte i % 4 of word i / 4) has its sign bit set iff query
// q0 + 16u + i is kept.
template <int HQ>
__device__ __forceinline__ void keep_bytes_col16(const PhiloxKey& pk, const KeepSwar8& ks, uint32_t group,
                                                 uint32_t q0, uint32_t (&kw)[HQ / 16][4])
{
    static_assert(HQ % 16 == 0, "query half-tile must be a multiple of 16");
    const uint32_t t = threadIdx.x & 15;
    const bool b8 = t & 8, b4 = t & 4, b2 = t & 2, b1 = t & 1;
    // all Philox calls first (independent chains the scheduler can interleave)
    uint4 w[HQ / 16];
#pragma unroll
    for (int u = 0; u < HQ / 16; ++u) w[u] = philox4x32_10_rk(group, q0 + 16u * (uint32_t)u + t, pk.bh, pk.offset, pk.rk);
#pragma unroll
    for (int u = 0; u < HQ / 16; ++u) {
        uint32_t W[4] = {ks(w[u].x), ks(w[u].y), ks(w[u].z), ks(w[u].w)};
        // bit 3: the off-diagonal 8 x 8 blocks (keys 8-15 of low lanes <-> keys 0-7 of high lanes)
        {
            const uint32_t s0 = __shfl_xor_sync(0xffffffffu, b8 ? W[0] : W[2], 8);
            const uint32_t s1 = __shfl_xor_sync(0xffffffffu, b8 ? W[1] : W[3], 8);
            if (b8) { W[0] = s0; W[1] = s1; } else { W[2] = s0; W[3] = s1; }
        }
        // bit 2: the off-diagonal 4 x 4 blocks within each 8 x 8 block (whole words)
        {
            const uint32_t s0 = __shfl_xor_sync(0xffffffffu, b4 ? W[0] : W[1], 4);
            const uint32_t s1 = __shfl_xor_sync(0xffffffffu, b4 ? W[2] : W[3], 4);
            if (b4) { W[0] = s0; W[2] = s1; } else { W[1] = s0; W[3] = s1; }
        }
        // bit 1: 16-bit halves of each word (keys 4k+2, 4k+3 of low lanes <-> 4k, 4k+1 of high lanes)
        {
            const uint32_t sel = b2 ? 0x5410u : 0x7632u;          // the halves this lane gives away
            const uint32_t s0 = __shfl_xor_sync(0xffffffffu, prmt(W[0], W[1], sel), 2);
            const uint32_t s1 = __shfl_xor_sync(0xffffffffu, prmt(W[2], W[3], sel), 2);
            // low lanes keep their low halves and take the partner's low halves as
            // their high halves; high lanes the other way round
            W[0] = prmt(W[0], s0, b2 ? 0x3254u : 0x5410u);
            W[1] = prmt(W[1], s0, b2 ? 0x3276u : 0x7610u);
            W[2] = prmt(W[2], s1, b2 ? 0x3254u : 0x5410u);
            W[3] = prmt(W[3], s1, b2 ? 0x3276u : 0x7610u);
        }
        // bit 0: bytes (keys 4k+1, 4k+3 of low lanes <-> 4k, 4k+2 of high lanes)
        {
            const uint32_t sel = b1 ? 0x6420u : 0x7531u;          // the bytes this lane gives away
            const uint32_t s0 = __shfl_xor_sync(0xffffffffu, prmt(W[0], W[1], sel), 1);
            const uint32_t s1 = __shfl_xor_sync(0xffffffffu, prmt(W[2], W[3], sel), 1);
            W[0] = prmt(W[0], s0, b1 ? 0x3514u : 0x5240u);
            W[1] = prmt(W[1], s0, b1 ? 0x3716u : 0x7260u);
            W[2] = prmt(W[2], s1, b1 ? 0x3514u : 0x5240u);
            W[3] = prmt(W[3], s1, b1 ? 0x3716u : 0x7260u);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) kw[u][k] = W[k];
    }
}

// Keep bits of four consecutive queries (bit t = query t) as the sign bits of
// four bytes (bit t -> bit 8t + 7).  Multiplying by 2^7 + 2^14 + 2^21 + 2^28
// moves bit t up by 7t + 7; a cross term t + 7u + 7 (u != t) never lands on a
// position 8k + 7 and no two terms share a position, so nothing carries.
__device__ __forceinline__ uint32_t keep_nibble_bytes(uint32_t nibble)
{
    return (nibble * 0x10204080u) & 0x80808080u;
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
