// sched.cuh -- static work split of the persistent kernels.
//
// The kernels launch one CTA per SM and walk a list of work tiles sorted
// longest first (under a causal mask a tile's work grows with its block
// index).  CTA c takes the tiles of positions c, 2G-1-c, 2G+c, 4G-1-c, ...
// (G CTAs): a serpentine deal that pairs the long tiles of one round with the
// short tiles of the next, so the per-CTA sums stay close to the mean.
#pragma once
#include <stdint.h>

#include "kernels.h"

namespace ac {

struct TileSched {
    int n_tiles, grid, cta;

    // Index of this CTA's u-th tile, or -1 when it has no more.
    __device__ __forceinline__ int tile(int u) const
    {
        const int pos = (u & 1) ? (grid - 1 - cta) : cta;
        const int64_t t = (int64_t)u * grid + pos;
        return t < n_tiles ? (int)t : -1;
    }
};

// The next tile with work of this CTA's list for the query-major kernels,
// scanning from position v (advanced past it): false when none is left.  A
// packed batch's list holds tiles past the end of short sequences, which every
// role of the kernel skips the same way.
template <bool PACKED>
__device__ __forceinline__ bool next_qtile(const TileSched& sched, const CommonArgs& a, int bn, int& v, QTile& w)
{
    for (;; ++v) {
        const int t = sched.tile(v);
        if (t < 0) return false;
        w = q_tile<PACKED>(a, t, bn);
        if (!w.empty) {
            ++v;
            return true;
        }
    }
}

}  // namespace ac
