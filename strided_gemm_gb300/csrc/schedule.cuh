// Work list of a persistent CTA, shared by the FFMA and TF32 kernels.
//
// Tiles [0, dp_tiles) are computed whole, tile t by CTA t % grid.  The K
// slices of the remaining tiles (sk_units = tiles x slices) are split evenly
// across the grid (stream-K): a CTA's share starts inside one tile (its tail:
// the last slices of that tile) and ends inside another (its head: the first
// slices).  A head's partial sums go to the workspace; the CTA owning the same
// tile's tail continues the same k-ordered accumulation from them, so results
// are bit-identical to the data-parallel schedule.
#pragma once

#include <cstdint>

namespace sbg {

// One unit of a CTA's work: slices [kb, ke) of one tile.  A HEAD item leaves
// its partial sums in the workspace for the next CTA; a TAIL item starts from
// the previous CTA's partial sums and finishes the tile.
enum : int { kFull = 0, kHead = 1, kTail = 2 };
struct Item { int64_t tile; int kb, ke, mode; };

// The CTA's ordered work list: its data-parallel tiles, then (stream-K) the
// head of the tile its K range ends in, the whole tiles inside the range, and
// last the tail of the tile its range starts in.  The head is produced first
// and the tail consumed last, so a tail's partial is normally long ready.
struct Schedule {
    int64_t n_dp, n_items;
    int64_t full_first, n_full;   // stream-K whole tiles
    int64_t head_tile, tail_tile;
    int head_end, tail_begin;     // head: slices [0, head_end); tail: [tail_begin, nk)
    int has_head, has_tail;

    __device__ __forceinline__ void init(int64_t dp_tiles, int64_t sk_units, int nk) {
        const int64_t c = blockIdx.x, G = gridDim.x;
        n_dp = dp_tiles > c ? (dp_tiles - 1 - c) / G + 1 : 0;
        has_head = has_tail = 0;
        n_full = 0;
        full_first = head_tile = tail_tile = 0;
        head_end = tail_begin = 0;
        if (sk_units > 0) {
            const int64_t u0 = c * sk_units / G, u1 = (c + 1) * sk_units / G;
            const int64_t t0 = u0 / nk, t1 = (u1 - 1) / nk;
            const int s0 = (int)(u0 % nk), e1 = (int)((u1 - 1) % nk);
            has_tail = s0 > 0;
            has_head = e1 < nk - 1;
            tail_tile = dp_tiles + t0;
            tail_begin = s0;
            head_tile = dp_tiles + t1;
            head_end = e1 + 1;
            full_first = t0 + has_tail;
            const int64_t last = t1 - has_head;
            n_full = last >= full_first ? last - full_first + 1 : 0;
            full_first += dp_tiles;
        }
        n_items = n_dp + has_head + n_full + has_tail;
    }

    __device__ __forceinline__ Item item(int64_t w, int nk) const {
        if (w < n_dp) return {blockIdx.x + w * (int64_t)gridDim.x, 0, nk, kFull};
        w -= n_dp;
        if (has_head) {
            if (w == 0) return {head_tile, 0, head_end, kHead};
            --w;
        }
        if (w < n_full) return {full_first + w, 0, nk, kFull};
        return {tail_tile, tail_begin, nk, kTail};
    }

    __device__ __forceinline__ int64_t slices(int nk) const {
        return (n_dp + n_full) * nk + (has_head ? head_end : 0) + (has_tail ? nk - tail_begin : 0);
    }
};

// Host-side choice of the split.  All but the last one or two waves stay
// data-parallel; their tiles' K slices are spread over the grid when the
// estimated time, in K slices of one CTA, drops by at least 3% after adding
// `overhead_slices` for the exchange of partial sums and the flag reset.
// Every CTA then covers at least one whole tile's worth of slices, so a tile
// is split at most once (one head, one tail).  Returns the number of
// data-parallel tiles, or -1 to stay fully data-parallel.
inline int64_t stream_k_dp_tiles(int64_t tiles, int64_t nk, int64_t grid, int64_t overhead_slices) {
    if (tiles < grid || nk < 8) return -1;
    const int64_t full_waves = tiles / grid - 1;
    const int64_t dp = full_waves * grid;
    const int64_t rem_units = (tiles - dp) * nk;
    const double t_dp = (double)((tiles + grid - 1) / grid) * nk;
    const double t_sk = (double)full_waves * nk + (double)((rem_units + grid - 1) / grid) +
                        (double)overhead_slices;
    return t_sk > 0.97 * t_dp ? -1 : dp;
}

}  // namespace sbg
