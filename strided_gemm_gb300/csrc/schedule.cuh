// Work list of a persistent CTA, shared by the FFMA and TF32 kernels.
//
// Tiles [0, dp_tiles) are computed whole, tile t by CTA t % grid.  The K
// slices of the remaining tiles (sk_units = tiles x slices) are split evenly
// across the grid in contiguous ranges: a CTA's range starts inside one tile
// (its tail: the last slices of that tile) and ends inside another (its head:
// the first slices), or lies strictly inside one tile (a middle piece).  Heads
// and middle pieces leave their partial sums in the workspace slot of their
// CTA, one slot per CTA.  Two ways of finishing a split tile:
//  - chained (stream-K over the last waves, every range at least one tile
//    long, so a tile has one head and one tail): the tail continues the head's
//    k-ordered accumulation from its partial sums, so results are
//    bit-identical to the data-parallel schedule;
//  - independent pieces (fewer tiles than CTAs, long K): every piece starts
//    from zero and runs at the same time as the others; the tail adds the
//    earlier pieces' partial sums in a fixed order (latest CTA first), so
//    results are deterministic from run to run but rounded differently from
//    the unsplit schedule.
#pragma once

#include <cstdint>

namespace sbg {

// One unit of a CTA's work: slices [kb, ke) of one tile.  A HEAD item (a head
// or a middle piece) leaves its partial sums in the workspace; a TAIL item
// finishes the tile from the earlier pieces' partial sums.
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
    int head_begin, head_end;     // head: slices [head_begin, head_end)
    int tail_begin;               // tail: slices [tail_begin, nk)
    int has_head, has_tail;
    int64_t cta, nctas;           // this worker and the number of workers (CTAs, or CTA pairs)

    __device__ __forceinline__ void init(int64_t dp_tiles, int64_t sk_units, int nk) {
        init(dp_tiles, sk_units, nk, blockIdx.x, gridDim.x);
    }

    __device__ __forceinline__ void init(int64_t dp_tiles, int64_t sk_units, int nk, int64_t c, int64_t G) {
        set(dp_tiles, sk_units, nk, c, G, c * sk_units / G, (c + 1) * sk_units / G);
    }

    // The split by cost instead of by unit: the first sk_full units cost wf
    // each and the rest wr (tiles whose later units are cheaper, ordered
    // last), so every CTA gets the same cost.  Each range must still span at
    // least one tile's units (the caller checks total cost >= G nk wf).
    __device__ __forceinline__ void init_weighted(int64_t dp_tiles, int64_t sk_units, int nk, int64_t sk_full,
                                                  int wf, int wr) {
        const int64_t c = blockIdx.x, G = gridDim.x;
        const int64_t total = unit_cost(sk_units, sk_full, wf, wr);
        set(dp_tiles, sk_units, nk, c, G, unit_at_cost(c * total / G, sk_full, wf, wr),
            unit_at_cost((c + 1) * total / G, sk_full, wf, wr));
    }

    // Cost of the units before unit x, and the first unit whose cost starts at
    // or after `cost`.
    __device__ __forceinline__ static int64_t unit_cost(int64_t x, int64_t sk_full, int wf, int wr) {
        return x <= sk_full ? x * wf : sk_full * wf + (x - sk_full) * wr;
    }
    __device__ __forceinline__ static int64_t unit_at_cost(int64_t cost, int64_t sk_full, int wf, int wr) {
        const int64_t cf = sk_full * wf;
        return cost <= cf ? (cost + wf - 1) / wf : sk_full + (cost - cf + wr - 1) / wr;
    }

    __device__ __forceinline__ void set(int64_t dp_tiles, int64_t sk_units, int nk, int64_t c, int64_t G,
                                        int64_t u0, int64_t u1) {
        cta = c;
        nctas = G;
        n_dp = dp_tiles > c ? (dp_tiles - 1 - c) / G + 1 : 0;
        has_head = has_tail = 0;
        n_full = 0;
        full_first = head_tile = tail_tile = 0;
        head_begin = head_end = tail_begin = 0;
        if (sk_units > 0) {
            const int64_t t0 = u0 / nk, t1 = (u1 - 1) / nk;
            const int s0 = (int)(u0 % nk), e1 = (int)((u1 - 1) % nk);
            has_tail = s0 > 0;
            has_head = e1 < nk - 1;
            if (t0 == t1 && has_tail && has_head) {   // strictly inside one tile
                has_tail = 0;
                head_begin = s0;
            }
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
        if (w < n_dp) return {cta + w * nctas, 0, nk, kFull};
        w -= n_dp;
        if (has_head) {
            if (w == 0) return {head_tile, head_begin, head_end, kHead};
            --w;
        }
        if (w < n_full) return {full_first + w, 0, nk, kFull};
        return {tail_tile, tail_begin, nk, kTail};
    }

    __device__ __forceinline__ int64_t slices(int nk) const {
        return (n_dp + n_full) * nk + (has_head ? head_end - head_begin : 0) +
               (has_tail ? nk - tail_begin : 0);
    }
};

// The CTA whose range holds unit x: the largest c with floor(c * units / grid) <= x.
__host__ __device__ __forceinline__ int64_t unit_owner(int64_t x, int64_t units, int64_t grid) {
    return ((x + 1) * grid - 1) / units;
}

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

// Independent pieces for problems with fewer tiles than CTAs: all of the
// tiles' K slices spread over up to `grid` CTAs of at least `min_slices`
// slices each.  Chosen when the estimated time (one CTA's share, plus
// `overhead_slices` and one slice per extra piece of a tile for the
// reduction) is at most 97% of one whole tile.  Returns the CTA count, or -1.
inline int64_t split_k_ctas(int64_t tiles, int64_t nk, int64_t grid, int64_t min_slices,
                            int64_t overhead_slices) {
    if (tiles <= 0 || tiles >= grid || nk < 2 * min_slices) return -1;
    const int64_t units = tiles * nk;
    int64_t g = units / min_slices;
    if (g > grid) g = grid;
    if (g <= tiles) return -1;
    const int64_t share = (units + g - 1) / g;
    const int64_t pieces = (nk + share - 1) / share + 1;   // most pieces one tile can have
    const double t_split = (double)share + (double)overhead_slices + (double)(pieces - 1);
    return t_split > 0.97 * (double)nk ? -1 : g;
}

}  // namespace sbg
