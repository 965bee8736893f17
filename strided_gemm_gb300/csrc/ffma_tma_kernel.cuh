// TMA-fed FFMA path for operands with a unit stride (K-major or MN-major) whose
// other strides are 16-byte multiples.
//
// Persistent CTAs (one per SM) of eight warps walk their work list: whole
// output tiles, and with a workspace the K ranges of the last waves split
// across CTAs (stream-K).  Each tile's K range is cut into 32-deep slices that
// TMA copies (one box of A, one of B) into a ring of shared-memory stages;
// "full" mbarriers signal a landed stage, "empty" mbarriers (one arrival per
// warp) its release.  Thread 0 doubles as the copy issuer, refilling the stage
// released one slice earlier, across tile boundaries too.
//
// The mainloop always reads both operands MN-major: a K-major slice (stored by
// TMA as 128-byte swizzled rows along K) is first transposed in shared memory
// into an MN-major buffer (two buffers, alternating by slice, synchronised by
// bounded mbarriers).  When both operands are transposed the raw stage is free
// as soon as its slice is, so two raw stages keep two slices in flight.
//
// Each warp computes a 64 x 64 warp tile as 16 x 8 register micro-tiles per
// thread (the register blocking of the StaleyNET "GPU Implementation" page,
// section "The matrix product", grown from 4 x 4).  The size follows from
// shared-memory bandwidth: an SM reads 32 fp32 words per clock from shared
// memory but retires 128 FMA lanes, so a thread needs at least 4 FMAs per word
// it loads; 16 x 8 does 128 per 24.  The FMAs are packed two lanes per
// instruction (FFMA2, fma.rn.f32x2) over pairs of adjacent A rows, with B
// broadcast; the next k's fragments load while this k's FMAs run.  Each output
// keeps one fused multiply-add chain in increasing k, so results are
// bit-identical to a scalar fmaf loop, to the gather path and across layouts.
// The epilogue writes alpha*acc (+ C_old) straight from registers with masks
// on ragged M / N; a fused addend and activation (epilogue.cuh) follow in a
// second pass over the thread's own outputs.  Every wait is bounded: on expiry the thread records a
// status code and returns (the copy issuer first waits, again bounded, for the
// copies it has in flight).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <type_traits>

#include "debug_check.cuh"
#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "schedule.cuh"

namespace sbg {
namespace {

constexpr int BK = 32;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int TM = 16, TN = 8;         // micro-tile per thread (rows of A x columns of B)
constexpr int WTM = 64, WTN = 64;      // warp tile: 4 lane-rows x 16, 8 lane-cols x 8

__device__ unsigned int g_wait_status = 0;

struct Params {
    float* C;
    int64_t rsC, csC, bsC;
    int64_t M, N, K;
    int64_t tiles_m, tiles_n, tiles_total;
    int nk;                 // K slices per tile
    float alpha;
    int accumulate;
    int a_bcast, b_bcast;   // batch stride 0: always batch coordinate 0
    int c_vec4;             // csC == 1 and 16-byte aligned rows: float4 epilogue
    // Schedule: tiles [0, dp_tiles) are computed whole, tile t by CTA t % grid.
    // The K slices of tiles [dp_tiles, tiles_total) are split evenly across
    // the grid (stream-K) when sk_units > 0.
    int64_t dp_tiles;
    int64_t sk_units;       // (tiles_total - dp_tiles) * nk
    int indep;              // split tiles as independent pieces (schedule.cuh)
    // Chained split of a product whose last tile column is at most half
    // full: those tiles run in about 2/3 of a full tile's time (their idle
    // warps are one per scheduler), so they are ordered after every full tile
    // (tile_coord) and the split counts their units at w_rag against w_full
    // (Schedule::init_weighted).  w_full == 0: plain order and split.
    int64_t full_tiles;     // tiles outside the last column
    int64_t sk_full_units;  // split units of full tiles: (full_tiles - dp_tiles) * nk
    int w_full, w_rag;
    EpiParams epi;          // fused epilogue (epilogue.cuh); epi.on == 0: none
    int epi_inline;         // ... a bias per column (or none), no activation or ReLU:
                            // applied in the register epilogue
    float2* ws_partial;     // [grid][kThreads * 64] partial accumulators
    unsigned int* ws_flag;  // [grid] partial-ready flags, zeroed before launch
    ElemSpan sc;            // debug builds: C's valid element offsets
};

// Debug builds: [p, p + n) lies inside C's span (records a violation if not).
__device__ __forceinline__ bool c_ok(const Params& p, const float* x, int n) {
    return dbg_in_span(p.C, x, p.sc, &g_wait_status) && dbg_in_span(p.C, x + (n - 1), p.sc, &g_wait_status);
}

// Copy issuer state (thread 0 only, kept in shared memory so that it costs
// no registers in the consumers' hot loop): the next (item, slice) to load.
struct Issuer {
    int64_t w;          // item of the next slice to load
    int kt;             // slice within that item's tile
    int pad;
    uint64_t issued;    // slices issued so far (global iteration count)
    int64_t total;      // slices this CTA loads in all
    // Item w's slice range and copy coordinates, worked out once per item
    // (the tile's coordinates take 64-bit divisions, which thread 0 would
    // otherwise pay on every slice while its warp is part of the mainloop).
    int64_t cw;         // the item they belong to (-1: none yet)
    int kb, ke;
    int m0, n0, ba, bb;
};

// Shared-memory plan of one tile shape.  TA / TB: the A / B operand is
// K-major and each of its slices is transposed in shared memory into an
// MN-major buffer (two buffers, alternating by slice), so the mainloop always
// reads both operands MN-major: 16-byte loads of 4 adjacent rows of A and 4
// adjacent columns of B per k.  When both are transposed the raw TMA stage is
// free as soon as its slice is transposed, so two raw stages keep two slices
// in flight.
constexpr size_t kSmemBudget = 232448 - 1024 - 512;   // opt-in limit - alignment - barriers

template <int BM, int BN, bool TA = false, bool TB = false>
struct Cfg {
    static constexpr int kWarpsM = BM / WTM, kWarpsN = BN / WTN;
    static_assert(kWarpsM * kWarpsN == kWarps, "8 warps of 64 x 64");
    static constexpr int kABytes = BM * BK * 4, kBBytes = BN * BK * 4;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr bool kRawEarly = TA && TB;
    // Transposed buffers: two (a slice is transposed while the previous one is
    // computed) unless that leaves fewer than two raw stages, as with 512-row
    // tiles; with one, the transpose waits for every warp to finish the slice.
    static constexpr size_t kT1Bytes = (size_t)((TA ? BK * BM : 0) + (TB ? BK * BN : 0)) * 4;
    static constexpr int kTBufs = (kSmemBudget - 2 * kT1Bytes) / kStageBytes >= 2 ? 2 : 1;
    static constexpr int kAtFloats = TA ? kTBufs * BK * BM : 4;
    static constexpr int kBtFloats = TB ? kTBufs * BK * BN : 4;
    static constexpr size_t kTBytes = (size_t)(kAtFloats + kBtFloats) * 4;
    static constexpr int kFit = (int)((kSmemBudget - kTBytes) / kStageBytes);
    static constexpr int kStages = kFit > 4 ? 4 : kFit;
    static_assert(kStages >= 2, "at least two raw stages");
    // TMA boxes span at most 256 rows: a 512-row K-major A comes in two.
    static constexpr int kABoxes = BM > 256 ? BM / 256 : 1;
    static_assert(BM <= 256 || TA, "an MN-major A box spans at most 256 rows");
    // Slices issued ahead of the one being computed.
    static constexpr int kLookahead = kRawEarly ? kStages : kStages - 1;
    struct Smem {
        float a[kStages][BM * BK];
        float b[kStages][BN * BK];
        float at[kAtFloats];          // TA: [kTBufs][BK][BM]
        float bt[kBtFloats];          // TB: [kTBufs][BK][BN]
        uint64_t full[kStages];
        uint64_t empty[kStages];
        uint64_t t_done[2];           // every thread wrote its part of buffer b
        uint64_t t_used[2];           // every thread finished reading buffer b
        uint64_t stored;    // every thread has written its partial (stream-K head)
        uint64_t ready;     // the predecessor's partial is visible (stream-K tail)
        Schedule sched;     // the CTA's work list, computed once by thread 0
        Issuer iss;         // copy issuer state (thread 0)
    };
    static constexpr size_t kSmemBytes = sizeof(Smem) + 1024;   // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// Transposes one K-major operand slice ([R rows][32 k], 128-byte swizzle) into
// [32 k][R] in 4-row x 4-k quads: four 16-byte loads and four 16-byte stores
// per task.  A 16-byte access is served a quarter-warp at a time; its 8 lanes
// (task bits 0..2 = x, y, z) take row quads nq = (x, y, z, ..) and k chunks
// c = (y ^ t3, z ^ t4, t5) (t = task bits), so the loads read chunk
// c ^ (row & 7), bits (y, z, x) up to a constant, and the stores write chunk
// nq & 7 of rows R floats apart: 8 distinct chunks either way, no bank
// conflict.  (A row-per-lane form with 4-byte stores, once used for 256-row
// slices, issued 2.5x the instructions and ran 2-4% slower on products with
// both operands K-major.)
// Quad task -> (row quad nq, k chunk c), see above.
__device__ __forceinline__ int quad_row(int task) { return (task & 7) | ((task >> 6) << 3); }
__device__ __forceinline__ int quad_chunk(int task) {
    return (((task >> 1) ^ (task >> 3)) & 1) | ((((task >> 2) ^ (task >> 4)) & 1) << 1) |
           (((task >> 5) & 1) << 2);
}

template <int R>
__device__ __forceinline__ void quad_load(const float* raw, int task, float4 (&v)[4]) {
    const int nq = quad_row(task), c = quad_chunk(task);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int row = 4 * nq + r;
        v[r] = *reinterpret_cast<const float4*>(reinterpret_cast<const char*>(raw) + row * 128 +
                                                (((c ^ (row & 7)) & 7) << 4));
    }
}

template <int R>
__device__ __forceinline__ void quad_store(float* dst, int task, const float4 (&v)[4]) {
    const int nq = quad_row(task), c = quad_chunk(task);
    float* d = dst + (4 * c) * R + 4 * nq;
    *reinterpret_cast<float4*>(d) = make_float4(v[0].x, v[1].x, v[2].x, v[3].x);
    *reinterpret_cast<float4*>(d + R) = make_float4(v[0].y, v[1].y, v[2].y, v[3].y);
    *reinterpret_cast<float4*>(d + 2 * R) = make_float4(v[0].z, v[1].z, v[2].z, v[3].z);
    *reinterpret_cast<float4*>(d + 3 * R) = make_float4(v[0].w, v[1].w, v[2].w, v[3].w);
}

// Transposes the K-major slices of A (RA rows) and B (RB rows; 0 = not
// transposed).  Every load of the thread's tasks is issued before any store:
// the compiler cannot move a load of one buffer above a store to another, and
// the transposes sit on every warp's path between two slices.
template <int RA, int RB>
__device__ __forceinline__ void transpose_slices(const float* rawA, float* dstA, const float* rawB,
                                                 float* dstB) {
    static_assert(BK / 4 == 8 && RA % 32 == 0 && RB % 32 == 0, "8 chunks; whole quarter-warps");
    constexpr int NA = RA / 4 * (BK / 4), NB = RB / 4 * (BK / 4);   // tasks
    constexpr int TA_ = (NA + kThreads - 1) / kThreads;             // tasks per thread
    constexpr int TB_ = (NB + kThreads - 1) / kThreads;
    static_assert(NA % 32 == 0 && NB % 32 == 0, "whole warps of tasks");
    float4 va[TA_ > 0 ? TA_ : 1][4], vb[TB_ > 0 ? TB_ : 1][4];
    // Only a part of the last round has a task when the count is not a
    // multiple of the block (64-row slices).
    auto has = [](int n, int j) { return n % kThreads == 0 || (int)threadIdx.x + j * kThreads < n; };
#pragma unroll
    for (int j = 0; j < TA_; ++j)
        if (has(NA, j)) quad_load<RA>(rawA, threadIdx.x + j * kThreads, va[j]);
#pragma unroll
    for (int j = 0; j < TB_; ++j)
        if (has(NB, j)) quad_load<RB>(rawB, threadIdx.x + j * kThreads, vb[j]);
#pragma unroll
    for (int j = 0; j < TA_; ++j)
        if (has(NA, j)) quad_store<RA>(dstA, threadIdx.x + j * kThreads, va[j]);
#pragma unroll
    for (int j = 0; j < TB_; ++j)
        if (has(NB, j)) quad_store<RB>(dstB, threadIdx.x + j * kThreads, vb[j]);
}

struct TileCoord { int64_t b, m0, n0; };

// Tile t -> (batch entry, first row, first column); grouped raster of 8
// tile-rows within a batch entry so concurrently resident CTAs share slices.
template <int BM, int BN>
__device__ __forceinline__ TileCoord raster_coord(int64_t t, int64_t tiles_m, int64_t tiles_n) {
    const int64_t per_batch = tiles_m * tiles_n;
    const int64_t b = t / per_batch;
    const int64_t r = t - b * per_batch;
    constexpr int64_t G = 8;
    const int64_t group = r / (G * tiles_n);
    const int64_t first_m = group * G;
    const int64_t gm = (tiles_m - first_m < G) ? (tiles_m - first_m) : G;
    const int64_t w = r - group * G * tiles_n;
    return {b, (first_m + w % gm) * BM, (w / gm) * BN};
}

// With a weighted split the tiles of the last column come after all others.
template <int BM, int BN>
__device__ __forceinline__ TileCoord tile_coord(const Params& p, int64_t t) {
    if (p.w_full == 0) return raster_coord<BM, BN>(t, p.tiles_m, p.tiles_n);
    if (t < p.full_tiles) return raster_coord<BM, BN>(t, p.tiles_m, p.tiles_n - 1);
    const int64_t r = t - p.full_tiles;
    const int64_t b = r / p.tiles_m;
    return {b, (r - b * p.tiles_m) * BM, (p.tiles_n - 1) * BN};
}

// Thread -> tile row of its i-th A row (16) / tile column of its j-th B column
// (8): runs of 4 adjacent values (one 16-byte load), the runs of a thread 16
// rows / 32 columns apart so the lanes of a warp cover 64 x 64.
__device__ __forceinline__ int row_of(int wbase, int lm, int i) {
    return wbase + (i >> 2) * 16 + lm * 4 + (i & 3);
}
__device__ __forceinline__ int col_of(int wbase, int ln, int j) {
    return wbase + (j >> 2) * 32 + ln * 4 + (j & 3);
}

// Accumulators of the 16 x 8 micro-tile as 64 float pairs.  PAIR_I pairs rows
// (i, i+1) of one column, otherwise columns (j, j+1) of one row.
template <bool PAIR_I>
__device__ __forceinline__ float& acc_at(float2 (&acc)[64], int i, int j) {
    if (PAIR_I) return (i & 1) ? acc[(i >> 1) * TN + j].y : acc[(i >> 1) * TN + j].x;
    return (j & 1) ? acc[i * (TN / 2) + (j >> 1)].y : acc[i * (TN / 2) + (j >> 1)].x;
}

// acc(i, j) += a[i] * b[j] for one k.
template <bool PAIR_I>
__device__ __forceinline__ void fma_step(float2 (&acc)[64], const float (&a)[TM], const float (&b)[TN]) {
    if (PAIR_I) {
#pragma unroll
        for (int ip = 0; ip < TM / 2; ++ip) {
            const float2 av = make_float2(a[2 * ip], a[2 * ip + 1]);
#pragma unroll
            for (int j = 0; j < TN; ++j)
                acc[ip * TN + j] = __ffma2_rn(av, make_float2(b[j], b[j]), acc[ip * TN + j]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const float2 av = make_float2(a[i], a[i]);
#pragma unroll
            for (int jp = 0; jp < TN / 2; ++jp)
                acc[i * (TN / 2) + jp] =
                    __ffma2_rn(av, make_float2(b[2 * jp], b[2 * jp + 1]), acc[i * (TN / 2) + jp]);
        }
    }
}

template <int BM, int BN, bool A_K, bool B_K>
__device__ __forceinline__ void issue_next(typename Cfg<BM, BN, A_K, B_K>::Smem& sh, const CUtensorMap* ta,
                                           const CUtensorMap* tb, const Params& p,
                                           const Schedule& sc, Issuer& is) {
    using C = Cfg<BM, BN, A_K, B_K>;
    if (is.cw != is.w) {
        const Item itm = sc.item(is.w, p.nk);
        const TileCoord tc = tile_coord<BM, BN>(p, itm.tile);
        is.cw = is.w;
        is.kb = itm.kb;
        is.ke = itm.ke;
        is.m0 = (int)tc.m0;
        is.n0 = (int)tc.n0;
        is.ba = p.a_bcast ? 0 : (int)tc.b;
        is.bb = p.b_bcast ? 0 : (int)tc.b;
        if (is.kt < is.kb) is.kt = is.kb;
    }
    const int s = (int)(is.issued % C::kStages);
    const int ba = is.ba, bb = is.bb;
    const int k0 = is.kt * BK;
    mbar_arrive_expect_tx(&sh.full[s], C::kStageBytes);
    if (A_K) {
#pragma unroll
        for (int j = 0; j < C::kABoxes; ++j)
            tma_load_3d(sh.a[s] + j * 256 * BK, ta, &sh.full[s], k0, is.m0 + 256 * j, ba);
    } else {
        tma_load_3d(sh.a[s], ta, &sh.full[s], is.m0, k0, ba);
    }
    if (B_K) tma_load_3d(sh.b[s], tb, &sh.full[s], k0, is.n0, bb);
    else     tma_load_3d(sh.b[s], tb, &sh.full[s], is.n0, k0, bb);
    ++is.issued;
    if (++is.kt == is.ke) { is.kt = 0; ++is.w; }
}

// On a failed wait the issuer may still have copies landing in shared memory;
// it waits (bounded) for every slice it issued beyond `consumed`.
template <int STAGES>
__device__ __forceinline__ void drain(uint64_t* full, uint64_t consumed, uint64_t issued) {
    for (uint64_t q = consumed; q < issued; ++q)
        if (!mbar_wait(&full[q % STAGES], (uint32_t)((q / STAGES) & 1))) {
            record_status(&g_wait_status, kWaitDrain);
            return;
        }
}

// Slices the issuer has loaded that the consumers have not yet taken, given the
// consumers' 32-bit running count (the issuer is never more than a few stages
// ahead, so the low 32 bits of the difference are exact).
__device__ __forceinline__ uint64_t in_flight(uint64_t issued, uint32_t consumed) {
    return (uint64_t)(uint32_t)((uint32_t)issued - consumed);
}


// Fused addend and activation over the outputs of one thread's micro-tile,
// which it has just stored, read back 4 rows x 8 columns at a time through L2
// (float4 when C is row-major), then D added and the activation applied, one
// function per instantiation.  An addend constant along M (a bias per column)
// is loaded once per tile.
template <int ACT>
__device__ __forceinline__ void fused_pass(const Params& p, const TileCoord& tc, int wm, int wn,
                                           int lm, int ln) {
    constexpr int G = 4;
    float* Cb = p.C + tc.b * p.bsC;
    const float* Db = p.epi.D ? p.epi.D + tc.b * p.epi.bsD : nullptr;
    const bool d_per_col = Db && p.epi.rsD == 0;
    int64_t ncol[TN];
    float d_col[TN];
#pragma unroll
    for (int j = 0; j < TN; ++j) {
        ncol[j] = tc.n0 + col_of(wn, ln, j);
        const float* d = Db ? Db + ncol[j] * p.epi.csD : nullptr;
        d_col[j] = (d_per_col && ncol[j] < p.N && dbg_in_span(p.epi.D, d, p.epi.d_span, &g_wait_status))
                       ? __ldg(d) : 0.0f;
    }
    const bool vec = p.c_vec4 && ncol[TN - 1] < p.N;   // both runs of 4 wholly inside C
    auto load = [&](float (&v)[G][TN], int i0) {
#pragma unroll
        for (int i = 0; i < G; ++i) {
            const int64_t m = tc.m0 + row_of(wm, lm, i0 + i);
            const float* crow = Cb + (m < p.M ? m : 0) * p.rsC;
            if (vec) {
#pragma unroll
                for (int h = 0; h < TN / 4; ++h) {
                    const float4 c4 = (m < p.M && c_ok(p, crow + ncol[4 * h], 4))
                                          ? __ldcg(reinterpret_cast<const float4*>(crow + ncol[4 * h]))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[i][4 * h] = c4.x; v[i][4 * h + 1] = c4.y; v[i][4 * h + 2] = c4.z; v[i][4 * h + 3] = c4.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < TN; ++j)
                    v[i][j] = (m < p.M && ncol[j] < p.N && c_ok(p, crow + ncol[j] * p.csC, 1))
                                  ? __ldcg(crow + ncol[j] * p.csC) : 0.0f;
            }
        }
    };
    auto finish_store = [&](float (&v)[G][TN], int i0) {
#pragma unroll
        for (int i = 0; i < G; ++i) {
            const int64_t m = tc.m0 + row_of(wm, lm, i0 + i);
            if (m >= p.M) continue;
            float* crow = Cb + m * p.rsC;
            const float* drow = (Db && !d_per_col) ? Db + m * p.epi.rsD : nullptr;
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                float z = v[i][j];
                if (d_per_col) {
                    z += d_col[j];
                } else if (drow && ncol[j] < p.N &&
                           dbg_in_span(p.epi.D, drow + ncol[j] * p.epi.csD, p.epi.d_span, &g_wait_status)) {
                    z += __ldg(drow + ncol[j] * p.epi.csD);
                }
                v[i][j] = act_fn<ACT>(z);
            }
            if (vec) {
#pragma unroll
                for (int h = 0; h < TN / 4; ++h)
                    if (c_ok(p, crow + ncol[4 * h], 4))
                        *reinterpret_cast<float4*>(crow + ncol[4 * h]) =
                            make_float4(v[i][4 * h], v[i][4 * h + 1], v[i][4 * h + 2], v[i][4 * h + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < TN; ++j)
                    if (ncol[j] < p.N && c_ok(p, crow + ncol[j] * p.csC, 1)) crow[ncol[j] * p.csC] = v[i][j];
            }
        }
    };
#pragma unroll 1
    for (int i0 = 0; i0 < TM; i0 += G) {
        float v[G][TN];
        load(v, i0);
        finish_store(v, i0);
    }
}

template <int BM, int BN, bool A_K, bool B_K>
__global__ void __launch_bounds__(kThreads, 1)
tma_ffma_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                const Params p) {
    constexpr bool TA = A_K, TB = B_K;   // K-major operands are transposed in smem
    constexpr bool TT = TA || TB;
    using C = Cfg<BM, BN, TA, TB>;
    constexpr int S = C::kStages;
    constexpr bool RAW_EARLY = C::kRawEarly;
    constexpr uint32_t NT = C::kTBufs;
    extern __shared__ uint8_t smem_raw[];
    auto& sh = *reinterpret_cast<typename C::Smem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const bool issuer = threadIdx.x == 0;
    const Schedule& sc = sh.sched;
    Issuer& is = sh.iss;
    if (issuer) {
        if (p.w_full)
            sh.sched.init_weighted(p.dp_tiles, p.sk_units, p.nk, p.sk_full_units, p.w_full, p.w_rag);
        else
            sh.sched.init(p.dp_tiles, p.sk_units, p.nk);
        is.w = 0;
        is.kt = 0;
        is.cw = -1;
        is.issued = 0;
        is.total = sh.sched.slices(p.nk);
        for (int s = 0; s < S; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], kWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.t_done[b], kThreads);
            mbar_init(&sh.t_used[b], kThreads);
        }
        mbar_init(&sh.stored, kThreads);
        mbar_init(&sh.ready, 1);
        fence_mbar_init();
        prefetch_tensormap(&ta);
        prefetch_tensormap(&tb);
    }
    __syncthreads();
    if (issuer) {
        for (int q = 0; q < C::kLookahead && (int64_t)is.issued < is.total; ++q)
            issue_next<BM, BN, A_K, B_K>(sh, &ta, &tb, p, sc, is);
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wm = (warp % C::kWarpsM) * WTM, wn = (warp / C::kWarpsM) * WTN;
    const int lm = lane >> 3, ln = lane & 7;
    // Both operands reach the mainloop MN-major: pair rows of A (adjacent in
    // one 16-byte load), broadcast B.
    constexpr bool PI = true;
    uint32_t it = 0;        // slices consumed so far (low 32 bits)
    int stage = 0;          // it % S, kept incrementally
    uint32_t phase = 0;     // (it / S) & 1
    const int64_t n_items = sc.n_items;
    if constexpr (TT) {
        // The first slice is transposed before the loop, every later one at
        // the end of the previous slice's iteration.
        if (is.total > 0) {
            if (!mbar_wait(&sh.full[0], 0)) {
                record_status(&g_wait_status, kWaitFull);
                if (issuer) drain<S>(sh.full, 0, is.issued);
                return;
            }
            transpose_slices<TA ? BM : 0, TB ? BN : 0>(sh.a[0], sh.at, sh.b[0], sh.bt);
            if constexpr (RAW_EARLY) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.empty[0]);
            }
            mbar_arrive(&sh.t_done[0]);
        }
    }
    for (int64_t w = 0; w < n_items; ++w) {
        float2 acc[64];
        if (sc.item(w, p.nk).mode == kTail && !p.indep) {
            // Continue the predecessor's FMA chains from its partial sums.
            const float2* src = p.ws_partial + (int64_t)(blockIdx.x - 1) * (kThreads * 64);
            if (issuer) {
                if (!wait_flag(p.ws_flag + (blockIdx.x - 1))) {
                    record_status(&g_wait_status, kWaitPartial);
                    drain<S>(sh.full, is.issued - in_flight(is.issued, it), is.issued);
                    return;
                }
                mbar_arrive(&sh.ready);
            }
            if (!mbar_wait(&sh.ready, 0)) {
                record_status(&g_wait_status, kWaitPartial);
                return;
            }
#pragma unroll
            for (int q = 0; q < 64; ++q) acc[q] = __ldcg(src + q * kThreads + threadIdx.x);
        } else {
#pragma unroll
            for (int q = 0; q < 64; ++q) acc[q] = make_float2(0.0f, 0.0f);
        }

        int kt_end;
        bool busy;          // this warp's 64 x 64 block holds outputs of the tile
        {
            const Item itm = sc.item(w, p.nk);
            kt_end = itm.ke - itm.kb;
            const TileCoord t0 = tile_coord<BM, BN>(p, itm.tile);
            busy = t0.m0 + wm < p.M && t0.n0 + wn < p.N;
        }
        for (int kt = 0; kt < kt_end; ++kt, ++it) {
            if (issuer && (int64_t)is.issued < is.total) {
                // Refill the stage every warp released at slice it-1.
                if (is.issued >= (uint64_t)S &&
                    !mbar_wait(&sh.empty[is.issued % S], (uint32_t)(((is.issued / S) - 1) & 1))) {
                    record_status(&g_wait_status, kWaitEmpty);
                    drain<S>(sh.full, is.issued - in_flight(is.issued, it), is.issued);
                    return;
                }
                issue_next<BM, BN, A_K, B_K>(sh, &ta, &tb, p, sc, is);
            }
            const int s = stage;
            if (!RAW_EARLY && !mbar_wait(&sh.full[s], phase)) {
                record_status(&g_wait_status, kWaitFull);
                if (issuer) drain<S>(sh.full, is.issued - in_flight(is.issued, it), is.issued);
                return;
            }
            if (++stage == S) { stage = 0; phase ^= 1u; }
            const float* As = TA ? sh.at + (it % NT) * (BK * BM) : sh.a[s];
            const float* Bs = TB ? sh.bt + (it % NT) * (BK * BN) : sh.b[s];
            if constexpr (TT) {
                if (!mbar_wait(&sh.t_done[it % NT], (it / NT) & 1)) {
                    record_status(&g_wait_status, kWaitFull);
                    if (issuer) drain<S>(sh.full, is.issued - in_flight(is.issued, it), is.issued);
                    return;
                }
            }
            // A warp whose block lies wholly past a ragged edge (N = 64 in a
            // 128-wide tile, say) skips the FMAs; it still takes its part in
            // the transposes and the stage barriers.
            if (busy) {
                // One k ahead: the next k's fragments (24 registers, 16-byte
                // loads of 4 adjacent rows of A and columns of B) load while
                // this k's 64 packed FMAs run.  Deeper unrolling spills.
                float fa[2][TM], fb[2][TN];
                const float* arow = As + wm + lm * 4;
                const float* brow = Bs + wn + ln * 4;
#pragma unroll
                for (int q = 0; q < TM / 4; ++q) {
                    const float4 v = *reinterpret_cast<const float4*>(arow + q * 16);
                    fa[0][4 * q] = v.x; fa[0][4 * q + 1] = v.y; fa[0][4 * q + 2] = v.z; fa[0][4 * q + 3] = v.w;
                }
#pragma unroll
                for (int q = 0; q < TN / 4; ++q) {
                    const float4 v = *reinterpret_cast<const float4*>(brow + q * 32);
                    fb[0][4 * q] = v.x; fb[0][4 * q + 1] = v.y; fb[0][4 * q + 2] = v.z; fb[0][4 * q + 3] = v.w;
                }
#pragma unroll 4
                for (int k = 0; k < BK; ++k) {
                    const int cur = k & 1;
                    if (k + 1 < BK) {
#pragma unroll
                        for (int q = 0; q < TM / 4; ++q) {
                            const float4 v = *reinterpret_cast<const float4*>(arow + (k + 1) * BM + q * 16);
                            fa[cur ^ 1][4 * q] = v.x; fa[cur ^ 1][4 * q + 1] = v.y;
                            fa[cur ^ 1][4 * q + 2] = v.z; fa[cur ^ 1][4 * q + 3] = v.w;
                        }
#pragma unroll
                        for (int q = 0; q < TN / 4; ++q) {
                            const float4 v = *reinterpret_cast<const float4*>(brow + (k + 1) * BN + q * 32);
                            fb[cur ^ 1][4 * q] = v.x; fb[cur ^ 1][4 * q + 1] = v.y;
                            fb[cur ^ 1][4 * q + 2] = v.z; fb[cur ^ 1][4 * q + 3] = v.w;
                        }
                    }
                    fma_step<PI>(acc, fa[cur], fb[cur]);
                }
            }
            if constexpr (!RAW_EARLY) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.empty[s]);
            }
            if constexpr (TT) {
                mbar_arrive(&sh.t_used[it % NT]);
                const uint32_t nx = it + 1;
                if ((int64_t)nx < is.total) {
                    const int nb = (int)(nx % NT);
                    // Buffer nb last held slice nx-NT: every thread must be done with it,
                    // and slice nx's raw tiles (stage `stage`, phase `phase`) must have landed.
                    const bool ok = (nx < NT || mbar_wait(&sh.t_used[nb], ((nx / NT) - 1) & 1)) &&
                                    mbar_wait(&sh.full[stage], phase);
                    if (!ok) {
                        record_status(&g_wait_status, kWaitFull);
                        if (issuer) drain<S>(sh.full, is.issued - in_flight(is.issued, nx), is.issued);
                        return;
                    }
                    transpose_slices<TA ? BM : 0, TB ? BN : 0>(sh.a[stage], sh.at + nb * (BK * BM),
                                                               sh.b[stage], sh.bt + nb * (BK * BN));
                    if constexpr (RAW_EARLY) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sh.empty[stage]);
                    }
                    mbar_arrive(&sh.t_done[nb]);
                }
            }
        }

        const Item itm = sc.item(w, p.nk);
        if (itm.mode == kHead) {
            // Leave the partial sums for the next CTA, then raise its flag once
            // every thread's stores are visible device-wide.
            float2* dst = p.ws_partial + (int64_t)blockIdx.x * (kThreads * 64);
#pragma unroll
            for (int q = 0; q < 64; ++q) __stcg(dst + q * kThreads + threadIdx.x, acc[q]);
            __threadfence();
            mbar_arrive(&sh.stored);
            if (issuer) {
                if (!mbar_wait(&sh.stored, 0)) {
                    record_status(&g_wait_status, kWaitPartial);
                    drain<S>(sh.full, is.issued - in_flight(is.issued, it), is.issued);
                    return;
                }
                st_release_gpu(p.ws_flag + blockIdx.x, 1u);
            }
            continue;
        }

        if (itm.mode == kTail && p.indep) {
            // Add the earlier pieces of this tile, latest CTA first, once all
            // of them are published.
            const int64_t first = unit_owner((itm.tile - p.dp_tiles) * p.nk, p.sk_units, gridDim.x);
            if (issuer) {
                for (int64_t c = first; c < (int64_t)blockIdx.x; ++c)
                    if (!wait_flag(p.ws_flag + c)) {
                        record_status(&g_wait_status, kWaitPartial);
                        drain<S>(sh.full, is.issued - in_flight(is.issued, it), is.issued);
                        return;
                    }
                mbar_arrive(&sh.ready);
            }
            if (!mbar_wait(&sh.ready, 0)) {
                record_status(&g_wait_status, kWaitPartial);
                return;
            }
#pragma unroll 1
            for (int64_t c = (int64_t)blockIdx.x - 1; c >= first; --c) {
                const float2* src = p.ws_partial + c * (kThreads * 64);
#pragma unroll
                for (int q = 0; q < 64; ++q) {
                    const float2 v = __ldcg(src + q * kThreads + threadIdx.x);
                    acc[q].x += v.x;
                    acc[q].y += v.y;
                }
            }
        }

        // Epilogue straight from registers.  A fused bias per column, with
        // ReLU or no activation, is applied here too (a few instructions per
        // output, in a copy of the epilogue of its own, so the plain one stays
        // as it is); any other fused epilogue runs as a second pass below.
        const TileCoord tc = tile_coord<BM, BN>(p, itm.tile);
        float* Cb = p.C + tc.b * p.bsC;
        auto store_acc = [&](auto fused) {
            constexpr bool F = decltype(fused)::value;
            float bias[TN];
            bool relu = false;
            if constexpr (F) {
#pragma unroll
                for (int j = 0; j < TN; ++j) {
                    const int64_t n = tc.n0 + col_of(wn, ln, j);
                    const float* d = p.epi.D ? p.epi.D + tc.b * p.epi.bsD + n * p.epi.csD : nullptr;
                    bias[j] = (p.epi.D && n < p.N && dbg_in_span(p.epi.D, d, p.epi.d_span, &g_wait_status))
                                  ? __ldg(d) : 0.0f;
                }
                relu = p.epi.act == kActRelu;
            }
            const int64_t n0c = tc.n0 + wn;
            auto ncol = [&](int j) { return n0c + col_of(0, ln, j); };
            // Both runs of 4 wholly inside a row-major, 16-byte aligned C: float4.
            const bool vec = p.c_vec4 && ncol(TN - 1) < p.N;
            auto put = [&](int i, float (&r)[TN]) {
                const int64_t m = tc.m0 + row_of(wm, lm, i);
                float* crow = Cb + m * p.rsC;
                if constexpr (F) {
#pragma unroll
                    for (int j = 0; j < TN; ++j) {
                        r[j] += bias[j];
                        if (relu) r[j] = fmaxf(r[j], 0.0f);
                    }
                }
                if (vec) {
#pragma unroll
                    for (int h = 0; h < TN / 4; ++h)
                        if (c_ok(p, crow + ncol(4 * h), 4))
                            *reinterpret_cast<float4*>(crow + ncol(4 * h)) =
                                make_float4(r[4 * h], r[4 * h + 1], r[4 * h + 2], r[4 * h + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < TN; ++j)
                        if (ncol(j) < p.N && c_ok(p, crow + ncol(j) * p.csC, 1)) crow[ncol(j) * p.csC] = r[j];
                }
            };
            if (p.accumulate) {
                // C_old of G rows is loaded before any of them is stored, so the
                // loads are in flight together (the compiler cannot move a load
                // of C above a store to C).
                constexpr int G = 4;   // 2 ran slower, 8 spilled
#pragma unroll
                for (int i0 = 0; i0 < TM; i0 += G) {
                    float old[G][TN];
#pragma unroll
                    for (int i = 0; i < G; ++i) {
                        const int64_t m = tc.m0 + row_of(wm, lm, i0 + i);
                        const float* crow = Cb + (m < p.M ? m : 0) * p.rsC;
                        if (vec) {
#pragma unroll
                            for (int h = 0; h < TN / 4; ++h) {
                                const float4 o = (m < p.M && c_ok(p, crow + ncol(4 * h), 4))
                                                     ? *reinterpret_cast<const float4*>(crow + ncol(4 * h))
                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                                old[i][4 * h] = o.x; old[i][4 * h + 1] = o.y;
                                old[i][4 * h + 2] = o.z; old[i][4 * h + 3] = o.w;
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < TN; ++j)
                                old[i][j] = (m < p.M && ncol(j) < p.N && c_ok(p, crow + ncol(j) * p.csC, 1))
                                                ? crow[ncol(j) * p.csC] : 0.0f;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < G; ++i) {
                        if (tc.m0 + row_of(wm, lm, i0 + i) >= p.M) continue;
                        float r[TN];
#pragma unroll
                        for (int j = 0; j < TN; ++j) r[j] = fmaf(p.alpha, acc_at<PI>(acc, i0 + i, j), old[i][j]);
                        put(i0 + i, r);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    if (tc.m0 + row_of(wm, lm, i) >= p.M) continue;
                    float r[TN];
#pragma unroll
                    for (int j = 0; j < TN; ++j) r[j] = p.alpha * acc_at<PI>(acc, i, j);
                    put(i, r);
                }
            }
        };
        if (p.epi_inline) store_acc(std::true_type{});
        else store_acc(std::false_type{});
        if (p.epi.on && !p.epi_inline) {
            // Fused addend and activation: every thread revisits the outputs it
            // has just stored (still in L2), so the register epilogue above
            // stays the plain product's.
            switch (p.epi.act) {
                case kActRelu: fused_pass<kActRelu>(p, tc, wm, wn, lm, ln); break;
                case kActSigmoid: fused_pass<kActSigmoid>(p, tc, wm, wn, lm, ln); break;
                case kActSilu: fused_pass<kActSilu>(p, tc, wm, wn, lm, ln); break;
                case kActGeluTanh: fused_pass<kActGeluTanh>(p, tc, wm, wn, lm, ln); break;
                case kActGeluErf: fused_pass<kActGeluErf>(p, tc, wm, wn, lm, ln); break;
                default: fused_pass<kActNone>(p, tc, wm, wn, lm, ln); break;
            }
        }
    }
}

// Operand tensor map: the inner index has unit stride.  `inner`, `outer` are
// the logical extents along the unit-stride index and the other index; `so`
// the other index's stride, `sb` the batch stride (elements); `box_rows` the
// tile extent along the non-k index.
bool make_map(CUtensorMap* map, const float* base, int64_t inner, int64_t outer, int64_t so,
              int64_t sb, int64_t batch, bool broadcast, bool k_major, int box_rows) {
    const int64_t nb = broadcast ? 1 : batch;
    // A stride over an extent of 1 is never used; give it a legal value.
    const int64_t so_b = outer > 1 ? so * 4 : ((inner * 4 + 15) / 16) * 16;
    const int64_t sb_b = nb > 1 ? sb * 4 : so_b * (outer > 1 ? outer : 1);
    const uint64_t dims[3] = {(uint64_t)inner, (uint64_t)outer, (uint64_t)nb};
    const uint64_t strides[2] = {(uint64_t)so_b, (uint64_t)sb_b};
    const uint32_t box[3] = {k_major ? (uint32_t)BK : (uint32_t)box_rows,
                             k_major ? (uint32_t)box_rows : (uint32_t)BK, 1};
    return encode_tmap_f32_3d(map, base, dims, strides, box, k_major);
}

template <int BM, int BN, bool A_K, bool B_K>
cudaError_t launch_impl(const Problem& pr, const Plan& plan, int sm_count, cudaStream_t stream) {
    using C = Cfg<BM, BN, A_K, B_K>;
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(tma_ffma_kernel<BM, BN, A_K, B_K>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    CUtensorMap ta, tb;
    const bool a_bc = pr.batch == 1 || pr.bsA == 0;
    const bool b_bc = pr.batch == 1 || pr.bsB == 0;
    // A: K-major -> inner K, outer M (stride rsA); MN-major -> inner M, outer K (csA).
    if (!make_map(&ta, pr.A, A_K ? pr.K : pr.M, A_K ? pr.M : pr.K, A_K ? pr.rsA : pr.csA,
                  pr.bsA, pr.batch, a_bc, A_K, BM / C::kABoxes))
        return cudaErrorInvalidValue;
    // B: K-major -> inner K, outer N (csB); MN-major -> inner N, outer K (rsB).
    if (!make_map(&tb, pr.B, B_K ? pr.K : pr.N, B_K ? pr.N : pr.K, B_K ? pr.csB : pr.rsB,
                  pr.bsB, pr.batch, b_bc, B_K, BN))
        return cudaErrorInvalidValue;
    Params p;
    p.C = pr.C; p.rsC = pr.rsC; p.csC = pr.csC; p.bsC = pr.bsC;
    p.M = pr.M; p.N = pr.N; p.K = pr.K;
    p.tiles_m = plan.tiles_m; p.tiles_n = plan.tiles_n; p.tiles_total = plan.tiles;
    p.nk = (int)((pr.K + BK - 1) / BK);
    p.alpha = pr.alpha;
    p.accumulate = pr.accumulate;
    p.a_bcast = a_bc;
    p.b_bcast = b_bc;
    p.c_vec4 = pr.csC == 1 && (reinterpret_cast<uintptr_t>(pr.C) % 16 == 0) &&
               (pr.M == 1 || pr.rsC % 4 == 0) && (pr.batch == 1 || pr.bsC % 4 == 0);
    const int64_t grid = plan.ctas;
    p.dp_tiles = plan.stream_k ? plan.dp_tiles : plan.tiles;
    p.sk_units = plan.stream_k ? (plan.tiles - plan.dp_tiles) * p.nk : 0;
    p.indep = plan.stream_k && plan.split_indep ? 1 : 0;
    p.full_tiles = p.sk_full_units = 0;
    p.w_full = p.w_rag = 0;
    const int64_t rag = pr.N % BN;
    if (plan.stream_k && !plan.split_indep && rag != 0 && 2 * rag <= BN && p.tiles_n > 1) {
        // The tiles of the last column hold at most BN / 2 columns: the warps
        // past it skip their FMAs, one per scheduler, and such a tile measured
        // 0.67 of a full one's time (N = 960 in 128-wide tiles).
        constexpr int kWf = 3, kWr = 2;
        const int64_t full = p.tiles_m * (p.tiles_n - 1) * pr.batch;
        if (p.dp_tiles <= full) {
            const int64_t skf = (full - p.dp_tiles) * p.nk;
            const int64_t total = skf * kWf + (p.sk_units - skf) * kWr;
            if (total >= grid * (int64_t)p.nk * kWf) {   // every range still spans a whole tile
                p.full_tiles = full;
                p.sk_full_units = skf;
                p.w_full = kWf;
                p.w_rag = kWr;
            }
        }
    }
    p.epi = pr.epi;
    p.epi_inline = pr.epi.on && (pr.epi.D == nullptr || pr.epi.rsD == 0) &&
                   (pr.epi.act == kActNone || pr.epi.act == kActRelu) ? 1 : 0;
    p.ws_partial = nullptr;
    p.ws_flag = nullptr;
    p.sc = pr.sc;
    if (plan.stream_k) {
        // Partials first, then one flag word per CTA (see workspace_bytes).
        p.ws_partial = static_cast<float2*>(plan.workspace);
        p.ws_flag = reinterpret_cast<unsigned int*>(
            static_cast<char*>(plan.workspace) + (size_t)grid * kThreads * 64 * sizeof(float2));
        cudaError_t e = cudaMemsetAsync(p.ws_flag, 0, (size_t)grid * sizeof(unsigned int), stream);
        if (e != cudaSuccess) return e;
        // CTAs wait on one another's partial sums: make them co-resident.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, tma_ffma_kernel<BM, BN, A_K, B_K>, ta, tb, p);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    tma_ffma_kernel<BM, BN, A_K, B_K><<<(unsigned)grid, kThreads, C::kSmemBytes, stream>>>(ta, tb, p);
    return cudaGetLastError();
}

template <int BM, int BN>
cudaError_t launch_tile(const Problem& p, const Plan& plan, int sm_count, cudaStream_t stream) {
    const bool ak = plan.a_layout == SBGEMM_LAYOUT_K_MAJOR;
    const bool bk = plan.b_layout == SBGEMM_LAYOUT_K_MAJOR;
    if (ak && bk) return launch_impl<BM, BN, true, true>(p, plan, sm_count, stream);
    if (ak) return launch_impl<BM, BN, true, false>(p, plan, sm_count, stream);
    if (bk) return launch_impl<BM, BN, false, true>(p, plan, sm_count, stream);
    return launch_impl<BM, BN, false, false>(p, plan, sm_count, stream);
}

// This translation unit's copy of the kernels' status word (each tile shape is
// compiled on its own), read and cleared by the host.
inline unsigned int read_and_clear_status(cudaStream_t stream) {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_wait_status, sizeof(v), 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_wait_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return v;
}

}  // namespace
}  // namespace sbg
