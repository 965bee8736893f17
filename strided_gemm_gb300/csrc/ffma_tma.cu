// TMA-fed FFMA path for operands with a unit stride (K-major or MN-major) whose
// other strides are 16-byte multiples.
//
// Persistent CTAs (one per SM) of eight warps walk their output tiles.  Each
// tile's K range is cut into BK-deep slices that TMA copies (one box of A, one
// of B) into a ring of shared-memory stages; "full" mbarriers signal a landed
// stage and "empty" mbarriers (one arrival per warp) its release.  Thread 0
// doubles as the copy issuer: at every slice it refills the stage that all
// warps released one slice earlier, so copies run kStages-1 slices ahead,
// across tile boundaries too (the next tile streams in during an epilogue).
//
// Each warp computes a 64 x 64 warp tile as 16 x 8 register micro-tiles per
// thread (the register blocking of the StaleyNET "GPU Implementation" page,
// section "The matrix product", grown from 4 x 4).  The micro-tile size is set
// by shared-memory bandwidth: an SM reads 32 fp32 words per clock from shared
// memory but retires 128 FMA lanes, so a thread must do at least 4 FMAs per
// word it loads; 16 x 8 does 128 per 24 (8 x 8 would sit exactly at the limit).
// The FMAs are packed two lanes per instruction (FFMA2, fma.rn.f32x2): pairs
// run along whichever operand arrives with adjacent values (an MN-major tile),
// the other operand is broadcast.  Each output still has one fused
// multiply-add chain in increasing k, so results are bit-identical to a
// scalar fmaf loop and across layouts.  The epilogue writes alpha*acc
// (+ C_old) straight from registers with masks on ragged M / N.
//
// Shared-memory layouts follow the operand's unit stride: a K-major tile is
// stored [row][32 k] with the TMA 128-byte swizzle (conflict-free 8-byte
// fragment reads along k), an MN-major tile [32 k][rows] unswizzled (16-byte
// fragment reads along m or n).  Out-of-range rows, columns and k are
// zero-filled by TMA.  Every mbarrier wait is bounded: on expiry the thread
// records a status code and returns (the copy issuer first waits, again
// bounded, for the copies it has in flight).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

#ifndef SBGEMM_FFMA2
#define SBGEMM_FFMA2 1
#endif
#ifndef SBGEMM_KUNROLL
#define SBGEMM_KUNROLL 2
#endif

namespace sbg {
namespace {

constexpr int BK = 32;
constexpr int kUnrollK = SBGEMM_KUNROLL;   // k-pair groups unrolled per slice
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
};

template <int BM, int BN>
struct Cfg {
    static constexpr int kWarpsM = BM / WTM, kWarpsN = BN / WTN;
    static_assert(kWarpsM * kWarpsN == kWarps, "8 warps of 64 x 64");
    static constexpr int kABytes = BM * BK * 4, kBBytes = BN * BK * 4;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = 4;
    struct Smem {
        float a[kStages][BM * BK];
        float b[kStages][BN * BK];
        uint64_t full[kStages];
        uint64_t empty[kStages];
    };
    static constexpr size_t kSmemBytes = sizeof(Smem) + 1024;   // + alignment slack
};

struct TileCoord { int64_t b, m0, n0; };

// Tile t -> (batch entry, first row, first column); grouped raster of 8
// tile-rows within a batch entry so concurrently resident CTAs share slices.
template <int BM, int BN>
__device__ __forceinline__ TileCoord tile_coord(const Params& p, int64_t t) {
    const int64_t per_batch = p.tiles_m * p.tiles_n;
    const int64_t b = t / per_batch;
    const int64_t r = t - b * per_batch;
    constexpr int64_t G = 8;
    const int64_t group = r / (G * p.tiles_n);
    const int64_t first_m = group * G;
    const int64_t gm = (p.tiles_m - first_m < G) ? (p.tiles_m - first_m) : G;
    const int64_t w = r - group * G * p.tiles_n;
    return {b, (first_m + w % gm) * BM, (w / gm) * BN};
}

// Thread -> tile row of its i-th A row (16) / tile column of its j-th B column
// (8).  K-major operands step by the lane count (distinct swizzle rows per
// load); MN-major operands take runs of 4 adjacent values (one 16-byte load).
template <bool K_MAJOR>
__device__ __forceinline__ int row_of(int wbase, int lm, int i) {
    return K_MAJOR ? wbase + lm + 4 * i : wbase + (i >> 2) * 16 + lm * 4 + (i & 3);
}
template <bool K_MAJOR>
__device__ __forceinline__ int col_of(int wbase, int ln, int j) {
    return K_MAJOR ? wbase + ln + 8 * j : wbase + (j >> 2) * 32 + ln * 4 + (j & 3);
}

// Fragments of one operand for k = k0, k0+1 (k0 even): R values per thread
// per k.  LANES distinct lane indices run along the dimension (4 for A rows, 8
// for B columns).  `lidx` is the lane index, `wbase` the warp's first row.
//
// K-major tiles are [row][32 k] with the 128-byte swizzle: the 16-byte chunk c
// of row r sits at chunk c ^ (r & 7).  A thread's rows wbase + lidx + LANES*i
// fall into at most two swizzle classes (r & 7 = lidx + LANES*(i&1) mod 8), so
// each k-chunk needs one XOR per class and every load is base + immediate.
// PAIRED (K-major pair operand): 4-byte loads of k0 and k0+1 separately, so
// values of neighbouring rows land in one register pair without moves.
// Otherwise K-major uses one 8-byte load per row (k0, k0+1).
// MN-major tiles are [k][TILE_ROWS]: 16-byte loads of 4 adjacent rows.
template <bool K_MAJOR, bool PAIRED, int R, int LANES, int TILE_ROWS>
__device__ __forceinline__ void load_frag2(const float* tile, int k0, int wbase, int lidx,
                                           float (&f)[R][2]) {
    if (K_MAJOR) {
        const char* base = reinterpret_cast<const char*>(tile) + (wbase + lidx) * 128;
        const int c = k0 >> 2;
        const int x0 = lidx & 7, x1 = (lidx + LANES) & 7;
        const char* b0 = base + (((c ^ x0) & 7) << 4) + ((k0 & 3) << 2);
        const char* b1 = base + (((c ^ x1) & 7) << 4) + ((k0 & 3) << 2);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const char* q = ((i & 1) ? b1 : b0) + i * LANES * 128;
            if (PAIRED) {
                f[i][0] = *reinterpret_cast<const float*>(q);
                f[i][1] = *reinterpret_cast<const float*>(q + 4);
            } else {
                const float2 v = *reinterpret_cast<const float2*>(q);
                f[i][0] = v.x;
                f[i][1] = v.y;
            }
        }
    } else {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const float* row = tile + (k0 + kk) * TILE_ROWS + wbase + lidx * 4;
#pragma unroll
            for (int q = 0; q < R / 4; ++q) {
                const float4 v = *reinterpret_cast<const float4*>(row + q * 4 * LANES);
                f[4 * q + 0][kk] = v.x; f[4 * q + 1][kk] = v.y;
                f[4 * q + 2][kk] = v.z; f[4 * q + 3][kk] = v.w;
            }
        }
    }
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
#if SBGEMM_FFMA2
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
#else
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc_at<PAIR_I>(acc, i, j) = fmaf(a[i], b[j], acc_at<PAIR_I>(acc, i, j));
#endif
}

// Copy issuer state (thread 0 only): the next (tile, slice) to load.
struct Issuer {
    int64_t t;          // tile index of the next slice to load
    int kt;             // slice within that tile
    uint64_t issued;    // slices issued so far (global iteration count)
};

template <int BM, int BN, bool A_K, bool B_K>
__device__ __forceinline__ void issue_next(typename Cfg<BM, BN>::Smem& sh, const CUtensorMap* ta,
                                           const CUtensorMap* tb, const Params& p, Issuer& is) {
    using C = Cfg<BM, BN>;
    const TileCoord tc = tile_coord<BM, BN>(p, is.t);
    const int s = (int)(is.issued % C::kStages);
    const int ba = p.a_bcast ? 0 : (int)tc.b;
    const int bb = p.b_bcast ? 0 : (int)tc.b;
    const int k0 = is.kt * BK;
    mbar_arrive_expect_tx(&sh.full[s], C::kStageBytes);
    if (A_K) tma_load_3d(sh.a[s], ta, &sh.full[s], k0, (int)tc.m0, ba);
    else     tma_load_3d(sh.a[s], ta, &sh.full[s], (int)tc.m0, k0, ba);
    if (B_K) tma_load_3d(sh.b[s], tb, &sh.full[s], k0, (int)tc.n0, bb);
    else     tma_load_3d(sh.b[s], tb, &sh.full[s], (int)tc.n0, k0, bb);
    ++is.issued;
    if (++is.kt == p.nk) { is.kt = 0; is.t += gridDim.x; }
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

template <int BM, int BN, bool A_K, bool B_K>
__global__ void __launch_bounds__(kThreads, 1)
tma_ffma_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                const Params p) {
    using C = Cfg<BM, BN>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    auto& sh = *reinterpret_cast<typename C::Smem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const bool issuer = threadIdx.x == 0;
    Issuer is{blockIdx.x, 0, 0};
    if (issuer) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], kWarps);
        }
        fence_mbar_init();
        prefetch_tensormap(&ta);
        prefetch_tensormap(&tb);
    }
    __syncthreads();
    const int64_t my_slices = (p.tiles_total > (int64_t)blockIdx.x)
        ? ((p.tiles_total - 1 - blockIdx.x) / gridDim.x + 1) * p.nk : 0;
    if (issuer) {
        for (int q = 0; q < S - 1 && (int64_t)is.issued < my_slices; ++q)
            issue_next<BM, BN, A_K, B_K>(sh, &ta, &tb, p, is);
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wm = (warp % C::kWarpsM) * WTM, wn = (warp / C::kWarpsM) * WTN;
    const int lm = lane >> 3, ln = lane & 7;
    // Pair along the dimension whose operand arrives with adjacent values:
    // rows when A is MN-major, otherwise columns.
    constexpr bool PI = !A_K;
    uint64_t it = 0;
    for (int64_t t = blockIdx.x; t < p.tiles_total; t += gridDim.x) {
        const TileCoord tc = tile_coord<BM, BN>(p, t);
        float2 acc[64];
#pragma unroll
        for (int q = 0; q < 64; ++q) acc[q] = make_float2(0.0f, 0.0f);

        for (int kt = 0; kt < p.nk; ++kt, ++it) {
            if (issuer && (int64_t)is.issued < my_slices) {
                // Refill the stage every warp released at slice it-1.
                if (is.issued >= (uint64_t)S &&
                    !mbar_wait(&sh.empty[is.issued % S], (uint32_t)(((is.issued / S) - 1) & 1))) {
                    record_status(&g_wait_status, kWaitEmpty);
                    drain<S>(sh.full, it, is.issued);
                    return;
                }
                issue_next<BM, BN, A_K, B_K>(sh, &ta, &tb, p, is);
            }
            const int s = (int)(it % S);
            if (!mbar_wait(&sh.full[s], (uint32_t)((it / S) & 1))) {
                record_status(&g_wait_status, kWaitFull);
                if (issuer) drain<S>(sh.full, it, is.issued);
                return;
            }
            const float* As = sh.a[s];
            const float* Bs = sh.b[s];
            // Unrolling deeper lets ptxas hoist fragment loads until the 128
            // accumulators spill; the warp's second neighbour on the scheduler
            // covers the shared-memory latency instead.
#pragma unroll kUnrollK
            for (int k = 0; k < BK; k += 2) {
                float fa[TM][2], fb[TN][2];
                // The pair operand is B unless A is MN-major (PI).
                load_frag2<A_K, false, TM, 4, BM>(As, k, wm, lm, fa);
                load_frag2<B_K, !PI, TN, 8, BN>(Bs, k, wn, ln, fb);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    float a[TM], b[TN];
#pragma unroll
                    for (int q = 0; q < TM; ++q) a[q] = fa[q][kk];
#pragma unroll
                    for (int q = 0; q < TN; ++q) b[q] = fb[q][kk];
                    fma_step<PI>(acc, a, b);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.empty[s]);
        }

        // Epilogue straight from registers.
        float* Cb = p.C + tc.b * p.bsC;
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int64_t m = tc.m0 + row_of<A_K>(wm, lm, i);
            if (m >= p.M) continue;
            float* crow = Cb + m * p.rsC;
            if (!B_K && p.c_vec4) {
#pragma unroll
                for (int h = 0; h < TN / 4; ++h) {
                    const int64_t n = tc.n0 + col_of<false>(wn, ln, 4 * h);
                    if (n + 3 < p.N) {
                        float4* cp = reinterpret_cast<float4*>(crow + n);
                        float4 v;
                        if (p.accumulate) {
                            const float4 o = *cp;
                            v.x = fmaf(p.alpha, acc_at<PI>(acc, i, 4 * h + 0), o.x);
                            v.y = fmaf(p.alpha, acc_at<PI>(acc, i, 4 * h + 1), o.y);
                            v.z = fmaf(p.alpha, acc_at<PI>(acc, i, 4 * h + 2), o.z);
                            v.w = fmaf(p.alpha, acc_at<PI>(acc, i, 4 * h + 3), o.w);
                        } else {
                            v.x = p.alpha * acc_at<PI>(acc, i, 4 * h + 0);
                            v.y = p.alpha * acc_at<PI>(acc, i, 4 * h + 1);
                            v.z = p.alpha * acc_at<PI>(acc, i, 4 * h + 2);
                            v.w = p.alpha * acc_at<PI>(acc, i, 4 * h + 3);
                        }
                        *cp = v;
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (n + e < p.N) {
                                float* c = crow + (n + e);
                                *c = p.accumulate ? fmaf(p.alpha, acc_at<PI>(acc, i, 4 * h + e), *c)
                                                  : p.alpha * acc_at<PI>(acc, i, 4 * h + e);
                            }
                        }
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < TN; ++j) {
                    const int64_t n = tc.n0 + col_of<B_K>(wn, ln, j);
                    if (n >= p.N) continue;
                    float* c = crow + n * p.csC;
                    *c = p.accumulate ? fmaf(p.alpha, acc_at<PI>(acc, i, j), *c)
                                      : p.alpha * acc_at<PI>(acc, i, j);
                }
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
    using C = Cfg<BM, BN>;
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
                  pr.bsA, pr.batch, a_bc, A_K, BM))
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
    const int64_t grid = plan.tiles < (int64_t)sm_count ? plan.tiles : (int64_t)sm_count;
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

constexpr TmaFfmaConfig kConfigs[] = {
    {256, 128, BK, Cfg<256, 128>::kStages, kThreads},
    {128, 256, BK, Cfg<128, 256>::kStages, kThreads},
};

}  // namespace

int tma_ffma_config_count() { return (int)(sizeof(kConfigs) / sizeof(kConfigs[0])); }

TmaFfmaConfig tma_ffma_config(int variant) { return kConfigs[variant]; }

// Picks the tile shape that wastes the least work, counting both the ragged
// edge of the last tiles and the idle SMs of the last wave.
int tma_ffma_pick_variant(const Problem& p, int sm_count) {
    int best = 0;
    double best_cost = 0.0;
    for (int v = 0; v < tma_ffma_config_count(); ++v) {
        const TmaFfmaConfig c = kConfigs[v];
        const int64_t tm = (p.M + c.bm - 1) / c.bm, tn = (p.N + c.bn - 1) / c.bn;
        const int64_t tiles = tm * tn * p.batch;
        const int64_t waves = (tiles + sm_count - 1) / sm_count;
        const double cost = (double)waves * c.bm * c.bn;   // time ~ waves x tile work
        if (v == 0 || cost < best_cost) { best = v; best_cost = cost; }
    }
    return best;
}

cudaError_t launch_tma_ffma(const Problem& p, const Plan& plan, int sm_count, cudaStream_t stream) {
    switch (plan.variant) {
        case 0: return launch_tile<256, 128>(p, plan, sm_count, stream);
        case 1: return launch_tile<128, 256>(p, plan, sm_count, stream);
        default: return cudaErrorInvalidValue;
    }
}

unsigned int read_and_clear_wait_status_tma_ffma(cudaStream_t stream) {
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

}  // namespace sbg
