// Strided-gather FFMA path: serves every stride pattern (unit, padded, zero,
// negative), so it is the path of last resort and the correctness baseline.
//
// Each CTA owns a BM x BN output tile of one batch entry and walks K in BK-deep
// slices.  The 256 threads load the next A and B slices with scalar loads whose
// thread-to-element map follows each operand's smaller stride (coalesced for a
// unit stride), stage them through registers into double-buffered shared memory
// laid out k-major ([k][m] and [k][n]), and compute TM x TN register micro-tiles
// with one fused multiply-add chain per output in increasing k (register
// blocking as in the StaleyNET "GPU Implementation" page, section "The matrix
// product", with the 4 x 4 block grown to 8 x 8).  The epilogue forms
// fmaf(alpha, acc, C_old) (or alpha*acc) and stores with masks on ragged M / N;
// ragged K is covered by zero-filled loads.
//
// Small products (a few dozen tiles, as a 256 x 512 layer) would leave most
// SMs idle, so with a caller workspace their K range is cut into pieces, one
// CTA per (tile, piece): each piece parks its partial sums, and the CTA that
// finishes a tile last (an atomic count per tile) adds the pieces in piece
// order and runs the epilogue.  Deterministic, but rounded differently from
// one chain, so only under k_split = ANY.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "debug_check.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace sbg {
namespace {

constexpr int kThreads = 256;

// Status word of this kernel's debug bounds checks (sbgemm_device_status).
__device__ unsigned int g_status = 0;
constexpr int kMinPieceSlices = 4;   // K slices (of 16) per piece at least
constexpr int kMaxPieces = 16;

struct Split {
    int pieces;                 // K pieces per tile (grid z); 1 = whole tiles
    float* part;                // [tile][piece][BM * BN] partial sums
    unsigned int* count;        // [tile] pieces finished, zeroed before launch
};

// Loads one operand's R x BK slice (R = rows of the tile: BM for A, BN for B).
// `rs` steps along R, `ks` along K.  RFAST: the thread-to-element map runs
// along R first (the operand's smaller stride is along R); otherwise along K.
// With a unit stride along that fast index and alignment to match (checked
// on the host), each thread fetches `vec` = 2 or 4 consecutive elements with
// one 8- or 16-byte load; a vector that crosses a ragged edge of the tile or
// of K falls back to guarded scalar loads of its elements.
template <int R, int BK, bool RFAST>
struct SliceLoader {
    static constexpr int kPer = R * BK / kThreads;   // elements per thread
    static_assert(kPer % 4 == 0, "whole vectors of 4");
    float v[kPer];
    int vec;           // elements per load: 1, 2 or 4 (vector i holds v[i * vec ..])
    int64_t off0;      // element offset of this thread's first element at k0 = 0
    int64_t step_i;    // offset between this thread's consecutive vectors
    int64_t step_k;    // offset step of one BK slice
    int r_first, k_first;
    int line_step;     // slow-index step between consecutive vectors

    __device__ __forceinline__ void init(int tid, int64_t r0, int64_t rs, int64_t ks, int vec_) {
        vec = vec_;
        const int per_line = (RFAST ? R : BK) / vec;    // threads along the fast index
        const int fast = (tid % per_line) * vec, slow = tid / per_line;
        line_step = kThreads / per_line;
        if (RFAST) {
            r_first = fast;
            k_first = slow;
            step_i = (int64_t)line_step * ks;
        } else {
            k_first = fast;
            r_first = slow;
            step_i = (int64_t)line_step * rs;
        }
        off0 = (r0 + r_first) * rs + (int64_t)k_first * ks;
        step_k = (int64_t)BK * ks;
    }

    template <int V>
    __device__ __forceinline__ void load_v(const float* __restrict__ base, int64_t off, int64_t rows_left,
                                           int64_t k_left, const float* op, const ElemSpan& span) {
#pragma unroll
        for (int i = 0; i < kPer / V; ++i) {
            const int r = RFAST ? r_first : r_first + i * line_step;
            const int k = RFAST ? k_first + i * line_step : k_first;
            const float* a = base + off + i * step_i;
            // The vector's elements run along the fast index, whose stride is
            // 1 when V > 1.
            const bool whole = RFAST ? (r + V - 1 < rows_left && k < k_left)
                                     : (r < rows_left && k + V - 1 < k_left);
            if (V == 4 && whole && dbg_in_span(op, a, span, &g_status) && dbg_in_span(op, a + 3, span, &g_status)) {
                const float4 x = __ldg(reinterpret_cast<const float4*>(a));
                v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
            } else if (V == 2 && whole && dbg_in_span(op, a, span, &g_status) &&
                       dbg_in_span(op, a + 1, span, &g_status)) {
                const float2 x = __ldg(reinterpret_cast<const float2*>(a));
                v[2 * i] = x.x; v[2 * i + 1] = x.y;
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const bool ok = RFAST ? (r + e < rows_left && k < k_left) : (r < rows_left && k + e < k_left);
                    v[V * i + e] = (ok && dbg_in_span(op, a + e, span, &g_status)) ? __ldg(a + e) : 0.0f;
                }
            }
        }
    }

    // Fetch slice kt (k0 = kt*BK).  rows_left = valid rows from r0, k_left = K - k0.
    // op / span: the operand's base pointer and valid offsets (debug checks).
    __device__ __forceinline__ void load(const float* __restrict__ base, int64_t kt,
                                         int64_t rows_left, int64_t k_left, const float* op,
                                         const ElemSpan& span) {
        const int64_t off = off0 + kt * step_k;
        if (vec == 4) load_v<4>(base, off, rows_left, k_left, op, span);
        else if (vec == 2) load_v<2>(base, off, rows_left, k_left, op, span);
        else load_v<1>(base, off, rows_left, k_left, op, span);
    }

    template <int V, int LD>
    __device__ __forceinline__ void store_v(float (*S)[LD]) const {
#pragma unroll
        for (int i = 0; i < kPer / V; ++i) {
            const int r = RFAST ? r_first : r_first + i * line_step;
            const int k = RFAST ? k_first + i * line_step : k_first;
            if (RFAST && V == 4) {
                *reinterpret_cast<float4*>(&S[k][r]) = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            } else if (RFAST && V == 2) {
                *reinterpret_cast<float2*>(&S[k][r]) = make_float2(v[2 * i], v[2 * i + 1]);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    if (RFAST) S[k][r + e] = v[V * i + e];
                    else S[k + e][r] = v[V * i + e];
                }
            }
        }
    }

    template <int LD>
    __device__ __forceinline__ void store(float (*S)[LD]) const {
        if (vec == 4) store_v<4>(S);
        else if (vec == 2) store_v<2>(S);
        else store_v<1>(S);
    }
};

// SPLIT: the instantiation for K pieces (64 x 64 tiles only), so that the
// others keep their registers.
template <int BM, int BN, int BK, int TM, int TN, bool A_MFAST, bool B_NFAST, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 2)
gather_ffma_kernel(const Problem p, const int64_t tiles_m, const int64_t tiles_n, const Split sp,
                   const int va, const int vb) {
    static_assert((BM / TM) * (BN / TN) == kThreads, "thread grid must cover the tile");
    static_assert(TM % 4 == 0 && TN % 4 == 0, "micro-tile is built from float4 rows");
    constexpr int LDA = BM + 4;   // +4 floats keeps float4 alignment of each k-row
    constexpr int LDB = BN + 4;
    __shared__ __align__(16) float As[2][BK][LDA];
    __shared__ __align__(16) float Bs[2][BK][LDB];
    __shared__ unsigned int last_piece;

    const int tid = threadIdx.x;
    const int tx = tid % (BN / TN);
    const int ty = tid / (BN / TN);

    // Grouped raster over (tile_m, tile_n): 8 tile-rows per group so that
    // concurrently running CTAs share A and B slices in L2.
    const int64_t t = blockIdx.x;
    constexpr int64_t kGroup = 8;
    const int64_t group_size = kGroup * tiles_n;
    const int64_t g = t / group_size;
    const int64_t first_m = g * kGroup;
    const int64_t gm = (tiles_m - first_m < kGroup) ? (tiles_m - first_m) : kGroup;
    const int64_t within = t % group_size;
    const int64_t tm = first_m + within % gm;
    const int64_t tn = within / gm;
    const int64_t m0 = tm * BM, n0 = tn * BN;
    const int64_t rows_a = p.M - m0, rows_b = p.N - n0;
    const int64_t nk = (p.K + BK - 1) / BK;
    // This CTA's K slices [kb, ke): all of them, or its piece's share.
    const int piece = SPLIT ? (int)blockIdx.z : 0;
    const int64_t kb = SPLIT ? nk * piece / sp.pieces : 0;
    const int64_t ke = SPLIT ? nk * (piece + 1) / sp.pieces : nk;

    for (int64_t b = blockIdx.y; b < p.batch; b += gridDim.y) {
        const float* __restrict__ Ab = p.A + b * p.bsA;
        const float* __restrict__ Bb = p.B + b * p.bsB;

        SliceLoader<BM, BK, A_MFAST> la;
        SliceLoader<BN, BK, B_NFAST> lb;
        la.init(tid, m0, p.rsA, p.csA, va);
        lb.init(tid, n0, p.csB, p.rsB, vb);

        // Accumulators of adjacent row pairs (i, i+1) of one column, for the
        // packed FMA (fma.rn.f32x2: each lane rounds like fmaf, so every output
        // keeps one k-ordered FMA chain).
        float2 acc2[TM][TN / 2];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN / 2; ++j) acc2[i][j] = make_float2(0.0f, 0.0f);
#define ACC(i, j) (((j) & 1) ? acc2[i][(j) >> 1].y : acc2[i][(j) >> 1].x)

        if (ke > kb) {
            la.load(Ab, kb, rows_a, p.K - kb * BK, p.A, p.sa);
            lb.load(Bb, kb, rows_b, p.K - kb * BK, p.B, p.sb);
            la.template store<LDA>(As[0]);
            lb.template store<LDB>(Bs[0]);
        }
        __syncthreads();

        for (int64_t kt = kb; kt < ke; ++kt) {
            const int buf = (int)((kt - kb) & 1);
            const bool more = kt + 1 < ke;
            if (more) {
                la.load(Ab, kt + 1, rows_a, p.K - (kt + 1) * BK, p.A, p.sa);
                lb.load(Bb, kt + 1, rows_b, p.K - (kt + 1) * BK, p.B, p.sb);
            }
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                float a[TM], bv[TN];
#pragma unroll
                for (int h = 0; h < TM / 4; ++h) {
                    float4 x = *reinterpret_cast<const float4*>(
                        &As[buf][kk][h * (BM / TM) * 4 + ty * 4]);
                    a[4 * h + 0] = x.x; a[4 * h + 1] = x.y; a[4 * h + 2] = x.z; a[4 * h + 3] = x.w;
                }
#pragma unroll
                for (int h = 0; h < TN / 4; ++h) {
                    float4 x = *reinterpret_cast<const float4*>(
                        &Bs[buf][kk][h * (BN / TN) * 4 + tx * 4]);
                    bv[4 * h + 0] = x.x; bv[4 * h + 1] = x.y; bv[4 * h + 2] = x.z; bv[4 * h + 3] = x.w;
                }
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const float2 av = make_float2(a[i], a[i]);
#pragma unroll
                    for (int jp = 0; jp < TN / 2; ++jp)
                        acc2[i][jp] = __ffma2_rn(av, make_float2(bv[2 * jp], bv[2 * jp + 1]), acc2[i][jp]);
                }
            }
            if (more) {
                la.template store<LDA>(As[buf ^ 1]);
                lb.template store<LDB>(Bs[buf ^ 1]);
            }
            __syncthreads();
        }

        if constexpr (SPLIT) {
            // Park this piece; the last piece of the tile to finish sums them
            // all in piece order (a warp's stores and loads are contiguous).
            const int64_t tile_id = b * (tiles_m * tiles_n) + t;
            float* slot = sp.part + (tile_id * sp.pieces + piece) * (int64_t)(BM * BN);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) __stcg(slot + (i * TN + j) * kThreads + tid, ACC(i, j));
            __threadfence();
            __syncthreads();
            if (tid == 0)
                last_piece = atomicAdd(sp.count + tile_id, 1u) == (unsigned int)(sp.pieces - 1);
            __syncthreads();
            if (!last_piece) continue;
            __threadfence();
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) ACC(i, j) = 0.0f;
            const float* first = sp.part + tile_id * sp.pieces * (int64_t)(BM * BN);
#pragma unroll 1
            for (int q = 0; q < sp.pieces; ++q) {
                const float* src = first + q * (int64_t)(BM * BN);
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) ACC(i, j) += __ldcg(src + (i * TN + j) * kThreads + tid);
            }
        }

        // Epilogue: alpha * acc (+ C_old), masked on ragged M / N.
        float* __restrict__ Cb = p.C + b * p.bsC;
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int64_t m = m0 + (i / 4) * (BM / TM) * 4 + ty * 4 + (i % 4);
            if (m >= p.M) continue;
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const int64_t n = n0 + (j / 4) * (BN / TN) * 4 + tx * 4 + (j % 4);
                if (n >= p.N) continue;
                float* c = Cb + m * p.rsC + n * p.csC;
                if (!dbg_in_span(p.C, c, p.sc, &g_status)) continue;
                *c = p.accumulate ? fmaf(p.alpha, ACC(i, j), *c) : p.alpha * ACC(i, j);
            }
        }
        if (p.epi.on) {
            // Fused addend and activation over the thread's own fresh outputs.
#pragma unroll 1
            for (int i = 0; i < TM; ++i) {
                const int64_t m = m0 + (i / 4) * (BM / TM) * 4 + ty * 4 + (i % 4);
                if (m >= p.M) continue;
#pragma unroll 1
                for (int j = 0; j < TN; ++j) {
                    const int64_t n = n0 + (j / 4) * (BN / TN) * 4 + tx * 4 + (j % 4);
                    if (n >= p.N) continue;
                    float* c = Cb + m * p.rsC + n * p.csC;
                    if (!dbg_in_span(p.C, c, p.sc, &g_status)) continue;
                    *c = finish(p.epi, *c, b, m, n, &g_status);
                }
            }
        }
    }
#undef ACC
}

// Products of a few thousand outputs with short K (a 64 x 48 x 32 layer):
// one 64 x 64 tile leaves each of its 256 threads 16 outputs' chains, run by
// 2 warps per scheduler with nothing to hide their latencies (about 10k
// cycles for such a product).  Here each thread computes one output straight
// from global memory (the L1 serves the reuse), so the work spreads over
// many SMs and each thread's chain is one dot product.  A warp covers 32
// consecutive columns of a row, a CTA 8 rows.  The loads of 32 k steps go
// out together before their FMAs; k runs in increasing order in one fmaf
// chain from +0, as in the tiled kernel, so the two agree to the bit.
constexpr int kDirectRows = kThreads / 32, kDirectCols = 32, kDirectChunk = 32;

__global__ void __launch_bounds__(kThreads)
gather_direct_kernel(const Problem p, const int64_t tiles_n) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t tile = blockIdx.x;
    const uint32_t tm = tile / (uint32_t)tiles_n, tn = tile - tm * (uint32_t)tiles_n;
    const int64_t m = (int64_t)tm * kDirectRows + w, n = (int64_t)tn * kDirectCols + lane;
    if (m >= p.M || n >= p.N) return;   // no barrier below
    for (int64_t b = blockIdx.y; b < p.batch; b += gridDim.y) {
        const float* __restrict__ arow = p.A + b * p.bsA + m * p.rsA;
        const float* __restrict__ bcol = p.B + b * p.bsB + n * p.csB;
        float acc = 0.0f;
        for (int64_t k0 = 0; k0 < p.K; k0 += kDirectChunk) {
            float av[kDirectChunk], bv[kDirectChunk];
#pragma unroll
            for (int k = 0; k < kDirectChunk; ++k) {
                const bool in = k0 + k < p.K;
                const float* pa = arow + (k0 + k) * p.csA;
                const float* pb = bcol + (k0 + k) * p.rsB;
                av[k] = (in && dbg_in_span(p.A, pa, p.sa, &g_status)) ? __ldg(pa) : 0.0f;
                bv[k] = (in && dbg_in_span(p.B, pb, p.sb, &g_status)) ? __ldg(pb) : 0.0f;
            }
#pragma unroll
            for (int k = 0; k < kDirectChunk; ++k)
                if (k0 + k < p.K) acc = fmaf(av[k], bv[k], acc);
        }
        float* c = p.C + b * p.bsC + m * p.rsC + n * p.csC;
        if (!dbg_in_span(p.C, c, p.sc, &g_status)) continue;
        float v = p.accumulate ? fmaf(p.alpha, acc, *c) : p.alpha * acc;
        if (p.epi.on) v = finish(p.epi, v, b, m, n, &g_status);
        *c = v;
    }
}

// Tiny products with long K (a 256 x 10 x 512 classifier layer), under
// k_split = ANY with a workspace: one warp per output, its lanes taking k =
// lane, lane + 32, ... in one fmaf chain each, then a butterfly of shuffles
// adds the 32 partial sums (a + b = b + a exactly, so every lane ends with
// the same sum, the same on every run).  The K split rounds differently from
// one chain, like the K pieces; consecutive lanes read consecutive k, so an
// operand with unit stride along K is read in whole lines.  A CTA holds 8
// outputs, consecutive in (batch, row, column) order.
constexpr int kDotWarps = kThreads / 32, kDotUnroll = 8;

__global__ void __launch_bounds__(kThreads)
gather_warpdot_kernel(const Problem p) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t o = blockIdx.x * (uint32_t)kDotWarps + (uint32_t)w;
    const uint32_t mn = (uint32_t)(p.M * p.N);
    if ((int64_t)o >= p.M * p.N * p.batch) return;   // whole warps; no barrier below
    const int64_t b = o / mn, r = o - (uint32_t)b * mn;
    const int64_t m = r / p.N, n = r - m * p.N;
    const float* __restrict__ arow = p.A + b * p.bsA + m * p.rsA;
    const float* __restrict__ bcol = p.B + b * p.bsB + n * p.csB;
    float acc = 0.0f;
    for (int64_t k0 = 0; k0 < p.K; k0 += 32 * kDotUnroll) {
        float av[kDotUnroll], bv[kDotUnroll];
#pragma unroll
        for (int i = 0; i < kDotUnroll; ++i) {
            const int64_t k = k0 + 32 * i + lane;
            const float* pa = arow + k * p.csA;
            const float* pb = bcol + k * p.rsB;
            av[i] = (k < p.K && dbg_in_span(p.A, pa, p.sa, &g_status)) ? __ldg(pa) : 0.0f;
            bv[i] = (k < p.K && dbg_in_span(p.B, pb, p.sb, &g_status)) ? __ldg(pb) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < kDotUnroll; ++i)
            if (k0 + 32 * i + lane < p.K) acc = fmaf(av[i], bv[i], acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane != 0) return;
    float* c = p.C + b * p.bsC + m * p.rsC + n * p.csC;
    if (!dbg_in_span(p.C, c, p.sc, &g_status)) return;
    float v = p.accumulate ? fmaf(p.alpha, acc, *c) : p.alpha * acc;
    if (p.epi.on) v = finish(p.epi, v, b, m, n, &g_status);
    *c = v;
}

// Bytes of the partial sums of `tiles` tiles cut into `pieces`, rounded up to
// 256 so that the counters after them stay aligned.
size_t split_part_bytes(int64_t tiles, int pieces, int tile_elems) {
    const size_t b = (size_t)tiles * (size_t)pieces * (size_t)tile_elems * sizeof(float);
    return (b + 255) / 256 * 256;
}

template <int BM, int BN, int BK, int TM, int TN, bool SPLIT>
cudaError_t launch_variant(const Problem& p, const Plan& plan, cudaStream_t stream) {
    // A: tile rows are M (stride rsA), k stride csA; B: tile rows are N (stride
    // csB), k stride rsB.  Consecutive threads walk whichever index has the
    // smaller stride magnitude (unit stride => coalesced; zero => broadcast).
    auto mag = [](int64_t x) { return x < 0 ? -x : x; };
    const bool a_fast = mag(p.rsA) < mag(p.csA);
    const bool b_fast = mag(p.csB) < mag(p.rsB);
    // Vector width of each operand's loads: the fast index has stride +1 and
    // the base and the other strides keep every vector of `v` elements
    // aligned to 4 v bytes (tile origins and thread offsets along the fast
    // index are multiples of 4).
    auto width = [&](const float* base, int64_t fast, int64_t other, int64_t bs) {
        if (fast != 1) return 1;
        for (int v : {4, 2})
            if (reinterpret_cast<uintptr_t>(base) % (4u * v) == 0 && other % v == 0 &&
                (p.batch == 1 || bs % v == 0))
                return v;
        return 1;
    };
    const int va = width(p.A, a_fast ? p.rsA : p.csA, a_fast ? p.csA : p.rsA, p.bsA);
    const int vb = width(p.B, b_fast ? p.csB : p.rsB, b_fast ? p.rsB : p.csB, p.bsB);
    Split sp{1, nullptr, nullptr};
    if (SPLIT) {
        sp.pieces = plan.k_pieces;
        sp.part = static_cast<float*>(plan.workspace);
        sp.count = reinterpret_cast<unsigned int*>(static_cast<char*>(plan.workspace) +
                                                   split_part_bytes(plan.tiles, plan.k_pieces, BM * BN));
        cudaError_t e = cudaMemsetAsync(sp.count, 0, (size_t)plan.tiles * sizeof(unsigned int), stream);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)(plan.tiles_m * plan.tiles_n),
              (unsigned)(p.batch < 65535 ? p.batch : 65535), (unsigned)sp.pieces);
    dim3 block(kThreads);
    if (a_fast && b_fast)
        gather_ffma_kernel<BM, BN, BK, TM, TN, true, true, SPLIT><<<grid, block, 0, stream>>>(p, plan.tiles_m, plan.tiles_n, sp, va, vb);
    else if (a_fast)
        gather_ffma_kernel<BM, BN, BK, TM, TN, true, false, SPLIT><<<grid, block, 0, stream>>>(p, plan.tiles_m, plan.tiles_n, sp, va, vb);
    else if (b_fast)
        gather_ffma_kernel<BM, BN, BK, TM, TN, false, true, SPLIT><<<grid, block, 0, stream>>>(p, plan.tiles_m, plan.tiles_n, sp, va, vb);
    else
        gather_ffma_kernel<BM, BN, BK, TM, TN, false, false, SPLIT><<<grid, block, 0, stream>>>(p, plan.tiles_m, plan.tiles_n, sp, va, vb);
    return cudaGetLastError();
}

constexpr GatherConfig kConfigs[] = {
    {128, 128, 16, kThreads, 2},   // 8 x 8 micro-tiles
    {64, 64, 16, kThreads, 2},     // 4 x 4 micro-tiles, for small problems
    {128, 64, 16, kThreads, 2},    // 8 x 4 micro-tiles, for narrow or ragged N
    {kDirectRows, kDirectCols, kDirectChunk, kThreads, 8},   // one output per thread
    {1, kDotWarps, 32, kThreads, 8},                          // one output per warp, K over lanes
};
constexpr int kDirectVariant = 3;
constexpr int kWarpDotVariant = 4;
// The direct kernel serves products of at most this many outputs (over the
// batch) and this K.
constexpr int64_t kDirectMaxOutputs = 16384, kDirectMaxK = 128;

}  // namespace

int gather_config_count() { return (int)(sizeof(kConfigs) / sizeof(kConfigs[0])); }

GatherConfig gather_config(int variant) { return kConfigs[variant]; }

int gather_pick_variant(const Problem& p, int sm_count) {
    // Tiny products: one output per thread (gather_direct_kernel).
    if (p.K <= kDirectMaxK && p.M <= kDirectMaxOutputs && p.N <= kDirectMaxOutputs &&
        p.batch <= kDirectMaxOutputs && p.M * p.N * p.batch <= kDirectMaxOutputs)
        return kDirectVariant;
    // The tile shape with the smallest estimated time: waves of CTAs (two
    // per SM) times the tile's work, the smaller tiles charged 4/3 (64 x 64)
    // and 7/6 (128 x 64) for their lower arithmetic per load.  Large tiles
    // win on big products; smaller ones when the large tiles would leave a
    // nearly empty last wave (a 64-clip spectrogram of 125 frames x 514
    // bins: 320 tiles of 128 x 128 on 304 slots, 576 of 128 x 64).
    auto cost = [&](int v, double charge) {
        const GatherConfig g = kConfigs[v];
        const int64_t tiles = ((p.M + g.bm - 1) / g.bm) * ((p.N + g.bn - 1) / g.bn) * p.batch;
        const int64_t slots = (int64_t)sm_count * g.ctas_per_sm;
        return (double)((tiles + slots - 1) / slots) * g.bm * g.bn * charge;
    };
    const double c0 = cost(0, 1.0), c1 = cost(1, 4.0 / 3.0), c2 = cost(2, 7.0 / 6.0);
    return c0 <= c1 && c0 <= c2 ? 0 : (c2 <= c1 ? 2 : 1);
}

void gather_schedule(const Problem& p, Plan& plan, int sm_count, size_t ws_bytes, const void* ws,
                     int k_split) {
    // Tiny products whose K is too long for one thread's chain: with the
    // caller's consent to split K, one warp per output.
    if (ws && k_split == SBGEMM_KSPLIT_ANY && p.K > kDirectMaxK && p.M <= kDirectMaxOutputs &&
        p.N <= kDirectMaxOutputs && p.batch <= kDirectMaxOutputs &&
        p.M * p.N * p.batch <= kDirectMaxOutputs) {
        const GatherConfig d = kConfigs[kWarpDotVariant];
        const int64_t outputs = p.M * p.N * p.batch;
        plan.variant = kWarpDotVariant;
        plan.tile_m = d.bm;
        plan.tile_n = d.bn;
        plan.tile_k = d.bk;
        plan.ctas_per_sm = d.ctas_per_sm;
        plan.tiles = (outputs + kDotWarps - 1) / kDotWarps;
        plan.tiles_m = plan.tiles;
        plan.tiles_n = 1;
        plan.ctas = plan.tiles;
        plan.k_slices = (int)((p.K + 31) / 32);
        plan.k_pieces = 32;
        plan.stream_k = true;      // reported as K pieces; no workspace is used
        plan.split_indep = true;
        plan.dp_tiles = 0;
        plan.workspace = nullptr;
        return;
    }
    const GatherConfig g = kConfigs[plan.variant];
    const int64_t nk = (p.K + g.bk - 1) / g.bk;
    plan.k_slices = (int)nk;
    plan.k_pieces = 1;
    // Only the 64 x 64 tiles of small products are cut.
    if (plan.variant != 1 || !ws || k_split != SBGEMM_KSPLIT_ANY || p.batch > 65535) return;
    if ((reinterpret_cast<uintptr_t>(ws) % 256) != 0) return;
    // Only when the tiles would fill less than half of the CTA slots; then
    // enough pieces to fill them about once, each at least 4 slices.
    const int64_t slots = (int64_t)sm_count * g.ctas_per_sm;
    if (plan.tiles * 2 > slots) return;
    int64_t pieces = (slots + plan.tiles - 1) / plan.tiles;
    pieces = std::min<int64_t>(pieces, nk / kMinPieceSlices);
    pieces = std::min<int64_t>(pieces, kMaxPieces);
    if (pieces < 2) return;
    const size_t need = split_part_bytes(plan.tiles, (int)pieces, g.bm * g.bn) +
                        (size_t)plan.tiles * sizeof(unsigned int);
    if (need > ws_bytes) return;
    plan.k_pieces = (int)pieces;
    plan.stream_k = true;
    plan.split_indep = true;
    plan.dp_tiles = 0;
    plan.ctas = plan.tiles * pieces;
    plan.workspace = const_cast<void*>(ws);
}

cudaError_t launch_gather_ffma(const Problem& p, const Plan& plan, cudaStream_t stream) {
    switch (plan.variant) {
        case 0: return launch_variant<128, 128, 16, 8, 8, false>(p, plan, stream);
        case 1:
            if (plan.k_pieces > 1) return launch_variant<64, 64, 16, 4, 4, true>(p, plan, stream);
            return launch_variant<64, 64, 16, 4, 4, false>(p, plan, stream);
        case 2: return launch_variant<128, 64, 16, 8, 4, false>(p, plan, stream);
        case kWarpDotVariant:
            gather_warpdot_kernel<<<(unsigned)plan.ctas, kThreads, 0, stream>>>(p);
            return cudaGetLastError();
        case kDirectVariant: {
            dim3 grid((unsigned)(plan.tiles_m * plan.tiles_n), (unsigned)(p.batch < 65535 ? p.batch : 65535));
            gather_direct_kernel<<<grid, kThreads, 0, stream>>>(p, plan.tiles_n);
            return cudaGetLastError();
        }
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sbg

namespace sbg {

unsigned int read_and_clear_status_gather(cudaStream_t stream) {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return v;
}

}  // namespace sbg
