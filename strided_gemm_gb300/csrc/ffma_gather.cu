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
// `rs` steps along R, `ks` along K.  RFAST: consecutive threads take
// consecutive R indices (unit stride along R); otherwise consecutive K.
template <int R, int BK, bool RFAST>
struct SliceLoader {
    static constexpr int kPer = R * BK / kThreads;   // elements per thread
    float v[kPer];
    int64_t off0;      // element offset of this thread's first element at k0 = 0
    int64_t step_i;    // offset between this thread's consecutive elements
    int64_t step_k;    // offset step of one BK slice
    int r_first, k_first;

    __device__ __forceinline__ void init(int tid, int64_t r0, int64_t rs, int64_t ks) {
        if (RFAST) {
            r_first = tid % R;
            k_first = tid / R;
            step_i = (int64_t)(kThreads / R) * ks;
        } else {
            k_first = tid % BK;
            r_first = tid / BK;
            step_i = (int64_t)(kThreads / BK) * rs;
        }
        off0 = (r0 + r_first) * rs + (int64_t)k_first * ks;
        step_k = (int64_t)BK * ks;
    }

    // Fetch slice kt (k0 = kt*BK).  rows_left = valid rows from r0, k_left = K - k0.
    // op / span: the operand's base pointer and valid offsets (debug checks).
    __device__ __forceinline__ void load(const float* __restrict__ base, int64_t kt,
                                         int64_t rows_left, int64_t k_left, const float* op,
                                         const ElemSpan& span) {
        const int64_t off = off0 + kt * step_k;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            int r = RFAST ? r_first : r_first + i * (kThreads / BK);
            int k = RFAST ? k_first + i * (kThreads / R) : k_first;
            bool ok = (r < rows_left) && (k < k_left);
            const float* a = base + off + i * step_i;
            v[i] = (ok && dbg_in_span(op, a, span, &g_status)) ? __ldg(a) : 0.0f;
        }
    }

    template <int LD>
    __device__ __forceinline__ void store(float (*S)[LD]) const {
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            int r = RFAST ? r_first : r_first + i * (kThreads / BK);
            int k = RFAST ? k_first + i * (kThreads / R) : k_first;
            S[k][r] = v[i];
        }
    }
};

// SPLIT: the instantiation for K pieces (64 x 64 tiles only), so that the
// others keep their registers.
template <int BM, int BN, int BK, int TM, int TN, bool A_MFAST, bool B_NFAST, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 2)
gather_ffma_kernel(const Problem p, const int64_t tiles_m, const int64_t tiles_n, const Split sp) {
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
        la.init(tid, m0, p.rsA, p.csA);
        lb.init(tid, n0, p.csB, p.rsB);

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
        gather_ffma_kernel<BM, BN, BK, TM, TN, true, true, SPLIT><<<grid, block, 0, stream>>>(p, plan.tiles_m, plan.tiles_n, sp);
    else if (a_fast)
        gather_ffma_kernel<BM, BN, BK, TM, TN, true, false, SPLIT><<<grid, block, 0, stream>>>(p, plan.tiles_m, plan.tiles_n, sp);
    else if (b_fast)
        gather_ffma_kernel<BM, BN, BK, TM, TN, false, true, SPLIT><<<grid, block, 0, stream>>>(p, plan.tiles_m, plan.tiles_n, sp);
    else
        gather_ffma_kernel<BM, BN, BK, TM, TN, false, false, SPLIT><<<grid, block, 0, stream>>>(p, plan.tiles_m, plan.tiles_n, sp);
    return cudaGetLastError();
}

constexpr GatherConfig kConfigs[] = {
    {128, 128, 16, kThreads, 2},   // 8 x 8 micro-tiles
    {64, 64, 16, kThreads, 2},     // 4 x 4 micro-tiles, for small problems
};

}  // namespace

int gather_config_count() { return (int)(sizeof(kConfigs) / sizeof(kConfigs[0])); }

GatherConfig gather_config(int variant) { return kConfigs[variant]; }

int gather_pick_variant(const Problem& p, int sm_count) {
    // Prefer the large tile when it still gives every SM at least one CTA.
    const int64_t big = ((p.M + 127) / 128) * ((p.N + 127) / 128) * p.batch;
    return big >= sm_count ? 0 : 1;
}

void gather_schedule(const Problem& p, Plan& plan, int sm_count, size_t ws_bytes, const void* ws,
                     int k_split) {
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
