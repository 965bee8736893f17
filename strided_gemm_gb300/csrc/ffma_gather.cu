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
#include <cuda_runtime.h>

#include <cstdint>

#include "epilogue.cuh"
#include "internal.h"

namespace sbg {
namespace {

constexpr int kThreads = 256;

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
    __device__ __forceinline__ void load(const float* __restrict__ base, int64_t kt,
                                         int64_t rows_left, int64_t k_left) {
        const int64_t off = off0 + kt * step_k;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            int r = RFAST ? r_first : r_first + i * (kThreads / BK);
            int k = RFAST ? k_first + i * (kThreads / R) : k_first;
            bool ok = (r < rows_left) && (k < k_left);
            v[i] = ok ? __ldg(base + off + i * step_i) : 0.0f;
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

template <int BM, int BN, int BK, int TM, int TN, bool A_MFAST, bool B_NFAST>
__global__ void __launch_bounds__(kThreads, 2)
gather_ffma_kernel(const Problem p, const int64_t tiles_m, const int64_t tiles_n) {
    static_assert((BM / TM) * (BN / TN) == kThreads, "thread grid must cover the tile");
    static_assert(TM % 4 == 0 && TN % 4 == 0, "micro-tile is built from float4 rows");
    constexpr int LDA = BM + 4;   // +4 floats keeps float4 alignment of each k-row
    constexpr int LDB = BN + 4;
    __shared__ __align__(16) float As[2][BK][LDA];
    __shared__ __align__(16) float Bs[2][BK][LDB];

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

    for (int64_t b = blockIdx.y; b < p.batch; b += gridDim.y) {
        const float* __restrict__ Ab = p.A + b * p.bsA;
        const float* __restrict__ Bb = p.B + b * p.bsB;

        SliceLoader<BM, BK, A_MFAST> la;
        SliceLoader<BN, BK, B_NFAST> lb;
        la.init(tid, m0, p.rsA, p.csA);
        lb.init(tid, n0, p.csB, p.rsB);

        float acc[TM][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

        if (nk > 0) {
            la.load(Ab, 0, rows_a, p.K);
            lb.load(Bb, 0, rows_b, p.K);
            la.template store<LDA>(As[0]);
            lb.template store<LDB>(Bs[0]);
        }
        __syncthreads();

        for (int64_t kt = 0; kt < nk; ++kt) {
            const int buf = (int)(kt & 1);
            const bool more = kt + 1 < nk;
            if (more) {
                la.load(Ab, kt + 1, rows_a, p.K - (kt + 1) * BK);
                lb.load(Bb, kt + 1, rows_b, p.K - (kt + 1) * BK);
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
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
            }
            if (more) {
                la.template store<LDA>(As[buf ^ 1]);
                lb.template store<LDB>(Bs[buf ^ 1]);
            }
            __syncthreads();
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
                *c = p.accumulate ? fmaf(p.alpha, acc[i][j], *c) : p.alpha * acc[i][j];
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
                    *c = finish(p.epi, *c, b, m, n);
                }
            }
        }
    }
}

template <int BM, int BN, int BK, int TM, int TN>
cudaError_t launch_variant(const Problem& p, const Plan& plan, cudaStream_t stream) {
    // A: tile rows are M (stride rsA), k stride csA; B: tile rows are N (stride
    // csB), k stride rsB.  Consecutive threads walk whichever index has the
    // smaller stride magnitude (unit stride => coalesced; zero => broadcast).
    auto mag = [](int64_t x) { return x < 0 ? -x : x; };
    const bool a_fast = mag(p.rsA) < mag(p.csA);
    const bool b_fast = mag(p.csB) < mag(p.rsB);
    dim3 grid((unsigned)(plan.tiles_m * plan.tiles_n),
              (unsigned)(p.batch < 65535 ? p.batch : 65535));
    dim3 block(kThreads);
    if (a_fast && b_fast)
        gather_ffma_kernel<BM, BN, BK, TM, TN, true, true><<<grid, block, 0, stream>>>(p, plan.tiles_m, plan.tiles_n);
    else if (a_fast)
        gather_ffma_kernel<BM, BN, BK, TM, TN, true, false><<<grid, block, 0, stream>>>(p, plan.tiles_m, plan.tiles_n);
    else if (b_fast)
        gather_ffma_kernel<BM, BN, BK, TM, TN, false, true><<<grid, block, 0, stream>>>(p, plan.tiles_m, plan.tiles_n);
    else
        gather_ffma_kernel<BM, BN, BK, TM, TN, false, false><<<grid, block, 0, stream>>>(p, plan.tiles_m, plan.tiles_n);
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

cudaError_t launch_gather_ffma(const Problem& p, const Plan& plan, cudaStream_t stream) {
    switch (plan.variant) {
        case 0: return launch_variant<128, 128, 16, 8, 8>(p, plan, stream);
        case 1: return launch_variant<64, 64, 16, 4, 4>(p, plan, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sbg
