// Fused attention on the tensor cores (opt-in TF32): O = softmax(alpha Q K^T
// [causal]) V per (sequence, head), the scores and probabilities kept on the
// chip, as the FP32 kernel in attention.cu computes it ("rvllm CUDA path",
// section "What's basic about it": three steps with the scores in global
// memory, which a fused kernel avoids).
//
// One CTA per 256 query rows of one batch entry: two tiles of 128 rows (the
// MMA's M) that share every K and V block, head dimension 64, keys in blocks
// of 128.  Per block j and tile t:
//   S_tj = Q_t K_j^T   tcgen05.mma kind::tf32, M 128 x N 128 x K 64, into TMEM
//   P_tj = exp2(alpha log2(e) S_tj - m_t)   one thread per query row, in one
//          pass over the row's 128 scores (tcgen05.ld, two 64-column
//          chunks), written back over S_tj (tcgen05.st); the row sum l_t in
//          registers
//   O_t += P_tj V_j   M 128 x N 64 x K 128, A = P_tj from TMEM, accumulated in
//          TMEM by the MMA
// and O_t / l_t is stored at the end.  The reference maximum m_t of a row is
// set from its first kept chunk and raised only when a chunk's exponent
// argument exceeds 8 (a factor of 2^8): then what the row has summed and
// written (l_t, the block's earlier P, O_t in TMEM) is scaled by exp2(m_old -
// m_new) by the row's own thread.  Between raises the exponentials stay below
// 2^8, and O / l is the same function either way.
//
// Q_t lands by TMA in the V^T buffers (not yet in use) and the row threads
// copy it into TMEM, the A operand of the score MMAs, so that shared memory
// holds two V^T buffers: the transpose of block j+1 then overlaps the P V
// MMAs of block j instead of waiting for them.
//
// The MMA lane issues, per block: P V_0, then (once P V_0 has read P_0) the
// scores of tile 0's next block, then the same for tile 1.  So each tile's
// softmax runs while the tensor cores work on the other tile, and since the
// next scores of a tile are issued only after its P V, they also tell its
// softmax that O_t is settled.  Measured on this GPU, a tcgen05.mma issue
// blocks until the one before it is nearly done, and a branch or wait between
// two MMAs costs the tensor pipe as much as an N = 64 MMA: hence 128-key
// blocks (N = 128 score MMAs, half the instructions per key of N = 64, and
// each lane's waits and commits spread over twice the keys) and straight-line
// MMA sequences with every operand one add away.
// Roles (12 warps), all waits bounded (a timeout records a status code and
// the role leaves its loop):
//   warp 0       TMA: both Q tiles once (into the V^T buffers); K_j (two
//                128-byte swizzled boxes of
//                32 along the head dimension) and V_j (eight raw 32 x 32
//                boxes) into a 2-stage ring;
//   warp 1       one lane issues the MMAs;
//   warps 2-3    rewrite V_j (rows along the keys) into V_j^T with rows along
//                the values, the K-major layout P V's B operand takes (4 x 4
//                quads, conflict-free under the swizzle);
//   warps 4-7    softmax of tile 0, one TMEM lane quarter each;
//   warps 8-11   softmax of tile 1.
// TMEM: S / P (2 tiles x 128 columns), O (2 x 64) and Q (2 x 64).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "attention_tc.h"
#include "ptx.cuh"

namespace sbg {
namespace {

constexpr int kD = 64;               // head dimension of Q, K and V
constexpr int kAtom = 32;            // fp32 values in one 128-byte swizzled row
constexpr int kDA = kD / kAtom;      // atoms along the head dimension
constexpr int BM = 128;              // query rows per tile (the MMA's M)
constexpr int kTiles = 2;            // query tiles per CTA, sharing each K and V block
constexpr int BN = 128;              // keys per block
constexpr int kKA = BN / kAtom;      // key atoms per block
constexpr int kMmaK = 8;             // tf32 elements per MMA
constexpr int kStages = 2;           // K and raw V blocks in flight
constexpr int kSoftWarps = 4;        // per tile: one TMEM lane quarter each
constexpr int kTransWarps = 2;
constexpr int kWarpSoft = 4;         // first softmax warp
constexpr int kWarps = kWarpSoft + kTiles * kSoftWarps;
constexpr int kThreads = kWarps * 32;
constexpr int kBox = 32 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                         // S / P [t] at t * BN
constexpr uint32_t kColO = kTiles * BN;               // O[t] at kColO + t * kD
constexpr uint32_t kColQ = kColO + kTiles * kD;       // Q[t] at kColQ + t * kD
static_assert(kColQ + kTiles * kD <= kTmemCols, "TMEM columns");
static_assert((kWarpSoft % 4) == 0 && kSoftWarps == 4, "each tile's softmax warps cover the four lane quarters");
static_assert(kTiles == 2, "the softmax warps pick their tile's block count from two");
static_assert(kD % 32 == 0 && BN == 128, "32-column TMEM transfers; 128-key blocks in two 64-column halves");
constexpr float kRaise = 8.0f;       // log2 headroom before the reference maximum is raised

// max(a, b, c) in one instruction (the three-input form of max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Instruction descriptors, kind::tf32: D fp32, A and B tf32 K-major, M 128;
// N = BN for the scores, kD for P V.
constexpr uint32_t idesc(int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}
constexpr uint32_t kIdescS = idesc(BN), kIdescPV = idesc(kD);

struct Smem {
    alignas(1024) float k[kStages][kDA][BN * kAtom];      // K_j, K-major, head-dim atoms
    alignas(1024) float vraw[kStages][kKA * kDA][kBox];   // V_j: box (key atom h, value atom g) at h kDA + g
    // V_j^T in buffer j % 2: rows along the values, key atoms.  Before the
    // first transpose, the Q tiles as TMA lands them ([tile][atom][row * 32]).
    alignas(1024) float vt[2][kKA][kD * kAtom];
    uint64_t q_full;
    uint64_t q_tmem;              // every row thread has copied its Q row into TMEM
    uint64_t k_full[kStages], k_empty[kStages];
    uint64_t v_full[kStages], v_empty[kStages];
    uint64_t vt_full[2], vt_empty[2];
    uint64_t s_full[kTiles];      // a tile's scores of the current block are in TMEM
    uint64_t p_full[kTiles];      // a tile's P of the current block is in TMEM
    uint64_t pv_done[kTiles];     // a tile's P V has read P and added into O
    uint64_t o_done[kTiles];      // a tile's last P V is done
    uint64_t mma_done;
    uint32_t tmem_base;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(sizeof(Smem::vt) == (size_t)kTiles * kDA * BM * kAtom * 4, "the Q tiles fill the V^T buffers");
static_assert(sizeof(Smem::k[0]) == (size_t)kDA * BM * kAtom * 4, "a K stage holds one tile of O");

// The landing place of Q tile t, atom a (in the V^T buffers).
__device__ __forceinline__ float* q_stage(Smem& sh, int t, int a) {
    return &sh.vt[0][0][0] + (size_t)(t * kDA + a) * BM * kAtom;
}

__device__ unsigned int g_wait_status = 0;

struct Params {
    float* O;
    int64_t rsO, csO, bsO;
    int64_t M, N;
    float scale_log2;                // alpha * log2(e)
    int causal;
    int64_t q_len;
    int bq, bk, bv;                  // batch coordinate follows blockIdx.x (else 0: broadcast)
    int o_vec;                       // O rows unit-stride and 16-byte aligned
    int o_tma;                       // O goes out through its tensor map
    int bo;                          // O's batch coordinate follows blockIdx.x
};

// Keys [0, n_end) a tile of rows starting at m0 needs: all of them, or
// (causal) those up to its rows' last position.  0 when the tile holds no row.
__device__ __forceinline__ int tile_blocks(const Params& p, int64_t m0) {
    if (m0 >= p.M) return 0;
    int64_t n_end = p.N;
    if (p.causal) {
        const int64_t m_last = (m0 + BM - 1 < p.M ? m0 + BM - 1 : p.M - 1);
        const int64_t r0 = m0 % p.q_len;
        const bool wraps = r0 + (m_last - m0) >= p.q_len;
        n_end = (wraps ? p.N - 1 : (m_last % p.q_len) + p.N - p.q_len) + 1;
    }
    return (int)((n_end + BN - 1) / BN);
}

// Rewrites one key atom of V_j: kDA raw boxes (32 keys x 32 values each) into
// V_j^T rows 0..kD-1 (values) x 32 keys, K-major 128-byte swizzle.  A
// quarter-warp's quads hit 8 distinct 16-byte chunks on both the loads and
// the stores.
__device__ __forceinline__ void transpose_atom(const float* raw, float* dst, int t) {
    constexpr int kQuads = kD / 4 * (kAtom / 4);
#pragma unroll
    for (int q = t; q < kQuads; q += kTransWarps * 32) {
        const int kq = ((q >> 2) & 1) | (((q ^ (q >> 1) ^ (q >> 3)) & 1) << 1) | (((q >> 4) & 1) << 2);
        const int mq = (q & 3) | ((q >> 5) << 2);    // 4-row group of values
        const float* box = raw + (mq >> 3) * kBox;
        const int mc = mq & 7;
        float4 v[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int k = 4 * kq + r;
            v[r] = *reinterpret_cast<const float4*>(box + k * 32 + ((mc ^ (k & 7)) << 2));
        }
        const int m = 4 * mq;
        *reinterpret_cast<float4*>(dst + (m + 0) * 32 + ((kq ^ ((m + 0) & 7)) << 2)) =
            make_float4(v[0].x, v[1].x, v[2].x, v[3].x);
        *reinterpret_cast<float4*>(dst + (m + 1) * 32 + ((kq ^ ((m + 1) & 7)) << 2)) =
            make_float4(v[0].y, v[1].y, v[2].y, v[3].y);
        *reinterpret_cast<float4*>(dst + (m + 2) * 32 + ((kq ^ ((m + 2) & 7)) << 2)) =
            make_float4(v[0].z, v[1].z, v[2].z, v[3].z);
        *reinterpret_cast<float4*>(dst + (m + 3) * 32 + ((kq ^ ((m + 3) & 7)) << 2)) =
            make_float4(v[0].w, v[1].w, v[2].w, v[3].w);
    }
}

// The scores of one tile: D = Q_t K_j^T, A (Q_t) in TMEM from column a, B
// (K_j) in 32-wide K-major swizzled atoms of BN rows (descriptor low word
// b_lo); kD / 8 MMAs in straight-line code.
__device__ __forceinline__ void mma_scores(uint32_t d, uint32_t a, uint32_t b_lo) {
    constexpr uint32_t kBAtom = (uint32_t)(BN * kAtom * 4) >> 4;   // next atom, in descriptor units
    constexpr int kSteps = kD / kMmaK;
    uint64_t bd[kSteps];
#pragma unroll
    for (int kk = 0; kk < kSteps; ++kk)
        bd[kk] = ((uint64_t)kDescHiSw128 << 32) | (b_lo + (uint32_t)(kk / 4) * kBAtom + (uint32_t)(kk & 3) * 2);
#pragma unroll
    for (int kk = 0; kk < kSteps; ++kk)
        mma_tf32_ts_desc(d, a + (uint32_t)(kk * kMmaK), bd[kk], kIdescS, kk > 0 ? 1u : 0u);
}

// P V of one tile: O (+)= P_t V_j, A (P_t) in TMEM from column a, B (V_j^T) in
// 32-wide K-major swizzled key atoms of kD rows (descriptor low word b_lo);
// BN / 8 MMAs in straight-line code.  en0: the first adds to O.
__device__ __forceinline__ void mma_pv(uint32_t d, uint32_t a, uint32_t b_lo, uint32_t en0) {
    constexpr uint32_t kBAtom = (uint32_t)(kD * kAtom * 4) >> 4;
    constexpr int kSteps = BN / kMmaK;
    uint64_t bd[kSteps];
#pragma unroll
    for (int kk = 0; kk < kSteps; ++kk)
        bd[kk] = ((uint64_t)kDescHiSw128 << 32) | (b_lo + (uint32_t)(kk / 4) * kBAtom + (uint32_t)(kk & 3) * 2);
#pragma unroll
    for (int kk = 0; kk < kSteps; ++kk)
        mma_tf32_ts_desc(d, a + (uint32_t)(kk * kMmaK), bd[kk], kIdescPV, kk > 0 ? 1u : en0);
}

__global__ void __launch_bounds__(kThreads, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                    const Params p) {
    extern __shared__ uint8_t smem_raw[];
    Smem& sh = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                        ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t b = blockIdx.x;
    const int64_t mb = p.causal ? (int64_t)gridDim.y - 1 - blockIdx.y : (int64_t)blockIdx.y;
    const int64_t m0 = mb * (kTiles * BM);
    int nb_t[kTiles];
    int nblk = 0;
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
        nb_t[t] = tile_blocks(p, m0 + t * BM);
        nblk = nb_t[t] > nblk ? nb_t[t] : nblk;
    }

    if (threadIdx.x == 0) {
        mbar_init(&sh.q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sh.k_full[s], 1);
            mbar_init(&sh.k_empty[s], 1);
            mbar_init(&sh.v_full[s], 1);
            mbar_init(&sh.v_empty[s], kTransWarps);
        }
        mbar_init(&sh.q_tmem, kTiles * kSoftWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.vt_full[i], kTransWarps);
            mbar_init(&sh.vt_empty[i], 1);
        }
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(&sh.s_full[t], 1);
            mbar_init(&sh.p_full[t], kSoftWarps);
            mbar_init(&sh.pv_done[t], 1);
            mbar_init(&sh.o_done[t], 1);
        }
        mbar_init(&sh.mma_done, 1);
        fence_mbar_init();
        prefetch_tensormap(&tq);
        prefetch_tensormap(&tk);
        prefetch_tensormap(&tv);
        if (p.o_tma) prefetch_tensormap(&to);
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        // ---- TMA producer -------------------------------------------------
        if (lane == 0) {
            const int zq = p.bq ? (int)b : 0, zk = p.bk ? (int)b : 0, zv = p.bv ? (int)b : 0;
            int tiles_in = 0;
#pragma unroll
            for (int t = 0; t < kTiles; ++t) tiles_in += nb_t[t] > 0 ? 1 : 0;
            mbar_arrive_expect_tx(&sh.q_full, (uint32_t)tiles_in * kDA * BM * kAtom * 4);
#pragma unroll
            for (int t = 0; t < kTiles; ++t) {
                if (nb_t[t] == 0) continue;
#pragma unroll
                for (int a = 0; a < kDA; ++a)
                    tma_load_3d(q_stage(sh, t, a), &tq, &sh.q_full, kAtom * a, (int)(m0 + t * BM), zq);
            }
            int j = 0;
            for (; j < nblk; ++j) {
                const int s = j % kStages;
                const uint32_t ph = (uint32_t)(((j / kStages) - 1) & 1);
                if (j >= kStages && (!mbar_wait(&sh.k_empty[s], ph) || !mbar_wait(&sh.v_empty[s], ph))) {
                    record_status(&g_wait_status, kWaitEmpty);
                    break;
                }
                const int n0 = j * BN;
                mbar_arrive_expect_tx(&sh.k_full[s], kDA * BN * kAtom * 4);
#pragma unroll
                for (int a = 0; a < kDA; ++a) tma_load_3d(sh.k[s][a], &tk, &sh.k_full[s], kAtom * a, n0, zk);
                mbar_arrive_expect_tx(&sh.v_full[s], kKA * kDA * kBox * 4);
#pragma unroll
                for (int h = 0; h < kKA; ++h)
#pragma unroll
                    for (int g = 0; g < kDA; ++g)
                        tma_load_3d(sh.vraw[s][h * kDA + g], &tv, &sh.v_full[s], 32 * g, n0 + 32 * h, zv);
            }
            // Wait for the copies still landing before the CTA may exit.
            for (int q = j > kStages ? j - kStages : 0; q < j; ++q) {
                const uint32_t ph = (uint32_t)((q / kStages) & 1);
                if (!mbar_wait(&sh.k_full[q % kStages], ph) || !mbar_wait(&sh.v_full[q % kStages], ph)) {
                    record_status(&g_wait_status, kWaitDrain);
                    break;
                }
            }
            if (!mbar_wait(&sh.q_full, 0)) record_status(&g_wait_status, kWaitDrain);
        }
    } else if (warp == 1) {
        // ---- MMA issuer ---------------------------------------------------
        if (lane == 0) {
            // Q in TMEM (every row thread's copy), which also frees the
            // V^T buffers for the transposer.
            bool ok = mbar_wait(&sh.q_tmem, 0);
            // Descriptor low words of every shared-memory operand: stage and
            // buffer offsets are whole multiples of 16 bytes.
            const uint32_t k_lo0 = desc_lo_sw128(smem_u32(sh.k[0][0]));
            constexpr uint32_t kKStage = (uint32_t)sizeof(sh.k[0]) >> 4;
            const uint32_t vt_lo0 = desc_lo_sw128(smem_u32(sh.vt[0][0]));
            constexpr uint32_t kVtBuf = (uint32_t)sizeof(sh.vt[0]) >> 4;
            // The scores of block j for tile t, once P V_t of block j-1 has
            // read P_t (the same TMEM columns).  K_j is released after the
            // last tile's scores.
            auto scores = [&](int t, int j) -> bool {
                if (j >= nb_t[t]) return true;
                if (j > 0 && !mbar_wait(&sh.pv_done[t], (uint32_t)((j - 1) & 1))) return false;
                tc_fence_after();
                mma_scores(tmem + kColS + (uint32_t)t * BN, tmem + kColQ + (uint32_t)t * kD,
                           k_lo0 + (uint32_t)(j % kStages) * kKStage);
                mma_commit(&sh.s_full[t]);
                return true;
            };
            auto release_k = [&](int j) { mma_commit(&sh.k_empty[j % kStages]); };
            if (ok && nblk > 0) {
                ok = mbar_wait(&sh.k_full[0], 0) && scores(0, 0) && scores(1, 0);
                release_k(0);
            }
            for (int j = 0; j < nblk && ok; ++j) {
                if (!mbar_wait(&sh.vt_full[j & 1], (uint32_t)((j >> 1) & 1))) { ok = false; break; }
                const bool next = j + 1 < nblk;
                if (next && !mbar_wait(&sh.k_full[(j + 1) % kStages], (uint32_t)(((j + 1) / kStages) & 1))) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int t = 0; t < kTiles; ++t) {
                    if (j < nb_t[t]) {
                        if (!mbar_wait(&sh.p_full[t], (uint32_t)(j & 1))) { ok = false; break; }
                        tc_fence_after();
                        mma_pv(tmem + kColO + (uint32_t)t * kD, tmem + kColS + (uint32_t)t * BN,
                               vt_lo0 + (uint32_t)(j & 1) * kVtBuf, j > 0 ? 1u : 0u);
                        mma_commit(&sh.pv_done[t]);
                        if (j == nb_t[t] - 1) mma_commit(&sh.o_done[t]);
                    }
                    if (t == kTiles - 1) mma_commit(&sh.vt_empty[j & 1]);   // after every P V of block j
                    if (next && !scores(t, j + 1)) { ok = false; break; }
                }
                if (!ok) break;
                if (next) release_k(j + 1);
            }
            if (!ok) record_status(&g_wait_status, kWaitFull);
            // Nothing may still be writing TMEM when it is freed.
            mma_commit(&sh.mma_done);
            if (!mbar_wait(&sh.mma_done, 0)) record_status(&g_wait_status, kWaitMma);
        }
    } else if (warp < kWarpSoft) {
        // ---- V_j -> V_j^T -------------------------------------------------
        const int t = threadIdx.x - 2 * 32;
        // The V^T buffers hold Q until the row threads have copied it.
        const bool q_out = nblk == 0 || mbar_wait(&sh.q_tmem, 0);
        if (!q_out) record_status(&g_wait_status, kWaitFull);
        for (int j = 0; q_out && j < nblk; ++j) {
            const int s = j % kStages, buf = j & 1;
            if (!mbar_wait(&sh.v_full[s], (uint32_t)((j / kStages) & 1))) {
                record_status(&g_wait_status, kWaitFull);
                break;
            }
            if (j >= 2 && !mbar_wait(&sh.vt_empty[buf], (uint32_t)(((j >> 1) - 1) & 1))) {
                record_status(&g_wait_status, kWaitEmpty);
                break;
            }
#pragma unroll
            for (int h = 0; h < kKA; ++h) transpose_atom(sh.vraw[s][h * kDA], sh.vt[buf][h], t);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sh.vt_full[buf]);
                mbar_arrive(&sh.v_empty[s]);
            }
        }
    } else {
        // ---- softmax and output, one query row per thread ------------------
        const int t = (warp - kWarpSoft) / kSoftWarps;   // query tile
        const int quarter = warp & 3;                    // TMEM lanes this warp may read
        const int row = quarter * 32 + lane;
        const int64_t m = m0 + t * BM + row;
        const int nbt = t == 0 ? nb_t[0] : nb_t[kTiles - 1];
        const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
        const uint32_t o_addr = tmem + lanes + kColO + (uint32_t)t * kD;
        const uint32_t s_addr = tmem + lanes + kColS + (uint32_t)t * BN;
        const int64_t pos = p.causal ? (m % p.q_len) + p.N - p.q_len : p.N - 1;
        const int64_t last_key = pos < p.N - 1 ? pos : p.N - 1;
        const float scale = p.scale_log2;
        float m_ref = -INFINITY, l_run = 0.0f;
        bool ok = nblk > 0;
        // The row's Q into TMEM (lane = row, one column per head-dim element).
        // Every row thread arrives, including those of a tile with no rows.
        if (ok) {
            ok = mbar_wait(&sh.q_full, 0);
            if (ok && nbt > 0) {
#pragma unroll
                for (int a = 0; a < kDA; ++a) {
                    const float* src = q_stage(sh, t, a);
                    float v[32];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 x = *reinterpret_cast<const float4*>(src + row * kAtom + ((c ^ (row & 7)) << 2));
                        v[4 * c] = x.x; v[4 * c + 1] = x.y; v[4 * c + 2] = x.z; v[4 * c + 3] = x.w;
                    }
                    tmem_st32_nowait(tmem + lanes + kColQ + (uint32_t)(t * kD + a * 32), v);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.q_tmem);
        }
        ok = ok && nbt > 0;
        for (int j = 0; ok && j < nbt; ++j) {
            // The scores of block j were issued after P V of block j-1, so
            // their barrier also tells that O is settled.
            if (!mbar_wait(&sh.s_full[t], (uint32_t)(j & 1))) { ok = false; break; }
            tc_fence_after();
            // Keys c <= lim of the block are kept (keys past N, or past the
            // row's causal position, are not).
            const int64_t last = last_key - (int64_t)j * BN;
            const int lim = last < 0 ? -1 : (last >= BN ? BN - 1 : (int)last);
            const bool whole = __all_sync(0xffffffffu, lim == BN - 1);
            // One pass over the block in two 64-column chunks: exponent
            // arguments against the row's reference maximum m_ref, their
            // largest value checked against the headroom.  Only a row's first
            // kept chunk needs its maximum first (m_ref is then -inf).
            float corr_blk = 1.0f;      // this block's scaling of O (raises)
            float psum[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) psum[i] = 0.0f;
#pragma unroll
            for (int hh = 0; hh < BN / 64; ++hh) {
                float s[64];
                tmem_ld64(s_addr + 64 * hh, s);
                if (__any_sync(0xffffffffu, m_ref == -INFINITY)) {
                    if (m_ref == -INFINITY) {
                        // The chunk's largest scaled score (-inf if every key
                        // of the chunk is masked).
                        float mx[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            if (whole || 64 * hh + c <= lim) mx[c & 7] = fmaxf(mx[c & 7], s[c] * scale);
                        m_ref = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                      fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                    }
                }
                const float neg = -m_ref;
                float am[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) am[i] = -INFINITY;
                if (whole) {
                    // In pairs on the FMA pipe (each lane rounds as fmaf), the
                    // running maxima three operands at a time: the softmax is
                    // bound by instruction issue (moving a share of its exp2
                    // to the FMA pipe made it slower), not by the MUFU.
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), make_float2(scale, scale),
                                                    make_float2(neg, neg));
                        s[c] = x.x;
                        s[c + 1] = x.y;
                        am[(c / 2) & 7] = fmax3(am[(c / 2) & 7], x.x, x.y);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        s[c] = 64 * hh + c <= lim ? fmaf(s[c], scale, neg) : -INFINITY;
                        am[c & 7] = fmaxf(am[c & 7], s[c]);
                    }
                }
                const float amax = fmaxf(fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3])),
                                         fmaxf(fmaxf(am[4], am[5]), fmaxf(am[6], am[7])));
                // Raise the reference past the headroom (rare): shift this
                // chunk's arguments, and scale what the row has summed and
                // written against the old reference by exp2(-shift).
                const bool raise = amax > kRaise;
                if (__any_sync(0xffffffffu, raise)) {
                    const float shift = raise ? amax : 0.0f;
                    const float corr = raise ? ex2_approx(-amax) : 1.0f;
                    m_ref += shift;
                    l_run *= corr;
                    corr_blk *= corr;
#pragma unroll
                    for (int i = 0; i < 8; ++i) psum[i] *= corr;
#pragma unroll
                    for (int c = 0; c < 64; ++c) s[c] -= shift;
                    // P of the block's earlier chunks, already in TMEM.
                    tmem_wait_st();
#pragma unroll
                    for (int g = 0; g < hh; ++g)
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            float q[32];
                            tmem_ld32(s_addr + 64 * g + 32 * h2, q);
#pragma unroll
                            for (int e = 0; e < 32; ++e) q[e] *= corr;
                            tmem_st32_nowait(s_addr + 64 * g + 32 * h2, q);
                        }
                }
                // The probabilities over the scores (masked keys: exp2(-inf) = 0).
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    s[c] = ex2_approx(s[c]);
                    s[c + 1] = ex2_approx(s[c + 1]);
                    const float2 ps = __fadd2_rn(make_float2(psum[c & 7], psum[(c + 1) & 7]),
                                                 make_float2(s[c], s[c + 1]));
                    psum[c & 7] = ps.x;
                    psum[(c + 1) & 7] = ps.y;
                }
                tmem_st64_nowait(s_addr + 64 * hh, s);
            }
            l_run += ((psum[0] + psum[1]) + (psum[2] + psum[3])) + ((psum[4] + psum[5]) + (psum[6] + psum[7]));
            if (j > 0 && __any_sync(0xffffffffu, corr_blk != 1.0f)) {
                // O row *= corr_blk (1 for the rows that did not raise).
#pragma unroll
                for (int h = 0; h < kD / 32; ++h) {
                    float o[32];
                    tmem_ld32(o_addr + 32 * h, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= corr_blk;
                    tmem_st32_nowait(o_addr + 32 * h, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.p_full[t]);
        }
        if (ok && nbt > 0) {
            if (!mbar_wait(&sh.o_done[t], 0)) ok = false;
        }
        if (!ok) {
            if (nbt > 0) record_status(&g_wait_status, kWaitMma);
        } else if (p.o_tma) {
            // O / l through K stage t in the swizzled layout of the O tensor
            // map; each warp stores its 32 rows with one bulk tensor copy per
            // head-dim atom, and the copy leaves out the rows past M.  The
            // other tile may still have blocks to go (causal rows), so K is
            // free only once every MMA of the CTA is done (and with them every
            // K load, all consumed by score MMAs).
            if (!mbar_wait(&sh.mma_done, 0)) {
                record_status(&g_wait_status, kWaitMma);
                ok = false;
            }
        }
        if (ok && p.o_tma) {
            tc_fence_after();
            const float inv = 1.0f / l_run;
#pragma unroll
            for (int a = 0; a < kDA; ++a) {
                float o[32];
                tmem_ld32(o_addr + 32 * a, o);
                float* st = sh.k[t][a];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<float4*>(st + row * kAtom + ((c ^ (row & 7)) << 2)) =
                        make_float4(o[4 * c] * inv, o[4 * c + 1] * inv, o[4 * c + 2] * inv, o[4 * c + 3] * inv);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && m0 + t * BM + quarter * 32 < p.M) {
#pragma unroll
                for (int a = 0; a < kDA; ++a)
                    tma_store_3d(&to, sh.k[t][a] + quarter * 32 * kAtom, kAtom * a,
                                 (int)(m0 + t * BM + quarter * 32), p.bo ? (int)b : 0);
                bulk_commit();
                // Shared memory must outlive the copies' reads of it; the
                // writes themselves complete with the grid.
                bulk_wait_read_all();
            }
        } else if (ok) {
            tc_fence_after();
            const float inv = 1.0f / l_run;
            float* orow = p.O + b * p.bsO + (m < p.M ? m : 0) * p.rsO;
#pragma unroll
            for (int h = 0; h < kD / 32; ++h) {
                float o[32];
                tmem_ld32(o_addr + 32 * h, o);    // whole warp, converged
                if (m < p.M) {
                    if (p.o_vec) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4*>(orow + 32 * h + e) =
                                make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) orow[(32 * h + e) * p.csO] = o[e] * inv;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// A 3-D map (head dimension inner, rows, batch) with 32-wide boxes of `rows`
// rows and the 128-byte swizzle.  A zero batch stride maps one batch entry.
bool make_map(CUtensorMap* map, const float* base, int64_t rows, int64_t rs, int64_t bs,
              int64_t batch, int64_t inner, uint32_t box_rows) {
    const bool bcast = batch == 1 || bs == 0;
    const int64_t nb = bcast ? 1 : batch;
    const int64_t rs_b = rows > 1 ? rs * 4 : ((inner * 4 + 15) / 16) * 16;
    const int64_t bs_b = nb > 1 ? bs * 4 : rs_b * (rows > 1 ? rows : 1);
    const uint64_t dims[3] = {(uint64_t)inner, (uint64_t)rows, (uint64_t)nb};
    const uint64_t strides[2] = {(uint64_t)rs_b, (uint64_t)bs_b};
    const uint32_t box[3] = {32, box_rows, 1};
    return encode_tmap_f32_3d(map, base, dims, strides, box, true);
}

bool tma_operand(const float* base, int64_t rows, int64_t rs, int64_t cs, int64_t bs, int64_t batch) {
    if (cs != 1) return false;
    if (reinterpret_cast<uintptr_t>(base) % 16 != 0) return false;
    const int64_t lim = (int64_t)1 << 31;
    if (rows >= lim || batch >= lim) return false;
    auto ok_stride = [](int64_t st) { return st > 0 && (st * 4) % 16 == 0 && st * 4 < ((int64_t)1 << 40); };
    if (rows > 1 && (!ok_stride(rs) || rs < kD)) return false;
    if (batch > 1 && bs != 0 && (!ok_stride(bs) || bs < rs * rows)) return false;
    return true;
}

}  // namespace

bool attention_tc_supported(const AttnProblem& a) {
    return a.D == kD && a.Dv == kD && tma_operand(a.Q, a.M, a.rsQ, a.csQ, a.bsQ, a.batch) &&
           tma_operand(a.K, a.N, a.rsK, a.csK, a.bsK, a.batch) &&
           tma_operand(a.V, a.N, a.rsV, a.csV, a.bsV, a.batch);
}

cudaError_t launch_attention_tc(const AttnProblem& a, cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, a.Q, a.M, a.rsQ, a.bsQ, a.batch, kD, BM) ||
        !make_map(&tk, a.K, a.N, a.rsK, a.bsK, a.batch, kD, BN) ||
        !make_map(&tv, a.V, a.N, a.rsV, a.bsV, a.batch, kD, 32))
        return cudaErrorInvalidValue;
    Params p;
    p.O = a.O; p.rsO = a.rsO; p.csO = a.csO; p.bsO = a.bsO;
    p.M = a.M; p.N = a.N;
    p.scale_log2 = a.alpha * 1.4426950408889634f;
    p.causal = a.causal;
    p.q_len = a.causal ? a.q_len : a.M;
    p.bq = !(a.batch == 1 || a.bsQ == 0);
    p.bk = !(a.batch == 1 || a.bsK == 0);
    p.bv = !(a.batch == 1 || a.bsV == 0);
    p.o_vec = a.csO == 1 && reinterpret_cast<uintptr_t>(a.O) % 16 == 0 && a.rsO % 4 == 0 &&
              (a.batch == 1 || a.bsO % 4 == 0);
    // O through a tensor map when it has the layout of one (unit stride along
    // the values, 16-byte strides laid out without overlap), else by the row
    // threads.  A zero batch stride is never an O layout (validated injective).
    CUtensorMap to;
    std::memset(&to, 0, sizeof(to));
    p.o_tma = tma_operand(a.O, a.M, a.rsO, a.csO, a.bsO, a.batch) && (a.batch == 1 || a.bsO != 0) &&
              make_map(&to, a.O, a.M, a.rsO, a.bsO, a.batch, kD, 32);
    p.bo = a.batch > 1;
    const int64_t rows = kTiles * BM;
    const dim3 grid((unsigned)a.batch, (unsigned)((a.M + rows - 1) / rows));
    attention_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError();
}

unsigned int read_and_clear_wait_status_attention_tc(cudaStream_t stream) {
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
