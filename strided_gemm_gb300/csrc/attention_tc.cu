// Fused attention on the tensor cores (opt-in TF32): O = softmax(alpha Q K^T
// [causal]) V per (sequence, head), the scores and probabilities kept on the
// chip, as the FP32 kernel in attention.cu computes it ("rvllm CUDA path",
// section "What's basic about it": three steps with the scores in global
// memory, which a fused kernel avoids).
//
// One CTA per 128 query rows of one batch entry, head dimension 64, keys in
// blocks of 64.  Per block j:
//   S_j  = Q K_j^T   tcgen05.mma kind::tf32, M 128 x N 64 x K 64, into TMEM
//   P_j  = exp2(alpha log2(e) S_j - m)   one thread per query row, read from
//          TMEM with tcgen05.ld, the running maximum m and sum l in registers,
//          written to shared memory as the next MMA's K-major operand
//   PV_j = P_j V_j   M 128 x N 64 x K 64, into TMEM
//   O    = O exp2(m_old - m_new) + PV_j   in the row thread's registers
// and O / l is stored at the end.  Roles, all waits bounded (a timeout records
// a status code and returns):
//   warp 0       TMA: Q once; K_j (two 128-byte swizzled boxes of 32 along
//                the head dimension) and V_j (four raw 32 x 32 boxes) into a
//                2-stage ring;
//   warp 1       one lane issues the MMAs: S_0, then S_{j+1} ahead of PV_j, so
//                the next block's scores are ready when its softmax starts;
//   warps 2-5    softmax and output, one TMEM lane quarter each;
//   warps 6-7    rewrite V_j (rows along the keys) into V_j^T with rows along
//                the values, the K-major layout P V's B operand takes
//                (4 x 4 quads, conflict-free under the swizzle).
// S and PV are double-buffered in TMEM (4 x 64 columns).  The adding of PV_j
// into O waits until P_{j+1} is written, so PV_j overlaps the next softmax.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "attention_tc.h"
#include "ptx.cuh"

namespace sbg {
namespace {

constexpr int kD = 64;               // head dimension of Q, K and V
constexpr int BM = 128;              // query rows per CTA (the MMA's M)
constexpr int BN = 64;               // keys per block
constexpr int kAtom = 32;            // fp32 values in one 128-byte swizzled row
constexpr int kMmaK = 8;             // tf32 elements per MMA
constexpr int kStages = 2;           // K and raw V blocks in flight
constexpr int kSoftWarps = 4, kTransWarps = 2;   // 8 warps: up to 255 registers a thread
constexpr int kWarps = 2 + kSoftWarps + kTransWarps;
constexpr int kThreads = kWarps * 32;
constexpr int kBox = 32 * 32;
constexpr uint32_t kTmemCols = 256;  // S[2], PV[2]
constexpr uint32_t kColS = 0, kColPV = 128;

// Instruction descriptor, kind::tf32: D fp32, A and B tf32 K-major, N 64
// (both products), M 128.
constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

struct Smem {
    alignas(1024) float q[2][BM * kAtom];           // Q, K-major: head-dim atoms 0-31, 32-63
    alignas(1024) float k[kStages][2][BN * kAtom];  // K_j, K-major, same atoms
    alignas(1024) float vraw[kStages][4][kBox];     // V_j: box (key half h, value half g) at 2h + g
    alignas(1024) float vt[2][2][kD * kAtom];       // V_j^T: rows along the values, key atoms
    alignas(1024) float p[2][BM * kAtom];           // P_j, K-major: key atoms 0-31, 32-63
    uint64_t q_full;
    uint64_t k_full[kStages], k_empty[kStages];
    uint64_t v_full[kStages], v_empty[kStages];
    uint64_t vt_full[2], vt_empty[2];
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full, p_empty;
    uint64_t pv_full[2], pv_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

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
};

// Rewrites one key atom of V_j: two raw boxes (32 keys x 32 values each, the
// value halves) into V_j^T rows 0..63 (values) x 32 keys, K-major 128-byte
// swizzle.  A quarter-warp's quads hit 8 distinct 16-byte chunks on both the
// loads and the stores.
__device__ __forceinline__ void transpose_atom(const float* raw, float* dst, int t) {
    constexpr int kQuads = kD / 4 * (kAtom / 4);     // 128: two per transposer thread
#pragma unroll
    for (int q = t; q < kQuads; q += kTransWarps * 32) {
        const int kq = ((q >> 2) & 1) | (((q ^ (q >> 1) ^ (q >> 3)) & 1) << 1) | (((q >> 4) & 1) << 2);
        const int mq = (q & 3) | ((q >> 5) << 2);    // 4-row group of values, 0..15
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

// The 8 MMAs (K = 64 in steps of 8) of one 128 x 64 x 64 product whose
// operands are two 32-wide K atoms each.
__device__ __forceinline__ void mma_128x64x64(uint32_t d, const float* a0, const float* a1,
                                              const float* b0, const float* b1) {
#pragma unroll
    for (int kk = 0; kk < kD / kMmaK; ++kk) {
        const uint32_t off = (uint32_t)(kk & 3) * kMmaK * 4;
        const uint64_t ad = umma_desc_kmajor_sw128(smem_u32(kk < 4 ? a0 : a1) + off);
        const uint64_t bd = umma_desc_kmajor_sw128(smem_u32(kk < 4 ? b0 : b1) + off);
        mma_tf32(d, ad, bd, kIdesc, kk > 0 ? 1u : 0u);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    Smem& sh = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                        ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t b = blockIdx.x;
    const int64_t mb = p.causal ? (int64_t)gridDim.y - 1 - blockIdx.y : (int64_t)blockIdx.y;
    const int64_t m0 = mb * BM;
    // Keys this CTA needs: all, or (causal) up to its rows' last position.
    int64_t n_end = p.N;
    if (p.causal) {
        const int64_t m_last = (m0 + BM - 1 < p.M ? m0 + BM - 1 : p.M - 1);
        const int64_t r0 = m0 % p.q_len;
        const bool wraps = r0 + (m_last - m0) >= p.q_len;
        n_end = (wraps ? p.N - 1 : (m_last % p.q_len) + p.N - p.q_len) + 1;
    }
    const int nblk = (int)((n_end + BN - 1) / BN);

    if (threadIdx.x == 0) {
        mbar_init(&sh.q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sh.k_full[s], 1);
            mbar_init(&sh.k_empty[s], 1);
            mbar_init(&sh.v_full[s], 1);
            mbar_init(&sh.v_empty[s], kTransWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.vt_full[i], kTransWarps);
            mbar_init(&sh.vt_empty[i], 1);
            mbar_init(&sh.s_full[i], 1);
            mbar_init(&sh.s_empty[i], kSoftWarps);
            mbar_init(&sh.pv_full[i], 1);
            mbar_init(&sh.pv_empty[i], kSoftWarps);
        }
        mbar_init(&sh.p_full, kSoftWarps);
        mbar_init(&sh.p_empty, 1);
        mbar_init(&sh.mma_done, 1);
        fence_mbar_init();
        prefetch_tensormap(&tq);
        prefetch_tensormap(&tk);
        prefetch_tensormap(&tv);
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
            mbar_arrive_expect_tx(&sh.q_full, 2 * BM * kAtom * 4);
            tma_load_3d(sh.q[0], &tq, &sh.q_full, 0, (int)m0, zq);
            tma_load_3d(sh.q[1], &tq, &sh.q_full, kAtom, (int)m0, zq);
            int j = 0;
            for (; j < nblk; ++j) {
                const int s = j % kStages;
                const uint32_t ph = (uint32_t)(((j / kStages) - 1) & 1);
                if (j >= kStages && (!mbar_wait(&sh.k_empty[s], ph) || !mbar_wait(&sh.v_empty[s], ph))) {
                    record_status(&g_wait_status, kWaitEmpty);
                    break;
                }
                const int n0 = j * BN;
                mbar_arrive_expect_tx(&sh.k_full[s], 2 * BN * kAtom * 4);
                tma_load_3d(sh.k[s][0], &tk, &sh.k_full[s], 0, n0, zk);
                tma_load_3d(sh.k[s][1], &tk, &sh.k_full[s], kAtom, n0, zk);
                mbar_arrive_expect_tx(&sh.v_full[s], 4 * kBox * 4);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int g = 0; g < 2; ++g)
                        tma_load_3d(sh.vraw[s][2 * h + g], &tv, &sh.v_full[s], 32 * g, n0 + 32 * h, zv);
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
            bool ok = mbar_wait(&sh.q_full, 0);
            auto issue_s = [&](int j) -> bool {
                const int s = j % kStages, buf = j & 1;
                if (!mbar_wait(&sh.k_full[s], (uint32_t)((j / kStages) & 1))) return false;
                if (j >= 2 && !mbar_wait(&sh.s_empty[buf], (uint32_t)(((j >> 1) - 1) & 1))) return false;
                tc_fence_after();
                mma_128x64x64(tmem + kColS + buf * BN, sh.q[0], sh.q[1], sh.k[s][0], sh.k[s][1]);
                mma_commit(&sh.k_empty[s]);
                mma_commit(&sh.s_full[buf]);
                return true;
            };
            if (ok && nblk > 0) ok = issue_s(0);
            for (int j = 0; j < nblk && ok; ++j) {
                if (j + 1 < nblk && !issue_s(j + 1)) { ok = false; break; }
                const int buf = j & 1;
                if (!mbar_wait(&sh.p_full, (uint32_t)(j & 1)) ||
                    !mbar_wait(&sh.vt_full[buf], (uint32_t)((j >> 1) & 1)) ||
                    (j >= 2 && !mbar_wait(&sh.pv_empty[buf], (uint32_t)(((j >> 1) - 1) & 1)))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                mma_128x64x64(tmem + kColPV + buf * kD, sh.p[0], sh.p[1], sh.vt[buf][0], sh.vt[buf][1]);
                mma_commit(&sh.p_empty);
                mma_commit(&sh.vt_empty[buf]);
                mma_commit(&sh.pv_full[buf]);
            }
            if (!ok) record_status(&g_wait_status, kWaitFull);
            // Nothing may still be writing TMEM when it is freed.
            mma_commit(&sh.mma_done);
            if (!mbar_wait(&sh.mma_done, 0)) record_status(&g_wait_status, kWaitMma);
        }
    } else if (warp < 2 + kSoftWarps) {
        // ---- softmax and output, one query row per thread ------------------
        const int quarter = warp & 3;                 // TMEM lanes this warp may read
        const int row = quarter * 32 + lane;
        const int64_t m = m0 + row;
        const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
        const int64_t pos = p.causal ? (m % p.q_len) + p.N - p.q_len : p.N - 1;
        float o[kD];
#pragma unroll
        for (int e = 0; e < kD; ++e) o[e] = 0.0f;
        float m_run = -INFINITY, l_run = 0.0f, corr_prev = 1.0f;
        bool ok = true;
        // O = O * corr_prev + PV_{j}, once PV_j has landed.
        auto add_pv = [&](int j) -> bool {
            const int buf = j & 1;
            if (!mbar_wait(&sh.pv_full[buf], (uint32_t)((j >> 1) & 1))) return false;
            tc_fence_after();
            float v[32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tmem_ld32(tmem + lanes + kColPV + buf * kD + h * 32, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[h * 32 + e] = fmaf(o[h * 32 + e], corr_prev, v[e]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.pv_empty[buf]);
            return true;
        };
        for (int j = 0; j < nblk; ++j) {
            const int buf = j & 1;
            if (!mbar_wait(&sh.s_full[buf], (uint32_t)((j >> 1) & 1))) { ok = false; break; }
            tc_fence_after();
            float s[BN];
            {
                float v[32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    tmem_ld32(tmem + lanes + kColS + buf * BN + h * 32, v);
#pragma unroll
                    for (int c = 0; c < 32; ++c) s[h * 32 + c] = v[c];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.s_empty[buf]);
            // Mask (keys past N, or past the row's causal position), scale to
            // the exp2 domain, and the running maximum.
            const int64_t n0 = (int64_t)j * BN;
            // Keys c <= lim of the block are kept.  Eight partial maxima and
            // sums, so that no chain runs through all 64 keys.
            const int64_t last = (pos < p.N - 1 ? pos : p.N - 1) - n0;
            const int lim = last < 0 ? -1 : (last >= BN ? BN - 1 : (int)last);
            float part[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) part[i] = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; ++c) {
                s[c] = c <= lim ? s[c] * p.scale_log2 : -INFINITY;
                part[c & 7] = fmaxf(part[c & 7], s[c]);
            }
            const float mx = fmaxf(fmaxf(fmaxf(part[0], part[1]), fmaxf(part[2], part[3])),
                                   fmaxf(fmaxf(part[4], part[5]), fmaxf(part[6], part[7])));
            const float m_new = fmaxf(m_run, mx);
            // A row with no kept key so far keeps m = -inf; its terms stay 0.
            const float base = m_new == -INFINITY ? 0.0f : m_new;
            const float corr = exp2f(m_run - base);
#pragma unroll
            for (int i = 0; i < 8; ++i) part[i] = 0.0f;
#pragma unroll
            for (int c = 0; c < BN; ++c) {
                s[c] = exp2f(s[c] - base);
                part[c & 7] += s[c];
            }
            const float sum = ((part[0] + part[1]) + (part[2] + part[3])) +
                              ((part[4] + part[5]) + (part[6] + part[7]));
            l_run = l_run * corr + sum;
            m_run = m_new;
            // P_j to shared memory once P V_{j-1} has read P_{j-1}.
            if (j > 0 && !mbar_wait(&sh.p_empty, (uint32_t)((j - 1) & 1))) { ok = false; break; }
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<float4*>(&sh.p[a][row * kAtom + ((q ^ (row & 7)) << 2)]) =
                        make_float4(s[a * 32 + 4 * q], s[a * 32 + 4 * q + 1], s[a * 32 + 4 * q + 2],
                                    s[a * 32 + 4 * q + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.p_full);
            // The previous block's P V joins O while this block's runs.
            if (j > 0 && !add_pv(j - 1)) { ok = false; break; }
            corr_prev = corr;
        }
        if (ok && nblk > 0) ok = add_pv(nblk - 1);
        if (!ok) {
            record_status(&g_wait_status, kWaitMma);
        } else if (m < p.M) {
            const float inv = 1.0f / l_run;
            float* orow = p.O + b * p.bsO + m * p.rsO;
            if (p.o_vec) {
#pragma unroll
                for (int e = 0; e < kD; e += 4)
                    *reinterpret_cast<float4*>(orow + e) =
                        make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
            } else {
#pragma unroll
                for (int e = 0; e < kD; ++e) orow[e * p.csO] = o[e] * inv;
            }
        }
    } else {
        // ---- V_j -> V_j^T -------------------------------------------------
        const int t = threadIdx.x - (2 + kSoftWarps) * 32;
        for (int j = 0; j < nblk; ++j) {
            const int s = j % kStages, buf = j & 1;
            if (!mbar_wait(&sh.v_full[s], (uint32_t)((j / kStages) & 1))) {
                record_status(&g_wait_status, kWaitFull);
                break;
            }
            if (j >= 2 && !mbar_wait(&sh.vt_empty[buf], (uint32_t)(((j >> 1) - 1) & 1))) {
                record_status(&g_wait_status, kWaitEmpty);
                break;
            }
            transpose_atom(sh.vraw[s][0], sh.vt[buf][0], t);    // keys 0..31 of the block
            transpose_atom(sh.vraw[s][2], sh.vt[buf][1], t);    // keys 32..63
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sh.vt_full[buf]);
                mbar_arrive(&sh.v_empty[s]);
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
    const dim3 grid((unsigned)a.batch, (unsigned)((a.M + BM - 1) / BM));
    attention_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
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
