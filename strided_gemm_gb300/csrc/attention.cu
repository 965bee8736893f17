// Fused attention: O = softmax(alpha * Q K^T [causal]) V over a batch of
// (sequence, head) problems laid out by strides, without the scores or the
// probabilities ever reaching global memory.  The pages compute attention as
// three launches, scores, softmax and probs @ V, with the scores matrix in
// global memory in between, and name a fused kernel as the way to avoid that
// ("rvllm CUDA path", section "What's basic about it"); grouped-query heads are
// rows of one batch entry stacked against one K ("rvllm CUDA path", section
// "Matmuls go to cuBLAS").
//
// One CTA of 128 threads per 128 query rows of one batch entry, walking the
// keys in blocks of 64 (flash-attention order):
//  * Q's block goes into shared memory once, transposed ([d][m]); each key
//    block's K is transposed into [d][n] and V kept as [n][e].
//  * Each thread owns 8 query rows x 8 keys of a score block and 8 rows x
//    DH/8 value columns (runs of 4, so that its 16-byte shared-memory reads of
//    Q, K, P and V are contiguous across the warp): S = Q K^T by FFMA
//    micro-tiles, then the online softmax per row: the row maximum across the
//    8 lanes sharing the row (shuffles), the running sum kept per thread until
//    the end, exp2 on scores pre-scaled by alpha * log2(e), and O rescaled by
//    exp2(m_old - m_new).
//  * P goes to shared memory transposed ([n][m]); O += P V by FFMA.
//  * Causal: keys after position(m) = (m mod q_len) + N - q_len are masked;
//    key blocks past the CTA's last position are skipped.
// Head dimension DH = 32, 64, 96 or 128, the same for Q, K and V.
//
// Paged K and V ("rvllm CUDA path", section "The kernels", and the paged read
// that section "What's basic about it" names instead of gathering the whole
// context every step): K and V are then the caches [num_blocks][block_size]
// [n_kv_heads][DH], and key n of batch entry b (sequence b / n_kv_heads, head
// b % n_kv_heads) is row n % block_size of block table[seq][n / block_size].
// The row offsets of each key block are looked up once per block into shared
// memory; a block id outside the cache, or a sequence length outside [1, N]
// (or below q_len when causal), records kPagedInput in the status word and
// the key reads as zero or the length is clamped, so no access leaves the
// caches.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "debug_check.cuh"
#include "internal.h"

namespace sbg {
namespace {

constexpr int BM = 128;         // query rows per CTA
constexpr int BN = 64;          // keys per block
constexpr int kThreads = 128;
constexpr int QP = BM + 4;      // pitch of Qs[d][m] and Ps[n][m]
constexpr int KP = BN + 4;      // pitch of Ks[d][n]

struct AttnParams {
    const float* Q; int64_t rsQ, csQ, bsQ;
    const float* K; int64_t rsK, csK, bsK;
    const float* V; int64_t rsV, csV, bsV;
    float* O; int64_t rsO, csO, bsO;
    int64_t M, N, batch;
    float scale_log2;            // alpha * log2(e)
    int causal;
    int64_t q_len;
    int v_vec, o_vec;            // unit stride along e and 16-byte aligned rows
    ElemSpan sq, sk, sv, so;     // debug builds: valid element offsets of the operands
    // Paged K / V (PAGED kernels only).
    const int32_t* table;
    const int32_t* seq_lens;
    int64_t max_blocks, block_size, n_kv_heads, num_blocks;
};

template <int DH>
struct Smem {
    float q[DH * QP];            // Q block, [d][m]
    float k[DH * KP];            // K block, [d][n]
    float v[BN * DH];            // V block, [n][e]
    float p[BN * QP];            // probabilities, [n][m]
    int64_t row[BN];             // paged: element offset of each key's row (-1: none)
};

// Rows of the CTA owned by thread row-group ty (0..15): two runs of 4.
__device__ __forceinline__ int row_of(int ty, int i) { return (i < 4 ? 0 : 64) + ty * 4 + (i & 3); }
// Keys of a block, or value dimensions, of column-group tx (0..7): runs of 4
// every 32.
__device__ __forceinline__ int col_of(int tx, int j) { return (j >> 2) * 32 + tx * 4 + (j & 3); }

// Status word of this kernel's debug bounds checks and paged-input checks
// (sbgemm_device_status).
__device__ unsigned int g_status = 0;

template <int DH, bool PAGED>
__global__ void __launch_bounds__(kThreads, DH <= 64 ? 2 : 1) attention_kernel(const AttnParams p) {
    constexpr int EC = DH / 8;   // value columns per thread
    extern __shared__ float4 smem4[];
    Smem<DH>& sh = *reinterpret_cast<Smem<DH>*>(smem4);
    const int t = threadIdx.x;
    const int lane = t & 31, warp = t >> 5;
    const int ty = warp * 4 + (lane >> 3), tx = lane & 7;
    // Blocks are launched batch entry fastest; causal row blocks late in a
    // head see more keys, so they go first and the short ones fill the last
    // wave.
    const int64_t b = blockIdx.x;
    const int64_t mb = p.causal ? (int64_t)gridDim.y - 1 - blockIdx.y : (int64_t)blockIdx.y;
    const int64_t m0 = mb * BM;
    const float* Qb = p.Q + b * p.bsQ;
    const float* Kb = PAGED ? p.K : p.K + b * p.bsK;
    const float* Vb = PAGED ? p.V : p.V + b * p.bsV;

    // This entry's keys: N, or (paged) its sequence's length.
    int64_t len = p.N;
    int64_t seq = 0, head = 0;
    if constexpr (PAGED) {
        seq = b / p.n_kv_heads;
        head = b - seq * p.n_kv_heads;
        if (p.seq_lens) {
            len = p.seq_lens[seq];
            const int64_t lo = p.causal ? p.q_len : 1;
            if (len < lo || len > p.N) {
                if (t == 0) record_status(&g_status, kPagedInput);
                len = len < lo ? lo : p.N;
            }
        }
    }

    // Q block, transposed: thread (d, m4) gathers 4 consecutive rows and
    // stores them as one 16-byte word of row d (conflict-free with pitch QP).
#pragma unroll 4
    for (int idx = t; idx < DH * (BM / 4); idx += kThreads) {
        const int d = idx % DH, m4 = idx / DH;
        float x[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t m = m0 + 4 * m4 + q;
            const float* a = Qb + m * p.rsQ + d * p.csQ;
            x[q] = (m < p.M && dbg_in_span(p.Q, a, p.sq, &g_status)) ? *a : 0.0f;
        }
        *reinterpret_cast<float4*>(&sh.q[d * QP + 4 * m4]) = make_float4(x[0], x[1], x[2], x[3]);
    }

    // Keys this CTA needs: all, or (causal) up to its rows' last position.
    int64_t n_end = len;
    if (p.causal) {
        const int64_t m_last = (m0 + BM - 1 < p.M ? m0 + BM - 1 : p.M - 1);
        const int64_t r0 = m0 % p.q_len;
        const bool wraps = r0 + (m_last - m0) >= p.q_len;
        const int64_t last_pos = wraps ? len - 1 : (m_last % p.q_len) + len - p.q_len;
        n_end = last_pos + 1;
    }
    int64_t pos[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t m = m0 + row_of(ty, i);
        pos[i] = p.causal ? (m % p.q_len) + len - p.q_len : len;
    }

    // Accumulators pair adjacent rows (2ip, 2ip+1) of one column: the packed
    // FMA (fma.rn.f32x2) takes the pair from one 16-byte shared-memory load
    // and broadcasts the column operand.
    float2 o[4][EC];
    float mrow[8], lrow[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        mrow[i] = -INFINITY;
        lrow[i] = 0.0f;
    }
#pragma unroll
    for (int ip = 0; ip < 4; ++ip)
#pragma unroll
        for (int j = 0; j < EC; ++j) o[ip][j] = make_float2(0.0f, 0.0f);

    for (int64_t n0 = 0; n0 < n_end; n0 += BN) {
        __syncthreads();   // the previous block's K, V, P and row offsets are no longer read
        if constexpr (PAGED) {
            if (t < BN) {
                const int64_t n = n0 + t;
                int64_t off = -1;
                if (n < len) {
                    const int64_t bp = n / p.block_size;
                    const int64_t blk = p.table[seq * p.max_blocks + bp];
                    if (blk >= 0 && blk < p.num_blocks)
                        off = ((blk * p.block_size + (n - bp * p.block_size)) * p.n_kv_heads + head) * DH;
                    else
                        record_status(&g_status, kPagedInput);
                }
                sh.row[t] = off;
            }
            __syncthreads();
        }
        {
            // K block, transposed like Q.
#pragma unroll 4
            for (int idx = t; idx < DH * (BN / 4); idx += kThreads) {
                const int d = idx % DH, n4 = idx / DH;
                float x[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if constexpr (PAGED) {
                        const int64_t off = sh.row[4 * n4 + q];
                        const float* a = Kb + off + d;
                        x[q] = (off >= 0 && dbg_in_span(p.K, a, p.sk, &g_status)) ? *a : 0.0f;
                    } else {
                        const int64_t n = n0 + 4 * n4 + q;
                        const float* a = Kb + n * p.rsK + d * p.csK;
                        x[q] = (n < len && dbg_in_span(p.K, a, p.sk, &g_status)) ? *a : 0.0f;
                    }
                }
                *reinterpret_cast<float4*>(&sh.k[d * KP + 4 * n4]) = make_float4(x[0], x[1], x[2], x[3]);
            }
            // V block as stored: DH/4 threads per row.
#pragma unroll 4
            for (int idx = t; idx < BN * (DH / 4); idx += kThreads) {
                const int r = idx / (DH / 4), e4 = idx % (DH / 4);
                const int64_t n = n0 + r;
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                const float* vrow;
                bool ok;
                if constexpr (PAGED) {
                    const int64_t off = sh.row[r];
                    vrow = Vb + (off < 0 ? 0 : off);
                    ok = off >= 0;
                } else {
                    vrow = Vb + n * p.rsV;
                    ok = n < len;
                }
                if (ok && dbg_in_span(p.V, vrow, p.sv, &g_status) &&
                    dbg_in_span(p.V, vrow + (4 * e4 + 3) * p.csV, p.sv, &g_status)) {
                    if (p.v_vec) {
                        x = __ldg(reinterpret_cast<const float4*>(vrow) + e4);
                    } else {
                        x.x = vrow[(4 * e4 + 0) * p.csV];
                        x.y = vrow[(4 * e4 + 1) * p.csV];
                        x.z = vrow[(4 * e4 + 2) * p.csV];
                        x.w = vrow[(4 * e4 + 3) * p.csV];
                    }
                }
                *reinterpret_cast<float4*>(&sh.v[r * DH + 4 * e4]) = x;
            }
        }
        __syncthreads();

        // Scores of this block: 8 rows x 8 keys per thread.
        float2 s2[4][8];
#pragma unroll
        for (int ip = 0; ip < 4; ++ip)
#pragma unroll
            for (int j = 0; j < 8; ++j) s2[ip][j] = make_float2(0.0f, 0.0f);
#pragma unroll 4
        for (int d = 0; d < DH; ++d) {
            const float4 qa = *reinterpret_cast<const float4*>(&sh.q[d * QP + ty * 4]);
            const float4 qb = *reinterpret_cast<const float4*>(&sh.q[d * QP + 64 + ty * 4]);
            const float4 ka = *reinterpret_cast<const float4*>(&sh.k[d * KP + tx * 4]);
            const float4 kb = *reinterpret_cast<const float4*>(&sh.k[d * KP + 32 + tx * 4]);
            const float2 a[4] = {make_float2(qa.x, qa.y), make_float2(qa.z, qa.w),
                                 make_float2(qb.x, qb.y), make_float2(qb.z, qb.w)};
            const float c[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
#pragma unroll
            for (int ip = 0; ip < 4; ++ip)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    s2[ip][j] = __ffma2_rn(a[ip], make_float2(c[j], c[j]), s2[ip][j]);
        }
        // Row i of column j of the score and output accumulators.
#define S_AT(i, j) (((i) & 1) ? s2[(i) >> 1][j].y : s2[(i) >> 1][j].x)
#define O_AT(i, j) (((i) & 1) ? o[(i) >> 1][j].y : o[(i) >> 1][j].x)

        // Online softmax per row.
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int64_t n = n0 + col_of(tx, j);
                const bool keep = n < len && n <= pos[i];
                S_AT(i, j) = keep ? S_AT(i, j) * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, S_AT(i, j));
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            const float m_new = fmaxf(mrow[i], mx);
            // A row with no kept key so far keeps m = -inf; its terms stay 0.
            const float base = m_new == -INFINITY ? 0.0f : m_new;
            const float corr = exp2f(mrow[i] - base);
            float sum = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                S_AT(i, j) = exp2f(S_AT(i, j) - base);
                sum += S_AT(i, j);
            }
            lrow[i] = lrow[i] * corr + sum;
            mrow[i] = m_new;
#pragma unroll
            for (int j = 0; j < EC; ++j) O_AT(i, j) *= corr;
        }

        // P to shared memory, transposed: Ps[n][m].
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int n = col_of(tx, j);
            *reinterpret_cast<float4*>(&sh.p[n * QP + ty * 4]) =
                make_float4(s2[0][j].x, s2[0][j].y, s2[1][j].x, s2[1][j].y);
            *reinterpret_cast<float4*>(&sh.p[n * QP + 64 + ty * 4]) =
                make_float4(s2[2][j].x, s2[2][j].y, s2[3][j].x, s2[3][j].y);
        }
        __syncthreads();

        // O += P V over the block's keys.
#pragma unroll 4
        for (int n = 0; n < BN; ++n) {
            const float4 pa = *reinterpret_cast<const float4*>(&sh.p[n * QP + ty * 4]);
            const float4 pb = *reinterpret_cast<const float4*>(&sh.p[n * QP + 64 + ty * 4]);
            const float2 a[4] = {make_float2(pa.x, pa.y), make_float2(pa.z, pa.w),
                                 make_float2(pb.x, pb.y), make_float2(pb.z, pb.w)};
#pragma unroll
            for (int r = 0; r < EC / 4; ++r) {
                const float4 vv = *reinterpret_cast<const float4*>(&sh.v[n * DH + r * 32 + tx * 4]);
                const float c[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                for (int ip = 0; ip < 4; ++ip)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        o[ip][4 * r + j] = __ffma2_rn(a[ip], make_float2(c[j], c[j]), o[ip][4 * r + j]);
            }
        }
#undef S_AT
    }

    // Normalise by the row sums (gathered over the 8 lanes of the row) and store.
    float* Ob = p.O + b * p.bsO;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float l = lrow[i];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        const int64_t m = m0 + row_of(ty, i);
        if (m >= p.M) continue;
        const float inv = 1.0f / l;
        float* orow = Ob + m * p.rsO;
        if (!dbg_in_span(p.O, orow, p.so, &g_status) ||
            !dbg_in_span(p.O, orow + (DH - 1) * p.csO, p.so, &g_status))
            continue;
        if (p.o_vec) {
#pragma unroll
            for (int r = 0; r < EC / 4; ++r)
                *reinterpret_cast<float4*>(orow + r * 32 + tx * 4) =
                    make_float4(O_AT(i, 4 * r) * inv, O_AT(i, 4 * r + 1) * inv,
                                O_AT(i, 4 * r + 2) * inv, O_AT(i, 4 * r + 3) * inv);
        } else {
#pragma unroll
            for (int j = 0; j < EC; ++j) orow[col_of(tx, j) * p.csO] = O_AT(i, j) * inv;
        }
    }
#undef O_AT
}

template <int DH, bool PAGED>
cudaError_t launch_dh(const AttnParams& p, const dim3& grid, cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(attention_kernel<DH, PAGED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(Smem<DH>));
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    attention_kernel<DH, PAGED><<<grid, kThreads, sizeof(Smem<DH>), stream>>>(p);
    return cudaGetLastError();
}

template <bool PAGED>
cudaError_t launch_paged(const AttnParams& p, int64_t D, const dim3& grid, cudaStream_t stream) {
    switch (D) {
        case 32: return launch_dh<32, PAGED>(p, grid, stream);
        case 64: return launch_dh<64, PAGED>(p, grid, stream);
        case 96: return launch_dh<96, PAGED>(p, grid, stream);
        case 128: return launch_dh<128, PAGED>(p, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool attention_supported(int64_t D, int64_t Dv) {
    return D == Dv && (D == 32 || D == 64 || D == 96 || D == 128);
}

int64_t attention_max_rows() { return (int64_t)65535 * BM; }

cudaError_t launch_attention(const AttnProblem& a, cudaStream_t stream) {
    if (!attention_supported(a.D, a.Dv)) return cudaErrorInvalidValue;
    AttnParams p;
    p.Q = a.Q; p.rsQ = a.rsQ; p.csQ = a.csQ; p.bsQ = a.bsQ;
    p.K = a.K; p.rsK = a.rsK; p.csK = a.csK; p.bsK = a.bsK;
    p.V = a.V; p.rsV = a.rsV; p.csV = a.csV; p.bsV = a.bsV;
    p.O = a.O; p.rsO = a.rsO; p.csO = a.csO; p.bsO = a.bsO;
    p.M = a.M; p.N = a.N; p.batch = a.batch;
    p.scale_log2 = a.alpha * 1.4426950408889634f;
    p.causal = a.causal;
    p.q_len = a.causal ? a.q_len : a.M;
    p.v_vec = a.csV == 1 && reinterpret_cast<uintptr_t>(a.V) % 16 == 0 && a.rsV % 4 == 0 &&
              (a.batch == 1 || a.paged || a.bsV % 4 == 0);
    p.o_vec = a.csO == 1 && reinterpret_cast<uintptr_t>(a.O) % 16 == 0 && a.rsO % 4 == 0 &&
              (a.batch == 1 || a.bsO % 4 == 0);
    p.sq = a.sq; p.sk = a.sk; p.sv = a.sv; p.so = a.so;
    p.table = a.table; p.seq_lens = a.seq_lens;
    p.max_blocks = a.max_blocks; p.block_size = a.block_size;
    p.n_kv_heads = a.n_kv_heads; p.num_blocks = a.num_blocks;
    const dim3 grid((unsigned)a.batch, (unsigned)((a.M + BM - 1) / BM));
    return a.paged ? launch_paged<true>(p, a.D, grid, stream)
                   : launch_paged<false>(p, a.D, grid, stream);
}

unsigned int read_and_clear_status_attention(cudaStream_t stream) {
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
