// Fused attention for few query rows per batch entry (a decode step: one new
// token per sequence, its grouped-query heads stacked as rows), reading K and
// V either by strides or straight out of a paged cache through the block
// table ("rvllm CUDA path", section "The kernels": the cache
// [num_blocks][block_size][n_kv_heads][head_dim] and the block-table lookup of
// position pos at block pos / block_size, offset pos % block_size; section
// "What's basic about it": a kernel that reads straight from the blocks
// instead of gathering the whole context every decode step).
//
// With a handful of rows the work is the stream of K and V rows out of HBM
// (about 2 * head_dim * 4 bytes per key and head against 4 * rows * head_dim
// flops), so the kernel is built for bandwidth, not for the FMA pipe:
//  * The keys of a batch entry are cut into chunks (with a workspace), one
//    CTA each, so that the grid fills the SMs even for a few long sequences.
//    (Handing (entry, chunk) items out from a counter to a grid the size of
//    the SMs' capacity measured slower: the hardware already places CTAs as
//    slots free up, and smaller items only add start-up.)
//  * A CTA streams its chunk in tiles of 32 keys through a 3-stage (4 at head dimension 32) ring of
//    16-byte cp.async copies (K and V rows are contiguous along the head
//    dimension); keys past the sequence, or with a bad block id, are zero
//    filled without a read.  The paged row offsets of 256 keys at a time are
//    looked up half a sub-chunk ahead of the copies that use them.
//  * Eight lanes share a key: each holds DH/8 of the head dimension (runs of
//    4 every 32) of every query row and of the key's K and V rows, and forms
//    its part of the dot products of the group's two keys of a tile with the
//    MR rows.  A reduce-scatter across the eight lanes (each round keeps half
//    of the values and adds the partner's other half) leaves every lane with
//    the full score of its own (key, row) pairs, so the masking and the exp2
//    of a pair happen once, not on all eight lanes; the probabilities then go
//    back to every lane by shuffles for O += P V.
//  * Each lane group keeps its own online softmax against a reference maximum
//    per row that moves only when a score passes it by 2^8 (then l and O are
//    scaled; warp-uniform and rare), so the common step is one exp2 per pair.
//  * The 16 lane groups of a CTA merge in shared memory; with one chunk the
//    CTA normalises and stores O, otherwise it writes (max, sum, O) of its
//    chunk to the caller's workspace and counts itself in on the entry's
//    counter; the last chunk to arrive merges all of them in chunk order (so
//    results do not depend on timing).  No second launch, no clearing of the
//    counters (each call tags them with its own epoch).  (A separate merge
//    launch cost about 8 us of a 80 us step; merging the chunks of an entry
//    inside a thread-block cluster was slower still on ragged batches, as a
//    short sequence's empty chunks hold their SM slots until the cluster's
//    longest chunk ends.)
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "debug_check.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace sbg {
namespace {

constexpr int kThreads = 128;
constexpr int kGroups = kThreads / 8;   // 8-lane key groups per CTA
constexpr int TK = 32;                  // keys per tile
// Ring stages: 4 for head dimension 32, 3 above (four CTAs of an SM at 64).
template <int DH>
__host__ __device__ constexpr int stages_of() { return DH <= 32 ? 4 : 3; }
// CTAs per SM the register budget aims at: 4 while a lane's rows and head
// slots are few (32 warps' worth of latency hiding), else 2.
template <int DH, int MR>
__host__ __device__ constexpr int min_ctas_of() { return DH * MR <= 256 ? 4 : 2; }
constexpr int SC = 256;                 // keys per sub-chunk of looked-up row offsets
constexpr int kTilesPerSub = SC / TK;
constexpr float kRaise = 8.0f;          // log2 headroom of the reference maximum

struct DecodeParams {
    const float* Q; int64_t rsQ, csQ, bsQ;
    const float* K; int64_t rsK, bsK;   // unit stride along the head dimension
    const float* V; int64_t rsV, bsV;
    float* O; int64_t rsO, csO, bsO;
    int64_t M, N;
    int64_t chunk_keys;
    int chunks;
    float scale_log2;                   // alpha * log2(e)
    int causal;
    int64_t q_len;
    float* part;                        // [entry][chunk][MR][2 + DH] when chunks > 1
    unsigned long long* counters;       // [entry]: chunks arrived, tagged with the call's epoch
    unsigned long long epoch;           // this call's tag (48 bits)
    const int32_t* table;
    const int32_t* seq_lens;
    int64_t max_blocks, block_size, n_kv_heads, num_blocks;
    ElemSpan sq, sk, sv, so;
};

template <int DH, int MR>
struct DecSmem {
    union {
        struct {
            float k[stages_of<DH>()][TK * DH];
            float v[stages_of<DH>()][TK * DH];
        } ring;
        struct {
            float m[kGroups][MR];
            float l[kGroups][MR];
            float o[kGroups][MR][DH];
        } merge;
    } u;
    int64_t off[2][SC];                 // paged: row index of each key of a sub-chunk (-1: none)
    float newref[kGroups][MR];          // a group's new reference maxima when one moves
    int last;                           // this CTA merges the entry's chunks
};

__device__ unsigned int g_status = 0;

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Head-dimension index of slot x (0 .. DH/8-1) of lane l8 of a key group.
template <int DH>
__device__ __forceinline__ int dim_of(int l8, int x) { return (x >> 2) * 32 + l8 * 4 + (x & 3); }

// The (key, row) pair index (kk * MR + m) that slot x of lane l8 finishes
// after the reduce-scatter of P values over 8 lanes: each round with lane bit
// b set keeps the upper half of the values left.
template <int P>
__device__ __forceinline__ int own_pair(int l8, int x) {
    int idx = x, c = P;
#pragma unroll
    for (int bit = 4; bit >= 1; bit >>= 1) {
        if (c > 1) {
            c /= 2;
            if (l8 & bit) idx += c;
        }
    }
    return idx;
}

// Row index (paged) of key n of sequence `seq`, head `head`; -1 when the key
// is past the sequence or its block id is out of range.
__device__ __forceinline__ int64_t paged_row(const DecodeParams& p, int64_t seq, int64_t head,
                                             int64_t n, int64_t len) {
    if (n >= len) return -1;
    const int64_t bp = n / p.block_size;
    const int64_t blk = p.table[seq * p.max_blocks + bp];
    if (blk < 0 || blk >= p.num_blocks) {
        record_status(&g_status, kPagedInput);
        return -1;
    }
    return (blk * p.block_size + (n - bp * p.block_size)) * p.n_kv_heads + head;
}

// Counts one chunk of an entry in and reports whether it was the last.  A
// counter holds (epoch << 16) | arrivals; one whose epoch is not this call's
// (left over from an earlier call, or whatever the workspace held) counts as
// zero, so the counters need no clearing.  Every failed compare-and-swap
// means another chunk of the entry got in, so the loop ends within `chunks`
// tries; the bound only guards against a corrupted workspace.
__device__ __forceinline__ bool arrive(unsigned long long* ctr, unsigned long long epoch, int chunks) {
    unsigned long long old = atomicAdd(ctr, 0ull);
    for (int it = 0; it < (1 << 20); ++it) {
        const unsigned long long cnt = (old >> 16) == epoch ? (old & 0xFFFFull) : 0ull;
        const unsigned long long seen = atomicCAS(ctr, old, (epoch << 16) | (cnt + 1));
        if (seen == old) return cnt + 1 == (unsigned long long)chunks;
        old = seen;
    }
    record_status(&g_status, kWaitPartial);
    return false;
}

// One work item: chunk `chunk` of batch entry b.
template <int DH, int MR, bool PAGED>
__device__ __forceinline__ void decode_item(const DecodeParams& p, DecSmem<DH, MR>& sh, const int64_t b,
                                            const int chunk) {
    constexpr int X = DH / 8;            // head-dimension slots per lane
    constexpr int PIECES = TK * DH / 4;  // 16-byte pieces of K (or V) per tile
    constexpr int kStages = stages_of<DH>();
    constexpr int KK = TK / kGroups;     // keys of a tile per lane group
    constexpr int P = KK * MR;           // (key, row) pairs of a group per tile
    constexpr int CF = P >= 8 ? P / 8 : 1;   // pairs each lane finishes
    constexpr int REP = P >= 8 ? 1 : 8 / P;  // lanes holding each finished pair
    const int t = threadIdx.x;
    const int grp = t >> 3, l8 = t & 7;

    int64_t len = p.N, seq = 0, head = 0;
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
    const int64_t kb = (int64_t)chunk * p.chunk_keys;
    const int64_t ke = min(kb + p.chunk_keys, len);
    const int64_t nkeys = ke > kb ? ke - kb : 0;
    const int tiles = (int)((nkeys + TK - 1) / TK);
    const float* Kb = PAGED ? p.K : p.K + b * p.bsK;
    const float* Vb = PAGED ? p.V : p.V + b * p.bsV;

    // Query rows in registers (rows past M are zero and never stored).
    float q[MR][X];
#pragma unroll
    for (int m = 0; m < MR; ++m) {
#pragma unroll
        for (int x = 0; x < X; ++x) {
            const float* a = p.Q + b * p.bsQ + (int64_t)m * p.rsQ + (int64_t)dim_of<DH>(l8, x) * p.csQ;
            q[m][x] = (m < p.M && dbg_in_span(p.Q, a, p.sq, &g_status)) ? *a : 0.0f;
        }
    }

    // Row offsets of sub-chunk 0 (paged).
    [[maybe_unused]] int32_t look[SC / kThreads];   // raw block-table entries of the next sub-chunk
    if constexpr (PAGED) {
#pragma unroll
        for (int r = 0; r < SC / kThreads; ++r) {
            const int j = t + r * kThreads;
            sh.off[0][j] = j < nkeys ? paged_row(p, seq, head, kb + j, len) : -1;
        }
        __syncthreads();
    }

    auto issue = [&](int tile) {
        if (tile < tiles) {
            const int slot = tile % kStages;
#pragma unroll
            for (int it = 0; it < PIECES / kThreads; ++it) {
                const int idx = t + it * kThreads;
                const int j = idx / (DH / 4), c = idx % (DH / 4);
                const int64_t kj = (int64_t)tile * TK + j;          // key within the chunk
                const float* ks = p.K;
                const float* vs = p.V;
                bool ok;
                if constexpr (PAGED) {
                    const int64_t row = sh.off[(tile / kTilesPerSub) & 1][kj % SC];
                    ok = row >= 0;
                    if (ok) {
                        ks = Kb + row * DH + 4 * c;
                        vs = Vb + row * DH + 4 * c;
                    }
                } else {
                    const int64_t n = kb + kj;
                    ok = kj < nkeys;
                    if (ok) {
                        ks = Kb + n * p.rsK + 4 * c;
                        vs = Vb + n * p.rsV + 4 * c;
                    }
                }
                ok = ok && dbg_in_span(p.K, ks, p.sk, &g_status) && dbg_in_span(p.V, vs, p.sv, &g_status) &&
                     dbg_in_span(p.K, ks + 3, p.sk, &g_status) && dbg_in_span(p.V, vs + 3, p.sv, &g_status);
                cp_async16(&sh.u.ring.k[slot][j * DH + 4 * c], ok ? ks : p.K, ok);
                cp_async16(&sh.u.ring.v[slot][j * DH + 4 * c], ok ? vs : p.V, ok);
            }
        }
        cp_async_commit();
    };

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) issue(s);

    // Softmax state.  Every lane of a group holds O's slice of every row and
    // each row's reference maximum (mref); after the reduce-scatter of a tile's
    // scores each lane finishes CF of the group's P (key, row) pairs, always
    // the same rows, and keeps the running sums of those rows (lsum).
    float2 o[MR][X / 2];         // (slot 2y, slot 2y+1) of each row: packed FMAs
    float mref[MR];
    float mown[CF], lsum[CF];
    int64_t pos_own[CF];
#pragma unroll
    for (int m = 0; m < MR; ++m) {
        mref[m] = -INFINITY;
#pragma unroll
        for (int y = 0; y < X / 2; ++y) o[m][y] = make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int i = 0; i < CF; ++i) {
        const int m = own_pair<P>(l8, i) % MR;
        mown[i] = -INFINITY;
        lsum[i] = 0.0f;
        pos_own[i] = p.causal ? (m % p.q_len) + len - p.q_len : len - 1;
    }

    for (int i = 0; i < tiles; ++i) {
        cp_async_wait<kStages - 2>();
        __syncthreads();          // tile i is in; every thread is done with tile i-1's slot
        if constexpr (PAGED) {
            // Row offsets of the next sub-chunk: its block-table entries are
            // loaded at its predecessor's start (nothing waits on them then),
            // turned into row offsets and stored at the middle, and first used
            // kStages-1 tiles before its own start.
            const int sub = i / kTilesPerSub, ph = i % kTilesPerSub;
            if (ph == 0) {
#pragma unroll
                for (int r = 0; r < SC / kThreads; ++r) {
                    const int64_t n = kb + (int64_t)(sub + 1) * SC + t + r * kThreads;
                    look[r] = n < ke ? p.table[seq * p.max_blocks + n / p.block_size] : -1;
                }
            } else if (ph == kTilesPerSub / 2) {
#pragma unroll
                for (int r = 0; r < SC / kThreads; ++r) {
                    const int64_t n = kb + (int64_t)(sub + 1) * SC + t + r * kThreads;
                    int64_t row = -1;
                    if (n < ke) {
                        const int64_t blk = look[r];
                        if (blk >= 0 && blk < p.num_blocks)
                            row = (blk * p.block_size + n % p.block_size) * p.n_kv_heads + head;
                        else
                            record_status(&g_status, kPagedInput);
                    }
                    sh.off[(sub + 1) & 1][t + r * kThreads] = row;
                }
            }
        }
        issue(i + kStages - 1);

        const int slot = i % kStages;
        // This group's KK keys of the tile: K and V slices, then the P partial
        // dot products (key kk, row m) at index kk * MR + m.
        float kv[KK][X], vv[KK][X];
#pragma unroll
        for (int kk = 0; kk < KK; ++kk) {
            const int j = grp + kk * kGroups;
#pragma unroll
            for (int r = 0; r < X / 4; ++r) {
                const float4 a = *reinterpret_cast<const float4*>(&sh.u.ring.k[slot][j * DH + r * 32 + l8 * 4]);
                const float4 c = *reinterpret_cast<const float4*>(&sh.u.ring.v[slot][j * DH + r * 32 + l8 * 4]);
                kv[kk][4 * r] = a.x; kv[kk][4 * r + 1] = a.y; kv[kk][4 * r + 2] = a.z; kv[kk][4 * r + 3] = a.w;
                vv[kk][4 * r] = c.x; vv[kk][4 * r + 1] = c.y; vv[kk][4 * r + 2] = c.z; vv[kk][4 * r + 3] = c.w;
            }
        }
        // Packed FMAs (fma.rn.f32x2): two rows at a time against one key
        // slot, or, with one row, the even and odd slots as two sums.
        float v[P];
#pragma unroll
        for (int kk = 0; kk < KK; ++kk) {
            if constexpr (MR >= 2) {
#pragma unroll
                for (int mp = 0; mp < MR / 2; ++mp) {
                    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int x = 0; x < X; ++x)
                        acc = __ffma2_rn(make_float2(q[2 * mp][x], q[2 * mp + 1][x]),
                                         make_float2(kv[kk][x], kv[kk][x]), acc);
                    v[kk * MR + 2 * mp] = acc.x;
                    v[kk * MR + 2 * mp + 1] = acc.y;
                }
            } else {
                float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int y = 0; y < X / 2; ++y)
                    acc = __ffma2_rn(make_float2(q[0][2 * y], q[0][2 * y + 1]),
                                     make_float2(kv[kk][2 * y], kv[kk][2 * y + 1]), acc);
                v[kk] = acc.x + acc.y;
            }
        }
        // Reduce-scatter across the 8 lanes: each round halves the values a
        // lane keeps (the half its lane bit selects) and adds its partner's
        // other half; once one value is left the rounds are plain sums.
        {
            int c = P;
#pragma unroll
            for (int bit = 4; bit >= 1; bit >>= 1) {
                if (c > 1) {
                    const int half = c / 2;
                    const bool up = (l8 & bit) != 0;
#pragma unroll
                    for (int x = 0; x < half; ++x) {
                        const float lo = v[x], hi = v[x + half];
                        const float mine = up ? hi : lo, other = up ? lo : hi;
                        v[x] = mine + __shfl_xor_sync(0xffffffffu, other, bit);
                    }
                    c = half;
                } else {
                    v[0] += __shfl_xor_sync(0xffffffffu, v[0], bit);
                }
            }
        }
        // The lane's own pairs: mask, scale, and the row maximum over the
        // tile's two keys of the row (the partner lane across bit 2 holds the
        // other key).
        float sc[CF], rmax[CF];
        bool raise = false;
#pragma unroll
        for (int x = 0; x < CF; ++x) {
            const int kk = own_pair<P>(l8, x) / MR;
            const int64_t n = kb + (int64_t)i * TK + grp + kk * kGroups;
            sc[x] = (n < ke && n <= pos_own[x]) ? v[x] * p.scale_log2 : -INFINITY;
            rmax[x] = fmaxf(sc[x], __shfl_xor_sync(0xffffffffu, sc[x], 4));
            raise |= rmax[x] > mown[x] + kRaise;
        }
        // A row's maximum passed its reference by 2^8 (or the first kept key):
        // move the reference there and scale the row's sums and O (rare, warp
        // uniform).
        if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
            for (int x = 0; x < CF; ++x) {
                const int m = own_pair<P>(l8, x) % MR;
                const float nr = rmax[x] > mown[x] + kRaise ? rmax[x] : mown[x];
                sh.newref[grp][m] = nr;         // every owner of the row writes the same value
            }
            __syncwarp();
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                const float nr = sh.newref[grp][m];
                if (nr > mref[m]) {
                    const float corr = ex2_approx(mref[m] - nr);
#pragma unroll
                    for (int y = 0; y < X / 2; ++y) {
                        o[m][y].x *= corr;
                        o[m][y].y *= corr;
                    }
                    mref[m] = nr;
                }
            }
#pragma unroll
            for (int x = 0; x < CF; ++x) {
                const float nr = sh.newref[grp][own_pair<P>(l8, x) % MR];
                if (nr > mown[x]) {
                    lsum[x] *= ex2_approx(mown[x] - nr);
                    mown[x] = nr;
                }
            }
            __syncwarp();
        }
        float pr[CF];
#pragma unroll
        for (int x = 0; x < CF; ++x) {
            pr[x] = sc[x] == -INFINITY ? 0.0f : ex2_approx(sc[x] - mown[x]);
            lsum[x] += pr[x];
        }
        // O += P V: every pair's probability from the lane that finished it.
        const int gbase = (t & 31) & ~7;
#pragma unroll
        for (int idx = 0; idx < P; ++idx) {
            const float pv = __shfl_sync(0xffffffffu, pr[idx % CF], gbase + (idx / CF) * REP);
            const int kk = idx / MR, m = idx % MR;
#pragma unroll
            for (int y = 0; y < X / 2; ++y)
                o[m][y] = __ffma2_rn(make_float2(pv, pv), make_float2(vv[kk][2 * y], vv[kk][2 * y + 1]), o[m][y]);
        }
    }
    cp_async_wait<0>();
    __syncthreads();              // the ring is free for the merge

    // Merge the lane groups.  A row's sum is its two key lanes' (across bit
    // 2); one owner writes it (copies made by the plain-sum rounds are equal).
#pragma unroll
    for (int x = 0; x < CF; ++x) {
        const float l = lsum[x] + __shfl_xor_sync(0xffffffffu, lsum[x], 4);
        if ((l8 & 4) == 0 && (l8 & (REP - 1)) == 0) {
            const int m = own_pair<P>(l8, x) % MR;
            sh.u.merge.m[grp][m] = mown[x];
            sh.u.merge.l[grp][m] = l;
        }
    }
#pragma unroll
    for (int m = 0; m < MR; ++m)
#pragma unroll
        for (int y = 0; y < X / 2; ++y) {
            sh.u.merge.o[grp][m][dim_of<DH>(l8, 2 * y)] = o[m][y].x;
            sh.u.merge.o[grp][m][dim_of<DH>(l8, 2 * y + 1)] = o[m][y].y;
        }
    __syncthreads();

    const int64_t rows = p.M < MR ? p.M : MR;
    for (int idx = t; idx < rows * DH; idx += kThreads) {
        const int m = idx / DH, e = idx % DH;
        float mx = -INFINITY;
#pragma unroll
        for (int g = 0; g < kGroups; ++g) mx = fmaxf(mx, sh.u.merge.m[g][m]);
        float l = 0.0f, acc = 0.0f;
        if (mx != -INFINITY) {
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
                const float gm = sh.u.merge.m[g][m];
                if (gm == -INFINITY) continue;
                const float w = exp2f(gm - mx);
                l = fmaf(sh.u.merge.l[g][m], w, l);
                acc = fmaf(sh.u.merge.o[g][m][e], w, acc);
            }
        }
        if (p.chunks == 1) {
            float* a = p.O + b * p.bsO + (int64_t)m * p.rsO + (int64_t)e * p.csO;
            if (dbg_in_span(p.O, a, p.so, &g_status)) *a = acc / l;
        } else {
            float* rec = p.part + ((b * p.chunks + chunk) * MR + m) * (int64_t)(2 + DH);
            if (e == 0) {
                rec[0] = mx;
                rec[1] = l;
            }
            rec[2 + e] = acc;
        }
    }
    if (p.chunks == 1) return;

    // The last chunk of the entry to finish merges all of them, in chunk
    // order, so the result does not depend on which one that is.
    __threadfence();              // this thread's part of the record is visible GPU-wide
    __syncthreads();
    if (t == 0) {
        sh.last = arrive(p.counters + b, p.epoch, p.chunks) ? 1 : 0;
    }
    __syncthreads();
    if (!sh.last) return;
    __threadfence();
    for (int idx = t; idx < rows * DH; idx += kThreads) {
        const int m = idx / DH, e = idx % DH;
        const float* rec0 = p.part + (b * p.chunks * MR + m) * (int64_t)(2 + DH);
        const int64_t cstride = (int64_t)MR * (2 + DH);
        float mx = -INFINITY;
        for (int c = 0; c < p.chunks; ++c) mx = fmaxf(mx, __ldcg(rec0 + c * cstride));
        float l = 0.0f, acc = 0.0f;
        for (int c = 0; c < p.chunks; ++c) {
            const float* rec = rec0 + c * cstride;
            const float cm = __ldcg(rec);
            if (cm == -INFINITY) continue;
            const float w = exp2f(cm - mx);
            l = fmaf(__ldcg(rec + 1), w, l);
            acc = fmaf(__ldcg(rec + 2 + e), w, acc);
        }
        float* a = p.O + b * p.bsO + (int64_t)m * p.rsO + (int64_t)e * p.csO;
        if (dbg_in_span(p.O, a, p.so, &g_status)) *a = acc / l;
    }
}

// One CTA per (entry, chunk): blockIdx.x the entry, blockIdx.y the chunk.
template <int DH, int MR, bool PAGED>
__global__ void __launch_bounds__(kThreads, min_ctas_of<DH, MR>()) attention_decode_kernel(const DecodeParams p) {
    extern __shared__ float4 smem4[];
    DecSmem<DH, MR>& sh = *reinterpret_cast<DecSmem<DH, MR>*>(smem4);
    decode_item<DH, MR, PAGED>(p, sh, blockIdx.x, (int)blockIdx.y);
}

template <int DH, int MR, bool PAGED>
cudaError_t launch_cfg(const DecodeParams& p, int64_t batch, cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    constexpr int kSmem = (int)sizeof(DecSmem<DH, MR>);
    if (!(attr_done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(attention_decode_kernel<DH, MR, PAGED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    const dim3 grid((unsigned)batch, (unsigned)p.chunks);
    attention_decode_kernel<DH, MR, PAGED><<<grid, kThreads, kSmem, stream>>>(p);
    return cudaGetLastError();
}

template <bool PAGED>
cudaError_t launch_dh(const DecodeParams& p, int64_t D, int mr, int64_t batch, cudaStream_t stream) {
    switch (D) {
        case 32: return mr == 1 ? launch_cfg<32, 1, PAGED>(p, batch, stream)
                      : mr == 4 ? launch_cfg<32, 4, PAGED>(p, batch, stream)
                                : launch_cfg<32, 8, PAGED>(p, batch, stream);
        case 64: return mr == 1 ? launch_cfg<64, 1, PAGED>(p, batch, stream)
                      : mr == 4 ? launch_cfg<64, 4, PAGED>(p, batch, stream)
                                : launch_cfg<64, 8, PAGED>(p, batch, stream);
        case 96: return mr == 1 ? launch_cfg<96, 1, PAGED>(p, batch, stream)
                                : launch_cfg<96, 4, PAGED>(p, batch, stream);
        case 128: return mr == 1 ? launch_cfg<128, 1, PAGED>(p, batch, stream)
                                 : launch_cfg<128, 4, PAGED>(p, batch, stream);
        default: return cudaErrorInvalidValue;
    }
}

// Rows per instantiation for M rows at head dimension D (0: none fits).
int rows_config(int64_t M, int64_t D) {
    const int cap = D <= 64 ? 8 : 4;
    if (M <= 1) return 1;
    if (M <= 4) return 4;
    if (M <= cap) return cap;
    return 0;
}

}  // namespace

bool attention_decode_supported(const AttnProblem& a) {
    if (!(a.D == a.Dv && (a.D == 32 || a.D == 64 || a.D == 96 || a.D == 128))) return false;
    if (rows_config(a.M, a.D) == 0) return false;
    if (a.batch >= 65536 * 32768LL) return false;
    auto a16 = [](const void* x) { return reinterpret_cast<uintptr_t>(x) % 16 == 0; };
    if (a.paged) return a16(a.K) && a16(a.V);
    // Rows of K and V contiguous along the head dimension, every row 16-byte aligned.
    return a.csK == 1 && a.csV == 1 && a16(a.K) && a16(a.V) && a.rsK % 4 == 0 && a.rsV % 4 == 0 &&
           (a.batch == 1 || (a.bsK % 4 == 0 && a.bsV % 4 == 0));
}

cudaError_t launch_attention_decode(const AttnProblem& a, cudaStream_t stream) {
    if (!attention_decode_supported(a)) return cudaErrorInvalidValue;
    const int mr = rows_config(a.M, a.D);
    DecodeParams p{};
    p.Q = a.Q; p.rsQ = a.rsQ; p.csQ = a.csQ; p.bsQ = a.bsQ;
    p.K = a.K; p.rsK = a.rsK; p.bsK = a.bsK;
    p.V = a.V; p.rsV = a.rsV; p.bsV = a.bsV;
    p.O = a.O; p.rsO = a.rsO; p.csO = a.csO; p.bsO = a.bsO;
    p.M = a.M; p.N = a.N;
    p.scale_log2 = a.alpha * 1.4426950408889634f;
    p.causal = a.causal;
    p.q_len = a.causal ? a.q_len : a.M;
    p.table = a.table; p.seq_lens = a.seq_lens;
    p.max_blocks = a.max_blocks; p.block_size = a.block_size;
    p.n_kv_heads = a.n_kv_heads; p.num_blocks = a.num_blocks;
    p.sq = a.sq; p.sk = a.sk; p.sv = a.sv; p.so = a.so;

    // Chunks: about four CTAs per SM in all (longer chunks lose less to each
    // CTA's start-up, measured against eight per SM on ragged decode
    // batches), each at least 4 tiles, as many as the workspace holds; one
    // chunk per entry without one.  Workspace: one counter per entry, then
    // the chunks' records.
    int sms = 152;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) {
        if (const DeviceProps* d = device_props(dev)) sms = d->sm_count;
    }
    cudaGetLastError();
    const int64_t target = (int64_t)sms * 4;
    int64_t chunks = std::max<int64_t>(1, (target + a.batch - 1) / a.batch);
    chunks = std::min<int64_t>(chunks, std::max<int64_t>(1, a.N / (4 * TK)));
    const int64_t rec_bytes = (int64_t)mr * (2 + a.D) * (int64_t)sizeof(float);
    const int64_t ctr_bytes = (a.batch * 8 + 255) / 256 * 256;
    const int64_t fit = a.workspace && (int64_t)a.workspace_bytes > ctr_bytes
                            ? ((int64_t)a.workspace_bytes - ctr_bytes) / (rec_bytes * a.batch)
                            : 0;
    if (chunks > fit) chunks = fit >= 2 ? fit : 1;
    chunks = std::min<int64_t>(chunks, 65535);
    int64_t ck = (a.N + chunks - 1) / chunks;
    ck = (ck + TK - 1) / TK * TK;
    chunks = (a.N + ck - 1) / ck;
    p.chunk_keys = ck;
    p.chunks = (int)chunks;
    p.counters = chunks > 1 ? static_cast<unsigned long long*>(a.workspace) : nullptr;
    p.part = chunks > 1 ? reinterpret_cast<float*>(static_cast<char*>(a.workspace) + ctr_bytes) : nullptr;
    static std::atomic<unsigned long long> next_epoch{1};
    p.epoch = next_epoch.fetch_add(1) & ((1ull << 48) - 1);
    return a.paged ? launch_dh<true>(p, a.D, mr, a.batch, stream)
                   : launch_dh<false>(p, a.D, mr, a.batch, stream);
}

unsigned int read_and_clear_status_attention_decode(cudaStream_t stream) {
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
