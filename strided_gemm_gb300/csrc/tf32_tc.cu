// TF32 tensor-core path (opt-in through sbgemm_options.math): tcgen05.mma
// kind::tf32 with fp32 accumulators in tensor memory.  The MMAs read both
// operands K-major (unit stride along K); one operand whose unit stride runs
// along M or N is transposed in shared memory on the way by four transposer
// warps (raw 32 x 32 boxes -> the K-major swizzled layout).
//
// Persistent, warp-specialised CTAs, one per SM, 192 threads:
//  * warp 0, one lane: TMA producer.  Walks the CTA's tiles and their 32-deep
//    K slices and loads a 128 x 32 box of A and a 256 x 32 box of B (128-byte
//    swizzle) into a 4-stage shared-memory ring ("full" / "empty" mbarriers).
//  * warp 1, one lane: MMA issuer.  Allocates 512 TMEM columns (two 128 x 256
//    fp32 accumulators), and per slice issues four 128x256x8 MMAs whose smem
//    descriptors advance 32 bytes along the swizzled rows; tcgen05.commit frees
//    the stage when its MMAs are done, and marks the accumulator full after the
//    tile's last slice.
//  * warps 2..5: epilogue.  Each warp reads its 32 TMEM lanes (rows) in 32-
//    column pieces (tcgen05.ld 32x32b.x32), stages each piece in shared
//    memory, and writes alpha*acc (+ C_old), with the fused addend and
//    activation if any, in 128-byte rows with masks on ragged M / N; then it
//    releases the accumulator, so the next tile's MMAs overlap these stores.
// With a workspace, tiles are split along K across the grid as independent
// pieces (the work list of schedule.cuh shared with the FFMA kernel): the last
// waves when there are at least as many tiles as SMs, all tiles otherwise.
// Every piece accumulates from zero, so no MMA ever waits for another CTA; a
// head or middle piece leaves its accumulator in the workspace, and the tail
// piece's epilogue adds the earlier pieces' partial sums, latest CTA first,
// after loading its own.  Results are deterministic but rounded differently
// from the unsplit tile.
// Every mbarrier wait is bounded; a role that gives up records a status code
// and leaves its loop, the producer then waits (bounded) for the copies it
// issued, the MMA issuer for its MMAs, and the allocating warp frees TMEM
// before the CTA exits.
//
// TF32 reads the top 19 bits of each fp32 operand; products accumulate in fp32.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "debug_check.cuh"
#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "schedule.cuh"

namespace sbg {
namespace {

constexpr int BM = 128, BN = 256, BK = 32;   // CTA tile; UMMA 128 x 256 x 8
constexpr int kMmaK = 8;                     // tf32 elements per MMA
constexpr int kABytes = BM * BK * 4;         // 16 KB
constexpr int kBBytes = BN * BK * 4;         // 32 KB
constexpr uint32_t kAccCols = BN;            // fp32 accumulator: one column per n
constexpr uint32_t kTmemCols = 2 * kAccCols; // double-buffered accumulator
constexpr int kEpiWarps = 4;
constexpr int kTransWarps = 4;               // transposers of the MN-major operands
constexpr int kBM128 = BM;                               // rows of a partial slot
constexpr int64_t kSlotFloat4 = (int64_t)BM * BN / 4;    // one partial tile, in float4
constexpr int kBox = 32 * 32;                // floats in one 32 x 32 raw box of an MN-major operand
constexpr int kPairVariant = 1;              // Plan::variant of the CTA-pair kernel
static_assert((size_t)kSlotFloat4 * sizeof(float4) + sizeof(unsigned int) == kWorkspaceBytesPerSm,
              "a partial tile and a flag per CTA fit the workspace sbgemm_workspace_bytes reports");

// Shared-memory plan by operand orientation.  MN: 0 both operands K-major;
// 1 A MN-major (unit stride along M); 2 B MN-major (along N); 3 both.  An
// MN-major slice lands as raw 32 x 32 boxes (rows along K, 128-byte swizzle)
// in a ring of its own (with both MN-major, A's boxes and then B's share one
// raw stage), and the transposer warps rewrite it into the K-major swizzled
// layout the MMAs read, in a ring of kTStages stages; an operand TMA brings
// in K-major has a ring of kStages stages.  The load latency is what the
// stages cover (each waits out about 1.1-1.3 us of it), so the TMA-fed rings
// get the depth and the transposed ring, filled from shared memory, two
// stages (3 transposed stages with 2 raw ones measured 11% slower).  With
// both operands MN-major a raw stage holds 48 KB and the shared memory has
// room for four such stages: 2 raw and 2 transposed measured 8% faster than
// 3 raw and 1 transposed (which makes the transposers wait on the MMAs).
// MN 4: both operands K-major on a CTA pair (cta_group::2): a 256 x 256 tile
// of which each CTA loads 128 rows of A and 128 of B's 256 columns and holds
// 128 rows of the accumulator; a stage is then 32 KB, so six fit.
template <int MN>
struct TCfg {
    static constexpr bool kPair = MN == 4;
    static constexpr bool kTA = MN == 1 || MN == 3, kTB = MN == 2 || MN == 3;
    static constexpr bool kTrans = kTA || kTB;
    static constexpr bool kKRing = !(kTA && kTB);          // an operand comes in K-major
    static constexpr int kWarps = 2 + kEpiWarps + (kTrans ? kTransWarps : 0);
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kStages = kPair ? 6 : 4;          // TMA-fed K-major ring
    static constexpr int kBRows = kPair ? BN / 2 : BN;     // rows of B (columns of C) a CTA loads
    static constexpr int kTStages = kTrans ? 2 : 1;        // transposed ring
    static constexpr int kStagesA = kTA ? kTStages : kStages;
    static constexpr int kStagesB = kTB ? kTStages : kStages;
    static constexpr int kRawRowsA = kTA ? BM : 0;         // A's rows lead a raw stage
    static constexpr int kRawRows = kRawRowsA + (kTB ? BN : 0);
    static constexpr int kRawStages = (kTA && kTB) ? 2 : (kTA ? 3 : (kTB ? 2 : 0));
    static constexpr int kStageBufs = kTrans ? 1 : 2;     // epilogue staging tiles per warp
    // Bytes the K-major operand copies bring into a stage.
    static constexpr uint32_t kKBytes = (kTA ? 0 : kABytes) + (kTB ? 0 : (uint32_t)kBRows * BK * 4);
    static constexpr uint32_t kRawBytes = kRawRows * BK * 4;
    static constexpr int kRawSlots = kRawStages > 0 ? kRawStages : 1;
    static constexpr int kRawFloats = kRawRows > 0 ? kRawRows * BK : 4;
    struct Smem {
        float a[kStagesA][BM * BK];
        float b[kStagesB][kBRows * BK];
        // Per epilogue warp: pieces of C (alternating by store when there are
        // two) in the 128-byte swizzled layout of its tensor map (16-byte chunk
        // q of row r at chunk q ^ (r & 7)).
        alignas(1024) float stage[kEpiWarps][kStageBufs][32 * 32];
        alignas(1024) float raw[kRawSlots][kRawFloats];
        uint64_t full[kStages];       // the K-major operand of stage s landed
        uint64_t empty[kStages];      // the MMAs that read it are done
        uint64_t tdone[kTStages];     // the transposers wrote transposed stage t
        uint64_t tempty[kTStages];    // the MMAs that read it are done
        uint64_t rfull[kRawSlots];
        uint64_t rempty[kRawSlots];
        uint64_t acc_full[2];
        uint64_t acc_empty[2];
        uint64_t mma_done;
        uint64_t stored;          // every epilogue thread wrote its head partial
        uint64_t c_old[kEpiWarps];   // a warp's C_old piece landed in its staging tile
        Schedule sched;
        uint32_t tmem_base;
    };
    static constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static_assert(kKRing == (kKBytes > 0), "the K-major ring carries an operand");
    static_assert(kRawBytes % 4096 == 0, "raw slices are whole 32 x 32 boxes");
};

__device__ unsigned int g_wait_status = 0;

struct Params {
    float* C;
    int64_t rsC, csC, bsC;
    int64_t M, N, K;
    int64_t tiles_m, tiles_n, tiles_total;
    int nk;
    float alpha;
    int accumulate;
    int a_bcast, b_bcast;
    int c_tma;                    // C goes out through its tensor map: 1 unit stride along N, 2 along M
    int a_blk4, b_blk4;           // the MN-major operand's map is rank 4: a slice's boxes in one copy
    int pair;                     // CTA-pair kernel: tiles of 2 BM rows, this CTA's half by its rank
    int64_t dp_tiles, sk_units;   // work list (see schedule.cuh)
    EpiParams epi;                // fused epilogue (epilogue.cuh); epi.on == 0: none
    float4* ws_partial;           // [grid][8 chunks][8 quads][128 rows] partial sums
    unsigned int* ws_flag;        // [grid] partial-ready flags, zeroed before launch
    ElemSpan sc;                  // debug builds: C's valid element offsets
};


// Instruction descriptor, kind::tf32: D fp32, A and B tf32, both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24.  N is set per tile (idesc_for).
constexpr uint32_t kIdescNoN = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(BM >> 4) << 24);

// The MMA width for a tile whose first column is n0: BN, or at a ragged N
// edge the valid columns rounded up to the 16 an M = 128 MMA takes.  The
// accumulator columns past it keep stale values that no store reads.
__device__ __forceinline__ uint32_t idesc_for(int64_t N, int64_t n0) {
    const int64_t nv = N - n0;
    const uint32_t nn = nv >= BN ? (uint32_t)BN : (uint32_t)((nv + 15) & ~(int64_t)15);
    return kIdescNoN | ((nn >> 3) << 17);
}

// Raw 32-row boxes of an MN-major tile that hold valid rows (ext of them).
template <int ROWS>
__device__ __forceinline__ int valid_boxes(int64_t ext) {
    return ext >= ROWS ? ROWS / 32 : (int)((ext + 31) / 32);
}

struct TileCoord { int64_t b, m0, n0; };

__device__ __forceinline__ TileCoord tile_coord(const Params& p, int64_t t) {
    const int64_t per_batch = p.tiles_m * p.tiles_n;
    const int64_t b = t / per_batch;
    const int64_t r = t - b * per_batch;
    constexpr int64_t G = 8;
    const int64_t group = r / (G * p.tiles_n);
    const int64_t first_m = group * G;
    const int64_t gm = (p.tiles_m - first_m < G) ? (p.tiles_m - first_m) : G;
    const int64_t w = r - group * G * p.tiles_n;
    const int64_t tm = p.pair ? 2 * BM : BM;
    const int64_t sub = p.pair ? (int64_t)BM * (cluster_rank() & 1) : 0;
    return {b, (first_m + w % gm) * tm + sub, (w / gm) * BN};
}

template <int MN>
__device__ __forceinline__ void producer(typename TCfg<MN>::Smem& sh, const CUtensorMap* ta,
                                         const CUtensorMap* tb, const Params& p) {
    using C = TCfg<MN>;
    constexpr int S = C::kStages, R = C::kRawSlots;
    uint64_t i = 0;   // slices issued
    bool ok = true;
    const int64_t n_items = sh.sched.n_items;
    for (int64_t w = 0; w < n_items && ok; ++w) {
        const Item itm = sh.sched.item(w, p.nk);
        const TileCoord tc = tile_coord(p, itm.tile);
        const int ba = p.a_bcast ? 0 : (int)tc.b;
        const int bb = p.b_bcast ? 0 : (int)tc.b;
        for (int kt = itm.kb; kt < itm.ke; ++kt, ++i) {
            if constexpr (C::kTrans) {
                // An MN-major operand: 32 x 32 boxes along M (A) or N (B), rows
                // along K, into the raw ring (A's boxes first when both are).
                const int r = (int)(i % R);
                if (i >= (uint64_t)R && !mbar_wait(&sh.rempty[r], (uint32_t)(((i / R) - 1) & 1))) {
                    record_status(&g_wait_status, kWaitEmpty);
                    ok = false;
                    break;
                }
                // With a rank-4 map (the extent a multiple of 32) one copy
                // brings all of a slice's boxes, those past a ragged edge
                // zero-filled; otherwise boxes wholly past the edge are not
                // fetched.
                const int boxes_a = C::kTA ? (p.a_blk4 ? BM / 32 : valid_boxes<BM>(p.M - tc.m0)) : 0;
                const int boxes_b = C::kTB ? (p.b_blk4 ? BN / 32 : valid_boxes<BN>(p.N - tc.n0)) : 0;
                mbar_arrive_expect_tx(&sh.rfull[r], (uint32_t)(boxes_a + boxes_b) * kBox * 4);
                float* raw_b = sh.raw[r] + (C::kRawRowsA / 32) * kBox;
                if constexpr (C::kTA) {
                    if (p.a_blk4) {
                        tma_load_4d(sh.raw[r], ta, &sh.rfull[r], 0, kt * BK, (int)(tc.m0 / 32), ba);
                    } else {
#pragma unroll 1
                        for (int j = 0; j < boxes_a; ++j)
                            tma_load_3d(sh.raw[r] + j * kBox, ta, &sh.rfull[r], (int)tc.m0 + 32 * j, kt * BK, ba);
                    }
                }
                if constexpr (C::kTB) {
                    if (p.b_blk4) {
                        tma_load_4d(raw_b, tb, &sh.rfull[r], 0, kt * BK, (int)(tc.n0 / 32), bb);
                    } else {
#pragma unroll 1
                        for (int j = 0; j < boxes_b; ++j)
                            tma_load_3d(raw_b + j * kBox, tb, &sh.rfull[r], (int)tc.n0 + 32 * j, kt * BK, bb);
                    }
                }
            }
            if constexpr (C::kKRing) {
                const int st = (int)(i % S);
                // (On a pair the leader's commits free this CTA's stages.)
                if (i >= (uint64_t)S && !mbar_wait(&sh.empty[st], (uint32_t)(((i / S) - 1) & 1))) {
                    record_status(&g_wait_status, kWaitEmpty);
                    ok = false;
                    break;
                }
                if constexpr (C::kPair) {
                    // Both CTAs' copies of a stage complete on the leader's
                    // barrier, which expects the bytes of both.
                    const uint32_t rank = cluster_rank() & 1;
                    if (rank == 0) mbar_arrive_expect_tx(&sh.full[st], 2 * C::kKBytes);
                    const uint32_t bar = cluster_addr(&sh.full[st], 0);
                    tma_load_3d_pair(sh.a[st], ta, bar, kt * BK, (int)tc.m0, ba);
                    tma_load_3d_pair(sh.b[st], tb, bar, kt * BK, (int)tc.n0 + C::kBRows * (int)rank, bb);
                } else {
                    mbar_arrive_expect_tx(&sh.full[st], C::kKBytes);
                    if constexpr (!C::kTA) tma_load_3d(sh.a[st], ta, &sh.full[st], kt * BK, (int)tc.m0, ba);
                    if constexpr (!C::kTB) tma_load_3d(sh.b[st], tb, &sh.full[st], kt * BK, (int)tc.n0, bb);
                }
            }
        }
    }
    // Wait for the copies still landing (on a pair, the leader's barrier
    // counts both CTAs' copies; the peer's own barrier is unused).
    if (C::kPair && (cluster_rank() & 1) != 0) return;
    if constexpr (C::kKRing) {
        for (uint64_t q = i > (uint64_t)S ? i - S : 0; q < i; ++q)
            if (!mbar_wait(&sh.full[q % S], (uint32_t)((q / S) & 1))) {
                record_status(&g_wait_status, kWaitDrain);
                return;
            }
    }
    if constexpr (C::kTrans) {
        for (uint64_t q = i > (uint64_t)R ? i - R : 0; q < i; ++q)
            if (!mbar_wait(&sh.rfull[q % R], (uint32_t)((q / R) & 1))) {
                record_status(&g_wait_status, kWaitDrain);
                return;
            }
    }
}

// Rewrites the raw boxes of one MN-major slice (rows along K, 128-byte
// swizzle) into the K-major swizzled layout of the MMA operand (row m = 32 k
// values, 16-byte chunk c at chunk c ^ (m & 7)), in 4 x 4 quads: four 16-byte
// loads of 4 rows of K, four 16-byte stores of 4 rows of M.  A 16-byte access
// is served a quarter-warp at a time, and the 8 lanes of a quarter take quads
// (mq, kq) with q bits 0..2 = (a, b, c) as mq = (a, b, ..), kq = (c, a^b^d, ..)
// (d = q bit 3): a load reads chunk (mq & 7) ^ (k & 7), whose bits are (a, b,
// mq2 ^ c) up to a constant, and a store writes chunk kq ^ (m & 7), bits (c,
// a^b^d, kq2 ^ a): 8 distinct chunks either way, so neither conflicts.
// Only the first `boxes` boxes are rewritten (the rows past a ragged edge
// are never multiplied into a stored output).
// One 4 x 4 quad q of transpose_mn_slice.
__device__ __forceinline__ void transpose_quad(const float* raw, float* dst, int q) {
    const int kq = ((q >> 2) & 1) | (((q ^ (q >> 1) ^ (q >> 3)) & 1) << 1) |
                   (((q >> 4) & 1) << 2);                    // 4-k group, 0..7
    const int mq = (q & 3) | ((q >> 5) << 2);                // 4-row group
    const float* box = raw + (mq >> 3) * kBox;
    const int mc = mq & 7;                                    // chunk of the box row
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

template <int ROWS>
__device__ __forceinline__ void transpose_mn_slice(const float* raw, float* dst, int t, int boxes) {
    static_assert(BK / 4 == 8 && ROWS % 32 == 0, "8 k groups; whole 32-row boxes");
    constexpr int kStep = kTransWarps * 32;
    if (boxes == ROWS / 32) {
        // Every box: a fixed trip count, unrolled so that all of a thread's
        // loads are in flight together.
#pragma unroll
        for (int q = t; q < ROWS * 2; q += kStep) transpose_quad(raw, dst, q);
    } else {
        const int quads = boxes * 64;     // 32 rows x 32 k per box, in 4 x 4 quads
#pragma unroll 1
        for (int q = t; q < quads; q += kStep) transpose_quad(raw, dst, q);
    }
}

// Transposer warps: per slice, wait for the raw boxes and for the stage's
// previous MMAs, rewrite the MN-major operand (A's boxes, then B's, when both
// are), order the writes before the tensor cores' reads (async proxy), then
// signal the MMA lane and free the raw slot.
template <int MN>
__device__ __forceinline__ void transposer(typename TCfg<MN>::Smem& sh, const Params& p, int t,
                                           int lane) {
    using C = TCfg<MN>;
    constexpr int T = C::kTStages, R = C::kRawSlots;
    uint64_t i = 0;
    const int64_t n_items = sh.sched.n_items;
    for (int64_t w = 0; w < n_items; ++w) {
        const Item itm = sh.sched.item(w, p.nk);
        const TileCoord tc = tile_coord(p, itm.tile);
        const int boxes_a = C::kTA ? valid_boxes<BM>(p.M - tc.m0) : 0;
        const int boxes_b = C::kTB ? valid_boxes<BN>(p.N - tc.n0) : 0;
        for (int kt = itm.kb; kt < itm.ke; ++kt, ++i) {
            const int r = (int)(i % R), ts = (int)(i % T);
            if (!mbar_wait(&sh.rfull[r], (uint32_t)((i / R) & 1))) {
                record_status(&g_wait_status, kWaitFull);
                return;
            }
            if (i >= (uint64_t)T && !mbar_wait(&sh.tempty[ts], (uint32_t)(((i / T) - 1) & 1))) {
                record_status(&g_wait_status, kWaitEmpty);
                return;
            }
            if constexpr (C::kTA) transpose_mn_slice<BM>(sh.raw[r], sh.a[ts], t, boxes_a);
            if constexpr (C::kTB)
                transpose_mn_slice<BN>(sh.raw[r] + (C::kRawRowsA / 32) * kBox, sh.b[ts], t, boxes_b);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sh.tdone[ts]);
                mbar_arrive(&sh.rempty[r]);
            }
        }
    }
}

template <int MN>
__device__ __forceinline__ void mma_issuer(typename TCfg<MN>::Smem& sh, uint32_t tmem, const Params& p) {
    using C = TCfg<MN>;
    constexpr int S = C::kStages;
    uint64_t i = 0;
    bool ok = true;
    const int64_t n_items = sh.sched.n_items;
    for (int64_t w = 0; w < n_items && ok; ++w) {
        const Item itm = sh.sched.item(w, p.nk);
        const uint32_t buf = (uint32_t)(w & 1);
        const uint64_t use = (uint64_t)w >> 1;
        if (use > 0 && !mbar_wait(&sh.acc_empty[buf], (uint32_t)((use - 1) & 1))) {
            record_status(&g_wait_status, kWaitAccFree);
            break;
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * kAccCols;
        const uint32_t idesc = idesc_for(p.N, tile_coord(p, itm.tile).n0);
        for (int kt = itm.kb; kt < itm.ke; ++kt, ++i) {
            const int st = (int)(i % S), ts = (int)(i % C::kTStages);
            if ((C::kKRing && !mbar_wait(&sh.full[st], (uint32_t)((i / S) & 1))) ||
                (C::kTrans && !mbar_wait(&sh.tdone[ts], (uint32_t)((i / C::kTStages) & 1)))) {
                record_status(&g_wait_status, kWaitFull);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sh.a[C::kTA ? ts : st]);
            const uint32_t b0 = smem_u32(sh.b[C::kTB ? ts : st]);
#pragma unroll
            for (int kk = 0; kk < BK / kMmaK; ++kk) {
                const uint64_t ad = umma_desc_kmajor_sw128(a0 + kk * kMmaK * 4);
                const uint64_t bd = umma_desc_kmajor_sw128(b0 + kk * kMmaK * 4);
                const bool acc = kt > itm.kb || kk > 0;
                mma_tf32(d, ad, bd, idesc, acc ? 1u : 0u);
            }
            if constexpr (C::kKRing) mma_commit(&sh.empty[st]);
            if constexpr (C::kTrans) mma_commit(&sh.tempty[ts]);
        }
        if (!ok) break;
        mma_commit(&sh.acc_full[buf]);
    }
    // Nothing may still be writing TMEM when it is freed.
    mma_commit(&sh.mma_done);
    if (!mbar_wait(&sh.mma_done, 0)) record_status(&g_wait_status, kWaitMma);
}

// CTA pair, leader (rank 0): per slice, wait for the stage of both CTAs (one
// barrier counts both CTAs' copies), then four 256 x 256 x 8 MMAs over both CTAs' shared
// memory into both CTAs' TMEM; the commits free the stage and fill the
// accumulator in both CTAs.  The accumulator is free again once the epilogue
// warps of both CTAs have drained it.
template <int MN>
__device__ __forceinline__ void mma_issuer_pair(typename TCfg<MN>::Smem& sh, uint32_t tmem, const Params& p) {
    using C = TCfg<MN>;
    constexpr int S = C::kStages;
    constexpr uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(BN >> 3) << 17) |
                               ((uint32_t)((2 * BM) >> 4) << 24);
    uint64_t i = 0;
    bool ok = true;
    const int64_t n_items = sh.sched.n_items;
    for (int64_t w = 0; w < n_items && ok; ++w) {
        const Item itm = sh.sched.item(w, p.nk);
        const uint32_t buf = (uint32_t)(w & 1);
        const uint64_t use = (uint64_t)w >> 1;
        if (use > 0 && !mbar_wait_cluster(&sh.acc_empty[buf], (uint32_t)((use - 1) & 1))) {
            record_status(&g_wait_status, kWaitAccFree);
            break;
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * kAccCols;
        for (int kt = itm.kb; kt < itm.ke; ++kt, ++i) {
            const int st = (int)(i % S);
            const uint32_t par = (uint32_t)((i / S) & 1);
            if (!mbar_wait(&sh.full[st], par)) {
                record_status(&g_wait_status, kWaitFull);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sh.a[st]);
            const uint32_t b0 = smem_u32(sh.b[st]);
#pragma unroll
            for (int kk = 0; kk < BK / kMmaK; ++kk) {
                const uint64_t ad = umma_desc_kmajor_sw128(a0 + kk * kMmaK * 4);
                const uint64_t bd = umma_desc_kmajor_sw128(b0 + kk * kMmaK * 4);
                mma_tf32_pair(d, ad, bd, idesc, (kt > itm.kb || kk > 0) ? 1u : 0u);
            }
            mma_commit_pair_both(&sh.empty[st]);
        }
        if (!ok) break;
        mma_commit_pair_both(&sh.acc_full[buf]);
    }
    // Nothing may still be writing either CTA's TMEM when it is freed.
    mma_commit_pair_local(&sh.mma_done);
    if (!mbar_wait(&sh.mma_done, 0)) record_status(&g_wait_status, kWaitMma);
}

// Partial sums of one 32-column piece of a row: 8 float4 at a stride of 128
// rows, so a warp's 16-byte accesses cover 512 contiguous bytes.
__device__ __forceinline__ float4* partial_piece(float4* slot, int c, int row) {
    return slot + (c * 8) * kBM128 + row;
}

// The split schedule's workers: CTAs, or on a pair clusters of two CTAs, each
// CTA of which parks and collects its own 128 rows of a tile's partial sums.
__device__ __forceinline__ int64_t worker(const Params& p) {
    return p.pair ? (int64_t)(blockIdx.x >> 1) : (int64_t)blockIdx.x;
}
__device__ __forceinline__ int64_t n_workers(const Params& p) {
    return p.pair ? (int64_t)(gridDim.x >> 1) : (int64_t)gridDim.x;
}
// The CTA of worker w that holds the same rows as this CTA.
__device__ __forceinline__ int64_t worker_cta(const Params& p, int64_t w) {
    return p.pair ? 2 * w + (int64_t)(blockIdx.x & 1) : w;
}

// Waits (bounded) until workers first..worker-1 have published their pieces
// of this tile; one lane spins, then every lane takes its own acquire.  False
// on timeout.
__device__ __forceinline__ bool wait_pieces(const Params& p, int64_t first, int lane) {
    for (int64_t w = first; w < worker(p); ++w) {
        const int64_t c = worker_cta(p, w);
        int up = 1;
        if (lane == 0) up = wait_flag(p.ws_flag + c) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, up, 0)) return false;
        (void)ld_acquire_gpu(p.ws_flag + c);
    }
    return true;
}

// One 32-column chunk of this thread's row of a piece's partial sums.
__device__ __forceinline__ void load_piece_chunk(float (&x)[32], const Params& p, int64_t cta, int chunk,
                                                 int row) {
    const float4* q = partial_piece(p.ws_partial + cta * kSlotFloat4, chunk, row);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 t = __ldcg(q + j * kBM128);
        x[4 * j] = t.x; x[4 * j + 1] = t.y; x[4 * j + 2] = t.z; x[4 * j + 3] = t.w;
    }
}

// Adds the partial sums of pieces from workers `from` down to `first` of one
// 32-column chunk of this thread's row (latest first: a fixed order).
__device__ __forceinline__ void add_pieces(float (&v)[32], const Params& p, int64_t first, int64_t from,
                                           int chunk, int row) {
#pragma unroll 1
    for (int64_t w = from; w >= first; --w) {
        float x[32];
        load_piece_chunk(x, p, worker_cta(p, w), chunk, row);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] += x[e];
    }
}

// Writes one finished tile's rows [quarter*32, +32) through the C tensor map:
// per 32-column piece the warp forms alpha*acc (+ C_old, itself brought in by
// a TMA load), adds the fused addend and applies ACT, writes the piece into
// its staging tile and lane 0 issues one bulk tensor store (the parts outside
// C are not written).  A row-major C (COLC false) stages a 128-byte row of C
// per lane, written as float4s; a column-major C stages one 128-byte column
// of the piece per n, each lane (one m) writing its element of every column,
// which the 128-byte swizzle keeps free of bank conflicts.  Returns false if
// a C_old load did not land in time.
template <int ACT, bool COLC, typename SmemT, int NBUF>
__device__ __forceinline__ bool store_tile_tma(SmemT& sh, const CUtensorMap* cmap, const Params& p,
                                               const TileCoord& tc, uint32_t taddr, int quarter,
                                               int lane, int ew, uint32_t& c_loads,
                                               uint32_t& stores, int64_t first_piece) {
    const int64_t m_base = tc.m0 + quarter * 32;
    const int64_t m = m_base + lane;
    const float* drow = (p.epi.D && m < p.M) ? p.epi.D + tc.b * p.epi.bsD + m * p.epi.rsD : nullptr;
    const bool rows_in = m_base < p.M;
    const int row = quarter * 32 + lane;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        const int64_t n0 = tc.n0 + c * 32;
        const bool piece_in = rows_in && n0 < p.N;
        // Stores alternate between the warp's two staging tiles; a tile is free
        // once the store before the most recent one has read it.  With
        // accumulation C_old must land there first; without, the tile is waited
        // for only just before it is written, so that the TMEM load and the
        // arithmetic overlap the earlier stores.
        float* st = sh.stage[ew][NBUF == 2 ? (stores & 1u) : 0u];
        if (p.accumulate) {
            if (lane == 0) {
                if (NBUF == 2) bulk_wait_read_all_but_one(); else bulk_wait_read_all();
                if (piece_in) {
                    mbar_arrive_expect_tx(&sh.c_old[ew], 32 * 32 * 4);
                    if (COLC) tma_load_3d(st, cmap, &sh.c_old[ew], (int)m_base, (int)n0, (int)tc.b);
                    else tma_load_3d(st, cmap, &sh.c_old[ew], (int)n0, (int)m_base, (int)tc.b);
                }
            }
            __syncwarp();
        }
        float v[32];
        tmem_ld32(taddr + c * 32, v);      // whole warp, converged: row m, columns n0..n0+31
        if (!piece_in) continue;
        // A tail adds the earlier pieces' partial sums before alpha.
        if (first_piece >= 0) add_pieces(v, p, first_piece, worker(p) - 1, c, row);
        if (p.accumulate) {
            if (!mbar_wait(&sh.c_old[ew], c_loads & 1u)) return false;
            ++c_loads;
if constexpr (COLC) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    v[e] = fmaf(p.alpha, v[e], st[e * 32 + (((lane >> 2) ^ (e & 7)) << 2) + (lane & 3)]);
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 o = *reinterpret_cast<const float4*>(st + lane * 32 + ((q ^ (lane & 7)) << 2));
                    v[4 * q + 0] = fmaf(p.alpha, v[4 * q + 0], o.x);
                    v[4 * q + 1] = fmaf(p.alpha, v[4 * q + 1], o.y);
                    v[4 * q + 2] = fmaf(p.alpha, v[4 * q + 2], o.z);
                    v[4 * q + 3] = fmaf(p.alpha, v[4 * q + 3], o.w);
                }
            }
            __syncwarp();                  // every lane has read its C_old row
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = p.alpha * v[e];
        }
        if (drow && (!kDebugChecks || (dbg_in_span(p.epi.D, drow + n0 * p.epi.csD, p.epi.d_span, &g_wait_status) &&
                                        dbg_in_span(p.epi.D, drow + (n0 + 31 < p.N ? n0 + 31 : p.N - 1) * p.epi.csD,
                                                    p.epi.d_span, &g_wait_status)))) {
            if (p.epi.d_vec4 && n0 + 32 <= p.N) {
                const float4* d4 = reinterpret_cast<const float4*>(drow + n0);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 d = __ldg(d4 + q);
                    v[4 * q + 0] += d.x;
                    v[4 * q + 1] += d.y;
                    v[4 * q + 2] += d.z;
                    v[4 * q + 3] += d.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (n0 + e < p.N) v[e] += __ldg(drow + (n0 + e) * p.epi.csD);
            }
        }
        if constexpr (ACT != kActNone) {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = act_fn<ACT>(v[e]);
        }
        if (!p.accumulate) {
            if (lane == 0) {
                if (NBUF == 2) bulk_wait_read_all_but_one(); else bulk_wait_read_all();
            }
            __syncwarp();
        }
if constexpr (COLC) {
#pragma unroll
            for (int e = 0; e < 32; ++e) st[e * 32 + (((lane >> 2) ^ (e & 7)) << 2) + (lane & 3)] = v[e];
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4*>(st + lane * 32 + ((q ^ (lane & 7)) << 2)) =
                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (COLC) tma_store_3d(cmap, st, (int)m_base, (int)n0, (int)tc.b);
            else tma_store_3d(cmap, st, (int)n0, (int)m_base, (int)tc.b);
            bulk_commit();
        }
        ++stores;
    }
    return true;
}

// store_tile_tma for the run-time activation.
template <bool COLC, typename SmemT, int NB>
__device__ __forceinline__ bool store_tile_act(SmemT& sh, const CUtensorMap* cmap, const Params& p,
                                               const TileCoord& tc, uint32_t taddr, int quarter,
                                               int lane, int ew, uint32_t& c_loads,
                                               uint32_t& stores, int64_t first_piece) {
    switch (p.epi.act) {
        case kActRelu: return store_tile_tma<kActRelu, COLC, SmemT, NB>(sh, cmap, p, tc, taddr, quarter, lane, ew, c_loads, stores, first_piece);
        case kActSigmoid: return store_tile_tma<kActSigmoid, COLC, SmemT, NB>(sh, cmap, p, tc, taddr, quarter, lane, ew, c_loads, stores, first_piece);
        case kActSilu: return store_tile_tma<kActSilu, COLC, SmemT, NB>(sh, cmap, p, tc, taddr, quarter, lane, ew, c_loads, stores, first_piece);
        case kActGeluTanh: return store_tile_tma<kActGeluTanh, COLC, SmemT, NB>(sh, cmap, p, tc, taddr, quarter, lane, ew, c_loads, stores, first_piece);
        case kActGeluErf: return store_tile_tma<kActGeluErf, COLC, SmemT, NB>(sh, cmap, p, tc, taddr, quarter, lane, ew, c_loads, stores, first_piece);
        default: return store_tile_tma<kActNone, COLC, SmemT, NB>(sh, cmap, p, tc, taddr, quarter, lane, ew, c_loads, stores, first_piece);
    }
}

template <int MN>
__device__ __forceinline__ void epilogue(typename TCfg<MN>::Smem& sh, uint32_t tmem,
                                         const CUtensorMap* cmap, const Params& p, int warp,
                                         int lane) {
    using SmemT = typename TCfg<MN>::Smem;
    constexpr int NB = TCfg<MN>::kStageBufs;
    const int quarter = warp & 3;               // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;
    const int ew = warp - 2;                    // epilogue warp index: staging tile, C_old barrier
    uint32_t c_loads = 0;                       // C_old pieces this warp has loaded
    uint32_t stores = 0;                        // bulk stores this warp has issued
    const int64_t n_items = sh.sched.n_items;
    for (int64_t w = 0; w < n_items; ++w) {
        const Item itm = sh.sched.item(w, p.nk);
        const uint32_t buf = (uint32_t)(w & 1);
        const uint32_t acc_parity = (uint32_t)((w >> 1) & 1);
        // A tail finishes its tile: the earlier pieces (CTAs first..this-1)
        // were computed at the same time and published as heads, normally
        // long before this point.
        int64_t first_piece = -1;
        if (itm.mode == kTail) {
            first_piece = unit_owner((itm.tile - p.dp_tiles) * p.nk, p.sk_units, n_workers(p));
            if (!wait_pieces(p, first_piece, lane)) {
                record_status(&g_wait_status, kWaitPartial);
                return;
            }
        }
        if (!mbar_wait(&sh.acc_full[buf], acc_parity)) {
            record_status(&g_wait_status, kWaitMma);
            return;
        }
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + buf * kAccCols;
        if (itm.mode == kHead) {
            // Partial sums to the workspace, then the successor's flag once every
            // epilogue thread's stores are visible device-wide.
            float4* dst = p.ws_partial + (int64_t)blockIdx.x * kSlotFloat4;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                float v[32];
                __syncwarp();
                tmem_ld32(taddr + c * 32, v);
                float4* q = partial_piece(dst, c, row);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    __stcg(q + j * kBM128, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
            }
            __threadfence();
            mbar_arrive(&sh.stored);
            if (warp == 2 && lane == 0) {
                if (!mbar_wait(&sh.stored, 0)) {
                    record_status(&g_wait_status, kWaitPartial);
                    return;
                }
                st_release_gpu(p.ws_flag + blockIdx.x, 1u);
            }
        } else if (p.c_tma) {
            const TileCoord tc = tile_coord(p, itm.tile);
            const bool ok = p.c_tma == 2
                ? store_tile_act<true, SmemT, NB>(sh, cmap, p, tc, taddr, quarter, lane, ew, c_loads, stores, first_piece)
                : store_tile_act<false, SmemT, NB>(sh, cmap, p, tc, taddr, quarter, lane, ew, c_loads, stores, first_piece);
            if (!ok) {
                record_status(&g_wait_status, kWaitFull);
                return;
            }
        } else {
            // Any other C: a lane per row, the columns in turn (128-byte rows
            // when C is column-major).
            const TileCoord tc = tile_coord(p, itm.tile);
            const int64_t m = tc.m0 + row;
            const bool row_ok = m < p.M;
            float* crow = p.C + tc.b * p.bsC + (row_ok ? m : 0) * p.rsC;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                float v[32];
                __syncwarp();
                tmem_ld32(taddr + c * 32, v);      // whole warp, converged, every row
                const int64_t n0 = tc.n0 + c * 32;
                if (!row_ok || n0 >= p.N) continue;
                if (first_piece >= 0) add_pieces(v, p, first_piece, worker(p) - 1, c, row);
                // C_old of the whole piece is loaded before any store, so the 32
                // loads are in flight together (the compiler cannot move a load
                // of C above a store to C).
                if (p.accumulate) {
                    float o[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = (n0 + e < p.N && dbg_in_span(p.C, crow + (n0 + e) * p.csC, p.sc, &g_wait_status))
                                   ? crow[(n0 + e) * p.csC] : 0.0f;
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = fmaf(p.alpha, v[e], o[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = p.alpha * v[e];
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int64_t n = n0 + e;
                    if (n < p.N && dbg_in_span(p.C, crow + n * p.csC, p.sc, &g_wait_status)) {
                        float r = v[e];
                        if (p.epi.on) r = finish(p.epi, r, tc.b, m, n, &g_wait_status);
                        crow[n * p.csC] = r;
                    }
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            // On a pair the leader's MMAs write both CTAs' accumulators: the
            // peer's epilogue warps free theirs on the leader's barrier.
            if (TCfg<MN>::kPair && (cluster_rank() & 1) != 0)
                mbar_arrive_remote(&sh.acc_empty[buf], 0);
            else
                mbar_arrive(&sh.acc_empty[buf]);
        }
    }
}

template <int MN>
__global__ void __launch_bounds__(TCfg<MN>::kThreads, 1)
tf32_tc_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
               const __grid_constant__ CUtensorMap tcm, const Params p) {
    using C = TCfg<MN>;
    using Smem = typename C::Smem;
    constexpr int kStages = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    Smem& sh = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        for (int s = 0; s < C::kTStages; ++s) {
            mbar_init(&sh.tdone[s], kTransWarps);
            mbar_init(&sh.tempty[s], 1);
        }
        for (int r = 0; r < C::kRawSlots; ++r) {
            mbar_init(&sh.rfull[r], 1);
            mbar_init(&sh.rempty[r], kTransWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.acc_full[b], 1);
            mbar_init(&sh.acc_empty[b], kEpiWarps * (C::kPair ? 2 : 1));
        }
        mbar_init(&sh.mma_done, 1);
        mbar_init(&sh.stored, kEpiWarps * 32);
        for (int w = 0; w < kEpiWarps; ++w) mbar_init(&sh.c_old[w], 1);
        if constexpr (C::kPair) {
            sh.sched.init(p.dp_tiles, p.sk_units, p.nk, blockIdx.x >> 1, gridDim.x >> 1);
            fence_mbar_init_cluster();
        } else {
            sh.sched.init(p.dp_tiles, p.sk_units, p.nk);
            fence_mbar_init();
        }
        prefetch_tensormap(&ta);
        prefetch_tensormap(&tb);
        if (p.c_tma) prefetch_tensormap(&tcm);
    }
    if (warp == 1) {
        if constexpr (C::kPair) {
            // One warp of each CTA of the pair: the same columns in both.
            tmem_alloc_pair(&sh.tmem_base, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&sh.tmem_base, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    // A pair's barriers and TMEM are set up in both CTAs before either uses
    // the other's.
    if constexpr (C::kPair) cluster_sync();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        if (lane == 0) producer<MN>(sh, &ta, &tb, p);
    } else if (warp == 1) {
        if constexpr (C::kPair) {
            // The leader issues the pair's MMAs; the peer's MMA lane has no work.
            if (lane == 0 && (cluster_rank() & 1) == 0) mma_issuer_pair<MN>(sh, tmem, p);
        } else {
            if (lane == 0) mma_issuer<MN>(sh, tmem, p);
        }
    } else if (warp < 2 + kEpiWarps) {
        epilogue<MN>(sh, tmem, &tcm, p, warp, lane);
        // Shared memory must outlive the bulk stores that read it.
        if (lane == 0) bulk_wait_all();
    } else if constexpr (C::kTrans) {
        transposer<MN>(sh, p, threadIdx.x - (2 + kEpiWarps) * 32, lane);
    }

    tc_fence_before();
    __syncthreads();
    // Neither CTA of a pair leaves (or frees TMEM) while the other may still
    // use its shared memory, barriers or TMEM.
    if constexpr (C::kPair) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (C::kPair) tmem_dealloc_pair(tmem, kTmemCols);
        else tmem_dealloc(tmem, kTmemCols);
    }
}

// An MN-major operand (unit stride along M or N): dims (M or N, K, batch), a
// 32 x 32 box (32 values along the unit stride, 32 rows along K), 128-byte
// swizzle.
bool make_mn_map(CUtensorMap* map, const float* base, int64_t inner, int64_t K, int64_t sk,
                 int64_t sb, int64_t batch, bool broadcast) {
    const int64_t nb = broadcast ? 1 : batch;
    const int64_t sk_b = K > 1 ? sk * 4 : ((inner * 4 + 15) / 16) * 16;
    const int64_t sb_b = nb > 1 ? sb * 4 : sk_b * (K > 1 ? K : 1);
    const uint64_t dims[3] = {(uint64_t)inner, (uint64_t)K, (uint64_t)nb};
    const uint64_t strides[2] = {(uint64_t)sk_b, (uint64_t)sb_b};
    const uint32_t box[3] = {32, 32, 1};
    return encode_tmap_f32_3d(map, base, dims, strides, box, true);
}

// The same operand as a rank-4 map for an extent that is a multiple of 32:
// dims (32 along M or N, K, blocks of 32, batch), so that one box of
// (32, 32, rows / 32) lands as the rows / 32 boxes of make_mn_map one after
// another.  False if the extent does not divide or the driver refuses it.
bool make_mn_map4(CUtensorMap* map, const float* base, int64_t inner, int64_t K, int64_t sk,
                  int64_t sb, int64_t batch, bool broadcast, int rows) {
    if (inner % 32 != 0 || inner / 32 >= ((int64_t)1 << 31)) return false;
    const int64_t nb = broadcast ? 1 : batch;
    const int64_t sk_b = K > 1 ? sk * 4 : ((inner * 4 + 15) / 16) * 16;
    const int64_t sb_b = nb > 1 ? sb * 4 : sk_b * (K > 1 ? K : 1);
    const uint64_t dims[4] = {32, (uint64_t)K, (uint64_t)(inner / 32), (uint64_t)nb};
    const uint64_t strides[3] = {(uint64_t)sk_b, 128, (uint64_t)sb_b};
    const uint32_t box[4] = {32, 32, (uint32_t)(rows / 32), 1};
    return encode_tmap_f32_4d(map, base, dims, strides, box, true);
}

bool make_kmajor_map(CUtensorMap* map, const float* base, int64_t K, int64_t rows, int64_t so,
                     int64_t sb, int64_t batch, bool broadcast, int box_rows) {
    const int64_t nb = broadcast ? 1 : batch;
    const int64_t so_b = rows > 1 ? so * 4 : ((K * 4 + 15) / 16) * 16;
    const int64_t sb_b = nb > 1 ? sb * 4 : so_b * (rows > 1 ? rows : 1);
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)rows, (uint64_t)nb};
    const uint64_t strides[2] = {(uint64_t)so_b, (uint64_t)sb_b};
    const uint32_t box[3] = {(uint32_t)BK, (uint32_t)box_rows, 1};
    return encode_tmap_f32_3d(map, base, dims, strides, box, true);
}

// C's tensor map for the epilogue's bulk stores and C_old loads: unit stride
// along N, a 16-byte aligned base, positive 16-byte multiple strides laid out
// without overlap (row stride >= N, batch stride >= one matrix), extents that
// fit 32-bit coordinates; a 32 x 32 box, 128-byte swizzle.  False: C is
// written by the threads directly.
// The C tensor map, 32x32 boxes: 1 when C has unit stride along N (inner
// dimension N), 2 when it has unit stride along M (inner dimension M), 0 when
// neither (or an extent, stride or alignment TMA cannot take).
int make_c_map(CUtensorMap* map, const Problem& pr) {
    const bool row_major = pr.csC == 1 || pr.N == 1;
    const bool col_major = !row_major && (pr.rsC == 1 || pr.M == 1);
    if (!row_major && !col_major) return 0;
    if (reinterpret_cast<uintptr_t>(pr.C) % 16 != 0) return 0;
    const int64_t lim = (int64_t)1 << 31;
    if (pr.N >= lim || pr.M >= lim || pr.batch >= lim) return 0;
    // inner: the unit-stride extent; outer: the other one and its stride.
    const int64_t inner = row_major ? pr.N : pr.M;
    const int64_t outer = row_major ? pr.M : pr.N;
    const int64_t so = row_major ? pr.rsC : pr.csC;
    auto ok_stride = [](int64_t st) { return st > 0 && (st * 4) % 16 == 0 && st * 4 < ((int64_t)1 << 40); };
    const int64_t outer_b = outer > 1 ? so * 4 : ((inner * 4 + 15) / 16) * 16;
    if (outer > 1 && (!ok_stride(so) || so < inner)) return 0;
    const bool batched = pr.batch > 1;
    if (batched && (!ok_stride(pr.bsC) || pr.bsC * 4 < outer_b * outer)) return 0;
    const uint64_t dims[3] = {(uint64_t)inner, (uint64_t)outer, (uint64_t)pr.batch};
    const uint64_t strides[2] = {(uint64_t)outer_b, batched ? (uint64_t)pr.bsC * 4 : (uint64_t)outer_b * outer};
    const uint32_t box[3] = {32, 32, 1};
    if (!encode_tmap_f32_3d(map, pr.C, dims, strides, box, true)) return 0;
    return row_major ? 1 : 2;
}

}  // namespace

TmaFfmaConfig tf32_tc_config() { return {BM, BN, BK, TCfg<0>::kStages, TCfg<0>::kThreads}; }

namespace {

template <int MN>
cudaError_t launch_mn(const Problem& pr, const Plan& plan, cudaStream_t stream) {
    using C = TCfg<MN>;
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(tf32_tc_kernel<MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    CUtensorMap ta, tb;
    const bool a_bc = pr.batch == 1 || pr.bsA == 0;
    const bool b_bc = pr.batch == 1 || pr.bsB == 0;
    // A[m][k] = A + m*rsA + k*csA; B[k][n] = B + k*rsB + n*csB.
    const int a4 = C::kTA && make_mn_map4(&ta, pr.A, pr.M, pr.K, pr.csA, pr.bsA, pr.batch, a_bc, BM) ? 1 : 0;
    const int b4 = C::kTB && make_mn_map4(&tb, pr.B, pr.N, pr.K, pr.rsB, pr.bsB, pr.batch, b_bc, BN) ? 1 : 0;
    const bool ok_a = a4 || (C::kTA ? make_mn_map(&ta, pr.A, pr.M, pr.K, pr.csA, pr.bsA, pr.batch, a_bc)
                                    : make_kmajor_map(&ta, pr.A, pr.K, pr.M, pr.rsA, pr.bsA, pr.batch, a_bc, BM));
    const bool ok_b = b4 || (C::kTB ? make_mn_map(&tb, pr.B, pr.N, pr.K, pr.rsB, pr.bsB, pr.batch, b_bc)
                                    : make_kmajor_map(&tb, pr.B, pr.K, pr.N, pr.csB, pr.bsB, pr.batch, b_bc,
                                                      C::kBRows));
    if (!ok_a || !ok_b) return cudaErrorInvalidValue;
    Params p;
    p.a_blk4 = a4;
    p.b_blk4 = b4;
    p.pair = C::kPair ? 1 : 0;
    p.C = pr.C; p.rsC = pr.rsC; p.csC = pr.csC; p.bsC = pr.bsC;
    p.M = pr.M; p.N = pr.N; p.K = pr.K;
    p.tiles_m = plan.tiles_m; p.tiles_n = plan.tiles_n; p.tiles_total = plan.tiles;
    p.nk = (int)((pr.K + BK - 1) / BK);
    p.alpha = pr.alpha;
    p.accumulate = pr.accumulate;
    p.a_bcast = a_bc;
    p.b_bcast = b_bc;
    CUtensorMap tcm;
    std::memset(&tcm, 0, sizeof(tcm));
    p.c_tma = make_c_map(&tcm, pr);
    const int64_t grid = plan.ctas;
    p.dp_tiles = plan.stream_k ? plan.dp_tiles : plan.tiles;
    p.sk_units = plan.stream_k ? (plan.tiles - plan.dp_tiles) * p.nk : 0;
    p.epi = pr.epi;
    p.ws_partial = nullptr;
    p.ws_flag = nullptr;
    p.sc = pr.sc;
    if (plan.stream_k) {
        p.ws_partial = static_cast<float4*>(plan.workspace);
        p.ws_flag = reinterpret_cast<unsigned int*>(static_cast<char*>(plan.workspace) +
                                                    (size_t)grid * kSlotFloat4 * sizeof(float4));
        const cudaError_t e = cudaMemsetAsync(p.ws_flag, 0, (size_t)grid * sizeof(unsigned int), stream);
        if (e != cudaSuccess) return e;
    }
    if (plan.stream_k || C::kPair) {
        // A split's CTAs wait on one another's partial sums: a cooperative
        // launch makes them co-resident.  A pair kernel runs in clusters of
        // two CTAs, each pair one worker; where the driver takes no
        // cooperative launch of clusters, the planner's bound on the pairs
        // (the clusters that fit the device at once) stands in for it.
        static std::atomic<int> coop_clusters{1};
        const bool coop = plan.stream_k && (!C::kPair || coop_clusters.load() != 0);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(C::kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        int na = 0;
        if (coop) {
            attr[na].id = cudaLaunchAttributeCooperative;
            attr[na].val.cooperative = 1;
            ++na;
        }
        if (C::kPair) {
            attr[na].id = cudaLaunchAttributeClusterDimension;
            attr[na].val.clusterDim.x = 2;
            attr[na].val.clusterDim.y = 1;
            attr[na].val.clusterDim.z = 1;
            ++na;
        }
        cfg.attrs = attr;
        cfg.numAttrs = na;
        cudaError_t e = cudaLaunchKernelEx(&cfg, tf32_tc_kernel<MN>, ta, tb, tcm, p);
        if (e != cudaSuccess && coop && C::kPair) {
            (void)cudaGetLastError();
            coop_clusters.store(0);
            cfg.attrs = attr + 1;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, tf32_tc_kernel<MN>, ta, tb, tcm, p);
        }
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    tf32_tc_kernel<MN><<<(unsigned)grid, C::kThreads, C::kSmemBytes, stream>>>(ta, tb, tcm, p);
    return cudaGetLastError();
}

// Clusters of two CTAs of the pair kernel the device holds at once (one CTA
// per SM), asked of the driver once per device; 0 if it does not say.
template <int MN>
int pair_clusters_fit(int sm_count) {
    using C = TCfg<MN>;
    static std::atomic<int> fit[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    std::atomic<int>& slot = fit[dev & 63];
    const int known = slot.load();
    if (known != 0) return known > 0 ? known : 0;
    int n = 0;
    cudaError_t e = cudaFuncSetAttribute(tf32_tc_kernel<MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::kSmemBytes);
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(sm_count / 2 * 2));
        cfg.blockDim = dim3(C::kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&n, tf32_tc_kernel<MN>, &cfg);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    slot.store(n > 0 ? n : -1);
    return n > 0 ? n : 0;
}

}  // namespace

cudaError_t launch_tf32_tc(const Problem& pr, const Plan& plan, int sm_count, cudaStream_t stream) {
    (void)sm_count;
    // Orientation of the problem as launched (the plan's layouts describe C's
    // own orientation, which differs when the plan computes C^T).
    const bool a_mn = !(pr.K == 1 || pr.csA == 1);
    const bool b_mn = !(pr.K == 1 || pr.rsB == 1);
    if (a_mn && b_mn) return launch_mn<3>(pr, plan, stream);
    if (a_mn) return launch_mn<1>(pr, plan, stream);
    if (b_mn) return launch_mn<2>(pr, plan, stream);
    if (plan.variant == kPairVariant) return launch_mn<4>(pr, plan, stream);
    return launch_mn<0>(pr, plan, stream);
}

// The FFMA path's rules (stream_k_dp_tiles, split_k_ctas), with independent
// pieces in both cases.  The exchange is off the MMA path (a piece's partial
// sums are written while the next item's MMAs run; only the tail's epilogue
// reads them), but the split still costs about 15 us against the slice model,
// whose data-parallel estimate ignores that a thin last wave runs faster than
// a full one: charged as 48 slices of 128 x 256 x 32 (0.37 us each), which
// reproduces every measured decision (long K or few tiles split; c5a, c5b and
// K <= 2048 stay data-parallel).  The result is not the unsplit rounding, so
// k_split = EXACT never splits.
void tf32_tc_schedule(const Problem& pr, Plan& plan, int sm_count, size_t ws_bytes, const void* ws,
                      int k_split) {
    const int64_t nk = (pr.K + BK - 1) / BK;
    const int64_t G = sm_count;
    plan.k_slices = (int)nk;
    plan.stream_k = false;
    plan.split_indep = false;
    plan.dp_tiles = plan.tiles;
    plan.ctas = plan.tiles < G ? plan.tiles : G;
    const size_t need = (size_t)G * (size_t)kSlotFloat4 * sizeof(float4) + (size_t)G * sizeof(unsigned int);
    if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) % 256) != 0) return;
    if (k_split != SBGEMM_KSPLIT_ANY) return;
    int64_t dp = stream_k_dp_tiles(plan.tiles, nk, G, 48);
    int64_t ctas = G;
    if (dp < 0) {
        ctas = split_k_ctas(plan.tiles, nk, G, 8, 48);
        if (ctas < 0) return;
        dp = 0;
    }
    plan.stream_k = true;
    plan.split_indep = true;
    plan.dp_tiles = dp;
    plan.ctas = ctas;
    plan.workspace = const_cast<void*>(ws);
}

// Both operands K-major, at least 8 K slices, and 256 x 256 tiles enough
// for a wave of pairs: the tiles go to CTA pairs.  Each CTA then reads
// half of B per slice: a 32 KB stage instead of 48, six stages instead of
// four, and a third less shared-memory traffic per MMA, which is what holds
// the one-CTA tile near 0.7 of the tensor rate.  With a workspace the last
// waves are split into independent K pieces as on one CTA, each pair one
// worker.  Returns false (nothing changed) when pairs do not apply.
bool tf32_tc_pair(const Problem& pr, Plan& plan, int sm_count, size_t ws_bytes, const void* ws,
                  int k_split) {
    // An MN-major A on pairs (each CTA transposing its 128 rows, the peer's
    // transposers signalling the leader by 16-byte bulk copies) measured 3-7%
    // slower than one CTA's tiles, split or not (c5c 235 against 227 us).
    const bool a_k = pr.K == 1 || pr.csA == 1;
    const bool b_k = pr.K == 1 || pr.rsB == 1;
    if (!a_k || !b_k) return false;
    const int64_t nk = (pr.K + BK - 1) / BK;
    // Short K (c3's 64: two slices) is bound by the C stores, and a pair's two
    // epilogues, which both must drain an accumulator before either is
    // reused, measured slower there (41 against 35 us back to back).
    if (nk < 8) return false;
    const int64_t tm = (pr.M + 2 * BM - 1) / (2 * BM), tn = (pr.N + BN - 1) / BN;
    const int64_t tiles = tm * tn * pr.batch;
    int64_t pairs = sm_count / 2;
    const int fit = pair_clusters_fit<4>(sm_count);
    if (fit > 0 && fit < pairs) pairs = fit;
    if (pairs < 1 || tiles < pairs) return false;
    plan.variant = kPairVariant;
    plan.tiles_m = tm;
    plan.tiles_n = tn;
    plan.tiles = tiles;
    plan.k_slices = (int)nk;
    plan.tile_m = plan.transposed ? BN : 2 * BM;   // reported in C's own orientation
    plan.tile_n = plan.transposed ? 2 * BM : BN;
    plan.stream_k = false;
    plan.split_indep = false;
    plan.dp_tiles = tiles;
    plan.ctas = 2 * pairs;
    const size_t need = (size_t)(2 * pairs) * (size_t)kSlotFloat4 * sizeof(float4) +
                        (size_t)(2 * pairs) * sizeof(unsigned int);
    if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) % 256) != 0) return true;
    if (k_split != SBGEMM_KSPLIT_ANY) return true;
    const int64_t dp = stream_k_dp_tiles(tiles, nk, pairs, 48);
    if (dp < 0) return true;
    plan.stream_k = true;
    plan.split_indep = true;
    plan.dp_tiles = dp;
    plan.workspace = const_cast<void*>(ws);
    return true;
}

unsigned int read_and_clear_wait_status_tf32(cudaStream_t stream) {
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
