// Host side of the TMA-fed FFMA path: tile shapes, the choice between them,
// the work-list split and the launch dispatch.  The kernels themselves are in
// ffma_tma_kernel.cuh, compiled once per tile shape (ffma_tma_256x128.cu,
// ffma_tma_128x256.cu, ffma_tma_512x64.cu) so that the shapes build in
// parallel.
#include "ffma_tma_kernel.cuh"

namespace sbg {
namespace {

constexpr TmaFfmaConfig kConfigs[] = {
    {256, 128, BK, Cfg<256, 128>::kStages, kThreads},
    {128, 256, BK, Cfg<128, 256>::kStages, kThreads},
    {512, 64, BK, Cfg<512, 64, true, false>::kStages, kThreads},   // N <= 64, K-major A only
};
constexpr int kNarrowVariant = 2;

}  // namespace

int tma_ffma_config_count() { return (int)(sizeof(kConfigs) / sizeof(kConfigs[0])); }

TmaFfmaConfig tma_ffma_config(int variant) { return kConfigs[variant]; }

// Picks the tile shape that wastes the least work, counting both the ragged
// edge of the last tiles and the idle SMs of the last wave.
int tma_ffma_pick_variant(const Problem& p, int sm_count) {
    // K-major operands are transposed in shared memory slice by slice, which
    // costs in proportion to the tile's rows of that operand: on equal wave
    // cost, prefer the shape whose transposed side is the shorter one.
    const bool a_k = p.K == 1 || p.csA == 1;
    const bool b_k = p.K == 1 || p.rsB == 1;
    int best = 0;
    double best_cost = 0.0;
    int best_rows = 0;
    for (int v = 0; v < tma_ffma_config_count(); ++v) {
        // 512 x 64 tiles, for N <= 64 with a K-major A: all 8 warps busy where a
        // 128-wide tile leaves half of them idle.
        if (v == kNarrowVariant && !(a_k && p.N <= 64)) continue;
        const TmaFfmaConfig c = kConfigs[v];
        const int64_t tm = (p.M + c.bm - 1) / c.bm, tn = (p.N + c.bn - 1) / c.bn;
        const int64_t tiles = tm * tn * p.batch;
        const int64_t waves = (tiles + sm_count - 1) / sm_count;
        const double cost = (double)waves * c.bm * c.bn;   // time ~ waves x tile work
        const int rows = (a_k ? c.bm : 0) + (b_k ? c.bn : 0);
        if (v == 0 || cost < best_cost || (cost == best_cost && rows < best_rows)) {
            best = v;
            best_cost = cost;
            best_rows = rows;
        }
    }
    return best;
}

size_t tma_ffma_workspace_bytes(int sm_count) {
    // One partial tile per CTA (every thread's 64 accumulator pairs) and one
    // flag word per CTA; the same for every tile shape (256 threads x 128).
    static_assert(kWorkspaceBytesPerSm == (size_t)kThreads * 64 * sizeof(float2) + sizeof(unsigned int),
                  "one partial tile of this kernel's accumulators and one flag per CTA");
    return (size_t)sm_count * kWorkspaceBytesPerSm;
}

// Data-parallel for all but the last one or two waves, whose K slices are
// split evenly over the grid.  Chosen only when it removes at least 3% of the
// estimated time, every CTA's share spans at least one whole tile (so a tile
// is split at most once), and a tile has enough slices to amortise the
// exchange of its partial sums.
void tma_ffma_schedule(const Problem& pr, Plan& plan, int sm_count, size_t ws_bytes,
                       const void* ws, int k_split) {
    const TmaFfmaConfig c = kConfigs[plan.variant];
    const int64_t nk = (pr.K + c.bk - 1) / c.bk;
    const int64_t G = sm_count;
    plan.k_slices = (int)nk;
    plan.stream_k = false;
    plan.dp_tiles = plan.tiles;
    plan.ctas = plan.tiles < G ? plan.tiles : G;
    if (!ws || ws_bytes < tma_ffma_workspace_bytes(sm_count)) return;
    if ((reinterpret_cast<uintptr_t>(ws) % 256) != 0) return;
    if (k_split == SBGEMM_KSPLIT_NONE) return;
    // About 20 us of exchange and reset cost: some 4 slices of a 256 x 128 tile.
    const int64_t dp = stream_k_dp_tiles(plan.tiles, nk, G, 4);
    if (dp >= 0) {
        plan.stream_k = true;
        plan.dp_tiles = dp;
        plan.ctas = G;
        plan.workspace = const_cast<void*>(ws);
        return;
    }
    if (k_split != SBGEMM_KSPLIT_ANY) return;
    // Fewer tiles than SMs: independent K pieces of at least 8 slices.
    const int64_t g = split_k_ctas(plan.tiles, nk, G, 8, 4);
    if (g < 0) return;
    plan.stream_k = true;
    plan.split_indep = true;
    plan.dp_tiles = 0;
    plan.ctas = g;
    plan.workspace = const_cast<void*>(ws);
}

cudaError_t launch_tma_ffma(const Problem& p, const Plan& plan, int sm_count, cudaStream_t stream) {
    switch (plan.variant) {
        case 0: return launch_tma_ffma_256x128(p, plan, sm_count, stream);
        case 1: return launch_tma_ffma_128x256(p, plan, sm_count, stream);
        case kNarrowVariant: return launch_tma_ffma_512x64(p, plan, sm_count, stream);
        default: return cudaErrorInvalidValue;
    }
}

unsigned int read_and_clear_wait_status_tma_ffma(cudaStream_t stream) {
    unsigned int v = read_and_clear_wait_status_tma_ffma_256x128(stream);
    const unsigned int v1 = read_and_clear_wait_status_tma_ffma_128x256(stream);
    const unsigned int v2 = read_and_clear_wait_status_tma_ffma_512x64(stream);
    if (v == 0) v = v1;
    if (v == 0) v = v2;
    return v;
}

}  // namespace sbg
