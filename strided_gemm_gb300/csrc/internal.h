// Internal declarations shared by the host API and the kernel translation units.
// Nothing here is exported from the shared library.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sbgemm.h"

namespace sbg {

// Codes written to a path's device status word (first writer wins).
enum : unsigned int {
    kWaitFull = 1,       // consumer waiting for a loaded stage
    kWaitEmpty = 2,      // producer waiting for a released stage
    kWaitDrain = 3,      // producer draining its last copies on the way out
    kWaitMma = 4,        // epilogue waiting for the accumulator
    kWaitAccFree = 5,    // MMA issuer waiting for the epilogue to free TMEM
    kWaitPartial = 6,    // stream-K: exchanging partial sums between CTAs
    kWaitSelftestMbar = 7,   // self-test: an mbarrier phase nothing completes
    kWaitSelftestFlag = 8,   // self-test: a global flag nothing sets
    kBoundsViolation = 9,    // debug build: an access outside its operand's span (skipped)
    kPagedInput = 10,        // paged attention: a block id or sequence length out of range (skipped)
};

// Element offsets [lo, hi] from an operand's base pointer that lie inside the
// memory the caller described (the host's span check before every launch).
// Only the bounds checks of a debug build (SBGEMM_DEBUG) read them.
struct ElemSpan { int64_t lo, hi; };

// One call of the product, strides in fp32 elements (see include/sbgemm.h).
// Fused epilogue of sbgemm_fused: out = act(alpha*acc (+ C_old) + D), with D
// read through its own strides (epilogue.cuh applies it on the device).
struct EpiParams {
    const float* D;          // nullptr: no addend
    int64_t rsD, csD, bsD;
    int act;                 // SBGEMM_ACT_*
    int on;                  // D != nullptr || act != SBGEMM_ACT_NONE
    int d_vec4;              // D has unit stride along N and 16-byte aligned rows
    ElemSpan d_span;         // debug builds: D's valid element offsets
};

struct Problem {
    const float* A; int64_t rsA, csA, bsA;
    const float* B; int64_t rsB, csB, bsB;
    float* C;       int64_t rsC, csC, bsC;
    int64_t M, N, K, batch;
    float alpha;
    int accumulate;
    EpiParams epi;           // all zero: the plain product
    ElemSpan sa, sb, sc;     // debug builds: valid element offsets of A, B and C
};

// Per-device properties, read once per device and immutable afterwards.
struct DeviceProps {
    int device;
    int sm_count;
    int max_smem_per_block_optin;   // bytes
    int max_smem_per_sm;            // bytes
    int cc_major, cc_minor;
};

// Returns NULL if the device cannot be queried.
const DeviceProps* device_props(int device);

// Kernel variant chosen by the planner.
struct Plan {
    int path = SBGEMM_PATH_NONE;
    int a_layout = SBGEMM_LAYOUT_GENERAL, b_layout = SBGEMM_LAYOUT_GENERAL,
        c_layout = SBGEMM_LAYOUT_GENERAL;
    bool a_broadcast = false, b_broadcast = false;
    bool a_tma = false, b_tma = false;
    int tile_m = 0, tile_n = 0, tile_k = 0;
    int ctas_per_sm = 0;
    int variant = 0;                // kernel-specific configuration index
    int64_t tiles_m = 0, tiles_n = 0;
    int64_t tiles = 0;              // tiles_m * tiles_n * batch
    int64_t ctas = 0;
    int k_slices = 0;               // K slices per tile
    bool stream_k = false;          // tiles split along K (needs workspace)
    bool split_indep = false;       // ... as independent pieces (fewer tiles than SMs)
    bool transposed = false;        // computed as C^T = B^T A^T (tiles, schedule and
                                    // launch are those of the transposed problem)
    int64_t dp_tiles = 0;           // tiles computed whole
    int k_pieces = 1;               // gather path: K pieces per tile (independent)
    void* workspace = nullptr;      // caller's scratch when stream_k
};

// ---- fused attention (attention.cu) -----------------------------------------
// O[b,m,:] = softmax_n(alpha * Q[b,m,:] . K[b,n,:], causal optional) V[b,n,:]
struct AttnProblem {
    const float* Q; int64_t rsQ, csQ, bsQ;
    const float* K; int64_t rsK, csK, bsK;
    const float* V; int64_t rsV, csV, bsV;
    float* O;       int64_t rsO, csO, bsO;
    int64_t M, N, D, Dv, batch;
    float alpha;
    int causal;
    int64_t q_len;           // rows per head for the causal position
    ElemSpan sq, sk, sv, so; // debug builds: valid element offsets of Q, K, V and O
    // Paged K and V: K and V are then caches [num_blocks][block_size][n_kv_heads]
    // [D or Dv]; batch entry b is (sequence b / n_kv_heads, head b % n_kv_heads)
    // and key n of a sequence lives in block table[seq][n / block_size] at
    // offset n % block_size.  seq_lens (or N for all) gives each sequence's keys.
    int paged = 0;
    const int32_t* table = nullptr;
    const int32_t* seq_lens = nullptr;
    int64_t max_blocks = 0, block_size = 0, n_kv_heads = 0, num_blocks = 0;
    // Scratch of the split-key decode kernel (caller's workspace; may be null).
    void* workspace = nullptr;
    size_t workspace_bytes = 0;
};
// C^T = B^T A^T as a problem of its own: A' = B^T, B' = A^T, C' = C^T, M' = N,
// N' = M (the fused addend transposed alike).
Problem transposed_problem(const Problem& p);

bool attention_supported(int64_t D, int64_t Dv);
int64_t attention_max_rows();   // M limit of one launch
cudaError_t launch_attention(const AttnProblem& a, cudaStream_t stream);
// Few query rows per batch entry (decode): keys split across CTAs.
bool attention_decode_supported(const AttnProblem& a);
cudaError_t launch_attention_decode(const AttnProblem& a, cudaStream_t stream);
unsigned int read_and_clear_status_attention_decode(cudaStream_t stream);

// ---- strided-gather FFMA path (ffma_gather.cu) --------------------------------
// Tile configurations of the gather kernel.
struct GatherConfig { int bm, bn, bk, threads, ctas_per_sm; };
int gather_config_count();
GatherConfig gather_config(int variant);
// Picks a variant for the problem size on a device with `sm_count` SMs.
int gather_pick_variant(const Problem& p, int sm_count);
// With a workspace and k_split = ANY, cuts the K range of products with few
// tiles into pieces (plan.k_pieces, summed in a fixed order).
void gather_schedule(const Problem& p, Plan& plan, int sm_count, size_t ws_bytes, const void* ws,
                     int k_split);
cudaError_t launch_gather_ffma(const Problem& p, const Plan& plan, cudaStream_t stream);

// ---- TMA-fed FFMA path (ffma_tma.cu; kernels in ffma_tma_<shape>.cu) ---------
struct TmaFfmaConfig { int bm, bn, bk, stages, threads; };
int tma_ffma_config_count();
TmaFfmaConfig tma_ffma_config(int variant);
int tma_ffma_pick_variant(const Problem& p, int sm_count);
// Stream-K scratch per SM (one CTA each): one tile of partial sums, kept as
// the 64 accumulator pairs of each of the 256 threads of a TMA FFMA CTA (the
// TF32 kernel's 128 x 256 fp32 tile is the same size), plus one flag word.
constexpr size_t kWorkspaceBytesPerSm = (size_t)256 * 64 * 2 * sizeof(float) + sizeof(unsigned int);
// Bytes of workspace the stream-K schedule needs on a device with sm_count SMs.
size_t tma_ffma_workspace_bytes(int sm_count);
// Fills plan.ctas / stream_k / dp_tiles / k_slices for the chosen variant.
// k_split: SBGEMM_KSPLIT_* policy of the caller's options.
void tma_ffma_schedule(const Problem& p, Plan& plan, int sm_count, size_t ws_bytes, const void* ws,
                       int k_split);
cudaError_t launch_tma_ffma(const Problem& p, const Plan& plan, int sm_count, cudaStream_t stream);
// One per tile shape (ffma_tma_<shape>.cu), each with its own status word.
cudaError_t launch_tma_ffma_256x128(const Problem& p, const Plan& plan, int sm_count, cudaStream_t stream);
cudaError_t launch_tma_ffma_128x256(const Problem& p, const Plan& plan, int sm_count, cudaStream_t stream);
cudaError_t launch_tma_ffma_512x64(const Problem& p, const Plan& plan, int sm_count, cudaStream_t stream);
unsigned int read_and_clear_wait_status_tma_ffma_256x128(cudaStream_t stream);
unsigned int read_and_clear_wait_status_tma_ffma_128x256(cudaStream_t stream);
unsigned int read_and_clear_wait_status_tma_ffma_512x64(cudaStream_t stream);

// Reads and clears the status words of the kernels that use bounded waits.
// Returns the first non-zero code found (0 if none).
unsigned int read_and_clear_wait_status_tma_ffma(cudaStream_t stream);

// ---- TF32 tensor-core path (tf32_tc.cu) ----------------------------------------
TmaFfmaConfig tf32_tc_config();
cudaError_t launch_tf32_tc(const Problem& p, const Plan& plan, int sm_count, cudaStream_t stream);
// Fills plan.ctas / stream_k / dp_tiles / k_slices for the TF32 kernel.
void tf32_tc_schedule(const Problem& p, Plan& plan, int sm_count, size_t ws_bytes, const void* ws,
                      int k_split);
// Switches a plan of two K-major operands to CTA-pair tiles where they apply
// (with their own split over the workspace); false leaves the plan as it was.
bool tf32_tc_pair(const Problem& pr, Plan& plan, int sm_count, size_t ws_bytes, const void* ws,
                  int k_split);
unsigned int read_and_clear_wait_status_tf32(cudaStream_t stream);

// ---- status words of the kernels without bounded waits (debug bounds checks) ----
unsigned int read_and_clear_status_gather(cudaStream_t stream);
unsigned int read_and_clear_status_attention(cudaStream_t stream);

// ---- failure-detection self-test (selftest.cu) ----------------------------------
unsigned int read_and_clear_wait_status_selftest(cudaStream_t stream);

// ---- driver entry points (driver.cpp) ---------------------------------------
// [base, base+size) of the allocation that contains `ptr`; false if `ptr` is not
// in a device-accessible allocation known to the driver.
bool device_allocation_range(const void* ptr, uintptr_t* base, size_t* size);

// Rank-3 fp32 tiled tensor map: dims innermost first, byte strides of dims 1
// and 2, box extents, optional 128-byte swizzle.  Zero fill out of bounds.
bool encode_tmap_f32_3d(CUtensorMap* map, const void* base, const uint64_t dims[3],
                        const uint64_t strides_bytes[2], const uint32_t box[3], bool swizzle128);
// The same with rank 4 (byte strides of dims 1, 2 and 3).
bool encode_tmap_f32_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                        const uint64_t strides_bytes[3], const uint32_t box[4], bool swizzle128);

}  // namespace sbg
