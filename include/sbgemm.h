/*
 * sbgemm: strided batched fp32 matrix product on one GB300 (sm_103a).
 *
 *     C[b] <- alpha * A[b] * B[b]            (accumulate == 0)
 *     C[b] <- alpha * A[b] * B[b] + C[b]     (accumulate != 0)
 *
 * for b = 0 .. batch-1, where A[b] is M x K, B[b] is K x N and C[b] is M x N.
 *
 * Source of the operation: StaleyNET, "GPU Implementation", section "The matrix
 * product" -- one kernel computes, for a batch of matrix pairs, alpha times A
 * times B with the previous C optionally added; every input is described by the
 * memory distance between neighbouring rows and between neighbouring columns,
 * so a transposed input is the same memory with the two distances exchanged,
 * and the batch covers all heads and sequences of attention in one launch.  The
 * argument list generalises the row-major cuBLAS call of "rvllm CUDA path"
 * (section "Matmuls go to cuBLAS": lda/ldb/ldc and a strided batch) and the
 * {batches, rows, inner, columns} sizes of the kael.cpp "CUDA backend" page.
 *
 * Layout.  Every operand is a base pointer plus three strides counted in fp32
 * ELEMENTS (not bytes), signed 64-bit:
 *     A[b][m][k] = A[b*bsA + m*rsA + k*csA]
 *     B[b][k][n] = B[b*bsB + k*rsB + n*csB]
 *     C[b][m][n] = C[b*bsC + m*rsC + n*csC]
 * A transposed read is the stored matrix with rs and cs exchanged (a row-major
 * W[N][K] read as B = W^T has rsB = 1, csB = K).  Strides of A and B may be
 * zero (broadcast: one matrix shared by every batch entry, or one row shared
 * by every row) or negative.  C's strides must map distinct (b, m, n) to
 * distinct elements.
 *
 * Numerics.  sbgemm and sbgemm_ex with math = SBGEMM_MATH_FP32 compute every
 * product and sum in fp32 with fused multiply-adds, each output's terms added
 * in increasing k, and the result formed as fmaf(alpha, sum, C_old).  Integer
 * inputs whose partial sums stay below 2^24 give exact results.
 * SBGEMM_MATH_TF32 (opt-in, sbgemm_ex only) rounds A and B to tf32 on the
 * tensor cores and accumulates in fp32.
 *
 * Ownership and synchronisation.  All pointers are device memory owned by the
 * caller (cudaMalloc, cudaMallocAsync, managed memory, or any allocator that
 * hands out such memory).  The library allocates nothing per call; it keeps
 * only immutable per-device properties, initialised once.  Calls are enqueued
 * on `stream` (a cudaStream_t; NULL = the legacy default stream) and return
 * without synchronising; errors raised inside a kernel surface at the
 * caller's next synchronisation.  The functions are thread-safe.
 *
 * Edge cases.  M, N or batch equal to 0: nothing is done (SBGEMM_OK, pointers
 * may be NULL).  K == 0: C <- alpha*0 (overwrite) or C is left as it was
 * (accumulate).  Without accumulation C is never read, so stale NaNs in C do
 * not leak into the result.
 *
 * Errors are returned as sbgemm_status codes; nothing is launched on error.
 */
#ifndef SBGEMM_H
#define SBGEMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SBGEMM_API __attribute__((visibility("default")))
#else
#define SBGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SBGEMM_OK = 0,
    SBGEMM_ERR_INVALID_VALUE = 1,   /* negative size, misaligned pointer, stride
                                       span overflowing int64, bad option value */
    SBGEMM_ERR_NULL_POINTER = 2,    /* a needed operand pointer is NULL */
    SBGEMM_ERR_OUTPUT_OVERLAP = 3,  /* C's strides map two outputs to one element,
                                       or C's address span meets A's or B's */
    SBGEMM_ERR_UNSUPPORTED = 4,     /* a forced path cannot serve this layout */
    SBGEMM_ERR_CUDA = 5,            /* CUDA runtime/driver error (launch, attribute,
                                       tensor-map encoding, no device) */
    SBGEMM_ERR_DEVICE_TIMEOUT = 6,  /* a bounded in-kernel wait expired; see
                                       sbgemm_device_status */
    SBGEMM_ERR_NOT_DEVICE_MEMORY = 7, /* an operand is not device-accessible memory,
                                       or its span leaves its allocation */
    SBGEMM_ERR_DEVICE_CHECK = 8     /* a kernel's own check found an input it
                                       could not use (a paged block id or
                                       sequence length out of range; a debug
                                       build's out-of-span address) and skipped
                                       it; see sbgemm_device_status */
} sbgemm_status;

/* Arithmetic of sbgemm_options.math. */
enum {
    SBGEMM_MATH_FP32 = 0,  /* fp32 FFMA on the CUDA cores (default, strict) */
    SBGEMM_MATH_TF32 = 1   /* tf32 inputs, fp32 accumulation, on the tensor cores */
};

/* Kernel paths; sbgemm_options.force_path and sbgemm_plan_info.path. */
enum {
    SBGEMM_PATH_NONE = -1,        /* nothing to launch (empty problem, or
                                     K == 0 with accumulate) */
    SBGEMM_PATH_AUTO = 0,         /* let the planner choose */
    SBGEMM_PATH_GATHER_FFMA = 1,  /* any strides: coalesced strided gather into
                                     shared memory, FFMA register micro-tiles */
    SBGEMM_PATH_TMA_FFMA = 2,     /* unit-stride operands: TMA + mbarrier ring,
                                     FFMA register micro-tiles */
    SBGEMM_PATH_TMA_TF32 = 3      /* unit-stride operands (an MN-major one is
                                     transposed in shared memory): TMA +
                                     tcgen05.mma kind::tf32 with the
                                     accumulator in TMEM */
};

/* Operand layout classes reported by sbgemm_plan. */
enum {
    SBGEMM_LAYOUT_K_MAJOR = 0,   /* unit stride along K (A: csA == 1, B: rsB == 1);
                                    for C: unit stride along N (csC == 1) */
    SBGEMM_LAYOUT_MN_MAJOR = 1,  /* unit stride along M (A) or N (B);
                                    for C: unit stride along M (rsC == 1) */
    SBGEMM_LAYOUT_GENERAL = 2    /* no unit stride */
};

/* How the planner may split a tile's K range across CTAs when a workspace is
 * given; sbgemm_options.k_split.  The split follows the work-list scheme of
 * persistent CTAs, and its partial sums are added in a fixed order, so every
 * choice is deterministic from run to run (the pages' "Chapter 09 CUDA
 * backend", section "Reductions", for device sums; "GPU Implementation",
 * section "Making the embedding gradient repeatable", for gradients). */
enum {
    SBGEMM_KSPLIT_ANY = 0,    /* default: chained stream-K over the last waves,
                                 or, with fewer tiles than SMs and long K
                                 (e.g. the weight gradient Gt*X), independent K
                                 pieces summed in a fixed order; the latter
                                 rounds differently from the unsplit product.
                                 Small products on the gather path are cut
                                 into K pieces the same way, and products of
                                 at most 16384 outputs with K > 128 split K
                                 across the 32 lanes of a warp (one output per
                                 warp, a fixed shuffle tree). */
    SBGEMM_KSPLIT_EXACT = 1,  /* only splits whose result is bit-identical to
                                 the unsplit schedule (chained stream-K) */
    SBGEMM_KSPLIT_NONE = 2    /* never split K */
};

/* sbgemm_plan_info.stream_k. */
enum {
    SBGEMM_STREAM_K_NONE = 0,     /* every tile computed whole by one CTA */
    SBGEMM_STREAM_K_CHAINED = 1,  /* last waves split; a tail continues its
                                     head's k-ordered accumulation, so results
                                     do not change */
    SBGEMM_STREAM_K_PIECES = 2    /* all tiles split into independent K pieces
                                     over the SMs, the tail adding the earlier
                                     pieces' partial sums latest first (on the
                                     gather path the tile's last CTA adds all
                                     pieces in piece order) */
};

typedef struct {
    int math;          /* SBGEMM_MATH_* */
    int force_path;    /* SBGEMM_PATH_AUTO or a specific path */
    void* workspace;   /* optional device scratch owned by the caller, 256-byte
                          aligned, at least sbgemm_workspace_bytes() long; NULL
                          = none.  With it the planner may split the last waves
                          of tiles along K across all SMs (stream-K).  The
                          library writes it on `stream` during the call; calls
                          that may run concurrently need separate workspaces. */
    size_t workspace_bytes;
    int k_split;       /* SBGEMM_KSPLIT_*; 0 = any */
    int reserved[1];   /* must be zero */
} sbgemm_options;

typedef struct {
    int path;                 /* SBGEMM_PATH_* chosen (NONE: no launch) */
    int a_layout, b_layout, c_layout;   /* SBGEMM_LAYOUT_* */
    int a_broadcast, b_broadcast;       /* batch stride 0 with batch > 1 */
    int a_tma, b_tma;         /* operand can be fetched by a TMA tensor map */
    int tile_m, tile_n, tile_k;
    int ctas_per_sm;          /* resident CTAs per SM the plan assumes */
    int64_t ctas;             /* CTAs launched (0 when path == NONE) */
    int64_t tiles;            /* output tiles over all batch entries */
    int stream_k;             /* SBGEMM_STREAM_K_*: how tiles are split along K
                                 (needs a workspace) */
    int k_slices;             /* K slices (tile_k deep) per tile */
    int64_t dp_tiles;         /* tiles computed whole, data-parallel */
    int reserved[4];
} sbgemm_plan_info;

/* Activation of the fused epilogue; sbgemm_epilogue.activation.  The pages
 * name ReLU, GeluTanh and GeluExact ("Chapter 09 CUDA backend", section
 * "Elementwise"), the sigmoid ("PyTorch demystified 3") and SiLU ("rvllm
 * CUDA path", the FFN's silu(gate)). */
enum {
    SBGEMM_ACT_NONE = 0,
    SBGEMM_ACT_RELU = 1,       /* max(z, 0) */
    SBGEMM_ACT_SIGMOID = 2,    /* 1 / (1 + e^-z) */
    SBGEMM_ACT_SILU = 3,       /* z / (1 + e^-z) */
    SBGEMM_ACT_GELU_TANH = 4,  /* z/2 (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))) */
    SBGEMM_ACT_GELU_ERF = 5    /* z/2 (1 + erf(z / sqrt(2))) */
};

/* Fused epilogue of sbgemm_fused:
 *     C[b,m,n] <- act(alpha * (A*B)[b,m,n] + (accumulate ? C_old[b,m,n] : 0) + D[b,m,n])
 * with D[b,m,n] = D[b*bsD + m*rsD + n*csD] (strides in fp32 elements; zero
 * strides broadcast, so a bias per output column is rsD = 0, csD = 1, bsD = 0,
 * and a bias per batch entry and column is bsD = N).  The fusion of
 * "PyTorch demystified 3", section "Summary": the feed-forward layer's bias is
 * added inside the matmul kernel, saving a pass over C and a launch.
 * Rounding: alpha*acc (+ C_old) as sbgemm forms it, one fp32 add of D, then
 * the activation in fp32 through the CUDA math library. */
typedef struct {
    const float* D;            /* NULL = no addend; device memory, 4-byte aligned,
                                  its span must not meet C's */
    int64_t rsD, csD, bsD;
    int activation;            /* SBGEMM_ACT_* */
    int reserved[3];           /* must be zero */
} sbgemm_epilogue;

/* Strict fp32 product on the CUDA cores; the planner picks the kernel.
 * Arguments as described above; stream is a cudaStream_t (NULL = default). */
SBGEMM_API int sbgemm(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
           const float* B, int64_t rsB, int64_t csB, int64_t bsB,
           float* C, int64_t rsC, int64_t csC, int64_t bsC,
           int64_t M, int64_t N, int64_t K, int64_t batch,
           float alpha, int accumulate, void* stream);

/* As sbgemm, with the arithmetic and the kernel path chosen by `opt` (NULL =
 * defaults).  math = SBGEMM_MATH_TF32 opts in to the tensor cores; when the
 * operands cannot be fetched by TMA (each needs a unit stride along K or
 * along its M / N index), the planner falls back to strict fp32 unless the
 * TF32 path was forced (then SBGEMM_ERR_UNSUPPORTED). */
SBGEMM_API int sbgemm_ex(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
              const float* B, int64_t rsB, int64_t csB, int64_t bsB,
              float* C, int64_t rsC, int64_t csC, int64_t bsC,
              int64_t M, int64_t N, int64_t K, int64_t batch,
              float alpha, int accumulate, void* stream,
              const sbgemm_options* opt);

/* As sbgemm_ex, with a fused epilogue (NULL = none: same as sbgemm_ex).  All
 * paths and schedules apply it once per output, after the last K slice.  With
 * an epilogue, K == 0 with accumulate writes act(C_old + D) instead of
 * leaving C unchanged.  Errors as sbgemm_ex, plus SBGEMM_ERR_INVALID_VALUE for
 * an unknown activation, non-zero reserved fields, a misaligned D or a D span
 * overflowing int64; SBGEMM_ERR_OUTPUT_OVERLAP when D's span meets C's (or the
 * workspace); SBGEMM_ERR_NOT_DEVICE_MEMORY when D is not inside one device
 * allocation. */
SBGEMM_API int sbgemm_fused(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
                 const float* B, int64_t rsB, int64_t csB, int64_t bsB,
                 float* C, int64_t rsC, int64_t csC, int64_t bsC,
                 int64_t M, int64_t N, int64_t K, int64_t batch,
                 float alpha, int accumulate, const sbgemm_epilogue* epi,
                 void* stream, const sbgemm_options* opt);

/* Fused attention over a batch of (sequence, head) problems, every operand
 * laid out by strides in fp32 elements like the product's:
 *     O[b,m,e] = sum_n softmax_n(alpha * sum_d Q[b,m,d] K[b,n,d]) V[b,n,e]
 * with Q[b,m,d] = Q[b*bsQ + m*rsQ + d*csQ], K[b,n,d], V[b,n,e] and O[b,m,e]
 * alike.  The pages compute attention as three steps (scores, softmax,
 * probs @ V) with the scores in global memory between them and name a fused
 * kernel as the fix ("rvllm CUDA path", section "What's basic about it");
 * here the scores and probabilities stay on chip.  Grouped-query heads are
 * rows of one batch entry stacked against one K and V ("rvllm CUDA path",
 * section "Matmuls go to cuBLAS").
 *   causal: 0, or 1 to mask keys n > position(m) = (m mod q_len) + N - q_len
 *           (q_len: query rows per head, 0 < q_len <= N; ignored when 0).
 *   D, Dv:  head dimensions; this build supports D = Dv = 32, 64, 96 or 128.
 * fp32 arithmetic: scores by FFMA, the softmax with exp2 of alpha*log2(e)
 * scaled scores, P V by FFMA.  Up to 8 query rows per batch entry (4 when D
 * is 96 or 128), a decode step, run a kernel that splits each entry's keys
 * across CTAs when sbgemm_attention_ex gives it a workspace (one CTA per
 * entry without one).  Asynchronous on `stream`; allocates nothing.
 * Errors: SBGEMM_ERR_INVALID_VALUE (negative size, N == 0 with rows to
 * compute, a bad causal flag or q_len, misaligned pointer, span overflow),
 * SBGEMM_ERR_NULL_POINTER, SBGEMM_ERR_OUTPUT_OVERLAP (O not injective or
 * meeting Q, K or V), SBGEMM_ERR_UNSUPPORTED (another head dimension, M over
 * 65535 x 128 rows), SBGEMM_ERR_NOT_DEVICE_MEMORY, SBGEMM_ERR_CUDA.  M, batch
 * or Dv zero: nothing to do. */
SBGEMM_API int sbgemm_attention(const float* Q, int64_t rsQ, int64_t csQ, int64_t bsQ,
                     const float* K, int64_t rsK, int64_t csK, int64_t bsK,
                     const float* V, int64_t rsV, int64_t csV, int64_t bsV,
                     float* O, int64_t rsO, int64_t csO, int64_t bsO,
                     int64_t M, int64_t N, int64_t D, int64_t Dv, int64_t batch,
                     float alpha, int causal, int64_t q_len, void* stream);

/* sbgemm_attention with options.  opt->math = SBGEMM_MATH_TF32 opts in to the
 * tensor-core kernel: S = Q K^T and P V by tcgen05 MMAs (tf32 inputs, fp32
 * accumulation), the softmax in fp32 as above.  It takes Q, K and V with unit
 * stride along the head dimension (csQ = csK = csV = 1), 16-byte aligned bases
 * and row / batch strides (a zero batch stride broadcasts); other layouts run
 * the fp32 kernel, unless opt->force_path = SBGEMM_PATH_TMA_TF32, which then
 * returns SBGEMM_ERR_UNSUPPORTED.  Problems of a few rows per entry (see
 * sbgemm_attention) run the fp32 decode kernel in either math unless the
 * tensor-core kernel is forced.  opt->workspace (caller-owned device memory
 * of opt->workspace_bytes, meeting no operand) lets the decode kernel split
 * the keys of an entry into chunks, each writing (2 + Dv) floats per row,
 * that a second launch merges in chunk order; sbgemm_workspace_bytes is
 * plenty.  k_split is ignored; force_path must be AUTO or TMA_TF32 (TMA_TF32
 * with math = TF32).  NULL opt is sbgemm_attention.  Errors as
 * sbgemm_attention, plus those of the options and of the workspace
 * (SBGEMM_ERR_NOT_DEVICE_MEMORY, SBGEMM_ERR_OUTPUT_OVERLAP). */
SBGEMM_API int sbgemm_attention_ex(const float* Q, int64_t rsQ, int64_t csQ, int64_t bsQ,
                        const float* K, int64_t rsK, int64_t csK, int64_t bsK,
                        const float* V, int64_t rsV, int64_t csV, int64_t bsV,
                        float* O, int64_t rsO, int64_t csO, int64_t bsO,
                        int64_t M, int64_t N, int64_t D, int64_t Dv, int64_t batch,
                        float alpha, int causal, int64_t q_len, void* stream,
                        const sbgemm_options* opt);

/* Fused attention reading K and V straight out of a paged cache through a
 * block table ("rvllm CUDA path", section "The kernels": the cache is one
 * buffer [num_blocks][block_size][n_kv_heads][head_dim], and context position
 * pos of a sequence lives in block block_table[seq * max_blocks + pos /
 * block_size] at offset pos % block_size; section "What's basic about it":
 * reading the blocks directly instead of gathering the whole context into a
 * contiguous buffer every decode step).
 *   K_cache, V_cache: [num_blocks][block_size][n_kv_heads][D] and [..][Dv]
 *           fp32, contiguous, 16-byte aligned.
 *   block_table: int32 [n_seqs][max_blocks] on the device; entries past a
 *           sequence's last block are never read.
 *   seq_lens: int32 [n_seqs] on the device, each sequence's context length
 *           (1..N, and >= q_len when causal), or NULL for N everywhere.
 *   N:      the longest context, at most max_blocks * block_size.
 *   Q, O:   strided like sbgemm_attention's, batch entry b = seq * n_kv_heads
 *           + head, M rows each (grouped-query heads stacked as rows);
 *           causal positions use the entry's own length:
 *           position(m) = (m mod q_len) + len - q_len.
 * O[b] is sbgemm_attention of Q[b] against the keys and values of positions
 * 0..len-1 of (seq, head).  D = Dv = 32, 64, 96 or 128; fp32 arithmetic as
 * sbgemm_attention (opt->math is not read); few-row problems use the decode
 * kernel and opt->workspace as sbgemm_attention_ex, others the row-block
 * kernel.  The host checks sizes, spans and overlaps as sbgemm_attention
 * (the caches, the table and seq_lens as operands O must not meet); the
 * table's and seq_lens' contents are device data and are checked by the
 * kernels: a block id outside [0, num_blocks) reads as a zero key and value,
 * a length out of range is clamped, and either makes the next
 * sbgemm_device_status return SBGEMM_ERR_DEVICE_CHECK (code 10); no access
 * leaves the caches.  opt->force_path must be AUTO.  Asynchronous on
 * `stream`; allocates nothing. */
SBGEMM_API int sbgemm_attention_paged(const float* Q, int64_t rsQ, int64_t csQ, int64_t bsQ,
                                      const float* K_cache, const float* V_cache,
                                      int64_t num_blocks, int64_t block_size, int64_t n_kv_heads,
                                      const int32_t* block_table, int64_t max_blocks,
                                      const int32_t* seq_lens,
                                      float* O, int64_t rsO, int64_t csO, int64_t bsO,
                                      int64_t M, int64_t N, int64_t D, int64_t Dv, int64_t n_seqs,
                                      float alpha, int causal, int64_t q_len, void* stream,
                                      const sbgemm_options* opt);

/* Validate and plan without launching or touching device memory: reports the
 * layout classes and the kernel path, tile and CTA count that sbgemm_ex would
 * use.  Pointers are only checked for NULL and alignment (no device query). */
SBGEMM_API int sbgemm_plan(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
                const float* B, int64_t rsB, int64_t csB, int64_t bsB,
                const float* C, int64_t rsC, int64_t csC, int64_t bsC,
                int64_t M, int64_t N, int64_t K, int64_t batch,
                int accumulate, const sbgemm_options* opt,
                sbgemm_plan_info* info);

/* Workspace size that lets sbgemm_ex use the stream-K schedule on `device`
 * (one fp32 tile of partial sums per SM plus one flag word per SM); the
 * gather path's K pieces of small products fit in it too.  Returns
 * SBGEMM_OK and writes *bytes, or SBGEMM_ERR_CUDA if the device cannot be
 * queried. */
SBGEMM_API int sbgemm_workspace_bytes(int device, size_t* bytes);

/* Size in bytes of sbgemm_noalloc's scratch array (20 MiB + 4 KiB). */
#define SBGEMM_NOALLOC_SCRATCH_BYTES ((size_t)20 * 1024 * 1024 + 4096)

/* The fp32 product for callers that cannot allocate device memory.
 * The paper has no counterpart: it exists because the stream-K schedule (and
 * the K pieces of small products) needs scratch that sbgemm_ex takes from its
 * caller, and some callers cannot make any (code running under CUDA graph
 * capture, plugins given only their input and output buffers, loops that
 * must not pay cudaMalloc's synchronisation, runtimes whose allocator owns
 * all device memory).
 *
 * Arguments, layout and errors are those of sbgemm.  The call is sbgemm_ex
 * with math = FP32, the automatic path, k_split = SBGEMM_KSPLIT_ANY and the
 * library's scratch as the workspace, so its results are bit-identical to
 * sbgemm_ex given those options and a workspace of
 * SBGEMM_NOALLOC_SCRATCH_BYTES.  Against sbgemm (no workspace) they can
 * differ in rounding, within the fp32 bound, for the products the planner
 * cuts into independent K pieces (few output tiles with a long K, or small
 * products on the gather path): those pieces are summed in a fixed order
 * rather than in one k-ordered chain.
 *
 * The scratch is a file-scope device array of SBGEMM_NOALLOC_SCRATCH_BYTES
 * inside the library (room for the schedule on devices of up to 160 SMs),
 * created when the library's module is loaded and held on every GPU that
 * loads the library until the process exits.  Nothing is allocated per call:
 * no cudaMalloc, cudaFree or allocating library routine runs.  The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current; make that first call before any stream capture
 * (a first call on a capturing stream returns SBGEMM_ERR_CUDA without
 * touching the stream, and a failed lookup is retried by the next call).
 * Every call shares the one array, which keeps the last call's contents; the
 * schedule clears its flags and counters on `stream` before each launch.
 * Calls that overlap on the GPU (different streams, or different host
 * threads) race on the scratch and must be serialised by the caller.
 * Returns SBGEMM_ERR_UNSUPPORTED if the current device would need more
 * scratch than the array holds (more than 160 SMs). */
SBGEMM_API int sbgemm_noalloc(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
                              const float* B, int64_t rsB, int64_t csB, int64_t bsB,
                              float* C, int64_t rsC, int64_t csC, int64_t bsC,
                              int64_t M, int64_t N, int64_t K, int64_t batch,
                              float alpha, int accumulate, void* stream);

/* Reads and clears the device-side status words that kernels set when a
 * bounded in-kernel wait gives up or a device-side check skips an input
 * (after synchronising `stream`; the first code recorded is kept).  Returns
 * SBGEMM_OK, SBGEMM_ERR_DEVICE_TIMEOUT (codes 1-8) or SBGEMM_ERR_DEVICE_CHECK
 * (codes 9-10); *where_out (may be NULL) receives the code (0 if none): 1 a
 * loaded stage, 2 a released stage, 3 copies in flight at exit, 4 the MMAs of
 * a tile, 5 a free accumulator, 6 a stream-K partial sum, 7 / 8 the
 * self-test's mbarrier / flag, 9 an address outside its operand's span (debug
 * builds only; the access was skipped), 10 a paged-attention block id or
 * sequence length out of range. */
SBGEMM_API int sbgemm_device_status(void* stream, int* where_out);

/* Failure-detection self-test (a diagnostic of the library, not part of the
 * product).  Launches one CTA on `stream` that waits, with the bounded-wait
 * helpers every kernel uses and a limit of `limit_us` microseconds (1 ..
 * 2,000,000), on a condition nothing satisfies: an mbarrier phase that never
 * completes (SBGEMM_SELFTEST_MBARRIER) or a global flag no code sets
 * (SBGEMM_SELFTEST_FLAG).  The wait gives up, records its code, and the kernel
 * returns; the context stays usable and the next sbgemm_device_status call
 * returns SBGEMM_ERR_DEVICE_TIMEOUT with that code.  Returns SBGEMM_OK once
 * launched, SBGEMM_ERR_INVALID_VALUE for an unknown test or limit. */
enum { SBGEMM_SELFTEST_MBARRIER = 1, SBGEMM_SELFTEST_FLAG = 2 };
SBGEMM_API int sbgemm_selftest(int what, int64_t limit_us, void* stream);

/* Static, human-readable name of a status code. */
SBGEMM_API const char* sbgemm_status_string(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
SBGEMM_API int sbgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SBGEMM_H */
