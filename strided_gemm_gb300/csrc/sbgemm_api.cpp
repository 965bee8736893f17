// C-ABI boundary: argument validation, operand layout classification, kernel
// planning and dispatch for the strided batched product.
//
// The checks follow the StaleyNET "GPU Implementation" page, section "Safety":
// every size the kernel depends on is checked before the launch, so a launch
// never reads or writes memory outside what the caller described.
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cstdint>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <utility>

#include "attention_tc.h"
#include "internal.h"
#include "sbgemm.h"

namespace sbg {

// ---- device properties ------------------------------------------------------

namespace {
constexpr int kMaxDevices = 64;
std::array<std::once_flag, kMaxDevices> g_props_once;
std::array<DeviceProps, kMaxDevices> g_props;
std::array<bool, kMaxDevices> g_props_ok{};
}  // namespace

const DeviceProps* device_props(int device) {
    if (device < 0 || device >= kMaxDevices) return nullptr;
    std::call_once(g_props_once[device], [device] {
        DeviceProps d{};
        d.device = device;
        bool ok = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.max_smem_per_block_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.max_smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, device) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, device) == cudaSuccess;
        g_props[device] = d;
        g_props_ok[device] = ok;
    });
    return g_props_ok[device] ? &g_props[device] : nullptr;
}

namespace {

inline int64_t mag(int64_t x) { return x < 0 ? -x : x; }

// Element-offset span [lo, hi] of an operand over its [batch][rows][cols] box.
// Returns false if the span does not fit comfortably in int64 byte offsets.
struct Span { int64_t lo, hi; };

bool operand_span(int64_t batch, int64_t rows, int64_t cols,
                  int64_t bs, int64_t rs, int64_t cs, Span* out) {
    __int128 lo = 0, hi = 0;
    const int64_t st[3] = {bs, rs, cs};
    const int64_t ex[3] = {batch, rows, cols};
    for (int i = 0; i < 3; ++i) {
        __int128 d = (__int128)st[i] * (ex[i] - 1);
        if (d < 0) lo += d; else hi += d;
    }
    const __int128 limit = (__int128)1 << 60;   // elements; 4x that in bytes
    if (lo < -limit || hi > limit) return false;
    out->lo = (int64_t)lo;
    out->hi = (int64_t)hi;
    return true;
}

// Distinct (b, m, n) map to distinct elements: sorted by stride magnitude,
// each stride must exceed the largest offset reachable by the smaller ones.
// This sufficient test rejects a few exotic injective layouts as overlapping.
bool output_injective(int64_t batch, int64_t M, int64_t N,
                      int64_t bs, int64_t rs, int64_t cs) {
    std::array<std::pair<int64_t, int64_t>, 3> d = {{{mag(bs), batch}, {mag(rs), M}, {mag(cs), N}}};
    std::sort(d.begin(), d.end());
    __int128 reach = 0;
    for (auto& [s, e] : d) {
        if (e <= 1) continue;
        if ((__int128)s <= reach) return false;
        reach += (__int128)s * (e - 1);
    }
    return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int classify_a(const Problem& p) {
    if (p.K == 1 || p.csA == 1) return SBGEMM_LAYOUT_K_MAJOR;
    if (p.M == 1 || p.rsA == 1) return SBGEMM_LAYOUT_MN_MAJOR;
    return SBGEMM_LAYOUT_GENERAL;
}
int classify_b(const Problem& p) {
    if (p.K == 1 || p.rsB == 1) return SBGEMM_LAYOUT_K_MAJOR;
    if (p.N == 1 || p.csB == 1) return SBGEMM_LAYOUT_MN_MAJOR;
    return SBGEMM_LAYOUT_GENERAL;
}
int classify_c(const Problem& p) {
    if (p.N == 1 || p.csC == 1) return SBGEMM_LAYOUT_K_MAJOR;
    if (p.M == 1 || p.rsC == 1) return SBGEMM_LAYOUT_MN_MAJOR;
    return SBGEMM_LAYOUT_GENERAL;
}

// A TMA tensor map can describe the operand: a unit stride on its inner index,
// a 16-byte aligned base, outer / batch strides that are positive multiples of
// 16 bytes below 2^40 laid out without overlap (outer stride >= inner extent,
// batch stride >= one matrix), and extents that fit 32-bit tile coordinates.
// A stride over an extent of 1 is never used and is not checked.
bool tma_eligible(const void* base, int layout, int64_t outer_stride, int64_t outer_extent,
                  int64_t bs, int64_t batch, int64_t inner_extent) {
    if (layout == SBGEMM_LAYOUT_GENERAL) return false;
    if (!aligned(base, 16)) return false;
    const int64_t lim = (int64_t)1 << 31;
    if (inner_extent >= lim || outer_extent >= lim || batch >= lim) return false;
    auto ok_stride = [](int64_t s) { return s > 0 && (s * 4) % 16 == 0 && (s * 4) < ((int64_t)1 << 40); };
    if (outer_extent > 1 && (!ok_stride(outer_stride) || outer_stride < inner_extent)) return false;
    if (batch > 1 && bs != 0) {
        if (!ok_stride(bs)) return false;
        const int64_t one = outer_extent > 1 ? outer_stride * outer_extent : inner_extent;
        if (bs < one) return false;
    }
    return true;
}

int check_options(const sbgemm_options* opt, sbgemm_options* out) {
    sbgemm_options o{};
    if (opt) o = *opt;
    if (o.math != SBGEMM_MATH_FP32 && o.math != SBGEMM_MATH_TF32) return SBGEMM_ERR_INVALID_VALUE;
    if (o.force_path < SBGEMM_PATH_AUTO || o.force_path > SBGEMM_PATH_TMA_TF32) return SBGEMM_ERR_INVALID_VALUE;
    if (o.k_split < SBGEMM_KSPLIT_ANY || o.k_split > SBGEMM_KSPLIT_NONE) return SBGEMM_ERR_INVALID_VALUE;
    for (int r : o.reserved) if (r != 0) return SBGEMM_ERR_INVALID_VALUE;
    if (o.workspace && (reinterpret_cast<uintptr_t>(o.workspace) % 256) != 0)
        return SBGEMM_ERR_INVALID_VALUE;
    *out = o;
    return SBGEMM_OK;
}

// Host-side checks that need no device.  Fills the spans of A, B and C.
int validate(const Problem& p, Span* sa, Span* sb, Span* sc, bool* empty) {
    if (p.M < 0 || p.N < 0 || p.K < 0 || p.batch < 0) return SBGEMM_ERR_INVALID_VALUE;
    *empty = (p.M == 0 || p.N == 0 || p.batch == 0);
    if (*empty) return SBGEMM_OK;
    if (!p.C) return SBGEMM_ERR_NULL_POINTER;
    if (p.K > 0 && (!p.A || !p.B)) return SBGEMM_ERR_NULL_POINTER;
    if (!aligned(p.C, 4) || (p.K > 0 && (!aligned(p.A, 4) || !aligned(p.B, 4))))
        return SBGEMM_ERR_INVALID_VALUE;
    if (!operand_span(p.batch, p.M, p.N, p.bsC, p.rsC, p.csC, sc)) return SBGEMM_ERR_INVALID_VALUE;
    if (p.K > 0) {
        if (!operand_span(p.batch, p.M, p.K, p.bsA, p.rsA, p.csA, sa)) return SBGEMM_ERR_INVALID_VALUE;
        if (!operand_span(p.batch, p.K, p.N, p.bsB, p.rsB, p.csB, sb)) return SBGEMM_ERR_INVALID_VALUE;
    }
    if (!output_injective(p.batch, p.M, p.N, p.bsC, p.rsC, p.csC)) return SBGEMM_ERR_OUTPUT_OVERLAP;
    if (p.K > 0) {
        auto bytes = [](const void* base, const Span& s, __int128* lo, __int128* hi) {
            *lo = (__int128)reinterpret_cast<uintptr_t>(base) + (__int128)s.lo * 4;
            *hi = (__int128)reinterpret_cast<uintptr_t>(base) + (__int128)s.hi * 4 + 4;
        };
        __int128 clo, chi, lo, hi;
        bytes(p.C, *sc, &clo, &chi);
        bytes(p.A, *sa, &lo, &hi);
        if (lo < chi && clo < hi) return SBGEMM_ERR_OUTPUT_OVERLAP;
        bytes(p.B, *sb, &lo, &hi);
        if (lo < chi && clo < hi) return SBGEMM_ERR_OUTPUT_OVERLAP;
    }
    return SBGEMM_OK;
}

// Allocation ranges already looked up during one call: an operand whose span
// lies inside one of them needs no driver query (operands in one pool
// segment, or views of one buffer, share a lookup).  Lives for one call only,
// so it never outlasts an allocation.
struct Ranges {
    int n = 0;
    uintptr_t base[8];
    size_t size[8];
};

// The operand's whole span lies inside one device-accessible allocation.
bool span_in_allocation(const void* base, const Span& s, Ranges* seen = nullptr) {
    const __int128 lo = (__int128)reinterpret_cast<uintptr_t>(base) + (__int128)s.lo * 4;
    const __int128 hi = (__int128)reinterpret_cast<uintptr_t>(base) + (__int128)s.hi * 4 + 4;
    if (seen)
        for (int i = 0; i < seen->n; ++i)
            if (lo >= (__int128)seen->base[i] && hi <= (__int128)seen->base[i] + (__int128)seen->size[i])
                return true;
    uintptr_t abase = 0;
    size_t asize = 0;
    if (!device_allocation_range(base, &abase, &asize)) return false;
    if (seen && seen->n < 8) {
        seen->base[seen->n] = abase;
        seen->size[seen->n] = asize;
        ++seen->n;
    }
    return lo >= (__int128)abase && hi <= (__int128)abase + (__int128)asize;
}

bool bytes_meet(const void* a, const Span& sa, const void* b, const Span& sb) {
    const __int128 alo = (__int128)reinterpret_cast<uintptr_t>(a) + (__int128)sa.lo * 4;
    const __int128 ahi = (__int128)reinterpret_cast<uintptr_t>(a) + (__int128)sa.hi * 4 + 4;
    const __int128 blo = (__int128)reinterpret_cast<uintptr_t>(b) + (__int128)sb.lo * 4;
    const __int128 bhi = (__int128)reinterpret_cast<uintptr_t>(b) + (__int128)sb.hi * 4 + 4;
    return alo < bhi && blo < ahi;
}

// An attention workspace, when given, is device memory that meets no operand
// (the decode kernel writes its per-chunk partial results there).
int check_attention_workspace(const sbgemm_options& o,
                              std::initializer_list<std::pair<const void*, Span>> operands) {
    if (!o.workspace) return SBGEMM_OK;
    if (o.workspace_bytes < 4) return SBGEMM_ERR_INVALID_VALUE;
    const Span sw{0, (int64_t)(o.workspace_bytes / 4) - 1};
    if (!span_in_allocation(o.workspace, sw)) return SBGEMM_ERR_NOT_DEVICE_MEMORY;
    for (const auto& op : operands)
        if (bytes_meet(op.first, op.second, o.workspace, sw)) return SBGEMM_ERR_OUTPUT_OVERLAP;
    return SBGEMM_OK;
}

int make_plan(const Problem& p, const sbgemm_options& o, int sm_count, bool empty, Plan* plan) {
    *plan = Plan{};
    // K == 0 with accumulation leaves C as it is, unless an epilogue applies.
    if (empty || (p.K == 0 && p.accumulate && !p.epi.on)) {
        plan->path = SBGEMM_PATH_NONE;
        return SBGEMM_OK;
    }
    plan->a_layout = classify_a(p);
    plan->b_layout = classify_b(p);
    plan->c_layout = classify_c(p);
    plan->a_broadcast = p.batch > 1 && p.bsA == 0;
    plan->b_broadcast = p.batch > 1 && p.bsB == 0;
    if (p.K > 0) {
        // A: inner index K (K-major) or M; B: inner index K (K-major) or N.
        const bool ak = plan->a_layout == SBGEMM_LAYOUT_K_MAJOR;
        const bool bk = plan->b_layout == SBGEMM_LAYOUT_K_MAJOR;
        plan->a_tma = tma_eligible(p.A, plan->a_layout, ak ? p.rsA : p.csA, ak ? p.M : p.K,
                                   p.bsA, p.batch, ak ? p.K : p.M);
        plan->b_tma = tma_eligible(p.B, plan->b_layout, bk ? p.csB : p.rsB, bk ? p.N : p.K,
                                   p.bsB, p.batch, bk ? p.K : p.N);
    }

    const bool tma_ok = p.K > 0 && plan->a_tma && plan->b_tma;
    // The tensor-core path reads its operands K-major (unit stride along K);
    // an MN-major operand is transposed in shared memory on the way.
    const bool tf32_ok = tma_ok;
    int path = o.force_path;
    if (path == SBGEMM_PATH_TMA_TF32 && !tf32_ok) return SBGEMM_ERR_UNSUPPORTED;
    if (path == SBGEMM_PATH_TMA_FFMA && !tma_ok) return SBGEMM_ERR_UNSUPPORTED;
    if (path == SBGEMM_PATH_AUTO) {
        if (o.math == SBGEMM_MATH_TF32 && tf32_ok) {
            path = SBGEMM_PATH_TMA_TF32;
        } else if (tma_ok) {
            // The persistent TMA kernel's 256x128 tiles leave most SMs idle on
            // small products; the gather kernel's 64x64 tiles spread them wider.
            const TmaFfmaConfig c = tma_ffma_config(tma_ffma_pick_variant(p, sm_count));
            const int64_t tma_tiles = ((p.M + c.bm - 1) / c.bm) * ((p.N + c.bn - 1) / c.bn) * p.batch;
            path = tma_tiles >= sm_count / 4 ? SBGEMM_PATH_TMA_FFMA : SBGEMM_PATH_GATHER_FFMA;
        } else {
            path = SBGEMM_PATH_GATHER_FFMA;
        }
    }
    plan->path = path;

    if (path == SBGEMM_PATH_TMA_TF32) {
        // A K-major A with an N-major B is computed as C^T = B^T A^T: the
        // MN-major operand to transpose in shared memory is then the 128-row
        // one (B^T as A') instead of the 256-row one, and C^T goes out
        // through a tensor map with M' inner.  Below N = 128 the transposed
        // problem fills only part of the 128-row MMA, which such a narrow,
        // HBM-bound product can afford (c4, N = 64: 51 -> 45 us).
        const bool swap = plan->a_layout == SBGEMM_LAYOUT_K_MAJOR &&
                          plan->b_layout != SBGEMM_LAYOUT_K_MAJOR;
        const Problem q = swap ? transposed_problem(p) : p;
        const TmaFfmaConfig c = tf32_tc_config();
        plan->transposed = swap;
        plan->tile_m = swap ? c.bn : c.bm;   // reported in C's own orientation
        plan->tile_n = swap ? c.bm : c.bn;
        plan->tile_k = c.bk;
        plan->ctas_per_sm = 1;
        plan->tiles_m = (q.M + c.bm - 1) / c.bm;
        plan->tiles_n = (q.N + c.bn - 1) / c.bn;
        plan->tiles = plan->tiles_m * plan->tiles_n * q.batch;
        tf32_tc_schedule(q, *plan, sm_count, o.workspace ? o.workspace_bytes : 0, o.workspace,
                         o.k_split);
        tf32_tc_pair(q, *plan, sm_count, o.workspace ? o.workspace_bytes : 0, o.workspace, o.k_split);
        return SBGEMM_OK;
    }

    if (path == SBGEMM_PATH_TMA_FFMA) {
        const int v = tma_ffma_pick_variant(p, sm_count);
        const TmaFfmaConfig c = tma_ffma_config(v);
        plan->variant = v;
        plan->tile_m = c.bm;
        plan->tile_n = c.bn;
        plan->tile_k = c.bk;
        plan->ctas_per_sm = 1;
        plan->tiles_m = (p.M + c.bm - 1) / c.bm;
        plan->tiles_n = (p.N + c.bn - 1) / c.bn;
        plan->tiles = plan->tiles_m * plan->tiles_n * p.batch;
        tma_ffma_schedule(p, *plan, sm_count, o.workspace ? o.workspace_bytes : 0, o.workspace,
                          o.k_split);
        return SBGEMM_OK;
    }

    const int v = gather_pick_variant(p, sm_count);
    const GatherConfig g = gather_config(v);
    plan->variant = v;
    plan->tile_m = g.bm;
    plan->tile_n = g.bn;
    plan->tile_k = g.bk;
    plan->ctas_per_sm = g.ctas_per_sm;
    plan->tiles_m = (p.M + g.bm - 1) / g.bm;
    plan->tiles_n = (p.N + g.bn - 1) / g.bn;
    if (plan->tiles_m * plan->tiles_n >= ((int64_t)1 << 31)) return SBGEMM_ERR_UNSUPPORTED;
    plan->tiles = plan->tiles_m * plan->tiles_n * p.batch;
    plan->ctas = plan->tiles_m * plan->tiles_n * std::min<int64_t>(p.batch, 65535);
    gather_schedule(p, *plan, sm_count, o.workspace ? o.workspace_bytes : 0, o.workspace, o.k_split);
    return SBGEMM_OK;
}

Problem make_problem(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
                     const float* B, int64_t rsB, int64_t csB, int64_t bsB,
                     const float* C, int64_t rsC, int64_t csC, int64_t bsC,
                     int64_t M, int64_t N, int64_t K, int64_t batch,
                     float alpha, int accumulate) {
    Problem p;
    p.A = A; p.rsA = rsA; p.csA = csA; p.bsA = bsA;
    p.B = B; p.rsB = rsB; p.csB = csB; p.bsB = bsB;
    p.C = const_cast<float*>(C); p.rsC = rsC; p.csC = csC; p.bsC = bsC;
    p.M = M; p.N = N; p.K = K; p.batch = batch;
    p.alpha = alpha;
    p.accumulate = accumulate ? 1 : 0;
    p.epi = EpiParams{nullptr, 0, 0, 0, SBGEMM_ACT_NONE, 0, 0, ElemSpan{0, -1}};
    p.sa = p.sb = p.sc = ElemSpan{0, -1};
    return p;
}

}  // namespace

Problem transposed_problem(const Problem& p) {
    Problem q = p;
    q.A = p.B; q.rsA = p.csB; q.csA = p.rsB; q.bsA = p.bsB;
    q.B = p.A; q.rsB = p.csA; q.csB = p.rsA; q.bsB = p.bsA;
    q.rsC = p.csC; q.csC = p.rsC;
    q.M = p.N; q.N = p.M;
    q.sa = p.sb; q.sb = p.sa;
    q.epi.rsD = p.epi.csD; q.epi.csD = p.epi.rsD;
    q.epi.d_vec4 = q.epi.D && (q.epi.csD == 1 || q.N == 1) &&
                   (reinterpret_cast<uintptr_t>(q.epi.D) % 16 == 0) && q.epi.rsD % 4 == 0 &&
                   q.epi.bsD % 4 == 0;
    return q;
}

namespace {

void fill_info(const Plan& plan, sbgemm_plan_info* info) {
    std::memset(info, 0, sizeof(*info));
    info->path = plan.path;
    info->a_layout = plan.a_layout;
    info->b_layout = plan.b_layout;
    info->c_layout = plan.c_layout;
    info->a_broadcast = plan.a_broadcast;
    info->b_broadcast = plan.b_broadcast;
    info->a_tma = plan.a_tma;
    info->b_tma = plan.b_tma;
    info->tile_m = plan.tile_m;
    info->tile_n = plan.tile_n;
    info->tile_k = plan.tile_k;
    info->ctas_per_sm = plan.ctas_per_sm;
    info->ctas = plan.ctas;
    info->tiles = plan.tiles;
    info->stream_k = plan.stream_k ? (plan.split_indep ? SBGEMM_STREAM_K_PIECES : SBGEMM_STREAM_K_CHAINED)
                                   : SBGEMM_STREAM_K_NONE;
    info->k_slices = plan.k_slices;
    info->dp_tiles = plan.dp_tiles;
}

// SM count for planning: the current device's when one is present, otherwise
// the GB300 figure, so sbgemm_plan works on machines without a GPU.
int planning_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) {
        if (const DeviceProps* d = device_props(dev)) return d->sm_count;
    }
    cudaGetLastError();
    return 152;
}

// Validates, plans and launches one product (with its fused epilogue, if
// any) on `stream`.
int run(Problem& p, const sbgemm_options& o, void* stream) {
    Span sa{}, sb{}, sc{};
    bool empty = false;
    int st = validate(p, &sa, &sb, &sc, &empty);
    if (st) return st;
    if (empty || (p.K == 0 && p.accumulate && !p.epi.on)) return SBGEMM_OK;
    Span sd{};
    if (p.epi.D) {
        // The addend is read while C is written: it must be device memory
        // outside C's span.
        if (!aligned(p.epi.D, 4)) return SBGEMM_ERR_INVALID_VALUE;
        if (!operand_span(p.batch, p.M, p.N, p.epi.bsD, p.epi.rsD, p.epi.csD, &sd))
            return SBGEMM_ERR_INVALID_VALUE;
        const __int128 dlo = (__int128)reinterpret_cast<uintptr_t>(p.epi.D) + (__int128)sd.lo * 4;
        const __int128 dhi = (__int128)reinterpret_cast<uintptr_t>(p.epi.D) + (__int128)sd.hi * 4 + 4;
        const __int128 clo = (__int128)reinterpret_cast<uintptr_t>(p.C) + (__int128)sc.lo * 4;
        const __int128 chi = (__int128)reinterpret_cast<uintptr_t>(p.C) + (__int128)sc.hi * 4 + 4;
        if (dlo < chi && clo < dhi) return SBGEMM_ERR_OUTPUT_OVERLAP;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return SBGEMM_ERR_CUDA; }
    const DeviceProps* props = device_props(dev);
    if (!props) return SBGEMM_ERR_CUDA;

    Ranges seen;
    if (!span_in_allocation(p.C, sc, &seen)) return SBGEMM_ERR_NOT_DEVICE_MEMORY;
    if (p.K > 0 && (!span_in_allocation(p.A, sa, &seen) || !span_in_allocation(p.B, sb, &seen)))
        return SBGEMM_ERR_NOT_DEVICE_MEMORY;
    if (p.epi.D && !span_in_allocation(p.epi.D, sd, &seen)) return SBGEMM_ERR_NOT_DEVICE_MEMORY;

    // The validated spans, for the bounds checks of a debug build.
    p.sa = ElemSpan{sa.lo, sa.hi};
    p.sb = ElemSpan{sb.lo, sb.hi};
    p.sc = ElemSpan{sc.lo, sc.hi};
    if (p.epi.D) p.epi.d_span = ElemSpan{sd.lo, sd.hi};

    Plan plan;
    st = make_plan(p, o, props->sm_count, false, &plan);
    if (st) return st;

    if (plan.stream_k && plan.workspace) {
        // The workspace is written by the kernel: it must be device memory and
        // must not meet any operand.
        const Span sw{0, (int64_t)(o.workspace_bytes / 4) - 1};
        if (!span_in_allocation(o.workspace, sw, &seen)) return SBGEMM_ERR_NOT_DEVICE_MEMORY;
        auto meets = [&](const void* base, const Span& sp) {
            const __int128 lo = (__int128)reinterpret_cast<uintptr_t>(base) + (__int128)sp.lo * 4;
            const __int128 hi = (__int128)reinterpret_cast<uintptr_t>(base) + (__int128)sp.hi * 4 + 4;
            const __int128 wlo = (__int128)reinterpret_cast<uintptr_t>(o.workspace);
            const __int128 whi = wlo + (__int128)o.workspace_bytes;
            return lo < whi && wlo < hi;
        };
        if (meets(p.C, sc) || meets(p.A, sa) || meets(p.B, sb) || (p.epi.D && meets(p.epi.D, sd)))
            return SBGEMM_ERR_OUTPUT_OVERLAP;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err = cudaSuccess;
    switch (plan.path) {
        case SBGEMM_PATH_GATHER_FFMA: err = launch_gather_ffma(p, plan, s); break;
        case SBGEMM_PATH_TMA_FFMA: err = launch_tma_ffma(p, plan, props->sm_count, s); break;
        case SBGEMM_PATH_TMA_TF32:
            err = launch_tf32_tc(plan.transposed ? transposed_problem(p) : p, plan, props->sm_count, s);
            break;
        default: return SBGEMM_ERR_UNSUPPORTED;
    }
    if (err != cudaSuccess) { cudaGetLastError(); return SBGEMM_ERR_CUDA; }
    return SBGEMM_OK;
}

}  // namespace
}  // namespace sbg

using namespace sbg;

extern "C" {

int sbgemm_version(void) { return 100; }

const char* sbgemm_status_string(int status) {
    switch (status) {
        case SBGEMM_OK: return "SBGEMM_OK";
        case SBGEMM_ERR_INVALID_VALUE: return "SBGEMM_ERR_INVALID_VALUE";
        case SBGEMM_ERR_NULL_POINTER: return "SBGEMM_ERR_NULL_POINTER";
        case SBGEMM_ERR_OUTPUT_OVERLAP: return "SBGEMM_ERR_OUTPUT_OVERLAP";
        case SBGEMM_ERR_UNSUPPORTED: return "SBGEMM_ERR_UNSUPPORTED";
        case SBGEMM_ERR_CUDA: return "SBGEMM_ERR_CUDA";
        case SBGEMM_ERR_DEVICE_TIMEOUT: return "SBGEMM_ERR_DEVICE_TIMEOUT";
        case SBGEMM_ERR_NOT_DEVICE_MEMORY: return "SBGEMM_ERR_NOT_DEVICE_MEMORY";
        case SBGEMM_ERR_DEVICE_CHECK: return "SBGEMM_ERR_DEVICE_CHECK";
        default: return "SBGEMM_ERR_UNKNOWN";
    }
}

int sbgemm_plan(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
                const float* B, int64_t rsB, int64_t csB, int64_t bsB,
                const float* C, int64_t rsC, int64_t csC, int64_t bsC,
                int64_t M, int64_t N, int64_t K, int64_t batch,
                int accumulate, const sbgemm_options* opt,
                sbgemm_plan_info* info) {
    if (!info) return SBGEMM_ERR_NULL_POINTER;
    sbgemm_options o;
    int st = check_options(opt, &o);
    if (st) return st;
    Problem p = make_problem(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                             M, N, K, batch, 1.0f, accumulate);
    Span sa{}, sb{}, sc{};
    bool empty = false;
    st = validate(p, &sa, &sb, &sc, &empty);
    if (st) return st;
    Plan plan;
    st = make_plan(p, o, planning_sm_count(), empty, &plan);
    if (st) return st;
    fill_info(plan, info);
    return SBGEMM_OK;
}

int sbgemm_ex(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
              const float* B, int64_t rsB, int64_t csB, int64_t bsB,
              float* C, int64_t rsC, int64_t csC, int64_t bsC,
              int64_t M, int64_t N, int64_t K, int64_t batch,
              float alpha, int accumulate, void* stream,
              const sbgemm_options* opt) {
    sbgemm_options o;
    int st = check_options(opt, &o);
    if (st) return st;
    Problem p = make_problem(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                             M, N, K, batch, alpha, accumulate);
    return run(p, o, stream);
}

int sbgemm_fused(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
                 const float* B, int64_t rsB, int64_t csB, int64_t bsB,
                 float* C, int64_t rsC, int64_t csC, int64_t bsC,
                 int64_t M, int64_t N, int64_t K, int64_t batch,
                 float alpha, int accumulate, const sbgemm_epilogue* epi,
                 void* stream, const sbgemm_options* opt) {
    sbgemm_options o;
    int st = check_options(opt, &o);
    if (st) return st;
    Problem p = make_problem(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                             M, N, K, batch, alpha, accumulate);
    if (epi) {
        if (epi->activation < SBGEMM_ACT_NONE || epi->activation > SBGEMM_ACT_GELU_ERF)
            return SBGEMM_ERR_INVALID_VALUE;
        for (int r : epi->reserved) if (r != 0) return SBGEMM_ERR_INVALID_VALUE;
        const bool d_vec4 = epi->D && (epi->csD == 1 || N == 1) && aligned(epi->D, 16) &&
                            epi->rsD % 4 == 0 && epi->bsD % 4 == 0;
        p.epi = EpiParams{epi->D, epi->rsD, epi->csD, epi->bsD, epi->activation,
                          (epi->D != nullptr || epi->activation != SBGEMM_ACT_NONE) ? 1 : 0,
                          d_vec4 ? 1 : 0, ElemSpan{0, -1}};
    }
    return run(p, o, stream);
}

int sbgemm_attention_ex(const float* Q, int64_t rsQ, int64_t csQ, int64_t bsQ,
                        const float* K, int64_t rsK, int64_t csK, int64_t bsK,
                        const float* V, int64_t rsV, int64_t csV, int64_t bsV,
                        float* O, int64_t rsO, int64_t csO, int64_t bsO,
                        int64_t M, int64_t N, int64_t D, int64_t Dv, int64_t batch,
                        float alpha, int causal, int64_t q_len, void* stream,
                        const sbgemm_options* opt) {
    sbgemm_options o;
    const int ost = check_options(opt, &o);
    if (ost) return ost;
    if (o.force_path != SBGEMM_PATH_AUTO && o.force_path != SBGEMM_PATH_TMA_TF32)
        return SBGEMM_ERR_UNSUPPORTED;
    if (o.force_path == SBGEMM_PATH_TMA_TF32 && o.math != SBGEMM_MATH_TF32) return SBGEMM_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || D < 0 || Dv < 0 || batch < 0) return SBGEMM_ERR_INVALID_VALUE;
    if (causal != 0 && causal != 1) return SBGEMM_ERR_INVALID_VALUE;
    if (M == 0 || batch == 0 || Dv == 0) return SBGEMM_OK;
    if (N == 0) return SBGEMM_ERR_INVALID_VALUE;          // a softmax over no keys
    if (causal && (q_len <= 0 || q_len > N)) return SBGEMM_ERR_INVALID_VALUE;
    if (!attention_supported(D, Dv)) return SBGEMM_ERR_UNSUPPORTED;
    if (M > attention_max_rows() || batch >= ((int64_t)1 << 31)) return SBGEMM_ERR_UNSUPPORTED;
    if (!Q || !K || !V || !O) return SBGEMM_ERR_NULL_POINTER;
    if (!aligned(Q, 4) || !aligned(K, 4) || !aligned(V, 4) || !aligned(O, 4))
        return SBGEMM_ERR_INVALID_VALUE;
    Span sq{}, sk{}, sv{}, so{};
    if (!operand_span(batch, M, D, bsQ, rsQ, csQ, &sq) || !operand_span(batch, N, D, bsK, rsK, csK, &sk) ||
        !operand_span(batch, N, Dv, bsV, rsV, csV, &sv) || !operand_span(batch, M, Dv, bsO, rsO, csO, &so))
        return SBGEMM_ERR_INVALID_VALUE;
    if (!output_injective(batch, M, Dv, bsO, rsO, csO)) return SBGEMM_ERR_OUTPUT_OVERLAP;
    if (bytes_meet(O, so, Q, sq) || bytes_meet(O, so, K, sk) || bytes_meet(O, so, V, sv))
        return SBGEMM_ERR_OUTPUT_OVERLAP;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return SBGEMM_ERR_CUDA; }
    Ranges seen;
    if (!span_in_allocation(Q, sq, &seen) || !span_in_allocation(K, sk, &seen) ||
        !span_in_allocation(V, sv, &seen) || !span_in_allocation(O, so, &seen))
        return SBGEMM_ERR_NOT_DEVICE_MEMORY;
    const int wst = check_attention_workspace(o, {{Q, sq}, {K, sk}, {V, sv}, {O, so}});
    if (wst) return wst;
    AttnProblem a{Q, rsQ, csQ, bsQ, K, rsK, csK, bsK, V, rsV, csV, bsV, O, rsO, csO, bsO,
                  M, N, D, Dv, batch, alpha, causal, causal ? q_len : M,
                  ElemSpan{sq.lo, sq.hi}, ElemSpan{sk.lo, sk.hi}, ElemSpan{sv.lo, sv.hi},
                  ElemSpan{so.lo, so.hi}};
    a.workspace = o.workspace;
    a.workspace_bytes = o.workspace ? o.workspace_bytes : 0;
    // Forced: the tensor-core kernel.  Otherwise a few rows per entry go to the
    // split-key decode kernel (fp32, in either math), and the rest to the
    // tensor-core kernel when TF32 is asked for and the operands suit tensor
    // maps, else to the fp32 kernel.
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (o.force_path == SBGEMM_PATH_TMA_TF32) {
        if (!attention_tc_supported(a)) return SBGEMM_ERR_UNSUPPORTED;
        e = launch_attention_tc(a, s);
    } else if (attention_decode_supported(a)) {
        e = launch_attention_decode(a, s);
    } else if (o.math == SBGEMM_MATH_TF32 && attention_tc_supported(a)) {
        e = launch_attention_tc(a, s);
    } else {
        e = launch_attention(a, s);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SBGEMM_ERR_CUDA;
    }
    return SBGEMM_OK;
}

int sbgemm_attention_paged(const float* Q, int64_t rsQ, int64_t csQ, int64_t bsQ,
                           const float* K_cache, const float* V_cache,
                           int64_t num_blocks, int64_t block_size, int64_t n_kv_heads,
                           const int32_t* block_table, int64_t max_blocks, const int32_t* seq_lens,
                           float* O, int64_t rsO, int64_t csO, int64_t bsO,
                           int64_t M, int64_t N, int64_t D, int64_t Dv, int64_t n_seqs,
                           float alpha, int causal, int64_t q_len, void* stream,
                           const sbgemm_options* opt) {
    sbgemm_options o;
    const int ost = check_options(opt, &o);
    if (ost) return ost;
    if (o.force_path != SBGEMM_PATH_AUTO) return SBGEMM_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || D < 0 || Dv < 0 || n_seqs < 0) return SBGEMM_ERR_INVALID_VALUE;
    if (causal != 0 && causal != 1) return SBGEMM_ERR_INVALID_VALUE;
    if (M == 0 || n_seqs == 0 || Dv == 0) return SBGEMM_OK;
    if (N == 0) return SBGEMM_ERR_INVALID_VALUE;
    if (causal && (q_len <= 0 || q_len > N)) return SBGEMM_ERR_INVALID_VALUE;
    if (num_blocks <= 0 || block_size <= 0 || n_kv_heads <= 0 || max_blocks <= 0)
        return SBGEMM_ERR_INVALID_VALUE;
    if ((__int128)max_blocks * block_size < (__int128)N) return SBGEMM_ERR_INVALID_VALUE;
    if (!attention_supported(D, Dv)) return SBGEMM_ERR_UNSUPPORTED;
    const __int128 batch128 = (__int128)n_seqs * n_kv_heads;
    if (M > attention_max_rows() || batch128 >= ((__int128)1 << 31)) return SBGEMM_ERR_UNSUPPORTED;
    const int64_t batch = (int64_t)batch128;
    if (!Q || !K_cache || !V_cache || !block_table || !O) return SBGEMM_ERR_NULL_POINTER;
    if (!aligned(Q, 4) || !aligned(O, 4) || !aligned(block_table, 4) || (seq_lens && !aligned(seq_lens, 4)))
        return SBGEMM_ERR_INVALID_VALUE;
    if (!aligned(K_cache, 16) || !aligned(V_cache, 16)) return SBGEMM_ERR_INVALID_VALUE;
    // Element counts of the caches and the int32 tables (4 bytes each, so the
    // float spans' byte arithmetic holds for them too).
    const __int128 rows = (__int128)num_blocks * block_size * n_kv_heads;
    const __int128 k_elems = rows * D, v_elems = rows * Dv, t_elems = (__int128)n_seqs * max_blocks;
    const __int128 lim = (__int128)1 << 60;
    if (k_elems >= lim || v_elems >= lim || t_elems >= lim) return SBGEMM_ERR_INVALID_VALUE;
    Span sq{}, so{};
    if (!operand_span(batch, M, D, bsQ, rsQ, csQ, &sq) || !operand_span(batch, M, Dv, bsO, rsO, csO, &so))
        return SBGEMM_ERR_INVALID_VALUE;
    const Span sk{0, (int64_t)k_elems - 1}, sv{0, (int64_t)v_elems - 1};
    const Span st{0, (int64_t)t_elems - 1}, sl{0, n_seqs - 1};
    if (!output_injective(batch, M, Dv, bsO, rsO, csO)) return SBGEMM_ERR_OUTPUT_OVERLAP;
    if (bytes_meet(O, so, Q, sq) || bytes_meet(O, so, K_cache, sk) || bytes_meet(O, so, V_cache, sv) ||
        bytes_meet(O, so, block_table, st) || (seq_lens && bytes_meet(O, so, seq_lens, sl)))
        return SBGEMM_ERR_OUTPUT_OVERLAP;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return SBGEMM_ERR_CUDA; }
    Ranges seen;
    if (!span_in_allocation(Q, sq, &seen) || !span_in_allocation(K_cache, sk, &seen) ||
        !span_in_allocation(V_cache, sv, &seen) || !span_in_allocation(block_table, st, &seen) ||
        (seq_lens && !span_in_allocation(seq_lens, sl, &seen)) || !span_in_allocation(O, so, &seen))
        return SBGEMM_ERR_NOT_DEVICE_MEMORY;
    const int wst = check_attention_workspace(
        o, {{Q, sq}, {K_cache, sk}, {V_cache, sv}, {block_table, st}, {O, so},
            {seq_lens ? static_cast<const void*>(seq_lens) : static_cast<const void*>(O), seq_lens ? sl : so}});
    if (wst) return wst;
    AttnProblem a{Q, rsQ, csQ, bsQ, K_cache, n_kv_heads * D, 1, 0, V_cache, n_kv_heads * Dv, 1, 0,
                  O, rsO, csO, bsO, M, N, D, Dv, batch, alpha, causal, causal ? q_len : M,
                  ElemSpan{sq.lo, sq.hi}, ElemSpan{sk.lo, sk.hi}, ElemSpan{sv.lo, sv.hi},
                  ElemSpan{so.lo, so.hi}};
    a.paged = 1;
    a.table = block_table;
    a.seq_lens = seq_lens;
    a.max_blocks = max_blocks;
    a.block_size = block_size;
    a.n_kv_heads = n_kv_heads;
    a.num_blocks = num_blocks;
    a.workspace = o.workspace;
    a.workspace_bytes = o.workspace ? o.workspace_bytes : 0;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = attention_decode_supported(a) ? launch_attention_decode(a, s)
                                                         : launch_attention(a, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SBGEMM_ERR_CUDA;
    }
    return SBGEMM_OK;
}

int sbgemm_attention(const float* Q, int64_t rsQ, int64_t csQ, int64_t bsQ,
                     const float* K, int64_t rsK, int64_t csK, int64_t bsK,
                     const float* V, int64_t rsV, int64_t csV, int64_t bsV,
                     float* O, int64_t rsO, int64_t csO, int64_t bsO,
                     int64_t M, int64_t N, int64_t D, int64_t Dv, int64_t batch,
                     float alpha, int causal, int64_t q_len, void* stream) {
    return sbgemm_attention_ex(Q, rsQ, csQ, bsQ, K, rsK, csK, bsK, V, rsV, csV, bsV,
                               O, rsO, csO, bsO, M, N, D, Dv, batch, alpha, causal, q_len,
                               stream, nullptr);
}

int sbgemm(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
           const float* B, int64_t rsB, int64_t csB, int64_t bsB,
           float* C, int64_t rsC, int64_t csC, int64_t bsC,
           int64_t M, int64_t N, int64_t K, int64_t batch,
           float alpha, int accumulate, void* stream) {
    return sbgemm_ex(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                     M, N, K, batch, alpha, accumulate, stream, nullptr);
}

int sbgemm_workspace_bytes(int device, size_t* bytes) {
    if (!bytes) return SBGEMM_ERR_NULL_POINTER;
    const DeviceProps* d = device_props(device);
    if (!d) { cudaGetLastError(); return SBGEMM_ERR_CUDA; }
    *bytes = tma_ffma_workspace_bytes(d->sm_count);
    return SBGEMM_OK;
}

int sbgemm_device_status(void* stream, int* where_out) {
    if (where_out) *where_out = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return SBGEMM_ERR_CUDA;
    }
    unsigned int code = read_and_clear_wait_status_tma_ffma(s);
    const unsigned int code_tc = read_and_clear_wait_status_tf32(s);
    const unsigned int code_st = read_and_clear_wait_status_selftest(s);
    const unsigned int code_at = read_and_clear_wait_status_attention_tc(s);
    const unsigned int code_g = read_and_clear_status_gather(s);
    const unsigned int code_a = read_and_clear_status_attention(s);
    const unsigned int code_d = read_and_clear_status_attention_decode(s);
    if (code == 0) code = code_tc;
    if (code == 0) code = code_st;
    if (code == 0) code = code_at;
    if (code == 0) code = code_g;
    if (code == 0) code = code_a;
    if (code == 0) code = code_d;
    if (code != 0) {
        if (where_out) *where_out = (int)code;
        return (code == kBoundsViolation || code == kPagedInput) ? SBGEMM_ERR_DEVICE_CHECK
                                                                  : SBGEMM_ERR_DEVICE_TIMEOUT;
    }
    return SBGEMM_OK;
}

}  // extern "C"
