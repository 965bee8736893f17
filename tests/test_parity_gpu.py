"""GPU parity: the CUDA path against the CPU oracle, element by element.

Tolerances follow the strided-batched problem statement: every element within
1e-5 * (|alpha| sum_k |a||b| + |C0|) on the fp32 path and 2e-3 times that bound
on the tf32 path; integer-valued inputs must match bit for bit.
"""

import dataclasses

import numpy as np
import pytest

import oracle
import strided_gemm_gb300 as sg
import workloads as wl
from strided_gemm_gb300 import build as sgbuild
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

FFMA_PATHS = [sg.PATH_AUTO, sg.PATH_GATHER_FFMA, sg.PATH_TMA_FFMA]


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need a CUDA device"
    sgbuild.build()
    sg.load()
    return t


def _supported(case, math, path):
    """Whether a forced path can serve the case (device allocations are at
    least 256-byte aligned, so only the element offsets matter)."""
    try:
        sg.sbgemm_plan(0x10000000 + 4 * case.A.offset, case.A.rs, case.A.cs, case.A.bs,
                       0x20000000 + 4 * case.B.offset, case.B.rs, case.B.cs, case.B.bs,
                       0x1000000000 + 4 * case.C.offset, case.C.rs, case.C.cs, case.C.bs,
                       case.M, case.N, case.K, case.batch, case.accumulate,
                       math=math, force_path=path)
        return True
    except sg.SbgemmError as e:
        assert e.status == sg.SBGEMM_ERR_UNSUPPORTED
        return False


# Workloads a tensor map cannot describe: the spectrogram's frames are
# overlapping rows of the signal (row stride 128 < 512 samples per frame) and
# its basis pitch (514 floats) is not a multiple of 16 bytes.
NOT_TMA = {"f4spec"}


@pytest.mark.parametrize("name", wl.WORKLOADS)
@pytest.mark.parametrize("values", ["real", "int"])
@pytest.mark.parametrize("path", FFMA_PATHS)
def test_workloads_small(torch, name, values, path):
    case = wl.make(name, values, **wl.small_shape(name))
    if name in NOT_TMA and path == sg.PATH_TMA_FFMA:
        assert not _supported(case, sg.MATH_FP32, path)
        pytest.skip("not TMA-eligible by construction")
    assert _supported(case, sg.MATH_FP32, path), "every other workload is TMA-eligible"
    got = gu.run_case(case, torch, force_path=path)
    gu.check_full(case, got, exact=(values == "int"))


# (M, K, N).  N <= 64 with a K-major A takes the 512 x 64 tiles on the TMA
# path; 1100 x 300 x 50 spans three of them with a ragged last one.
AWKWARD = [(17, 9, 33), (5, 31, 129), (1, 1, 1), (4, 4, 4), (5, 9, 3), (8, 7, 16),
           (33, 65, 20), (64, 64, 1), (1, 1, 64), (130, 70, 257), (257, 129, 131),
           (1100, 300, 50)]
LAYOUT_PAIRS = [("row", "row"), ("row", "col"), ("col", "row"), ("col", "col"),
                ("neg_row", "gap"), ("gap", "bcast_row"), ("bcast_row", "neg_row"),
                ("row16", "row16"), ("row16", "col16"), ("col16", "row16"), ("col16", "col16")]


@pytest.mark.parametrize("mkn", AWKWARD, ids=[f"{m}x{k}x{n}" for m, k, n in AWKWARD])
@pytest.mark.parametrize("layouts", LAYOUT_PAIRS, ids=["-".join(l) for l in LAYOUT_PAIRS])
def test_awkward_shapes_all_layouts(torch, mkn, layouts):
    M, K, N = mkn
    rng = np.random.default_rng(M * 1000 + K * 10 + N)
    for i, (bsm, c_layout, acc, alpha) in enumerate([
            (("dense", "dense"), "row", 0, 1.0),
            (("zero", "neg"), "col", 1, -0.5),
            (("neg", "zero"), "row", 1, 0.125)]):
        batch = [1, 3, 2][i]
        for values in ("int", "real"):
            case = wl.random_strided(rng, M, N, K, batch, layouts[0], layouts[1],
                                     c_layout=c_layout, bs_mode=bsm, values=values,
                                     accumulate=acc, alpha=alpha)
            for path in FFMA_PATHS:
                if not _supported(case, sg.MATH_FP32, path):
                    continue
                got = gu.run_case(case, torch, force_path=path)
                gu.check_full(case, got, exact=(values == "int"))


TINY = [(17, 9, 33), (5, 31, 129), (1, 1, 1), (4, 4, 4), (5, 9, 3), (8, 7, 16), (64, 64, 1),
        (1, 1, 64), (64, 32, 48)]
TINY_LAYOUTS = [("row", "row"), ("col", "col"), ("neg_row", "gap"), ("bcast_row", "neg_row"),
                ("col16", "row16")]


@pytest.mark.parametrize("mkn", TINY, ids=[f"{m}x{k}x{n}" for m, k, n in TINY])
@pytest.mark.parametrize("layouts", TINY_LAYOUTS, ids=["-".join(l) for l in TINY_LAYOUTS])
def test_tiny_products_direct_and_tiled_agree(torch, mkn, layouts):
    """A product of at most 16384 outputs with K <= 128 runs one output per
    thread (8 x 32 blocks); the same shapes over a batch large enough to pass
    that bound take the tiled kernel.  Both match the oracle on every
    element, and batch entry 0 of the tiled run equals the one-entry direct
    run to the bit (one k-ordered fmaf chain per output in both)."""
    M, K, N = mkn
    rng = np.random.default_rng(M * 7 + K * 3 + N)
    batch = 16384 // (M * N) + 1
    for acc, alpha in ((0, 1.0), (1, -0.75)):
        big = wl.random_strided(rng, M, N, K, batch, layouts[0], layouts[1], c_layout="row",
                                values="real", accumulate=acc, alpha=alpha)
        one = dataclasses.replace(big, batch=1)
        kw = dict(force_path=sg.PATH_GATHER_FFMA)
        p_big = sg.sbgemm_plan(0x10000000 + 4 * big.A.offset, big.A.rs, big.A.cs, big.A.bs,
                               0x20000000 + 4 * big.B.offset, big.B.rs, big.B.cs, big.B.bs,
                               0x1000000000, big.C.rs, big.C.cs, big.C.bs, M, N, K, batch, acc, **kw)
        p_one = sg.sbgemm_plan(0x10000000 + 4 * big.A.offset, big.A.rs, big.A.cs, big.A.bs,
                               0x20000000 + 4 * big.B.offset, big.B.rs, big.B.cs, big.B.bs,
                               0x1000000000, big.C.rs, big.C.cs, big.C.bs, M, N, K, 1, acc, **kw)
        assert (p_one["tile_m"], p_one["tile_n"]) == (8, 32), p_one
        assert (p_big["tile_m"], p_big["tile_n"]) != (8, 32), p_big
        got_big = gu.run_case(big, torch, **kw)
        gu.check_full(big, got_big)
        got_one = gu.run_case(one, torch, **kw)
        gu.check_full(one, got_one)
        c0_big = gu.logical_c(big, got_big)[0]
        c0_one = gu.logical_c(one, got_one)[0]
        assert np.array_equal(c0_big.view(np.uint32), c0_one.view(np.uint32))


@pytest.mark.parametrize("name", wl.WORKLOADS)
def test_workloads_full_size_sampled(torch, name):
    """Full-size inputs through the default entry point (the call the benchmark
    times), checked at sampled outputs including every corner."""
    case = wl.make(name, "real")
    got = gu.run_case(case, torch, entry="sbgemm")
    gu.check_points(case, got)
    case_i = wl.make(name, "int")
    got = gu.run_case(case_i, torch, entry="sbgemm")
    gu.check_points(case_i, got, exact=True)


def test_overwrite_never_reads_c(torch):
    case = wl.make("c2a", "real")
    nan_c = np.full_like(case.C.storage, np.nan)
    got = gu.run_case(case, torch, c_init=nan_c)
    assert not np.isnan(gu.logical_c(case, got)).any()
    gu.check_full(case, got)


def test_k_zero(torch):
    rng = np.random.default_rng(11)
    case = wl.random_strided(rng, 37, 21, 0, 2, "row", "row", values="real", accumulate=0,
                             alpha=3.0)
    case.C.storage[:] = 7.0
    got = gu.run_case(case, torch)
    assert np.all(gu.logical_c(case, got) == 0.0)
    case.accumulate = 1
    got = gu.run_case(case, torch)
    assert np.all(gu.logical_c(case, got) == 7.0)


def test_batch_beyond_grid_limit(torch):
    rng = np.random.default_rng(12)
    case = wl.random_strided(rng, 2, 3, 4, 70000, "row", "col", values="int",
                             accumulate=1, alpha=1.0)
    got = gu.run_case(case, torch)
    gu.check_full(case, got, exact=True)


def test_swapped_strides_bitwise_equal_to_transposed_copy(torch):
    rng = np.random.default_rng(13)
    M, K, N = 300, 516, 260     # pitches that are 16-byte multiples: every path applies
    a_km = rng.standard_normal((K, M)).astype(np.float32)
    b_nk = rng.standard_normal((N, K)).astype(np.float32)
    c = np.zeros(M * N, np.float32)
    swapped = wl.Case("swapped", wl.Operand(a_km.reshape(-1), 0, 1, M, 0),
                      wl.Operand(b_nk.reshape(-1), 0, 1, K, 0),
                      wl.Operand(c.copy(), 0, N, 1, 0), M, N, K, 1, 1.0, 0, "real")
    copied = wl.Case("copied", wl.Operand(np.ascontiguousarray(a_km.T).reshape(-1), 0, K, 1, 0),
                     wl.Operand(np.ascontiguousarray(b_nk.T).reshape(-1), 0, N, 1, 0),
                     wl.Operand(c.copy(), 0, N, 1, 0), M, N, K, 1, 1.0, 0, "real")
    for path in FFMA_PATHS:
        assert _supported(swapped, sg.MATH_FP32, path) and _supported(copied, sg.MATH_FP32, path)
        g1 = gu.run_case(swapped, torch, force_path=path)
        g2 = gu.run_case(copied, torch, force_path=path)
        assert np.array_equal(g1, g2)
    gu.check_full(swapped, g1)


def test_alpha_power_of_two_and_batch_permutation_bitwise(torch):
    case = wl.make("c3", "real", batch=4, M=200, N=130, K=64)
    base = gu.logical_c(case, gu.run_case(case, torch))
    case.alpha = 0.5
    half = gu.logical_c(case, gu.run_case(case, torch))
    assert np.array_equal(half, base * 4)     # alpha 1/8 -> 1/2 is a factor 4
    perm = [3, 1, 0, 2]
    a = case.A.storage.reshape(4, -1)[perm].reshape(-1).copy()
    b = case.B.storage.reshape(4, -1)[perm].reshape(-1).copy()
    case.A.storage, case.B.storage = a, b
    case.alpha = 0.125
    permuted = gu.logical_c(case, gu.run_case(case, torch))
    assert np.array_equal(permuted, base[perm])


def test_identity_reproduces_operand_bitwise(torch):
    rng = np.random.default_rng(14)
    M = K = 150
    N = 333
    eye = np.eye(M, dtype=np.float32).reshape(-1)
    b = rng.standard_normal(K * N).astype(np.float32)
    case = wl.Case("eye", wl.Operand(eye, 0, K, 1, 0), wl.Operand(b, 0, N, 1, 0),
                   wl.Operand(np.zeros(M * N, np.float32), 0, N, 1, 0), M, N, K, 1, 1.0, 0, "real")
    got = gu.logical_c(case, gu.run_case(case, torch))
    assert np.array_equal(got[0], b.reshape(K, N))


def test_errors_surface_as_status(torch):
    x = torch.zeros(64, device="cuda")
    # C overlapping A.
    with pytest.raises(sg.SbgemmError) as e:
        sg.sbgemm(x.data_ptr(), 4, 1, 0, x.data_ptr(), 4, 1, 0, x.data_ptr() + 4 * 8, 4, 1, 0,
                  4, 4, 4, 1, 1.0, 0)
    assert e.value.status == sg.SBGEMM_ERR_OUTPUT_OVERLAP
    # Span leaving the allocation: a 16-float tensor sits in a small-block
    # segment of a few MB; rows 64 M floats apart leave any such segment.
    # The rows walk away from C so that the spans do not meet (which would be
    # reported as an overlap first).
    y = torch.zeros(16, device="cuda")
    z = torch.zeros(16, device="cuda")
    rs = -(1 << 26) if z.data_ptr() > y.data_ptr() else (1 << 26)
    with pytest.raises(sg.SbgemmError) as e:
        sg.sbgemm(y.data_ptr(), rs, 1, 0, y.data_ptr(), 4, 1, 0, z.data_ptr(), 4, 1, 0,
                  4, 4, 4, 1, 1.0, 0)
    assert e.value.status == sg.SBGEMM_ERR_NOT_DEVICE_MEMORY
    # Host memory is not accepted.
    h = np.zeros(16, np.float32)
    with pytest.raises(sg.SbgemmError) as e:
        sg.sbgemm(h.ctypes.data, 4, 1, 0, y.data_ptr(), 4, 1, 0, z.data_ptr(), 4, 1, 0,
                  4, 4, 4, 1, 1.0, 0)
    assert e.value.status == sg.SBGEMM_ERR_NOT_DEVICE_MEMORY
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK and where == 0


def test_torch_tensor_helper(torch):
    g = torch.Generator(device="cpu").manual_seed(5)
    A = torch.randn(3, 70, 90, generator=g).cuda()
    W = torch.randn(50, 90, generator=g).cuda()
    C = torch.empty(3, 70, 50, device="cuda")
    sg.matmul(A, W.t().unsqueeze(0).expand(3, 90, 50), C)
    torch.cuda.synchronize()
    # The oracle on the same memory: W [50, 90] read as B[k][n] = W[n][k],
    # shared by the three batch entries.
    a = wl.Operand(A.cpu().numpy().ravel(), 0, 90, 1, 70 * 90)
    w = wl.Operand(W.cpu().numpy().ravel(), 0, 1, 90, 0)
    c0 = wl.Operand(np.zeros(3 * 70 * 50, np.float32), 0, 50, 1, 70 * 50)
    ref, bound = oracle.product(a, w, c0, 70, 50, 90, 3, 1.0, 0)
    got = C.cpu().numpy().astype(np.float64)
    assert bool((np.abs(got - ref) <= gu.TOL_FFMA * bound).all())


STREAM_K_SHAPES = [
    # (name, M, N, K, batch, a_layout, b_layout, accumulate)
    ("160_tiles_all_split", 2048, 2560, 1024, 1, "row16", "col16", 0),
    ("ragged_k", 2048, 2600, 1000, 1, "row16", "row16", 1),
    ("batched", 1024, 1024, 768, 5, "col16", "row16", 1),
    ("mn_major_both", 4100, 1200, 640, 1, "col16", "row16", 0),
    # the last 128-wide tile column half full: its units weighted lighter, its
    # tiles ordered last
    ("ragged_last_column", 8192, 960, 2560, 1, "row16", "col16", 0),
    ("ragged_last_column_batched", 2048, 936, 1536, 3, "row16", "col16", 1),
]


@pytest.fixture(scope="module")
def workspace(torch):
    nbytes = sg.sbgemm_workspace_bytes(torch.cuda.current_device())
    return torch.empty(nbytes, dtype=torch.uint8, device="cuda")


def _run_ws(case, torch, ws, entry_kw=None):
    kw = dict(workspace=ws.data_ptr(), workspace_bytes=ws.numel()) if ws is not None else {}
    dA, dB = gu.to_device(case.A, torch), gu.to_device(case.B, torch)
    dC = torch.from_numpy(case.C.storage.copy()).to("cuda")
    args = (dA.data_ptr() + 4 * case.A.offset, case.A.rs, case.A.cs, case.A.bs,
            dB.data_ptr() + 4 * case.B.offset, case.B.rs, case.B.cs, case.B.bs,
            dC.data_ptr() + 4 * case.C.offset, case.C.rs, case.C.cs, case.C.bs,
            case.M, case.N, case.K, case.batch, case.alpha, case.accumulate,
            torch.cuda.current_stream().cuda_stream)
    kw.update(entry_kw or {})
    plan = sg.sbgemm_plan(*args[:16], case.accumulate, **kw)
    sg.sbgemm_ex(*args, **kw)
    torch.cuda.synchronize()
    return dC.cpu().numpy(), plan


@pytest.mark.parametrize("shape", STREAM_K_SHAPES, ids=[s[0] for s in STREAM_K_SHAPES])
def test_stream_k_bitwise_equals_data_parallel(torch, workspace, shape):
    """Split tiles continue one k-ordered FMA chain through the workspace, so
    the stream-K schedule reproduces the data-parallel result bit for bit."""
    _, M, N, K, batch, la, lb, acc = shape
    rng = np.random.default_rng(M + N + K)
    case = wl.random_strided(rng, M, N, K, batch, la, lb, values="real", accumulate=acc,
                             alpha=0.75)
    dp, plan_dp = _run_ws(case, torch, None)
    sk, plan_sk = _run_ws(case, torch, workspace)
    assert not plan_dp["stream_k"] and plan_sk["stream_k"], (plan_dp, plan_sk)
    assert np.array_equal(dp, sk)
    gu.check_points(case, sk, n=4000)
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where


def test_stream_k_repeated_calls_reuse_workspace(torch, workspace):
    """The flags are cleared on the stream before every launch, so back-to-back
    calls through one workspace stay exact (integer inputs)."""
    rng = np.random.default_rng(3)
    case = wl.random_strided(rng, 2048, 2560, 1024, 1, "row16", "row16", values="int")
    first, plan = _run_ws(case, torch, workspace)
    assert plan["stream_k"]
    for _ in range(3):
        again, _ = _run_ws(case, torch, workspace)
        assert np.array_equal(again, first)
    gu.check_full(case, first, exact=True)


# ---- independent K pieces (fewer tiles than SMs, long K) --------------------------

SPLIT_SHAPES = [
    # (name, M, N, K, batch, a_layout, b_layout, accumulate); 38..151 TMA tiles
    ("weight_grad_like", 2560, 960, 8192, 1, "col16", "row16", 1),   # 80 tiles, 2-3 pieces each
    ("ragged", 2000, 1000, 3000, 1, "row16", "col16", 0),            # ragged M, N and K
    ("batched", 512, 512, 2048, 12, "col16", "row16", 1),
    ("many_pieces", 1536, 1024, 4096, 1, "row16", "row16", 0),       # 48 tiles, ~4 pieces each
]


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=[s[0] for s in SPLIT_SHAPES])
def test_split_k_pieces_parity_and_determinism(torch, workspace, shape):
    """Every piece starts from zero and the tail adds the earlier pieces in a
    fixed order: within the FFMA bound of the oracle, identical on every run,
    and k_split = EXACT restores the unsplit result bit for bit."""
    _, M, N, K, batch, la, lb, acc = shape
    rng = np.random.default_rng(M * 7 + N + K + batch)
    case = wl.random_strided(rng, M, N, K, batch, la, lb, values="real", accumulate=acc,
                             alpha=0.5)
    first, plan = _run_ws(case, torch, workspace)
    assert plan["path"] == sg.PATH_TMA_FFMA and plan["stream_k"] == sg.STREAM_K_PIECES, plan
    gu.check_points(case, first, n=4000)
    again, _ = _run_ws(case, torch, workspace)
    assert np.array_equal(first, again)
    whole, _ = _run_ws(case, torch, None)
    exact, plan_x = _run_ws(case, torch, workspace, dict(k_split=sg.KSPLIT_EXACT))
    assert plan_x["stream_k"] == sg.STREAM_K_NONE
    assert np.array_equal(exact, whole)
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where


@pytest.mark.parametrize("name", ["c2a", "c2b", "strided"])
def test_gather_k_pieces_parity_and_determinism(torch, workspace, name):
    """Small products on the gather path cut K into pieces (one CTA per tile
    and piece, summed in piece order by the tile's last CTA; c2b, 2560
    outputs, splits K across a warp's lanes instead): within the oracle's
    bound, exact on integers, identical on every run; k_split = EXACT keeps
    one chain per output, bit for bit the result without a workspace."""
    rng = np.random.default_rng(23 + len(name))
    for values in ("real", "int"):
        if name == "strided":
            # Gapped and negative strides (no tensor map), ragged, batched, +C.
            case = wl.random_strided(rng, 100, 70, 900, 3, "gap", "neg_row", values=values,
                                     accumulate=1, alpha=-0.5)
        else:
            case = wl.make(name, values)
        first, plan = _run_ws(case, torch, workspace)
        assert plan["path"] == sg.PATH_GATHER_FFMA and plan["stream_k"] == sg.STREAM_K_PIECES, plan
        gu.check_full(case, first, exact=(values == "int"))
        again, _ = _run_ws(case, torch, workspace)
        assert np.array_equal(first, again)
    whole, _ = _run_ws(case, torch, None)
    exact, plan_x = _run_ws(case, torch, workspace, dict(k_split=sg.KSPLIT_EXACT))
    assert plan_x["stream_k"] == sg.STREAM_K_NONE
    assert np.array_equal(exact, whole)
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where


WARPDOT = [(5, 300, 7, 3), (1, 1000, 1, 1), (17, 129, 33, 2), (64, 512, 10, 4), (3, 4097, 5, 1)]
WARPDOT_LAYOUTS = [("row", "col"), ("col", "row"), ("gap", "neg_row"), ("bcast_row", "gap")]


@pytest.mark.parametrize("mknb", WARPDOT, ids=[f"{m}x{k}x{n}x{b}" for m, k, n, b in WARPDOT])
@pytest.mark.parametrize("layouts", WARPDOT_LAYOUTS, ids=["-".join(l) for l in WARPDOT_LAYOUTS])
def test_tiny_long_k_one_warp_per_output(torch, workspace, mknb, layouts):
    """At most 16384 outputs with K > 128, a workspace and k_split = ANY: one
    warp per output, its lanes splitting K and a shuffle butterfly adding
    them (reported as K pieces, 1 x 8 outputs per CTA).  Within the oracle's
    bound, exact on integers, identical from run to run; k_split = EXACT keeps
    one chain per output, bit for bit the result without a workspace."""
    M, K, N, batch = mknb
    rng = np.random.default_rng(M * 13 + K + N * 7 + batch)
    for values, acc, alpha in (("real", 0, 1.0), ("int", 1, -0.5)):
        case = wl.random_strided(rng, M, N, K, batch, layouts[0], layouts[1], values=values,
                                 accumulate=acc, alpha=alpha)
        first, plan = _run_ws(case, torch, workspace)
        assert plan["path"] == sg.PATH_GATHER_FFMA and plan["stream_k"] == sg.STREAM_K_PIECES, plan
        assert (plan["tile_m"], plan["tile_n"]) == (1, 8), plan
        gu.check_full(case, first, exact=(values == "int"))
        again, _ = _run_ws(case, torch, workspace)
        assert np.array_equal(first, again)
        whole, plan_w = _run_ws(case, torch, None)
        exact, plan_x = _run_ws(case, torch, workspace, dict(k_split=sg.KSPLIT_EXACT))
        assert plan_x["stream_k"] == sg.STREAM_K_NONE and (plan_x["tile_m"], plan_x["tile_n"]) != (1, 8)
        assert np.array_equal(exact, whole)
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where


def test_split_k_pieces_integer_exact(torch, workspace):
    """Integer inputs: every partial sum is exact, so the split result is the
    exact product whatever the order of the pieces."""
    rng = np.random.default_rng(17)
    case = wl.random_strided(rng, 1536, 1024, 4096, 1, "col16", "row16", values="int",
                             accumulate=1)
    got, plan = _run_ws(case, torch, workspace)
    assert plan["stream_k"] == sg.STREAM_K_PIECES
    gu.check_points(case, got, n=6000, exact=True)


@pytest.mark.parametrize("name", wl.BACKWARD)
def test_backward_products_full_size_with_workspace(torch, workspace, name):
    """The backward products at full size through the schedule a caller with a
    workspace gets (chained stream-K for dX, independent pieces for dW)."""
    for values in ("real", "int"):
        case = wl.make(name, values)
        got, plan = _run_ws(case, torch, workspace)
        assert plan["path"] == sg.PATH_TMA_FFMA
        want_mode = sg.STREAM_K_PIECES if name.startswith("f1dw") else sg.STREAM_K_CHAINED
        assert plan["stream_k"] == want_mode, plan
        if values == "int":
            gu.check_points(case, got, n=3000, exact=True)
        else:
            gu.check_points(case, got, n=3000)
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where


@pytest.mark.parametrize("math", ["fp32", "tf32"])
def test_linear_backward_helper(torch, workspace, math):
    """sg.linear_backward on torch tensors: dX = G W and dW += G^T X against
    float64 torch on the CPU, on either arithmetic path."""
    m = sg.MATH_TF32 if math == "tf32" else sg.MATH_FP32
    tol = gu.TOL_TF32 if math == "tf32" else gu.TOL_FFMA
    gen = torch.Generator().manual_seed(5)
    T, d_in, d_out = 2048, 384, 640
    X = torch.randn(T, d_in, generator=gen)
    W = torch.randn(d_out, d_in, generator=gen) * 0.02
    G = torch.randn(T, d_out, generator=gen)
    dW0 = torch.randn(d_out, d_in, generator=gen) * 0.01
    dX = torch.empty(T, d_in, device="cuda")
    dW = dW0.clone().cuda()
    sg.linear_backward(G.cuda(), X.cuda(), W.cuda(), dX, dW, accumulate_dW=True,
                       workspace=workspace, math=m)
    torch.cuda.synchronize()
    # The oracle on the same memory: dX = G W (G [T, out], W [out, in]) and
    # dW = dW0 + G^T X (G read with swapped strides, X [T, in]).
    g = G.numpy().ravel()
    zero = wl.Operand(np.zeros(T * d_in, np.float32), 0, d_in, 1, 0)
    want_dX, bound_dX = oracle.product(wl.Operand(g, 0, d_out, 1, 0), wl.Operand(W.numpy().ravel(), 0, d_in, 1, 0),
                                       zero, T, d_in, d_out, 1, 1.0, 0)
    want_dW, bound_dW = oracle.product(wl.Operand(g, 0, 1, d_out, 0), wl.Operand(X.numpy().ravel(), 0, d_in, 1, 0),
                                       wl.Operand(dW0.numpy().ravel(), 0, d_in, 1, 0), d_out, d_in, T, 1, 1.0, 1)
    assert bool((np.abs(dX.cpu().double().numpy() - want_dX[0]) <= tol * bound_dX[0]).all())
    assert bool((np.abs(dW.cpu().double().numpy() - want_dW[0]) <= tol * bound_dW[0]).all())


# ---- TF32 tensor-core path (opt-in) -------------------------------------------

# Both operands K-major, one MN-major or both (transposed in shared memory):
# c4's V and c5c's B are N-major, c5d's A is M-major, and the weight
# gradients' G^T and X are M-major and N-major.
TF32_WORKLOADS = ["c2a", "c2b", "c3", "c3gqa", "c4", "c5a", "c5b", "c5c", "c5d",
                  "f1dxa", "f1dwa", "f1dxb", "f1dwb", "f4dist"]


@pytest.mark.parametrize("name", TF32_WORKLOADS)
@pytest.mark.parametrize("values", ["real", "int"])
def test_tf32_workloads_small(torch, name, values):
    case = wl.make(name, values, **wl.small_shape(name))
    assert _supported(case, sg.MATH_TF32, sg.PATH_TMA_TF32)
    got = gu.run_case(case, torch, math=sg.MATH_TF32, force_path=sg.PATH_TMA_TF32)
    gu.check_full(case, got, tol=gu.TOL_TF32, exact=(values == "int"))


TF32_SHAPES = [(17, 9, 33), (5, 31, 129), (1, 1, 1), (130, 70, 257), (257, 129, 300),
               (128, 32, 256), (300, 1000, 520)]


# (A, B): both K-major; A M-major with B K-major; A K-major with B N-major;
# both MN-major.
TF32_LAYOUTS = [("row16", "col16"), ("col16", "col16"), ("row16", "row16"), ("col16", "row16")]


@pytest.mark.parametrize("mkn", TF32_SHAPES, ids=[f"{m}x{k}x{n}" for m, k, n in TF32_SHAPES])
@pytest.mark.parametrize("layouts", TF32_LAYOUTS, ids=["-".join(l) for l in TF32_LAYOUTS])
def test_tf32_awkward_shapes(torch, mkn, layouts):
    """Every unit-stride orientation of A and B; zero batch strides,
    column-major C, ragged edges."""
    M, K, N = mkn
    rng = np.random.default_rng(M * 31 + K * 7 + N)
    for i, (bsm, c_layout, acc, alpha) in enumerate([
            (("dense", "dense"), "row", 0, 1.0),
            (("zero", "dense"), "col", 1, -0.5),
            (("dense", "zero"), "row", 1, 0.125)]):
        batch = [1, 3, 2][i]
        for values in ("int", "real"):
            case = wl.random_strided(rng, M, N, K, batch, layouts[0], layouts[1], c_layout=c_layout,
                                     bs_mode=bsm, values=values, accumulate=acc, alpha=alpha)
            assert _supported(case, sg.MATH_TF32, sg.PATH_TMA_TF32)
            got = gu.run_case(case, torch, math=sg.MATH_TF32, force_path=sg.PATH_TMA_TF32)
            gu.check_full(case, got, tol=gu.TOL_TF32, exact=(values == "int"))


def test_tf32_opt_in_falls_back_to_fp32(torch):
    """math=TF32 without a forced path serves operands the tensor-core path
    does not take (strides TMA cannot fetch) with strict fp32."""
    rng = np.random.default_rng(21)
    general = wl.random_strided(rng, 70, 90, 50, 2, "gap", "neg_row", values="real",
                                accumulate=1, alpha=0.5)
    for c, want_path in ((general, (sg.PATH_GATHER_FFMA,)),):
        plan = sg.sbgemm_plan(0x10000000 + 4 * c.A.offset, c.A.rs, c.A.cs, c.A.bs,
                              0x20000000 + 4 * c.B.offset, c.B.rs, c.B.cs, c.B.bs,
                              0x1000000000, c.C.rs, c.C.cs, c.C.bs,
                              c.M, c.N, c.K, c.batch, c.accumulate, math=sg.MATH_TF32)
        assert plan["path"] in want_path
        assert not _supported(c, sg.MATH_TF32, sg.PATH_TMA_TF32)
        got = gu.run_case(c, torch, math=sg.MATH_TF32)
        gu.check_full(c, got)


TF32_STREAM_K_SHAPES = [
    # (name, M, N, K, batch, accumulate[, A layout, B layout]); by default A
    # row-major and B column-major (both K-major)
    ("160_tiles_long_k", 2048, 2560, 4096, 1, 0),
    ("ragged_k", 2560, 2560, 4000, 1, 1),
    ("batched", 1024, 1024, 4096, 5, 1),
    ("320_tiles", 2048, 5120, 4096, 1, 0),
    ("few_tiles_pieces", 1024, 1024, 8192, 1, 1),      # 32 tiles: several pieces per tile
    ("weight_grad_both_mn", 2560, 960, 8192, 1, 1, "col16", "row16"),   # dW = G^T X
]


@pytest.mark.parametrize("shape", TF32_STREAM_K_SHAPES, ids=[s[0] for s in TF32_STREAM_K_SHAPES])
def test_tf32_split_pieces_parity_and_determinism(torch, workspace, shape):
    """On the tensor cores a split tile's pieces accumulate independently and
    the tail adds the earlier ones in a fixed order: within the TF32 bound,
    identical from run to run; k_split = EXACT keeps the unsplit result."""
    _, M, N, K, batch, acc = shape[:6]
    la, lb = shape[6:] if len(shape) > 6 else ("row16", "col16")
    rng = np.random.default_rng(M * 3 + N + K)
    case = wl.random_strided(rng, M, N, K, batch, la, lb, values="real",
                             accumulate=acc, alpha=0.75)
    kw = dict(math=sg.MATH_TF32, force_path=sg.PATH_TMA_TF32)
    first, plan = _run_ws(case, torch, workspace, kw)
    assert plan["path"] == sg.PATH_TMA_TF32 and plan["stream_k"] == sg.STREAM_K_PIECES, plan
    gu.check_points(case, first, n=4000, tol=gu.TOL_TF32)
    again, _ = _run_ws(case, torch, workspace, kw)
    assert np.array_equal(first, again)
    whole, _ = _run_ws(case, torch, None, kw)
    exact, plan_x = _run_ws(case, torch, workspace, dict(kw, k_split=sg.KSPLIT_EXACT))
    assert plan_x["stream_k"] == sg.STREAM_K_NONE and np.array_equal(exact, whole)
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where


TF32_PAIR_SPLIT_SHAPES = [
    # (name, M, N, K, A layout, tile): B column-major (K-major), ragged M, N
    # and K edges, every tile split into K pieces: two K-major operands on
    # 100 tiles of 256 x 256 (CTA pairs), an M-major A on one CTA's tiles
    ("k_major_pairs", 2500, 2470, 4100, "row16", (256, 256)),
    ("a_m_major", 2500, 2470, 4100, "col16", (128, 256)),
]


@pytest.mark.parametrize("shape", TF32_PAIR_SPLIT_SHAPES, ids=[s[0] for s in TF32_PAIR_SPLIT_SHAPES])
def test_tf32_pair_split_parity(torch, workspace, shape):
    """Tiles whose K slices are split into pieces (on CTA pairs each pair is
    one worker, and each CTA of a pair parks and collects its own rows):
    within the TF32 bound at sampled points and along the ragged last rows
    and columns, identical from run to run; integers exact."""
    _, M, N, K, la, tile = shape
    rng = np.random.default_rng(M + 7 * N + K)
    kw = dict(math=sg.MATH_TF32, force_path=sg.PATH_TMA_TF32)
    for values in ("real", "int"):
        case = wl.random_strided(rng, M, N, K, 1, la, "col16", values=values, accumulate=1, alpha=0.75)
        first, plan = _run_ws(case, torch, workspace, kw)
        assert plan["stream_k"] == sg.STREAM_K_PIECES and (plan["tile_m"], plan["tile_n"]) == tile, plan
        gu.check_points(case, first, n=4000, tol=gu.TOL_TF32, exact=(values == "int"))
        edge = [(0, m, n) for m in range(M - 200, M) for n in range(N - 3, N)] + \
               [(0, m, n) for m in range(0, M, 97) for n in range(N - 200, N, 7)]
        gu.check_points(case, first, points=edge, tol=gu.TOL_TF32, exact=(values == "int"))
        again, _ = _run_ws(case, torch, workspace, kw)
        assert np.array_equal(first, again)
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where


def test_tf32_stream_k_integer_exact(torch, workspace):
    """Small integers are exact in TF32, so the split schedule must give the
    exact product; repeated calls reuse the workspace flags."""
    rng = np.random.default_rng(5)
    case = wl.random_strided(rng, 2048, 2560, 4096, 1, "row16", "col16", values="int")
    kw = dict(math=sg.MATH_TF32, force_path=sg.PATH_TMA_TF32)
    first, plan = _run_ws(case, torch, workspace, kw)
    assert plan["stream_k"]
    for _ in range(2):
        again, _ = _run_ws(case, torch, workspace, kw)
        assert np.array_equal(again, first)
    gu.check_points(case, first, n=4000, exact=True)


@pytest.mark.parametrize("name", ["c3", "c3gqa", "c4", "c5a", "c5b", "c5c", "c5d", "f1dwa", "f1dwb"])
def test_tf32_full_size_sampled(torch, name):
    case = wl.make(name, "real")
    assert _supported(case, sg.MATH_TF32, sg.PATH_TMA_TF32)
    got = gu.run_case(case, torch, math=sg.MATH_TF32)
    gu.check_points(case, got, tol=gu.TOL_TF32)
    case_i = wl.make(name, "int")
    got = gu.run_case(case_i, torch, math=sg.MATH_TF32)
    gu.check_points(case_i, got, exact=True)
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where
