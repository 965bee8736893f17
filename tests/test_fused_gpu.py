"""Fused epilogue C <- act(alpha*A*B (+C) + D) through sbgemm_fused, on every
kernel path, against the oracle's fused product.

Tolerance: the product's own bound carried through the activation, whose
slope is at most 1.2 in magnitude for all six functions, plus the fp32
evaluation of the activation itself (16 units of 2^-24 on |f| + |z|)."""

import numpy as np
import pytest

import oracle
import strided_gemm_gb300 as sg
import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
SLOPE = 1.2
ACTS = list(sg.ACTIVATIONS)


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    return t


def make_D(rng, case, kind, values):
    """An addend of the given broadcast kind, or None."""
    M, N, batch = case.M, case.N, case.batch
    draw = ((lambda n: rng.integers(-8, 9, size=n).astype(np.float32)) if values == "int"
            else (lambda n: rng.standard_normal(n).astype(np.float32)))
    if kind == "none":
        return None
    if kind == "col_bias":            # one bias per output column
        return wl.Operand(draw(N), 0, 0, 1, 0)
    if kind == "batch_bias":          # a bias per batch entry and column
        return wl.Operand(draw(batch * N), 0, 0, 1, N)
    if kind == "matrix_colmajor":     # a full addend, column-major per batch entry
        return wl.Operand(draw(batch * M * N + 3), 3, 1, M, M * N)
    raise ValueError(kind)


def run_fused(case, D, act, torch, math=sg.MATH_FP32, force_path=sg.PATH_AUTO,
              workspace=None, k_split=sg.KSPLIT_ANY):
    dA, dB = gu.to_device(case.A, torch), gu.to_device(case.B, torch)
    dC = torch.from_numpy(case.C.storage.copy()).to("cuda")
    d_ptr = rs = cs = bs = 0
    if D is not None:
        dD = torch.from_numpy(D.storage).to("cuda")
        d_ptr, rs, cs, bs = dD.data_ptr() + 4 * D.offset, D.rs, D.cs, D.bs
    kw = {}
    if workspace is not None:
        kw = dict(workspace=workspace.data_ptr(), workspace_bytes=workspace.numel())
    sg.sbgemm_fused(dA.data_ptr() + 4 * case.A.offset, case.A.rs, case.A.cs, case.A.bs,
                    dB.data_ptr() + 4 * case.B.offset, case.B.rs, case.B.cs, case.B.bs,
                    dC.data_ptr() + 4 * case.C.offset, case.C.rs, case.C.cs, case.C.bs,
                    case.M, case.N, case.K, case.batch, case.alpha, case.accumulate,
                    d_ptr, rs, cs, bs, sg.ACTIVATIONS[act] if isinstance(act, str) else act,
                    torch.cuda.current_stream().cuda_stream, math, force_path, k_split=k_split,
                    **kw)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


def check_fused(case, D, act, got_storage, tol=gu.TOL_FFMA, exact=False, idx=None):
    code = oracle.ACTIVATIONS[act]
    args = (case.A, case.B, case.C, case.M, case.N, case.K, case.batch, case.alpha,
            case.accumulate, D, code)
    if idx is None:
        out, z, bound = oracle.fused_product(*args)
        got = gu.logical_c(case, got_storage).astype(np.float64)
    else:
        out, z, bound = oracle.fused_points(*args, idx)
        got = gu.c_storage_at(case, got_storage, idx)
    if exact:
        want = out.astype(np.float32).astype(np.float64)
        bad = np.flatnonzero(got.reshape(-1) != want.reshape(-1))
        assert bad.size == 0, f"{act}: {bad.size} inexact elements"
        return
    lim = SLOPE * tol * bound + 16 * U * (np.abs(out) + np.abs(z))
    err = np.abs(got - out)
    bad = np.flatnonzero(~(err <= lim).reshape(-1))
    assert bad.size == 0, (f"{act}: {bad.size} elements outside the bound; first flat {bad[0]}: "
                           f"got {got.reshape(-1)[bad[0]]} want {out.reshape(-1)[bad[0]]} "
                           f"z {z.reshape(-1)[bad[0]]} lim {lim.reshape(-1)[bad[0]]}")


# (path, math, A layout, B layout): the gather path gets layouts TMA cannot fetch.
PATHS = [
    ("gather", sg.MATH_FP32, sg.PATH_GATHER_FFMA, "gap", "neg_row"),
    ("tma", sg.MATH_FP32, sg.PATH_TMA_FFMA, "col16", "row16"),
    ("tf32", sg.MATH_TF32, sg.PATH_TMA_TF32, "row16", "col16"),
]


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
def test_fused_every_path_activation_and_addend(torch, path, act):
    name, math, force, la, lb = path
    tol = gu.TOL_TF32 if math == sg.MATH_TF32 else gu.TOL_FFMA
    rng = np.random.default_rng(len(act) * 31 + len(name))
    for i, (kind, acc, c_layout) in enumerate([("none", 0, "row"), ("col_bias", 1, "row"),
                                                ("batch_bias", 0, "col"),
                                                ("matrix_colmajor", 1, "row")]):
        case = wl.random_strided(rng, 130, 260, 96, 2, la, lb, c_layout=c_layout,
                                 values="real", accumulate=acc, alpha=[1.0, 0.5, -0.25, 2.0][i])
        D = make_D(rng, case, kind, "real")
        got = run_fused(case, D, act, torch, math, force)
        check_fused(case, D, act, got, tol=tol)


@pytest.mark.parametrize("act", ACTS)
def test_fused_tf32_column_major_c_through_tma(torch, act):
    """TF32 with a column-major C whose pitch (256 rows) suits a tensor map.
    Both operands K-major: the epilogue stages each 32 x 32 piece column by
    column and writes it with a TMA store through an M-inner map (C_old comes
    in the same way).  A K-major with B N-major: the plan is the transposed
    product, whose C^T is row-major."""
    rng = np.random.default_rng(40 + len(act))
    for la, lb, kind in (("row16", "col16", "col_bias"), ("row16", "row16", "matrix_colmajor")):
        case = wl.random_strided(rng, 256, 200, 96, 2, la, lb, c_layout="col", values="real",
                                 accumulate=1, alpha=0.75)
        D = make_D(rng, case, kind, "real")
        got = run_fused(case, D, act, torch, sg.MATH_TF32, sg.PATH_TMA_TF32)
        check_fused(case, D, act, got, tol=gu.TOL_TF32)


@pytest.mark.parametrize("act", ["none", "relu"])
@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
def test_fused_integer_inputs_exact(torch, path, act):
    """Integer A, B, C0 and D: every partial sum is exact, and so are the
    addend and ReLU."""
    name, math, force, la, lb = path
    rng = np.random.default_rng(7 + len(name))
    for kind in ("col_bias", "matrix_colmajor"):
        case = wl.random_strided(rng, 257, 300, 129, 3, la, lb, values="int", accumulate=1)
        D = make_D(rng, case, kind, "int")
        got = run_fused(case, D, act, torch, math, force)
        check_fused(case, D, act, got, exact=True)


@pytest.fixture(scope="module")
def workspace(torch):
    return torch.empty(sg.sbgemm_workspace_bytes(torch.cuda.current_device()),
                       dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("shape", [
    ("chained", 2048, 2560, 1024, "row16", "col16", sg.STREAM_K_CHAINED),
    ("pieces", 2560, 960, 8192, "col16", "row16", sg.STREAM_K_PIECES),
    ("gather_pieces", 256, 512, 784, "gap", "neg_row", sg.STREAM_K_PIECES),
    ("warp_per_output", 40, 30, 700, "gap", "neg_row", sg.STREAM_K_PIECES),
], ids=["chained", "pieces", "gather_pieces", "warp_per_output"])
def test_fused_after_split_k(torch, workspace, shape):
    """Split tiles apply the epilogue once, after the last piece."""
    _, M, N, K, la, lb, mode = shape
    rng = np.random.default_rng(M + K)
    case = wl.random_strided(rng, M, N, K, 1, la, lb, values="real", accumulate=1)
    plan = sg.sbgemm_plan(0x10000000, case.A.rs, case.A.cs, case.A.bs,
                          0x2000000000, case.B.rs, case.B.cs, case.B.bs,
                          0x4000000000, case.C.rs, case.C.cs, case.C.bs,
                          M, N, K, 1, 1, workspace=workspace.data_ptr(),
                          workspace_bytes=workspace.numel())
    assert plan["stream_k"] == mode
    D = make_D(rng, case, "col_bias", "real")
    got = run_fused(case, D, "gelu_tanh", torch, workspace=workspace)
    check_fused(case, D, "gelu_tanh", got, idx=gu.sample_points(case, 3000))
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where


def test_fused_k_zero(torch):
    """K = 0: C <- act(C_old + D) with accumulate, act(D) without."""
    rng = np.random.default_rng(3)
    for acc in (1, 0):
        case = wl.random_strided(rng, 40, 50, 0, 2, "row", "row", values="real", accumulate=acc)
        D = make_D(rng, case, "batch_bias", "real")
        got = run_fused(case, D, "silu", torch)
        check_fused(case, D, "silu", got)


def test_full_size_projection_with_bias_and_gelu(torch):
    """The feed-forward case: c5a (x W^T) with a bias per output feature and
    GELU, at full size, on sampled outputs; FP32 and TF32."""
    case = wl.make("c5a", "real")
    rng = np.random.default_rng(9)
    D = make_D(rng, case, "col_bias", "real")
    idx = gu.sample_points(case, 3000)
    for math, tol in ((sg.MATH_FP32, gu.TOL_FFMA), (sg.MATH_TF32, gu.TOL_TF32)):
        got = run_fused(case, D, "gelu_erf", torch, math=math)
        check_fused(case, D, "gelu_erf", got, tol=tol, idx=idx)


def test_fused_errors(torch):
    A = torch.zeros(64 * 64, device="cuda")
    B = torch.zeros(64 * 64, device="cuda")
    C = torch.zeros(64 * 64 + 64, device="cuda")
    base = (A.data_ptr(), 64, 1, 0, B.data_ptr(), 64, 1, 0, C.data_ptr(), 64, 1, 0,
            64, 64, 64, 1, 1.0, 0)

    def status(**kw):
        try:
            sg.sbgemm_fused(*base, **kw)
            torch.cuda.synchronize()
            return sg.SBGEMM_OK
        except sg.SbgemmError as e:
            return e.status

    bias = torch.zeros(64, device="cuda")
    assert status(D=bias.data_ptr(), csD=1, activation=sg.ACT_RELU) == sg.SBGEMM_OK
    assert status(activation=6) == sg.SBGEMM_ERR_INVALID_VALUE
    assert status(activation=-1) == sg.SBGEMM_ERR_INVALID_VALUE
    assert status(D=bias.data_ptr() + 2, csD=1) == sg.SBGEMM_ERR_INVALID_VALUE
    # D inside C's span (the row past C's last element is outside it).
    assert status(D=C.data_ptr() + 4 * 10, csD=1) == sg.SBGEMM_ERR_OUTPUT_OVERLAP
    assert status(D=C.data_ptr() + 4 * 64 * 64, csD=1) == sg.SBGEMM_OK
    host = np.zeros(64, dtype=np.float32)
    assert status(D=host.ctypes.data, csD=1) == sg.SBGEMM_ERR_NOT_DEVICE_MEMORY


def test_matmul_helper_bias_and_activation(torch):
    """sg.matmul(bias=..., activation=...) on torch tensors: a linear layer
    y = gelu(x W^T + b), against float64 torch on the CPU."""
    gen = torch.Generator().manual_seed(4)
    x = torch.randn(1000, 384, generator=gen)
    W = torch.randn(520, 384, generator=gen) * 0.05
    b = torch.randn(520, generator=gen)
    y = torch.empty(1000, 520, device="cuda")
    sg.matmul(x.cuda(), W.cuda().t(), y, bias=b.cuda(), activation="gelu_erf")
    torch.cuda.synchronize()
    z = x.double() @ W.double().t() + b.double()
    want = torch.nn.functional.gelu(z)
    bound = x.double().abs() @ W.double().abs().t() + b.double().abs()
    lim = SLOPE * gu.TOL_FFMA * bound + 16 * U * (want.abs() + z.abs())
    assert bool(((y.cpu().double() - want).abs() <= lim).all())
