"""Fused attention O = softmax(alpha * Q K^T [causal]) V through the C ABI
against the fp64 oracle.

Tolerance, from the products' convention: the scores carry 1e-5 of their
magnitude (smag, the largest |alpha| sum_d |q k| of the row) plus a few
units of 2^-24 for the scale and exp2, which perturbs each probability by
at most delta = 1e-5 * smag + 8u relative; P V carries 1e-5 of sum_n P |V|
(the oracle's weight W).  So |O - O_ref| <= (1e-5 + 2 delta) W + 4u |O_ref|.
The TF32 tensor-core kernel rounds Q, K, P and V to tf32: the same bound with
2e-3 in place of 1e-5 (the products' TF32 reading)."""

import numpy as np
import pytest

import oracle
import strided_gemm_gb300 as sg
import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    return t


def run_attention(case, torch, O_init=None, math=sg.MATH_FP32, force=sg.PATH_AUTO):
    dQ, dK, dV = (gu.to_device(op, torch) for op in (case.Q, case.K, case.V))
    dO = torch.from_numpy(case.O.storage.copy() if O_init is None else O_init.copy()).to("cuda")
    sg.sbgemm_attention(dQ.data_ptr() + 4 * case.Q.offset, case.Q.rs, case.Q.cs, case.Q.bs,
                        dK.data_ptr() + 4 * case.K.offset, case.K.rs, case.K.cs, case.K.bs,
                        dV.data_ptr() + 4 * case.V.offset, case.V.rs, case.V.cs, case.V.bs,
                        dO.data_ptr() + 4 * case.O.offset, case.O.rs, case.O.cs, case.O.bs,
                        case.M, case.N, case.D, case.Dv, case.batch, case.alpha, case.causal,
                        case.q_len, torch.cuda.current_stream().cuda_stream, math=math,
                        force_path=force)
    torch.cuda.synchronize()
    return dO.cpu().numpy()


def _sub(op, b):
    """The operand restricted to batch entry b (a one-entry view)."""
    return wl.Operand(op.storage, op.offset + b * op.bs, op.rs, op.cs, 0)


def check_attention(case, got_storage, batches=None, tol=1e-5):
    batches = range(case.batch) if batches is None else batches
    for b in batches:
        O, W, S = oracle.attention(_sub(case.Q, b), _sub(case.K, b), _sub(case.V, b), case.M, case.N,
                                   case.D, case.Dv, 1, case.alpha, case.causal, case.q_len)
        o = case.O
        got = np.array(wl.Operand(got_storage, o.offset + b * o.bs, o.rs, o.cs, 0).view(1, case.M, case.Dv),
                       dtype=np.float64)
        delta = tol * S[..., None] + 8 * U
        lim = (tol + 2 * delta) * W + 4 * U * np.abs(O)
        err = np.abs(got - O)
        bad = np.argwhere(~(err <= lim))
        assert bad.size == 0, (f"{case.name} batch {b}: {len(bad)} outputs outside the bound; first "
                               f"{tuple(bad[0])}: got {got[tuple(bad[0])]} want {O[tuple(bad[0])]} "
                               f"lim {lim[tuple(bad[0])]}")


SMALL = [
    # (M, N, batch, layout, causal, q_len)
    (100, 130, 3, "row", 0, 0),            # ragged rows and keys
    (192, 300, 2, "row", 1, 192),          # causal, queries end-aligned with the keys
    (128, 128, 4, "mixed", 1, 128),        # K read transposed, V and O column-major, Q batches reversed
    (384, 96, 2, "row", 1, 96),            # 4 heads stacked as rows against one K (grouped query)
    (1, 777, 3, "row", 1, 1),              # one decode row against a long context
    (70, 5, 2, "mixed", 0, 0),             # fewer keys than one block
]


@pytest.mark.parametrize("shape", SMALL, ids=[f"{s[0]}x{s[1]}x{s[2]}-{s[3]}-c{s[4]}" for s in SMALL])
def test_attention_small_against_oracle(torch, shape):
    M, N, batch, layout, causal, q_len = shape
    rng = np.random.default_rng(M * 7 + N)
    case = wl.random_attention(rng, M, N, 64, batch, layout, causal=causal, q_len=q_len)
    got = run_attention(case, torch)
    check_attention(case, got)


def test_attention_saturated_scores(torch):
    """Scores of several hundred: the running maximum keeps exp2 in range."""
    rng = np.random.default_rng(2)
    case = wl.random_attention(rng, 200, 333, 64, 2, "row", alpha=1.0, scale=3.0)
    got = run_attention(case, torch)
    assert np.isfinite(got).all()
    check_attention(case, got)


@pytest.mark.parametrize("name", list(wl.ATTENTION))
def test_attention_full_size_sampled_batches(torch, name):
    case = wl.make_attention(name)
    got = run_attention(case, torch)
    check_attention(case, got, batches=[0, case.batch // 2, case.batch - 1])


def test_attention_does_not_read_O(torch):
    """O's previous content (NaN here) never leaks into the result."""
    rng = np.random.default_rng(4)
    case = wl.random_attention(rng, 65, 70, 64, 2, "row")
    got = run_attention(case, torch, O_init=np.full(case.O.storage.shape, np.nan, np.float32))
    check_attention(case, got)


def test_attention_errors(torch):
    Q = torch.zeros(2 * 128 * 64, device="cuda")
    K = torch.zeros(2 * 128 * 64, device="cuda")
    V = torch.zeros(2 * 128 * 64, device="cuda")
    O = torch.zeros(2 * 128 * 64, device="cuda")

    def status(M=128, N=128, D=64, Dv=64, causal=0, q_len=0, o_ptr=None, q_ptr=None):
        try:
            sg.sbgemm_attention(q_ptr or Q.data_ptr(), 64, 1, 128 * 64, K.data_ptr(), 64, 1, 128 * 64,
                                V.data_ptr(), 64, 1, 128 * 64, o_ptr or O.data_ptr(), 64, 1, 128 * 64,
                                M, N, D, Dv, 2, 0.125, causal, q_len)
            torch.cuda.synchronize()
            return sg.SBGEMM_OK
        except sg.SbgemmError as e:
            return e.status

    assert status() == sg.SBGEMM_OK
    assert status(D=48, Dv=48) == sg.SBGEMM_ERR_UNSUPPORTED
    assert status(D=64, Dv=32) == sg.SBGEMM_ERR_UNSUPPORTED
    assert status(N=0) == sg.SBGEMM_ERR_INVALID_VALUE
    assert status(M=0, N=0) == sg.SBGEMM_OK
    assert status(causal=1, q_len=0) == sg.SBGEMM_ERR_INVALID_VALUE
    assert status(causal=1, q_len=129) == sg.SBGEMM_ERR_INVALID_VALUE
    assert status(causal=2, q_len=1) == sg.SBGEMM_ERR_INVALID_VALUE
    assert status(o_ptr=K.data_ptr() + 4 * 64) == sg.SBGEMM_ERR_OUTPUT_OVERLAP
    host = np.zeros(2 * 128 * 64, dtype=np.float32)
    assert status(q_ptr=host.ctypes.data) == sg.SBGEMM_ERR_NOT_DEVICE_MEMORY


def test_attention_torch_helper_shared_kv(torch):
    """sg.attention on tensors: 4 query heads stacked against one shared K, V
    (batch 1 broadcast), causal per head, against float64 torch on the CPU."""
    gen = torch.Generator().manual_seed(8)
    T, H = 200, 4
    q = torch.randn(3, H * T, 64, generator=gen)
    k = torch.randn(1, T, 64, generator=gen)
    v = torch.randn(1, T, 64, generator=gen)
    o = torch.empty(3, H * T, 64, device="cuda")
    sg.attention(q.cuda(), k.cuda(), v.cuda(), o, causal=True, q_len=T)
    torch.cuda.synchronize()
    s = (q.double() @ k.double().transpose(1, 2)) / 8.0
    pos = torch.arange(H * T) % T
    mask = torch.arange(T)[None, :] > pos[:, None]
    s = s.masked_fill(mask[None], float("-inf"))
    p = torch.softmax(s, dim=-1)
    want = p @ v.double()
    w = p @ v.double().abs()
    assert bool(((o.cpu().double() - want).abs() <= 2e-4 * w + 1e-6).all())


# ---- TF32 tensor-core kernel (opt-in) -------------------------------------------

TOL_TF32 = 2e-3
# (M, N, batch, causal, q_len); row-major operands, which suit its tensor maps.
TF32_SMALL = [
    (100, 130, 3, 0, 0),          # ragged rows and keys
    (192, 300, 2, 1, 192),        # causal, end-aligned
    (384, 96, 2, 1, 96),          # 4 heads stacked as rows against one K (grouped query)
    (1, 777, 3, 1, 1),            # one decode row against a long context
    (70, 5, 2, 0, 0),             # fewer keys than one block
    (256, 512, 2, 0, 0),          # whole blocks: 2 row blocks, 8 key blocks
]


@pytest.mark.parametrize("shape", TF32_SMALL, ids=[f"{s[0]}x{s[1]}x{s[2]}-c{s[3]}" for s in TF32_SMALL])
def test_attention_tf32_small_against_oracle(torch, shape):
    M, N, batch, causal, q_len = shape
    rng = np.random.default_rng(M * 11 + N)
    case = wl.random_attention(rng, M, N, 64, batch, "row", causal=causal, q_len=q_len)
    got = run_attention(case, torch, math=sg.MATH_TF32, force=sg.PATH_TMA_TF32)
    check_attention(case, got, tol=TOL_TF32)
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where


@pytest.mark.parametrize("name", list(wl.ATTENTION))
def test_attention_tf32_full_size_sampled_batches(torch, name):
    case = wl.make_attention(name)
    got = run_attention(case, torch, math=sg.MATH_TF32, force=sg.PATH_TMA_TF32)
    check_attention(case, got, batches=[0, case.batch // 2, case.batch - 1], tol=TOL_TF32)


def test_attention_tf32_saturated_scores_and_stale_output(torch):
    """Scores of several hundred, and O's previous content (NaN) never read."""
    rng = np.random.default_rng(12)
    case = wl.random_attention(rng, 200, 333, 64, 2, "row", alpha=1.0, scale=3.0)
    got = run_attention(case, torch, O_init=np.full(case.O.storage.shape, np.nan, np.float32),
                        math=sg.MATH_TF32, force=sg.PATH_TMA_TF32)
    assert np.isfinite(got).all()
    check_attention(case, got, tol=TOL_TF32)


@pytest.mark.parametrize("ramp", ["every_chunk", "second_chunk"])
def test_attention_tf32_reference_raises_inside_blocks(torch, ramp):
    """Scores that climb along the keys, so that a row's reference maximum
    moves by more than 2^8 inside later blocks: in every 64-key chunk, or only
    in the second chunk of each 128-key block (then the block's first half of
    P and O are rescaled after that half's exponentials were written, before
    P V reads it)."""
    rng = np.random.default_rng(31 if ramp == "every_chunk" else 32)
    M, N, D, batch = 256, 512, 64, 2
    case = wl.random_attention(rng, M, N, D, batch, "row", alpha=1.0, scale=0.1)
    q = case.Q.storage.reshape(batch, M, D)
    k = case.K.storage.reshape(batch, N, D)
    q[:, :, 0] += 1.0
    n = np.arange(N, dtype=np.float32)
    climb = 0.15 * n if ramp == "every_chunk" else np.where(n % 128 >= 64, 0.15 * n, 0.0)
    k[:, :, 0] += climb.astype(np.float32)
    got = run_attention(case, torch, math=sg.MATH_TF32, force=sg.PATH_TMA_TF32)
    assert np.isfinite(got).all()
    check_attention(case, got, tol=TOL_TF32)
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where


def test_attention_tf32_other_layouts_fall_back_or_refuse(torch):
    """K read transposed (no unit stride along the head dimension): with
    math = TF32 the fp32 kernel runs (fp32 bound); forcing the tensor-core
    kernel is refused."""
    rng = np.random.default_rng(13)
    case = wl.random_attention(rng, 128, 128, 64, 2, "mixed", causal=1, q_len=128)
    got = run_attention(case, torch, math=sg.MATH_TF32)
    check_attention(case, got)
    with pytest.raises(sg.SbgemmError) as e:
        run_attention(case, torch, math=sg.MATH_TF32, force=sg.PATH_TMA_TF32)
    assert e.value.status == sg.SBGEMM_ERR_UNSUPPORTED
    with pytest.raises(sg.SbgemmError) as e:
        run_attention(case, torch, math=sg.MATH_FP32, force=sg.PATH_TMA_TF32)
    assert e.value.status == sg.SBGEMM_ERR_INVALID_VALUE
    with pytest.raises(sg.SbgemmError) as e:
        run_attention(case, torch, math=sg.MATH_TF32, force=sg.PATH_GATHER_FFMA)
    assert e.value.status == sg.SBGEMM_ERR_UNSUPPORTED


def test_attention_tf32_torch_helper(torch):
    """sg.attention(math=TF32) on tensors against float64 torch on the CPU."""
    gen = torch.Generator().manual_seed(9)
    q = torch.randn(4, 300, 64, generator=gen)
    k = torch.randn(4, 260, 64, generator=gen)
    v = torch.randn(4, 260, 64, generator=gen)
    o = torch.empty(4, 300, 64, device="cuda")
    sg.attention(q.cuda(), k.cuda(), v.cuda(), o, math=sg.MATH_TF32)
    torch.cuda.synchronize()
    p = torch.softmax((q.double() @ k.double().transpose(1, 2)) / 8.0, dim=-1)
    want = p @ v.double()
    w = p @ v.double().abs()
    assert bool(((o.cpu().double() - want).abs() <= 2e-2 * w + 1e-6).all())


def test_attention_tf32_shared_kv_and_column_major_o(torch):
    """TF32 kernel with K and V shared by every batch entry (zero batch
    stride, grouped-query heads stacked as rows, causal per head) and O
    written column-major (strided stores)."""
    rng = np.random.default_rng(21)
    T, H, batch = 160, 3, 2
    M, N, D = H * T, T, 64
    q = rng.standard_normal(batch * M * D).astype(np.float32)
    k = rng.standard_normal(N * D).astype(np.float32)
    v = rng.standard_normal(N * D).astype(np.float32)
    case = wl.AttnCase("tf32_shared", wl.Operand(q, 0, D, 1, M * D), wl.Operand(k, 0, D, 1, 0),
                       wl.Operand(v, 0, D, 1, 0),
                       wl.Operand(np.zeros(batch * M * D, np.float32), 0, 1, M, M * D),
                       M, N, D, D, batch, 0.125, 1, T)
    got = run_attention(case, torch, math=sg.MATH_TF32, force=sg.PATH_TMA_TF32)
    check_attention(case, got, tol=TOL_TF32)
