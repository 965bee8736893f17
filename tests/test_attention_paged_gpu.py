"""Fused attention at head dimensions 32, 64, 96 and 128, the split-key decode
kernel for a few query rows, and attention over a paged K / V cache read
through a block table ("rvllm CUDA path", sections "The kernels" and "What's
basic about it"), all through the C ABI against the fp64 oracle.

The bound is the fused-attention one (tests/test_attention_gpu.py):
|O - O_ref| <= (1e-5 + 2 delta) W + 4u |O_ref| with delta = 1e-5 smag + 8u,
W = sum_n P |V| and smag the largest |alpha| sum_d |q k| of the row.  Paged
caches hold NaN in every slot no sequence owns and the block tables -1 past
each sequence's blocks, so a kernel that reads one of them fails the test."""

import numpy as np
import pytest

import oracle
import strided_gemm_gb300 as sg
import workloads as wl
from tests import gpu_util as gu
from tests.test_attention_gpu import check_attention, run_attention

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
TOL = 1e-5


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    return t


@pytest.fixture(scope="module")
def workspace(torch):
    return torch.empty(sg.sbgemm_workspace_bytes(torch.cuda.current_device()), dtype=torch.uint8,
                       device="cuda")


def check_result(O, W, S, got, name, tol=TOL):
    """got [batch, M, Dv] against the oracle's O, W, S."""
    delta = tol * S[..., None] + 8 * U
    lim = (tol + 2 * delta) * W + 4 * U * np.abs(O)
    err = np.abs(got - O)
    bad = np.argwhere(~(err <= lim))
    assert bad.size == 0, (f"{name}: {len(bad)} outputs outside the bound; first {tuple(bad[0])}: "
                           f"got {got[tuple(bad[0])]} want {O[tuple(bad[0])]} lim {lim[tuple(bad[0])]}")


# ---- head dimensions, row-block kernel -------------------------------------------

HEAD_DIMS = [
    # (D, M, N, batch, layout, causal, q_len)
    (32, 100, 130, 3, "row", 0, 0),
    (32, 192, 300, 2, "mixed", 1, 192),
    (96, 100, 130, 2, "row", 1, 100),
    (96, 70, 5, 2, "mixed", 0, 0),
    (128, 130, 257, 2, "row", 0, 0),
    (128, 384, 96, 1, "row", 1, 96),
]


@pytest.mark.parametrize("shape", HEAD_DIMS, ids=[f"d{s[0]}-{s[1]}x{s[2]}x{s[3]}-{s[4]}-c{s[5]}"
                                                  for s in HEAD_DIMS])
def test_head_dims_against_oracle(torch, shape):
    D, M, N, batch, layout, causal, q_len = shape
    rng = np.random.default_rng(D * 1000 + M + N)
    case = wl.random_attention(rng, M, N, D, batch, layout, causal=causal, q_len=q_len,
                               alpha=1.0 / np.sqrt(D))
    got = run_attention(case, torch)
    check_attention(case, got)


@pytest.mark.parametrize("D", [32, 96, 128])
def test_head_dims_saturated_scores(torch, D):
    rng = np.random.default_rng(D)
    case = wl.random_attention(rng, 150, 200, D, 2, "row", alpha=1.0, scale=3.0)
    got = run_attention(case, torch)
    assert np.isfinite(got).all()
    check_attention(case, got)


# ---- decode kernel (few rows per entry), strided operands -------------------------

DECODE = [
    # (D, M, N, batch, causal, q_len, with workspace)
    (64, 1, 777, 3, 1, 1, True),
    (64, 1, 777, 3, 1, 1, False),
    (64, 4, 2000, 5, 1, 1, True),          # 4 query heads stacked against one KV head
    (64, 8, 1500, 2, 1, 2, True),          # 4 heads x 2 new tokens, causal per head
    (64, 3, 65, 4, 0, 0, True),
    (32, 8, 999, 3, 1, 4, True),
    (32, 5, 40, 2, 0, 0, False),
    (96, 4, 1234, 2, 1, 1, True),
    (96, 1, 31, 2, 0, 0, True),
    (128, 4, 3001, 2, 1, 2, True),
    (128, 2, 100, 3, 1, 1, False),
]


@pytest.mark.parametrize("shape", DECODE, ids=[f"d{s[0]}-m{s[1]}-n{s[2]}-b{s[3]}-c{s[4]}q{s[5]}"
                                               f"-{'ws' if s[6] else 'nows'}" for s in DECODE])
def test_decode_against_oracle(torch, workspace, shape):
    D, M, N, batch, causal, q_len, use_ws = shape
    rng = np.random.default_rng(D + 3 * M + N)
    case = wl.random_attention(rng, M, N, D, batch, "row", causal=causal, q_len=q_len,
                               alpha=1.0 / np.sqrt(D))
    dQ, dK, dV = (gu.to_device(op, torch) for op in (case.Q, case.K, case.V))
    dO = torch.full((case.O.storage.size,), float("nan"), device="cuda")
    ws = dict(workspace=workspace.data_ptr(), workspace_bytes=workspace.numel()) if use_ws else {}
    sg.sbgemm_attention(dQ.data_ptr(), case.Q.rs, case.Q.cs, case.Q.bs, dK.data_ptr(), case.K.rs,
                        case.K.cs, case.K.bs, dV.data_ptr(), case.V.rs, case.V.cs, case.V.bs,
                        dO.data_ptr(), case.O.rs, case.O.cs, case.O.bs, case.M, case.N, case.D,
                        case.Dv, case.batch, case.alpha, case.causal, case.q_len,
                        torch.cuda.current_stream().cuda_stream, **ws)
    torch.cuda.synchronize()
    check_attention(case, dO.cpu().numpy())


def test_decode_same_result_in_tf32_math(torch, workspace):
    """A few rows per entry run the fp32 decode kernel in either math: the
    two results are identical."""
    rng = np.random.default_rng(77)
    case = wl.random_attention(rng, 4, 900, 64, 3, "row", causal=1, q_len=1)
    a = run_attention(case, torch, math=sg.MATH_FP32)
    b = run_attention(case, torch, math=sg.MATH_TF32)
    assert np.array_equal(a, b)
    check_attention(case, a)


# ---- paged K / V -----------------------------------------------------------------

def run_paged(case, torch, workspace=None, seq_lens=True, table=None, lens=None):
    """Runs sbgemm_attention_paged; returns O [batch, M, D] (numpy)."""
    dQ = gu.to_device(case.Q, torch)
    dK = torch.from_numpy(np.ascontiguousarray(case.K_cache).reshape(-1)).to("cuda")
    dV = torch.from_numpy(np.ascontiguousarray(case.V_cache).reshape(-1)).to("cuda")
    dT = torch.from_numpy(np.ascontiguousarray(case.block_table if table is None else table)).to("cuda")
    dL = torch.from_numpy(np.ascontiguousarray(case.seq_lens if lens is None else lens)).to("cuda")
    dO = torch.full((case.O.storage.size,), float("nan"), device="cuda")
    ws = dict(workspace=workspace.data_ptr(), workspace_bytes=workspace.numel()) if workspace is not None else {}
    sg.sbgemm_attention_paged(dQ.data_ptr() + 4 * case.Q.offset, case.Q.rs, case.Q.cs, case.Q.bs,
                              dK.data_ptr(), dV.data_ptr(), case.K_cache.shape[0], case.block_size,
                              case.n_kv_heads, dT.data_ptr(), case.block_table.shape[1],
                              dL.data_ptr() if seq_lens else 0,
                              dO.data_ptr(), case.O.rs, case.O.cs, case.O.bs, case.M, case.N, case.D,
                              case.D, case.n_seqs, case.alpha, case.causal, case.q_len,
                              torch.cuda.current_stream().cuda_stream, **ws)
    torch.cuda.synchronize()
    return dO.cpu().numpy().reshape(case.batch, case.M, case.D).astype(np.float64)


def paged_oracle(case, entries=None):
    O, W, S = oracle.attention_paged(case.Q, case.K_cache, case.V_cache, case.block_table,
                                     case.seq_lens, case.M, case.alpha, case.causal, case.q_len)
    return O, W, S


PAGED = [
    # (lens, n_kv_heads, group, q_len, D, block_size, causal, workspace)
    ([777, 5, 300], 2, 4, 1, 64, 16, 1, True),       # decode kernel, ragged contexts
    ([777, 5, 300], 2, 4, 1, 64, 16, 1, False),      # one CTA per entry
    ([64, 65, 129], 3, 1, 1, 64, 1, 1, True),        # one token per block
    ([200, 33], 2, 8, 1, 32, 5, 1, True),            # a block size that divides nothing
    ([500, 1000], 1, 2, 2, 96, 64, 1, True),         # two new tokens per sequence
    ([300, 301], 2, 4, 1, 128, 16, 0, True),
    ([400, 257, 130], 2, 4, 40, 64, 16, 1, True),    # row-block kernel: 160 rows (prefill chunk)
    ([129, 64], 2, 3, 64, 32, 7, 1, True),           # row-block kernel, D 32
    ([300, 150], 1, 1, 130, 128, 16, 1, True),       # row-block kernel, D 128
    ([90, 200], 2, 2, 50, 96, 3, 0, True),           # row-block kernel, D 96, no mask
]


@pytest.mark.parametrize("shape", PAGED, ids=[f"n{'-'.join(map(str, s[0]))}-h{s[1]}g{s[2]}q{s[3]}-d{s[4]}"
                                              f"-bs{s[5]}-c{s[6]}-{'ws' if s[7] else 'nows'}" for s in PAGED])
def test_paged_against_oracle(torch, workspace, shape):
    lens, heads, group, q_len, D, bsz, causal, use_ws = shape
    rng = np.random.default_rng(sum(lens) + D + bsz)
    case = wl.random_paged_attention(rng, lens, heads, group, q_len, D, bsz, causal=causal)
    got = run_paged(case, torch, workspace if use_ws else None)
    O, W, S = paged_oracle(case)
    check_result(O, W, S, got, "paged")


def test_paged_equal_lengths_without_seq_lens(torch, workspace):
    """seq_lens NULL: every sequence has N keys."""
    rng = np.random.default_rng(5)
    case = wl.random_paged_attention(rng, [333, 333, 333], 2, 4, 1, 64, 16, causal=1)
    got = run_paged(case, torch, workspace, seq_lens=False)
    O, W, S = paged_oracle(case)
    check_result(O, W, S, got, "paged, no seq_lens")


def test_paged_matches_strided_on_the_same_context(torch, workspace):
    """The paged read and the strided read of the same keys give the same
    bits (same kernel arithmetic, only the row addresses differ)."""
    rng = np.random.default_rng(6)
    n = 700
    case = wl.random_paged_attention(rng, [n, n], 2, 4, 1, 64, 16, causal=1)
    got = run_paged(case, torch, workspace)
    K = np.ascontiguousarray(case.K_ctx[:, :, :n]).reshape(-1)
    V = np.ascontiguousarray(case.V_ctx[:, :, :n]).reshape(-1)
    D, M = case.D, case.M
    strided = wl.AttnCase("strided", case.Q, wl.Operand(K, 0, D, 1, n * D), wl.Operand(V, 0, D, 1, n * D),
                          wl.Operand(np.zeros(case.batch * M * D, np.float32), 0, D, 1, M * D),
                          M, n, D, D, case.batch, case.alpha, 1, case.q_len)
    dQ, dK, dV = (gu.to_device(op, torch) for op in (strided.Q, strided.K, strided.V))
    dO = torch.zeros(case.batch * M * D, device="cuda")
    sg.sbgemm_attention(dQ.data_ptr(), strided.Q.rs, 1, strided.Q.bs, dK.data_ptr(), D, 1, n * D,
                        dV.data_ptr(), D, 1, n * D, dO.data_ptr(), D, 1, M * D, M, n, D, D, case.batch,
                        case.alpha, 1, case.q_len, torch.cuda.current_stream().cuda_stream,
                        workspace=workspace.data_ptr(), workspace_bytes=workspace.numel())
    torch.cuda.synchronize()
    assert np.array_equal(dO.cpu().numpy().reshape(got.shape), got.astype(np.float32))


@pytest.mark.parametrize("name", list(wl.PAGED))
def test_paged_full_size_sampled_entries(torch, workspace, name):
    """The decode workload at full size; the oracle checks every row of a
    few entries (the first, the longest context's, the last)."""
    case = wl.make_paged(name)
    got = run_paged(case, torch, workspace)
    H = case.n_kv_heads
    seqs = sorted({0, int(np.argmax(case.seq_lens)), case.n_seqs - 1})
    for s in seqs:
        n = int(case.seq_lens[s])
        for h in (0, H - 1):
            b = s * H + h
            Qb = wl.Operand(case.Q.storage, case.Q.offset + b * case.Q.bs, case.Q.rs, case.Q.cs, 0)
            Kc = oracle.kv_gather(case.K_cache, case.block_table, s, h, n).reshape(-1)
            Vc = oracle.kv_gather(case.V_cache, case.block_table, s, h, n).reshape(-1)
            O, W, S = oracle.attention(Qb, wl.Operand(Kc, 0, case.D, 1, 0), wl.Operand(Vc, 0, case.D, 1, 0),
                                       case.M, n, case.D, case.D, 1, case.alpha, case.causal, case.q_len)
            check_result(O, W, S, got[b:b + 1], f"{name} seq {s} head {h}")


def test_paged_bad_table_entry_is_reported_not_read(torch, workspace):
    """A block id outside the cache: the kernel reads nothing there, the
    other entries are exact, and the device status says which check fired."""
    rng = np.random.default_rng(8)
    case = wl.random_paged_attention(rng, [100, 200], 1, 4, 1, 64, 16, causal=1)
    table = case.block_table.copy()
    table[1, 3] = case.K_cache.shape[0] + 1000
    for ws in (workspace, None):
        got = run_paged(case, torch, ws, table=table)
        st, where = sg.sbgemm_device_status()
        assert st == sg.SBGEMM_ERR_DEVICE_CHECK and where == 10, (st, where)
        O, W, S = paged_oracle(case)
        check_result(O[:1], W[:1], S[:1], got[:1], "untouched sequence")
    # A length past N is clamped and reported the same way.
    lens = case.seq_lens.copy()
    lens[0] = case.N + 5
    run_paged(case, torch, workspace, lens=lens)
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_ERR_DEVICE_CHECK and where == 10, (st, where)
    assert sg.sbgemm_device_status() == (sg.SBGEMM_OK, 0)


def test_paged_errors(torch, workspace):
    rng = np.random.default_rng(9)
    case = wl.random_paged_attention(rng, [40, 20], 2, 2, 1, 64, 8, causal=1)
    dQ = gu.to_device(case.Q, torch)
    dK = torch.from_numpy(case.K_cache.reshape(-1)).to("cuda")
    dV = torch.from_numpy(case.V_cache.reshape(-1)).to("cuda")
    dT = torch.from_numpy(case.block_table).to("cuda")
    dL = torch.from_numpy(case.seq_lens).to("cuda")
    dO = torch.zeros(case.O.storage.size, device="cuda")
    nb, mb = case.K_cache.shape[0], case.block_table.shape[1]

    def status(**kw):
        a = dict(Q=dQ.data_ptr(), K=dK.data_ptr(), V=dV.data_ptr(), nb=nb, bsz=8, H=2, T=dT.data_ptr(),
                 mb=mb, L=dL.data_ptr(), O=dO.data_ptr(), M=case.M, N=case.N, D=64, Dv=64, S=2,
                 causal=1, q_len=1, ws=0, wsb=0)
        a.update(kw)
        try:
            sg.sbgemm_attention_paged(a["Q"], 64, 1, case.M * 64, a["K"], a["V"], a["nb"], a["bsz"], a["H"],
                                      a["T"], a["mb"], a["L"], a["O"], 64, 1, case.M * 64, a["M"], a["N"],
                                      a["D"], a["Dv"], a["S"], 0.125, a["causal"], a["q_len"],
                                      workspace=a["ws"], workspace_bytes=a["wsb"])
            torch.cuda.synchronize()
            return sg.SBGEMM_OK
        except sg.SbgemmError as e:
            return e.status

    assert status() == sg.SBGEMM_OK
    assert status(N=mb * 8 + 1) == sg.SBGEMM_ERR_INVALID_VALUE       # past the table
    assert status(bsz=0) == sg.SBGEMM_ERR_INVALID_VALUE
    assert status(D=48, Dv=48) == sg.SBGEMM_ERR_UNSUPPORTED
    assert status(D=64, Dv=32) == sg.SBGEMM_ERR_UNSUPPORTED
    assert status(K=dK.data_ptr() + 4) == sg.SBGEMM_ERR_INVALID_VALUE   # not 16-byte aligned
    assert status(T=0) == sg.SBGEMM_ERR_NULL_POINTER
    assert status(causal=1, q_len=0) == sg.SBGEMM_ERR_INVALID_VALUE
    assert status(O=dK.data_ptr()) == sg.SBGEMM_ERR_OUTPUT_OVERLAP
    assert status(O=dT.data_ptr()) == sg.SBGEMM_ERR_OUTPUT_OVERLAP
    host = np.zeros(case.block_table.size, np.int32)
    assert status(T=host.ctypes.data) == sg.SBGEMM_ERR_NOT_DEVICE_MEMORY
    host_cache = np.zeros(case.K_cache.size + 16, np.float32)
    aligned = host_cache.ctypes.data + (-host_cache.ctypes.data) % 16
    assert status(K=aligned) == sg.SBGEMM_ERR_NOT_DEVICE_MEMORY
    assert status(ws=dK.data_ptr(), wsb=4096) == sg.SBGEMM_ERR_OUTPUT_OVERLAP
    assert status(ws=workspace.data_ptr(), wsb=workspace.numel()) == sg.SBGEMM_OK
    assert status(M=0) == sg.SBGEMM_OK and status(S=0) == sg.SBGEMM_OK
