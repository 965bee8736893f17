"""Helpers for the GPU parity tests: place a workloads.Case on the device, run
it through the C-ABI, read C back and compare it with the CPU oracle."""

from __future__ import annotations

import numpy as np

import oracle
import strided_gemm_gb300 as sg

# Tolerances of the strided-batched problem statement, relative to the oracle's
# bound |alpha| * sum_k |a||b| + |C0| of each element.
TOL_FFMA = 1e-5
TOL_TF32 = 2e-3


def to_device(op, torch):
    t = torch.from_numpy(op.storage).to("cuda")
    return t


def run_case(case, torch, math=sg.MATH_FP32, force_path=sg.PATH_AUTO, c_init=None,
             stream=None, entry="sbgemm_ex"):
    """Runs ``case`` on the GPU; returns the whole C storage after the call (numpy)."""
    dA, dB = to_device(case.A, torch), to_device(case.B, torch)
    c_host = case.C.storage.copy() if c_init is None else c_init.copy()
    dC = torch.from_numpy(c_host).to("cuda")
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    args = (dA.data_ptr() + 4 * case.A.offset, case.A.rs, case.A.cs, case.A.bs,
            dB.data_ptr() + 4 * case.B.offset, case.B.rs, case.B.cs, case.B.bs,
            dC.data_ptr() + 4 * case.C.offset, case.C.rs, case.C.cs, case.C.bs,
            case.M, case.N, case.K, case.batch, case.alpha, case.accumulate, s)
    if entry == "sbgemm":
        sg.sbgemm(*args)
    else:
        sg.sbgemm_ex(*args, math=math, force_path=force_path)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


def logical_c(case, c_storage):
    """[batch, M, N] view of C over a storage array."""
    op = type(case.C)(c_storage, case.C.offset, case.C.rs, case.C.cs, case.C.bs)
    return np.array(op.view(case.batch, case.M, case.N))


def check_full(case, got_storage, tol=TOL_FFMA, exact=False):
    """Compare every element of C with the oracle."""
    ref, bound = oracle.case_product(case)
    got = logical_c(case, got_storage).astype(np.float64)
    if exact:
        want = ref.astype(np.float32).astype(np.float64)
        bad = np.argwhere(got != want)
        assert bad.size == 0, (f"{case.name}: {len(bad)} inexact elements, first "
                               f"{tuple(bad[0])}: got {got[tuple(bad[0])]} want {want[tuple(bad[0])]}")
    else:
        err = np.abs(got - ref)
        lim = tol * bound
        bad = np.argwhere(~(err <= lim))
        assert bad.size == 0, (f"{case.name}: {len(bad)} elements outside {tol}*bound, first "
                               f"{tuple(bad[0])}: got {got[tuple(bad[0])]} ref {ref[tuple(bad[0])]} "
                               f"bound {bound[tuple(bad[0])]}")
    return ref


def sample_points(case, n=1500, seed=0):
    """Indices (b, m, n) that always include the corners and the last row and
    column of the first and last batch entry, plus random interior points."""
    rng = np.random.default_rng(seed)
    pts = []
    for b in {0, case.batch - 1}:
        for m in {0, case.M - 1}:
            for nn in {0, case.N - 1}:
                pts.append((b, m, nn))
        for _ in range(16):
            pts.append((b, case.M - 1, int(rng.integers(0, case.N))))
            pts.append((b, int(rng.integers(0, case.M)), case.N - 1))
    r = np.stack([rng.integers(0, case.batch, n), rng.integers(0, case.M, n),
                  rng.integers(0, case.N, n)], axis=1)
    return np.concatenate([np.array(pts, dtype=np.int64), r.astype(np.int64)])


def check_points(case, got_storage, tol=TOL_FFMA, exact=False, n=1500, points=None):
    """Compares sampled elements (or the given (b, m, n) points) with the
    oracle, one by one."""
    idx = sample_points(case, n) if points is None else np.asarray(points, dtype=np.int64)
    ref, bound = oracle.case_points(case, idx)
    c = case.C
    got = c_storage_at(case, got_storage, idx)
    if exact:
        want = ref.astype(np.float32).astype(np.float64)
        assert np.array_equal(got, want), f"{case.name}: inexact sampled elements"
    else:
        err = np.abs(got - ref)
        bad = np.flatnonzero(~(err <= tol * bound))
        assert bad.size == 0, (f"{case.name}: {bad.size} sampled elements outside {tol}*bound; "
                               f"first idx {idx[bad[0]]} got {got[bad[0]]} ref {ref[bad[0]]}")


def c_storage_at(case, storage, idx):
    c = case.C
    off = c.offset + idx[:, 0] * c.bs + idx[:, 1] * c.rs + idx[:, 2] * c.cs
    return storage[off].astype(np.float64)
