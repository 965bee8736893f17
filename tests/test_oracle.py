"""Pins for the CPU oracle, run without a GPU.

Each test checks the oracle against something other than itself: values the
pages print (tests/golden), closed forms, special cases that reduce to a numpy
library routine on explicitly materialised matrices, exact integer brute force,
and invariants of the product's definition (StaleyNET "GPU Implementation",
section "The matrix product").
"""

import os

import numpy as np
import pytest

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# Awkward sizes: StaleyNET "Testing the kernels" (17 x 33 x 9, 5 x 129 x 31) and
# the kael "How it is tested" matmul shapes (rows, inner, columns).
AWKWARD_MNK = [(17, 9, 33), (5, 31, 129), (1, 1, 1), (4, 4, 4), (5, 9, 3),
               (8, 7, 16), (33, 65, 20), (64, 64, 1), (1, 1, 64)]
LAYOUTS = ["row", "col", "neg_row", "gap", "bcast_row"]


def _int_expected(case):
    """alpha*A@B + C0 for integer-valued operands, computed exactly with numpy's
    int64 matmul on the materialised strided views."""
    A = case.A.view(case.batch, case.M, case.K).astype(np.int64)
    B = case.B.view(case.batch, case.K, case.N).astype(np.int64)
    s = np.matmul(A, B)
    t = np.matmul(np.abs(A), np.abs(B))
    ref = case.alpha * s.astype(np.float64)
    bound = abs(case.alpha) * t.astype(np.float64)
    if case.accumulate:
        c0 = case.C.view(case.batch, case.M, case.N).astype(np.float64)
        ref = ref + c0
        bound = bound + np.abs(c0)
    return ref, bound


def _cases(seed=0):
    rng = np.random.default_rng(seed)
    out = []
    j = 0
    for i, (M, K, N) in enumerate(AWKWARD_MNK):
        for la in LAYOUTS:
            lb = LAYOUTS[(i + LAYOUTS.index(la)) % len(LAYOUTS)]
            bsm = [("dense", "dense"), ("zero", "dense"), ("dense", "neg"),
                   ("neg", "zero")][(i + len(la)) % 4]
            batch = [1, 3, 2][i % 3]
            # alpha and accumulate cycle independently so every pairing occurs.
            alpha = [1.0, 0.125, -2.0][j % 3]
            acc = (j // 3) % 2
            j += 1
            out.append(wl.random_strided(rng, M, N, K, batch, la, lb,
                                         c_layout="col" if i % 2 else "row",
                                         bs_mode=bsm, values="int",
                                         accumulate=acc, alpha=alpha))
    return out


def run_int_pins(lib=None):
    """Exact brute-force comparison over every layout; returns the number of
    mismatching cases (0 for a correct oracle).  Also used on mutated builds."""
    bad = 0
    for case in _cases():
        ref, bound = oracle.case_product(case, lib=lib, nthreads=3)
        eref, ebound = _int_expected(case)
        if not (np.array_equal(ref, eref) and np.array_equal(bound, ebound)):
            bad += 1
    return bad


def test_brute_force_integers_all_layouts(oracle_lib):
    assert run_int_pins() == 0


def test_real_values_match_numpy_float64():
    rng = np.random.default_rng(1)
    for la, lb in [("row", "col"), ("col", "row"), ("neg_row", "gap"), ("gap", "bcast_row")]:
        case = wl.random_strided(rng, 37, 29, 131, 2, la, lb, values="real",
                                 accumulate=1, alpha=0.7)
        ref, bound = oracle.case_product(case)
        A = case.A.view(case.batch, case.M, case.K).astype(np.float64)
        B = case.B.view(case.batch, case.K, case.N).astype(np.float64)
        C0 = case.C.view(case.batch, case.M, case.N).astype(np.float64)
        want = np.float64(np.float32(0.7)) * np.einsum("bmk,bkn->bmn", A, B) + C0
        assert np.all(np.abs(ref - want) <= 1e-12 * bound + 1e-300)


def test_golden_transposed_view():
    """kael trace: x [2,3] = 0..5 read with strides (1,3) is [[0,3],[1,4],[2,5]].
    I(3) * x^T through the oracle must reproduce the printed read-out."""
    g = {}
    for line in open(os.path.join(GOLDEN, "kael_transpose_view.txt")):
        if line.startswith("#") or not line.strip():
            continue
        key, *vals = line.split()
        g[key] = [int(v) for v in vals]
    storage = np.array(g["storage"], dtype=np.float32)
    rs, cs = g["xT_strides"]
    K, N = g["xT_shape"]           # x^T is [3, 2]: it plays B with K=3, N=2
    eye = np.eye(K, dtype=np.float32).reshape(-1)
    A = wl.Operand(eye, 0, K, 1, 0)
    B = wl.Operand(storage, 0, rs, cs, 0)
    C = wl.Operand(np.zeros(K * N, np.float32), 0, N, 1, 0)
    ref, _ = oracle.product(A, B, C, K, N, K, 1, 1.0, 0)
    assert ref.reshape(-1).tolist() == [float(v) for v in g["xT_rowmajor"]]


def test_identity_exact_real_values():
    rng = np.random.default_rng(2)
    M, K, N = 19, 19, 23
    a = rng.standard_normal(M * K).astype(np.float32)
    b = rng.standard_normal(K * N).astype(np.float32)
    eye = np.eye(19, dtype=np.float32).reshape(-1)
    C = wl.Operand(np.zeros(M * N, np.float32), 0, N, 1, 0)
    # A = I  =>  C = B bitwise (one non-zero term per sum).
    ref, _ = oracle.product(wl.Operand(eye, 0, K, 1, 0), wl.Operand(b, 0, N, 1, 0),
                            C, M, N, K, 1, 1.0, 0)
    assert np.array_equal(ref[0], b.reshape(K, N).astype(np.float64))
    # B = I read with swapped strides (still I)  =>  C = A.
    C2 = wl.Operand(np.zeros(M * K, np.float32), 0, K, 1, 0)
    ref, _ = oracle.product(wl.Operand(a, 0, K, 1, 0), wl.Operand(eye, 0, 1, 19, 0),
                            C2, M, K, K, 1, 1.0, 0)
    assert np.array_equal(ref[0], a.reshape(M, K).astype(np.float64))


def test_zero_operand_and_overwrite_does_not_read_c():
    M, K, N = 7, 5, 6
    zeros = np.zeros(M * K, np.float32)
    b = np.arange(K * N, dtype=np.float32)
    c0 = np.random.default_rng(3).standard_normal(M * N).astype(np.float32)
    nan_c = np.full(M * N, np.nan, np.float32)
    A, B = wl.Operand(zeros, 0, K, 1, 0), wl.Operand(b, 0, N, 1, 0)
    ref, _ = oracle.product(A, B, wl.Operand(nan_c, 0, N, 1, 0), M, N, K, 1, 1.0, 0)
    assert np.all(ref == 0.0)
    ref, bound = oracle.product(A, B, wl.Operand(c0, 0, N, 1, 0), M, N, K, 1, 3.0, 1)
    assert np.array_equal(ref[0], c0.reshape(M, N).astype(np.float64))
    assert np.array_equal(bound[0], np.abs(c0.reshape(M, N)).astype(np.float64))


def test_swapped_strides_equal_explicit_transpose_copy():
    rng = np.random.default_rng(4)
    M, K, N = 13, 21, 17
    a_km = rng.standard_normal((K, M)).astype(np.float32)   # stores A^T
    b_nk = rng.standard_normal((N, K)).astype(np.float32)   # stores B^T
    C = wl.Operand(np.zeros(M * N, np.float32), 0, N, 1, 0)
    swapped, _ = oracle.product(wl.Operand(a_km.reshape(-1), 0, 1, M, 0),
                                wl.Operand(b_nk.reshape(-1), 0, 1, K, 0),
                                C, M, N, K, 1, 1.0, 0)
    a_copy = np.ascontiguousarray(a_km.T).reshape(-1)
    b_copy = np.ascontiguousarray(b_nk.T).reshape(-1)
    copied, _ = oracle.product(wl.Operand(a_copy, 0, K, 1, 0),
                               wl.Operand(b_copy, 0, N, 1, 0),
                               C, M, N, K, 1, 1.0, 0)
    assert np.array_equal(swapped, copied)


def test_alpha_power_of_two_scaling_exact():
    case = wl.make("c1", "real")
    base, _ = oracle.case_product(case)
    for j in (-3, 1, 5):
        case.alpha = 2.0 ** j
        scaled, _ = oracle.case_product(case)
        assert np.array_equal(scaled, base * 2.0 ** j)


def test_accumulate_minus_c0_equals_overwrite_integers():
    rng = np.random.default_rng(5)
    case = wl.random_strided(rng, 23, 11, 40, 2, "row", "col", values="int",
                             accumulate=1, alpha=0.125)
    acc, _ = oracle.case_product(case)
    case.accumulate = 0
    over, _ = oracle.case_product(case)
    c0 = case.C.view(case.batch, case.M, case.N).astype(np.float64)
    assert np.array_equal(acc - c0, over)


def test_batch_permutation_and_zero_batch_stride():
    rng = np.random.default_rng(6)
    M, K, N, batch = 9, 12, 10, 4
    a = rng.standard_normal(batch * M * K).astype(np.float32)
    b = rng.standard_normal(batch * K * N).astype(np.float32)
    C = wl.Operand(np.zeros(batch * M * N, np.float32), 0, N, 1, M * N)
    ref, _ = oracle.product(wl.Operand(a, 0, K, 1, M * K), wl.Operand(b, 0, N, 1, K * N),
                            C, M, N, K, batch, 1.0, 0)
    perm = [2, 0, 3, 1]
    ap = a.reshape(batch, -1)[perm].reshape(-1).copy()
    bp = b.reshape(batch, -1)[perm].reshape(-1).copy()
    refp, _ = oracle.product(wl.Operand(ap, 0, K, 1, M * K), wl.Operand(bp, 0, N, 1, K * N),
                             C, M, N, K, batch, 1.0, 0)
    assert np.array_equal(refp, ref[perm])
    # Batch stride 0 on A and B: every batch entry is the same product.
    ref0, _ = oracle.product(wl.Operand(a, 0, K, 1, 0), wl.Operand(b, 0, N, 1, 0),
                             C, M, N, K, batch, 1.0, 0)
    for i in range(1, batch):
        assert np.array_equal(ref0[i], ref0[0])
    assert np.array_equal(ref0[0], ref[0])


def test_all_ones_closed_form_and_softmax_rows():
    M, K, N = 8, 300, 5
    ones_a = np.ones(M * K, np.float32)
    ones_b = np.ones(K * N, np.float32)
    C = wl.Operand(np.zeros(M * N, np.float32), 0, N, 1, 0)
    ref, bound = oracle.product(wl.Operand(ones_a, 0, K, 1, 0),
                                wl.Operand(ones_b, 0, N, 1, 0), C, M, N, K, 1, 1.0, 0)
    assert np.all(ref == K) and np.all(bound == K)
    # Softmax rows of the attention-output workload times a ones column sum to 1.
    case = wl.make("c4", "real", batch=2, M=16, K=512, N=1)
    ones = wl.Operand(np.ones(512, np.float32), 0, 1, 0, 0)
    ref, _ = oracle.product(case.A, ones, wl.Operand(np.zeros(32, np.float32), 0, 1, 1, 16),
                            16, 1, 512, 2, 1.0, 0)
    assert np.all(np.abs(ref - 1.0) <= 1e-6)


def test_thread_count_and_reverse_order_do_not_change_results():
    case = wl.make("c2b", "real")
    r1, b1 = oracle.case_product(case, nthreads=1)
    r7, b7 = oracle.case_product(case, nthreads=7, reverse=True)
    assert np.array_equal(r1, r7) and np.array_equal(b1, b7)


def test_points_match_full_product():
    rng = np.random.default_rng(7)
    case = wl.random_strided(rng, 31, 27, 45, 3, "neg_row", "col", values="real",
                             accumulate=1, alpha=-0.5, bs_mode=("neg", "dense"))
    ref, bound = oracle.case_product(case)
    idx = np.stack([rng.integers(0, 3, 50), rng.integers(0, 31, 50),
                    rng.integers(0, 27, 50)], axis=1)
    pr, pb = oracle.case_points(case, idx)
    assert np.array_equal(pr, ref[idx[:, 0], idx[:, 1], idx[:, 2]])
    assert np.array_equal(pb, bound[idx[:, 0], idx[:, 1], idx[:, 2]])


def test_degenerate_sizes():
    a = np.arange(12, dtype=np.float32)
    c0 = np.arange(12, dtype=np.float32) - 5
    A = wl.Operand(a, 0, 3, 1, 0)
    # K = 0: overwrite gives zeros, accumulate gives C0 unchanged.
    ref, _ = oracle.product(A, A, wl.Operand(c0, 0, 4, 1, 0), 3, 4, 0, 1, 2.0, 0)
    assert np.all(ref == 0)
    ref, _ = oracle.product(A, A, wl.Operand(c0, 0, 4, 1, 0), 3, 4, 0, 1, 2.0, 1)
    assert np.array_equal(ref[0], c0.reshape(3, 4).astype(np.float64))
    # Empty M, N or batch: nothing to compute.
    for M, N, batch in ((0, 4, 1), (3, 0, 1), (3, 4, 0)):
        ref, _ = oracle.product(A, A, wl.Operand(c0, 0, 4, 1, 0), M, N, 2, batch, 1.0, 0)
        assert ref.size == 0


def test_golden_flop_convention():
    """The rate the pages print is 2*d0*d1*d2 / CPU time (printed rounded)."""
    rows = [l.split() for l in open(os.path.join(GOLDEN, "pytorch_demystified_gflops.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 21
    for d0, d1, d2, _wall, t, g in rows:
        decimals = len(t.split(".")[1]) if "." in t else 0
        half = 0.5 * 10.0 ** (-decimals)
        t_us = float(t)
        lo = wl.gflops_per_s(int(d0), int(d1), int(d2), 1, (t_us + half) * 1e-6)
        hi = wl.gflops_per_s(int(d0), int(d1), int(d2), 1, (t_us - half) * 1e-6)
        assert lo <= float(g) <= hi, (d0, d1, d2, t, g)


def test_spans_outside_storage_are_refused():
    a = np.zeros(6, np.float32)
    with pytest.raises(ValueError):
        oracle.product(wl.Operand(a, 0, 3, 1, 0), wl.Operand(a, 0, 3, 1, 0),
                       wl.Operand(a, 0, 3, 1, 0), 3, 3, 3, 1, 1.0, 0)


def test_backward_layouts_are_the_linear_layer_gradients():
    """Pins the backward workloads' layouts (G read transposed through swapped
    strides for dW; W read as stored for dX) to the definition of a gradient.
    For L(X, W) = sum(G * (X W^T)) with integer entries, L is linear in W and in
    X, so dL/dW[i, j] = L(W + E_ij) - L(W) and dL/dX[t, j] = L(X + E_tj) - L(X)
    exactly in int64, with no product routine involved ("PyTorch demystified
    3", section "Opt. 3 - Speed up matmul in the backward block through kernel
    fusion": dA = G B^T, dB = A^T G)."""
    rng = np.random.default_rng(11)
    T, d_in, d_out = 7, 5, 6
    X = rng.integers(-8, 9, size=(T, d_in)).astype(np.int64)
    W = rng.integers(-8, 9, size=(d_out, d_in)).astype(np.int64)
    G = rng.integers(-8, 9, size=(T, d_out)).astype(np.int64)

    def loss(X, W):
        total = 0
        for t in range(T):
            for o in range(d_out):
                y = 0
                for i in range(d_in):
                    y += int(X[t, i]) * int(W[o, i])
                total += int(G[t, o]) * y
        return total

    base = loss(X, W)
    want_dW = np.zeros((d_out, d_in), dtype=np.int64)
    for o in range(d_out):
        for i in range(d_in):
            W2 = W.copy(); W2[o, i] += 1
            want_dW[o, i] = loss(X, W2) - base
    want_dX = np.zeros((T, d_in), dtype=np.int64)
    for t in range(T):
        for i in range(d_in):
            X2 = X.copy(); X2[t, i] += 1
            want_dX[t, i] = loss(X2, W) - base

    f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32).reshape(-1)
    zeros = lambda n: np.zeros(n, dtype=np.float32)
    # dW = G^T X: A[m][k] = G[k][m] (rsA = 1, csA = d_out), B = X row-major.
    ref, _ = oracle.product(wl.Operand(f32(G), 0, 1, d_out, 0), wl.Operand(f32(X), 0, d_in, 1, 0),
                            wl.Operand(zeros(d_out * d_in), 0, d_in, 1, 0),
                            d_out, d_in, T, 1, 1.0, 0)
    assert np.array_equal(ref[0], want_dW.astype(np.float64))
    # dX = G W: A = G row-major, B[k][n] = W[k][n] read as stored.
    ref, _ = oracle.product(wl.Operand(f32(G), 0, d_out, 1, 0), wl.Operand(f32(W), 0, d_in, 1, 0),
                            wl.Operand(zeros(T * d_in), 0, d_in, 1, 0),
                            T, d_in, d_out, 1, 1.0, 0)
    assert np.array_equal(ref[0], want_dX.astype(np.float64))
    # The workloads' own dW layout, shrunk: same definition through make().
    case = wl.make("f1dwa", "int", M=6, N=5, K=7)
    Gs = case.A.storage.reshape(7, 6).astype(np.int64)    # stored [T, out]
    Xs = case.B.storage.reshape(7, 5).astype(np.int64)    # stored [T, in]
    C0 = case.C.storage.reshape(6, 5).astype(np.int64)
    ref, _ = oracle.case_product(case)
    want = C0 + np.array([[sum(int(Gs[t, o]) * int(Xs[t, i]) for t in range(7))
                           for i in range(5)] for o in range(6)])
    assert np.array_equal(ref[0], want.astype(np.float64))


# ---- fused epilogue: activations and the added operand D ----------------------

def run_activation_pins(lib=None):
    """Pins of the oracle's activations against facts independent of its
    formulas; returns the number of failed checks (0 for a correct oracle).
    Also used on mutated builds."""
    A = oracle.ACTIVATIONS
    act = lambda name, z: oracle.activation(A[name], np.asarray(z, dtype=np.float64), lib=lib)
    z = np.linspace(-9.0, 9.0, 3601)
    ln3 = np.log(3.0)
    checks = []
    # none and relu: exact identities.
    checks.append(np.array_equal(act("none", z), z))
    r = act("relu", z)
    checks.append(np.array_equal(r - act("relu", -z), z) and np.array_equal(r + act("relu", -z), np.abs(z)))
    # sigmoid: symmetric about 1/2, and 1/(1 + 1/3) at ln 3.
    s = act("sigmoid", z)
    checks.append(np.abs(s + act("sigmoid", -z) - 1.0).max() < 1e-15)
    checks.append(abs(act("sigmoid", [ln3])[0] - 0.75) < 1e-15 and act("sigmoid", [0.0])[0] == 0.5)
    # silu: odd part z/2, and (3/4) ln 3 at ln 3.
    checks.append(np.abs(act("silu", z) - act("silu", -z) - z).max() < 1e-13)
    checks.append(abs(act("silu", [ln3])[0] - 0.75 * ln3) < 1e-15)
    # gelu_erf: z * Phi(z), the standard normal CDF of scipy; Phi(1) = 0.841344746068543.
    from scipy.stats import norm
    ge = act("gelu_erf", z)
    checks.append(np.abs(ge - z * norm.cdf(z)).max() < 1e-14)
    checks.append(abs(act("gelu_erf", [1.0])[0] - 0.841344746068543) < 1e-15)
    checks.append(np.abs(ge - act("gelu_erf", -z) - z).max() < 1e-13)
    # gelu_tanh: odd part z/2; the tanh approximation of z * Phi(z) deviates from
    # it by 4.73e-4 at most (a wrong coefficient moves that by 2x or more).
    gt = act("gelu_tanh", z)
    checks.append(np.abs(gt - act("gelu_tanh", -z) - z).max() < 1e-13)
    zz = np.linspace(-8.0, 8.0, 160001)
    dev = np.abs(act("gelu_tanh", zz) - zz * norm.cdf(zz)).max()
    checks.append(4.6e-4 < dev < 4.8e-4)
    return sum(1 for c in checks if not c)


def test_activation_pins():
    assert run_activation_pins() == 0


def test_unknown_activation_is_refused():
    with pytest.raises(ValueError):
        oracle.activation(6, np.zeros(3))


def run_epilogue_pins(lib=None):
    """Integer A, B, C0 and D: z is exact and so is relu(z); the sampled-points
    variant (D added in C) reproduces the full fused product (D added here with
    numpy) for every activation; D broadcast over rows (a bias per column) and
    over batches.  Returns the number of failed checks."""
    rng = np.random.default_rng(23)
    bad = 0
    for acc, d_rs, d_bs in ((0, 0, 0), (1, 0, 1), (1, 1, 0)):
        M, N, K, batch = 19, 21, 33, 3
        case = wl.random_strided(rng, M, N, K, batch, "row", "col", values="int",
                                 accumulate=acc, alpha=0.5)
        dst = rng.integers(-8, 9, size=batch * M * N).astype(np.float32)
        D = wl.Operand(dst, 0, d_rs * N, 1, d_bs * M * N)
        out, z, bound = oracle.fused_product(case.A, case.B, case.C, M, N, K, batch,
                                             case.alpha, acc, D, oracle.ACTIVATIONS["relu"],
                                             lib=lib)
        eref, ebound = _int_expected(case)
        d = D.view(batch, M, N).astype(np.float64)
        bad += not (np.array_equal(z, eref + d) and np.array_equal(bound, ebound + np.abs(d)))
        bad += not np.array_equal(out, np.where(z > 0, z, 0.0))
        idx = np.stack([rng.integers(0, batch, 200), rng.integers(0, M, 200),
                        rng.integers(0, N, 200)], axis=1)
        sel = (idx[:, 0], idx[:, 1], idx[:, 2])
        for code in oracle.ACTIVATIONS.values():
            fo, fz, fb = oracle.fused_points(case.A, case.B, case.C, M, N, K, batch, case.alpha,
                                             acc, D, code, idx, lib=lib)
            full, fullz, fullb = oracle.fused_product(case.A, case.B, case.C, M, N, K, batch,
                                                      case.alpha, acc, D, code, lib=lib)
            bad += not (np.array_equal(fo, full[sel]) and np.array_equal(fz, fullz[sel]) and
                        np.array_equal(fb, fullb[sel]))
    return bad


def test_fused_epilogue_pins():
    assert run_epilogue_pins() == 0


# ---- fused attention ----------------------------------------------------------

def _attn(Qa, Ka, Va, alpha, causal=False, q_len=0, lib=None):
    """Oracle attention on dense arrays Q [b,M,D], K [b,N,D], V [b,N,Dv]."""
    b, M, D = Qa.shape
    N, Dv = Ka.shape[1], Va.shape[2]
    op = lambda a: wl.Operand(np.ascontiguousarray(a, dtype=np.float32).reshape(-1), 0,
                              a.shape[2], 1, a.shape[1] * a.shape[2])
    return oracle.attention(op(Qa), op(Ka), op(Va), M, N, D, Dv, b, alpha, causal, q_len, lib=lib)


def run_attention_pins(lib=None):
    """Pins of the attention oracle against facts that do not restate its
    formula; returns the number of failed checks (also used on mutated builds)."""
    rng = np.random.default_rng(31)
    attn = lambda *a, **k: _attn(*a, lib=lib, **k)
    bad = 0
    b, M, N, D = 2, 6, 9, 5
    K = rng.standard_normal((b, N, D)).astype(np.float32)
    V = rng.standard_normal((b, N, D)).astype(np.float32)
    # Zero queries: every score equal, so O is the mean of the kept value rows.
    O, W, _ = attn(np.zeros((b, M, D), np.float32), K, V, 0.5)
    bad += not np.allclose(O, np.broadcast_to(V.astype(np.float64).mean(axis=1, keepdims=True), O.shape),
                           rtol=0, atol=1e-12)
    O, _, _ = attn(np.zeros((b, M, D), np.float32), K, V, 0.5, causal=True, q_len=M)
    for m in range(M):
        kept = m + N - M + 1
        bad += not np.allclose(O[:, m], V[:, :kept].astype(np.float64).mean(axis=1), rtol=0, atol=1e-12)
    # Causal, q_len = N: the first query sees the first key only.
    Q = rng.standard_normal((b, N, D)).astype(np.float32)
    O, _, _ = attn(Q, K, V, 0.7, causal=True, q_len=N)
    bad += not np.array_equal(O[:, 0], V[:, 0].astype(np.float64))
    # One-hot queries and keys: score alpha on the diagonal, 0 elsewhere.
    Nh, a = 7, 3.0
    E = np.eye(Nh, dtype=np.float32)[None]
    Vh = rng.standard_normal((1, Nh, 4)).astype(np.float32).astype(np.float64)
    O, _, _ = attn(E, E, Vh, a)
    want = (np.exp(a) * Vh[0] + (Vh[0].sum(axis=0, keepdims=True) - Vh[0])) / (np.exp(a) + Nh - 1)
    bad += not np.allclose(O[0], want, rtol=0, atol=1e-12)
    # A per-row shift of every score (an extra dimension: K = 1, Q = c) changes nothing.
    c = rng.standard_normal((b, M, 1)).astype(np.float32) * 4
    Qr = rng.standard_normal((b, M, D)).astype(np.float32)
    O1, _, _ = attn(Qr, K, V, 0.5)
    O2, _, _ = attn(np.concatenate([Qr, c], 2), np.concatenate([K, np.ones((b, N, 1), np.float32)], 2), V, 0.5)
    bad += not np.allclose(O1, O2, rtol=0, atol=1e-12)
    # Keys and values permuted together (no mask): nothing changes.
    perm = rng.permutation(N)
    O3, _, _ = attn(Qr, K[:, perm], V[:, perm], 0.5)
    bad += not np.allclose(O1, O3, rtol=0, atol=1e-12)
    # Linear in V (integer values, so V1 + V2 is exact in fp32).
    V1 = rng.integers(-8, 9, size=(b, N, D)).astype(np.float32)
    V2 = rng.integers(-8, 9, size=(b, N, D)).astype(np.float32)
    Oa, _, _ = attn(Qr, K, V1, 0.5)
    Ob, _, _ = attn(Qr, K, V2, 0.5)
    Oc, _, _ = attn(Qr, K, V1 + V2, 0.5)
    bad += not np.allclose(Oc, Oa + Ob, rtol=0, atol=1e-12)
    # The tolerance weight dominates |O| and equals O when V >= 0.
    O6, W6, S6 = attn(Qr, K, V, 0.5)
    bad += not bool((W6 + 1e-15 >= np.abs(O6)).all())
    Op, Wp, _ = attn(Qr, K, np.abs(V), 0.5)
    bad += not np.allclose(Op, Wp, rtol=1e-14, atol=0)
    # Two steps through the product oracle and a numpy softmax.
    S = np.einsum("bmd,bnd->bmn", Qr.astype(np.float64), K.astype(np.float64)) * 0.5
    P = np.exp(S - S.max(axis=2, keepdims=True))
    P /= P.sum(axis=2, keepdims=True)
    bad += not np.allclose(O6, np.einsum("bmn,bne->bme", P, V.astype(np.float64)), rtol=0, atol=1e-12)
    bad += not np.allclose(S6, (np.abs(Qr).astype(np.float64) @ np.abs(K.astype(np.float64)).transpose(0, 2, 1)).max(axis=2) * 0.5,
                           rtol=1e-14, atol=0)
    # The head dimensions the kernels take (32, 64, 96, 128): zero queries give
    # the mean of the value rows; one-hot queries against one-hot keys give the
    # closed form above, with the remaining dimensions zero.
    for Dh in (32, 64, 96, 128):
        Kd = rng.standard_normal((1, 11, Dh)).astype(np.float32)
        Vd = rng.standard_normal((1, 11, Dh)).astype(np.float32)
        O, _, _ = attn(np.zeros((1, 3, Dh), np.float32), Kd, Vd, 1.0 / np.sqrt(Dh))
        bad += not np.allclose(O[0], np.broadcast_to(Vd[0].astype(np.float64).mean(axis=0), O[0].shape),
                               rtol=0, atol=1e-12)
        Eh = np.zeros((1, Nh, Dh), np.float32)
        Eh[0, np.arange(Nh), np.arange(Nh) * (Dh // Nh)] = 1.0
        Vh = rng.standard_normal((1, Nh, Dh)).astype(np.float32).astype(np.float64)
        O, _, _ = attn(Eh, Eh, Vh, a)
        want = (np.exp(a) * Vh[0] + (Vh[0].sum(axis=0, keepdims=True) - Vh[0])) / (np.exp(a) + Nh - 1)
        bad += not np.allclose(O[0], want, rtol=0, atol=1e-12)
    return bad


def test_attention_pins():
    assert run_attention_pins() == 0


def test_attention_strided_layouts_match_dense():
    """The 'mixed' layout (K read transposed, V and O column-major with a
    padded pitch, Q batches walked backwards) reads the same logical operands."""
    rng = np.random.default_rng(5)
    c = wl.random_attention(rng, 11, 13, 8, 3, "mixed", causal=1, q_len=11)
    Qd, Kd, Vd = (np.array(op.view(c.batch, r, cc)) for op, r, cc in
                  ((c.Q, c.M, c.D), (c.K, c.N, c.D), (c.V, c.N, c.Dv)))
    O, W, S = oracle.attention_case(c)
    O2, W2, S2 = _attn(Qd, Kd, Vd, c.alpha, True, 11)
    assert np.array_equal(O, O2) and np.array_equal(W, W2) and np.array_equal(S, S2)


# ---- paged key / value reads ----------------------------------------------------

def run_paged_pins(lib=None):
    """Pins of the paged-cache reader and of paged attention.  The caches come
    from the workload generator, which writes each token at the offset it
    counts up inside the block it takes from a shuffled free list (the
    scheduler's side of the page's layout); the oracle divides positions back
    into (block, offset) through the table.  Returns the number of failures."""
    rng = np.random.default_rng(41)
    bad = 0

    def gather(cache, table, s, h, n):
        try:
            return oracle.kv_gather(cache, table, s, h, n, lib=lib)
        except ValueError:            # a refusal where the pages' layout has the row
            return np.full((n, cache.shape[3]), np.nan, np.float32)

    for bsz, lens, heads, Dh in ((4, [1, 5, 16, 17, 40], 3, 8), (1, [3, 9], 2, 4),
                                 (64, [64, 2, 65], 2, 4), (5, [23, 24, 25], 4, 3)):
        Kc, Vc, table, seq_lens, K_ctx, V_ctx = wl.paged_cache(rng, lens, heads, Dh, bsz)
        for s, n in enumerate(lens):
            for h in range(heads):
                bad += not np.array_equal(gather(Kc, table, s, h, n), K_ctx[s, h, :n])
                bad += not np.array_equal(gather(Vc, table, s, h, n), V_ctx[s, h, :n])
        # No slot outside a sequence's tokens is ever read (they hold NaN).
        bad += not all(np.isfinite(gather(Kc, table, s, h, n)).all()
                       for s, n in enumerate(lens) for h in range(heads))
    # A block id outside the cache, or a position past the table, is refused.
    Kc, Vc, table, seq_lens, K_ctx, V_ctx = wl.paged_cache(rng, [9, 4], 1, 2, 4)
    t2 = table.copy()
    t2[0, 1] = Kc.shape[0]
    for tab, n in ((t2, 9), (table, 4 * table.shape[1] + 1)):
        try:
            oracle.kv_gather(Kc, tab, 0, 0, n, lib=lib)
            bad += 1
        except ValueError:
            pass
    # Paged attention equals the attention oracle on the contiguous context
    # of each (sequence, head), with causal positions taken from that
    # sequence's own length.
    case = wl.random_paged_attention(rng, [3, 30, 19], 2, 3, 2, 8, 4, causal=1)
    try:
        O, W, S = oracle.attention_paged(case.Q, case.K_cache, case.V_cache, case.block_table,
                                         case.seq_lens, case.M, case.alpha, True, case.q_len, lib=lib)
    except ValueError:
        return bad + 1
    Qd = np.array(case.Q.view(case.batch, case.M, case.D))
    for s, n in enumerate(case.seq_lens):
        for h in range(case.n_kv_heads):
            b = s * case.n_kv_heads + h
            O2, W2, S2 = _attn(Qd[b:b + 1], case.K_ctx[s:s + 1, h, :n], case.V_ctx[s:s + 1, h, :n],
                               case.alpha, True, case.q_len, lib=lib)
            bad += not (np.array_equal(O[b:b + 1], O2) and np.array_equal(W[b:b + 1], W2) and
                        np.array_equal(S[b:b + 1], S2))
    return bad


def test_paged_pins():
    assert run_paged_pins() == 0


def test_spectrogram_workload_is_the_windowed_dft():
    """f4spec's product, frames read as overlapping strided rows times the
    basis, equals numpy's real FFT of the Hann-windowed frames (a library
    routine of its own): real parts in the first 257 columns, imaginary
    parts in the next 257."""
    case = wl.make("f4spec", "real", batch=2, M=9)
    ref, _ = oracle.case_product(case)
    K, hop = case.K, case.A.rs
    L = case.A.bs
    sig = case.A.storage.reshape(case.batch, L).astype(np.float64)
    w = np.sin(np.pi * np.arange(K) / K) ** 2
    for b in range(case.batch):
        frames = np.stack([sig[b, t * hop: t * hop + K] for t in range(case.M)]) * w
        X = np.fft.rfft(frames, axis=1)
        got = ref[b]
        assert np.allclose(got[:, :257], X.real, rtol=0, atol=1e-4 * np.abs(X).max())
        assert np.allclose(got[:, 257:], X.imag, rtol=0, atol=1e-4 * np.abs(X).max())


def test_distance_workload_is_the_squared_distance():
    """f4dist's product (-2 X C^T onto |x|^2 + |c|^2) equals the brute-force
    squared Euclidean distance of every embedding to every codebook entry."""
    case = wl.make("f4dist", "int", M=23, N=17, K=31)
    ref, _ = oracle.case_product(case)
    X = case.A.storage.reshape(23, 31).astype(np.int64)
    Cb = case.B.storage.reshape(17, 31).astype(np.int64)
    want = ((X[:, None, :] - Cb[None, :, :]) ** 2).sum(axis=2)
    assert np.array_equal(ref[0], want.astype(np.float64))
