"""Seeded synthetic inputs for the strided batched product C <- alpha*A*B (+C).

This module is shared by the tests, the benchmark and the smoke check. It only
draws random storage and describes how each operand is laid over that storage
(pointer offset plus row / column / batch strides, in fp32 elements). It holds
none of the product's arithmetic: the oracle and the CUDA library each compute
the product on their own from these inputs.

The workloads restate the five cases of the strided-batched problem statement
(StaleyNET "GPU Implementation", section "The matrix product"; the linear-layer
and attention shapes of "rvllm CUDA path", section "Matmuls go to cuBLAS"):

  c1      one 64x48x32 product, row-major, overwrite
  c2a     MLP layer y = x W^T, x [256,784], W [512,784] read transposed via strides
  c2b     follow-on layer [256,512] . W2^T, W2 stored [10,512] (out, in)
  c3      128 attention score products Q[512,64] K^T, alpha = 1/8
  c3gqa   grouped-query variant: 4 Q heads stacked as 2048 rows against one K
  c4      128 products P[512,512] V[512,64] + C0 (accumulate)
  c5a     8192 x 960 -> 2560, W [2560,960] read transposed
  c5b     8192 x 2560 -> 960, W [960,2560] read transposed
  c5c     4096^3, row-major, accumulate
  c5d     4096^3, A and B both read transposed by swapped strides, accumulate

and the backward products of the two projection layers (dX = G W, dW = G^T X for
Y = X W^T; "PyTorch demystified 3", section "Opt. 3 - Speed up matmul in the
backward block through kernel fusion"), transposes read through strides:

  f1dxa   dX of c5a's layer: G [8192,2560] . W [2560,960] (W read as stored)
  f1dwa   dW of c5a's layer: G^T [2560,8192] . X [8192,960], accumulate into dW
  f1dxb   dX of c5b's layer: G [8192,960] . W [960,2560]
  f1dwb   dW of c5b's layer: G^T [960,8192] . X [8192,2560], accumulate into dW

and two more products the StaleyNET page routes through the kernel ("GPU
Implementation", section "The matrix product": the spectrogram and the
tokenizer's distances), in the plain reading given there no formula:

  f4spec  power-spectrum basis product of 64 clips of 16384 samples: frames of
          512 samples every 128 (overlapping rows of the signal, rsA = 128, no
          framing copy) times the windowed DFT basis [w cos | -w sin] (512 x 514)
  f4dist  squared distances of 8192 embeddings (256-d) to a 4096-entry codebook:
          -2 X C^T accumulated onto |x|^2 + |c|^2

Every workload also has an integer pass (values uniform in {-8..8}) in which
every partial sum is an exact fp32 integer.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import numpy as np

__all__ = ["Operand", "Case", "WORKLOADS", "BACKWARD", "make", "flops", "gflops_per_s",
           "alg_bytes", "SEEDS", "AttnCase", "ATTENTION", "make_attention", "random_attention",
           "PagedCase", "PAGED", "paged_cache", "random_paged_attention", "make_paged"]


@dataclasses.dataclass
class Operand:
    """One operand laid over a flat fp32 storage array.

    Element (b, i, j) of the logical [batch, rows, cols] operand lives at
    ``storage[offset + b*bs + i*rs + j*cs]``.
    """
    storage: np.ndarray          # 1-D float32, C-contiguous
    offset: int                  # element offset of (0, 0, 0)
    rs: int
    cs: int
    bs: int

    def view(self, batch: int, rows: int, cols: int) -> np.ndarray:
        """Strided numpy view of the logical [batch, rows, cols] operand (no copy).

        Used only by tests to materialise operands for library cross-checks.
        """
        base = self.storage[self.offset:]
        item = self.storage.itemsize
        return np.lib.stride_tricks.as_strided(
            base, shape=(batch, rows, cols),
            strides=(self.bs * item, self.rs * item, self.cs * item),
            writeable=False)


@dataclasses.dataclass
class Case:
    name: str
    A: Operand
    B: Operand
    C: Operand                   # C0 lives in C.storage when accumulate
    M: int
    N: int
    K: int
    batch: int
    alpha: float
    accumulate: int
    values: str                  # "real" or "int"
    note: str = ""

    @property
    def flops(self) -> int:
        return flops(self.M, self.N, self.K, self.batch)


def flops(M: int, N: int, K: int, batch: int = 1) -> int:
    """Multiply-adds counted as two operations, one pair per (b, m, n, k).

    This is the counting the pages' own GFLOP/s tables use (checked against the
    printed google-benchmark rows in the golden test)."""
    return 2 * int(M) * int(N) * int(K) * int(batch)


def gflops_per_s(M: int, N: int, K: int, batch: int, seconds: float) -> float:
    return flops(M, N, K, batch) / seconds / 1e9


def alg_bytes(case: "Case") -> int:
    """Algorithmic HBM bytes of one product: A and B read once, C written once,
    C0 read once when accumulating (fp32 elements; broadcast operands once)."""
    a_batches = 1 if case.A.bs == 0 else case.batch
    b_batches = 1 if case.B.bs == 0 else case.batch
    n = (a_batches * case.M * case.K + b_batches * case.K * case.N
         + case.batch * case.M * case.N * (2 if case.accumulate else 1))
    return 4 * n


# Seeds follow the order of the workload list: c1 = 0 (as the problem states),
# c2 = 1, c3 = 2, c4 = 3, c5 = 4.
SEEDS = {"c1": 0, "c2a": 1, "c2b": 1, "c3": 2, "c3gqa": 2, "c4": 3,
         "c5a": 4, "c5b": 4, "c5c": 4, "c5d": 4,
         "f1dxa": 5, "f1dwa": 5, "f1dxb": 5, "f1dwb": 5, "f4spec": 7, "f4dist": 7}
# Sub-stream per workload sharing a seed, so c2a and c2b draw different values.
_STREAM = {"c1": 0, "c2a": 0, "c2b": 1, "c3": 0, "c3gqa": 1, "c4": 0,
           "c5a": 0, "c5b": 1, "c5c": 2, "c5d": 2,
           "f1dxa": 0, "f1dwa": 1, "f1dxb": 2, "f1dwb": 3, "f4spec": 0, "f4dist": 1}

# Full-size shapes.  Keys that a caller may override to shrink a case for the
# oracle: batch, M, N, K (and heads/seqs for the attention cases).
FULL: Dict[str, Dict[str, int]] = {
    "c1": dict(batch=1, M=64, N=48, K=32),
    "c2a": dict(batch=1, M=256, N=512, K=784),
    "c2b": dict(batch=1, M=256, N=10, K=512),
    "c3": dict(batch=128, M=512, N=512, K=64),          # 8 sequences x 16 heads
    "c3gqa": dict(batch=32, M=2048, N=512, K=64),       # 8 seqs x 4 KV heads, 4 Q heads each
    "c4": dict(batch=128, M=512, N=64, K=512),
    "c5a": dict(batch=1, M=8192, N=2560, K=960),
    "c5b": dict(batch=1, M=8192, N=960, K=2560),
    "c5c": dict(batch=1, M=4096, N=4096, K=4096),
    "c5d": dict(batch=1, M=4096, N=4096, K=4096),
    "f1dxa": dict(batch=1, M=8192, N=960, K=2560),
    "f1dwa": dict(batch=1, M=2560, N=960, K=8192),
    "f1dxb": dict(batch=1, M=8192, N=2560, K=960),
    "f1dwb": dict(batch=1, M=960, N=2560, K=8192),
    # frames (16384 - 512) / 128 + 1 = 125 per clip; 257 bins x (cos, sin)
    "f4spec": dict(batch=64, M=125, N=514, K=512),
    "f4dist": dict(batch=1, M=8192, N=4096, K=256),
}
WORKLOADS = tuple(FULL)
BACKWARD = ("f1dxa", "f1dwa", "f1dxb", "f1dwb")


def _rng(name: str, values: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(
        [SEEDS[name], _STREAM[name], 0 if values == "real" else 1]))


def _flat(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).reshape(-1)


def _ints(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.integers(-8, 9, size=shape).astype(np.float32)


def _uniform(rng, lo, hi, shape):
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def _normal(rng, std, shape):
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std))


def _softmax_rows(logits: np.ndarray) -> np.ndarray:
    """Row-wise softmax, used only to shape the config-4 probability inputs."""
    z = logits.astype(np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def make(name: str, values: str = "real", **shape) -> Case:
    """Build workload ``name`` with ``values`` in {"real", "int"}.

    ``shape`` may override batch / M / N / K to obtain a smaller case of the
    same layout (for the oracle); strides follow the (possibly shrunk) sizes.
    """
    if name not in FULL:
        raise KeyError(name)
    if values not in ("real", "int"):
        raise ValueError(values)
    dims = dict(FULL[name])
    dims.update({k: int(v) for k, v in shape.items()})
    batch, M, N, K = dims["batch"], dims["M"], dims["N"], dims["K"]
    rng = _rng(name, values)
    is_int = values == "int"

    def draw(kind: str, shp, *args):
        if is_int:
            return _ints(rng, shp)
        if kind == "u":
            return _uniform(rng, args[0], args[1], shp)
        if kind == "n":
            return _normal(rng, args[0], shp)
        if kind == "softmax":
            return _softmax_rows(_normal(rng, args[0], shp))
        raise ValueError(kind)

    empty_c = lambda: np.zeros(batch * M * N, dtype=np.float32)

    if name == "c1":
        a = draw("u", (M, K), -1.0, 1.0)
        b = draw("u", (K, N), -1.0, 1.0)
        return Case(name, Operand(_flat(a), 0, K, 1, M * K),
                    Operand(_flat(b), 0, N, 1, K * N),
                    Operand(empty_c(), 0, N, 1, M * N),
                    M, N, K, batch, 1.0, 0, values,
                    "row-major A and B, overwrite")

    if name in ("c2a", "c2b"):
        x = draw("u", (M, K), 0.0, 1.0)
        w = draw("n", (N, K), 0.05)
        # y = x W^T: B[k][n] = W[n][k] -> rsB = 1, csB = K (W's row length).
        return Case(name, Operand(_flat(x), 0, K, 1, M * K),
                    Operand(_flat(w), 0, 1, K, N * K),
                    Operand(empty_c(), 0, N, 1, M * N),
                    M, N, K, batch, 1.0, 0, values,
                    "weights [out,in] read transposed by swapped strides")

    if name == "c3":
        # Q and K head-major, contiguous per (sequence, head): [batch, T, D].
        q = draw("n", (batch, M, K), 1.0)
        k = draw("n", (batch, N, K), 1.0)
        return Case(name, Operand(_flat(q), 0, K, 1, M * K),
                    Operand(_flat(k), 0, 1, K, N * K),
                    Operand(empty_c(), 0, N, 1, M * N),
                    M, N, K, batch, 0.125, 0, values,
                    "S = Q K^T / sqrt(64), K read transposed")

    if name == "c3gqa":
        # Q stored [seqs, kv_heads, 4 q heads, T, D]; the 4 Q heads of a group
        # are consecutive, so they read as M = 4*T rows with rsA = D.
        q = draw("n", (batch, M, K), 1.0)
        k = draw("n", (batch, N, K), 1.0)
        return Case(name, Operand(_flat(q), 0, K, 1, M * K),
                    Operand(_flat(k), 0, 1, K, N * K),
                    Operand(empty_c(), 0, N, 1, M * N),
                    M, N, K, batch, 0.125, 0, values,
                    "grouped-query: 4 Q heads stacked as rows against one K")

    if name == "c4":
        p = draw("softmax", (batch, M, K), 2.0)
        v = draw("n", (batch, K, N), 1.0)
        c0 = draw("n", (batch, M, N), 1.0)
        return Case(name, Operand(_flat(p), 0, K, 1, M * K),
                    Operand(_flat(v), 0, N, 1, K * N),
                    Operand(_flat(c0), 0, N, 1, M * N),
                    M, N, K, batch, 1.0, 1, values,
                    "O = P V + C0, P rows softmax of normal(0,2) logits")

    if name in ("c5a", "c5b"):
        act = draw("n", (M, K), 1.0)
        w = draw("n", (N, K), 0.02)
        return Case(name, Operand(_flat(act), 0, K, 1, M * K),
                    Operand(_flat(w), 0, 1, K, N * K),
                    Operand(empty_c(), 0, N, 1, M * N),
                    M, N, K, batch, 1.0, 0, values,
                    "projection, W [out,in] read transposed")

    if name in ("c5c", "c5d"):
        # The square workloads may be shrunk to a non-square box; storage
        # stays row-major in each operand's own stored shape.
        a = draw("n", (M, K), 1.0) if name == "c5c" else draw("n", (K, M), 1.0)
        b = draw("n", (K, N), 0.02) if name == "c5c" else draw("n", (N, K), 0.02)
        c0 = draw("n", (M, N), 1.0)
        if name == "c5c":
            A = Operand(_flat(a), 0, K, 1, M * K)
            B = Operand(_flat(b), 0, N, 1, K * N)
            note = "square, row-major, accumulate"
        else:
            # A stored row-major [K, M] and read transposed: rsA = 1, csA = M.
            A = Operand(_flat(a), 0, 1, M, M * K)
            B = Operand(_flat(b), 0, 1, K, K * N)
            note = "square, A and B read transposed by swapped strides, accumulate"
        return Case(name, A, B, Operand(_flat(c0), 0, N, 1, M * N),
                    M, N, K, batch, 1.0, 1, values, note)

    if name in ("f1dxa", "f1dxb"):
        # dX [T, in] = G [T, out] . W [out, in]: M = T, K = out, N = in.
        g = draw("n", (M, K), 1.0)
        w = draw("n", (K, N), 0.02)
        return Case(name, Operand(_flat(g), 0, K, 1, M * K),
                    Operand(_flat(w), 0, N, 1, K * N),
                    Operand(empty_c(), 0, N, 1, M * N),
                    M, N, K, batch, 1.0, 0, values,
                    "input gradient, W [out,in] read as stored (N-major)")

    if name in ("f1dwa", "f1dwb"):
        # dW [out, in] += G^T . X: M = out, K = T, N = in.  G is stored [T, out]
        # and read transposed: A[m][k] = G[k][m], rsA = 1, csA = out.
        g = draw("n", (K, M), 1.0)
        x = draw("n", (K, N), 1.0)
        c0 = draw("n", (M, N), 0.01)
        return Case(name, Operand(_flat(g), 0, 1, M, M * K),
                    Operand(_flat(x), 0, N, 1, K * N),
                    Operand(_flat(c0), 0, N, 1, M * N),
                    M, N, K, batch, 1.0, 1, values,
                    "weight gradient, G read transposed by swapped strides, accumulate")

    if name == "f4spec":
        # Signal of each clip: (M - 1) * hop + K samples; frame t = samples
        # [t*hop, t*hop + K): A[b, t, k] = signal[b*L + t*hop + k].
        hop = 128
        L = (M - 1) * hop + K
        sig = draw("n", (batch, L), 1.0)
        # The integer pass keeps the layout with an integer basis.
        basis = _ints(rng, (K, N)) if is_int else spectrogram_basis(K, N // 2)
        return Case(name, Operand(_flat(sig), 0, hop, 1, L),
                    Operand(_flat(basis), 0, N, 1, 0),
                    Operand(empty_c(), 0, N, 1, M * N),
                    M, N, K, batch, 1.0, 0, values,
                    "overlapping frames read by strides times a windowed DFT basis")

    if name == "f4dist":
        x = draw("n", (M, K), 1.0)
        c = draw("n", (N, K), 1.0)
        # C0 = |x_m|^2 + |c_n|^2, computed in float64 and rounded once.
        x64, c64 = x.astype(np.float64), c.astype(np.float64)
        c0 = ((x64 * x64).sum(1)[:, None] + (c64 * c64).sum(1)[None, :]).astype(np.float32)
        return Case(name, Operand(_flat(x), 0, K, 1, M * K),
                    Operand(_flat(c), 0, 1, K, N * K),
                    Operand(_flat(c0), 0, N, 1, M * N),
                    M, N, K, batch, -2.0, 1, values,
                    "squared distances: -2 X C^T accumulated onto |x|^2 + |c|^2")

    raise AssertionError(name)


def spectrogram_basis(K: int, F: int) -> np.ndarray:
    """[K, 2F] basis of the windowed DFT: column f is w[k] cos(2 pi f k / K),
    column F + f is -w[k] sin(2 pi f k / K), with the periodic Hann window
    w[k] = sin^2(pi k / K).  Frames times this basis give the real and
    imaginary parts of the first F bins of the windowed frames' DFT."""
    k = np.arange(K, dtype=np.float64)[:, None]
    f = np.arange(F, dtype=np.float64)[None, :]
    w = np.sin(np.pi * k / K) ** 2
    ang = 2.0 * np.pi * f * k / K
    return np.concatenate([w * np.cos(ang), -w * np.sin(ang)], axis=1).astype(np.float32)


def small_shape(name: str) -> Dict[str, int]:
    """A reduced size of each workload that the CPU oracle computes in about a
    second while still spanning several 128x128 tiles and a ragged tail."""
    return {
        "c1": dict(FULL["c1"]),
        "c2a": dict(FULL["c2a"]),
        "c2b": dict(FULL["c2b"]),
        "c3": dict(batch=3, M=512, N=512, K=64),
        "c3gqa": dict(batch=2, M=2048, N=512, K=64),
        "c4": dict(batch=3, M=512, N=64, K=512),
        "c5a": dict(batch=1, M=300, N=2560, K=960),
        "c5b": dict(batch=1, M=300, N=960, K=2560),
        "c5c": dict(batch=1, M=260, N=1028, K=1024),
        "c5d": dict(batch=1, M=260, N=1028, K=1024),
        "f1dxa": dict(batch=1, M=300, N=960, K=2560),
        "f1dwa": dict(batch=1, M=260, N=300, K=2052),
        "f1dxb": dict(batch=1, M=300, N=1028, K=960),
        "f1dwb": dict(batch=1, M=300, N=260, K=2052),
        "f4spec": dict(batch=3, M=41, N=514, K=512),
        "f4dist": dict(batch=1, M=300, N=260, K=256),
    }[name]


def random_strided(rng: np.random.Generator, M: int, N: int, K: int, batch: int,
                   a_layout: str, b_layout: str, c_layout: str = "row",
                   bs_mode: Tuple[str, str] = ("dense", "dense"),
                   values: str = "int", accumulate: int = 0, alpha: float = 1.0,
                   pad: int = 0) -> Case:
    """Small case with a chosen layout per operand.

    Layouts: "row" (unit column stride), "col" (unit row stride), "neg_row"
    (row-major but rows walked backwards: negative row stride), "gap" (row-major
    with a padded row pitch), "bcast_row" (row stride 0: every row is the same
    memory), "row16" / "col16" (row- / column-major with the pitch rounded up
    to a multiple of 4 elements, i.e. 16 bytes). ``bs_mode`` per A/B: "dense",
    "zero" (batch stride 0, one shared matrix), "neg" (batches walked
    backwards).
    """
    def up4(x):
        return (x + 3) // 4 * 4

    def lay(rows, cols, layout, bsm):
        if layout in ("row", "neg_row", "gap", "row16"):
            rs = cols + (3 if layout == "gap" else 0) + pad
            if layout == "row16":
                rs = up4(rs)
            cs = 1
            span = rows * rs
        elif layout in ("col", "col16"):
            rs, cs = 1, rows + pad
            if layout == "col16":
                cs = up4(cs)
            span = cols * cs
        elif layout == "bcast_row":
            rs, cs = 0, 1
            span = cols
        else:
            raise ValueError(layout)
        nb = 1 if bsm == "zero" else batch
        bs = 0 if bsm == "zero" else span
        total = max(1, nb * span)
        if values == "int":
            st = rng.integers(-8, 9, size=total).astype(np.float32)
        else:
            st = rng.uniform(-1, 1, size=total).astype(np.float32)
        off = 0
        if layout == "neg_row":
            off += (rows - 1) * rs
            rs = -rs
        if bsm == "neg":
            off += (nb - 1) * bs
            bs = -bs
        return Operand(st, off, rs, cs, bs)

    A = lay(M, K, a_layout, bs_mode[0])
    B = lay(K, N, b_layout, bs_mode[1])
    if c_layout == "row":
        C = Operand(np.zeros(max(1, batch * M * N), np.float32), 0, N, 1, M * N)
    elif c_layout == "col":
        C = Operand(np.zeros(max(1, batch * M * N), np.float32), 0, 1, M, M * N)
    else:
        raise ValueError(c_layout)
    if accumulate:
        if values == "int":
            C.storage[:] = rng.integers(-8, 9, size=C.storage.size)
        else:
            C.storage[:] = rng.uniform(-1, 1, size=C.storage.size)
    return Case(f"rand_{a_layout}_{b_layout}_{c_layout}", A, B, C, M, N, K, batch,
                alpha, accumulate, values)


# ---- fused attention ---------------------------------------------------------
# O = softmax(alpha * Q K^T, causal optional) V for a batch of (sequence, head)
# problems: the scores of c3 and the probabilities of c4 computed in one pass
# ("rvllm CUDA path", section "What's basic about it": scores, softmax and
# probs @ V as three steps with the scores in global memory is the thing a
# fused kernel avoids).

@dataclasses.dataclass
class AttnCase:
    name: str
    Q: Operand          # [batch, M, D]
    K: Operand          # [batch, N, D]
    V: Operand          # [batch, N, Dv]
    O: Operand          # [batch, M, Dv] (output; storage is its initial content)
    M: int
    N: int
    D: int
    Dv: int
    batch: int
    alpha: float
    causal: int
    q_len: int          # rows per head for the causal position (M for one head)

    @property
    def flops(self) -> int:
        """2*M*N*D for the scores plus 2*M*N*Dv for probs @ V (the products'
        convention), counting every key even where the causal mask drops it."""
        return 2 * self.batch * self.M * self.N * (self.D + self.Dv)


ATTENTION = {
    # name: (batch, M, N, D, causal, q_len); alpha = 1/sqrt(D)
    "f2": (128, 512, 512, 64, 0, 512),          # the c3 / c4 problems: 8 sequences x 16 heads
    "f2causal": (128, 512, 512, 64, 1, 512),    # the same, causal
    "f2gqa": (32, 2048, 512, 64, 1, 512),       # 4 Q heads stacked as rows per KV head, causal
}


def make_attention(name: str, **shape) -> AttnCase:
    """Head-major Q, K, V [batch, T, D] as in c3; values N(0,1) (seed 6)."""
    batch, M, N, D, causal, q_len = ATTENTION[name]
    dims = dict(batch=batch, M=M, N=N, D=D, q_len=q_len)
    dims.update({k: int(v) for k, v in shape.items()})
    batch, M, N, D, q_len = dims["batch"], dims["M"], dims["N"], dims["D"], dims["q_len"]
    rng = np.random.Generator(np.random.PCG64([6, list(ATTENTION).index(name), 0]))
    q = _normal(rng, 1.0, (batch, M, D))
    k = _normal(rng, 1.0, (batch, N, D))
    v = _normal(rng, 1.0, (batch, N, D))
    return AttnCase(name, Operand(_flat(q), 0, D, 1, M * D), Operand(_flat(k), 0, D, 1, N * D),
                    Operand(_flat(v), 0, D, 1, N * D),
                    Operand(np.zeros(batch * M * D, dtype=np.float32), 0, D, 1, M * D),
                    M, N, D, D, batch, 1.0 / float(np.sqrt(D)), causal, q_len)


def random_attention(rng: np.random.Generator, M: int, N: int, D: int, batch: int,
                     layout: str = "row", causal: int = 0, q_len: int = 0,
                     alpha: float = 0.125, scale: float = 1.0) -> AttnCase:
    """A small attention case.  layout "row": every operand [batch, rows, D]
    row-major; "mixed": K stored [batch, D, N] and read transposed, V
    column-major with a padded pitch, O column-major, batches of Q walked
    backwards."""
    q = (rng.standard_normal(batch * M * D) * scale).astype(np.float32)
    k = (rng.standard_normal(batch * N * D) * scale).astype(np.float32)
    q_len = q_len or M
    if layout == "row":
        Q = Operand(q, 0, D, 1, M * D)
        K = Operand(k, 0, D, 1, N * D)
        V = Operand(rng.standard_normal(batch * N * D).astype(np.float32), 0, D, 1, N * D)
        O = Operand(np.zeros(batch * M * D, dtype=np.float32), 0, D, 1, M * D)
    elif layout == "mixed":
        Q = Operand(q, (batch - 1) * M * D, D, 1, -M * D)
        K = Operand(k, 0, 1, N, N * D)                  # K[b,n,d] at b*N*D + d*N + n
        pitch = N + 3
        V = Operand(rng.standard_normal(batch * D * pitch).astype(np.float32), 0, 1, pitch, D * pitch)
        O = Operand(np.zeros(batch * M * D, dtype=np.float32), 0, 1, M, M * D)
    else:
        raise ValueError(layout)
    return AttnCase(f"attn_{layout}_{M}x{N}x{D}", Q, K, V, O, M, N, D, D, batch, alpha,
                    int(bool(causal)), q_len)


# ---- paged key / value cache ---------------------------------------------------
# "rvllm CUDA path", section "The kernels": the cache is one buffer
# [num_blocks, block_size, n_kv_heads, head_dim]; each new token's K and V go
# to a block id and an offset handed out by the cache scheduler, and a
# sequence's block table lists its blocks in order.  The generator below plays
# the scheduler: sequences append one token per step (a batched decode loop),
# each takes the next block of a shuffled free list when its current block is
# full, and the token is written at (current block, next free offset).  It
# counts offsets up instead of dividing positions, so it is an independent
# statement of the layout the readers (oracle and kernels) divide back out.

@dataclasses.dataclass
class PagedCase:
    name: str
    Q: Operand                 # [n_seqs * n_kv_heads, M, D]; entry b = seq * n_kv_heads + head
    O: Operand                 # [n_seqs * n_kv_heads, M, D] (output)
    K_cache: np.ndarray        # float32 [num_blocks, block_size, n_kv_heads, D]; unused slots NaN
    V_cache: np.ndarray
    block_table: np.ndarray    # int32 [n_seqs, max_blocks]; entries past a sequence's blocks -1
    seq_lens: np.ndarray       # int32 [n_seqs]
    K_ctx: np.ndarray          # float32 [n_seqs, n_kv_heads, N, D]: the keys appended, in order
    V_ctx: np.ndarray          #   (positions past a sequence's length are zero)
    M: int
    N: int                     # longest context
    D: int
    n_kv_heads: int
    block_size: int
    alpha: float
    causal: int
    q_len: int

    @property
    def n_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def batch(self) -> int:
        return self.n_seqs * self.n_kv_heads

    @property
    def keys(self) -> int:
        """Keys read over the batch: every head of every context position."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.n_kv_heads

    @property
    def flops(self) -> int:
        """2*M*len*(D + Dv) per entry, every key counted."""
        return 2 * self.M * self.keys * 2 * self.D

    @property
    def alg_bytes(self) -> int:
        """K and V rows of every context position read once, Q read and O
        written once, the table and lengths read once."""
        return (self.keys * 2 * self.D * 4 + 2 * self.batch * self.M * self.D * 4 +
                self.block_table.size * 4 + self.seq_lens.size * 4)


def paged_cache(rng: np.random.Generator, lens, n_kv_heads: int, D: int, block_size: int,
                spare_blocks: int = 3, scale: float = 1.0):
    """A paged cache holding, for each sequence s, lens[s] tokens of random K
    and V.  Returns (K_cache, V_cache, block_table, seq_lens, K_ctx, V_ctx)."""
    lens = np.asarray(lens, dtype=np.int64)
    n_seqs, N = len(lens), int(lens.max())
    need = np.zeros(n_seqs, dtype=np.int64)
    for s in range(n_seqs):          # blocks each sequence will fill, by counting
        c = 0
        while c * block_size < lens[s]:
            c += 1
        need[s] = c
    num_blocks = int(need.sum()) + spare_blocks
    max_blocks = int(need.max()) + 1
    K_ctx = np.zeros((n_seqs, n_kv_heads, N, D), dtype=np.float32)
    V_ctx = np.zeros((n_seqs, n_kv_heads, N, D), dtype=np.float32)
    for s in range(n_seqs):
        K_ctx[s, :, :lens[s]] = _normal(rng, scale, (n_kv_heads, int(lens[s]), D))
        V_ctx[s, :, :lens[s]] = _normal(rng, 1.0, (n_kv_heads, int(lens[s]), D))
    K_cache = np.full((num_blocks, block_size, n_kv_heads, D), np.nan, dtype=np.float32)
    V_cache = np.full((num_blocks, block_size, n_kv_heads, D), np.nan, dtype=np.float32)
    table = np.full((n_seqs, max_blocks), -1, dtype=np.int32)
    free = list(rng.permutation(num_blocks))
    cur_block = np.full(n_seqs, -1, dtype=np.int64)
    cur_off = np.full(n_seqs, block_size, dtype=np.int64)   # "full": take a block first
    n_blocks = np.zeros(n_seqs, dtype=np.int64)
    for t in range(N):
        active = np.nonzero(lens > t)[0]
        for s in active[cur_off[active] == block_size]:
            cur_block[s] = free.pop(0)
            cur_off[s] = 0
            table[s, n_blocks[s]] = cur_block[s]
            n_blocks[s] += 1
        K_cache[cur_block[active], cur_off[active]] = K_ctx[active, :, t]
        V_cache[cur_block[active], cur_off[active]] = V_ctx[active, :, t]
        cur_off[active] += 1
    return K_cache, V_cache, table, lens.astype(np.int32), K_ctx, V_ctx


def random_paged_attention(rng: np.random.Generator, lens, n_kv_heads: int, group: int,
                           q_len: int, D: int, block_size: int, causal: int = 1,
                           alpha: Optional[float] = None, scale: float = 1.0,
                           name: str = "paged") -> PagedCase:
    """Attention of M = group * q_len query rows per (sequence, kv head)
    (grouped-query heads stacked as rows) over a paged cache of the given
    context lengths."""
    Kc, Vc, table, seq_lens, K_ctx, V_ctx = paged_cache(rng, lens, n_kv_heads, D, block_size,
                                                        scale=scale)
    n_seqs = len(seq_lens)
    M = group * q_len
    batch = n_seqs * n_kv_heads
    q = _normal(rng, 1.0, (batch, M, D))
    return PagedCase(name, Operand(_flat(q), 0, D, 1, M * D),
                     Operand(np.zeros(batch * M * D, dtype=np.float32), 0, D, 1, M * D),
                     Kc, Vc, table, seq_lens, K_ctx, V_ctx, M, int(seq_lens.max()), D, n_kv_heads,
                     block_size, 1.0 / float(np.sqrt(D)) if alpha is None else alpha,
                     int(bool(causal)), q_len)


PAGED = {
    # name: (n_seqs, n_kv_heads, group, q_len, D, block_size, context lengths)
    # A batched decode step: 32 sequences (the pages' largest batch), 8 KV heads
    # with 4 query heads each, head dimension 64, 16-token blocks, contexts
    # drawn uniformly from 1024..4096 tokens.
    "f2paged": (32, 8, 4, 1, 64, 16, (1024, 4096)),
}


def make_paged(name: str) -> PagedCase:
    n_seqs, heads, group, q_len, D, bsz, (lo, hi) = PAGED[name]
    rng = np.random.Generator(np.random.PCG64([7, list(PAGED).index(name), 0]))
    lens = rng.integers(lo, hi + 1, size=n_seqs)
    return random_paged_attention(rng, lens, heads, group, q_len, D, bsz, causal=1, name=name)
