"""CPU oracle for the strided batched product C <- alpha*A*B (+C0).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg are the only callers.  The CUDA library never imports or calls
anything here, and nothing here imports the CUDA library.

The arithmetic lives in ``sbgemm_ref.c`` (plain C, fp64 accumulation); this
module builds it with gcc and marshals numpy arrays to it.  Operands are passed
as objects with ``storage`` (1-D float32 numpy array), ``offset``, ``rs``,
``cs`` and ``bs`` attributes: element (b, i, j) is
``storage[offset + b*bs + i*rs + j*cs]``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
import types

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sbgemm_ref.c")
_LIB_PATH = os.path.join(_HERE, "libsbgemm_ref.so")
# A build with AddressSanitizer and UndefinedBehaviorSanitizer, loaded instead
# of the plain one when SBGEMM_ORACLE_SANITIZE=1 (the process must then start
# with the sanitizer runtimes preloaded, as tests/test_oracle_sanitized.py
# arranges).
_SAN_LIB_PATH = os.path.join(_HERE, "libsbgemm_ref_san.so")
SANITIZE_FLAGS = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all",
                  "-fno-omit-frame-pointer", "-g"]
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_fp = ctypes.c_void_p


def build(force: bool = False, src: str = _SRC, out: str | None = None,
          sanitize: bool = False) -> str:
    """Compile the oracle with gcc.  Contraction of a*b+c into fused
    multiply-adds is switched off so the fp64 arithmetic is the same on every
    host architecture.  ``sanitize`` adds AddressSanitizer and
    UndefinedBehaviorSanitizer (any report aborts the process)."""
    if out is None:
        out = _SAN_LIB_PATH if sanitize else _LIB_PATH
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        "-ffp-contract=off", "-fno-fast-math"] +
                       (SANITIZE_FLAGS if sanitize else []) + ["-o", tmp, src, "-lm"],
                       check=True)
        os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.sbgemm_ref.restype = ctypes.c_int
    lib.sbgemm_ref.argtypes = [
        _fp, _i64, _i64, _i64, _fp, _i64, _i64, _i64, _fp, _i64, _i64, _i64,
        _i64, _i64, _i64, _i64, ctypes.c_float, ctypes.c_int,
        _fp, _fp, ctypes.c_int, ctypes.c_int]
    lib.sbgemm_ref_points.restype = ctypes.c_int
    lib.sbgemm_ref_points.argtypes = [
        _fp, _i64, _i64, _i64, _fp, _i64, _i64, _i64, _fp, _i64, _i64, _i64,
        _i64, _i64, _i64, _i64, ctypes.c_float, ctypes.c_int,
        _fp, _i64, _fp, _fp]
    lib.sbgemm_ref_activation.restype = ctypes.c_int
    lib.sbgemm_ref_activation.argtypes = [ctypes.c_int, _fp, _fp, _i64]
    lib.sbgemm_ref_epilogue_points.restype = ctypes.c_int
    lib.sbgemm_ref_epilogue_points.argtypes = [_fp, _i64, _i64, _i64, ctypes.c_int,
                                               _fp, _i64, _fp, _fp, _fp]
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library.  ``path`` selects
    another build of the same source, e.g. a mutated copy in a test."""
    global _lib
    if path is not None:
        return _bind(path)
    with _lock:
        if _lib is None:
            san = os.environ.get("SBGEMM_ORACLE_SANITIZE") == "1"
            _lib = _bind(build(sanitize=san))
        return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _span_ok(op, batch, rows, cols) -> bool:
    """Every element the strides can reach lies inside the storage."""
    if batch == 0 or rows == 0 or cols == 0:
        return True
    lo = hi = op.offset
    for stride, extent in ((op.bs, batch), (op.rs, rows), (op.cs, cols)):
        d = stride * (extent - 1)
        lo, hi = (lo + d, hi) if d < 0 else (lo, hi + d)
    return lo >= 0 and hi < op.storage.size


def _ptr(op):
    st = op.storage
    assert st.dtype == np.float32 and st.flags.c_contiguous and st.ndim == 1
    return st.ctypes.data + 4 * int(op.offset)


def _check(A, B, C, M, N, K, batch, accumulate):
    if not _span_ok(A, batch, M, K):
        raise ValueError("oracle: A strides reach outside its storage")
    if not _span_ok(B, batch, K, N):
        raise ValueError("oracle: B strides reach outside its storage")
    if accumulate and not _span_ok(C, batch, M, N):
        raise ValueError("oracle: C strides reach outside its storage")


def product(A, B, C, M, N, K, batch, alpha, accumulate, nthreads=None,
            reverse=False, lib=None):
    """Full product.  Returns (ref, bound), float64 arrays of shape [batch, M, N]."""
    _check(A, B, C, M, N, K, batch, accumulate)
    lib = lib or load()
    ref = np.zeros((batch, M, N), dtype=np.float64)
    bound = np.zeros((batch, M, N), dtype=np.float64)
    rc = lib.sbgemm_ref(_ptr(A), A.rs, A.cs, A.bs, _ptr(B), B.rs, B.cs, B.bs,
                        _ptr(C), C.rs, C.cs, C.bs, M, N, K, batch,
                        float(alpha), int(accumulate),
                        ref.ctypes.data, bound.ctypes.data,
                        int(nthreads or default_threads()), int(bool(reverse)))
    if rc != 0:
        raise RuntimeError(f"oracle sbgemm_ref failed with {rc}")
    return ref, bound


def product_points(A, B, C, M, N, K, batch, alpha, accumulate, idx, lib=None):
    """The product at selected outputs.  ``idx`` is an int64 array [P, 3] of
    (b, m, n).  Returns (ref, bound), float64 arrays of length P."""
    _check(A, B, C, M, N, K, batch, accumulate)
    lib = lib or load()
    idx = np.ascontiguousarray(idx, dtype=np.int64).reshape(-1, 3)
    P = idx.shape[0]
    ref = np.zeros(P, dtype=np.float64)
    bound = np.zeros(P, dtype=np.float64)
    rc = lib.sbgemm_ref_points(_ptr(A), A.rs, A.cs, A.bs, _ptr(B), B.rs, B.cs, B.bs,
                               _ptr(C), C.rs, C.cs, C.bs, M, N, K, batch,
                               float(alpha), int(accumulate),
                               idx.ctypes.data, P, ref.ctypes.data, bound.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle sbgemm_ref_points failed with {rc}")
    return ref, bound


def case_product(case, **kw):
    """Full product of a workloads.Case."""
    return product(case.A, case.B, case.C, case.M, case.N, case.K, case.batch,
                   case.alpha, case.accumulate, **kw)


def case_points(case, idx, **kw):
    return product_points(case.A, case.B, case.C, case.M, case.N, case.K,
                          case.batch, case.alpha, case.accumulate, idx, **kw)


# ---- fused epilogue: out = act(alpha*A*B (+C0) + D) ------------------------------
# Activation codes of sbgemm_ref.c: 0 none, 1 relu, 2 sigmoid, 3 silu,
# 4 gelu_tanh, 5 gelu_erf.
ACTIVATIONS = {"none": 0, "relu": 1, "sigmoid": 2, "silu": 3, "gelu_tanh": 4, "gelu_erf": 5}


def activation(act, z, lib=None):
    """act(z) in fp64, elementwise (sbgemm_ref_activation)."""
    lib = lib or load()
    z = np.ascontiguousarray(z, dtype=np.float64)
    out = np.empty_like(z)
    if lib.sbgemm_ref_activation(int(act), z.ctypes.data, out.ctypes.data, z.size) != 0:
        raise ValueError(f"oracle: unknown activation {act}")
    return out


def fused_product(A, B, C, M, N, K, batch, alpha, accumulate, D, act, lib=None, **kw):
    """Full fused product.  D (an operand, or None) is added to the product and
    act applied: returns (out, z, bound) with z the pre-activation value and
    bound its error scale |alpha|sum|a||b| + |C0| + |D|."""
    z, bound = product(A, B, C, M, N, K, batch, alpha, accumulate, lib=lib, **kw)
    if D is not None:
        if not _span_ok(D, batch, M, N):
            raise ValueError("oracle: D strides reach outside its storage")
        b, m, n = np.meshgrid(np.arange(batch), np.arange(M), np.arange(N), indexing="ij")
        d = D.storage[D.offset + b * D.bs + m * D.rs + n * D.cs].astype(np.float64)
        z = z + d
        bound = bound + np.abs(d)
    return activation(act, z, lib=lib), z, bound


def fused_points(A, B, C, M, N, K, batch, alpha, accumulate, D, act, idx, lib=None):
    """The fused product at selected outputs (idx [P, 3] of (b, m, n))."""
    lib = lib or load()
    idx = np.ascontiguousarray(idx, dtype=np.int64).reshape(-1, 3)
    z, bound = product_points(A, B, C, M, N, K, batch, alpha, accumulate, idx, lib=lib)
    out = np.empty_like(z)
    if D is not None and not _span_ok(D, batch, M, N):
        raise ValueError("oracle: D strides reach outside its storage")
    rc = lib.sbgemm_ref_epilogue_points(_ptr(D) if D is not None else None,
                                        D.rs if D is not None else 0, D.cs if D is not None else 0,
                                        D.bs if D is not None else 0, int(act),
                                        idx.ctypes.data, idx.shape[0], z.ctypes.data,
                                        bound.ctypes.data, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle: unknown activation {act}")
    return out, z, bound


# ---- fused attention: O = softmax(alpha * Q K^T [causal]) V ----------------------

def attention(Q, K, V, M, N, D, Dv, batch, alpha, causal=False, q_len=0, lib=None):
    """The attention oracle (sbgemm_ref_attention).  Q, K, V are operands
    (storage, offset, rs, cs, bs): Q[b,m,d], K[b,n,d], V[b,n,e].  Returns (O,
    weight, smag): O and weight = sum_n P|V| of shape [batch, M, Dv], and smag
    [batch, M], the largest |alpha| * sum_d |q k| over the kept keys."""
    lib = lib or load()
    if not hasattr(lib, "_attn_bound"):
        lib.sbgemm_ref_attention.restype = ctypes.c_int
        lib.sbgemm_ref_attention.argtypes = [
            _fp, _i64, _i64, _i64, _fp, _i64, _i64, _i64, _fp, _i64, _i64, _i64,
            _i64, _i64, _i64, _i64, _i64, ctypes.c_float, ctypes.c_int, _i64, _fp, _fp, _fp]
        lib._attn_bound = True
    q_len = int(q_len) if q_len else M
    if causal and not (0 < q_len <= N):
        raise ValueError("oracle: causal attention needs 0 < q_len <= N")
    for op, rows, cols, name in ((Q, M, D, "Q"), (K, N, D, "K"), (V, N, Dv, "V")):
        if not _span_ok(op, batch, rows, cols):
            raise ValueError(f"oracle: {name} strides reach outside its storage")
    O = np.zeros((batch, M, Dv), dtype=np.float64)
    W = np.zeros((batch, M, Dv), dtype=np.float64)
    S = np.zeros((batch, M), dtype=np.float64)
    rc = lib.sbgemm_ref_attention(_ptr(Q), Q.rs, Q.cs, Q.bs, _ptr(K), K.rs, K.cs, K.bs,
                                  _ptr(V), V.rs, V.cs, V.bs, M, N, D, Dv, batch,
                                  float(alpha), int(bool(causal)), q_len,
                                  O.ctypes.data, W.ctypes.data, S.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle sbgemm_ref_attention failed with {rc}")
    return O, W, S


def attention_case(case, lib=None):
    return attention(case.Q, case.K, case.V, case.M, case.N, case.D, case.Dv, case.batch,
                     case.alpha, case.causal, case.q_len, lib=lib)


def kv_gather(cache, block_table, seq, head, length, lib=None):
    """Rows 0..length-1 of one (sequence, head) of a paged cache, gathered into
    a contiguous [length, head_dim] float32 array (sbgemm_ref_kv_gather).
    ``cache`` is float32 [num_blocks, block_size, n_kv_heads, head_dim] and
    ``block_table`` int32 [n_seqs, max_blocks]."""
    lib = lib or load()
    if not hasattr(lib, "_kvg_bound"):
        lib.sbgemm_ref_kv_gather.restype = ctypes.c_int
        lib.sbgemm_ref_kv_gather.argtypes = [_fp, _i64, _i64, _i64, _i64, _fp, _i64,
                                             _i64, _i64, _i64, _fp]
        lib._kvg_bound = True
    cache = np.ascontiguousarray(cache, dtype=np.float32)
    table = np.ascontiguousarray(block_table, dtype=np.int32)
    if cache.ndim != 4 or table.ndim != 2 or not 0 <= seq < table.shape[0]:
        raise ValueError("oracle: kv_gather needs a 4-d cache and a 2-d block table")
    nb, bsz, heads, hd = cache.shape
    out = np.empty((int(length), hd), dtype=np.float32)
    rc = lib.sbgemm_ref_kv_gather(cache.ctypes.data, nb, bsz, heads, hd, table.ctypes.data,
                                  table.shape[1], int(seq), int(head), int(length),
                                  out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle: a position maps outside the block table or the cache")
    return out


def attention_paged(Q, K_cache, V_cache, block_table, seq_lens, M, alpha, causal=False,
                    q_len=0, lib=None):
    """Attention of every (sequence, kv head) over its keys in a paged cache:
    the page's gather of the context into contiguous K and V, then the
    attention oracle with N = that sequence's length.  Q is an operand of
    batch n_seqs * n_kv_heads (entry b = seq * n_kv_heads + head, M rows of
    D); the caches are [num_blocks, block_size, n_kv_heads, D or Dv].
    Returns (O, weight, smag) as ``attention``, over the whole batch."""
    lib = lib or load()
    n_seqs = int(np.asarray(block_table).shape[0])
    heads, D, Dv = K_cache.shape[2], K_cache.shape[3], V_cache.shape[3]
    batch = n_seqs * heads
    if not _span_ok(Q, batch, M, D):
        raise ValueError("oracle: Q strides reach outside its storage")
    O = np.zeros((batch, M, Dv), dtype=np.float64)
    W = np.zeros((batch, M, Dv), dtype=np.float64)
    S = np.zeros((batch, M), dtype=np.float64)
    for s in range(n_seqs):
        n = int(seq_lens[s])
        for h in range(heads):
            b = s * heads + h
            Kc = kv_gather(K_cache, block_table, s, h, n, lib=lib).reshape(-1)
            Vc = kv_gather(V_cache, block_table, s, h, n, lib=lib).reshape(-1)
            Qb = types.SimpleNamespace(storage=Q.storage, offset=Q.offset + b * Q.bs,
                                       rs=Q.rs, cs=Q.cs, bs=0)
            Kb = types.SimpleNamespace(storage=Kc, offset=0, rs=D, cs=1, bs=0)
            Vb = types.SimpleNamespace(storage=Vc, offset=0, rs=Dv, cs=1, bs=0)
            O[b:b + 1], W[b:b + 1], S[b:b + 1] = attention(Qb, Kb, Vb, M, n, D, Dv, 1, alpha,
                                                           causal, q_len, lib=lib)
    return O, W, S
