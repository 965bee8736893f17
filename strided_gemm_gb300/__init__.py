"""Python binding of libsbgemm, the strided batched fp32 product for GB300.

The functions below carry the C names and arguments of include/sbgemm.h and do
argument marshalling only: every step of the product runs in the library's
CUDA kernels.  Pointers are plain integers (device addresses); strides are in
fp32 elements.  A non-zero status raises SbgemmError.

``matmul`` is a convenience over torch CUDA tensors viewed as [batch, rows,
cols] (any strides, including expand()-ed zero strides).
"""

from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "SbgemmError", "load", "sbgemm", "sbgemm_ex", "sbgemm_plan", "sbgemm_workspace_bytes",
    "sbgemm_noalloc", "sbgemm_selftest", "SELFTEST_MBARRIER", "SELFTEST_FLAG",
    "sbgemm_device_status", "sbgemm_status_string", "sbgemm_version", "matmul",
    "SBGEMM_OK", "SBGEMM_ERR_INVALID_VALUE", "SBGEMM_ERR_NULL_POINTER",
    "SBGEMM_ERR_OUTPUT_OVERLAP", "SBGEMM_ERR_UNSUPPORTED", "SBGEMM_ERR_CUDA",
    "SBGEMM_ERR_DEVICE_TIMEOUT", "SBGEMM_ERR_NOT_DEVICE_MEMORY", "SBGEMM_ERR_DEVICE_CHECK",
    "MATH_FP32", "MATH_TF32", "PATH_NONE", "PATH_AUTO", "PATH_GATHER_FFMA",
    "PATH_TMA_FFMA", "PATH_TMA_TF32", "LAYOUT_K_MAJOR", "LAYOUT_MN_MAJOR",
    "LAYOUT_GENERAL", "EXPORTED_SYMBOLS", "LIB_PATH", "sbgemm_fused", "linear_backward",
    "sbgemm_attention", "sbgemm_attention_ex", "sbgemm_attention_paged", "attention",
    "ACT_NONE", "ACT_RELU", "ACT_SIGMOID", "ACT_SILU", "ACT_GELU_TANH", "ACT_GELU_ERF",
    "ACTIVATIONS", "KSPLIT_ANY", "KSPLIT_EXACT", "KSPLIT_NONE", "STREAM_K_NONE",
    "STREAM_K_CHAINED", "STREAM_K_PIECES", "NOALLOC_SCRATCH_BYTES",
]

HERE = os.path.dirname(os.path.abspath(__file__))
# SBGEMM_LIBRARY selects another build of the library, e.g. the debug build
# (build(debug=True): libsbgemm_debug.so, with device bounds checks).
LIB_PATH = os.environ.get("SBGEMM_LIBRARY") or os.path.join(HERE, "libsbgemm.so")

SBGEMM_OK = 0
SBGEMM_ERR_INVALID_VALUE = 1
SBGEMM_ERR_NULL_POINTER = 2
SBGEMM_ERR_OUTPUT_OVERLAP = 3
SBGEMM_ERR_UNSUPPORTED = 4
SBGEMM_ERR_CUDA = 5
SBGEMM_ERR_DEVICE_TIMEOUT = 6
SBGEMM_ERR_NOT_DEVICE_MEMORY = 7
SBGEMM_ERR_DEVICE_CHECK = 8

MATH_FP32, MATH_TF32 = 0, 1
PATH_NONE, PATH_AUTO, PATH_GATHER_FFMA, PATH_TMA_FFMA, PATH_TMA_TF32 = -1, 0, 1, 2, 3
LAYOUT_K_MAJOR, LAYOUT_MN_MAJOR, LAYOUT_GENERAL = 0, 1, 2
PATH_NAMES = {PATH_NONE: "none", PATH_GATHER_FFMA: "gather_ffma",
              PATH_TMA_FFMA: "tma_ffma", PATH_TMA_TF32: "tma_tf32"}

# Every function include/sbgemm.h declares.
EXPORTED_SYMBOLS = ("sbgemm", "sbgemm_ex", "sbgemm_fused", "sbgemm_attention",
                    "sbgemm_attention_ex", "sbgemm_attention_paged", "sbgemm_plan",
                    "sbgemm_workspace_bytes", "sbgemm_noalloc", "sbgemm_selftest",
                    "sbgemm_device_status", "sbgemm_status_string", "sbgemm_version")
ACT_NONE, ACT_RELU, ACT_SIGMOID, ACT_SILU, ACT_GELU_TANH, ACT_GELU_ERF = 0, 1, 2, 3, 4, 5
ACTIVATIONS = {"none": ACT_NONE, "relu": ACT_RELU, "sigmoid": ACT_SIGMOID, "silu": ACT_SILU,
               "gelu_tanh": ACT_GELU_TANH, "gelu_erf": ACT_GELU_ERF}
SELFTEST_MBARRIER, SELFTEST_FLAG = 1, 2
KSPLIT_ANY, KSPLIT_EXACT, KSPLIT_NONE = 0, 1, 2
# Bytes of sbgemm_noalloc's static scratch (SBGEMM_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 20 * 1024 * 1024 + 4096
STREAM_K_NONE, STREAM_K_CHAINED, STREAM_K_PIECES = 0, 1, 2


class SbgemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {sbgemm_status_string(status)} ({status})")


class _Options(ctypes.Structure):
    _fields_ = [("math", ctypes.c_int), ("force_path", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("k_split", ctypes.c_int), ("reserved", ctypes.c_int * 1)]


class _Epilogue(ctypes.Structure):
    _fields_ = [("D", ctypes.c_void_p), ("rsD", ctypes.c_int64), ("csD", ctypes.c_int64),
                ("bsD", ctypes.c_int64), ("activation", ctypes.c_int),
                ("reserved", ctypes.c_int * 3)]


class _PlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("a_layout", ctypes.c_int),
                ("b_layout", ctypes.c_int), ("c_layout", ctypes.c_int),
                ("a_broadcast", ctypes.c_int), ("b_broadcast", ctypes.c_int),
                ("a_tma", ctypes.c_int), ("b_tma", ctypes.c_int),
                ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("tile_k", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("ctas", ctypes.c_int64), ("tiles", ctypes.c_int64),
                ("stream_k", ctypes.c_int), ("k_slices", ctypes.c_int),
                ("dp_tiles", ctypes.c_int64), ("reserved", ctypes.c_int * 4)]


_lock = threading.Lock()
_lib = None
# The fast-call module (csrc/fastcall.c), bound to the loaded library's
# sbgemm_ex and sbgemm: the same calls with cheaper argument conversion.
# None where it was not built; the ctypes calls below then serve.
_fast = None
_i64, _vp = ctypes.c_int64, ctypes.c_void_p
_ARGS = [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _i64,
         _i64, _i64, _i64, _i64]


def load(path: str = LIB_PATH):
    """Load libsbgemm.so.  Raises if the library has not been built: there is
    no fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"the library is missing at {path}; build it with "
                "`python -m strided_gemm_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(path)
        lib.sbgemm.restype = ctypes.c_int
        lib.sbgemm.argtypes = _ARGS + [ctypes.c_float, ctypes.c_int, _vp]
        lib.sbgemm_fused.restype = ctypes.c_int
        lib.sbgemm_fused.argtypes = _ARGS + [ctypes.c_float, ctypes.c_int,
                                             ctypes.POINTER(_Epilogue), _vp,
                                             ctypes.POINTER(_Options)]
        lib.sbgemm_attention.restype = ctypes.c_int
        op4 = [_vp, _i64, _i64, _i64]
        lib.sbgemm_attention.argtypes = (op4 * 4 + [_i64] * 5 +
                                         [ctypes.c_float, ctypes.c_int, _i64, _vp])
        lib.sbgemm_attention_ex.restype = ctypes.c_int
        lib.sbgemm_attention_ex.argtypes = (op4 * 4 + [_i64] * 5 +
                                            [ctypes.c_float, ctypes.c_int, _i64, _vp,
                                             ctypes.POINTER(_Options)])
        lib.sbgemm_attention_paged.restype = ctypes.c_int
        lib.sbgemm_attention_paged.argtypes = (op4 + [_vp, _vp, _i64, _i64, _i64, _vp, _i64, _vp] +
                                               op4 + [_i64] * 5 +
                                               [ctypes.c_float, ctypes.c_int, _i64, _vp,
                                                ctypes.POINTER(_Options)])
        lib.sbgemm_ex.restype = ctypes.c_int
        lib.sbgemm_ex.argtypes = _ARGS + [ctypes.c_float, ctypes.c_int, _vp,
                                          ctypes.POINTER(_Options)]
        lib.sbgemm_plan.restype = ctypes.c_int
        lib.sbgemm_plan.argtypes = _ARGS + [ctypes.c_int, ctypes.POINTER(_Options),
                                            ctypes.POINTER(_PlanInfo)]
        lib.sbgemm_noalloc.restype = ctypes.c_int
        lib.sbgemm_noalloc.argtypes = _ARGS + [ctypes.c_float, ctypes.c_int, _vp]
        lib.sbgemm_workspace_bytes.restype = ctypes.c_int
        lib.sbgemm_workspace_bytes.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
        lib.sbgemm_selftest.restype = ctypes.c_int
        lib.sbgemm_selftest.argtypes = [ctypes.c_int, _i64, _vp]
        lib.sbgemm_device_status.restype = ctypes.c_int
        lib.sbgemm_device_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_int)]
        lib.sbgemm_status_string.restype = ctypes.c_char_p
        lib.sbgemm_status_string.argtypes = [ctypes.c_int]
        lib.sbgemm_version.restype = ctypes.c_int
        lib.sbgemm_version.argtypes = []
        global _fast
        try:
            from . import _fastcall
            _fastcall.bind(ctypes.cast(lib.sbgemm_ex, ctypes.c_void_p).value,
                           ctypes.cast(lib.sbgemm, ctypes.c_void_p).value)
            _fast = _fastcall
        except ImportError:
            _fast = None
        _lib = lib
        return lib


def _opts(math: int, force_path: int, workspace=0, workspace_bytes=0, k_split=KSPLIT_ANY):
    o = _Options()
    o.math = int(math)
    o.force_path = int(force_path)
    o.workspace = int(workspace) or None
    o.workspace_bytes = int(workspace_bytes)
    o.k_split = int(k_split)
    return o


# Option structs by value, reused across calls (the library reads them only
# during the call): a call with options it has seen before builds nothing.
_opts_cache: dict = {}


def _opts_ref(math, force_path, workspace, workspace_bytes, k_split):
    key = (math, force_path, workspace, workspace_bytes, k_split)
    r = _opts_cache.get(key)
    if r is None:
        o = _opts(math, force_path, workspace, workspace_bytes, k_split)
        if len(_opts_cache) >= 256:
            _opts_cache.clear()
        r = _opts_cache[key] = (o, ctypes.byref(o), ctypes.addressof(o))
    return r


def sbgemm_workspace_bytes(device: int = 0) -> int:
    """Bytes of caller-owned workspace that enable the stream-K schedule."""
    n = ctypes.c_size_t(0)
    st = load().sbgemm_workspace_bytes(int(device), ctypes.byref(n))
    if st:
        raise SbgemmError(st, "sbgemm_workspace_bytes")
    return n.value


def sbgemm_status_string(status: int) -> str:
    return load().sbgemm_status_string(int(status)).decode()


def sbgemm_version() -> int:
    return load().sbgemm_version()


def sbgemm(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
           M, N, K, batch, alpha, accumulate, stream=0) -> None:
    lib = _lib if _lib is not None else load()
    if _fast is not None:
        st = _fast.sbgemm(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                          M, N, K, batch, alpha, 1 if accumulate else 0, stream or 0)
    else:
        st = lib.sbgemm(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                        M, N, K, batch, alpha, 1 if accumulate else 0, stream or None)
    if st:
        raise SbgemmError(st, "sbgemm")


def sbgemm_noalloc(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                   M, N, K, batch, alpha, accumulate, stream=0) -> None:
    """As sbgemm_ex with k_split = KSPLIT_ANY, for callers that cannot
    allocate device memory: the scratch of the stream-K schedule and of the K
    pieces is the library's own static device array of NOALLOC_SCRATCH_BYTES
    (shared by all calls, so calls that overlap on the GPU must be
    serialised).  Make the first call on a device outside stream capture."""
    st = load().sbgemm_noalloc(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                               M, N, K, batch, float(alpha), int(bool(accumulate)),
                               stream or None)
    if st:
        raise SbgemmError(st, "sbgemm_noalloc")


def sbgemm_ex(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
              M, N, K, batch, alpha, accumulate, stream=0,
              math: int = MATH_FP32, force_path: int = PATH_AUTO,
              workspace: int = 0, workspace_bytes: int = 0, k_split: int = KSPLIT_ANY) -> None:
    lib = _lib if _lib is not None else load()
    o = _opts_ref(math, force_path, workspace, workspace_bytes, k_split)
    if _fast is not None:
        st = _fast.sbgemm_ex(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                             M, N, K, batch, alpha, 1 if accumulate else 0, stream or 0, o[2])
    else:
        st = lib.sbgemm_ex(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                           M, N, K, batch, alpha, 1 if accumulate else 0, stream or None, o[1])
    if st:
        raise SbgemmError(st, "sbgemm_ex")


def sbgemm_fused(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                 M, N, K, batch, alpha, accumulate, D=0, rsD=0, csD=0, bsD=0,
                 activation: int = ACT_NONE, stream=0, math: int = MATH_FP32,
                 force_path: int = PATH_AUTO, workspace: int = 0, workspace_bytes: int = 0,
                 k_split: int = KSPLIT_ANY) -> None:
    """C <- act(alpha*A*B (+C) + D) with D read through (rsD, csD, bsD)."""
    e = _Epilogue()
    e.D = int(D) or None
    e.rsD, e.csD, e.bsD = int(rsD), int(csD), int(bsD)
    e.activation = int(activation)
    o = _opts(math, force_path, workspace, workspace_bytes, k_split)
    st = load().sbgemm_fused(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                             M, N, K, batch, float(alpha), int(bool(accumulate)),
                             ctypes.byref(e), stream or None, ctypes.byref(o))
    if st:
        raise SbgemmError(st, "sbgemm_fused")


def sbgemm_attention(Q, rsQ, csQ, bsQ, K, rsK, csK, bsK, V, rsV, csV, bsV,
                     O, rsO, csO, bsO, M, N, D, Dv, batch, alpha, causal=0, q_len=0,
                     stream=0, math: int = MATH_FP32, force_path: int = PATH_AUTO,
                     workspace: int = 0, workspace_bytes: int = 0) -> None:
    """O = softmax(alpha * Q K^T [causal]) V over strided operands; math =
    MATH_TF32 opts in to the tensor-core kernel, and a workspace lets the
    decode kernel split keys (sbgemm_attention_ex)."""
    if math != MATH_FP32 or force_path != PATH_AUTO or workspace:
        sbgemm_attention_ex(Q, rsQ, csQ, bsQ, K, rsK, csK, bsK, V, rsV, csV, bsV,
                            O, rsO, csO, bsO, M, N, D, Dv, batch, alpha, causal, q_len,
                            stream, math=math, force_path=force_path, workspace=workspace,
                            workspace_bytes=workspace_bytes)
        return
    st = load().sbgemm_attention(Q, rsQ, csQ, bsQ, K, rsK, csK, bsK, V, rsV, csV, bsV,
                                 O, rsO, csO, bsO, M, N, D, Dv, batch, float(alpha),
                                 int(causal), int(q_len), stream or None)
    if st:
        raise SbgemmError(st, "sbgemm_attention")


def sbgemm_attention_ex(Q, rsQ, csQ, bsQ, K, rsK, csK, bsK, V, rsV, csV, bsV,
                        O, rsO, csO, bsO, M, N, D, Dv, batch, alpha, causal=0, q_len=0,
                        stream=0, math: int = MATH_FP32, force_path: int = PATH_AUTO,
                        workspace: int = 0, workspace_bytes: int = 0) -> None:
    """sbgemm_attention with options: math = MATH_TF32 runs the tensor-core
    kernel when Q, K and V suit tensor maps (force_path = PATH_TMA_TF32 makes
    that a requirement); a workspace lets the decode kernel split each entry's
    keys across CTAs."""
    o = _opts(math, force_path, workspace, workspace_bytes)
    st = load().sbgemm_attention_ex(Q, rsQ, csQ, bsQ, K, rsK, csK, bsK, V, rsV, csV, bsV,
                                    O, rsO, csO, bsO, M, N, D, Dv, batch, float(alpha),
                                    int(causal), int(q_len), stream or None, ctypes.byref(o))
    if st:
        raise SbgemmError(st, "sbgemm_attention_ex")


def sbgemm_attention_paged(Q, rsQ, csQ, bsQ, K_cache, V_cache, num_blocks, block_size,
                           n_kv_heads, block_table, max_blocks, seq_lens, O, rsO, csO, bsO,
                           M, N, D, Dv, n_seqs, alpha, causal=0, q_len=0, stream=0,
                           workspace: int = 0, workspace_bytes: int = 0) -> None:
    """Attention with K and V read from a paged cache [num_blocks, block_size,
    n_kv_heads, D] through an int32 block table [n_seqs, max_blocks] and
    optional int32 sequence lengths (device pointers; 0 for seq_lens means N
    keys everywhere).  Batch entry b of Q and O is (sequence b // n_kv_heads,
    head b % n_kv_heads)."""
    o = _opts(MATH_FP32, PATH_AUTO, workspace, workspace_bytes)
    st = load().sbgemm_attention_paged(Q, rsQ, csQ, bsQ, K_cache, V_cache, num_blocks, block_size,
                                       n_kv_heads, block_table, max_blocks, seq_lens or None,
                                       O, rsO, csO, bsO, M, N, D, Dv, n_seqs, float(alpha),
                                       int(causal), int(q_len), stream or None, ctypes.byref(o))
    if st:
        raise SbgemmError(st, "sbgemm_attention_paged")


def attention(Q, K, V, O, alpha=None, causal=False, q_len=0, stream=None, math=MATH_FP32):
    """Torch helper: Q [batch, M, D], K [batch, N, D], V [batch, N, Dv] and O
    [batch, M, Dv] float32 CUDA tensors with any strides (2-D means batch 1;
    K and V may have batch 1 to be shared).  alpha defaults to 1/sqrt(D);
    math = MATH_TF32 opts in to the tensor cores.  Returns O."""
    import torch
    Q3, K3, V3, O3 = _as3(Q, "Q"), _as3(K, "K"), _as3(V, "V"), _as3(O, "O")
    for t, n in ((Q3, "Q"), (K3, "K"), (V3, "V"), (O3, "O")):
        if t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError(f"{n} must be a float32 CUDA tensor")
    batch, M, D = Q3.shape
    N, Dv = K3.shape[1], V3.shape[2]
    if K3.shape[2] != D or V3.shape[1] != N or tuple(O3.shape) != (batch, M, Dv):
        raise ValueError(f"shape mismatch: Q{tuple(Q3.shape)} K{tuple(K3.shape)} "
                         f"V{tuple(V3.shape)} O{tuple(O3.shape)}")
    bs = lambda t: t.stride(0) if t.shape[0] == batch else 0
    if stream is None:
        stream = torch.cuda.current_stream(O3.device).cuda_stream
    sbgemm_attention(Q3.data_ptr(), Q3.stride(1), Q3.stride(2), Q3.stride(0),
                     K3.data_ptr(), K3.stride(1), K3.stride(2), bs(K3),
                     V3.data_ptr(), V3.stride(1), V3.stride(2), bs(V3),
                     O3.data_ptr(), O3.stride(1), O3.stride(2), O3.stride(0),
                     M, N, D, Dv, batch, (1.0 / D ** 0.5) if alpha is None else alpha,
                     int(bool(causal)), int(q_len) if causal else 0, stream, math=math)
    return O


def sbgemm_plan(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                M, N, K, batch, accumulate=0, math: int = MATH_FP32,
                force_path: int = PATH_AUTO, workspace: int = 0,
                workspace_bytes: int = 0, k_split: int = KSPLIT_ANY) -> dict:
    """Validate and plan without launching; returns the plan as a dict."""
    o = _opts(math, force_path, workspace, workspace_bytes, k_split)
    info = _PlanInfo()
    st = load().sbgemm_plan(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC,
                            M, N, K, batch, int(bool(accumulate)), ctypes.byref(o),
                            ctypes.byref(info))
    if st:
        raise SbgemmError(st, "sbgemm_plan")
    d = {name: getattr(info, name) for name, _ in _PlanInfo._fields_ if name != "reserved"}
    d["path_name"] = PATH_NAMES.get(d["path"], "?")
    return d


def sbgemm_selftest(what: int, limit_us: int, stream=0) -> None:
    """Launch the failure-detection self-test (a wait that must run out)."""
    st = load().sbgemm_selftest(int(what), int(limit_us), stream or None)
    if st:
        raise SbgemmError(st, "sbgemm_selftest")


def sbgemm_device_status(stream=0):
    """Synchronise `stream`, then read and clear the in-kernel wait status.
    Returns (status, where)."""
    where = ctypes.c_int(0)
    st = load().sbgemm_device_status(stream or None, ctypes.byref(where))
    return st, where.value


def _as3(t, name):
    if t.dim() == 2:
        t = t.unsqueeze(0)
    if t.dim() != 3:
        raise ValueError(f"{name} must be 2-D or 3-D, got {tuple(t.shape)}")
    return t


def matmul(A, B, C, alpha: float = 1.0, accumulate: bool = False,
           math: int = MATH_FP32, force_path: int = PATH_AUTO, stream=None,
           workspace=None, k_split: int = KSPLIT_ANY, bias=None, activation=ACT_NONE):
    """C <- alpha*A@B (+C) on torch CUDA float32 tensors viewed as [batch, M, K],
    [batch, K, N] and [batch, M, N] (2-D means batch 1).  Strides are taken from
    the tensors, so transposed or expanded views need no copy.  With `bias` (a
    tensor broadcastable to C, e.g. [N] per column) or an `activation` (an
    ACT_* code or its name) the epilogue is fused: C <- act(alpha*A@B (+C) +
    bias).  Returns C."""
    import torch
    A3, B3, C3 = _as3(A, "A"), _as3(B, "B"), _as3(C, "C")
    for t, n in ((A3, "A"), (B3, "B"), (C3, "C")):
        if t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError(f"{n} must be a float32 CUDA tensor")
    batch, M, K = C3.shape[0], C3.shape[1], A3.shape[2]
    N = C3.shape[2]
    if A3.shape[1] != M or B3.shape[1] != K or B3.shape[2] != N:
        raise ValueError(f"shape mismatch: A{tuple(A3.shape)} B{tuple(B3.shape)} C{tuple(C3.shape)}")
    for t, n in ((A3, "A"), (B3, "B")):
        if t.shape[0] not in (1, batch):
            raise ValueError(f"{n} batch {t.shape[0]} does not match {batch}")
    bsA = A3.stride(0) if A3.shape[0] == batch else 0
    bsB = B3.stride(0) if B3.shape[0] == batch else 0
    if stream is None:
        stream = torch.cuda.current_stream(C3.device).cuda_stream
    ws, ws_bytes = 0, 0
    if workspace is not None:
        ws, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    args = (A3.data_ptr(), A3.stride(1), A3.stride(2), bsA,
            B3.data_ptr(), B3.stride(1), B3.stride(2), bsB,
            C3.data_ptr(), C3.stride(1), C3.stride(2), C3.stride(0),
            M, N, K, batch, alpha, accumulate)
    act = ACTIVATIONS[activation] if isinstance(activation, str) else int(activation)
    if bias is None and act == ACT_NONE:
        sbgemm_ex(*args, stream, math, force_path, ws, ws_bytes, k_split)
        return C
    D, rsD, csD, bsD = 0, 0, 0, 0
    if bias is not None:
        if bias.dtype != torch.float32 or not bias.is_cuda:
            raise TypeError("bias must be a float32 CUDA tensor")
        Dv = bias.expand(C3.shape) if bias.dim() == 3 else bias.expand(C3.shape[1:]).unsqueeze(0)
        Dv = Dv.expand(C3.shape)
        D, rsD, csD, bsD = Dv.data_ptr(), Dv.stride(1), Dv.stride(2), Dv.stride(0)
    sbgemm_fused(*args, D, rsD, csD, bsD, act, stream, math, force_path, ws, ws_bytes, k_split)
    return C


def linear_backward(G, X, W, dX, dW, accumulate_dW: bool = False, stream=None,
                    workspace=None, k_split: int = KSPLIT_ANY, math: int = MATH_FP32):
    """Gradients of the linear layer Y = X W^T (X [T, in], W [out, in], upstream
    gradient G = dL/dY [T, out]), as two strided products that read the
    transposes through swapped strides, with no copy (the pages' "PyTorch
    demystified 3", section "Opt. 3 - Speed up matmul in the backward block
    through kernel fusion"):
        dX = G W        [T, in]   (B = W read row-major, N-major)
        dW = G^T X      [out, in] (A = G read with swapped strides; K = T)
    dW accumulates into the existing gradient when accumulate_dW is set.  With
    a workspace the long-K dW product may be split into independent K pieces
    (deterministic; k_split = KSPLIT_EXACT keeps the unsplit rounding).
    math = MATH_TF32 runs both on the tensor cores (dW's operands are both
    MN-major and are transposed in shared memory)."""
    matmul(G, W, dX, math=math, stream=stream, workspace=workspace, k_split=k_split)
    matmul(G.t(), X, dW, accumulate=accumulate_dW, math=math, stream=stream, workspace=workspace,
           k_split=k_split)
    return dX, dW
