"""C-ABI checks that need no GPU: the library loads, exports every function the
header declares, and validates / classifies / plans without a device.  No
compute call is made here."""

import ctypes
import os
import re
import subprocess

import pytest

import strided_gemm_gb300 as sg
from strided_gemm_gb300 import build as sgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sbgemm.h")

BASE = 0x7F0000000000   # fake, 256-byte aligned addresses: sbgemm_plan never dereferences


@pytest.fixture(scope="module", autouse=True)
def built():
    sgbuild.build()
    sg.load()


def header_functions():
    txt = open(HEADER).read()
    return re.findall(r"SBGEMM_API\s+[\w\s\*]+?\b(sbgemm\w*)\s*\(", txt)


def test_header_and_binding_agree():
    assert sorted(header_functions()) == sorted(sg.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(sg.LIB_PATH)
    for name in header_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", sg.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == set(header_functions()), exported


def test_noalloc_scratch_size_matches_header():
    # The binding's copy of SBGEMM_NOALLOC_SCRATCH_BYTES (the size the no-alloc
    # test gives sbgemm_ex's workspace to reproduce sbgemm_noalloc bit for bit).
    src = open(os.path.join(ROOT, "include", "sbgemm.h")).read()
    m = re.search(r"#define SBGEMM_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) \* (\d+) \* (\d+) \+ (\d+)\)", src)
    assert m, "macro not found"
    a, b, c, d = (int(x) for x in m.groups())
    assert a * b * c + d == sg.NOALLOC_SCRATCH_BYTES
    # Room for the stream-K scratch of 160 SMs: 256 threads x 64 float pairs + a flag each.
    assert sg.NOALLOC_SCRATCH_BYTES >= 160 * (256 * 64 * 8 + 4)


def test_status_strings_and_version():
    assert sg.sbgemm_status_string(0) == "SBGEMM_OK"
    assert sg.sbgemm_status_string(3) == "SBGEMM_ERR_OUTPUT_OVERLAP"
    assert sg.sbgemm_status_string(99) == "SBGEMM_ERR_UNKNOWN"
    assert sg.sbgemm_version() >= 100


def call_plan(A, B, C, M, N, K, batch, accumulate=0, **kw):
    return sg.sbgemm_plan(*A, *B, *C, M, N, K, batch, accumulate, **kw)


def rowmajor(base, rows, cols, batch):
    return (base, cols, 1, rows * cols)


def test_classifier_layouts():
    M, N, K = 256, 512, 784
    # y = x W^T: A row-major (K-major), B = W^T with rsB = 1 (K-major), C row-major.
    p = call_plan(rowmajor(BASE, M, K, 1), (BASE + (1 << 32), 1, K, N * K),
                  rowmajor(BASE + (2 << 32), M, N, 1), M, N, K, 1)
    assert (p["a_layout"], p["b_layout"], p["c_layout"]) == (sg.LAYOUT_K_MAJOR,) * 3
    assert p["a_tma"] and p["b_tma"]
    # P V: B row-major -> unit stride along N.
    p = call_plan(rowmajor(BASE, 512, 512, 1), rowmajor(BASE + (1 << 32), 512, 64, 1),
                  rowmajor(BASE + (2 << 32), 512, 64, 1), 512, 64, 512, 1)
    assert p["b_layout"] == sg.LAYOUT_MN_MAJOR
    # Both operands read transposed via swapped strides.
    p = call_plan((BASE, 1, 4096, 0), (BASE + (1 << 32), 1, 4096, 0),
                  rowmajor(BASE + (2 << 32), 4096, 4096, 1), 4096, 4096, 4096, 1)
    assert (p["a_layout"], p["b_layout"]) == (sg.LAYOUT_MN_MAJOR, sg.LAYOUT_K_MAJOR)
    # General strides (no unit stride) are not TMA-eligible.
    p = call_plan((BASE, 3, 7, 0), (BASE + (1 << 32), 5, 2, 0),
                  rowmajor(BASE + (2 << 32), 10, 10, 1), 10, 10, 10, 1)
    assert p["a_layout"] == sg.LAYOUT_GENERAL and not p["a_tma"]
    assert p["path"] == sg.PATH_GATHER_FFMA


def test_tma_eligibility_rules():
    M, N, K = 64, 48, 32
    good = call_plan(rowmajor(BASE, M, K, 1), rowmajor(BASE + (1 << 32), K, N, 1),
                     rowmajor(BASE + (2 << 32), M, N, 1), M, N, K, 1)
    assert good["a_tma"] and good["b_tma"]
    # Base not 16-byte aligned.
    p = call_plan((BASE + 4, K, 1, 0), rowmajor(BASE + (1 << 32), K, N, 1),
                  rowmajor(BASE + (2 << 32), M, N, 1), M, N, K, 1)
    assert not p["a_tma"]
    # Row pitch not a multiple of 16 bytes (33 floats).
    p = call_plan((BASE, 33, 1, 0), rowmajor(BASE + (1 << 32), K, N, 1),
                  rowmajor(BASE + (2 << 32), M, N, 1), M, N, K, 1)
    assert not p["a_tma"]
    # Negative row stride.
    p = call_plan((BASE + 4096 * 64, -K, 1, 0), rowmajor(BASE + (1 << 32), K, N, 1),
                  rowmajor(BASE + (2 << 32), M, N, 1), M, N, K, 1)
    assert not p["a_tma"] and p["path"] == sg.PATH_GATHER_FFMA
    # Zero batch stride (shared operand) keeps TMA eligibility and is flagged.
    p = call_plan((BASE, K, 1, 0), rowmajor(BASE + (1 << 32), K, N, 1),
                  (BASE + (2 << 32), N, 1, M * N), M, N, K, 4)
    assert p["a_tma"] and p["a_broadcast"] and not p["b_broadcast"]


def test_validation_errors():
    A = rowmajor(BASE, 8, 8, 1)
    B = rowmajor(BASE + (1 << 32), 8, 8, 1)
    C = rowmajor(BASE + (2 << 32), 8, 8, 1)

    def code(*args, **kw):
        with pytest.raises(sg.SbgemmError) as e:
            call_plan(*args, **kw)
        return e.value.status

    assert code(A, B, C, -1, 8, 8, 1) == sg.SBGEMM_ERR_INVALID_VALUE
    assert code(A, B, C, 8, 8, 8, -2) == sg.SBGEMM_ERR_INVALID_VALUE
    assert code(A, B, (0, 8, 1, 64), 8, 8, 8, 1) == sg.SBGEMM_ERR_NULL_POINTER
    assert code((0, 8, 1, 64), B, C, 8, 8, 8, 1) == sg.SBGEMM_ERR_NULL_POINTER
    assert code((BASE + 2, 8, 1, 64), B, C, 8, 8, 8, 1) == sg.SBGEMM_ERR_INVALID_VALUE
    # C not injective: zero batch stride with batch > 1, zero row stride, or
    # a row pitch shorter than the row.
    assert code(A, B, (C[0], 8, 1, 0), 8, 8, 8, 2) == sg.SBGEMM_ERR_OUTPUT_OVERLAP
    assert code(A, B, (C[0], 0, 1, 64), 8, 8, 8, 1) == sg.SBGEMM_ERR_OUTPUT_OVERLAP
    assert code(A, B, (C[0], 4, 1, 64), 8, 8, 8, 1) == sg.SBGEMM_ERR_OUTPUT_OVERLAP
    # C overlapping A's span.
    assert code(A, B, (BASE + 4 * 32, 8, 1, 64), 8, 8, 8, 1) == sg.SBGEMM_ERR_OUTPUT_OVERLAP
    # Spans that overflow.
    assert code((BASE, 1 << 62, 1, 0), B, C, 8, 8, 8, 1) == sg.SBGEMM_ERR_INVALID_VALUE
    # Bad options.
    assert code(A, B, C, 8, 8, 8, 1, math=7) == sg.SBGEMM_ERR_INVALID_VALUE
    assert code(A, B, C, 8, 8, 8, 1, force_path=9) == sg.SBGEMM_ERR_INVALID_VALUE


def test_fastcall_statuses_match_ctypes():
    """The fast-call module converts the arguments itself and calls the same
    sbgemm_ex / sbgemm: on calls the host checks settle (no device is
    touched) it returns the same status as the ctypes call, takes objects
    with __index__ for sizes, and refuses a wrong argument count."""
    if sg._fast is None:
        pytest.skip("the fast-call module is not built (no Python headers)")
    import numpy as np
    lib = sg.load()
    A = rowmajor(BASE, 8, 8, 1)
    B = rowmajor(BASE + (1 << 32), 8, 8, 1)
    C = rowmajor(BASE + (2 << 32), 8, 8, 1)
    cases = [(A, B, C, -1, 8, 8, 1), (A, B, C, 8, 8, 8, -2), (A, B, (0, 8, 1, 64), 8, 8, 8, 1),
             ((BASE + 2, 8, 1, 64), B, C, 8, 8, 8, 1), (A, B, (C[0], 8, 1, 0), 8, 8, 8, 2),
             (A, B, (BASE + 4 * 32, 8, 1, 64), 8, 8, 8, 1), ((BASE, 1 << 62, 1, 0), B, C, 8, 8, 8, 1),
             (A, B, C, 0, 8, 8, 1), (A, B, C, 8, 8, 8, 0)]
    bad_opts = sg._opts_ref(7, sg.PATH_AUTO, 0, 0, sg.KSPLIT_ANY)
    ok_opts = sg._opts_ref(sg.MATH_FP32, sg.PATH_AUTO, 0, 0, sg.KSPLIT_ANY)
    for a, b, c, M, N, K, batch in cases:
        args = (*a, *b, *c, M, N, K, batch, 0.5, 1)
        for o in (ok_opts, bad_opts):
            want = lib.sbgemm_ex(*args, None, o[1])
            assert sg._fast.sbgemm_ex(*args, 0, o[2]) == want, (args, want)
        want = lib.sbgemm(*args, None)
        assert sg._fast.sbgemm(*args, None) == want
        if want:
            with pytest.raises(sg.SbgemmError) as e:
                sg.sbgemm_ex(*args)
            assert e.value.status == want
    sizes = tuple(np.int64(v) for v in (8, 8, 8, 1))
    assert sg._fast.sbgemm_ex(*A, *B, *C, -1, *sizes[1:], 1.0, 0, 0, 0) == sg.SBGEMM_ERR_INVALID_VALUE
    with pytest.raises(TypeError):
        sg._fast.sbgemm_ex(*A, *B, *C, 8, 8, 8, 1, 1.0, 0, 0)
    with pytest.raises(TypeError):
        sg._fast.sbgemm(*A, *B, *C, "8", 8, 8, 1, 1.0, 0, 0)


def test_ctypes_path_without_the_fast_call_module(monkeypatch, tmp_path):
    """Without Python's headers the build skips the fast-call module, and the
    binding's ctypes calls give the same statuses."""
    import sysconfig
    real = sysconfig.get_paths
    monkeypatch.setattr(sysconfig, "get_paths", lambda *a, **k: dict(real(*a, **k), include=str(tmp_path)))
    assert sgbuild.build_fastcall(force=True) is None
    monkeypatch.setattr(sg, "_fast", None)
    A = rowmajor(BASE, 8, 8, 1)
    B = rowmajor(BASE + (1 << 32), 8, 8, 1)
    C = rowmajor(BASE + (2 << 32), 8, 8, 1)
    for M, batch, want in ((-1, 1, sg.SBGEMM_ERR_INVALID_VALUE), (8, -2, sg.SBGEMM_ERR_INVALID_VALUE)):
        for call in (sg.sbgemm, sg.sbgemm_ex):
            with pytest.raises(sg.SbgemmError) as e:
                call(*A, *B, *C, M, 8, 8, batch, 1.0, 0)
            assert e.value.status == want
    sg.sbgemm_ex(*A, *B, *C, 0, 8, 8, 1, 1.0, 0)   # empty: nothing to do


def test_injective_layouts_accepted():
    A = rowmajor(BASE, 8, 8, 1)
    B = rowmajor(BASE + (1 << 32), 8, 8, 1)
    # Column-major C, padded pitch, negative strides, batch-innermost layout.
    for C in [(BASE + (2 << 32), 1, 8, 64), (BASE + (2 << 32), 11, 1, 100),
              (BASE + (2 << 32) + 4 * 1000, -8, -1, 64), (BASE + (2 << 32), 24, 3, 1)]:
        p = call_plan(A, B, C, 8, 8, 8, 3)
        assert p["path"] != sg.PATH_NONE


def test_empty_and_degenerate_plans():
    A = rowmajor(BASE, 8, 8, 1)
    B = rowmajor(BASE + (1 << 32), 8, 8, 1)
    C = rowmajor(BASE + (2 << 32), 8, 8, 1)
    for M, N, batch in ((0, 8, 1), (8, 0, 1), (8, 8, 0)):
        assert call_plan(A, B, C, M, N, 8, batch)["path"] == sg.PATH_NONE
    # Null pointers are fine when there is nothing to do.
    assert call_plan((0, 0, 0, 0), (0, 0, 0, 0), (0, 0, 0, 0), 0, 0, 0, 0)["path"] == sg.PATH_NONE
    # K == 0: overwrite still writes zeros (a launch); accumulate leaves C alone.
    assert call_plan((0, 0, 0, 0), (0, 0, 0, 0), C, 8, 8, 0, 1)["path"] != sg.PATH_NONE
    assert call_plan((0, 0, 0, 0), (0, 0, 0, 0), C, 8, 8, 0, 1, accumulate=1)["path"] == sg.PATH_NONE


def test_plan_tiles_and_ctas():
    M, N, K = 8192, 2560, 960
    p = call_plan(rowmajor(BASE, M, K, 1), (BASE + (1 << 32), 1, K, 0),
                  rowmajor(BASE + (2 << 32), M, N, 1), M, N, K, 1)
    assert p["tiles"] == -(-M // p["tile_m"]) * -(-N // p["tile_n"])
    assert p["ctas"] >= 1
    # Batch over the 65535 grid limit still plans (the kernel loops over batch).
    p = call_plan((BASE, 1, 1, 1), (BASE + (1 << 32), 1, 1, 1), (BASE + (2 << 32), 1, 1, 1),
                  1, 1, 1, 70000)
    assert p["tiles"] == 70000


def test_stream_k_planning():
    """With a workspace the last waves of tiles are split along K; without
    one, or for problems that fill whole waves or have few K slices, the
    schedule stays data-parallel."""
    ws = BASE + (8 << 32)
    big = 1 << 30
    M = N = K = 4096
    A = rowmajor(BASE, M, K, 1)
    B = rowmajor(BASE + (1 << 32), K, N, 1)
    C = rowmajor(BASE + (2 << 32), M, N, 1)
    p0 = call_plan(A, B, C, M, N, K, 1)
    assert p0["path"] == sg.PATH_TMA_FFMA and not p0["stream_k"]
    assert p0["dp_tiles"] == p0["tiles"] and p0["ctas"] == min(p0["tiles"], 152)
    p1 = call_plan(A, B, C, M, N, K, 1, workspace=ws, workspace_bytes=big)
    assert p1["stream_k"] and p1["ctas"] == 152
    assert p1["dp_tiles"] % 152 == 0 and p1["tiles"] - p1["dp_tiles"] >= 152
    assert p1["k_slices"] == 4096 // p1["tile_k"]
    # Too small a workspace, or a misaligned one.
    assert not call_plan(A, B, C, M, N, K, 1, workspace=ws, workspace_bytes=1024)["stream_k"]
    with pytest.raises(sg.SbgemmError) as e:
        call_plan(A, B, C, M, N, K, 1, workspace=ws + 16, workspace_bytes=big)
    assert e.value.status == sg.SBGEMM_ERR_INVALID_VALUE
    # Fewer tiles than a quarter of the SMs: the gather path, whose 64 tiles
    # are cut into K pieces (test_gather_k_pieces_planning); few K slices:
    # nothing to gain.
    small = call_plan(rowmajor(BASE, 512, 512, 1), rowmajor(BASE + (1 << 32), 512, 512, 1),
                      rowmajor(BASE + (2 << 32), 512, 512, 1), 512, 512, 512, 1,
                      workspace=ws, workspace_bytes=big)
    assert small["path"] == sg.PATH_GATHER_FFMA and small["stream_k"] == sg.STREAM_K_PIECES
    shortk = call_plan(rowmajor(BASE, 4096, 64, 1), (BASE + (1 << 32), 1, 64, 0),
                       rowmajor(BASE + (2 << 32), 4096, 4096, 1), 4096, 4096, 64, 1,
                       workspace=ws, workspace_bytes=big)
    assert not shortk["stream_k"]


def test_tf32_stream_k_planning():
    """The tensor-core path splits with independent pieces: the last waves of
    a many-tile long-K problem, or all tiles of a few-tile long-K one.  Two
    K-major operands with a wave of 256 x 256 tiles run on CTA pairs, split or
    not (each pair one worker of the split); fewer tiles keep one CTA's
    128 x 256 tiles with 32-wide K slices."""
    ws = BASE + (8 << 32)
    big = 1 << 30
    M, N = 2048, 5120
    for K, split in ((4096, True), (1024, False)):
        A = rowmajor(BASE, M, K, 1)
        B = (BASE + (1 << 32), 1, K, 0)                 # column-major: K-major
        C = rowmajor(BASE + (2 << 32), M, N, 1)
        p0 = call_plan(A, B, C, M, N, K, 1, math=sg.MATH_TF32)
        assert p0["path"] == sg.PATH_TMA_TF32 and p0["stream_k"] == sg.STREAM_K_NONE
        assert (p0["tile_m"], p0["tile_n"], p0["tile_k"]) == (256, 256, 32)   # CTA pairs
        assert p0["tiles"] == 160 and p0["ctas"] == 152
        p1 = call_plan(A, B, C, M, N, K, 1, math=sg.MATH_TF32, workspace=ws, workspace_bytes=big)
        assert p1["k_slices"] == K // 32
        assert (p1["tile_m"], p1["tile_n"]) == (256, 256) and p1["ctas"] == 152
        if split:
            # 160 pair tiles on 76 pairs: one data-parallel wave, the rest split.
            assert p1["stream_k"] == sg.STREAM_K_PIECES and p1["tiles"] == 160
            assert p1["dp_tiles"] == 76
        else:
            assert p1["stream_k"] == sg.STREAM_K_NONE and p1["tiles"] == 160
        px = call_plan(A, B, C, M, N, K, 1, math=sg.MATH_TF32, workspace=ws, workspace_bytes=big,
                       k_split=sg.KSPLIT_EXACT)
        assert px["stream_k"] == sg.STREAM_K_NONE and (px["tile_m"], px["tile_n"]) == (256, 256)
    # 32 tiles of 1024 x 1024 with K = 8192: every tile split into pieces.
    M = N = 1024
    K = 8192
    p = call_plan(rowmajor(BASE, M, K, 1), (BASE + (1 << 32), 1, K, 0),
                  rowmajor(BASE + (2 << 32), M, N, 1), M, N, K, 1, math=sg.MATH_TF32,
                  workspace=ws, workspace_bytes=big)
    assert p["stream_k"] == sg.STREAM_K_PIECES and p["dp_tiles"] == 0 and p["ctas"] == 152


def test_split_k_pieces_planning():
    """Fewer tiles than SMs and long K (the weight gradient G^T X of a
    projection layer): with a workspace the tiles' K slices are spread as
    independent pieces over all SMs; k_split = EXACT or NONE keeps whole tiles,
    and NONE also turns off the chained stream-K of many-tile problems."""
    ws = BASE + (8 << 32)
    big = 1 << 30
    M, N, K = 2560, 960, 8192
    A = (BASE, 1, M, 0)                                  # G^T: G stored [K, M]
    B = rowmajor(BASE + (1 << 32), K, N, 1)
    C = rowmajor(BASE + (2 << 32), M, N, 1)
    p0 = call_plan(A, B, C, M, N, K, 1, 1)
    assert p0["path"] == sg.PATH_TMA_FFMA and p0["stream_k"] == sg.STREAM_K_NONE
    assert p0["tiles"] == 80 and p0["ctas"] == 80
    p1 = call_plan(A, B, C, M, N, K, 1, 1, workspace=ws, workspace_bytes=big)
    assert p1["stream_k"] == sg.STREAM_K_PIECES
    assert p1["ctas"] == 152 and p1["dp_tiles"] == 0 and p1["k_slices"] == K // 32
    for policy in (sg.KSPLIT_EXACT, sg.KSPLIT_NONE):
        p = call_plan(A, B, C, M, N, K, 1, 1, workspace=ws, workspace_bytes=big, k_split=policy)
        assert p["stream_k"] == sg.STREAM_K_NONE and p["ctas"] == 80
    # Many tiles: chained stream-K under ANY and EXACT, none under NONE.
    Mb = Nb = Kb = 4096
    A2, B2, C2 = (rowmajor(BASE, Mb, Kb, 1), rowmajor(BASE + (1 << 32), Kb, Nb, 1),
                  rowmajor(BASE + (2 << 32), Mb, Nb, 1))
    for policy, want in ((sg.KSPLIT_ANY, sg.STREAM_K_CHAINED), (sg.KSPLIT_EXACT, sg.STREAM_K_CHAINED),
                         (sg.KSPLIT_NONE, sg.STREAM_K_NONE)):
        p = call_plan(A2, B2, C2, Mb, Nb, Kb, 1, workspace=ws, workspace_bytes=big, k_split=policy)
        assert p["stream_k"] == want, (policy, p)
    # Short K does not split, and an unknown policy is refused.
    short = call_plan((BASE, 1, M, 0), rowmajor(BASE + (1 << 32), 256, N, 1), C, M, N, 256, 1,
                      workspace=ws, workspace_bytes=big)
    assert short["stream_k"] == sg.STREAM_K_NONE
    with pytest.raises(sg.SbgemmError) as e:
        call_plan(A, B, C, M, N, K, 1, workspace=ws, workspace_bytes=big, k_split=3)
    assert e.value.status == sg.SBGEMM_ERR_INVALID_VALUE


def test_tf32_takes_mn_major_operands():
    """TF32 reads operands K-major; an MN-major operand (A M-major or B
    N-major, or both) is transposed in shared memory.  Both MN-major is the
    weight gradient G^T X and is planned as it stands (its transpose is
    both MN-major as well)."""
    M, N, K = 1024, 768, 512
    A_k, A_m = rowmajor(BASE, M, K, 1), (BASE, 1, M, 0)
    B_k, B_n = (BASE + (1 << 32), 1, K, 0), rowmajor(BASE + (1 << 32), K, N, 1)
    C = rowmajor(BASE + (2 << 32), M, N, 1)
    for A, B in ((A_k, B_k), (A_m, B_k), (A_k, B_n), (A_m, B_n)):
        p = call_plan(A, B, C, M, N, K, 1, math=sg.MATH_TF32)
        assert p["path"] == sg.PATH_TMA_TF32, (A, B, p)
    p = call_plan(A_m, B_n, C, M, N, K, 1, math=sg.MATH_TF32, force_path=sg.PATH_TMA_TF32)
    assert p["a_layout"] == sg.LAYOUT_MN_MAJOR and p["b_layout"] == sg.LAYOUT_MN_MAJOR
    assert (p["tile_m"], p["tile_n"]) == (128, 256), p   # not transposed
    # A gathered A (no unit stride) still falls back, and refuses a forced TF32.
    A_g = (BASE, 2, 2 * M, 0)
    assert call_plan(A_g, B_n, C, M, N, K, 1, math=sg.MATH_TF32)["path"] != sg.PATH_TMA_TF32
    with pytest.raises(sg.SbgemmError) as e:
        call_plan(A_g, B_n, C, M, N, K, 1, math=sg.MATH_TF32, force_path=sg.PATH_TMA_TF32)
    assert e.value.status == sg.SBGEMM_ERR_UNSUPPORTED


@pytest.mark.parametrize("N", [64, 768])
def test_tf32_k_major_a_with_n_major_b_runs_transposed(N):
    """K-major A with N-major B is planned as C^T = B^T A^T, whatever N: the
    tile is reported in C's orientation, 256 rows by 128 columns, against
    128 x 256 for the untransposed plan of A M-major with B K-major."""
    M, K = 1024, 512
    A_k, A_m = rowmajor(BASE, M, K, 1), (BASE, 1, M, 0)
    B_k, B_n = (BASE + (1 << 32), 1, K, 0), rowmajor(BASE + (1 << 32), K, N, 1)
    C = rowmajor(BASE + (2 << 32), M, N, 1)
    p = call_plan(A_k, B_n, C, M, N, K, 1, math=sg.MATH_TF32)
    assert p["path"] == sg.PATH_TMA_TF32 and (p["tile_m"], p["tile_n"]) == (256, 128), p
    q = call_plan(A_m, B_k, C, M, N, K, 1, math=sg.MATH_TF32)
    assert q["path"] == sg.PATH_TMA_TF32 and (q["tile_m"], q["tile_n"]) == (128, 256), q


def test_gather_k_pieces_planning():
    """The gather path cuts K into pieces only for products whose tiles fill
    less than half of the CTA slots, with a workspace and k_split = ANY; each
    piece keeps at least 4 slices of 16."""
    ws, big = BASE + (8 << 32), 64 << 20
    M, N, K = 256, 512, 784
    A = (BASE, 786, 1, 0)                    # gapped rows: no tensor map, gather path
    B = (BASE + (1 << 32), 1, K + 3, 0)
    C = rowmajor(BASE + (2 << 32), M, N, 1)
    p = call_plan(A, B, C, M, N, K, 1, workspace=ws, workspace_bytes=big)
    assert p["path"] == sg.PATH_GATHER_FFMA and p["stream_k"] == sg.STREAM_K_PIECES, p
    pieces = p["ctas"] // p["tiles"]
    assert p["ctas"] == p["tiles"] * pieces and 2 <= pieces <= 16
    assert pieces * 4 <= -(-K // 16)
    for kw in ({}, dict(workspace=ws, workspace_bytes=big, k_split=sg.KSPLIT_EXACT),
               dict(workspace=ws, workspace_bytes=1024)):
        q = call_plan(A, B, C, M, N, K, 1, **kw)
        assert q["path"] == sg.PATH_GATHER_FFMA and q["stream_k"] == sg.STREAM_K_NONE, (kw, q)
    # Short K (2 slices) or enough tiles to fill the GPU: whole tiles.
    q = call_plan(A, B, C, M, N, 32, 1, workspace=ws, workspace_bytes=big)
    assert q["stream_k"] == sg.STREAM_K_NONE
    q = call_plan(A, B, C, M, N, K, 40, workspace=ws, workspace_bytes=big)
    assert q["stream_k"] == sg.STREAM_K_NONE


def test_attention_ex_option_checks():
    """sbgemm_attention_ex refuses options it cannot honour before touching the
    device: a forced path other than the tensor-core one, the tensor-core path
    without math = TF32, and non-zero reserved fields."""
    q, k, v, o = BASE, BASE + (1 << 32), BASE + (2 << 32), BASE + (3 << 32)
    args = (q, 64, 1, 128 * 64, k, 64, 1, 128 * 64, v, 64, 1, 128 * 64, o, 64, 1, 128 * 64,
            128, 128, 64, 64, 2, 0.125, 0, 0, 0)
    for math, force, want in ((sg.MATH_TF32, sg.PATH_GATHER_FFMA, sg.SBGEMM_ERR_UNSUPPORTED),
                              (sg.MATH_FP32, sg.PATH_TMA_FFMA, sg.SBGEMM_ERR_UNSUPPORTED),
                              (sg.MATH_FP32, sg.PATH_TMA_TF32, sg.SBGEMM_ERR_INVALID_VALUE),
                              (7, sg.PATH_AUTO, sg.SBGEMM_ERR_INVALID_VALUE)):
        with pytest.raises(sg.SbgemmError) as e:
            sg.sbgemm_attention_ex(*args, math=math, force_path=force)
        assert e.value.status == want, (math, force, e.value.status)


def test_tf32_pair_tiles_need_a_wave_of_pairs():
    """Two K-major operands run on CTA pairs only when the 256 x 256 tiles fill
    at least one wave of pairs (76 on 152 SMs) and K has at least 8 slices;
    otherwise they stay on one CTA's 128 x 256 tiles, and an MN-major operand
    never takes pairs."""
    K = 1024
    for M, N, pair in ((2048, 2304, False), (2560, 2048, True)):   # 72 and 80 pair tiles
        A = rowmajor(BASE, M, K, 1)
        B = (BASE + (1 << 32), 1, K, 0)
        C = rowmajor(BASE + (2 << 32), M, N, 1)
        p = call_plan(A, B, C, M, N, K, 1, math=sg.MATH_TF32)
        assert (p["tile_m"], p["tile_n"]) == ((256, 256) if pair else (128, 256)), p
    M, N = 4096, 4096
    A_m = (BASE, 1, M, 0)
    B = (BASE + (1 << 32), 1, K, 0)
    p = call_plan(A_m, B, rowmajor(BASE + (2 << 32), M, N, 1), M, N, K, 1, math=sg.MATH_TF32)
    assert (p["tile_m"], p["tile_n"]) == (128, 256), p
    # Short K (under 8 slices of 32) stays on one CTA: the C stores set the pace.
    Ks = 128
    p = call_plan(rowmajor(BASE, M, Ks, 1), (BASE + (1 << 32), 1, Ks, 0), rowmajor(BASE + (2 << 32), M, N, 1),
                  M, N, Ks, 1, math=sg.MATH_TF32)
    assert (p["tile_m"], p["tile_n"]) == (128, 256), p
