"""The debug build of the library (build(debug=True): every kernel checks each
global address it loads or stores against the operand span the host
validated, records a violation in its status word and skips the access).
The parity cases with awkward shapes, every stride layout, fused addends and
small attention problems run against it in a child process that loads that
build, and after every test the device status must be clean.  (The sanitizer
substitute for compute-sanitizer, which is closed on this machine; the StaleyNET
"GPU Implementation" page, section "Safety".)"""

import os
import subprocess
import sys

import pytest

import strided_gemm_gb300 as sg
from strided_gemm_gb300 import build as sgbuild

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    "tests/test_parity_gpu.py::test_workloads_small",
    "tests/test_parity_gpu.py::test_awkward_shapes_all_layouts",
    "tests/test_parity_gpu.py::test_tf32_awkward_shapes",
    "tests/test_fused_gpu.py::test_fused_every_path_activation_and_addend",
    "tests/test_attention_gpu.py::test_attention_small_against_oracle",
    "tests/test_attention_gpu.py::test_attention_tf32_small_against_oracle",
    "tests/test_attention_paged_gpu.py::test_head_dims_against_oracle",
    "tests/test_attention_paged_gpu.py::test_decode_against_oracle",
    "tests/test_attention_paged_gpu.py::test_paged_against_oracle",
]


def test_debug_build_passes_the_parity_cases_with_clean_status():
    path = sgbuild.build(debug=True)
    assert os.path.basename(path) == "libsbgemm_debug.so"
    env = dict(os.environ, SBGEMM_LIBRARY=path, SBGEMM_CHECK_STATUS="1")
    code = ("import strided_gemm_gb300 as sg, sys; "
            f"assert sg.LIB_PATH == {path!r}, sg.LIB_PATH; "
            "import pytest; sys.exit(pytest.main(sys.argv[1:]))")
    r = subprocess.run([sys.executable, "-c", code, *CASES, "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=1800)
    out = r.stdout + r.stderr
    assert r.returncode == 0, out[-4000:]
    assert " passed" in out and " failed" not in out, out[-2000:]
