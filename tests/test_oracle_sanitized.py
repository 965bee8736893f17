"""The oracle's pins again, on a build of the oracle with AddressSanitizer and
UndefinedBehaviorSanitizer: an out-of-bounds read or write, a use after free,
a signed overflow or a misaligned access anywhere in the C source aborts the
run.  (The host-emulation chapter of the kael pages runs its tests under these
sanitizers; compute-sanitizer, their device-side counterpart, is closed on
this pool.)

The pins run in a child process that starts with the sanitizer runtimes
preloaded, since the Python interpreter itself is not instrumented."""

import os
import shutil
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _runtime(name):
    cc = shutil.which("gcc")
    if cc is None:
        return None
    p = subprocess.run([cc, f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_oracle_pins_under_address_and_undefined_behavior_sanitizers():
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not asan or not ubsan:
        pytest.skip("gcc sanitizer runtimes not installed")
    oracle.build(sanitize=True)
    env = dict(os.environ)
    env.update({
        "LD_PRELOAD": f"{asan}:{ubsan}",
        "ASAN_OPTIONS": "detect_leaks=0:abort_on_error=0:exitcode=86",
        "UBSAN_OPTIONS": "halt_on_error=1:print_stacktrace=1:exitcode=87",
        "SBGEMM_ORACLE_SANITIZE": "1",
    })
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle.py", "-q", "-x",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    out = r.stdout + r.stderr
    assert "AddressSanitizer" not in out and "runtime error:" not in out, out[-4000:]
    assert r.returncode == 0, out[-4000:]
    assert " passed" in out, out[-2000:]
