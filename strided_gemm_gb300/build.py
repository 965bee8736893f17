"""Builds libsbgemm.so in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library next to this file.  A stamp holding a hash of the sources and flags
lets an unchanged tree skip the compile.

build(debug=True) makes libsbgemm_debug.so instead: the same sources with
SBGEMM_DEBUG defined, so that every kernel checks the global addresses it
loads and stores against the operand spans the host validated (a violation
is reported by sbgemm_device_status and the access skipped).
"""

from __future__ import annotations

import glob
import hashlib
import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(HERE, "libsbgemm.so")
STAMP = os.path.join(HERE, ".libsbgemm.stamp")
DEBUG_LIB_PATH = os.path.join(HERE, "libsbgemm_debug.so")
DEBUG_STAMP = os.path.join(HERE, ".libsbgemm_debug.stamp")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
          "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    deps = sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))
    return srcs, deps


def _digest(srcs, deps, extra) -> str:
    h = hashlib.sha256()
    for f in srcs + deps:
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + COMMON + extra).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=None, debug: bool = False) -> str:
    extra = list(extra_flags or []) + (["-DSBGEMM_DEBUG"] if debug else [])
    lib_path, stamp = (DEBUG_LIB_PATH, DEBUG_STAMP) if debug else (LIB_PATH, STAMP)
    srcs, deps = _sources()
    digest = _digest(srcs, deps, extra)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp):
        with open(stamp) as fh:
            if fh.read().strip() == digest:
                return lib_path
    with tempfile.TemporaryDirectory(prefix="sbgemm_build_") as tmp:
        procs = []
        objs = []
        for src in srcs:
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            cmd = [nvcc()] + ARCH + COMMON + extra + ["-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
            objs.append(obj)
        failed = []
        for src, pr in procs:
            out, _ = pr.communicate()
            if pr.returncode != 0:
                failed.append((src, out))
            elif verbose and out.strip():
                print(out, file=sys.stderr)
        if failed:
            msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
            raise RuntimeError(f"nvcc failed:\n{msg}")
        tmp_lib = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp_lib] + objs + ["-cudart", "static"]
        subprocess.run(cmd, check=True)
        os.replace(tmp_lib, lib_path)
    with open(stamp, "w") as fh:
        fh.write(digest + "\n")
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
