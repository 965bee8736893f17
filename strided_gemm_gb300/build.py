"""Builds libsbgemm.so in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library next to this file.  A stamp holding a hash of the sources and flags
lets an unchanged tree skip the compile.

build(debug=True) makes libsbgemm_debug.so instead: the same sources with
SBGEMM_DEBUG defined, so that every kernel checks the global addresses it
loads and stores against the operand spans the host validated (a violation
is reported by sbgemm_device_status and the access skipped).

build() also compiles the binding's fast-call module (csrc/fastcall.c, with
the host C compiler against Python's headers) when those headers are
present; without it the binding calls the library through ctypes alone.
"""

from __future__ import annotations

import glob
import hashlib
import os
import shutil
import subprocess
import sys
import sysconfig
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


FASTCALL_SRC = os.path.join(CSRC, "fastcall.c")
FASTCALL_PATH = os.path.join(HERE, "_fastcall" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))
FASTCALL_STAMP = os.path.join(HERE, ".fastcall.stamp")


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


def build_fastcall(force: bool = False) -> str | None:
    """Compiles the fast-call module next to the library; None when Python's
    headers or a C compiler are missing (the binding then uses ctypes)."""
    inc = sysconfig.get_paths().get("include") or ""
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if not cc or not os.path.exists(os.path.join(inc, "Python.h")):
        return None
    h = hashlib.sha256()
    for f in (FASTCALL_SRC, os.path.join(INCLUDE, "sbgemm.h")):
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update((cc + inc + FASTCALL_PATH).encode())
    digest = h.hexdigest()
    if not force and os.path.exists(FASTCALL_PATH) and os.path.exists(FASTCALL_STAMP):
        with open(FASTCALL_STAMP) as fh:
            if fh.read().strip() == digest:
                return FASTCALL_PATH
    tmp = FASTCALL_PATH + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-shared", "-fPIC", "-fvisibility=hidden", "-I", inc, "-I", INCLUDE,
           FASTCALL_SRC, "-o", tmp]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"the fast-call module failed to compile:\n{r.stdout}")
    os.replace(tmp, FASTCALL_PATH)
    with open(FASTCALL_STAMP, "w") as fh:
        fh.write(digest + "\n")
    return FASTCALL_PATH


def build(force: bool = False, verbose: bool = False, extra_flags=None, debug: bool = False) -> str:
    build_fastcall(force)
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
