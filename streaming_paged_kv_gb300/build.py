"""Build libkvc.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in its own nvcc process (in parallel), then one
link step writes ``streaming_paged_kv_gb300/libkvc.so``.  Objects live in
``streaming_paged_kv_gb300/_build/<machine>/`` so that x86 and Arm builds do
not mix; the library is rebuilt whenever a source is newer than it or it was
built for another machine.
"""

import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libkvc.so")
STAMP = os.path.join(PKG, "libkvc.machine")
# KVC_CHECKED=1: the same library with device-side bounds checks, built beside it.
LIB_CHECKED = os.path.join(PKG, "libkvc_checked.so")
STAMP_CHECKED = os.path.join(PKG, "libkvc_checked.machine")
SOURCES = ["kvc_host.cpp", "kvc_kernels.cu", "kvc_attn_tc.cu", "kvc_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(lib=LIB, stamp=STAMP):
    if not os.path.exists(lib) or not os.path.exists(stamp):
        return True
    if open(stamp).read().strip() != platform.machine():
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "kvc.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False, extra_flags=(), checked=None):
    """Compile and link libkvc.so (with checked=True, or KVC_CHECKED=1 in the
    environment: libkvc_checked.so, with -DKVC_CHECKED=1); returns its path."""
    if checked is None:
        checked = os.environ.get("KVC_CHECKED") == "1"
    lib, stamp = (LIB_CHECKED, STAMP_CHECKED) if checked else (LIB, STAMP)
    if checked:
        extra_flags = tuple(extra_flags) + ("-DKVC_CHECKED=1",)
    if not force and not _stale(lib, stamp):
        return lib
    out_dir = os.path.join(PKG, "_build", platform.machine() + ("-checked" if checked else ""))
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(out_dir, src + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose and src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(platform.machine() + "\n")
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
