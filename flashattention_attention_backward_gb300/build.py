"""Builds the in-tree shared library ``libattnbwd.so`` with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel into ``_build/`` and the
objects are linked into ``libattnbwd.so`` next to this file. A unit is
recompiled only when it, or a header it may include, is newer than its
object file.
"""
import concurrent.futures
import glob
import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT_DIR = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libattnbwd.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
SOURCES = ["attn_bwd.cu", "attn_bwd256.cu", "attn_fwd.cu", "attn_fwd_ref.cu", "attn_prepost.cu",
           "attn_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fno-strict-aliasing"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or add CUDA's bin directory to PATH)")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT_DIR, "include", "*.h"))


def _stale(obj, src):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in [src] + _headers())


def _compile(nvcc, src, obj, extra):
    cmd = [nvcc] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (os.path.basename(src), r.stdout, r.stderr))
    return r.stderr


def build(force=False, verbose=False, extra_flags=()):
    """Compile (if needed) and link the library; returns its path."""
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    jobs = []
    for name in SOURCES:
        src = os.path.join(CSRC, name)
        obj = os.path.join(BUILD_DIR, name.replace(".cu", ".o"))
        if force or _stale(obj, src):
            jobs.append((src, obj))
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            futs = [ex.submit(_compile, nvcc, s, o, list(extra_flags)) for s, o in jobs]
            for f in futs:
                msg = f.result()
                if verbose and msg:
                    print(msg)
    objs = [os.path.join(BUILD_DIR, n.replace(".cu", ".o")) for n in SOURCES]
    if force or jobs or not os.path.exists(LIB_PATH):
        tmp = LIB_PATH + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose=True))
