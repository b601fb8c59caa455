"""Builds tests/c_abi_client.c (plain C99, gcc) against include/attnbwd.h and
the in-tree libattnbwd.so; shared by the CPU test (build only) and the GPU
test (build and run)."""
import os
import shutil
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def cuda_home():
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def build_client(out_path):
    from flashattention_attention_backward_gb300.build import LIB_PATH, build

    build()
    cuda = cuda_home()
    libdir = os.path.dirname(LIB_PATH)
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_abi_client.c"), "-o", out_path,
           "-L", libdir, "-lattnbwd", "-Wl,-rpath," + libdir,
           "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64"),
           "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, "gcc failed:\n%s\n%s" % (r.stdout, r.stderr)
    return out_path
