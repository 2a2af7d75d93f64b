"""In-tree build of libpd_attn.so: every CUDA source compiled for sm_103a
(one -gencode, parallel nvcc processes), the host C++ with g++, linked with
nvcc into ``_build/libpd_attn.so`` next to this file.  No cmake."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libpd_attn.so")

CUDA_SOURCES = ["capi.cu", "store_copy.cu", "kv_pack.cu", "decode.cu", "decode_static.cu",
                "selftest.cu", "copy_bytes.cu",
                "prefill.cu"]
CXX_SOURCES = ["block_manager.cpp", "prefix_cache.cpp"]
HEADERS = ["pd_device.cuh", "pd_internal.h", "pd_tcgen05.cuh", "pd_mma.cuh", "pd_tmap.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "bin", "nvcc")):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise FileNotFoundError("nvcc not found (set CUDA_HOME)")


def _inputs():
    files = [os.path.join(CSRC, f) for f in CUDA_SOURCES + CXX_SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "pd_attn.h"))
    files.append(os.path.abspath(__file__))
    return [f for f in files if os.path.exists(f)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    obj_dir = os.path.join(BUILD, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    common_inc = ["-I", INCLUDE, "-I", CSRC]
    procs = []
    objs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(obj_dir, src + ".o")
        cmd = [nvcc, *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
               "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
               *common_inc, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    for src in CXX_SOURCES:
        obj = os.path.join(obj_dir, src + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-fvisibility=hidden",
               *common_inc, "-I", os.path.join(cuda, "include"),
               "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append(src)
            sys.stderr.write(f"--- {src} ---\n{text}\n")
        elif verbose or ptxas_verbose:
            sys.stdout.write(f"--- {src} ---\n{text}\n")
    if failed:
        raise RuntimeError(f"compilation failed: {failed}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv)
    print(LIB)
