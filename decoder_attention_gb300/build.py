"""Build libdecattn.so (the C-ABI library) in-tree with nvcc for sm_103a.

    python -m decoder_attention_gb300.build          # or __graft_entry__.build()

Each translation unit is compiled in parallel; the objects go to decoder_attention_gb300/_build/ and the
shared library to decoder_attention_gb300/libdecattn.so. The CUDA runtime is linked statically, so the
library loads without libcudart on the library path; the driver entry point it needs for tensor maps is
resolved at run time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdecattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cpp", "block_pool.cpp", "errors.cu", "rope_kv.cu", "attn_generic.cu", "attn_decode.cu", "attn_prefill.cu", "mla.cu", "mla_pair.cu", "proj.cu"]


def nvcc_path():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin on PATH)")


def _compile(nvcc, src, extra):
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj, "-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC,
           "-Xcompiler", "-fPIC", "-lineinfo"] + ARCH + extra
    if src.endswith(".cu"):
        cmd += ["--expt-relaxed-constexpr", "-Xptxas", "-v"] if os.environ.get("DA_PTXAS_VERBOSE") else ["--expt-relaxed-constexpr"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, res.returncode, res.stdout + res.stderr, " ".join(cmd)


def build(verbose: bool = False, extra_flags: list | None = None) -> str:
    """Compile every source and link libdecattn.so; returns the library path. Raises on failure."""
    nvcc = nvcc_path()
    os.makedirs(BUILD, exist_ok=True)
    extra = list(extra_flags or [])
    objs = []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for src, obj, rc, out, cmd in ex.map(lambda s: _compile(nvcc, s, extra), SOURCES):
            if verbose or rc != 0:
                sys.stderr.write(f"[build] {cmd}\n{out}")
            if rc != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{out}")
            objs.append(obj)
    tmp = LIB + ".tmp"
    cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
