"""Builds libkvc.so in place with nvcc for sm_103a (no cmake, no torch extension).

Every translation unit is compiled in parallel, then linked into one shared
library next to this file. Run ``python -m paged_kv_cache_157_gb300.build_lib``
or call ``build()``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkvc.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = [
    "runtime.cu",
    "append.cu",
    "decode_gqa_api.cu",
    "decode_gqa_f32.cu",
    "decode_gqa_f16.cu",
    "decode_gqa_bf16.cu",
    "decode_gqa_f32_ext.cu",
    "decode_gqa_f16_ext.cu",
    "decode_gqa_bf16_ext.cu",
    "decode_gqa_fp8.cu",
    "decode_gqa_int8.cu",
    "decode_gqa_mma_bf16.cu",
    "decode_gqa_mma_f16.cu",
    "decode_gqa_mma_fp8.cu",
    "decode_gqa_mma_int8.cu",
    "decode_wide.cu",
    "decode_mla.cu",
    "pool.cpp",
]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvc.so")
    return exe


def _extra_flags():
    """Extra nvcc flags from KVC_NVCC_FLAGS (space separated), e.g. tuning macros."""
    return os.environ.get("KVC_NVCC_FLAGS", "").split()


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
           "--expt-relaxed-constexpr", *_extra_flags(), "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    workers = min(len(SOURCES), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
