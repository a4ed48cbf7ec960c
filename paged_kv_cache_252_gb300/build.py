"""Build libpagedkv.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel to an object file under
``paged_kv_cache_252_gb300/_build/`` and linked into
``paged_kv_cache_252_gb300/libpagedkv.so`` (CUDA runtime linked statically;
the driver's tensor-map encoder is looked up at run time).

A profiling variant, ``libpagedkv_timeline.so`` (objects under ``_build_timeline/``),
is the same library compiled with ``-DPKV_TIMELINE``: its decode kernels record
per-CTA event times (``csrc/pkv_timeline.cuh``; driven by ``timeline.py``). The
product library never contains that code.

Usage: ``python -m paged_kv_cache_252_gb300.build [--verbose-ptxas] [--timeline]``
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpagedkv.so")
VARIANTS = {  # name -> (object dir, library, extra nvcc flags)
    "": (OUT_DIR, LIB, []),
    "timeline": (os.path.join(HERE, "_build_timeline"), os.path.join(HERE, "libpagedkv_timeline.so"),
                 ["-DPKV_TIMELINE"]),
}

SOURCES = ["capi.cu", "kv_cache_write.cu", "decode_f16.cu", "decode_bf16.cu", "decode_e5m2.cu",
           "decode_tc.cu", "decode_int8.cu", "noalloc.cu", "copy_blocks.cu", "chunked.cu", "selftest.cu",
           "block_allocator.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


def _compile(src: str, ptxas_verbose: bool, out_dir: str = OUT_DIR, extra=()) -> tuple[str, str]:
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", *extra,
           "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "pagedkv.h"),
                                                               os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, ptxas_verbose: bool = False, variant: str = "") -> str:
    out_dir, lib, extra = VARIANTS[variant]
    if not force and not ptxas_verbose and not _stale(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_verbose, out_dir, extra), SOURCES))
    if ptxas_verbose:
        with open(os.path.join(out_dir, "ptxas.log"), "w") as f:
            for (obj, log), src in zip(results, SOURCES):
                f.write(f"== {src}\n{log}\n")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--timeline", action="store_true", help="build the profiling variant")
    args = ap.parse_args()
    variant = "timeline" if args.timeline else ""
    print(build(force=args.force, ptxas_verbose=args.verbose_ptxas, variant=variant))
    if args.verbose_ptxas:
        print(open(os.path.join(VARIANTS[variant][0], "ptxas.log")).read())
    sys.exit(0)
