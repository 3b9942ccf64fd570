"""Builds libattn.so (the C-ABI attention library) in-tree for sm_103a.

Each CUDA translation unit is compiled in parallel with nvcc, then linked into
`causal_head_attention_fwd_gb300/libattn.so`. Rebuilds only when a source or
header is newer than the library.

    python -m causal_head_attention_fwd_gb300.build [--force] [-v]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import pathlib
import shutil
import subprocess
import sys

PKG = pathlib.Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = ROOT / "_build"
LIB = PKG / "libattn.so"

SOURCES = ["attn_api.cu", "attn_fwd.cu", "attn_bwd.cu", "attn_f32.cu", "attn_bwd_noalloc.cu", "attn_selftest.cu", "attn_att.cu", "attn_decode.cu",
           "attn_fwd_fp8.cu", "attn_linear.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-I", str(INCLUDE), "-I", str(CSRC)]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and pathlib.Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libattn.so")


def _inputs():
    return [CSRC / s for s in SOURCES] + list(CSRC.glob("*.cuh")) + list(INCLUDE.glob("*.h"))


def up_to_date(lib: pathlib.Path = LIB) -> bool:
    if not lib.exists():
        return False
    t = lib.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _inputs())


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    return r


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib: pathlib.Path | None = None,
          build_dir: pathlib.Path | None = None) -> pathlib.Path:
    """Compile and link libattn.so; returns its path.

    `extra_flags` (e.g. a -D that changes a compile-time limit), `lib` and
    `build_dir` build a variant of the library elsewhere, leaving the in-tree
    libattn.so and its objects untouched."""
    lib = LIB if lib is None else pathlib.Path(lib)
    bdir = BUILD if build_dir is None else pathlib.Path(build_dir)
    if not force and up_to_date(lib):
        return lib
    bdir.mkdir(parents=True, exist_ok=True)
    lib.parent.mkdir(parents=True, exist_ok=True)
    cc = nvcc()
    jobs = []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for s in SOURCES:
            obj = bdir / (pathlib.Path(s).stem + ".o")
            cmd = [cc, *NVCC_FLAGS, *extra_flags, "-c", str(CSRC / s), "-o", str(obj)]
            jobs.append((obj, ex.submit(_run, cmd, verbose)))
        objs = []
        for obj, fut in jobs:
            fut.result()
            objs.append(str(obj))
    tmp = lib.with_suffix(".so.tmp")
    _run([cc, *ARCH, "-shared", "-o", str(tmp), *objs], verbose)
    os.replace(tmp, lib)
    return lib


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose))


if __name__ == "__main__":
    sys.exit(main())
