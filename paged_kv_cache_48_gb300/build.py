"""Build the sm_103a shared library ``libpagedkv.so`` in-tree with nvcc.

Each CUDA translation unit compiles in parallel to an object under
``_build/``; the objects link into ``paged_kv_cache_48_gb300/libpagedkv.so``.
No relocatable device code, a single ``-gencode`` target (sm_103a).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIBRARY = PKG / "libpagedkv.so"
SOURCES = ["kv_write_zero.cu", "attention_decode.cu", "pkv_api.cu",
           "attention_noalloc.cu", "kv_blocks.cu", "input_prep.cu",
           "attention_prefill.cu"]
HEADERS = ["e4m3_encode.cuh", "pkv_device.cuh", "pkv_host.h", "tcgen05.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
          "-Xcompiler", "-Wall", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    return str(Path(home) / "bin" / "nvcc")


def _stale(target: Path, deps) -> bool:
    if not target.exists():
        return True
    t = target.stat().st_mtime
    return any(Path(d).stat().st_mtime > t for d in deps)


def build(verbose: bool = False, force: bool = False,
          extra_flags: tuple = ()) -> Path:
    """Compile and link the library (incrementally); returns its path."""
    BUILD.mkdir(exist_ok=True)
    nvcc = _nvcc()
    header_deps = [CSRC / h for h in HEADERS] + \
        sorted((PKG.parent / "include").glob("*.h"))

    def compile_one(src: str) -> Path:
        obj = BUILD / (Path(src).stem + ".o")
        deps = [CSRC / src, *header_deps]
        if force or _stale(obj, deps):
            cmd = [nvcc, *ARCH, *CFLAGS, *extra_flags, "-c", str(CSRC / src),
                   "-o", str(obj)]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            subprocess.run(cmd, check=True)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(LIBRARY, objs):
        tmp = LIBRARY.with_name(LIBRARY.name + f".tmp{os.getpid()}")
        cmd = [nvcc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv))
