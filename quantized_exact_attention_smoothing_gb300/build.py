"""Builds libsattn.so (the C-ABI library) in-tree with nvcc for sm_103a.

The translation units compile in parallel, then link into
``quantized_exact_attention_smoothing_gb300/_build/libsattn.so`` against the
shared CUDA runtime (so that the library and PyTorch share one runtime).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libsattn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsattn")
    return cand


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "sattn.h"),
                                                                 os.path.abspath(__file__)]


DEBUG_DIR = os.path.join(OUT_DIR, "debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_DIR, "libsattn_dbg.so")


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build_debug(force: bool = False, verbose: bool = False) -> str:
    """The same library built with SATTN_DEBUG_DUMP: the forward kernel can write
    the intermediates of its first tile (raw QK accumulators, P8 bytes, the
    first PV partial) to a buffer set with sattn_debug_set_dump.  For tests."""
    return build(force, verbose, ["-DSATTN_DEBUG_DUMP"], out_dir=DEBUG_DIR, lib_path=DEBUG_LIB_PATH)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          out_dir: str = OUT_DIR, lib_path: str = LIB_PATH) -> str:
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(out_dir, exist_ok=True)
    flags = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
             "-I", os.path.join(ROOT, "include"), *(extra_flags or [])]
    procs, objs = [], []
    for src in sources():
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0 or verbose:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-Xlinker",
           "-rpath," + _cuda_lib_dir(nvcc), *objs, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
