"""Builds the C-ABI library libqli_gb300.so in-tree (sparse_attention_indexer_qli_gb300/_build/).

Every CUDA source is compiled for sm_103a only (one -gencode), translation
units in parallel, then linked against the shared CUDA runtime so the library
shares the process's runtime with PyTorch. A stamp of the sources and flags
avoids needless rebuilds.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libqli_gb300.so")

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "-I", INCLUDE, "-I", CSRC]
UNITS = ["qli_api.cpp", "qli_plan.cu", "qli_score.cu", "qli_prefill.cu", "qli_select.cu",
         "qli_static.cu", "qli_quant.cu", "qli_attn.cu", "qli_small.cu"]
HEADERS = ["qli_internal.h", "qli_ptx.cuh"]


def _stamp() -> str:
    h = hashlib.sha256()
    for name in UNITS + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(INCLUDE, "qli.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(ARCH + COMMON).encode())
    return h.hexdigest()


def _compile(unit: str, verbose: bool, out_dir: str = OUT_DIR, defines=()) -> str:
    src = os.path.join(CSRC, unit)
    obj = os.path.join(out_dir, unit + ".o")
    cmd = [NVCC] + ARCH + COMMON + ["-D" + d for d in defines] + ["-c", src, "-o", obj]
    if unit.endswith(".cu") and verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (unit, r.stdout, r.stderr))
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, out_dir: str = OUT_DIR,
          defines=()) -> str:
    """Builds the library into out_dir (default: the package's _build/).
    `defines` are extra preprocessor symbols for diagnostic variants."""
    lib = os.path.join(out_dir, "libqli_gb300.so")
    os.makedirs(out_dir, exist_ok=True)
    stamp_path = os.path.join(out_dir, "stamp")
    stamp = _stamp() + ":" + ",".join(defines)
    if not force and os.path.exists(lib) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read() == stamp:
                return lib
    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        objs = list(ex.map(lambda u: _compile(u, verbose, out_dir, defines), UNITS))
    tmp = lib + ".tmp.%d" % os.getpid()
    cmd = [NVCC] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
