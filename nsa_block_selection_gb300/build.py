"""Build the sm_103a C-ABI library in-tree with nvcc.

``python -m nsa_block_selection_gb300.build`` (or ``build()``) compiles
``csrc/*.cu`` (one object per translation unit, in parallel) and links them
into ``nsa_block_selection_gb300/lib/libnsa_sel_attn.so``.
Only one ``-gencode`` (arch=compute_103a, code=sm_103a) is produced: the
library targets GB300 and nothing else.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from typing import Iterable, Optional

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "lib")
LIB_NAME = "libnsa_sel_attn.so"
GENCODE = "arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def sources() -> list:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile_flags(defines: Iterable[str], ptxas_info: bool) -> list:
    flags = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-gencode", GENCODE, "-lineinfo",
             "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if ptxas_info:
        flags += ["-Xptxas", "-v"]
    return flags + [f"-D{d}" for d in defines]


def build(out: Optional[str] = None, defines: Iterable[str] = (), verbose: bool = False,
          ptxas_info: bool = False) -> str:
    """Compile the library; returns the path of the shared object.

    Each translation unit is compiled to an object in parallel (one
    ``-gencode``), then the objects are linked into the shared library.
    """
    import concurrent.futures as cf

    out = out or os.path.join(LIB_DIR, LIB_NAME)
    os.makedirs(os.path.dirname(out), exist_ok=True)
    objdir = os.path.join(os.path.dirname(out), "_build",
                          os.path.splitext(os.path.basename(out))[0])
    os.makedirs(objdir, exist_ok=True)
    nvcc = nvcc_path()
    flags = _compile_flags(defines, ptxas_info)

    def compile_one(src: str):
        obj = os.path.join(objdir, os.path.splitext(os.path.basename(src))[0] + ".o")
        cmd = [nvcc, "-c"] + flags + [src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        return obj, subprocess.run(cmd, capture_output=True, text=True)

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, srcs))
    errors = [r for _, r in results if r.returncode != 0]
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(r.stdout + r.stderr for r in errors))
    if ptxas_info or verbose:
        for _, r in results:
            sys.stderr.write(r.stderr)
    link = [nvcc, "-shared", "-gencode", GENCODE] + [o for o, _ in results] + ["-o", out + ".tmp"]
    if verbose:
        print(" ".join(link), file=sys.stderr)
    res = subprocess.run(link, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc link failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))
