"""Build the sm_103a C-ABI library in-tree with nvcc.

``python -m nsa_block_selection_gb300.build`` (or ``build()``) compiles
``csrc/*.cu`` into ``nsa_block_selection_gb300/lib/libnsa_sel_attn.so``.
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


def build(out: Optional[str] = None, defines: Iterable[str] = (), verbose: bool = False,
          ptxas_info: bool = False) -> str:
    """Compile the library; returns the path of the shared object."""
    out = out or os.path.join(LIB_DIR, LIB_NAME)
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = [
        nvcc_path(), "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
        "-gencode", GENCODE, "-lineinfo", "-I", INCLUDE, "-I", CSRC,
        "--expt-relaxed-constexpr",
    ]
    if ptxas_info:
        cmd += ["-Xptxas", "-v"]
    cmd += [f"-D{d}" for d in defines]
    cmd += sources() + ["-o", out + ".tmp"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    if ptxas_info or verbose:
        sys.stderr.write(res.stderr)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))
