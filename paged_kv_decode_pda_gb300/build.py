"""In-tree build of ``libpda.so`` (the C ABI + sm_103a kernels) with nvcc."""

from __future__ import annotations

import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libpda.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared", "-Xptxas", "-v"]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + [os.path.join(ROOT, "include", "pda.h")])


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def build(force: bool = False, verbose: bool = False, out: str = LIB, defines: tuple[str, ...] = ()) -> str:
    """Compile csrc/pda_api.cu (one translation unit) into ``out``."""
    if not force and os.path.exists(out):
        newest = max(os.path.getmtime(s) for s in sources())
        if os.path.getmtime(out) >= newest:
            return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = [nvcc()] + ARCH + FLAGS + ["-D" + d for d in defines] + [os.path.join(CSRC, "pda_api.cu"), "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    if verbose:
        print(r.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    build(force=True, verbose=True)
