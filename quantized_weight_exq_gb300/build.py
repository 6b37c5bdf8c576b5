"""Build libexq.so in-tree: one nvcc job per translation unit, in parallel,
for sm_103a only, then a shared-library link with the static CUDA runtime
(so the library loads on hosts without a GPU driver)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIB = PKG / "libexq.so"

SOURCES = ["exq_api.cu", "exq_gemv.cu", "exq_dequant.cu", "exq_gemm.cu", "exq_kv.cu", "exq_convert.cu", "exq_pack.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; libexq needs the CUDA toolkit to build")
    return cand


def _flags(src: str) -> list[str]:
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O3", f"-I{ROOT / 'include'}", f"-I{CSRC}"]
    if src.endswith(".cu"):
        return ARCH + ["-lineinfo", "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"] + common
    return common + ["-x", "c++"]


def _compile(src: str, verbose: bool) -> tuple[str, str]:
    obj = BUILD / (src + ".o")
    s = CSRC / src
    if obj.exists() and obj.stat().st_mtime >= max(
            s.stat().st_mtime, *(p.stat().st_mtime for p in CSRC.glob("*.cuh")),
            *(p.stat().st_mtime for p in CSRC.glob("*.h")), *(p.stat().st_mtime for p in (ROOT / "include").glob("*.h"))):
        return str(obj), ""
    cmd = [nvcc(), "-c", str(s), "-o", str(obj)] + _flags(src)
    if verbose and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return str(obj), r.stdout + r.stderr


def build(verbose: bool = False, force: bool = False) -> Path:
    BUILD.mkdir(exist_ok=True)
    if force:
        for o in BUILD.glob("*.o"):
            o.unlink()
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    if verbose:
        for _, log in results:
            if log:
                print(log)
    objs = [o for o, _ in results]
    if not force and LIB.exists() and LIB.stat().st_mtime >= max(os.path.getmtime(o) for o in objs):
        return LIB
    tmp = LIB.with_suffix(".so.tmp")
    cmd = [nvcc(), "-shared", "-o", str(tmp)] + objs + ARCH + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(verbose="-v" in sys.argv, force="-f" in sys.argv)
    print(LIB)
