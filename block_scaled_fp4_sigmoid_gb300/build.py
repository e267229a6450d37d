"""Builds libfp4moe.so (the CUDA library behind include/fp4moe.h) in-tree for
sm_103a: every .cu under csrc/ is compiled in parallel with nvcc, then linked
into one shared library (CUDA runtime linked statically).

    python -m block_scaled_fp4_sigmoid_gb300.build [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
SRC = PKG / "csrc"
OUT = PKG / "libfp4moe.so"
BUILD = PKG / "_build"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the fp4moe CUDA library cannot be built")


def _compile(src: Path, obj: Path) -> None:
    cmd = [nvcc(), *ARCH, *FLAGS, "-c", str(src), "-o", str(obj)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src.name}:\n{r.stdout}\n{r.stderr}")


def _stale(out: Path, deps) -> bool:
    if not out.exists():
        return True
    t = out.stat().st_mtime
    return any(d.stat().st_mtime > t for d in deps)


def build_library(force: bool = False, sources: Path = SRC, out: Path = OUT, build_dir: Path = BUILD) -> Path:
    cus = sorted(sources.glob("*.cu"))
    deps = cus + sorted(sources.glob("*.cuh")) + sorted(sources.glob("*.h")) + [PKG.parent / "include" / "fp4moe.h"]
    if not force and not _stale(out, deps):
        return out
    build_dir.mkdir(exist_ok=True)
    objs = [build_dir / (c.stem + ".o") for c in cus]
    with cf.ThreadPoolExecutor(max_workers=min(len(cus), os.cpu_count() or 4)) as ex:
        list(ex.map(lambda p: _compile(*p), zip(cus, objs)))
    tmp = out.with_suffix(".so.tmp")
    cmd = [nvcc(), *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv))
