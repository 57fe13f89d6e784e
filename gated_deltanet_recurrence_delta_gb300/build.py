"""Build ``libgdn.so`` in-tree with nvcc for sm_103a (GB300).

Each ``csrc/*.cu`` compiles to an object in parallel, then one shared library
is linked (CUDA runtime linked statically, so loading needs no extra paths).
Usage: ``python -m gated_deltanet_recurrence_delta_gb300.build [--force]``.
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
INCLUDE = PKG.parent / "include"
OUT_DIR = PKG / "_build"
LIB = OUT_DIR / "libgdn.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdn")


def _sources():
    return sorted(CSRC.glob("*.cu"))


def _deps():
    return list(CSRC.glob("*.cu")) + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + list(INCLUDE.glob("*.h"))


def up_to_date(lib: Path = LIB) -> bool:
    if not lib.exists():
        return False
    t = lib.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _deps() + [Path(__file__)])


def build(force: bool = False, verbose: bool = False, out_dir: Path | None = None,
          defines: tuple[str, ...] = ()) -> Path:
    """Build libgdn.so (in-tree by default). out_dir / defines: a separate
    library built with extra preprocessor definitions (the tests' variant
    builds), never the in-tree one."""
    odir = Path(out_dir) if out_dir else OUT_DIR
    lib = odir / "libgdn.so"
    if not force and up_to_date(lib):
        return lib
    odir.mkdir(parents=True, exist_ok=True)
    cc = nvcc()
    srcs = _sources()
    dflags = [f"-D{d}" for d in defines]

    def compile_one(src: Path) -> Path:
        obj = odir / (src.stem + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *dflags, "-I", str(INCLUDE), "-c", str(src), "-o", str(obj)]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src.name}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr, flush=True)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib.with_suffix(f".{os.getpid()}.tmp")
    cmd = [cc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs), "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)
