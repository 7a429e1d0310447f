"""Build libfvf.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` file is compiled to an object in parallel, then linked
into ``finite_volume_field_gb300/libfvf.so`` (CUDA runtime linked statically,
only the ``include/fvf.h`` symbols exported).  ``-Xptxas -v`` resource usage
(registers, spills, shared memory) of every kernel is written to
``_build/ptxas.txt``.  Run as ``python -m finite_volume_field_gb300.buildlib``.
"""
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
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
LIB = PKG / "libfvf.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    "-O3", "-std=c++17", *ARCH, "-lineinfo",
    # No contraction of multiplies and adds anywhere: the kernels' arithmetic
    # already uses round-to-nearest intrinsics; this is a second guard.
    "--fmad=false",
    "-Xcompiler", "-fPIC,-fvisibility=hidden,-O2",
    "-Xptxas", "-v",
    f"-I{INCLUDE}",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfvf.so")


def sources():
    return sorted(CSRC.glob("*.cu"))


CHECK_BUILD = PKG / "_build_check"
CHECK_LIB = PKG / "libfvf_check.so"


def _stale(lib: Path) -> bool:
    if not lib.exists():
        return True
    t = lib.stat().st_mtime
    deps = list(CSRC.glob("*")) + list(INCLUDE.glob("*.h")) + [Path(__file__)]
    return any(p.stat().st_mtime > t for p in deps)


def build(force: bool = False, verbose: bool = False, bounds_check: bool = False) -> Path:
    """Compile and link libfvf.so if it is missing or older than a source.

    With ``bounds_check`` the same sources are built with
    -DFVF_BOUNDS_CHECK=1 into libfvf_check.so: a debug build (for small
    grids) whose kernels test every global index before using it and record
    a failure instead of accessing memory (read back by fvf_device_error)."""
    lib, build_dir = (CHECK_LIB, CHECK_BUILD) if bounds_check else (LIB, BUILD)
    if not force and not _stale(lib):
        return lib
    build_dir.mkdir(exist_ok=True)
    cc = nvcc()
    extra = ["-DFVF_BOUNDS_CHECK=1"] if bounds_check else []

    def compile_one(src: Path):
        obj = build_dir / (src.stem + ".o")
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", str(src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        results = list(ex.map(compile_one, sources()))
    report = []
    for src, obj, r in results:
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src.name}:\n{r.stdout}\n{r.stderr}")
        report.append(f"== {src.name}\n{r.stderr}")
    (build_dir / "ptxas.txt").write_text("\n".join(report))
    tmp = lib.with_suffix(f".so.tmp{os.getpid()}")
    link = [cc, "-shared", *ARCH, "-cudart", "static", *[str(o) for _, o, _ in results],
            "-o", str(tmp)]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print((build_dir / "ptxas.txt").read_text())
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
