"""In-tree build of the CUDA libraries with nvcc (sm_103a only).

``build()`` compiles every translation unit of ``csrc/`` in parallel and links
``libeagle.so`` next to this file; it also builds the fixture generator
``fixtures/libfixtures_gen.so``. Rebuilds only when a source is newer than
the library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
LIB = PKG / "libeagle.so"
FIX_SRC = ROOT / "fixtures" / "gen.cu"
FIX_LIB = ROOT / "fixtures" / "libfixtures_gen.so"
FIX_CPU_SRC = ROOT / "fixtures" / "gen_cpu.c"
FIX_CPU_LIB = ROOT / "fixtures" / "libfixtures_cpu.so"
BUILD_DIR = ROOT / "_build"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xcompiler", "-Wall,-Wno-unused-function"]


def nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = Path(cuda) / "bin" / "nvcc"
    return str(p) if p.exists() else (shutil.which("nvcc") or "nvcc")


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")


def _stale(out: Path, srcs: list[Path]) -> bool:
    if not out.exists():
        return True
    t = out.stat().st_mtime
    return any(s.stat().st_mtime > t for s in srcs)


def build_lib(force: bool = False, verbose: bool = False) -> Path:
    cus = sorted(CSRC.glob("*.cu"))
    deps = cus + sorted(CSRC.glob("*.h")) + sorted(CSRC.glob("*.cuh")) + [ROOT / "include" / "eagle.h"]
    if not force and not _stale(LIB, deps):
        return LIB
    BUILD_DIR.mkdir(exist_ok=True)
    objs = [BUILD_DIR / (cu.stem + ".o") for cu in cus]

    def comp(pair):
        cu, o = pair
        _run([nvcc(), *ARCH, *NVCC_FLAGS, "-I", str(ROOT / "include"), "-c", str(cu), "-o", str(o)])
        return o

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        list(ex.map(comp, zip(cus, objs)))
    tmp = LIB.with_suffix(".so.tmp")
    cuda_lib = str(Path(nvcc()).resolve().parent.parent / "lib64")
    _run([nvcc(), *ARCH, "-shared", "-o", str(tmp), *map(str, objs), "-lcudart", "-Xlinker", "-rpath",
          "-Xlinker", cuda_lib])
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}")
    return LIB


def build_fixtures(force: bool = False) -> Path:
    if not force and not _stale(FIX_LIB, [FIX_SRC]):
        return FIX_LIB
    tmp = FIX_LIB.with_suffix(".so.tmp")
    cuda_lib = str(Path(nvcc()).resolve().parent.parent / "lib64")
    _run([nvcc(), *ARCH, *NVCC_FLAGS, "-shared", "-o", str(tmp), str(FIX_SRC), "-Xlinker", "-rpath", "-Xlinker",
          cuda_lib])
    os.replace(tmp, FIX_LIB)
    return FIX_LIB


def build_fixtures_cpu(force: bool = False) -> Path:
    """Host-side fixture generator (gcc + OpenMP; the same recipe as the numpy one)."""
    if not force and not _stale(FIX_CPU_LIB, [FIX_CPU_SRC]):
        return FIX_CPU_LIB
    tmp = FIX_CPU_LIB.with_suffix(".so.tmp")
    _run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math", "-o", str(tmp), str(FIX_CPU_SRC), "-lm"])
    os.replace(tmp, FIX_CPU_LIB)
    return FIX_CPU_LIB


def build(force: bool = False, verbose: bool = False) -> None:
    with ThreadPoolExecutor(max_workers=3) as ex:
        jobs = [ex.submit(build_lib, force, verbose), ex.submit(build_fixtures, force),
                ex.submit(build_fixtures_cpu, force)]
        for j in jobs:
            j.result()


if __name__ == "__main__":
    build(force=True, verbose=True)
