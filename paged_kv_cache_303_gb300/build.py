"""Build libpagedkv.so (the sm_103a CUDA library) in-tree.

Each .cu translation unit under csrc/ is compiled in parallel by nvcc for
sm_103a only, then linked into paged_kv_cache_303_gb300/libpagedkv.so with a
static CUDA runtime.  Object files go to _build/ at the repository root.
Run ``python -m paged_kv_cache_303_gb300.build`` or call ``build()``.
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
BUILD = ROOT / "_build"
LIB = PKG / "libpagedkv.so"
SOURCES = ["api.cu", "kv_store.cu", "decode.cu", "prefill.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv")


def _flags(verbose: bool):
    f = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", str(ROOT / "include"),
         "--expt-relaxed-constexpr", *ARCH]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _stale(target: Path, deps) -> bool:
    if not target.exists():
        return True
    t = target.stat().st_mtime
    return any(Path(d).stat().st_mtime > t for d in deps)


def build(force: bool = False, verbose: bool = False, jobs: int | None = None) -> Path:
    return _build_into(LIB, BUILD, [], force, verbose, jobs)


def build_test_variant(tag: str, defines, force: bool = False) -> Path:
    """A test-only copy of the library compiled with extra -D definitions
    (for example a short device wait bound and the test hooks), under
    _build/<tag>/.  The product library is never built with them."""
    out = BUILD / tag
    return _build_into(out / f"libpagedkv_{tag}.so", out, [f"-D{d}" for d in defines], force,
                       False, None)


def _build_into(lib: Path, objdir: Path, extra, force, verbose, jobs) -> Path:
    objdir.mkdir(parents=True, exist_ok=True)
    headers = list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + [ROOT / "include" / "pagedkv.h"]
    cc = nvcc()
    objs, todo = [], []
    for src in SOURCES:
        s = CSRC / src
        o = objdir / (s.stem + ".o")
        objs.append(o)
        if force or _stale(o, [s, *headers]):
            todo.append((s, o))

    def compile_one(job):
        s, o = job
        cmd = [cc, *_flags(verbose), *extra, "-c", str(s), "-o", str(o)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {s.name}:\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    if todo:
        with ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            for log in ex.map(compile_one, todo):
                if verbose and log:
                    sys.stderr.write(log)
    if force or todo or _stale(lib, objs):
        tmp = lib.with_suffix(f".so.tmp{os.getpid()}")
        cmd = [cc, "-shared", *ARCH, "-o", str(tmp), *map(str, objs), "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(force="-f" in sys.argv, verbose=v))
