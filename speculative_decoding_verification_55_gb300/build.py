"""Builds libspecverify.so in-tree with nvcc for sm_103a: the translation units compile in
parallel, then link into one shared library (static cudart)."""
from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

PKG_DIR = Path(__file__).resolve().parent
CSRC = PKG_DIR / "csrc"
SOURCES = [CSRC / "sv_api.cu", CSRC / "sv_stream.cu", CSRC / "sv_element.cu", CSRC / "sv_noalloc.cu",
           CSRC / "sv_rollback.cu", CSRC / "sv_threshold.cu", CSRC / "sv_listed.cu",
           CSRC / "sv_staged.cu"]
DEPS = [CSRC / "sv_common.cuh", PKG_DIR.parent / "include" / "spec_verify.h"]
LIB_NAME = "libspecverify.so"
LIB_PATH = PKG_DIR / LIB_NAME

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
]


def find_nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libspecverify.so")


def needs_build() -> bool:
    if not LIB_PATH.exists():
        return True
    lib_m = LIB_PATH.stat().st_mtime
    return any(p.stat().st_mtime > lib_m for p in (*SOURCES, *DEPS, Path(__file__)))


def build_library(force: bool = False, verbose: bool = False, extra_flags=(), out: Path = None) -> Path:
    """Compiles csrc/*.cu and links libspecverify.so next to this file (atomic rename)."""
    out = Path(out) if out is not None else LIB_PATH
    if out == LIB_PATH and not force and not needs_build():
        return LIB_PATH
    nvcc = find_nvcc()
    tag = f"{os.getpid()}"
    objs, procs = [], []
    for src in SOURCES:
        obj = out.parent / f".{src.stem}.{tag}.o"
        cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c", str(src), "-o", str(obj)]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True), cmd))
        objs.append(obj)
    errors = []
    for proc, cmd in procs:
        o, e = proc.communicate()
        if proc.returncode != 0:
            errors.append(f"{' '.join(cmd)}\n{o}\n{e}")
    try:
        if errors:
            raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
        tmp = out.with_suffix(f".so.tmp{tag}")
        cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", str(tmp),
               *[str(o) for o in objs]]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, out)
    finally:
        for o in objs:
            if o.exists():
                o.unlink()
    return out


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
